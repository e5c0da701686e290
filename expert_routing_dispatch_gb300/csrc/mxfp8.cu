// mxfp8.cu -- the MXFP8 variant of the expert FFN ("Hosting Qwen on Blackwell",
// section "MoE GEMM": the deployed expert GEMMs run in MXFP8).
//
//   quantise : bf16 rows -> OCP MX v1.0 MXFP8 (E4M3 codes + one UE8M0 scale per 32
//              elements along the row); one thread per 32-element block
//   gather   : the MXFP8 rows of x into the grouped x_perm layout (dispatch)
//   gate/up  : block-scaled tcgen05 GEMM, SiLU*up, h quantised to MXFP8 in the epilogue
//   down     : block-scaled tcgen05 GEMM -> y_perm (fp32)
// The GEMM core is in grouped_gemm_mx.cuh.
#include "grouped_gemm_mx.cuh"
#include "kernels.h"

namespace moe {

namespace {

// ------------------------------------------------------------------ quantise
// block b of the [rows, K] matrix = elements [32 b, 32 b + 32) of the flat array
__global__ void __launch_bounds__(256) mx_quantize_kernel(const uint4* __restrict__ src, long long blocks,
                                                          uint4* __restrict__ q, uint8_t* __restrict__ s) {
    const long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= blocks) return;
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 u = __ldg(src + b * 4 + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[8 * i + 2 * j] = bf16_lo(w[j]);
            v[8 * i + 2 * j + 1] = bf16_hi(w[j]);
        }
    }
    uint32_t w[8];
    s[b] = (uint8_t)mx::mx_quantize32(v, w);
    q[b * 2] = make_uint4(w[0], w[1], w[2], w[3]);
    q[b * 2 + 1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// ------------------------------------------------------------------ gather
// one CTA per token: its E4M3 row (H16 16-byte vectors) and scale words (S4 per row)
// go to every grouped row of its local slots
__global__ void __launch_bounds__(128) mx_gather_kernel(const uint4* __restrict__ xq, const uint32_t* __restrict__ xs,
                                                        int H16, int S4, int k, const int32_t* __restrict__ pair_row,
                                                        uint4* __restrict__ xpq, uint32_t* __restrict__ xps) {
    __shared__ int rows[32];
    __shared__ int nrows;
    const int t = blockIdx.x;
    if (threadIdx.x < 32) {
        const int r = (threadIdx.x < k) ? __ldg(pair_row + (size_t)t * k + threadIdx.x) : -1;
        const unsigned m = __ballot_sync(0xffffffffu, r >= 0);
        if (r >= 0) rows[__popc(m & ((1u << threadIdx.x) - 1u))] = r;
        if (threadIdx.x == 0) nrows = __popc(m);
    }
    __syncthreads();
    const int nr = nrows;
    if (nr == 0) return;
    for (int v = threadIdx.x; v < H16; v += blockDim.x) {
        const uint4 val = __ldg(xq + (size_t)t * H16 + v);
        for (int i = 0; i < nr; ++i) xpq[(size_t)rows[i] * H16 + v] = val;
    }
    for (int v = threadIdx.x; v < S4; v += blockDim.x) {
        const uint32_t sv = __ldg(xs + (size_t)t * S4 + v);
        for (int i = 0; i < nr; ++i) xps[(size_t)rows[i] * S4 + v] = sv;
    }
}

// ------------------------------------------------------------------ GEMMs
template <int MODE>
__global__ void __launch_bounds__(mx::NUM_THREADS, 1)
    grouped_ffn_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                          const __grid_constant__ CUtensorMap tmB1, const int32_t* __restrict__ offsets,
                          const mx::Args args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t ring = mx::ring_base(smem_raw);
    mx::Ctl& c = mx::ctl_of(smem_raw);
    const int n = args.n;
    mx::init(c, args.stall);
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB0);
        if (MODE == mx::MODE_GATEUP) tma_prefetch_desc(&tmB1);
    }
    for (int i = threadIdx.x; i <= n; i += mx::NUM_THREADS) c.row_off[i] = __ldg(offsets + i);
    __syncthreads();
    mx::build_tile_table(c, n, args.ntiles_n);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    mx::run<MODE>(c, ring, &tmA, &tmB0, &tmB1, args);
    __syncthreads();
    mx::teardown(c, args.status);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// byte matrix [rows, cols]: boxes of 128 bytes x box_rows, 128-byte swizzle
bool make_tmap_u8(CUtensorMap* m, const void* ptr, long long rows, int cols, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {(cuuint32_t)mx::BKB, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_mx_gemm(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                           const int32_t* offsets, const mx::Args& args, cudaStream_t s) {
    const cudaError_t attr =
        ensure_dynamic_smem(reinterpret_cast<const void*>(&grouped_ffn_mx_kernel<MODE>), (int)mx::SMEM_BYTES);
    if (attr != cudaSuccess) return attr;
    grouped_ffn_mx_kernel<MODE><<<sm_count(), mx::NUM_THREADS, mx::SMEM_BYTES, s>>>(a, b0, b1, offsets, args);
    return cudaGetLastError();
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

cudaError_t launch_mx_quantize(const uint16_t* src, long long rows, int K, uint8_t* q, uint8_t* s, cudaStream_t st) {
    const long long blocks = rows * (K / 32);
    if (blocks == 0) return cudaSuccess;
    mx_quantize_kernel<<<(unsigned)((blocks + 255) / 256), 256, 0, st>>>(reinterpret_cast<const uint4*>(src), blocks,
                                                                         reinterpret_cast<uint4*>(q), s);
    return cudaGetLastError();
}

cudaError_t launch_mx_gather(const uint8_t* xq, const uint8_t* xs, int T, int H, int k, const int32_t* pair_row,
                             uint8_t* xpq, uint8_t* xps, cudaStream_t s) {
    mx_gather_kernel<<<T, 128, 0, s>>>(reinterpret_cast<const uint4*>(xq), reinterpret_cast<const uint32_t*>(xs),
                                       H / 16, H / 128, k, pair_row, reinterpret_cast<uint4*>(xpq),
                                       reinterpret_cast<uint32_t*>(xps));
    return cudaGetLastError();
}

size_t mx_ffn_scratch_bytes(long long rows, int I) {
    return align256((size_t)rows * (size_t)I) + align256((size_t)rows * (size_t)(I / 32));
}

cudaError_t launch_mx_expert_ffn(const uint8_t* xq, const uint8_t* xs, const int32_t* offsets, const uint8_t* wgq,
                                 const uint8_t* wgs, const uint8_t* wuq, const uint8_t* wus, const uint8_t* wdq,
                                 const uint8_t* wds, float* y_perm, long long rows, int H, int I, int n,
                                 void* scratch, int32_t* status, cudaStream_t s, int stall_gate_up) {
    uint8_t* hq = static_cast<uint8_t*>(scratch);
    uint8_t* hs = hq + align256((size_t)rows * (size_t)I);
    const int nt_gu = (I + mx::BN / 2 - 1) / (mx::BN / 2), nt_dn = (H + mx::BN - 1) / mx::BN;
    CUtensorMap mX, mG, mU, mH, mD;
    if (!make_tmap_u8(&mX, xq, rows, H, mx::BM) || !make_tmap_u8(&mG, wgq, (long long)n * I, H, mx::BN / 2) ||
        !make_tmap_u8(&mU, wuq, (long long)n * I, H, mx::BN / 2) || !make_tmap_u8(&mH, hq, rows, I, mx::BM) ||
        !make_tmap_u8(&mD, wdq, (long long)n * H, I, mx::BN))
        return cudaErrorInvalidValue;
    const mx::Args ga{hq,
                      hs,
                      reinterpret_cast<const uint32_t*>(xs),
                      reinterpret_cast<const uint32_t*>(wgs),
                      reinterpret_cast<const uint32_t*>(wus),
                      rows,
                      status,
                      n,
                      H / mx::BKB,
                      nt_gu,
                      I,
                      I,
                      mx::BN / 2,
                      stall_gate_up};
    cudaError_t e = launch_mx_gemm<mx::MODE_GATEUP>(mX, mG, mU, offsets, ga, s);
    if (e != cudaSuccess) return e;
    const mx::Args da{y_perm,
                      nullptr,
                      reinterpret_cast<const uint32_t*>(hs),
                      reinterpret_cast<const uint32_t*>(wds),
                      reinterpret_cast<const uint32_t*>(wds),
                      rows,
                      status,
                      n,
                      I / mx::BKB,
                      nt_dn,
                      H,
                      H,
                      mx::BN,
                      0};
    return launch_mx_gemm<mx::MODE_DOWN>(mH, mD, mD, offsets, da, s);
}

}  // namespace moe

#ifdef MOE_GEMM_PROFILE
// tuning builds only: read (and optionally reset) the role counters of grouped_gemm_mx.cuh
extern "C" int moe_debug_mx_prof(unsigned long long* host24, int reset) {
    cudaError_t e = cudaMemcpyFromSymbol(host24, moe::mx::g_mx_prof, sizeof(unsigned long long) * 24);
    if (reset) {
        unsigned long long z[24] = {};
        e = cudaMemcpyToSymbol(moe::mx::g_mx_prof, z, sizeof(z));
    }
    return e == cudaSuccess ? 0 : 4;
}
#endif
