// grouped_ffn.cu -- K3/K4: the split-path grouped SwiGLU expert FFN launches.
//
// Two persistent launches over the grouped rows made by dispatch (the prefill
// path of "Hosting Qwen on Blackwell", section "Expert Parallel": the prefill
// layer is split into several kernels): the gate/up GEMM with the SiLU*up
// epilogue writes h as two bf16 terms (hi + lo, split layout [rows, 2 I]), the
// down GEMM writes y_perm (fp32) from both terms.  The tile loop, the TMA/tcgen05
// pipeline on CTA pairs and the epilogues live in grouped_gemm_pair.cuh.  This
// file also builds the TMA descriptors that the fused decode kernel uses.
#include <mutex>

#include "grouped_gemm.cuh"
#include "grouped_gemm_pair.cuh"
#include "kernels.h"

namespace moe {

namespace {

using namespace gemm;

static_assert(pair::SMEM_BYTES <= 232448, "CTA-pair GEMM exceeds the 227 KB shared-memory limit");

// The split path's GEMMs: one tile stream over CTA pairs (grouped_gemm_pair.cuh).
template <int MODE>
__global__ void __launch_bounds__(pair::NUM_THREADS, 1)
    grouped_ffn_pair_kernel(const __grid_constant__ pair::Maps maps, const int32_t* __restrict__ offsets,
                            const pair::Args args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t ring = pair::ring_base(smem_raw);
    pair::Ctl& c = pair::ctl_of(smem_raw);
    const int n = args.n;

    pair::init(c, args.stall);
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&maps.w0);
        if (MODE == pair::MODE_GATEUP) tma_prefetch_desc(&maps.w1);
        for (int i = 0; i < pair::TOKEN_BOXES; ++i) tma_prefetch_desc(&maps.tok[i]);
    }
    for (int i = threadIdx.x; i <= n; i += pair::NUM_THREADS) c.row_off[i] = __ldg(offsets + i);
    __syncthreads();
    pair::build_tile_table(c, n, args.nwb, (int)pair::cluster_count());
    tc_fence_before();
    __syncthreads();
    pair::cluster_sync();  // both CTAs' barriers exist before any copy or arrive crosses over
    tc_fence_after();

    pair::run<MODE>(c, ring, &maps, args);

    __syncthreads();
    pair::teardown(c, args.status);
}

}  // namespace

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
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

// bf16 row-major [rows, cols] matrix; box = BK columns x box_rows, swizzle span = BK * 2 bytes
bool make_tmap_bf16(CUtensorMap* m, const void* ptr, long long rows, int cols, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle swz = (BK == 64) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Weight maps of a GEMM whose tiles cover `rows` weight rows of each map: boxes of
// rows, rows / 2 and rows / 4 (the split pieces of the last round)
bool make_wmaps(WMaps* m, const void* w0, const void* w1, long long total_rows, int cols, int rows) {
    for (int i = 0; i < 3; ++i) {
        if (!make_tmap_bf16(&m->b0[i], w0, total_rows, cols, rows >> i)) return false;
        if (!make_tmap_bf16(&m->b1[i], w1 ? w1 : w0, total_rows, cols, rows >> i)) return false;
    }
    return true;
}

namespace {

// Launch a CTA-pair GEMM: as many pairs as fit on the device at once, one tile
// stream over them.
template <int MODE>
cudaError_t launch_pair(const pair::Maps& maps, const int32_t* offsets, const pair::Args& args, cudaStream_t s) {
    const void* fn = reinterpret_cast<const void*>(&grouped_ffn_pair_kernel<MODE>);
    cudaError_t e = ensure_dynamic_smem(fn, (int)pair::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int clusters = 0;
    if ((e = max_active_clusters(fn, 2, pair::NUM_THREADS, (int)pair::SMEM_BYTES, &clusters)) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(pair::NUM_THREADS);
    cfg.dynamicSmemBytes = pair::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, grouped_ffn_pair_kernel<MODE>, maps, offsets, args);
}

// token maps of the pair GEMMs: boxes of 16, 32, ..., 128 rows
bool make_token_maps(pair::Maps* m, const void* tokens, long long rows, int cols) {
    for (int i = 0; i < pair::TOKEN_BOXES; ++i)
        if (!make_tmap_bf16(&m->tok[i], tokens, rows, cols, 16 * (i + 1))) return false;
    return true;
}

}  // namespace

// h as hi and lo bf16 terms: [rows, 2 I]
size_t ffn_scratch_bytes(long long rows, int I) { return (size_t)rows * (size_t)I * 4; }

cudaError_t launch_gate_up(const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_gate,
                           const uint16_t* w_up, uint16_t* h, long long rows, int H, int I, int n, int32_t* status,
                           cudaStream_t s, int stall) {
    pair::Maps maps;
    if (!make_token_maps(&maps, x_perm, rows, H) || !make_tmap_bf16(&maps.w0, w_gate, (long long)n * I, H, 64) ||
        !make_tmap_bf16(&maps.w1, w_up, (long long)n * I, H, 64))
        return cudaErrorInvalidValue;
    const pair::Args a{h, status, n, H / pair::BK, (I + 127) / 128, I, I, 0, stall};
    return launch_pair<pair::MODE_GATEUP>(maps, offsets, a, s);
}

cudaError_t launch_down(const uint16_t* h, const int32_t* offsets, const uint16_t* w_down, float* y_perm,
                        long long rows, int H, int I, int n, int32_t* status, cudaStream_t s) {
    pair::Maps maps;
    if (!make_token_maps(&maps, h, rows, 2 * I) || !make_tmap_bf16(&maps.w0, w_down, (long long)n * H, I, 128))
        return cudaErrorInvalidValue;
    maps.w1 = maps.w0;
    // K = 2 I: the k-blocks alternate hi and lo of h against the same W_down k-block
    const pair::Args a{y_perm, status, n, 2 * I / pair::BK, (H + 255) / 256, H, H, 1, 0};
    return launch_pair<pair::MODE_DOWN>(maps, offsets, a, s);
}

cudaError_t launch_expert_ffn(const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_gate,
                              const uint16_t* w_up, const uint16_t* w_down, float* y_perm, long long rows, int H,
                              int I, int n, void* scratch, int32_t* status, cudaStream_t s) {
    uint16_t* h = static_cast<uint16_t*>(scratch);
    cudaError_t e = launch_gate_up(x_perm, offsets, w_gate, w_up, h, rows, H, I, n, status, s);
    if (e != cudaSuccess) return e;
    return launch_down(h, offsets, w_down, y_perm, rows, H, I, n, status, s);
}

}  // namespace moe

#ifdef MOE_GEMM_PROFILE
// tuning builds only: reset / read the role wait counters of grouped_gemm_pair.cuh
// ([0..7] gate/up, [8..15] down)
extern "C" int moe_debug_gemm_prof(unsigned long long* host16, int reset) {
    cudaError_t e = cudaMemcpyFromSymbol(host16, moe::pair::g_pair_prof, sizeof(unsigned long long) * 16);
    if (reset) {
        unsigned long long z[16] = {};
        e = cudaMemcpyToSymbol(moe::pair::g_pair_prof, z, sizeof(z));
    }
    return e == cudaSuccess ? 0 : 4;
}
#endif
