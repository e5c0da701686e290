// grouped_ffn.cu -- K3/K4: the split-path grouped SwiGLU expert FFN launches.
//
// Two persistent launches over the grouped rows made by dispatch (the prefill
// path of "Hosting Qwen on Blackwell", section "Expert Parallel": the prefill
// layer is split into several kernels): the gate/up GEMM with the SiLU*up
// epilogue writes h (bf16), the down GEMM writes y_perm (fp32).  The tile
// loop, the TMA/tcgen05 pipeline and the epilogues live in grouped_gemm.cuh.
#include <mutex>

#include "grouped_gemm.cuh"
#include "kernels.h"

namespace moe {

namespace {

using namespace gemm;
static_assert(SMEM_BYTES <= 232448, "grouped GEMM exceeds the 227 KB shared-memory limit");

// L2 prefetch of weight boxes by the first m-tile of each weight tile (k-blocks
// ahead; GB300 measurements: down -5% at 6000 tokens and -6% at 16384 with 8,
// gate/up within noise; the fused decode launch is faster without it)
constexpr int kPrefetchGateUp = 0;
constexpr int kPrefetchDown = 8;

struct FfnArgs {
    const int32_t* offsets;
    Args g;
};

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_ffn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ WMaps wm,
                       const FfnArgs args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t ring = ring_base(smem_raw);
    Ctl& c = ctl_of(smem_raw);
    const int n = args.g.n;

    init(c, args.g.stall);
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        for (int i = 0; i < 3; ++i) {
            tma_prefetch_desc(&wm.b0[i]);
            if (MODE == MODE_GATEUP) tma_prefetch_desc(&wm.b1[i]);
        }
    }
    for (int i = threadIdx.x; i <= n; i += NUM_THREADS) c.row_off[i] = __ldg(args.offsets + i);
    __syncthreads();
    build_tile_table(c, n, args.g.ntiles_n, args.g.bn);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    Pipe p;
    pipe_reset(p);
    run_phase<MODE>(c, ring, p, &tmA, &wm, args.g);

    __syncthreads();
    teardown(c, p, args.g.status);
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

template <int MODE>
cudaError_t set_smem_attr() {
    return ensure_dynamic_smem(reinterpret_cast<const void*>(&grouped_ffn_kernel<MODE>), (int)SMEM_BYTES);
}

}  // namespace

size_t ffn_scratch_bytes(long long rows, int I) { return (size_t)rows * (size_t)I * 2; }

cudaError_t launch_gate_up(const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_gate,
                           const uint16_t* w_up, uint16_t* h, long long rows, int H, int I, int n, int32_t* status,
                           cudaStream_t s, int stall) {
    cudaError_t e;
    if ((e = set_smem_attr<MODE_GATEUP>()) != cudaSuccess) return e;
    CUtensorMap mA;
    WMaps wm;
    if (!make_tmap_bf16(&mA, x_perm, rows, H, BM) || !make_wmaps(&wm, w_gate, w_up, (long long)n * I, H, BN / 2))
        return cudaErrorInvalidValue;
    FfnArgs a{offsets,
              {h, status, n, H / BK, (I + BN / 2 - 1) / (BN / 2), I, I, BN / 2, kPrefetchGateUp, BN, 0, stall}};
    grouped_ffn_kernel<MODE_GATEUP><<<sm_count(), NUM_THREADS, SMEM_BYTES, s>>>(mA, wm, a);
    return cudaGetLastError();
}

cudaError_t launch_down(const uint16_t* h, const int32_t* offsets, const uint16_t* w_down, float* y_perm,
                        long long rows, int H, int I, int n, int32_t* status, cudaStream_t s) {
    cudaError_t e;
    if ((e = set_smem_attr<MODE_DOWN>()) != cudaSuccess) return e;
    CUtensorMap mH;
    WMaps wm;
    if (!make_tmap_bf16(&mH, h, rows, I, BM) || !make_wmaps(&wm, w_down, nullptr, (long long)n * H, I, BN))
        return cudaErrorInvalidValue;
    FfnArgs a{offsets, {y_perm, status, n, I / BK, (H + BN - 1) / BN, H, H, BN, kPrefetchDown, BN, 0}};
    grouped_ffn_kernel<MODE_DOWN><<<sm_count(), NUM_THREADS, SMEM_BYTES, s>>>(mH, wm, a);
    return cudaGetLastError();
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
// tuning builds only: reset / read the role wait counters of grouped_gemm.cuh
extern "C" int moe_debug_gemm_prof(unsigned long long* host8, int reset) {
    cudaError_t e = cudaMemcpyFromSymbol(host8, moe::gemm::g_gemm_prof, sizeof(unsigned long long) * 8);
    if (reset) {
        unsigned long long z[8] = {};
        e = cudaMemcpyToSymbol(moe::gemm::g_gemm_prof, z, sizeof(z));
    }
    return e == cudaSuccess ? 0 : 4;
}
#endif
