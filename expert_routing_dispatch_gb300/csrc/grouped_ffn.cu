// grouped_ffn.cu -- K3/K4: grouped SwiGLU expert FFN on the tcgen05 tensor cores.
//
// "Hosting Qwen on Blackwell", section "MoE GEMM": the expert FFN is a grouped
// GEMM over the experts; at ~375 tokens per expert ("Prefillers" section) it is a
// dense, compute-bound problem, while at decode it is bound by streaming the
// expert weights from HBM ("Decoders" section).  The pages use CUTLASS grouped
// GEMMs on GB200; this is a from-scratch sm_103a kernel.
//
// Two persistent launches over the grouped rows produced by dispatch:
//   gate/up : acc[128 x 256] = x_perm[rows] . [W_gate[e] rows n..n+127 ; W_up[e] rows n..n+127]^T
//             epilogue h = bf16(silu(acc[:, 0:128]) * acc[:, 128:256])          (fp32 math)
//   down    : acc[128 x 256] = h[rows] . W_down[e][n..n+255]^T  ->  y_perm = acc (fp32)
// Tiles are (expert, m-tile of 128 rows, n-tile); the tile list is derived on
// the device from offsets (no host sync).  Within an expert the m-tiles of one
// n-tile are consecutive, so CTAs running side by side share the weight tile
// through L2.
//
// CTA = 6 warps: warp 0 issues TMA loads (128-byte swizzle) into a 4-stage
// shared-memory ring; warp 1 allocates 512 TMEM columns (two 256-column fp32
// accumulators) and one thread issues tcgen05.mma (M=128, N=256, K=16);
// warps 2..5 drain TMEM with tcgen05.ld and run the epilogue while the next
// tile accumulates into the other TMEM buffer.  All waits are bounded.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int MAX_LOCAL = 1024;
constexpr long long WAIT_LIMIT = 1ll << 31;  // clock cycles (~1 s)
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

enum { MODE_GATEUP = 0, MODE_DOWN = 1 };

struct Ctl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int tile_start[MAX_LOCAL + 1];  // exclusive prefix of tiles per expert
    int row_off[MAX_LOCAL + 1];     // copy of offsets
};
constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + (size_t)STAGES * STAGE_BYTES + sizeof(Ctl);

struct FfnArgs {
    const int32_t* offsets;
    void* out;          // h bf16 (gate/up) or y_perm fp32 (down), row-major [rows, out_cols]
    int32_t* status;
    int n;              // local experts
    int kblocks;        // K / 64
    int ntiles_n;       // n-tiles per expert
    int out_cols;       // I (gate/up) or H (down)
    int b_rows;         // weight rows per expert in the B tensor map (I or H)
    int n_step;         // output columns per n-tile (128 or 256)
};

struct TileCoord {
    int e, mt, nt, cnt;
};

__device__ __forceinline__ bool next_tile(const Ctl& c, int n, int ntiles_n, int tile, int& e_hint, TileCoord& tc) {
    if (tile >= c.tile_start[n]) return false;
    int e = e_hint;
    while (c.tile_start[e + 1] <= tile) ++e;  // tiles increase monotonically per CTA
    e_hint = e;
    int cnt = c.row_off[e + 1] - c.row_off[e];
    int mtiles = (cnt + BM - 1) / BM;
    int local = tile - c.tile_start[e];
    tc.e = e;
    tc.nt = local / mtiles;
    tc.mt = local - tc.nt * mtiles;
    tc.cnt = cnt;
    (void)ntiles_n;
    return true;
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_ffn_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1, const FfnArgs args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_addr - raw_addr);
    Ctl& c = *reinterpret_cast<Ctl*>(base + (size_t)STAGES * STAGE_BYTES);
    auto a_addr = [&](int s) { return base_addr + (uint32_t)(s * STAGE_BYTES); };
    auto b_addr = [&](int s) { return base_addr + (uint32_t)(s * STAGE_BYTES + A_BYTES); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = args.n;

    // ---- prologue: barriers, TMEM, tile table
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&c.full[s]), 1);
            mbar_init(smem_u32(&c.empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&c.tfull[a]), 1);
            mbar_init(smem_u32(&c.tempty[a]), 4);
        }
        mbar_init(smem_u32(&c.drain), 1);
        c.abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB0);
        if (MODE == MODE_GATEUP) tma_prefetch_desc(&tmB1);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&c.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    for (int i = threadIdx.x; i <= n; i += NUM_THREADS) c.row_off[i] = __ldg(args.offsets + i);
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int b0 = 0; b0 < n; b0 += 32) {
            int e = b0 + lane;
            int v = 0;
            if (e < n) v = ((c.row_off[e + 1] - c.row_off[e] + BM - 1) / BM) * args.ntiles_n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            if (e < n) c.tile_start[e + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) c.tile_start[0] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = c.tmem_base;
    volatile int* abort_flag = &c.abort_flag;

    int issued[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issued[s] = 0;

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            const uint64_t pol_a = l2_policy_evict_last();
            const uint64_t pol_b = l2_policy_evict_first();
            int g = 0, e_hint = 0;
            TileCoord tc;
            bool ok = true;
            for (int tile = blockIdx.x; ok && next_tile(c, n, args.ntiles_n, tile, e_hint, tc); tile += gridDim.x) {
                const int a_row = c.row_off[tc.e] + tc.mt * BM;
                const int b_row = tc.e * args.b_rows + tc.nt * args.n_step;
                for (int kb = 0; kb < args.kblocks; ++kb, ++g) {
                    const int s = g % STAGES, r = g / STAGES;
                    if (!mbar_wait_bounded(smem_u32(&c.empty[s]), (r & 1) ^ 1, abort_flag, args.status, WAIT_LIMIT)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&c.full[s]);
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    issued[s] = r + 1;
                    tma_load_2d(a_addr(s), &tmA, kb * BK, a_row, fb, pol_a);
                    if (MODE == MODE_GATEUP) {
                        tma_load_2d(b_addr(s), &tmB0, kb * BK, b_row, fb, pol_b);
                        tma_load_2d(b_addr(s) + B_BYTES / 2, &tmB1, kb * BK, b_row, fb, pol_b);
                    } else {
                        tma_load_2d(b_addr(s), &tmB0, kb * BK, b_row, fb, pol_b);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            int g = 0, it = 0, e_hint = 0;
            TileCoord tc;
            bool ok = true;
            for (int tile = blockIdx.x; ok && next_tile(c, n, args.ntiles_n, tile, e_hint, tc);
                 tile += gridDim.x, ++it) {
                const int acc = it & 1, use = it >> 1;
                if (!mbar_wait_bounded(smem_u32(&c.tempty[acc]), (use & 1) ^ 1, abort_flag, args.status,
                                       WAIT_LIMIT))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < args.kblocks; ++kb, ++g) {
                    const int s = g % STAGES, r = g / STAGES;
                    if (!mbar_wait_bounded(smem_u32(&c.full[s]), r & 1, abort_flag, args.status, WAIT_LIMIT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = sdesc_k_sw128(a_addr(s) + kk * 32);
                        const uint64_t bd = sdesc_k_sw128(b_addr(s) + kk * 32);
                        tc_mma_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0);
                    }
                    tc_commit(smem_u32(&c.empty[s]));
                }
                if (!ok) break;
                tc_commit(smem_u32(&c.tfull[acc]));
            }
        }
    } else {
        // ================= epilogue (warps 2..5, TMEM lane quarter = warp % 4) =================
        const int q = warp & 3;
        int it = 0, e_hint = 0;
        TileCoord tc;
        for (int tile = blockIdx.x; next_tile(c, n, args.ntiles_n, tile, e_hint, tc); tile += gridDim.x, ++it) {
            const int acc = it & 1, use = it >> 1;
            if (!mbar_wait_bounded(smem_u32(&c.tfull[acc]), use & 1, abort_flag, args.status, WAIT_LIMIT)) break;
            tc_fence_after();
            const int row_in_e = tc.mt * BM + q * 32 + lane;
            const bool valid = row_in_e < tc.cnt;
            const long long grow = (long long)c.row_off[tc.e] + row_in_e;
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            const int col0 = tc.nt * args.n_step;
            if (MODE == MODE_GATEUP) {
                uint16_t* orow = static_cast<uint16_t*>(args.out) + grow * args.out_cols;
#pragma unroll 1
                for (int cc = 0; cc < BN / 2; cc += 16) {
                    uint32_t g[16], u[16];
                    tmem_ld16(taddr + cc, g);
                    tmem_ld16(taddr + BN / 2 + cc, u);
                    tmem_ld_wait();
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                        float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
                        float h0 = g0 / (1.f + __expf(-g0)) * u0;
                        float h1 = g1 / (1.f + __expf(-g1)) * u1;
                        pk[i] = pack_bf16x2(h0, h1);
                    }
                    if (valid && col0 + cc < args.out_cols) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + col0 + cc);
                        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                }
            } else {
                float* orow = static_cast<float*>(args.out) + grow * args.out_cols;
#pragma unroll 1
                for (int cc = 0; cc < BN; cc += 16) {
                    uint32_t v[16];
                    tmem_ld16(taddr + cc, v);
                    tmem_ld_wait();
                    if (valid && col0 + cc < args.out_cols) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + col0 + cc);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&c.tempty[acc]));
        }
    }

    // ---- teardown: drain in-flight copies and MMAs (bounded), free TMEM
    __syncthreads();
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s)
            if (issued[s] > 0) {
                volatile int never = 0;
                mbar_wait_bounded(smem_u32(&c.full[s]), (issued[s] - 1) & 1, &never, args.status, WAIT_LIMIT);
            }
    }
    if (warp == 1) {
        if (lane == 0) {
            tc_commit(smem_u32(&c.drain));
            volatile int never = 0;
            mbar_wait_bounded(smem_u32(&c.drain), 0, &never, args.status, WAIT_LIMIT);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side
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

// bf16 row-major [rows, cols] matrix; box = 64 columns (128 B) x box_rows, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* ptr, long long rows, int cols, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t set_smem_attr() {
    static cudaError_t err = cudaFuncSetAttribute(grouped_ffn_kernel<MODE>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    return err;
}

}  // namespace

size_t ffn_scratch_bytes(long long rows, int I) { return (size_t)rows * (size_t)I * 2; }

cudaError_t launch_gate_up(const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_gate,
                           const uint16_t* w_up, uint16_t* h, long long rows, int H, int I, int n, int32_t* status,
                           cudaStream_t s) {
    cudaError_t e;
    if ((e = set_smem_attr<MODE_GATEUP>()) != cudaSuccess) return e;
    CUtensorMap mA, mG, mU;
    if (!make_map(&mA, x_perm, rows, H, BM) || !make_map(&mG, w_gate, (long long)n * I, H, BN / 2) ||
        !make_map(&mU, w_up, (long long)n * I, H, BN / 2))
        return cudaErrorInvalidValue;
    FfnArgs a{offsets, h, status, n, H / BK, (I + BN / 2 - 1) / (BN / 2), I, I, BN / 2};
    grouped_ffn_kernel<MODE_GATEUP><<<sm_count(), NUM_THREADS, SMEM_BYTES, s>>>(mA, mG, mU, a);
    return cudaGetLastError();
}

cudaError_t launch_down(const uint16_t* h, const int32_t* offsets, const uint16_t* w_down, float* y_perm,
                        long long rows, int H, int I, int n, int32_t* status, cudaStream_t s) {
    cudaError_t e;
    if ((e = set_smem_attr<MODE_DOWN>()) != cudaSuccess) return e;
    CUtensorMap mH, mD;
    if (!make_map(&mH, h, rows, I, BM) || !make_map(&mD, w_down, (long long)n * H, I, BN))
        return cudaErrorInvalidValue;
    FfnArgs a{offsets, y_perm, status, n, I / BK, (H + BN - 1) / BN, H, H, BN};
    grouped_ffn_kernel<MODE_DOWN><<<sm_count(), NUM_THREADS, SMEM_BYTES, s>>>(mH, mD, mD, a);
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
