// mxfp8.cu -- the MXFP8 variant of the expert FFN ("Hosting Qwen on Blackwell",
// section "MoE GEMM": the deployed expert GEMMs run in MXFP8).
//
//   quantise : bf16 rows -> OCP MX v1.0 MXFP8 (E4M3 codes + one UE8M0 scale per 32
//              elements along the row); one thread per 32-element block
//   gather   : the MXFP8 rows of x into the grouped x_perm layout (dispatch)
//   gate/up  : block-scaled tcgen05 GEMM, SiLU*up, h quantised to MXFP8 in the epilogue
//   down     : block-scaled tcgen05 GEMM -> y_perm (fp32)
// The GEMM core is in grouped_gemm_mx.cuh.
#include "combine.cuh"
#include "grouped_gemm_mx.cuh"
#include "kernels.h"
#include "route.cuh"

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

// ------------------------------------------------------------------ dispatch copy
// one CTA per token: its x row is quantised to MXFP8 once (one 32-element block per
// thread, the arithmetic of mx_quantize_kernel) and the codes and scale of each block
// go to every grouped row of its local slots
__global__ void __launch_bounds__(128) mx_dispatch_quantize_kernel(const uint4* __restrict__ x, int H, int k,
                                                                   const int32_t* __restrict__ pair_row,
                                                                   uint8_t* __restrict__ xpq,
                                                                   uint8_t* __restrict__ xps) {
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
    const int nblk = H / 32;
    const uint4* src = x + (size_t)t * (H / 8);
    for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 u = __ldg(src + b * 4 + i);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * i + 2 * j] = bf16_lo(w4[j]);
                v[8 * i + 2 * j + 1] = bf16_hi(w4[j]);
            }
        }
        uint32_t w[8];
        const uint8_t code = (uint8_t)mx::mx_quantize32(v, w);
        for (int i = 0; i < nr; ++i) {
            const size_t row = (size_t)rows[i];
            uint4* dst = reinterpret_cast<uint4*>(xpq + row * H + 32 * b);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            xps[row * nblk + b] = code;
        }
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
    auto& c = mx::ctl_of<mx::GeoPrefill>(smem_raw);
    const int n = args.n;
    mx::init(c, args.stall);
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB0);
        if (MODE == mx::MODE_GATEUP) tma_prefetch_desc(&tmB1);
    }
    for (int i = threadIdx.x; i <= n; i += mx::NUM_THREADS) c.row_off[i] = __ldg(offsets + i);
    __syncthreads();
    mx::build_tile_table<mx::GeoPrefill>(c, n, args.ntiles_n);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    mx::Pipe pipe{0, 0};
    mx::run<MODE, mx::GeoPrefill>(c, ring, pipe, &tmA, &tmB0, &tmB1, args);
    __syncthreads();
    mx::teardown(c, args.status);
}

// ------------------------------------------------------------------ fused decode
// "Hosting Qwen on Blackwell", section "Expert Parallel": for decode the whole
// expert-parallel kernel is one fused kernel.  The MXFP8 layer in one cooperative
// launch of one CTA per SM, phases separated by bounded grid-wide barriers:
//   P0 route; P1 dispatch (every CTA counts all pairs, scatters its own token slice,
//   quantises each of its tokens' x rows to MXFP8 once and writes the codes and
//   scales to every local row); P2 MX gate/up; P3 MX down; P4 combine.  The MX GEMM
//   core (grouped_gemm_mx.cuh) keeps its ring and accumulator counters across P2
//   and P3.  sync[0] (arrivals) and sync[1] (abort) are zero at launch.
#ifdef MOE_GEMM_PROFILE
// Tuning builds only: %globaltimer (ns) of every CTA at the phase boundaries of the
// fused launch (after a block barrier), read back by moe_debug_phase_mx.
__device__ unsigned long long g_phase_mx[1024][12];
#define PHASE_STAMP(i)                                                              \
    do {                                                                            \
        __syncthreads();                                                            \
        if (threadIdx.x == 0 && blockIdx.x < 1024) {                                \
            unsigned long long t_;                                                  \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));              \
            g_phase_mx[blockIdx.x][i] = t_;                                          \
        }                                                                           \
    } while (0)
#else
#define PHASE_STAMP(i) ((void)0)
#endif

constexpr long long MX_GRID_WAIT_LIMIT = 1ll << 31;  // clock cycles (~1 s)
constexpr int MX_SMALL_ROWS = 32;                     // token rows of the fused launch's m-tiles and boxes
constexpr int MX_FUSED_MAX_CTA_PAIRS = 256;           // pairs of one CTA's token slice (ceil(T / grid) * k)

struct MxFusedArgs {
    const float* logits;
    const uint4* x;  // bf16 [T, H] as 16-byte vectors
    int32_t* topk_idx;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* row_pair;
    int32_t* pair_row;
    uint8_t* xpq;  // [T*k, H] E4M3 codes of the grouped rows
    uint8_t* xps;  // [T*k, H/32] their scales
    uint8_t* hq;   // [T*k, I]
    uint8_t* hs;   // [T*k, I/32]
    const uint8_t* wgs;
    const uint8_t* wus;
    const uint8_t* wds;
    float* y_perm;
    float* out;
    unsigned* sync;
    int32_t* status;
    int T, H, I, E, k, e0, e1;
};

struct MxFusedSmem {
    int hist_before[mx::MAX_LOCAL];  // local pairs of each expert before this CTA's slice
    int cursor[mx::MAX_LOCAL];       // next grouped row of each expert for this CTA
    int prow[MX_FUSED_MAX_CTA_PAIRS];  // grouped row (or -1) of each pair of this CTA's tokens
    int rows[32];
    CombineSmem comb;
    int ok;
};
constexpr size_t MX_FUSED_SMEM_BYTES = mx::smem_bytes<mx::GeoDecode>() + sizeof(MxFusedSmem);
static_assert(MX_FUSED_SMEM_BYTES <= 232448, "fused MXFP8 kernel exceeds the 227 KB shared-memory limit");

__device__ __forceinline__ unsigned ld_acquire_gpu_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier (all CTAs co-resident): false, uniformly over the CTA, on
// timeout or when another CTA aborted.
__device__ bool mx_grid_sync(const MxFusedArgs& a, unsigned target, MxFusedSmem& fs) {
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        __threadfence();
        atomicAdd(&a.sync[0], 1u);
        const long long t0 = clock64();
        for (;;) {
            if (ld_acquire_gpu_u32(&a.sync[0]) >= target) break;
            if (ld_acquire_gpu_u32(&a.sync[1]) != 0u) {
                ok = 0;
                break;
            }
            if (clock64() - t0 > MX_GRID_WAIT_LIMIT) {
                atomicExch(&a.sync[1], 1u);
                set_status(a.status, MOE_ERR_TIMEOUT);
                ok = 0;
                break;
            }
            __nanosleep(128);
        }
        __threadfence();
        fs.ok = ok;
    }
    __syncthreads();
    return fs.ok != 0;
}

__global__ void __launch_bounds__(mx::NUM_THREADS, 1)
    moe_layer_mx_fused_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmU,
                              const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmXs,
                              const __grid_constant__ CUtensorMap tmHs, const MxFusedArgs a) {
    // tmXs / tmHs: the x and h codes with MX_SMALL_ROWS-row boxes, the m-tiles of the
    // decode ring geometry (decode has ~16 rows per expert)
    using GD = mx::GeoDecode;
    static_assert(GD::AR == MX_SMALL_ROWS, "token boxes are the decode m-tiles");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t ring = mx::ring_base(smem_raw);
    auto& c = mx::ctl_of<GD>(smem_raw);
    MxFusedSmem& fs = *reinterpret_cast<MxFusedSmem*>(reinterpret_cast<uint8_t*>(&c) + sizeof(c));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = a.e1 - a.e0, T = a.T, k = a.k;
    const unsigned G = gridDim.x;

    mx::init(c, 0);
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmG);
        tma_prefetch_desc(&tmU);
        tma_prefetch_desc(&tmD);
        tma_prefetch_desc(&tmXs);
        tma_prefetch_desc(&tmHs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    mx::Pipe pipe{0, 0};
    PHASE_STAMP(0);

    // ---------------- P0: route
    {
        const int warps = mx::NUM_THREADS / 32;
        for (int t = blockIdx.x * warps + warp; t < T; t += G * warps)
            route_token_any(a.logits, t, a.E, k, a.topk_idx, a.topk_w, a.status);
    }
    PHASE_STAMP(1);
    bool ok = mx_grid_sync(a, 1u * G, fs);
    PHASE_STAMP(2);

    // ---------------- P1: dispatch, x quantised to MXFP8 once per token
    if (ok) {
        const long long P = (long long)T * k;
        const int tpc = (T + (int)G - 1) / (int)G;
        const int t0 = min(T, (int)blockIdx.x * tpc), t1 = min(T, t0 + tpc);
        const long long p0 = (long long)t0 * k, p1 = (long long)t1 * k;
        int* hist_all = c.tile_start;  // scratch until the tile table is built
        for (int e = threadIdx.x; e < n; e += mx::NUM_THREADS) {
            hist_all[e] = 0;
            fs.hist_before[e] = 0;
        }
        __syncthreads();
        for (long long q0 = threadIdx.x; q0 < P; q0 += 8ll * mx::NUM_THREADS) {
            int ev[8];  // eight independent loads in flight, then the counts
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const long long q = q0 + (long long)u * mx::NUM_THREADS;
                ev[u] = q < P ? __ldcg(a.topk_idx + q) - a.e0 : -1;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const long long q = q0 + (long long)u * mx::NUM_THREADS;
                const int e = ev[u];
                if (e >= 0 && e < n) {
                    atomicAdd(&hist_all[e], 1);
                    if (q < p0) atomicAdd(&fs.hist_before[e], 1);
                }
            }
        }
        __syncthreads();
        if (warp == 0) {  // exclusive scan -> row_off
            int carry = 0;
            for (int b0 = 0; b0 < n; b0 += 32) {
                const int e = b0 + lane;
                const int v0 = (e < n) ? hist_all[e] : 0;
                int v = v0;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += y;
                }
                if (e < n) c.row_off[e] = carry + v - v0;
                carry += __shfl_sync(0xffffffffu, v, 31);
            }
            if (lane == 0) c.row_off[n] = carry;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < n; e += mx::NUM_THREADS) {
            fs.cursor[e] = c.row_off[e] + fs.hist_before[e];
            if (blockIdx.x == 0) {
                a.counts[e] = hist_all[e];
                a.offsets[e] = c.row_off[e];
            }
        }
        if (blockIdx.x == 0 && threadIdx.x == 0) a.offsets[n] = c.row_off[n];
        __syncthreads();
        if (warp == 0) {  // this CTA's pairs, in pair order
            const unsigned lt = (1u << lane) - 1u;
            for (long long b = p0; b < p1; b += 32) {
                const long long q = b + lane;
                const bool valid = q < p1;
                const int e = valid ? __ldcg(a.topk_idx + q) - a.e0 : -1;
                const bool local = valid && e >= 0 && e < n;
                const unsigned peers = __match_any_sync(0xffffffffu, local ? e : -1);
                const int base = local ? fs.cursor[e] : 0;
                __syncwarp();
                if (local) {
                    const int row = base + __popc(peers & lt);
                    if ((peers & lt) == 0) fs.cursor[e] = base + __popc(peers);
                    a.row_pair[row] = (int32_t)q;
                    a.pair_row[q] = row;
                    fs.prow[q - p0] = row;
                } else if (valid) {
                    a.pair_row[q] = -1;
                    fs.prow[q - p0] = -1;
                }
                __syncwarp();
            }
        }
        __syncthreads();
        // quantise each token row of this CTA's slice once and copy it to the token's
        // local rows: one item per (token, 32-element block), all in flight together
        const int H8 = a.H / 8, nblk = a.H / 32;
        for (int i = threadIdx.x; i < (t1 - t0) * nblk; i += mx::NUM_THREADS) {
            const int tl = i / nblk, b = i - tl * nblk;
            const size_t t = (size_t)(t0 + tl);
            float v[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 u = __ldg(a.x + t * H8 + b * 4 + j);
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    v[8 * j + 2 * jj] = bf16_lo(w4[jj]);
                    v[8 * j + 2 * jj + 1] = bf16_hi(w4[jj]);
                }
            }
            uint32_t w[8];
            const uint8_t code = (uint8_t)mx::mx_quantize32(v, w);
            for (int j = 0; j < k; ++j) {
                const int r = fs.prow[tl * k + j];
                if (r < 0) continue;
                uint4* dst = reinterpret_cast<uint4*>(a.xpq + (size_t)r * a.H + 32 * b);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                a.xps[(size_t)r * nblk + b] = code;
            }
        }
        __syncthreads();
        asm volatile("fence.proxy.async.global;" ::: "memory");  // xpq is read by TMA next
        PHASE_STAMP(3);
        ok = mx_grid_sync(a, 2u * G, fs);
        PHASE_STAMP(4);
    }

    // ---------------- P2: MX gate/up GEMM + SiLU*up, h quantised to MXFP8
    if (ok) {
        const int nt = (a.I + mx::BN / 2 - 1) / (mx::BN / 2);
        const mx::Args ga{a.hq,
                          a.hs,
                          reinterpret_cast<const uint32_t*>(a.xps),
                          reinterpret_cast<const uint32_t*>(a.wgs),
                          reinterpret_cast<const uint32_t*>(a.wus),
                          (long long)T * k,
                          a.status,
                          n,
                          a.H / mx::BKB,
                          nt,
                          a.I,
                          a.I,
                          mx::BN / 2,
                          0,
                          0};
        mx::build_tile_table<GD>(c, n, nt);
        __syncthreads();
        mx::run<mx::MODE_GATEUP, GD>(c, ring, pipe, &tmXs, &tmG, &tmU, ga);
        mx::pipe_advance(c, pipe, n, ga.kblocks);
        PHASE_STAMP(5);
        ok = mx_grid_sync(a, 3u * G, fs) && !c.abort_flag;
        PHASE_STAMP(6);
    }

    // ---------------- P3: MX down GEMM
    if (ok) {
        const int nt = (a.H + mx::BN - 1) / mx::BN;
        const mx::Args da{a.y_perm,
                          nullptr,
                          reinterpret_cast<const uint32_t*>(a.hs),
                          reinterpret_cast<const uint32_t*>(a.wds),
                          reinterpret_cast<const uint32_t*>(a.wds),
                          (long long)T * k,
                          a.status,
                          n,
                          a.I / mx::BKB,
                          nt,
                          a.H,
                          a.H,
                          mx::BN,
                          0,
                          0};
        mx::build_tile_table<GD>(c, n, nt);
        __syncthreads();
        mx::run<mx::MODE_DOWN, GD>(c, ring, pipe, &tmHs, &tmD, &tmD, da);
        mx::pipe_advance(c, pipe, n, da.kblocks);
        PHASE_STAMP(7);
        ok = mx_grid_sync(a, 4u * G, fs) && !c.abort_flag;
        PHASE_STAMP(8);
    }

    // ---------------- P4: combine
    if (ok) {
        const int H4 = a.H / 4;
        for (int t = blockIdx.x; t < T; t += G)
            combine_token<8>(reinterpret_cast<const float4*>(a.y_perm), a.pair_row, a.topk_w, t, H4, k,
                             reinterpret_cast<float4*>(a.out), fs.comb, true);
    }

    __syncthreads();
    PHASE_STAMP(9);
    mx::teardown(c, a.status);
    PHASE_STAMP(10);
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
        ensure_dynamic_smem(reinterpret_cast<const void*>(&grouped_ffn_mx_kernel<MODE>),
                            (int)mx::smem_bytes<mx::GeoPrefill>());
    if (attr != cudaSuccess) return attr;
    grouped_ffn_mx_kernel<MODE>
        <<<sm_count(), mx::NUM_THREADS, mx::smem_bytes<mx::GeoPrefill>(), s>>>(a, b0, b1, offsets, args);
    return cudaGetLastError();
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

cudaError_t launch_layer_mx_fused(const uint16_t* x, const float* logits, const uint8_t* wgq, const uint8_t* wgs,
                                  const uint8_t* wuq, const uint8_t* wus, const uint8_t* wdq, const uint8_t* wds,
                                  float* out, int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                  int32_t* row_pair, int32_t* pair_row, uint8_t* xpq, uint8_t* xps, uint8_t* hq,
                                  uint8_t* hs, float* y_perm, unsigned* sync, int T, int H, int I, int E, int k,
                                  int e0, int e1, int32_t* status, cudaStream_t s) {
    const cudaError_t attr =
        ensure_dynamic_smem(reinterpret_cast<const void*>(&moe_layer_mx_fused_kernel), (int)MX_FUSED_SMEM_BYTES);
    if (attr != cudaSuccess) return attr;
    const int n = e1 - e0;
    const long long rows = (long long)T * k;
    if ((long long)((T + sm_count() - 1) / sm_count()) * k > MX_FUSED_MAX_CTA_PAIRS) return cudaErrorInvalidConfiguration;
    CUtensorMap mG, mU, mD, mXs, mHs;
    if (!make_tmap_u8(&mG, wgq, (long long)n * I, H, mx::BN / 2) ||
        !make_tmap_u8(&mU, wuq, (long long)n * I, H, mx::BN / 2) ||
        !make_tmap_u8(&mD, wdq, (long long)n * H, I, mx::BN) || !make_tmap_u8(&mXs, xpq, rows, H, MX_SMALL_ROWS) ||
        !make_tmap_u8(&mHs, hq, rows, I, MX_SMALL_ROWS))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(sync, 0, 2 * sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    MxFusedArgs a{logits, reinterpret_cast<const uint4*>(x), topk_idx, topk_w, counts, offsets, row_pair, pair_row,
                  xpq, xps, hq, hs, wgs, wus, wds, y_perm, out, sync, status, T, H, I, E, k, e0, e1};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sm_count());
    cfg.blockDim = dim3(mx::NUM_THREADS);
    cfg.dynamicSmemBytes = MX_FUSED_SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_layer_mx_fused_kernel, mG, mU, mD, mXs, mHs, a);
}

cudaError_t launch_mx_quantize(const uint16_t* src, long long rows, int K, uint8_t* q, uint8_t* s, cudaStream_t st) {
    const long long blocks = rows * (K / 32);
    if (blocks == 0) return cudaSuccess;
    mx_quantize_kernel<<<(unsigned)((blocks + 255) / 256), 256, 0, st>>>(reinterpret_cast<const uint4*>(src), blocks,
                                                                         reinterpret_cast<uint4*>(q), s);
    return cudaGetLastError();
}

cudaError_t launch_mx_dispatch_quantize(const uint16_t* x, int T, int H, int k, const int32_t* pair_row,
                                       uint8_t* xpq, uint8_t* xps, cudaStream_t s) {
    mx_dispatch_quantize_kernel<<<T, 128, 0, s>>>(reinterpret_cast<const uint4*>(x), H, k, pair_row, xpq, xps);
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
                      stall_gate_up,
                      0};
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
                      0,
                      0};
    return launch_mx_gemm<mx::MODE_DOWN>(mH, mD, mD, offsets, da, s);
}

}  // namespace moe

#ifdef MOE_GEMM_PROFILE
// tuning builds only: read (and optionally reset) the role counters of grouped_gemm_mx.cuh
extern "C" int moe_debug_phase_mx(unsigned long long* host) {
    return cudaMemcpyFromSymbol(host, moe::g_phase_mx, sizeof(moe::g_phase_mx)) == cudaSuccess ? 0 : 4;
}
extern "C" int moe_debug_mx_prof(unsigned long long* host24, int reset) {
    cudaError_t e = cudaMemcpyFromSymbol(host24, moe::mx::g_mx_prof, sizeof(unsigned long long) * 24);
    if (reset) {
        unsigned long long z[24] = {};
        e = cudaMemcpyToSymbol(moe::mx::g_mx_prof, z, sizeof(z));
    }
    return e == cudaSuccess ? 0 : 4;
}
#endif
