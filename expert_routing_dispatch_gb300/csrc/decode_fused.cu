// decode_fused.cu -- K6: the whole local MoE layer in one persistent launch.
//
// "Hosting Qwen on Blackwell", section "Expert Parallel": for decode the whole
// expert-parallel kernel is fused into a single kernel (prefill is split into
// several, see the split launches).  Here one cooperative launch of one CTA per
// SM runs, separated by grid-wide barriers:
//   P0  route       every warp of the grid routes tokens (route.cuh)
//   --  barrier 1
//   P1  dispatch    every CTA counts all pairs in shared memory (the offsets and
//                   the tile table need no further exchange), then scatters the
//                   pairs of its own token slice in pair order and copies their
//                   x rows into x_perm
//   --  barrier 2
//   P2  gate/up     grouped tcgen05 GEMM + SiLU*up (grouped_gemm.cuh) -> h, as
//                   bf16 hi + lo terms
//   --  barrier 3
//   P3  down        grouped tcgen05 GEMM over both terms -> y_perm
//   --  barrier 4
//   P4  combine     tokens striped over the CTAs (combine.cuh) -> out
// Intermediates go through global memory; at decode sizes (T*k <= 8192 rows)
// they stay in L2.  TMEM is allocated once for the launch and the mbarrier
// ring carries over between the two GEMM phases.
//
// Every barrier wait is bounded (~1 s of clock cycles): on timeout the CTA sets
// MOE_ERR_TIMEOUT and a global abort word, and all CTAs skip the remaining
// phases, free TMEM and return.  sync[0] (arrivals) and sync[1] (abort) must be
// zero at launch; the launcher clears them on the stream.
#include "combine.cuh"
#include "grouped_gemm.cuh"
#include "kernels.h"
#include "route.cuh"

namespace moe {

namespace {

using namespace gemm;

#ifdef MOE_GEMM_PROFILE
// Tuning builds only: %globaltimer (ns) of every CTA at the phase boundaries of the
// fused launch (after a block barrier), read back by moe_debug_phase_bf.
__device__ unsigned long long g_phase_bf[1024][12];
#define PHASE_STAMP(i)                                                              \
    do {                                                                            \
        __syncthreads();                                                            \
        if (threadIdx.x == 0 && blockIdx.x < 1024) {                                \
            unsigned long long t_;                                                  \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));              \
            g_phase_bf[blockIdx.x][i] = t_;                                          \
        }                                                                           \
    } while (0)
#else
#define PHASE_STAMP(i) ((void)0)
#endif

constexpr long long GRID_WAIT_LIMIT = 1ll << 31;  // clock cycles
constexpr int SMALL_ROWS = 32;                    // token rows of the m-tiles and their boxes
constexpr int FUSED_MAX_CTA_PAIRS = 256;          // pairs of one CTA's token slice (ceil(T / grid) * k)
static_assert(SMALL_ROWS == AR, "token boxes are the GEMM core's m-tiles");

struct FusedArgs {
    const float* logits;
    const uint4* x;
    int32_t* topk_idx;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* row_pair;
    int32_t* pair_row;
    uint4* x_perm;
    uint16_t* h;
    float* y_perm;
    float* out;
    unsigned* sync;
    int32_t* status;
    int T, H, I, E, k, e0, e1;
    int bn;     // MMA N (weight rows per GEMM tile): 256, or 128 when there are few local experts
    int stall;  // testing hook: extra arrivals the first barrier waits for (0 in normal use)
    int gather; // 1: no x_perm; the gate/up GEMM gathers its token rows from x (tile::gather4)
};

struct FusedSmem {
    int hist_before[MAX_LOCAL];  // local pairs of each expert before this CTA's slice
    int cursor[MAX_LOCAL];       // next grouped row of each expert for this CTA
    int prow[FUSED_MAX_CTA_PAIRS];  // grouped row (or -1) of each pair of this CTA's tokens
    int rows[32];
    CombineSmem comb;
    int ok;
};
constexpr size_t FUSED_SMEM_BYTES = SMEM_BYTES + sizeof(FusedSmem);
static_assert(FUSED_SMEM_BYTES <= 232448, "fused kernel exceeds the 227 KB shared-memory limit");

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier number `phase` (1, 2, ...): all CTAs are co-resident
// (cooperative launch).  Returns false, uniformly over the CTA, on timeout or
// when another CTA aborted.
__device__ bool grid_sync(const FusedArgs& a, unsigned target, FusedSmem& fs) {
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        __threadfence();
        atomicAdd(&a.sync[0], 1u);
        const long long t0 = clock64();
        for (;;) {
            if (ld_acquire_gpu(&a.sync[0]) >= target) break;
            if (ld_acquire_gpu(&a.sync[1]) != 0u) {
                ok = 0;
                break;
            }
            if (clock64() - t0 > GRID_WAIT_LIMIT) {
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

__global__ void __launch_bounds__(NUM_THREADS, 1)
    moe_layer_fused_kernel(const __grid_constant__ WMaps wmGU, const __grid_constant__ WMaps wmD,
                           const __grid_constant__ CUtensorMap tmXs, const __grid_constant__ CUtensorMap tmHs,
                           const __grid_constant__ CUtensorMap tmXg, const FusedArgs a) {
    // tmXs / tmHs: x_perm / h with SMALL_ROWS-row boxes, the m-tiles of the GEMM core
    // (decode has ~16 tokens per expert); tmXg: x [T, H] with one-row boxes, the
    // source of the gate/up token rows when a.gather is set
    extern __shared__ uint8_t smem_raw[];
    const uint32_t ring = ring_base(smem_raw);
    Ctl& c = ctl_of(smem_raw);
    FusedSmem& fs = *reinterpret_cast<FusedSmem*>(reinterpret_cast<uint8_t*>(&c) + sizeof(Ctl));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = a.e1 - a.e0;
    const int T = a.T, k = a.k;
    const unsigned G = gridDim.x;

    init(c);
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmXs);
        tma_prefetch_desc(&tmXg);
        tma_prefetch_desc(&tmHs);
        for (int i = 0; i < 3; ++i) {
            tma_prefetch_desc(&wmGU.b0[i]);
            tma_prefetch_desc(&wmGU.b1[i]);
            tma_prefetch_desc(&wmD.b0[i]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    Pipe p;
    pipe_reset(p);
    PHASE_STAMP(0);

    // ---------------- P0: route
    {
        const int warps = NUM_THREADS / 32;
        for (int t = blockIdx.x * warps + warp; t < T; t += G * warps)
            route_token_any(a.logits, t, a.E, k, a.topk_idx, a.topk_w, a.status);
    }
    PHASE_STAMP(1);
    bool ok = grid_sync(a, 1u * G + (unsigned)a.stall, fs);
    PHASE_STAMP(2);

    // ---------------- P1: dispatch
    if (ok) {
        const long long P = (long long)T * k;
        const int tpc = (T + (int)G - 1) / (int)G;
        const int t0 = min(T, (int)blockIdx.x * tpc), t1 = min(T, t0 + tpc);
        const long long p0 = (long long)t0 * k, p1 = (long long)t1 * k;
        int* hist_all = c.tile_start;  // scratch until the tile table is built
        for (int e = threadIdx.x; e < n; e += NUM_THREADS) {
            hist_all[e] = 0;
            fs.hist_before[e] = 0;
        }
        __syncthreads();
        for (long long q0 = threadIdx.x; q0 < P; q0 += 8ll * NUM_THREADS) {
            int ev[8];  // eight independent loads in flight, then the counts
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const long long q = q0 + (long long)u * NUM_THREADS;
                ev[u] = q < P ? __ldcg(a.topk_idx + q) - a.e0 : -1;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const long long q = q0 + (long long)u * NUM_THREADS;
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
        for (int e = threadIdx.x; e < n; e += NUM_THREADS) {
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
        // copy the x rows of this CTA's tokens to their local rows: one item per (token,
        // 16-byte vector), four loads in flight per thread, then their stores
        const int H8 = a.H / 8;
        const int items = a.gather ? 0 : (t1 - t0) * H8;
        for (int i0 = threadIdx.x; i0 < items; i0 += 4 * NUM_THREADS) {
            uint4 val[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * NUM_THREADS;
                if (i < items) val[u] = __ldg(a.x + (size_t)t0 * H8 + i);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u * NUM_THREADS;
                if (i >= items) break;
                const int tl = i / H8, v = i - tl * H8;
                for (int j = 0; j < k; ++j) {
                    const int r = fs.prow[tl * k + j];
                    if (r >= 0) a.x_perm[(size_t)r * H8 + v] = val[u];
                }
            }
        }
        __syncthreads();
        asm volatile("fence.proxy.async.global;" ::: "memory");  // x_perm is read by TMA next
        PHASE_STAMP(3);
        ok = grid_sync(a, 2u * G + (unsigned)a.stall, fs);
        PHASE_STAMP(4);
    }

    // ---------------- P2: gate/up GEMM + SiLU*up
    if (ok) {
        const Args ga{a.h, a.status, n, a.H / BK, (a.I + a.bn / 2 - 1) / (a.bn / 2), a.I, a.I, a.bn / 2, a.bn, 0, 0};
        build_tile_table(c, n, ga.ntiles_n, ga.bn);
        __syncthreads();
        if (a.gather)
            run_phase<MODE_GATEUP>(c, ring, p, &tmXg, &wmGU, ga, a.row_pair, k);
        else
            run_phase<MODE_GATEUP>(c, ring, p, &tmXs, &wmGU, ga);
        PHASE_STAMP(5);
        ok = grid_sync(a, 3u * G + (unsigned)a.stall, fs) && !c.abort_flag;
        PHASE_STAMP(6);
    }

    // ---------------- P3: down GEMM
    if (ok) {
        // h as hi and lo terms: every stage holds a W_down k-block with the hi and the lo
        // k-block of h that use it (K = I weight k-blocks, 2 I columns of h)
        const Args da{a.y_perm, a.status, n, a.I / BK, (a.H + a.bn - 1) / a.bn, a.H, a.H, a.bn, a.bn, 1, 0};
        build_tile_table(c, n, da.ntiles_n, da.bn);
        __syncthreads();
        run_phase<MODE_DOWN>(c, ring, p, &tmHs, &wmD, da);
        PHASE_STAMP(7);
        ok = grid_sync(a, 4u * G + (unsigned)a.stall, fs) && !c.abort_flag;
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
    teardown(c, p, a.status);
    PHASE_STAMP(10);
}

}  // namespace

cudaError_t launch_layer_fused(const uint16_t* x, const float* logits, const uint16_t* w_gate, const uint16_t* w_up,
                               const uint16_t* w_down, float* out, int32_t* topk_idx, float* topk_w,
                               int32_t* counts, int32_t* offsets, int32_t* row_pair, int32_t* pair_row,
                               uint16_t* x_perm, uint16_t* h, float* y_perm, unsigned* sync, int T, int H, int I,
                               int E, int k, int e0, int e1, int32_t* status, int stall_first_barrier,
                               cudaStream_t s, int gather) {
    const cudaError_t attr =
        ensure_dynamic_smem(reinterpret_cast<const void*>(&moe_layer_fused_kernel), (int)FUSED_SMEM_BYTES);
    if (attr != cudaSuccess) return attr;
    const int n = e1 - e0;
    const long long rows = (long long)T * k;
    if ((long long)((T + sm_count() - 1) / sm_count()) * k > FUSED_MAX_CTA_PAIRS) return cudaErrorInvalidConfiguration;
    // 256-row weight tiles.  (128-row tiles for few local experts measured slower:
    // each tile then reloads its token tile for half the work.)
    const int grid = sm_count();
    const int bn = BN;
    CUtensorMap mXs, mHs, mXg;
    WMaps wGU, wD;
    if (!make_tmap_bf16(&mXs, x_perm, rows, H, SMALL_ROWS) || !make_tmap_bf16(&mHs, h, rows, 2 * I, SMALL_ROWS) ||
        !make_tmap_bf16(&mXg, x, T, H, 1) ||
        !make_wmaps(&wGU, w_gate, w_up, (long long)n * I, H, bn / 2) ||
        !make_wmaps(&wD, w_down, nullptr, (long long)n * H, I, bn))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(sync, 0, 2 * sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    FusedArgs a{logits, reinterpret_cast<const uint4*>(x), topk_idx, topk_w, counts, offsets, row_pair, pair_row,
                reinterpret_cast<uint4*>(x_perm), h, y_perm, out, sync, status, T, H, I, E, k, e0, e1, bn,
                stall_first_barrier, gather};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = FUSED_SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_layer_fused_kernel, wGU, wD, mXs, mHs, mXg, a);
}

}  // namespace moe

#ifdef MOE_GEMM_PROFILE
// tuning builds only: the phase timestamps of the fused launch ([1024][12] ns)
extern "C" int moe_debug_phase_bf(unsigned long long* host) {
    return cudaMemcpyFromSymbol(host, moe::g_phase_bf, sizeof(moe::g_phase_bf)) == cudaSuccess ? 0 : 4;
}
#endif
