// grouped_gemm_pair.cuh -- the split path's grouped expert GEMMs on CTA pairs
// (tcgen05 .cta_group::2).
//
// "Hosting Qwen on Blackwell", section "MoE GEMM": the expert FFN is a grouped
// GEMM over the experts, dense at prefill ("Prefillers": ~375 rows per expert).
//
// A cluster of two CTAs (a pair) computes one tile with one MMA stream issued by
// the even CTA: M = 256 weight rows (each CTA holds 128 of them in its own shared
// memory) by N <= 256 tokens of one expert (each CTA holds N / 2 token rows); the
// accumulator of each CTA's 128 weight rows x N tokens sits in its own tensor
// memory.  Per SM and k-block that is 16 KB of weights + up to 16 KB of tokens
// for a 128 x 256 x 64 product, against 48 KB in a one-CTA 128 x 256 tile, and
// the token side pads an expert's rows to a multiple of 16 instead of 128.
//
//   gate/up : CTA r of the pair holds W_gate rows j0..j0+63 and W_up rows
//             j0..j0+63 (j0 = 128 wb + 64 r); its accumulator lanes 0-63 are
//             gate, 64-127 up, for the same h columns.  Epilogue warps of lane
//             quarters q and q+2 swap halves of each 32-token chunk through
//             shared memory and write h = silu(g) * u as two bf16 terms (hi +
//             lo, the split layout [rows, 2 I] of common.cuh), transposed to
//             h[token][column].
//   down    : CTA r holds W_down rows 256 wb + 128 r .. +127; K = 2 I, the token
//             k-blocks alternating hi and lo of h against the same weight k-block;
//             the epilogue writes y_perm[token][column] in fp32, one 128-byte row
//             segment per store.
//
// Tiles are (expert, weight block wb, token tile tt) with tt fastest, so the
// pairs working side by side share each weight block through L2 (a block read by
// two pairs at the same time comes from HBM once).  An expert's c rows are cut
// into ceil(c / 256) token tiles of equal size (a multiple of 16; 375 rows give
// 192 + 183), so the tiles of one expert cost the same.  Cluster c of G takes
// stream positions k G + c for even k and k G + G-1-c for odd k, which evens out
// the differences between experts.  When the last round is sparse (r tiles,
// r <= G / 2), each of its tiles runs as up to 4 pieces along N on different
// pairs, so the last round spreads over more SMs.
//
// Roles (6 warps per CTA): warp 0 issues the TMA loads of its CTA's halves into
// a 6-stage ring, all completing on the even CTA's `full` barrier (.cta_group::2
// copies); warp 1 owns 512 TMEM columns (two 256-column accumulators) and, in the
// even CTA, issues the MMAs and the commits that release both CTAs' ring slots
// and accumulators (multicast); warps 2..5 drain the accumulators and arrive on
// the even CTA's `tempty` barrier.  Every wait is bounded; on timeout the status
// word gets MOE_ERR_TIMEOUT and every role of the CTA stops.
#pragma once

#include "common.cuh"

namespace moe {
namespace pair {

constexpr int WROWS = 128;                   // weight rows per CTA (the pair's MMA M = 256)
constexpr int TN = 256;                      // most tokens per tile (MMA N); each CTA holds up to TN / 2
constexpr int BK = 64;                       // k-block: 64 bf16 = 128-byte rows, 128-byte swizzle
constexpr int STAGES = 6;
constexpr int A_BYTES = WROWS * BK * 2;      // 16 KB
constexpr int B_BYTES = (TN / 2) * BK * 2;   // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 2 * TN;
constexpr int MAX_LOCAL = 1024;
constexpr int TOKEN_BOXES = 8;               // token boxes of 16, 32, ..., 128 rows
constexpr int MAX_TAIL = 256;                // most tiles of a last round that is split into pieces
constexpr int MAX_PIECES = 4;                // pieces per tile of the split last round
constexpr long long WAIT_LIMIT = 1ll << 31;  // clock cycles (~1 s)
// Down GEMM stage layout: one W_down k-block with the hi and the lo token k-blocks
// that use it (48 KB, 4 stages), instead of one token k-block per stage with the
// weight k-block loaded for each (32 KB, 6 stages).
constexpr bool DOWN_SHARED_W = true;

enum { MODE_GATEUP = 0, MODE_DOWN = 1 };

#ifdef MOE_GEMM_PROFILE
// Tuning builds only: clock cycles each role spends waiting, summed over CTAs
// (the MMA entries come from even CTAs only).
// [0] producer waits on a free stage   [1] producer total
// [2] MMA waits on a free accumulator  [3] MMA waits on loaded data  [4] MMA total
// [5] epilogue waits on an accumulator (per warp)  [6] epilogue total (per warp)  [7] tiles
__device__ unsigned long long g_pair_prof[2][8];
#define PAIR_PROF_WAIT(acc, call)               \
    ([&]() {                                    \
        const long long _t = clock64();         \
        const bool _r = (call);                 \
        acc += clock64() - _t;                  \
        return _r;                              \
    }())
#define PAIR_PROF_ADD(i, v) atomicAdd(&g_pair_prof[MODE][i], (unsigned long long)(v))
#else
#define PAIR_PROF_WAIT(acc, call) (call)
#define PAIR_PROF_ADD(i, v) ((void)0)
#endif

struct Ctl {
    // gate/up epilogue exchange: [lane-quarter pair][chunk parity][0: gate tokens 16-31,
    // 1: up tokens 0-15][token][lane]
    float xchg[2][2][2][16][32];
    uint64_t full[STAGES];   // even CTA: both CTAs' copies of a stage (expect-tx) ; odd CTA: unused
    uint64_t empty[STAGES];  // each CTA: its ring slot is free (MMA commit, multicast)
    uint64_t tfull[2];       // each CTA: accumulator ready (MMA commit, multicast)
    uint64_t tempty[2];      // even CTA: accumulator drained by both CTAs' epilogues (8 arrivals)
    uint64_t drain;          // each CTA: all MMAs done (teardown)
    uint64_t xbar[2][2];     // gate/up epilogue: both warps of a quarter pair wrote a chunk's halves (64 arrivals)
    uint32_t tmem_base;
    int abort_flag;
    int tile_start[MAX_LOCAL + 1];  // exclusive prefix of tiles per expert
    int row_off[MAX_LOCAL + 1];     // grouped-row offsets of the local experts
    int tail_first;                 // first tile of the split last round (= tiles when none)
    int stream_len;                 // whole tiles before the last round + pieces of its tiles
    int tail_start[MAX_TAIL + 1];   // exclusive prefix of pieces over the last round's tiles
};
constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + (size_t)STAGES * STAGE_BYTES + sizeof(Ctl);

struct Args {
    void* out;        // h bf16 [rows, I] (gate/up) or y_perm fp32 [rows, H] (down)
    int32_t* status;  // device status word or NULL
    int n;            // local experts
    int kblocks;      // k-blocks of the token operand: H / 64 (gate/up) or 2 I / 64 (down)
    int nwb;          // weight blocks per expert: ceil(I / 128) (gate/up) or ceil(H / 256) (down)
    int out_cols;     // I or H
    int w_rows;       // weight rows per expert in each weight map (I or H)
    int ksplit;       // weight k-block of token k-block kb: kb >> ksplit (1 for down: hi and lo share it)
    int stall;        // testing hook: extra arrivals ring stage 0 waits for (0 in normal use)
};

// w0 = W_gate (64-row boxes) or W_down (128-row boxes), w1 = W_up (64-row boxes,
// gate/up only); tok[i] = the grouped token matrix with 16 (i + 1)-row boxes
struct Maps {
    CUtensorMap w0;
    CUtensorMap w1;
    CUtensorMap tok[TOKEN_BOXES];
};

struct Tile {
    int e, wb, tok0, cnt, ntok;  // expert, weight block, first token (within the expert), rows of the expert,
                                 // tokens in the piece (<= 256)
};



// ------------------------------------------------------------------ cluster PTX
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait (acquire at cluster scope: the phase may be completed by the peer
// CTA); same contract as mbar_wait_bounded.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             int32_t* status, long long limit) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > limit) {
                *abort_flag = 1;
                set_status(status, MOE_ERR_TIMEOUT);
                return false;
            }
        }
    }
}
// 2-D tiled TMA load into this CTA's shared memory whose completion is counted on
// `mbar_cluster` (a shared::cluster address: the even CTA's barrier)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int32_t c0, int32_t c1,
                                                 uint32_t mbar_cluster, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(mbar_cluster), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem of both CTAs] (+)= A[smem of both CTAs] * B[smem of both CTAs]^T (M = 256)
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive once on the barrier at this shared offset in both CTAs of the pair when
// all previously issued tcgen05 operations of this thread have completed
__device__ __forceinline__ void commit_pair(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .b16 m;\n\tmov.b16 m, 3;\n\t"
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], m;\n\t}" ::"r"(
            bar)
        : "memory");
}

// ------------------------------------------------------------------ set-up
__device__ __forceinline__ uint32_t ring_base(uint8_t* raw) { return (smem_u32(raw) + 1023u) & ~1023u; }
__device__ __forceinline__ Ctl& ctl_of(uint8_t* raw) {
    const uint32_t b = ring_base(raw);
    return *reinterpret_cast<Ctl*>(raw + (b - smem_u32(raw)) + (size_t)STAGES * STAGE_BYTES);
}

// thread 0: barriers; warp 1 of each CTA: the pair's TMEM (a collective of the two
// CTAs).  The caller syncs the cluster afterwards.  `stall` > 0 (a testing hook)
// makes stage 0's `full` barrier wait for arrivals that never come.
__device__ __forceinline__ void init(Ctl& c, int stall) {
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&c.full[s]), 1 + (s == 0 ? stall : 0));
            mbar_init(smem_u32(&c.empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&c.tfull[a]), 1);
            mbar_init(smem_u32(&c.tempty[a]), 8);
        }
        mbar_init(smem_u32(&c.drain), 1);
        for (int p = 0; p < 2; ++p)
            for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&c.xbar[p][b]), 64);
        c.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&c.tmem_base), TMEM_COLS);
        tmem_relinquish_pair();
    }
}

// rows of token tile tt of an expert with cnt rows: [tt ts, min(cnt, (tt + 1) ts))
// with ts = ceil(cnt / ntt) rounded up to 16, ntt = ceil(cnt / 256)
__device__ __forceinline__ int token_tiles(int cnt) { return (cnt + TN - 1) / TN; }
__device__ __forceinline__ int token_tile_size(int cnt) {
    const int ntt = token_tiles(cnt);
    return ntt ? (((cnt + ntt - 1) / ntt + 15) & ~15) : 0;
}

// whole tile `tile` of the stream -> expert, weight block, token range
__device__ __forceinline__ void tile_coords(const Ctl& c, int tile, int& e_hint, Tile& t) {
    int e = e_hint;
    while (c.tile_start[e + 1] <= tile) ++e;  // tiles increase along a cluster's stream
    e_hint = e;
    const int cnt = c.row_off[e + 1] - c.row_off[e];
    const int ntt = token_tiles(cnt), ts = token_tile_size(cnt);
    const int local = tile - c.tile_start[e];
    const int tt = local % ntt;
    t.e = e;
    t.wb = local / ntt;
    t.cnt = cnt;
    t.tok0 = tt * ts;
    t.ntok = min(ts, cnt - t.tok0);
}

// pieces of a last-round tile with ntok tokens when the round holds r tiles
__device__ __forceinline__ int tail_pieces(int ntok, int r, int G) {
    int s = min(MAX_PIECES, G / r);
    s = min(s, (ntok + 31) / 32);  // pieces of at least 32 tokens
    return max(s, 1);
}

// warp 0: tile_start from row_off (already in shared memory), then the split of
// a sparse last round.  Every CTA of the grid computes the same table.
__device__ __forceinline__ void build_tile_table(Ctl& c, int n, int nwb, int G) {
    if ((threadIdx.x >> 5) != 0) return;
    const int lane = threadIdx.x & 31;
    int carry = 0;
    for (int b0 = 0; b0 < n; b0 += 32) {
        const int e = b0 + lane;
        int v = 0;
        if (e < n) v = token_tiles(c.row_off[e + 1] - c.row_off[e]) * nwb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (e < n) c.tile_start[e + 1] = carry + v;
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) c.tile_start[0] = 0;
    __syncwarp();
    const int total = carry, r = total % G;
    const bool split = r > 0 && 2 * r <= G && r <= MAX_TAIL;
    const int tail_first = split ? total - r : total;
    int pieces = 0;
    if (split) {
        int e_hint = 0;
        for (int b0 = 0; b0 < r; b0 += 32) {
            const int i = b0 + lane;
            int v = 0;
            if (i < r) {
                Tile t;
                tile_coords(c, tail_first + i, e_hint, t);
                v = tail_pieces(t.ntok, r, G);
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            if (i < r) c.tail_start[i + 1] = pieces + v;
            pieces += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    if (lane == 0) {
        c.tail_start[0] = 0;
        c.tail_first = tail_first;
        c.stream_len = tail_first + pieces;
    }
}

// stream position of this cluster's k-th piece (alternating direction per round)
__device__ __forceinline__ int tile_of(int k, int cid, int G) { return k * G + ((k & 1) ? G - 1 - cid : cid); }

// Stream position -> the piece to compute.  Positions increase along a cluster's
// stream, so the hints only move forward.
__device__ __forceinline__ bool next_tile(const Ctl& c, int pos, int& e_hint, int& tail_hint, Tile& t) {
    if (pos >= c.stream_len) return false;
    if (pos < c.tail_first) {
        tile_coords(c, pos, e_hint, t);
        return true;
    }
    const int q = pos - c.tail_first;
    int i = tail_hint;
    while (c.tail_start[i + 1] <= q) ++i;
    tail_hint = i;
    tile_coords(c, c.tail_first + i, e_hint, t);
    const int s = c.tail_start[i + 1] - c.tail_start[i], p = q - c.tail_start[i];
    const int ps = ((t.ntok + s - 1) / s + 15) & ~15;
    const int lo = min(t.ntok, p * ps), hi = min(t.ntok, (p + 1) * ps);
    t.tok0 += lo;
    t.ntok = hi - lo;
    return true;
}

// MMA N of a tile: its tokens rounded up to 16 (each CTA then holds a whole number
// of 8-row swizzle atoms)
__device__ __forceinline__ int tile_n(const Tile& t) { return (t.ntok + 15) & ~15; }

// ------------------------------------------------------------------ the GEMM
// Every thread of both CTAs calls it and plays its role.
template <int MODE>
__device__ __forceinline__ void run(Ctl& c, uint32_t ring, const Maps* maps, const Args& args) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int cid = (int)cluster_id(), G = (int)cluster_count();
    volatile int* abort_flag = &c.abort_flag;
    // stage geometry: KSUB token k-blocks per weight k-block in each of NST stages of SB bytes
    constexpr bool SHARED_W = MODE == MODE_DOWN && DOWN_SHARED_W;
    constexpr int KSUB = SHARED_W ? 2 : 1;
    constexpr int NST = SHARED_W ? 4 : STAGES;
    constexpr int SB = A_BYTES + KSUB * B_BYTES;
    static_assert(NST * SB <= STAGES * STAGE_BYTES && NST <= STAGES, "stage layout exceeds the ring");
    const int nsteps = args.kblocks / KSUB;
    auto a_addr = [&](int s) { return ring + (uint32_t)(s * SB); };
    auto b_addr = [&](int s) { return ring + (uint32_t)(s * SB + A_BYTES); };
    Tile t;

    if (warp == 0) {
        // ================= TMA producer (both CTAs): the whole warp loops, the elected lane issues
        long long w_empty = 0, t_begin = clock64();
        (void)w_empty;
        (void)t_begin;
        const uint64_t pol_w = l2_policy_evict_last();  // a weight block is read by every token tile of its expert
        const uint64_t pol_t = l2_policy_evict_last();  // token rows are read by every weight block of the expert
        const uint32_t full0 = map_to_rank(smem_u32(&c.full[0]), 0);
        int g = 0;
        bool ok = !__any_sync(0xffffffffu, *abort_flag);
        int e_hint = 0, tail_hint = 0;
        for (int k = 0; ok && next_tile(c, tile_of(k, cid, G), e_hint, tail_hint, t); ++k) {
            if (t.ntok <= 0) continue;  // an empty piece of the split last round: every role skips it
            const int N = tile_n(t), half = N >> 1;
            const int box = (half + 15) / 16 - 1;  // token box of 16 (box + 1) >= half rows
            const int tok_row = c.row_off[t.e] + t.tok0 + (int)rank * half;
            const int w_row = MODE == MODE_GATEUP ? t.e * args.w_rows + t.wb * 128 + (int)rank * 64
                                                  : t.e * args.w_rows + t.wb * 256 + (int)rank * 128;
            const uint32_t stage_tx = 2u * (uint32_t)(A_BYTES + KSUB * 16 * (box + 1) * BK * 2);
            for (int kb = 0; kb < nsteps; ++kb, ++g) {
                const int s = g % NST, r = g / NST;
                if (!__all_sync(0xffffffffu,
                                PAIR_PROF_WAIT(w_empty, wait_bounded(smem_u32(&c.empty[s]), (r & 1) ^ 1, abort_flag,
                                                                     args.status, WAIT_LIMIT)))) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    const uint32_t fb = full0 + (uint32_t)(s * 8);
                    const int wk = (SHARED_W ? kb : kb >> args.ksplit) * BK;  // weight k-block of this stage
                    if (rank == 0) mbar_arrive_expect_tx(smem_u32(&c.full[s]), stage_tx);
                    if (MODE == MODE_GATEUP) {  // [64 gate rows | 64 up rows] of the same h columns
                        tma_load_2d_pair(a_addr(s), &maps->w0, wk, w_row, fb, pol_w);
                        tma_load_2d_pair(a_addr(s) + 64 * BK * 2, &maps->w1, wk, w_row, fb, pol_w);
                    } else {
                        tma_load_2d_pair(a_addr(s), &maps->w0, wk, w_row, fb, pol_w);
                    }
#pragma unroll
                    for (int sub = 0; sub < KSUB; ++sub)  // down, shared W: hi then lo k-block of h
                        tma_load_2d_pair(b_addr(s) + (uint32_t)(sub * B_BYTES), &maps->tok[box], (kb * KSUB + sub) * BK,
                                         tok_row, fb, pol_t);
                }
                __syncwarp();
            }
        }
        if (lane == 0) {
            PAIR_PROF_ADD(0, w_empty);
            PAIR_PROF_ADD(1, clock64() - t_begin);
        }
    } else if (warp == 1) {
        // ================= MMA issuer (even CTA): the whole warp loops, the elected lane issues
        if (rank != 0) return;
        long long w_acc = 0, w_full = 0, t_begin = clock64(), ntiles = 0;
        (void)w_acc;
        (void)w_full;
        (void)t_begin;
        (void)ntiles;
        const uint32_t tmem = c.tmem_base;
        const uint64_t a_desc0 = sdesc_k_swz<128>(a_addr(0)), b_desc0 = sdesc_k_swz<128>(b_addr(0));
        int g = 0;
        bool ok = !__any_sync(0xffffffffu, *abort_flag);
        int e_hint = 0, tail_hint = 0, it = 0;
        for (int k = 0; ok && next_tile(c, tile_of(k, cid, G), e_hint, tail_hint, t); ++k) {
            if (t.ntok <= 0) continue;
            const int acc = it & 1, use = it >> 1;
            ++it;
            ++ntiles;
            if (!__all_sync(0xffffffffu, PAIR_PROF_WAIT(w_acc, wait_bounded(smem_u32(&c.tempty[acc]), (use & 1) ^ 1,
                                                                             abort_flag, args.status, WAIT_LIMIT))))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)(acc * TN);
            const uint32_t idesc = idesc_bf16_f32(2 * WROWS, tile_n(t));
            for (int kb = 0; kb < nsteps; ++kb, ++g) {
                const int s = g % NST, r = g / NST;
                if (!__all_sync(0xffffffffu, PAIR_PROF_WAIT(w_full, wait_bounded(smem_u32(&c.full[s]), r & 1,
                                                                                  abort_flag, args.status,
                                                                                  WAIT_LIMIT)))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    // descriptors are linear in the address (bits 0-13 hold address >> 4)
                    const uint64_t ad = a_desc0 + (uint64_t)((s * SB) >> 4);
                    const uint64_t bd = b_desc0 + (uint64_t)((s * SB) >> 4);
#pragma unroll
                    for (int sub = 0; sub < KSUB; ++sub)
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)  // K = 16 bf16 = 32 bytes per MMA
                            mma_bf16_pair(d_tmem, ad + 2 * kk, bd + (uint64_t)((sub * B_BYTES) >> 4) + 2 * kk, idesc,
                                          (kb | kk | sub) != 0);
                    commit_pair(smem_u32(&c.empty[s]));
                }
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one()) commit_pair(smem_u32(&c.tfull[acc]));
            __syncwarp();
        }
        if (lane == 0) {
            PAIR_PROF_ADD(2, w_acc);
            PAIR_PROF_ADD(3, w_full);
            PAIR_PROF_ADD(4, clock64() - t_begin);
            PAIR_PROF_ADD(7, ntiles);
        }
    } else {
        // ================= epilogue (warps 2..5 of both CTAs; TMEM lane quarter q = warp % 4)
        const int q = warp & 3;
        long long w_tf = 0, t_begin = clock64();
        (void)w_tf;
        (void)t_begin;
        const uint32_t tempty0 = map_to_rank(smem_u32(&c.tempty[0]), 0);
        int chunk_seq = 0;  // chunks exchanged so far (the two warps of a pair count alike)
        int e_hint = 0, tail_hint = 0, it = 0;
        for (int k = 0; !*abort_flag && next_tile(c, tile_of(k, cid, G), e_hint, tail_hint, t); ++k) {
            if (t.ntok <= 0) continue;
            const int acc = it & 1, use = it >> 1;
            ++it;
            if (!PAIR_PROF_WAIT(w_tf, wait_bounded(smem_u32(&c.tfull[acc]), use & 1, abort_flag, args.status,
                                                   WAIT_LIMIT)))
                break;
            tc_fence_after();
            const int N = tile_n(t);
            const int tok0 = t.tok0;  // token (within the expert) of accumulator column 0
            const long long row0 = (long long)c.row_off[t.e] + tok0;
            const uint32_t taddr = c.tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * TN);
            if (MODE == MODE_GATEUP) {
                // quarters 0/1: gate of h columns j0 + 32 q + lane; quarters 2/3: up of the same
                const int j0 = t.wb * 128 + (int)rank * 64;
                const int pr = q & 1;
                const bool is_gate = q < 2;
                const int col = j0 + 32 * pr + lane;
                const int hcol = h_hi_col(col & ~1);  // even column of this lane pair, hi term
                const long long ld = 2ll * args.out_cols;
                uint16_t* out = static_cast<uint16_t*>(args.out);
                if (j0 < args.out_cols) {
#pragma unroll 1
                    for (int cc = 0; cc < N; cc += 32) {
                        uint32_t v0[16], v1[16];
                        tmem_ld16(taddr + cc, v0);
                        tmem_ld16(taddr + cc + 16, v1);
                        tmem_ld_wait();
                        // buffer `par` serves chunks par, par + 2, ...; its barrier completes once per use
                        const int par = chunk_seq & 1, use_x = chunk_seq >> 1;
                        ++chunk_seq;
                        // the gate quarter keeps tokens 0-15 and hands over 16-31; the up quarter the reverse
                        float(*xg)[32] = c.xchg[pr][par][0];
                        float(*xu)[32] = c.xchg[pr][par][1];
                        if (is_gate) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) xg[i][lane] = __uint_as_float(v1[i]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) xu[i][lane] = __uint_as_float(v0[i]);
                        }
                        // bounded, unlike a named barrier: if the partner warp stopped, this one stops too
                        mbar_arrive(smem_u32(&c.xbar[pr][par]));
                        if (!__all_sync(0xffffffffu, wait_bounded(smem_u32(&c.xbar[pr][par]), use_x & 1, abort_flag,
                                                                  args.status, WAIT_LIMIT)))
                            break;
                        float hv[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float g_ = is_gate ? __uint_as_float(v0[i]) : xg[i][lane];
                            const float u_ = is_gate ? xu[i][lane] : __uint_as_float(v1[i]);
                            hv[i] = silu(g_) * u_;
                        }
                        // rows: tokens cc + i (gate quarter) or cc + 16 + i (up quarter).  Lane pairs
                        // swap one value so that each lane stores two adjacent columns of one token,
                        // as hi and lo bf16 terms (split layout [rows, 2 I]).
                        const int tb = cc + (is_gate ? 0 : 16);
                        const int odd = lane & 1;
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const float send = odd ? hv[i] : hv[i + 1];
                            const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
                            uint32_t lo;
                            const uint32_t hi = odd ? pack_bf16x2_hi_lo(recv, hv[i + 1], lo)
                                                    : pack_bf16x2_hi_lo(hv[i], recv, lo);
                            const int tok = tb + i + odd;
                            if (tok < t.ntok) {  // columns past the piece belong to other pieces
                                uint16_t* dst = out + (row0 + tok) * ld + hcol;
                                *reinterpret_cast<uint32_t*>(dst) = hi;
                                *reinterpret_cast<uint32_t*>(dst + 64) = lo;
                            }
                        }
                    }
                }
            } else {
                const int col = t.wb * 256 + (int)rank * 128 + 32 * q + lane;
                float* out = static_cast<float*>(args.out);
                if (col - lane < args.out_cols) {
#pragma unroll 1
                    for (int cc = 0; cc < N; cc += 32) {
                        uint32_t v0[16], v1[16];
                        tmem_ld16(taddr + cc, v0);
                        tmem_ld16(taddr + cc + 16, v1);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int tok = cc + i;
                            if (tok < t.ntok)  // columns past the piece belong to other pieces
                                out[(row0 + tok) * args.out_cols + col] = __uint_as_float(i < 16 ? v0[i] : v1[i - 16]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty0 + (uint32_t)(acc * 8));
        }
        // the stores above are read later through TMA (async proxy)
        asm volatile("fence.proxy.async.global;" ::: "memory");
        if (lane == 0) {
            PAIR_PROF_ADD(5, w_tf);
            PAIR_PROF_ADD(6, clock64() - t_begin);
        }
    }
}

// After a __syncthreads in each CTA: the even CTA's MMAs drain (bounded) and both
// CTAs learn of it; a CTA whose roles stopped early lets its copies in flight land;
// then the cluster syncs (no CTA leaves while its peer may still touch its shared
// memory) and frees the pair's TMEM.
__device__ __forceinline__ void teardown(Ctl& c, int32_t* status) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 1) {
        if (cluster_rank() == 0) {
            // the lane that issued the MMAs (elect_one() of the converged warp) commits the drain
            if (elect_one()) commit_pair(smem_u32(&c.drain));
            __syncwarp();
        }
        if (lane == 0) {
            volatile int never = 0;
            wait_bounded(smem_u32(&c.drain), 0, &never, status, WAIT_LIMIT);
        }
        __syncwarp();
    }
    if (threadIdx.x == 0 && c.abort_flag) {  // copies may still be in flight: let them land
        const long long t0 = clock64();
        while (clock64() - t0 < (1ll << 20)) {
        }
    }
    __syncthreads();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(c.tmem_base, TMEM_COLS);
    }
}

}  // namespace pair
}  // namespace moe
