// grouped_gemm.cuh -- device core of the one-CTA grouped expert GEMMs on the
// tcgen05 tensor cores, used by the fused decode kernel (decode_fused.cu).  The
// split prefill path runs the CTA-pair core of grouped_gemm_pair.cuh instead.
//
// "Hosting Qwen on Blackwell", section "MoE GEMM": the expert FFN is a grouped
// GEMM over the experts, bound by streaming the weights from HBM at decode
// ("Decoders").
//
// Two phases over the grouped rows made by dispatch:
//   gate/up : acc[128 x 256] = x_perm[rows] . [W_gate[e] rows n..n+127 ; W_up[e] rows n..n+127]^T
//             epilogue h = silu(acc[:, 0:128]) * acc[:, 128:256] (fp32 math), stored
//             as two bf16 terms hi + lo in the split layout [rows, 2 I] (common.cuh)
//   down    : acc[128 x 256] = h[rows] . W_down[e][n..n+255]^T over K = I weight
//             k-blocks: each stage holds a W_down k-block with the hi and the lo
//             k-block of h that use it, so y_perm = W_down (hi + lo) (fp32)
// Tiles are (expert, m-tile of 32 rows, n-tile); the tile table is built on
// the device from the row offsets.  Decode has ~16 rows per expert, so a stage
// carries 32-row token k-blocks (4 KB each: gate/up uses one, down its hi and lo)
// next to a 32 KB weight k-block; the MMA keeps M = 128, its A rows 32..127 read
// the bytes after the token slot (inside the ring) and only feed accumulator rows
// that are never stored.  Within an expert the m-tiles of one n-tile are
// consecutive, so CTAs running side by side share a weight tile through L2.
// When the last round of tiles would leave most CTAs idle (r tiles, 2r or 4r <=
// CTAs), each of those r tiles is split along N into 2 or 4 pieces (narrower
// MMA N, weight boxes and epilogue), which spreads the last round over more SMs.
//
// CTA = 6 warps: warp 0 issues TMA loads (128-byte swizzle) into a 5-stage
// shared-memory ring of 40 KB stages (160 KB of weights in flight, in both phases);
// warp 1 owns 512 TMEM columns (two 256-column fp32 accumulators) and issues
// tcgen05.mma (M=128, N=256, K=16) from one elected lane while all 32 lanes run
// the loop; warps 2..5 drain TMEM with tcgen05.ld and run the epilogue while the
// next tile accumulates into the other buffer.
// Every wait is bounded: on timeout the status word gets MOE_ERR_TIMEOUT and
// all roles bail out.
#pragma once

#include "common.cuh"

namespace moe {
namespace gemm {

// MMA shape M = BM, N = BN; BK = 64 bf16 (128-byte rows, 128-byte swizzle);
// m-tiles of AR token rows; 5 ring stages.
constexpr int BM = 128, BN = 256, BK = 64, AR = 32, STAGES = 5;
static_assert(AR <= 32 && AR % 4 == 0, "one producer lane per m-tile row; four-row gathers");
constexpr int ROW_BYTES = BK * 2;     // bytes of one K-row of a tile = swizzle span
constexpr int A_BYTES = AR * BK * 2;  // 4 KB per token k-block
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
// a stage: [token k-block (gate/up; hi of h for down) | lo of h (down) | weight k-block]
constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;
constexpr int MAX_LOCAL = 1024;
constexpr long long WAIT_LIMIT = 1ll << 31;  // clock cycles (~1 s)

enum { MODE_GATEUP = 0, MODE_DOWN = 1 };

// Four rows r0..r3 of a 2-D tensor, columns [c0, c0 + box width), gathered into
// four consecutive box-rows at `dst` (the map's box is one row high); completion
// on `bar` (tx bytes)
__device__ __forceinline__ void tma_gather4_2d(uint32_t dst, const void* tmap, int32_t c0, int32_t r0, int32_t r1,
                                               int32_t r2, int32_t r3, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar), "l"(policy)
        : "memory");
}


struct Ctl {
    // per epilogue warp: a 32-row x 128-byte staging tile (16-byte slots XOR-swizzled by
    // row) that turns per-row TMEM reads into whole 128-byte row segments in global memory
    alignas(128) uint4 stage[AR / 32][32 * 8];
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int tail_first;                 // first tile of the last round
    int tail_shift;                 // its tiles are split into 1 << tail_shift pieces along N
    int tile_total;                 // tiles plus extra pieces: the length of the tile stream
    int tile_start[MAX_LOCAL + 1];  // exclusive prefix of tiles per expert
    int row_off[MAX_LOCAL + 1];     // grouped-row offsets of the local experts
};
constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + (size_t)STAGES * STAGE_BYTES + sizeof(Ctl);

struct Args {
    void* out;        // h bf16 [rows, 2 I] (gate/up, split hi/lo layout) or y_perm fp32 [rows, H] (down)
    int32_t* status;  // device status word or NULL
    int n;            // local experts
    int kblocks;      // k-blocks of the token operand: H / 64 (gate/up) or 2 I / 64 (down)
    int ntiles_n;     // n-tiles per expert
    int out_cols;     // I (gate/up) or H (down)
    int b_rows;       // weight rows per expert in the B tensor map (I or H)
    int n_step;       // output columns per n-tile (bn / 2 for gate/up, bn for down)
    int bn;           // MMA N = weight rows per tile (256; 128 also supported)
    int hilo;         // 1 (down): a stage carries the hi and the lo token k-block of its weight k-block
    int stall;        // testing hook: extra arrivals ring stage 0 waits for (0 in normal use)
};

// Per-thread pipeline counters; they carry over from one GEMM phase to the next
// inside one launch so the mbarrier phases stay in step.
struct Pipe {
    int g;   // k-blocks loaded (producer) / consumed (MMA)
    int it;  // tiles accumulated (MMA) / drained (epilogue)
    int issued[STAGES];
};

struct TileCoord {
    int e, mt, nt, cnt;
    int shift, piece;  // piece `piece` of 1 << shift along N (0, 0 for a whole tile)
};

// Weight maps of one GEMM: box heights of a whole tile and of its half and quarter
// pieces.  b0 = W_gate (gate/up) or W_down, b1 = W_up (gate/up only).
struct WMaps {
    CUtensorMap b0[3];
    CUtensorMap b1[3];
};

// Shared memory: 1024-aligned stage ring followed by the control block.
__device__ __forceinline__ uint32_t ring_base(uint8_t* raw) { return (smem_u32(raw) + 1023u) & ~1023u; }
__device__ __forceinline__ Ctl& ctl_of(uint8_t* raw) {
    const uint32_t b = ring_base(raw);
    return *reinterpret_cast<Ctl*>(raw + (b - smem_u32(raw)) + (size_t)STAGES * STAGE_BYTES);
}

// thread 0: barriers; warp 1: TMEM.  Caller syncs afterwards.  `stall` > 0 (a
// testing hook) makes stage 0's `full` barrier wait for arrivals that never come,
// so the MMA warp's bounded wait runs out and the timeout path is exercised.
__device__ __forceinline__ void init(Ctl& c, int stall = 0) {
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&c.full[s]), 1 + (s == 0 ? stall : 0));
            mbar_init(smem_u32(&c.empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&c.tfull[a]), 1);
            mbar_init(smem_u32(&c.tempty[a]), 4);
        }
        mbar_init(smem_u32(&c.drain), 1);
        c.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&c.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
}

__device__ __forceinline__ void pipe_reset(Pipe& p) {
    p.g = 0;
    p.it = 0;
#pragma unroll
    for (int s = 0; s < STAGES; ++s) p.issued[s] = 0;
}

// warp 0: tile_start from row_off (must be in shared memory already), then the
// split of the last round (pieces at least 64 weight rows wide).
__device__ __forceinline__ void build_tile_table(Ctl& c, int n, int ntiles_n, int bn) {
    if ((threadIdx.x >> 5) != 0) return;
    const int lane = threadIdx.x & 31;
    int carry = 0;
    for (int b0 = 0; b0 < n; b0 += 32) {
        const int e = b0 + lane;
        int v = 0;
        if (e < n) v = ((c.row_off[e + 1] - c.row_off[e] + AR - 1) / AR) * ntiles_n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (e < n) c.tile_start[e + 1] = carry + v;
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) {
        c.tile_start[0] = 0;
        const int total = carry, G = (int)gridDim.x, r = total % G;
        int sh = 0;
        if (r > 0 && 4 * r <= G && (bn >> 2) >= 64)
            sh = 2;
        else if (r > 0 && 2 * r <= G && (bn >> 1) >= 64)
            sh = 1;
        c.tail_first = total - r;
        c.tail_shift = sh;
        c.tile_total = total - r + (r << sh);
    }
}

__device__ __forceinline__ bool next_tile(const Ctl& c, int n, int tile, int& e_hint, TileCoord& tc) {
    if (tile >= c.tile_total) return false;
    int f = tile;  // whole tile of this stream position
    tc.shift = 0;
    tc.piece = 0;
    if (tile >= c.tail_first) {
        const int h = tile - c.tail_first;
        tc.shift = c.tail_shift;
        f = c.tail_first + (h >> tc.shift);
        tc.piece = h & ((1 << tc.shift) - 1);
    }
    int e = e_hint;
    while (c.tile_start[e + 1] <= f) ++e;  // tiles increase monotonically per CTA
    e_hint = e;
    const int cnt = c.row_off[e + 1] - c.row_off[e];
    const int mtiles = (cnt + AR - 1) / AR;
    const int local = f - c.tile_start[e];
    tc.e = e;
    tc.nt = local / mtiles;
    tc.mt = local - tc.nt * mtiles;
    tc.cnt = cnt;
    return true;
}

// One GEMM phase, every thread of the CTA calls it and plays its role.
//   tmA: the token matrix with AR-row boxes, or (gather_pairs != NULL) the token-major
//   x [T, H] with one-row boxes: row i of an m-tile is then x[gather_pairs[row] /
//   gather_k], loaded by tile::gather4, four rows per copy (the grouped copy x_perm is
//   never written).  Rows past the expert's count repeat the m-tile's first token.
template <int MODE>
__device__ __forceinline__ void run_phase(Ctl& c, uint32_t ring, Pipe& p, const CUtensorMap* tmA, const WMaps* wm,
                                          const Args& args, const int32_t* gather_pairs = nullptr,
                                          int gather_k = 1) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = args.n;
    volatile int* abort_flag = &c.abort_flag;
    auto a_addr = [&](int s) { return ring + (uint32_t)(s * STAGE_BYTES); };
    auto b_addr = [&](int s) { return ring + (uint32_t)(s * STAGE_BYTES + 2 * A_BYTES); };

    if (warp == 0) {
        // ================= TMA producer: the whole warp loops, the elected lane issues =================
        const uint64_t pol_a = l2_policy_evict_last();  // token rows are reread for every n-tile
        // a weight tile is read by every m-tile of its expert; the down phase streams its
        // weights while it writes y_perm, which the combine phase reads next, so those
        // weights go first out of L2
        const uint64_t pol_b = MODE == MODE_DOWN ? l2_policy_evict_first() : l2_policy_evict_last();
        int e_hint = 0;
        TileCoord tc;
        bool ok = !__any_sync(0xffffffffu, *abort_flag);
        for (int tile = blockIdx.x; ok && next_tile(c, n, tile, e_hint, tc); tile += gridDim.x) {
            const int a_row = c.row_off[tc.e] + tc.mt * AR;
            const int piece_rows = args.n_step >> tc.shift;  // weight rows of one map's box
            const int b_row = tc.e * args.b_rows + tc.nt * args.n_step + tc.piece * piece_rows;
            const int bn_t = args.bn >> tc.shift;
            const CUtensorMap* tmB0 = &wm->b0[tc.shift];
            const CUtensorMap* tmB1 = &wm->b1[tc.shift];
            const CUtensorMap* tma_a = tmA;
            const uint32_t stage_tx = (uint32_t)((1 + args.hilo) * AR * BK * 2 + bn_t * BK * 2);
            int tok = 0;  // gather: lane i holds the token of m-tile row i (written earlier in the launch)
            if (gather_pairs != nullptr) {
                const int valid = tc.cnt - tc.mt * AR;
                tok = __ldcg(gather_pairs + a_row + (lane < valid ? lane : 0)) / gather_k;
            }
            for (int kb = 0; kb < args.kblocks; ++kb, ++p.g) {
                const int s = p.g % STAGES, r = p.g / STAGES;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c.empty[s]), (r & 1) ^ 1, abort_flag,
                                                               args.status, WAIT_LIMIT))) {
                    ok = false;
                    break;
                }
                p.issued[s] = r + 1;
                const bool leader = elect_one();
                const uint32_t fb = smem_u32(&c.full[s]);
                if (leader) {
                    // Each copy takes ~100 cycles to issue.  Gate/up issues its two weight
                    // boxes before the token box; down keeps the token box first.
                    const int wk = kb * BK;
                    mbar_arrive_expect_tx(fb, stage_tx);
                    if (MODE == MODE_GATEUP) {  // [gate rows | up rows], bn_t/2 each
                        tma_load_2d(b_addr(s), tmB0, wk, b_row, fb, pol_b);
                        tma_load_2d(b_addr(s) + (uint32_t)(bn_t / 2) * BK * 2, tmB1, wk, b_row, fb, pol_b);
                        if (gather_pairs == nullptr) tma_load_2d(a_addr(s), tma_a, kb * BK, a_row, fb, pol_a);
                    } else if (args.hilo) {  // h k-blocks 2 kb (hi) and 2 kb + 1 (lo) of the split layout
                        tma_load_2d(a_addr(s), tma_a, 2 * kb * BK, a_row, fb, pol_a);
                        tma_load_2d(a_addr(s) + (uint32_t)A_BYTES, tma_a, (2 * kb + 1) * BK, a_row, fb, pol_a);
                        tma_load_2d(b_addr(s), tmB0, wk, b_row, fb, pol_b);
                    } else {
                        tma_load_2d(a_addr(s), tma_a, kb * BK, a_row, fb, pol_a);
                        tma_load_2d(b_addr(s), tmB0, wk, b_row, fb, pol_b);
                    }
                }
                if (MODE == MODE_GATEUP && gather_pairs != nullptr) {
                    // AR rows as AR / 4 four-row gathers into consecutive 512-byte row groups
#pragma unroll
                    for (int j = 0; j < AR / 4; ++j) {
                        const int t0 = __shfl_sync(0xffffffffu, tok, 4 * j);
                        const int t1 = __shfl_sync(0xffffffffu, tok, 4 * j + 1);
                        const int t2 = __shfl_sync(0xffffffffu, tok, 4 * j + 2);
                        const int t3 = __shfl_sync(0xffffffffu, tok, 4 * j + 3);
                        if (leader)
                            tma_gather4_2d(a_addr(s) + (uint32_t)(j * 4 * ROW_BYTES), tma_a, kb * BK, t0, t1, t2, t3,
                                           fb, pol_a);
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // ================= MMA issuer: the whole warp loops, the elected lane issues =================
        // (every branch is warp-uniform, so elect_one() always picks the same lane)
        int e_hint = 0;
        TileCoord tc;
        bool ok = !__any_sync(0xffffffffu, *abort_flag);
        const uint64_t a_desc0 = sdesc_k_swz<ROW_BYTES>(a_addr(0)), b_desc0 = sdesc_k_swz<ROW_BYTES>(b_addr(0));
        for (int tile = blockIdx.x; ok && next_tile(c, n, tile, e_hint, tc); tile += gridDim.x, ++p.it) {
            const int acc = p.it & 1, use = p.it >> 1;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c.tempty[acc]), (use & 1) ^ 1, abort_flag,
                                                           args.status, WAIT_LIMIT)))
                break;
            tc_fence_after();
            const uint32_t d_tmem = c.tmem_base + (uint32_t)(acc * BN);
            const uint32_t idesc = idesc_bf16_f32(BM, args.bn >> tc.shift);
            for (int kb = 0; kb < args.kblocks; ++kb, ++p.g) {
                const int s = p.g % STAGES, r = p.g / STAGES;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&c.full[s]), r & 1, abort_flag, args.status,
                                                               WAIT_LIMIT))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    // descriptors are linear in the address (bits 0-13 hold address >> 4)
                    const uint64_t ad = a_desc0 + (uint64_t)((s * STAGE_BYTES) >> 4);
                    const uint64_t bd = b_desc0 + (uint64_t)((s * STAGE_BYTES) >> 4);
                    // hilo: the hi k-block's four MMAs, then the lo k-block's against the same
                    // weight k-block (the order of the split path's down GEMM)
                    for (int sub = 0; sub <= args.hilo; ++sub) {
                        const uint64_t as = ad + (uint64_t)((sub * A_BYTES) >> 4);
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)  // K = 16 bf16 = 32 bytes per MMA
                            tc_mma_bf16(d_tmem, as + 2 * kk, bd + 2 * kk, idesc, (kb | kk | sub) != 0);
                    }
                    tc_commit(smem_u32(&c.empty[s]));
                }
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one()) tc_commit(smem_u32(&c.tfull[acc]));
            __syncwarp();
        }
    } else {
        // ================= epilogue (warps 2..5, TMEM lane quarter = warp % 4) =================
        const int q = warp & 3;
        int e_hint = 0;
        TileCoord tc;
        for (int tile = blockIdx.x; !*abort_flag && next_tile(c, n, tile, e_hint, tc); tile += gridDim.x, ++p.it) {
            const int acc = p.it & 1, use = p.it >> 1;
            if (!mbar_wait_bounded(smem_u32(&c.tfull[acc]), use & 1, abort_flag, args.status, WAIT_LIMIT)) break;
            tc_fence_after();
            const int row0_in_e = tc.mt * AR + q * 32;  // first row of this warp's block
            const long long grow0 = (long long)c.row_off[tc.e] + row0_in_e;
            const uint32_t taddr = c.tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            const int bn_t = args.bn >> tc.shift;
            const int col0 = tc.nt * args.n_step + tc.piece * (args.n_step >> tc.shift);
            uint4* st = c.stage[q < AR / 32 ? q : 0];
            if (q * 32 >= AR) {
                // accumulator rows past the m-tile: computed from stale A rows, not stored
            } else if (MODE == MODE_GATEUP) {
                // 32 h columns per chunk (one half of a 64-column block of the split layout):
                // 64 B of hi and 64 B of lo per row, each staged as 4 slots; slot = piece ^ ((row >> 1) & 3)
                uint16_t* out = static_cast<uint16_t*>(args.out);
                const long long ld = 2ll * args.out_cols;
#pragma unroll 1
                for (int cc = 0; cc < bn_t / 2; cc += 32) {
                    uint32_t g0[16], g1[16], u0[16], u1[16];
                    tmem_ld16(taddr + cc, g0);
                    tmem_ld16(taddr + cc + 16, g1);
                    tmem_ld16(taddr + bn_t / 2 + cc, u0);
                    tmem_ld16(taddr + bn_t / 2 + cc + 16, u1);
                    tmem_ld_wait();
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float a0 = __uint_as_float(g0[2 * i]), a1 = __uint_as_float(g0[2 * i + 1]);
                        const float b0 = __uint_as_float(u0[2 * i]), b1 = __uint_as_float(u0[2 * i + 1]);
                        hi[i] = pack_bf16x2_hi_lo(silu(a0) * b0, silu(a1) * b1, lo[i]);
                        const float c0 = __uint_as_float(g1[2 * i]), c1 = __uint_as_float(g1[2 * i + 1]);
                        const float d0 = __uint_as_float(u1[2 * i]), d1 = __uint_as_float(u1[2 * i + 1]);
                        hi[8 + i] = pack_bf16x2_hi_lo(silu(c0) * d0, silu(c1) * d1, lo[8 + i]);
                    }
                    const int sw = (lane >> 1) & 3;
                    const int hcol = h_hi_col(col0 + cc);
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        const uint32_t* pk = part ? lo : hi;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            st[lane * 4 + (j ^ sw)] =
                                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                        __syncwarp();
                        if (col0 + cc < args.out_cols) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int r = i * 8 + (lane >> 2), piece = lane & 3;
                                const uint4 v = st[r * 4 + (piece ^ ((r >> 1) & 3))];
                                if (row0_in_e + r < tc.cnt)
                                    *reinterpret_cast<uint4*>(out + (grow0 + r) * ld + hcol + 64 * part + 8 * piece) =
                                        v;
                            }
                        }
                        __syncwarp();
                    }
                }
            } else {
                // 32 fp32 columns per chunk: 128 B per row, 8 slots; slot = piece ^ (row & 7)
                float* out = static_cast<float*>(args.out);
#pragma unroll 1
                for (int cc = 0; cc < bn_t; cc += 32) {
                    uint32_t v0[16], v1[16];
                    tmem_ld16(taddr + cc, v0);
                    tmem_ld16(taddr + cc + 16, v1);
                    tmem_ld_wait();
                    const int sw = lane & 7;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        st[lane * 8 + (j ^ sw)] = make_uint4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
                        st[lane * 8 + ((j + 4) ^ sw)] =
                            make_uint4(v1[4 * j], v1[4 * j + 1], v1[4 * j + 2], v1[4 * j + 3]);
                    }
                    __syncwarp();
                    if (col0 + cc < args.out_cols) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int r = i * 4 + (lane >> 3), piece = lane & 7;
                            const uint4 v = st[r * 8 + (piece ^ (r & 7))];
                            if (row0_in_e + r < tc.cnt)
                                *reinterpret_cast<uint4*>(out + (grow0 + r) * args.out_cols + col0 + cc + 4 * piece) = v;
                        }
                    }
                    __syncwarp();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&c.tempty[acc]));
        }
        // the stores above are read later through TMA (async proxy)
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
}

// After a __syncthreads: drain in-flight copies and MMAs (bounded), free TMEM.
__device__ __forceinline__ void teardown(Ctl& c, Pipe& p, int32_t* status) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s)
            if (p.issued[s] > 0) {
                volatile int never = 0;
                mbar_wait_bounded(smem_u32(&c.full[s]), (p.issued[s] - 1) & 1, &never, status, WAIT_LIMIT);
            }
    }
    if (warp == 1) {
        // the lane that issued the MMAs (elect_one() of the converged warp) commits the drain
        if (elect_one()) tc_commit(smem_u32(&c.drain));
        __syncwarp();
        if (lane == 0) {
            volatile int never = 0;
            mbar_wait_bounded(smem_u32(&c.drain), 0, &never, status, WAIT_LIMIT);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(c.tmem_base, TMEM_COLS);
    }
}

}  // namespace gemm
}  // namespace moe
