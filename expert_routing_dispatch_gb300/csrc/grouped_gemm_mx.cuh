// grouped_gemm_mx.cuh -- the grouped expert GEMMs with MXFP8 operands on the
// block-scaled tcgen05 tensor cores (kind::mxf8f6f4).
//
// "Hosting Qwen on Blackwell", section "MoE GEMM": the deployed expert GEMMs run
// in MXFP8.  Operands are OCP MX v1.0 MXFP8: E4M3 codes (one byte per element,
// K-major) and one UE8M0 scale per 32 elements along K.  The scales of a row are
// read as 32-bit words, four per 128-element k-block, so K is a multiple of 128.
//
//   gate/up : acc[128 x 192] = x[rows] . [W_gate rows n..n+95 ; W_up rows n..n+95]^T
//             epilogue h = silu(acc[:, 0:96]) * acc[:, 96:192] (fp32), quantised to
//             MXFP8 along I (each 32-column chunk of a row is one MX block)
//   down    : acc[128 x 192] = h[rows] . W_down[e][n..n+191]^T  ->  y_perm (fp32)
//
// One MMA instruction covers K = 32 (one scale per row of A and column of B); a
// 128-byte k-block is four of them, scale ID j picking byte j of each scale word.
// Block-scale factors live in tensor memory: for M = 128 the scale of row m is at
// lane m, column m / 32 of the A slot; the scale of B row n at lane n % 32, column
// n / 32 of the B slot, repeated in every 32-lane quadrant (each quadrant of
// accumulator rows reads the B scales from its own lanes).
//
// CTA = 10 warps: warp 0 issues the TMA loads of the E4M3 tiles into the ring
// (4 stages of 128 token rows + 192 weight rows for the split path, 6 stages of
// 32 token rows + 192 weight rows for the fused decode, see Geo below); warp 1
// owns TMEM (two 192-column accumulators and one 12-column scale slot per stage)
// and one of its threads issues, per k-block, three tcgen05.cp of the stage's
// scale words (shared memory -> TMEM, each 32 rows x 16 bytes copied to all four
// lane quadrants) and the four MMAs, in order in the tensor pipe; warps 2..5 run
// the epilogue; warps 6..9 gather the scale words from global memory into the
// shared-memory chunks of the ring: warp 6 + j fills the stages g with g % 4 == j
// and keeps the words of its next two stages in registers, loading the second
// right after publishing one, so the loads have eight stages of MMAs to land
// before they are needed.
// Every wait is bounded.
#pragma once

#include "common.cuh"

namespace moe {
namespace mx {

constexpr int BM = 128, BN = 192, BKB = 128;  // MMA shape M x N; k-block: 128 E4M3 = 128 bytes per row
constexpr int B_BYTES = BN * BKB;              // 24 KB
constexpr int NUM_THREADS = 320;
constexpr int SCALE_WARPS = 4;
constexpr int ACC_COLS = BN;
constexpr int SF_COL0 = 2 * ACC_COLS;  // first scale slot column (384)
constexpr int SF_SLOT = 12;            // columns per slot: 4 for A, 6 (of 8) for B
constexpr int TMEM_COLS = 512;
constexpr int MAX_LOCAL = 1024;
constexpr long long WAIT_LIMIT = 1ll << 31;

// Ring geometry: AR token rows per m-tile (the rows of a stage's A slot) and S
// stages.  The MMA always has M = 128; with AR = 32 its A rows 32..127 read the
// bytes after the A slot (inside the ring) and only feed accumulator rows that
// are never stored, so a stage carries 4 KB of tokens instead of 16 KB and more
// stages of weights fit in shared memory.
template <int AR_, int S_>
struct Geo {
    static constexpr int AR = AR_;
    static constexpr int STAGES = S_;
    static constexpr int A_BYTES = AR * BKB;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static_assert(AR == 32 || AR == 128, "m-tiles of 32 or 128 token rows");
    static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte alignment of the 128-byte swizzle");
    static_assert(SF_COL0 + S_ * SF_SLOT <= TMEM_COLS, "scale slots exceed the TMEM allocation");
};
using GeoPrefill = Geo<128, 4>;  // split path: 128-token m-tiles, 4 stages of 40 KB
using GeoDecode = Geo<32, 6>;    // fused decode: 32-token m-tiles, 6 stages of 28 KB (144 KB of weights in flight)

enum { MODE_GATEUP = 0, MODE_DOWN = 1 };

#ifdef MOE_GEMM_PROFILE
// Tuning builds only: clock cycles per role, summed over CTAs, per GEMM (gate/up, down).
// [0] producer waits on a free stage [1] producer total [2] MMA waits on an accumulator
// [3] MMA waits on a stage (data and scales) [4] unused [5] MMA total
// [6] epilogue waits (per warp) [7] epilogue total [8] scale warps wait on a free slot
// [9] scale warps total [10] tiles [11] CTAs
__device__ unsigned long long g_mx_prof[2][12];
#define MX_PROF_WAIT(acc, call)                 \
    ([&]() {                                    \
        const long long _t = clock64();         \
        const bool _r = (call);                 \
        acc += clock64() - _t;                  \
        return _r;                              \
    }())
#define MX_PROF_ADD(i, v) atomicAdd(&g_mx_prof[MODE][i], (unsigned long long)(v))
#else
#define MX_PROF_WAIT(acc, call) (call)
#define MX_PROF_ADD(i, v) ((void)0)
#endif

template <int S>
struct Ctl {
    alignas(128) uint4 stage[4][32 * 8];  // down epilogue: 32-row x 128-byte fp32 staging per warp
    // scale words per ring stage: [A | B columns 0-3 | B columns 4-5, 2 spare], each 32 rows x 16 bytes
    alignas(128) uint4 sf[S][3][32];
    uint64_t full[S];  // the stage's TMA bytes (producer's expect-tx arrival) and its scale chunk (scale warp)
    uint64_t empty[S];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
    int tile_start[MAX_LOCAL + 1];
    int row_off[MAX_LOCAL + 1];
};
template <class G>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)G::STAGES * G::STAGE_BYTES + sizeof(Ctl<G::STAGES>);
}
static_assert(smem_bytes<GeoPrefill>() <= 232448, "MX GEMM exceeds the 227 KB shared-memory limit");

struct Args {
    void* out;               // gate/up: h codes uint8 [rows, I]; down: y_perm fp32 [rows, H]
    uint8_t* out_s;          // gate/up: h scales uint8 [rows, I/32]
    const uint32_t* a_s;     // token scale words [a_rows, K/128]
    const uint32_t* b0_s;    // W_gate (gate/up) or W_down scale words [n * w_rows, K/128]
    const uint32_t* b1_s;    // W_up scale words (gate/up)
    long long a_rows;        // rows of the token buffers
    int32_t* status;
    int n;                   // local experts
    int kblocks;             // K / 128
    int ntiles_n;            // n-tiles per expert
    int out_cols;            // I (gate/up) or H (down)
    int w_rows;              // weight rows per expert (I or H)
    int n_step;              // output columns per n-tile: 96 (gate/up) or 192 (down)
    int stall;               // testing hook: extra arrivals ring stage 0 waits for (0 in normal use)
    int a_small;             // box rows of the optional small token map (0 = none)
};

struct TileCoord {
    int e, mt, nt, cnt;
};

// Pipeline counters of one thread: ring k-blocks and accumulator tiles used so far.
// They carry over from one GEMM phase to the next inside one launch (the fused
// decode kernel), so that the mbarrier phases stay in step.
struct Pipe {
    int g;   // k-blocks through the ring
    int it;  // tiles through the two TMEM accumulators
};

// tiles this CTA takes in the current phase (tile_start built)
template <class C>
__device__ __forceinline__ int tiles_of_cta(const C& c, int n) {
    const int total = c.tile_start[n];
    return total > (int)blockIdx.x ? (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
}

__device__ __forceinline__ uint32_t ring_base(uint8_t* raw) { return (smem_u32(raw) + 1023u) & ~1023u; }
template <class G>
__device__ __forceinline__ Ctl<G::STAGES>& ctl_of(uint8_t* raw) {
    const uint32_t b = ring_base(raw);
    return *reinterpret_cast<Ctl<G::STAGES>*>(raw + (b - smem_u32(raw)) + (size_t)G::STAGES * G::STAGE_BYTES);
}

// Instruction descriptor of kind::mxf8f6f4 with E4M3 A and B, UE8M0 scales:
//   bits 4-5 B scale ID, 7-9 A format (0 = E4M3), 10-12 B format, 17-22 N >> 3,
//   23 scale type (1 = UE8M0), 24-28 M >> 4, 29-30 A scale ID
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int sf_id) {
    return ((uint32_t)sf_id << 4) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24) |
           ((uint32_t)sf_id << 29);
}

__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// 32 rows x 16 bytes of shared memory (rows contiguous, no swizzle) -> lanes r of every
// 32-lane quadrant, 4 columns from taddr
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;   // leading byte offset (one 16-byte column)
    d |= (uint64_t)(128u >> 4) << 32;  // stride byte offset: 8-row groups of 16-byte rows
    d |= (uint64_t)1 << 46;            // descriptor version; layout 0 = no swizzle
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

// UE8M0 code of a block whose largest magnitude is amax (OCP MX: floor(log2(amax))
// - 8 + 127, clamped to [0, 254]; 0 for amax = 0 or below the normal range)
__device__ __forceinline__ uint32_t mx_scale_code(float amax) {
    const int eb = (int)((__float_as_uint(amax) >> 23) & 0xffu);  // amax >= 0
    const int c = eb - 8;                                           // floor(log2) - 8 + 127
    return (uint32_t)(c < 0 ? 0 : c > 254 ? 254 : c);
}
// two floats -> two E4M3 codes (round to nearest even, saturating at 448), lo in bits 0..7
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// 32 fp32 values of one MX block -> 32 E4M3 codes (8 words) and the scale code
__device__ __forceinline__ uint32_t mx_quantize32(const float (&v)[32], uint32_t (&w)[8]) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const uint32_t code = mx_scale_code(amax);
    const float inv = __uint_as_float((254u - code) << 23);  // 2^(127 - code): exact
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) | (e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
    return code;
}

// `stall` > 0 (a testing hook) makes stage 0's `full` barrier wait for arrivals
// that never come, so the MMA warp's bounded wait runs out.
template <int S>
__device__ __forceinline__ void init(Ctl<S>& c, int stall = 0) {
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&c.full[s]), 2 + (s == 0 ? stall : 0));
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

// warp 0: tile_start from row_off (m-tiles of G::AR token rows)
template <class G>
__device__ __forceinline__ void build_tile_table(Ctl<G::STAGES>& c, int n, int ntiles_n) {
    if ((threadIdx.x >> 5) != 0) return;
    const int lane = threadIdx.x & 31;
    int carry = 0;
    for (int b0 = 0; b0 < n; b0 += 32) {
        const int e = b0 + lane;
        int v = 0;
        if (e < n) v = ((c.row_off[e + 1] - c.row_off[e] + G::AR - 1) / G::AR) * ntiles_n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        if (e < n) c.tile_start[e + 1] = carry + v;
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) c.tile_start[0] = 0;
}

template <class G>
__device__ __forceinline__ bool next_tile(const Ctl<G::STAGES>& c, int n, int tile, int& e_hint, TileCoord& tc) {
    if (tile >= c.tile_start[n]) return false;
    int e = e_hint;
    while (c.tile_start[e + 1] <= tile) ++e;
    e_hint = e;
    const int cnt = c.row_off[e + 1] - c.row_off[e];
    const int mtiles = (cnt + G::AR - 1) / G::AR;
    const int local = tile - c.tile_start[e];
    tc.e = e;
    tc.nt = local / mtiles;
    tc.mt = local - tc.nt * mtiles;
    tc.cnt = cnt;
    return true;
}

// One GEMM over all tiles; every thread of the CTA calls it and plays its role.
//   tmA: token codes [a_rows, K], 128-row boxes (tmA_small, optional: the same codes
//   with args.a_small-row boxes, loaded for m-tiles with that few rows; the MMA still
//   reads 128 rows and the stale ones only feed output rows that are not stored);
//   tmB0 / tmB1: weight codes with
//   boxes of n_step rows (gate/up: W_gate / W_up) or BN rows (down: W_down twice)
template <int MODE, class G>
__device__ __forceinline__ void run(Ctl<G::STAGES>& c, uint32_t ring, Pipe& pipe, const CUtensorMap* tmA,
                                    const CUtensorMap* tmB0, const CUtensorMap* tmB1, const Args& args,
                                    const CUtensorMap* tmA_small = nullptr) {
    constexpr int STAGES = G::STAGES, STAGE_BYTES = G::STAGE_BYTES, A_BYTES = G::A_BYTES, AR = G::AR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = args.n;
    volatile int* abort_flag = &c.abort_flag;
    auto a_addr = [&](int s) { return ring + (uint32_t)(s * STAGE_BYTES); };
    auto b_addr = [&](int s) { return ring + (uint32_t)(s * STAGE_BYTES + A_BYTES); };
    int e_hint = 0;
    TileCoord tc;

    if (warp == 0) {
        // ================= TMA producer: the whole warp loops, the elected lane issues =================
        long long w0 = 0, t0 = clock64();
        (void)w0;
        (void)t0;
        const uint64_t pol = l2_policy_evict_last();
        // the fused decode's down phase streams its weights once while it writes y_perm,
        // which the combine phase reads next: those weights go first out of L2
        const uint64_t wpol = (AR == 32 && MODE == MODE_DOWN) ? l2_policy_evict_first() : pol;
        int g = pipe.g;
        bool ok = true;
        for (int tile = blockIdx.x; ok && !__any_sync(0xffffffffu, *abort_flag) && next_tile<G>(c, n, tile, e_hint, tc);
             tile += gridDim.x) {
            const int a_row = c.row_off[tc.e] + tc.mt * AR;
            // 128-row m-tiles with few rows load only a small box of tokens
            const bool small = AR == BM && tmA_small != nullptr && tc.cnt - tc.mt * BM <= args.a_small;
            const CUtensorMap* tma = small ? tmA_small : tmA;
            const uint32_t stage_tx = (uint32_t)((small ? args.a_small : AR) * BKB + B_BYTES);
            const int b_row = tc.e * args.w_rows + tc.nt * args.n_step;
            for (int kb = 0; kb < args.kblocks; ++kb, ++g) {
                const int s = g % STAGES, r = g / STAGES;
                if (!__all_sync(0xffffffffu, MX_PROF_WAIT(w0, mbar_wait_bounded(smem_u32(&c.empty[s]), (r & 1) ^ 1,
                                                                               abort_flag, args.status, WAIT_LIMIT)))) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    // gate/up: weight boxes before the token box; down: token box first
                    const uint32_t fb = smem_u32(&c.full[s]);
                    mbar_arrive_expect_tx(fb, stage_tx);
                    if (MODE == MODE_GATEUP) {  // [96 gate rows | 96 up rows]
                        tma_load_2d(b_addr(s), tmB0, kb * BKB, b_row, fb, wpol);
                        tma_load_2d(b_addr(s) + (uint32_t)(BN / 2) * BKB, tmB1, kb * BKB, b_row, fb, wpol);
                        tma_load_2d(a_addr(s), tma, kb * BKB, a_row, fb, pol);
                    } else {
                        tma_load_2d(a_addr(s), tma, kb * BKB, a_row, fb, pol);
                        tma_load_2d(b_addr(s), tmB0, kb * BKB, b_row, fb, wpol);
                    }
                }
                __syncwarp();
            }
        }
        if (lane == 0) {
            MX_PROF_ADD(0, w0);
            MX_PROF_ADD(1, clock64() - t0);
            MX_PROF_ADD(11, 1);
        }
    } else if (warp == 1) {
        // ================= MMA issuer: the whole warp loops, the elected lane issues =================
        // Every branch below is warp-uniform (waits and the abort flag are combined over the
        // warp), so elect_one() always sees 32 lanes and picks the same one.
        long long wa = 0, wf = 0, t0 = clock64();
        (void)wa;
        (void)wf;
        (void)t0;
        int g = pipe.g, it = pipe.it;
        bool ok = true;
        const uint32_t sf_smem = smem_u32(&c.sf[0][0][0]);
        const uint32_t tmem = c.tmem_base;  // a register copy: the asm memory clobbers would reload it
        const uint64_t a_desc0 = sdesc_k_swz<128>(a_addr(0)), b_desc0 = sdesc_k_swz<128>(b_addr(0));
        for (int tile = blockIdx.x; ok && !__any_sync(0xffffffffu, *abort_flag) && next_tile<G>(c, n, tile, e_hint, tc);
             tile += gridDim.x, ++it) {
            const int acc = it & 1, use = it >> 1;
            if (!__all_sync(0xffffffffu, MX_PROF_WAIT(wa, mbar_wait_bounded(smem_u32(&c.tempty[acc]), (use & 1) ^ 1,
                                                                           abort_flag, args.status, WAIT_LIMIT))))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)(acc * ACC_COLS);
            for (int kb = 0; kb < args.kblocks; ++kb, ++g) {
                const int s = g % STAGES, r = g / STAGES;
                if (!__all_sync(0xffffffffu, MX_PROF_WAIT(wf, mbar_wait_bounded(smem_u32(&c.full[s]), r & 1,
                                                                               abort_flag, args.status, WAIT_LIMIT)))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t sfa = tmem + (uint32_t)(SF_COL0 + s * SF_SLOT);
                    const uint32_t sfs = sf_smem + (uint32_t)(s * 3 * 32 * 16);
                    tmem_cp_32x128b_x4(sfa, sfs);
                    tmem_cp_32x128b_x4(sfa + 4, sfs + 32 * 16);
                    tmem_cp_32x128b_x4(sfa + 8, sfs + 2 * 32 * 16);
                    // descriptors are linear in the address (bits 0-13 hold address >> 4)
                    const uint64_t ad = a_desc0 + (uint64_t)((s * STAGE_BYTES) >> 4);
                    const uint64_t bd = b_desc0 + (uint64_t)((s * STAGE_BYTES) >> 4);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_mxf8(d_tmem, ad + 2 * j, bd + 2 * j, idesc_mxf8(BM, BN, j), sfa, sfa + 4, (kb | j) != 0);
                    tc_commit(smem_u32(&c.empty[s]));
                }
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one()) tc_commit(smem_u32(&c.tfull[acc]));
            __syncwarp();
        }
        if (lane == 0) {
            MX_PROF_ADD(2, wa);
            MX_PROF_ADD(3, wf);
            MX_PROF_ADD(5, clock64() - t0);
            MX_PROF_ADD(10, it);
        }
    } else if (warp >= 6) {
        // ================= scale-factor warps: warp 6 + j fills the stages g with g % 4 == j =================
        // (ring slot g % STAGES; with 4 stages warp 6 + j always fills slot j)
        const int j = warp - 6;
        const long long b_total = (long long)n * args.w_rows;
        // stage g (counted from this phase's first stage g0) = k-block g % kblocks of this
        // CTA's tile number g / kblocks; lane r = row r of each chunk
        const int g0 = pipe.g;
        auto load = [&](int gabs, uint32_t (&w)[10]) -> bool {
            const int g = gabs - g0;
            const int kb = g % args.kblocks;
            if (!next_tile<G>(c, n, blockIdx.x + (g / args.kblocks) * (int)gridDim.x, e_hint, tc)) return false;
            const long long a_row = (long long)c.row_off[tc.e] + tc.mt * AR + lane;
            const long long b_row = (long long)tc.e * args.w_rows + tc.nt * args.n_step + lane;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const long long row = a_row + 32 * i;
                // L2-coherent loads: the fused decode kernel writes these words earlier in the launch
                w[i] = (32 * i < AR && row < args.a_rows) ? __ldcg(args.a_s + row * args.kblocks + kb) : 0u;
            }
#pragma unroll
            for (int i = 0; i < 6; ++i) {
                long long row;
                const uint32_t* src;
                if (MODE == MODE_GATEUP) {  // columns 0-2: gate rows, 3-5: up rows of the same h columns
                    row = b_row + 32 * (i % 3);
                    src = i < 3 ? args.b0_s : args.b1_s;
                } else {
                    row = b_row + 32 * i;
                    src = args.b0_s;
                }
                // weight scales are read-only in every launch: cached loads, and the 32 (or 12)
                // k-blocks of a tile read the same lines
                w[4 + i] = row < b_total ? __ldg(src + row * args.kblocks + kb) : 0u;
            }
            return true;
        };
        long long wsf = 0, tsf = clock64();
        (void)wsf;
        (void)tsf;
        // two items in flight: the words of this warp's next stage and of the one after
        // it are loaded before the warp waits for that stage's slot to free up
        uint32_t w[10], wn[10];
        const int gj = g0 + (((j - g0) % SCALE_WARPS) + SCALE_WARPS) % SCALE_WARPS;  // this warp's first stage
        bool have = load(gj, w);
        bool have_n = have && load(gj + SCALE_WARPS, wn);
        for (int g = gj; have && !*abort_flag; g += SCALE_WARPS) {
            const int sl = g % STAGES, r = g / STAGES;
            // the copies of this slot's previous round have completed with its MMAs
            if (!MX_PROF_WAIT(wsf, mbar_wait_bounded(smem_u32(&c.empty[sl]), (r & 1) ^ 1, abort_flag, args.status,
                                                     WAIT_LIMIT)))
                break;
            c.sf[sl][0][lane] = make_uint4(w[0], w[1], w[2], w[3]);
            c.sf[sl][1][lane] = make_uint4(w[4], w[5], w[6], w[7]);
            c.sf[sl][2][lane] = make_uint4(w[8], w[9], 0u, 0u);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // read by tcgen05.cp (async proxy)
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&c.full[sl]));
#pragma unroll
            for (int i = 0; i < 10; ++i) w[i] = wn[i];
            have = have_n;
            if (have_n) have_n = load(g + 2 * SCALE_WARPS, wn);
        }
        if (lane == 0) {
            MX_PROF_ADD(8, wsf);
            MX_PROF_ADD(9, clock64() - tsf);
        }
    } else {
        // ================= epilogue (warps 2..5, TMEM lane quarter q = warp % 4) =================
        const int q = warp & 3;
        long long wt = 0, t0 = clock64();
        (void)wt;
        (void)t0;
        int it = pipe.it;
        for (int tile = blockIdx.x; !*abort_flag && next_tile<G>(c, n, tile, e_hint, tc); tile += gridDim.x, ++it) {
            const int acc = it & 1, use = it >> 1;
            if (!MX_PROF_WAIT(wt, mbar_wait_bounded(smem_u32(&c.tfull[acc]), use & 1, abort_flag, args.status,
                                                    WAIT_LIMIT)))
                break;
            tc_fence_after();
            const int row0_in_e = tc.mt * AR + q * 32;
            const long long grow0 = (long long)c.row_off[tc.e] + row0_in_e;
            const uint32_t taddr = c.tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
            const int col0 = tc.nt * args.n_step;
            if (q * 32 >= AR) {
                // accumulator rows past the m-tile (AR = 32): computed from stale A rows, not stored
            } else if (MODE == MODE_GATEUP) {
                // thread = one token row; 32 h columns per chunk = one MX block
                uint8_t* hq = static_cast<uint8_t*>(args.out);
                const bool row_ok = row0_in_e + lane < tc.cnt;
                const long long grow = grow0 + lane;
#pragma unroll 1
                for (int cc = 0; cc < BN / 2; cc += 32) {
                    uint32_t g0[16], g1[16], u0[16], u1[16];
                    tmem_ld16(taddr + cc, g0);
                    tmem_ld16(taddr + cc + 16, g1);
                    tmem_ld16(taddr + BN / 2 + cc, u0);
                    tmem_ld16(taddr + BN / 2 + cc + 16, u1);
                    tmem_ld_wait();
                    float h[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float a0 = __uint_as_float(g0[i]), b0 = __uint_as_float(u0[i]);
                        const float a1 = __uint_as_float(g1[i]), b1 = __uint_as_float(u1[i]);
                        h[i] = silu(a0) * b0;
                        h[16 + i] = silu(a1) * b1;
                    }
                    uint32_t w[8];
                    const uint32_t code = mx_quantize32(h, w);
                    if (row_ok && col0 + cc < args.out_cols) {
                        uint4* dst = reinterpret_cast<uint4*>(hq + grow * args.out_cols + col0 + cc);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                        args.out_s[grow * (args.out_cols / 32) + (col0 + cc) / 32] = (uint8_t)code;
                    }
                }
            } else {
                // 32 fp32 columns per chunk: 128 B per row, 8 slots; slot = piece ^ (row & 7)
                float* out = static_cast<float*>(args.out);
                uint4* st = c.stage[q];
#pragma unroll 1
                for (int cc = 0; cc < BN; cc += 32) {
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
        // the h codes are read later through TMA (async proxy)
        asm volatile("fence.proxy.async.global;" ::: "memory");
        if (lane == 0) {
            MX_PROF_ADD(6, wt);
            MX_PROF_ADD(7, clock64() - t0);
        }
    }
}

// Every thread: its counters after a phase that ran to completion.
template <class C>
__device__ __forceinline__ void pipe_advance(const C& c, Pipe& p, int n, int kblocks) {
    const int nt = tiles_of_cta(c, n);
    p.g += nt * kblocks;
    p.it += nt;
}

// After a __syncthreads: drain the MMAs (bounded), free TMEM.  Every load the
// producer issued was consumed by an MMA unless a wait gave up; then the loads
// still land within the bounded drain below.
template <class C>
__device__ __forceinline__ void teardown(C& c, int32_t* status) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 1) {
        // the lane that issued the MMAs (elect_one() of the converged warp) commits the drain
        if (elect_one()) tc_commit(smem_u32(&c.drain));
        __syncwarp();
        if (lane == 0) {
            volatile int never = 0;
            mbar_wait_bounded(smem_u32(&c.drain), 0, &never, status, WAIT_LIMIT);
            if (c.abort_flag) {  // copies may still be in flight: let them land
                const long long t0 = clock64();
                while (clock64() - t0 < (1ll << 20)) {
                }
            }
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(c.tmem_base, TMEM_COLS);
    }
}

}  // namespace mx
}  // namespace moe
