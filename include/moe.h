/*
 * moe.h -- C ABI of the GB300 (sm_103a) local mixture-of-experts layer of one
 * expert-parallel rank: route -> dispatch -> grouped SwiGLU expert FFN -> combine.
 *
 * The operations follow "Hosting Qwen on Blackwell" (Perplexity, 2026):
 *   - section "Expert Parallel": inputs are replicated on every rank; dispatch
 *     only selects the tokens routed to this rank's experts, gathers the routing
 *     information and stages the tokens in the buffers the MoE GEMM reads;
 *     combine first accumulates locally, with weights, the contributions of the
 *     tokens routed to this rank's experts (the cross-rank all-reduce that
 *     follows is not part of this library);
 *   - same section: for decode the whole layer is one fused kernel, for prefill
 *     it is split into several kernels;
 *   - section "MoE GEMM": the expert GEMM is a grouped GEMM over the experts;
 *   - section "Prefillers": T*k/E tokens reach each expert on average.
 * The router formula and the SwiGLU expert body are not on those pages; this
 * library computes softmax-over-logits top-k with renormalised weights and
 * FFN_e(x) = W_down[e] (silu(W_gate[e] x) * (W_up[e] x)).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers (cudaMalloc'd or PyTorch CUDA
 *     tensors), row-major, contiguous, 16-byte aligned.  bf16 tensors are passed
 *     as raw 16-bit patterns (uint16_t).
 *   - The caller allocates and owns every buffer, including the workspace; the
 *     library never allocates or frees device memory and never synchronises the
 *     stream.  `stream` is a cudaStream_t (NULL = legacy default stream); all
 *     work is enqueued asynchronously on it.
 *   - Argument errors detected on the host return a status and launch nothing.
 *     Launch failures return MOE_ERR_CUDA.  Data-dependent errors (non-finite
 *     logit, an internal wait that timed out) are written to the device word
 *     *status_dev when one is given (first error wins, 0 is never written: the
 *     caller clears it); outputs are then undefined but every write stays in
 *     bounds.  Nothing aborts, traps or throws across the ABI.
 *   - Weight pointers cover the LOCAL experts only: index 0 is expert e0.
 *   - The routed row count R lives on the device (offsets[n] = R); buffers
 *     sized for T*k rows always suffice.
 *   - Requires an sm_103 device (GB300); otherwise MOE_ERR_UNSUPPORTED.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* shape, range or null-pointer error            */
    MOE_ERR_UNSUPPORTED = 2, /* device is not sm_103, or a size limit is hit  */
    MOE_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small    */
    MOE_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed          */
    MOE_ERR_NONFINITE = 5,   /* (device status) a router logit is NaN or Inf  */
    MOE_ERR_TIMEOUT = 6      /* (device status) an internal wait ran out      */
} moe_status;

/*
 * Problem shape.  T tokens, hidden size H, expert intermediate size I, E experts
 * in total, top-k routing, local expert range [e0, e1) (n = e1 - e0 experts).
 * Limits: T >= 1, T*k < 2^31, 1 <= k <= min(E, 32), 1 <= E <= 1024,
 * 0 <= e0 < e1 <= E, H and I multiples of 64, 64 <= H, I <= 16384.
 */
typedef struct {
    int32_t T, H, I, E, k, e0, e1;
} moe_dims;

/* Human-readable name of a moe_status value (static storage). */
const char* moe_status_string(int status);

/* Workspace bytes needed by moe_dispatch / moe_expert_ffn / moe_layer for
 * these dims; 0 if the dims are invalid.  Workspace must be 256-byte aligned. */
size_t moe_dispatch_workspace_size(const moe_dims* d);
size_t moe_expert_ffn_workspace_size(const moe_dims* d);
size_t moe_workspace_size(const moe_dims* d);

/*
 * Routing ("Expert Parallel" section: the routing information dispatch gathers).
 * For each token t: the k largest logits[t, :] in descending order, ties broken
 * to the lower expert id (-0.0 ties +0.0); slot j holds the j-th pick.
 * topk_w[t, j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k picks, in fp32
 * (= the softmax over all E logits renormalised over the picks).
 *   logits    fp32  [T, E]  in
 *   topk_idx  int32 [T, k]  out, global expert ids in [0, E)
 *   topk_w    fp32  [T, k]  out
 *   status_dev int32[1] or NULL: set to MOE_ERR_NONFINITE if a logit is NaN/Inf
 */
int moe_route(const moe_dims* d, const float* logits, int32_t* topk_idx, float* topk_w,
              int32_t* status_dev, void* stream);

/*
 * Dispatch ("Expert Parallel" section: select the tokens routed to the local
 * experts and stage them in the grouped GEMM buffers).  A pair p = t*k + j is
 * local when e0 <= topk_idx[p] < e1.
 *   counts    int32 [n]        out, local pairs per local expert
 *   offsets   int32 [n+1]      out, exclusive prefix sum, offsets[n] = R
 *   row_pair  int32 [T*k]      out, rows [0, R): the pair each grouped row holds;
 *                              one expert's rows hold its pairs in ascending p
 *   pair_row  int32 [T*k]      out, row of pair p, or -1 if p is not local
 *   x_perm    bf16  [T*k, H]   out, rows [0, R): x_perm[r] = x[row_pair[r] / k]
 *   ws        >= moe_dispatch_workspace_size(d) bytes of scratch
 * Deterministic: identical inputs give identical outputs, bit for bit.
 */
int moe_dispatch(const moe_dims* d, const uint16_t* x, const int32_t* topk_idx,
                 int32_t* counts, int32_t* offsets, int32_t* row_pair, int32_t* pair_row,
                 uint16_t* x_perm, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_dispatch for callers that cannot allocate device memory -- for example a
 * plug-in inside a host runtime that owns every device buffer and hands it no
 * allocator, or a latency-critical serving loop where cudaMalloc is forbidden
 * because it can synchronise the whole device.  The paper has no counterpart:
 * it is an interface convenience of this library.
 *
 * Same arguments, outputs and determinism as moe_dispatch, minus the workspace:
 * its scratch (per-chunk expert histograms) is a fixed 1 MiB array compiled
 * into the library, which every GPU that loads the library keeps until the
 * process exits.  Limit: ceil(T*k / 2048) * (e1 - e0) <= 262144, e.g. T*k up to
 * 4,194,304 pairs with 128 local experts; larger problems return
 * MOE_ERR_UNSUPPORTED without launching.  It never calls cudaMalloc or cudaFree.
 * The first call on each device (with that device current) looks up the array's
 * device address with cudaGetSymbolAddress, which allocates nothing, and keeps it
 * for that device's context; the first call after a cudaDeviceReset looks it up
 * again.  That lookup may load the library's device code, so make the first call
 * on each device (and after a reset) before any stream capture.
 * All calls share the one array: calls whose work overlaps on the GPU (for
 * instance on two streams) race and give undefined results; calls ordered on one
 * stream are fine.  Its scan step reads n * ceil(T*k / 2048) histogram entries,
 * one warp per local expert; at the size limit that is 262144 entries.
 */
int moe_dispatch_noalloc(const moe_dims* d, const uint16_t* x, const int32_t* topk_idx,
                         int32_t* counts, int32_t* offsets, int32_t* row_pair, int32_t* pair_row,
                         uint16_t* x_perm, void* stream);

/*
 * Grouped SwiGLU expert FFN ("MoE GEMM" section), on the grouped rows made by
 * moe_dispatch: for each local expert e and row r in [offsets[e], offsets[e+1]):
 *   h[r]      = silu(x_perm[r] . W_gate[e]^T) * (x_perm[r] . W_up[e]^T)      (fp32)
 *   y_perm[r] = h[r] . W_down[e]^T                                          (fp32)
 * bf16 operands, fp32 accumulation on the tcgen05 tensor cores, SiLU*up in fp32.
 * h is the second GEMM's operand, which the bf16 tensor cores take as bf16: it is
 * carried as two bf16 terms, hi = bf16(h) and lo = bf16(h - hi) (hi + lo equals h
 * to about 2^-17), and the down GEMM runs over both (K = 2 I); y is kept in fp32.
 * The split layout of h is [T*k, 2 I]: each 64-column block j of h becomes
 * columns 128 j .. 128 j + 63 (hi) followed by 128 j + 64 .. 128 j + 127 (lo).
 *   x_perm   bf16 [T*k, H]; offsets int32 [n+1] (device, read by the kernels)
 *   w_gate, w_up  bf16 [n, I, H]; w_down bf16 [n, H, I]
 *   y_perm   fp32 [T*k, H] out (rows >= R are left untouched)
 *   ws       >= moe_expert_ffn_workspace_size(d) bytes (holds h, T*k * 2 I bf16)
 *   status_dev as in moe_route (MOE_ERR_TIMEOUT if an internal wait ran out)
 */
int moe_expert_ffn(const moe_dims* d, const uint16_t* x_perm, const int32_t* offsets,
                   const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                   float* y_perm, void* ws, size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * The two halves of moe_expert_ffn, for callers that keep h themselves (or
 * time the GEMMs apart).  Same row grouping, operands and rounding.
 *   moe_expert_gate_up: h[r] = silu(x_perm[r] . W_gate[e]^T) * (x_perm[r] . W_up[e]^T) as bf16
 *                       hi + lo terms, h bf16 [T*k, 2 I] out in the split layout
 *                       above (rows >= R untouched)
 *   moe_expert_down:    y_perm[r] = (hi[r] + lo[r]) . W_down[e]^T,  y_perm fp32 [T*k, H] out
 */
int moe_expert_gate_up(const moe_dims* d, const uint16_t* x_perm, const int32_t* offsets,
                       const uint16_t* w_gate, const uint16_t* w_up, uint16_t* h,
                       int32_t* status_dev, void* stream);
int moe_expert_down(const moe_dims* d, const uint16_t* h, const int32_t* offsets,
                    const uint16_t* w_down, float* y_perm, int32_t* status_dev, void* stream);

/*
 * Testing hook for failure detection without a GPU fault: moe_expert_gate_up
 * with the first stage of every CTA's shared-memory ring told to wait for one
 * arrival more than is ever made.  The MMA warp's bounded wait on that stage runs
 * out (~1 s of GPU clock cycles); the kernel writes MOE_ERR_TIMEOUT to
 * *status_dev, stops every role, waits (bounded) for its own copies in flight,
 * frees its tensor memory and returns, and the CUDA context stays usable.  h is
 * undefined afterwards.  Arguments as for moe_expert_gate_up.
 */
int moe_testing_expert_gate_up_stalled(const moe_dims* d, const uint16_t* x_perm, const int32_t* offsets,
                                       const uint16_t* w_gate, const uint16_t* w_up, uint16_t* h,
                                       int32_t* status_dev, void* stream);

/*
 * Combine ("Expert Parallel" and "MoE Dispatch - Combine" sections: weighted
 * local accumulation).  For each token t, in slot order j = 0..k-1 and in fp32:
 *   out[t] = sum_{j : pair_row[t*k+j] >= 0} topk_w[t, j] * y_perm[pair_row[t*k+j]]
 * Tokens with no local pair get exact zeros.  out is fp32 [T, H], overwritten: it
 * is this rank's partial sum, ready for a cross-rank all-reduce.
 */
int moe_combine(const moe_dims* d, const float* y_perm, const int32_t* pair_row,
                const float* topk_w, float* out, void* stream);

/*
 * Combine that adds into `out` instead of overwriting it: out[t] += the same
 * slot-ordered fp32 sum.  "Data Parallel and Expert Parallel" section: the DP-EP
 * kernel returns each expert's results to the tokens' source rank and
 * accumulates them there; with several expert ranges (or token shards) on one
 * GPU, each range's combine accumulates into one output buffer.  Arguments as
 * for moe_combine; out must hold the running sum (e.g. zeros) on entry.
 */
int moe_combine_accumulate(const moe_dims* d, const float* y_perm, const int32_t* pair_row,
                           const float* topk_w, float* out, void* stream);

/* T*k at or below which moe_layer runs the fused single-launch (decode) path. */
#define MOE_FUSED_MAX_PAIRS 8192

/*
 * The whole local layer, all intermediates in `ws` (>= moe_workspace_size(d)
 * bytes).  "Expert Parallel" section: for decode the whole kernel is fused into
 * one, prefill is split into several kernels.  Accordingly:
 *   - T*k <= MOE_FUSED_MAX_PAIRS: one persistent cooperative launch (one CTA per
 *     SM) that routes, dispatches, runs both grouped GEMMs and combines, with
 *     grid-wide barriers between the phases (plus a 8-byte memset of its barrier
 *     words on the stream);
 *   - otherwise moe_route, moe_dispatch, moe_expert_ffn and moe_combine back to back.
 * Both give bit-identical results for the same inputs.  topk_idx_opt /
 * topk_w_opt, when not NULL, receive the routing ([T, k] each); when NULL the
 * workspace holds it.  status_dev: MOE_ERR_NONFINITE, or MOE_ERR_TIMEOUT if an
 * internal wait (a grid barrier of the fused path) ran out.
 */
int moe_layer(const moe_dims* d, const uint16_t* x, const float* logits,
              const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
              float* out, int32_t* topk_idx_opt, float* topk_w_opt,
              void* ws, size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * moe_layer's fused path with dispatch by TMA row gather ("Expert Parallel"
 * section: dispatch stages the tokens routed to the local experts for the grouped
 * GEMM).  Dispatch writes no grouped copy of x: the gate/up GEMM loads the token
 * rows of each m-tile straight from x [T, H] into its operand tiles with
 * tile::gather4 copies (four rows each), indexed by row_pair (token = pair / k).
 * Same arguments, outputs and workspace as moe_layer, and bit-identical results;
 * the x_perm part of the workspace is left unwritten.  Requires
 * T*k <= MOE_FUSED_MAX_PAIRS (else MOE_ERR_UNSUPPORTED, nothing launched).
 */
int moe_layer_gather(const moe_dims* d, const uint16_t* x, const float* logits,
                     const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                     float* out, int32_t* topk_idx_opt, float* topk_w_opt,
                     void* ws, size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * Testing hook for failure detection without a GPU fault: the fused path of
 * moe_layer with its first grid-wide barrier told to wait for one CTA more than
 * the grid holds, so that wait runs out (~1 s of GPU clock cycles).  The kernel
 * then writes MOE_ERR_TIMEOUT to *status_dev, skips the remaining phases, frees
 * its tensor memory and returns; the CUDA context stays usable.  Outputs are
 * undefined.  Requires T*k <= MOE_FUSED_MAX_PAIRS (else MOE_ERR_INVALID_ARG).
 */
int moe_testing_layer_stalled_barrier(const moe_dims* d, const uint16_t* x, const float* logits,
                                      const uint16_t* w_gate, const uint16_t* w_up,
                                      const uint16_t* w_down, float* out, void* ws, size_t ws_bytes,
                                      int32_t* status_dev, void* stream);

/*
 * MXFP8 expert FFN ("MoE GEMM" section: the deployed expert GEMMs run in MXFP8).
 * The pages name the format only; it is read as OCP Microscaling (MX) v1.0 MXFP8:
 *   - an MXFP8 matrix [rows, K] is q uint8 [rows, K] (E4M3 codes: sign, 4 exponent
 *     bits with bias 7, 3 mantissa bits, no infinities, 0x7f/0xff NaN) and
 *     s uint8 [rows, K/32] (UE8M0 codes: the scale of elements 32b..32b+31 of a row
 *     is 2^(s[row, b] - 127));
 *   - quantisation of a block: X = 2^(floor(log2(amax)) - 8) (code 0 for a zero
 *     block, clamped to [0, 254]), each element = v / X rounded to the nearest E4M3
 *     value, ties to even, saturating at +-448.
 * The MX GEMMs accumulate in fp32 on the block-scaled tcgen05 tensor cores
 * (kind::mxf8f6f4); h = silu(g) * u is computed in fp32 and quantised to MXFP8
 * along I before the down GEMM; y_perm and the layer output are fp32.
 * Limits on top of moe_dims': H and I multiples of 128 (else MOE_ERR_UNSUPPORTED).
 * All q and s pointers must be 16-byte aligned.
 */

/* q, s = MXFP8 of the bf16 matrix src [rows, K] (K a multiple of 32).  Bit-exact
 * with the definition above. */
int moe_quantize_mxfp8(const uint16_t* src, int64_t rows, int32_t K, uint8_t* q, uint8_t* s, void* stream);

/*
 * moe_expert_ffn with MXFP8 operands: x_perm (q [T*k, H], s [T*k, H/32]) grouped
 * by `offsets` as moe_dispatch makes them; w_gate, w_up (q [n, I, H], s [n, I, H/32])
 * and w_down (q [n, H, I], s [n, H, I/32]), e.g. from moe_quantize_mxfp8.
 *   y_perm fp32 [T*k, H] out (rows >= R untouched)
 *   ws >= moe_expert_ffn_mxfp8_workspace_size(d) bytes, 256-byte aligned; it holds
 *   the quantised h: codes [T*k, I] at offset 0, then scales [T*k, I/32] at the
 *   next multiple of 256 bytes
 */
size_t moe_expert_ffn_mxfp8_workspace_size(const moe_dims* d);
int moe_expert_ffn_mxfp8(const moe_dims* d, const uint8_t* x_perm_q, const uint8_t* x_perm_s, const int32_t* offsets,
                         const uint8_t* w_gate_q, const uint8_t* w_gate_s, const uint8_t* w_up_q,
                         const uint8_t* w_up_s, const uint8_t* w_down_q, const uint8_t* w_down_s, float* y_perm,
                         void* ws, size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * Testing hook, as moe_testing_expert_gate_up_stalled for the MXFP8 FFN: its
 * gate/up GEMM's first ring stage waits for an arrival that never comes, so the
 * MMA warp's bounded wait runs out and *status_dev gets MOE_ERR_TIMEOUT; the down
 * GEMM then runs on an undefined h.  Arguments as for moe_expert_ffn_mxfp8.
 */
int moe_testing_expert_ffn_mxfp8_stalled(const moe_dims* d, const uint8_t* x_perm_q, const uint8_t* x_perm_s,
                                         const int32_t* offsets, const uint8_t* w_gate_q, const uint8_t* w_gate_s,
                                         const uint8_t* w_up_q, const uint8_t* w_up_s, const uint8_t* w_down_q,
                                         const uint8_t* w_down_s, float* y_perm, void* ws, size_t ws_bytes,
                                         int32_t* status_dev, void* stream);

/*
 * The whole local layer with MXFP8 expert weights: route, dispatch (x quantised to
 * MXFP8 once per token, rows copied in that format), the MXFP8 expert FFN and the
 * weighted fp32 combine into out fp32 [T, H].  As for moe_layer ("Expert Parallel"
 * section): T*k <= MOE_FUSED_MAX_PAIRS runs one persistent cooperative launch with
 * bounded grid-wide barriers between the phases (plus an 8-byte memset of its
 * barrier words), larger problems the split kernels; both give bit-identical
 * results.  Routing, counts, offsets and the permutation are those of moe_layer.
 * ws >= moe_layer_mxfp8_workspace_size(d) bytes, 256-byte aligned.
 */
size_t moe_layer_mxfp8_workspace_size(const moe_dims* d);
int moe_layer_mxfp8(const moe_dims* d, const uint16_t* x, const float* logits, const uint8_t* w_gate_q,
                    const uint8_t* w_gate_s, const uint8_t* w_up_q, const uint8_t* w_up_s, const uint8_t* w_down_q,
                    const uint8_t* w_down_s, float* out, int32_t* topk_idx_opt, float* topk_w_opt, void* ws,
                    size_t ws_bytes, int32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
