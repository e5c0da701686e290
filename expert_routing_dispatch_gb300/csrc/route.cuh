// route.cuh -- per-token top-k routing (device function), used by the router
// kernel and by the fused decode kernel.
//
// "Hosting Qwen on Blackwell", section "Expert Parallel": routing is the light
// part of the EP kernel.  Per token: the k largest fp32 logits in descending
// order, ties to the lower expert id; weights = softmax over the k picks (equal
// to the full softmax renormalised over them).
//
// Selection is exact: each logit maps to 32 bits whose unsigned order is the
// float order (-0.0 folded onto +0.0).  Each of the k passes takes the warp
// maximum of those bits (redux.sync), then the lowest expert id holding it (a
// second redux.sync), so ties go to the lower id.  Lane l holds the logits of
// experts l, l+32, l+64, ... in registers (coalesced loads).
#pragma once

#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint32_t route_ordered_bits(float v) {
    uint32_t u = __float_as_uint(v);
    if ((u << 1) == 0) u = 0;  // -0.0 ties +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The whole warp routes token t.  NPL = logits per lane, E <= 32 * NPL.
// Returns, in lane j < k, the expert of slot j (-1 in the other lanes).
template <int NPL>
__device__ __forceinline__ int route_token(const float* __restrict__ logits, int t, int E, int k,
                                            int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                            int32_t* status) {
    const int lane = threadIdx.x & 31;
    const float* row = logits + (size_t)t * E;
    uint32_t key[NPL];  // ordered bits, 0 = removed or absent
    bool finite = true;
#pragma unroll
    for (int c = 0; c < NPL; ++c) {
        const int e = c * 32 + lane;
        key[c] = 0;
        if (e < E) {
            const float v = __ldg(row + e);
            finite &= isfinite(v);
            key[c] = max(route_ordered_bits(v), 1u);  // 0 only for a NaN pattern, which is flagged below
        }
    }
    if (__any_sync(0xffffffffu, !finite) && lane == 0) set_status(status, MOE_ERR_NONFINITE);

    // k passes: warp max of the bits, then the lowest id holding it; lane j keeps pick j
    int id = -1, top = 0;
    for (int j = 0; j < k; ++j) {
        uint32_t lb = 0;
#pragma unroll
        for (int c = 0; c < NPL; ++c) lb = max(lb, key[c]);
        const uint32_t best = __reduce_max_sync(0xffffffffu, lb);
        uint32_t mine = 0xffffffffu;
#pragma unroll
        for (int c = NPL - 1; c >= 0; --c)
            if (key[c] == best) mine = (uint32_t)(c * 32 + lane);  // ends at the lane's lowest id
        const int pick = (int)__reduce_min_sync(0xffffffffu, mine);
#pragma unroll
        for (int c = 0; c < NPL; ++c)
            if (c * 32 + lane == pick) key[c] = 0;
        if (lane == j) id = pick;
        if (j == 0) top = pick;
    }
    const float v = (lane < k) ? __ldg(row + id) : 0.f;
    const float m = __ldg(row + top);
    const float ex = (lane < k) ? expf(v - m) : 0.f;
    // sum over the k picks in slot order, the same sequential order in every lane
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
        topk_idx[(size_t)t * k + lane] = id;
        topk_w[(size_t)t * k + lane] = ex / sum;
    }
    return lane < k ? id : -1;
}

// Runtime choice of the register layout for E experts (E <= 1024).
__device__ __forceinline__ void route_token_any(const float* logits, int t, int E, int k, int32_t* topk_idx,
                                                float* topk_w, int32_t* status) {
    if (E <= 32)
        route_token<1>(logits, t, E, k, topk_idx, topk_w, status);
    else if (E <= 64)
        route_token<2>(logits, t, E, k, topk_idx, topk_w, status);
    else if (E <= 128)
        route_token<4>(logits, t, E, k, topk_idx, topk_w, status);
    else if (E <= 256)
        route_token<8>(logits, t, E, k, topk_idx, topk_w, status);
    else if (E <= 512)
        route_token<16>(logits, t, E, k, topk_idx, topk_w, status);
    else
        route_token<32>(logits, t, E, k, topk_idx, topk_w, status);
}

}  // namespace moe
