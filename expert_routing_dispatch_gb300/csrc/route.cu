// route.cu -- K1: top-k router, one warp per token.
//
// "Hosting Qwen on Blackwell", section "Expert Parallel": routing is the light
// part of the prefill EP kernel (it needs fewer blocks than the local combine).
// Per token: the k largest fp32 logits in descending order, ties to the lower
// expert id; weights = softmax over the picks (= full softmax renormalised).
//
// Selection is exact: each (logit, id) is mapped to a 64-bit key whose unsigned
// order is "larger logit first, then lower id" (-0.0 folded onto +0.0), so each
// of the k passes is a plain warp max over keys.  Lane l holds the logits of
// experts l, l+32, l+64, ... in registers (coalesced loads).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

__device__ __forceinline__ uint32_t ordered_bits(float v) {
    uint32_t u = __float_as_uint(v);
    if ((u << 1) == 0) u = 0;  // -0.0 ties +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

template <int NPL>  // logits per lane; E <= 32 * NPL
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                                         int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float* row = logits + (size_t)t * E;

    uint64_t key[NPL];
    bool finite = true;
#pragma unroll
    for (int c = 0; c < NPL; ++c) {
        int e = c * 32 + lane;
        if (e < E) {
            float v = __ldg(row + e);
            finite &= isfinite(v);
            key[c] = ((uint64_t)ordered_bits(v) << 32) | (uint32_t)(0xffffffffu - (uint32_t)e);
        } else {
            key[c] = 0;  // below every real key
        }
    }
    if (__any_sync(0xffffffffu, !finite) && lane == 0) set_status(status, MOE_ERR_NONFINITE);

    // k passes of warp argmax; lane j keeps the j-th pick
    uint64_t mine = 0;
    for (int j = 0; j < k; ++j) {
        uint64_t best = 0;
#pragma unroll
        for (int c = 0; c < NPL; ++c) best = key[c] > best ? key[c] : best;
        best = warp_max_u64(best);
#pragma unroll
        for (int c = 0; c < NPL; ++c)
            if (key[c] == best) key[c] = 0;  // remove the pick (keys are unique)
        if (lane == j) mine = best;
    }
    // top logit (slot 0) from lane 0
    uint64_t top = __shfl_sync(0xffffffffu, mine, 0);
    int id = (int)(0xffffffffu - (uint32_t)(mine & 0xffffffffu));
    float v = (lane < k) ? __ldg(row + id) : 0.f;
    float m = __ldg(row + (int)(0xffffffffu - (uint32_t)(top & 0xffffffffu)));
    float ex = (lane < k) ? expf(v - m) : 0.f;
    // sum over the k picks in slot order (lane 0 adds sequentially: deterministic)
    float sum = 0.f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
        topk_idx[(size_t)t * k + lane] = id;
        topk_w[(size_t)t * k + lane] = ex / sum;
    }
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* topk_idx, float* topk_w, int32_t* status,
                         cudaStream_t s) {
    const int warps = 8;
    dim3 grid((T + warps - 1) / warps), block(32 * warps);
    if (E <= 32)
        route_topk_kernel<1><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status);
    else if (E <= 64)
        route_topk_kernel<2><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status);
    else if (E <= 128)
        route_topk_kernel<4><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status);
    else if (E <= 256)
        route_topk_kernel<8><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status);
    else if (E <= 512)
        route_topk_kernel<16><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status);
    else
        route_topk_kernel<32><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status);
    return cudaGetLastError();
}

}  // namespace moe
