// route.cu -- K1: top-k router, one warp per token (the per-token work is in
// route.cuh, shared with the fused decode kernel).
#include "kernels.h"
#include "route.cuh"

namespace moe {

namespace {

// hist (optional): per-chunk histogram of the local experts [e0, e0 + n) over
// chunks of chunk_t tokens, accumulated with atomics (order-free, so the counts
// are deterministic); it must be zero on entry.  The dispatch place kernel
// consumes it, which saves a separate counting pass.
template <int NPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                                         int32_t* status, int32_t* hist, int chunk_t, int e0, int n) {
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int id = route_token<NPL>(logits, t, E, k, topk_idx, topk_w, status);
    if (hist) {
        const int e = id - e0;
        if (id >= 0 && e >= 0 && e < n) atomicAdd(hist + (size_t)(t / chunk_t) * n + e, 1);
    }
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* topk_idx, float* topk_w, int32_t* status,
                         cudaStream_t s) {
    return launch_route_hist(logits, T, E, k, topk_idx, topk_w, status, nullptr, 1, 0, 1, s);
}

cudaError_t launch_route_hist(const float* logits, int T, int E, int k, int32_t* topk_idx, float* topk_w,
                              int32_t* status, int32_t* hist, int chunk_t, int e0, int n, cudaStream_t s) {
    const int warps = 8;
    dim3 grid((T + warps - 1) / warps), block(32 * warps);
    if (E <= 32)
        route_topk_kernel<1><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status, hist, chunk_t, e0, n);
    else if (E <= 64)
        route_topk_kernel<2><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status, hist, chunk_t, e0, n);
    else if (E <= 128)
        route_topk_kernel<4><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status, hist, chunk_t, e0, n);
    else if (E <= 256)
        route_topk_kernel<8><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status, hist, chunk_t, e0, n);
    else if (E <= 512)
        route_topk_kernel<16><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status, hist, chunk_t, e0, n);
    else
        route_topk_kernel<32><<<grid, block, 0, s>>>(logits, T, E, k, topk_idx, topk_w, status, hist, chunk_t, e0, n);
    return cudaGetLastError();
}

}  // namespace moe
