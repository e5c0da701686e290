// combine.cu -- K5: weighted local accumulation of the expert outputs, one
// 256-thread CTA per token (the per-token work is in combine.cuh, shared with the fused
// decode kernel).
#include "combine.cuh"
#include "kernels.h"

namespace moe {

namespace {

template <bool ACC>
__global__ void __launch_bounds__(256) combine_kernel(const float4* __restrict__ y_perm,
                                                      const int32_t* __restrict__ pair_row,
                                                      const float* __restrict__ topk_w, int H4, int k,
                                                      float4* __restrict__ out) {
    __shared__ CombineSmem sm;
    combine_token(y_perm, pair_row, topk_w, blockIdx.x, H4, k, out, sm, false, ACC);
}

}  // namespace

cudaError_t launch_combine(const float* y_perm, const int32_t* pair_row, const float* topk_w, int T, int H, int k,
                           float* out, cudaStream_t s, bool accumulate) {
    if (accumulate)
        combine_kernel<true><<<T, 256, 0, s>>>(reinterpret_cast<const float4*>(y_perm), pair_row, topk_w, H / 4, k,
                                               reinterpret_cast<float4*>(out));
    else
        combine_kernel<false><<<T, 256, 0, s>>>(reinterpret_cast<const float4*>(y_perm), pair_row, topk_w, H / 4, k,
                                                reinterpret_cast<float4*>(out));
    return cudaGetLastError();
}

}  // namespace moe
