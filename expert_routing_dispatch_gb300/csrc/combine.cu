// combine.cu -- K5: weighted local accumulation of the expert outputs.
//
// "Hosting Qwen on Blackwell", sections "MoE Dispatch - Combine" and "Expert
// Parallel": combine accumulates, with the routing weights, the contributions of
// the tokens routed to this rank's experts (before a cross-rank all-reduce).
//   out[t] = sum_{j=0..k-1, pair_row[t*k+j] >= 0} topk_w[t,j] * y_perm[pair_row[t*k+j]]
// in fp32 registers, slot order fixed (deterministic); tokens without a local
// slot get zeros.  One CTA per token, 16-byte loads and stores of 4 fp32.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

__global__ void __launch_bounds__(128) combine_kernel(const float4* __restrict__ y_perm,
                                                      const int32_t* __restrict__ pair_row,
                                                      const float* __restrict__ topk_w, int H4, int k,
                                                      float4* __restrict__ out) {
    __shared__ int rows[32];
    __shared__ float wts[32];
    __shared__ int nrows;
    const int t = blockIdx.x;
    if (threadIdx.x < 32) {
        int j = threadIdx.x;
        int r = (j < k) ? __ldg(pair_row + (size_t)t * k + j) : -1;
        float w = (j < k) ? __ldg(topk_w + (size_t)t * k + j) : 0.f;
        unsigned m = __ballot_sync(0xffffffffu, r >= 0);
        if (r >= 0) {
            int q = __popc(m & ((1u << j) - 1u));  // keeps slot order
            rows[q] = r;
            wts[q] = w;
        }
        if (j == 0) nrows = __popc(m);
    }
    __syncthreads();
    const int nr = nrows;
    float4* o = out + (size_t)t * H4;
    for (int v = threadIdx.x; v < H4; v += blockDim.x) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = 0; q < nr; ++q) {
            const float4 y = __ldg(y_perm + (size_t)rows[q] * H4 + v);
            const float w = wts[q];
            a.x = fmaf(w, y.x, a.x);
            a.y = fmaf(w, y.y, a.y);
            a.z = fmaf(w, y.z, a.z);
            a.w = fmaf(w, y.w, a.w);
        }
        o[v] = a;
    }
}

}  // namespace

cudaError_t launch_combine(const float* y_perm, const int32_t* pair_row, const float* topk_w, int T, int H, int k,
                           float* out, cudaStream_t s) {
    combine_kernel<<<T, 128, 0, s>>>(reinterpret_cast<const float4*>(y_perm), pair_row, topk_w, H / 4, k,
                                     reinterpret_cast<float4*>(out));
    return cudaGetLastError();
}

}  // namespace moe
