// combine.cuh -- weighted local accumulation of one token (device function),
// used by the combine kernel and by the fused decode kernel.
//
// "Hosting Qwen on Blackwell", sections "MoE Dispatch - Combine" and "Expert
// Parallel": combine accumulates, with the routing weights, the contributions of
// the tokens routed to this rank's experts (before a cross-rank all-reduce).
//   out[t] = sum_{j=0..k-1, pair_row[t*k+j] >= 0} topk_w[t,j] * y_perm[pair_row[t*k+j]]
// in fp32 registers, slot order fixed (deterministic); tokens without a local
// slot get zeros.  16-byte loads and stores of 4 fp32.
#pragma once

#include "common.cuh"

namespace moe {

struct CombineSmem {
    int rows[32];
    float wts[32];
    int nrows;
};

// The whole CTA (nthreads threads) combines token t.  `cg` selects L2-coherent
// loads for indices written earlier in the same launch by other CTAs.  With
// `accumulate` the sum starts from the current out[t] instead of zero.
__device__ __forceinline__ void combine_token(const float4* __restrict__ y_perm, const int32_t* pair_row,
                                              const float* topk_w, int t, int H4, int k, float4* __restrict__ out,
                                              CombineSmem& sm, bool cg, bool accumulate = false) {
    if (threadIdx.x < 32) {
        const int j = threadIdx.x;
        int r = -1;
        float w = 0.f;
        if (j < k) {
            r = cg ? __ldcg(pair_row + (size_t)t * k + j) : __ldg(pair_row + (size_t)t * k + j);
            w = cg ? __ldcg(topk_w + (size_t)t * k + j) : __ldg(topk_w + (size_t)t * k + j);
        }
        const unsigned m = __ballot_sync(0xffffffffu, r >= 0);
        if (r >= 0) {
            const int q = __popc(m & ((1u << j) - 1u));  // keeps slot order
            sm.rows[q] = r;
            sm.wts[q] = w;
        }
        if (j == 0) sm.nrows = __popc(m);
    }
    __syncthreads();
    const int nr = sm.nrows;
    float4* o = out + (size_t)t * H4;
    // two output vectors per thread per pass: twice the independent loads in flight
    for (int v0 = threadIdx.x; v0 < H4; v0 += 2 * blockDim.x) {
        const int v1 = v0 + blockDim.x;
        const bool has1 = v1 < H4;
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
        if (accumulate) {
            a0 = o[v0];
            if (has1) a1 = o[v1];
        }
        for (int q = 0; q < nr; ++q) {
            const float4* row = y_perm + (size_t)sm.rows[q] * H4;
            const float4 y0 = cg ? __ldcg(row + v0) : __ldg(row + v0);
            float4 y1 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (has1) y1 = cg ? __ldcg(row + v1) : __ldg(row + v1);
            const float w = sm.wts[q];
            a0.x = fmaf(w, y0.x, a0.x);
            a0.y = fmaf(w, y0.y, a0.y);
            a0.z = fmaf(w, y0.z, a0.z);
            a0.w = fmaf(w, y0.w, a0.w);
            a1.x = fmaf(w, y1.x, a1.x);
            a1.y = fmaf(w, y1.y, a1.y);
            a1.z = fmaf(w, y1.z, a1.z);
            a1.w = fmaf(w, y1.w, a1.w);
        }
        o[v0] = a0;
        if (has1) o[v1] = a1;
    }
    __syncthreads();  // sm is reused by the next token
}

}  // namespace moe
