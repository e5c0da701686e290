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
// `accumulate` the sum starts from the current out[t] instead of zero.  RB > 1
// issues the loads of RB rows before their fma steps (for launches with only a
// token or two per CTA, where the rows' L2 round trips would otherwise run one
// after another); the fma order per element, and so the result, is the same.
template <int RB = 1>
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
    // four output vectors per thread per pass: four independent 16-byte loads of
    // every row in flight (the per-element fma chain is in slot order either way)
    constexpr int U = 4;
    const int bd = blockDim.x;
    for (int v0 = threadIdx.x; v0 < H4; v0 += U * bd) {
        float4 a[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (accumulate && v0 + u * bd < H4) a[u] = o[v0 + u * bd];
        }
        for (int q0 = 0; q0 < nr; q0 += RB) {
            float4 y[RB][U];
#pragma unroll
            for (int qq = 0; qq < RB; ++qq) {
                const bool live = q0 + qq < nr;
                const float4* row = y_perm + (size_t)sm.rows[live ? q0 + qq : 0] * H4;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + u * bd;
                    y[qq][u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (live && v < H4) y[qq][u] = cg ? __ldcg(row + v) : __ldg(row + v);
                }
            }
#pragma unroll
            for (int qq = 0; qq < RB; ++qq) {
                if (q0 + qq >= nr) break;
                const float w = sm.wts[q0 + qq];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    a[u].x = fmaf(w, y[qq][u].x, a[u].x);
                    a[u].y = fmaf(w, y[qq][u].y, a[u].y);
                    a[u].z = fmaf(w, y[qq][u].z, a[u].z);
                    a[u].w = fmaf(w, y[qq][u].w, a[u].w);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v0 + u * bd < H4) o[v0 + u * bd] = a[u];
    }
    __syncthreads();  // sm is reused by the next token
}

}  // namespace moe
