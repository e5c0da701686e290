/*
 * oracle.c -- plain, slow, obviously-correct CPU reference of one expert-parallel
 * rank's local MoE layer: route -> dispatch -> SwiGLU expert FFN -> weighted combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA path.
 *
 * Source: "Hosting Qwen on Blackwell" (Perplexity, 2026), section "Expert Parallel":
 * the inputs are replicated on every rank, dispatch keeps only the tokens routed
 * to the rank's experts, gathers the routing information and stages those tokens
 * in the buffers the MoE GEMM reads; combine first accumulates, with weights, the
 * contributions of those tokens locally (the cross-rank all-reduce that follows
 * is out of scope).  Section "MoE Dispatch - Combine": combine is a weighted
 * accumulation.  Section "Prefillers": T*k/E tokens reach each expert on average.
 * The router formula (softmax over the expert logits, top-k, renormalised
 * weights) and the SwiGLU expert body are the workload's own statement; the
 * pages give neither.
 *
 * Readings where the pages are silent (each listed again in the design notes):
 *   - selection is on the fp32 logits, strict order (a > b) or (a == b and
 *     id_a < id_b): ties go to the lower expert id, and -0.0 ties +0.0;
 *   - slot j of a token is its j-th pick, i.e. descending logit;
 *   - weights: exp(l_j - m) / sum_i exp(l_i - m) over the k picks, m = the top
 *     logit.  This equals the full softmax renormalised over the k picks;
 *   - a non-finite logit is an error (status 5), no output is defined;
 *   - within one expert's rows, pairs p = t*k + j are in ascending p order
 *     (ascending token, since a token picks an expert at most once);
 *   - out[t] = sum over the token's slots j in order 0..k-1 whose expert is in
 *     [e0, e1) of w_tj * FFN_e(x_t); a token with no local slot gets 0;
 *   - FFN_e(x) = W_down[e] (silu(W_gate[e] x) * (W_up[e] x)), silu(z) = z/(1+e^-z);
 *   - arithmetic in fp64 (bf16 inputs widened exactly), no bf16 rounding of
 *     intermediates.
 *
 * Layouts (row-major): logits fp32 [T,E]; x bf16 bits [T,H]; w_gate, w_up bf16
 * [n,I,H]; w_down bf16 [n,H,I], local experts only (index 0 = expert e0).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NONFINITE 5

/* exact widening of a bf16 bit pattern */
static double bf16_widen(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Route one token: k passes of "largest remaining logit, lowest id on ties". */
static int route_one(int E, int k, const float* l, int32_t* idx, double* w) {
    for (int e = 0; e < E; ++e)
        if (!isfinite(l[e])) return ORACLE_ERR_NONFINITE;
    char picked[4096];
    memset(picked, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (picked[e]) continue;
            if (best < 0 || l[e] > l[best]) best = e; /* strict >: first (lowest) id wins ties */
        }
        picked[best] = 1;
        idx[j] = best;
    }
    double m = (double)l[idx[0]];
    double s = 0.0;
    for (int j = 0; j < k; ++j) s += exp((double)l[idx[j]] - m);
    for (int j = 0; j < k; ++j) w[j] = exp((double)l[idx[j]] - m) / s;
    return ORACLE_OK;
}

/* Routing for all tokens: topk_idx int32 [T,k], topk_w fp64 [T,k]. */
int oracle_route(int64_t T, int E, int k, const float* logits, int32_t* topk_idx, double* topk_w) {
    if (T < 0 || E < 1 || E > 4096 || k < 1 || k > E) return ORACLE_ERR_ARG;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(static) reduction(max : status)
    for (int64_t t = 0; t < T; ++t) {
        int s = route_one(E, k, logits + t * E, topk_idx + t * k, topk_w + t * k);
        if (s > status) status = s;
    }
    return status;
}

/*
 * Dispatch = stable counting sort of the in-range pairs by local expert.
 *   counts[e-e0]  = number of pairs (t, j) with topk_idx[t,j] == e
 *   offsets       = exclusive prefix sum of counts, offsets[n] = R
 *   row_pair[r]   = pair p = t*k + j placed at row r; rows of one expert hold
 *                   its pairs in ascending p
 *   pair_row[p]   = row of pair p, or -1 when its expert is outside [e0, e1)
 * Returns R (>= 0) or -1 on bad arguments.
 */
int64_t oracle_dispatch(int64_t T, int k, int e0, int e1, const int32_t* topk_idx,
                        int32_t* counts, int32_t* offsets, int32_t* row_pair, int32_t* pair_row) {
    if (T < 0 || k < 1 || e0 < 0 || e1 <= e0) return -1;
    int n = e1 - e0;
    int64_t P = T * k;
    for (int e = 0; e < n; ++e) counts[e] = 0;
    for (int64_t p = 0; p < P; ++p) {
        int e = topk_idx[p];
        if (e >= e0 && e < e1) counts[e - e0] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < n; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* fill = (int32_t*)calloc((size_t)n, sizeof(int32_t));
    for (int64_t p = 0; p < P; ++p) {
        int e = topk_idx[p];
        if (e >= e0 && e < e1) {
            int32_t r = offsets[e - e0] + fill[e - e0]++;
            row_pair[r] = (int32_t)p;
            pair_row[p] = r;
        } else {
            pair_row[p] = -1;
        }
    }
    free(fill);
    return offsets[n];
}

/* y[H] = W_down (silu(W_gate x) * (W_up x)) for one expert; x already widened. */
static void swiglu_ffn(int H, int I, const double* x, const uint16_t* wg, const uint16_t* wu,
                       const uint16_t* wd, double* act /*[I]*/, double* y /*[H]*/) {
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        const uint16_t* rg = wg + (int64_t)i * H;
        const uint16_t* ru = wu + (int64_t)i * H;
        for (int h = 0; h < H; ++h) g += bf16_widen(rg[h]) * x[h];
        for (int h = 0; h < H; ++h) u += bf16_widen(ru[h]) * x[h];
        double silu = g / (1.0 + exp(-g));
        act[i] = silu * u;
    }
    for (int h = 0; h < H; ++h) {
        double acc = 0.0;
        const uint16_t* rd = wd + (int64_t)h * I;
        for (int i = 0; i < I; ++i) acc += bf16_widen(rd[i]) * act[i];
        y[h] = acc;
    }
}

/*
 * Expert FFN on grouped rows (the dispatch layout): for each row r in
 * [row_lo, row_hi) find its local expert e (offsets[e] <= r < offsets[e+1]) and
 * write y[r-row_lo, :] = FFN_e(x_perm[r]).  Rows at or past offsets[n] get 0.
 */
void oracle_expert_ffn_rows(int H, int I, int n, const uint16_t* x_perm, const int32_t* offsets,
                            const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                            int64_t row_lo, int64_t row_hi, double* y) {
#pragma omp parallel
    {
        double* xd = (double*)malloc(sizeof(double) * (size_t)H);
        double* act = (double*)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = row_lo; r < row_hi; ++r) {
            double* yr = y + (r - row_lo) * H;
            int e = -1;
            for (int q = 0; q < n; ++q)
                if (r >= offsets[q] && r < offsets[q + 1]) { e = q; break; }
            if (e < 0) {
                for (int h = 0; h < H; ++h) yr[h] = 0.0;
                continue;
            }
            for (int h = 0; h < H; ++h) xd[h] = bf16_widen(x_perm[r * H + h]);
            swiglu_ffn(H, I, xd, w_gate + (int64_t)e * I * H, w_up + (int64_t)e * I * H,
                       w_down + (int64_t)e * H * I, act, yr);
        }
        free(xd);
        free(act);
    }
}

/* Same as oracle_expert_ffn_rows for an explicit list of grouped rows. */
void oracle_expert_ffn_rowlist(int H, int I, int n, const uint16_t* x_perm, const int32_t* offsets,
                               const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                               const int64_t* rows, int64_t nrows, double* y) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < nrows; ++q)
        oracle_expert_ffn_rows(H, I, n, x_perm, offsets, w_gate, w_up, w_down, rows[q], rows[q] + 1, y + q * H);
}

/*
 * Combine for the listed tokens: out[q, :] = sum_{j=0..k-1, pair_row[t*k+j] >= 0}
 * topk_w[t,j] * y_perm[pair_row[t*k+j], :], t = tokens[q], summed in slot order
 * (y_perm holds fp32 expert-output rows).
 */
void oracle_combine_tokens(int H, int k, const float* y_perm, const int32_t* pair_row,
                           const float* topk_w, const int64_t* tokens, int64_t ntok, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t q = 0; q < ntok; ++q) {
        int64_t t = tokens[q];
        double* o = out + q * H;
        for (int h = 0; h < H; ++h) o[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            int32_t r = pair_row[t * k + j];
            if (r < 0) continue;
            double w = (double)topk_w[t * k + j];
            for (int h = 0; h < H; ++h) o[h] += w * (double)y_perm[(int64_t)r * H + h];
        }
    }
}

/*
 * The whole local layer, token-major, for the listed tokens (never builds the
 * grouped buffers): route token t, then out[q] = sum over slots j in order of
 * w_tj * FFN_{idx_tj}(x_t) for the slots whose expert lies in [e0, e1).
 * Returns 0, or 5 if a listed token has a non-finite logit.
 */
int oracle_moe_layer_tokens(int H, int I, int E, int k, int e0, int e1, const float* logits,
                            const uint16_t* x, const uint16_t* w_gate, const uint16_t* w_up,
                            const uint16_t* w_down, const int64_t* tokens, int64_t ntok, double* out) {
    if (E < 1 || E > 4096 || k < 1 || k > E || e0 < 0 || e1 <= e0 || e1 > E) return ORACLE_ERR_ARG;
    int status = ORACLE_OK;
#pragma omp parallel reduction(max : status)
    {
        double* xd = (double*)malloc(sizeof(double) * (size_t)H);
        double* act = (double*)malloc(sizeof(double) * (size_t)I);
        double* y = (double*)malloc(sizeof(double) * (size_t)H);
        int32_t idx[4096];
        double w[4096];
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < ntok; ++q) {
            int64_t t = tokens[q];
            double* o = out + q * H;
            for (int h = 0; h < H; ++h) o[h] = 0.0;
            int s = route_one(E, k, logits + t * E, idx, w);
            if (s != ORACLE_OK) {
                if (s > status) status = s;
                continue;
            }
            int have_x = 0;
            for (int j = 0; j < k; ++j) {
                int e = idx[j];
                if (e < e0 || e >= e1) continue;
                if (!have_x) {
                    for (int h = 0; h < H; ++h) xd[h] = bf16_widen(x[t * H + h]);
                    have_x = 1;
                }
                int el = e - e0;
                swiglu_ffn(H, I, xd, w_gate + (int64_t)el * I * H, w_up + (int64_t)el * I * H,
                           w_down + (int64_t)el * H * I, act, y);
                for (int h = 0; h < H; ++h) o[h] += w[j] * y[h];
            }
        }
        free(xd);
        free(act);
        free(y);
    }
    return status;
}

/* number of OpenMP threads a parallel region uses (1 without OpenMP) */
int oracle_num_threads(void) {
#ifdef _OPENMP
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
#else
    return 1;
#endif
}
