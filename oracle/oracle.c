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

/*
 * MXFP8: "Hosting Qwen on Blackwell", section "MoE GEMM": the deployed expert
 * GEMMs use MXFP8.  The pages give no format details; the plain reading is the
 * OCP Microscaling Formats (MX) v1.0 definition of MXFP8:
 *   - blocks of 32 consecutive elements along K share one UE8M0 scale
 *     X = 2^(code - 127) (code 255 = NaN is never produced);
 *   - X = 2^(floor(log2(amax)) - 8), 8 being the largest exponent of an E4M3
 *     normal number (448 = 1.75 * 2^8), with amax the block's largest |v|; a
 *     block of zeros gets code 0; the code is clamped to [0, 254];
 *   - each element is v / X rounded to the nearest E4M3 value (ties to an even
 *     mantissa), saturating at +-448 (E4M3 has no infinities; 0x7f / 0xff are
 *     NaN); a negative value keeps its sign bit even when it rounds to zero.
 * E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 holds the
 * subnormals m * 2^-9.
 */
static double e4m3_decode(uint8_t b) {
    const int e = (b >> 3) & 15, m = b & 7;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (b & 0x80) ? -v : v;
}

/* nearest E4M3 code of v (|v| is the element divided by its block scale) */
static uint8_t e4m3_encode(double v) {
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7e; /* saturate (also the rounding of 448..464) */
    int e;
    double q;                           /* quantum of a's binade */
    if (a < ldexp(1.0, -6)) {
        e = -6;                         /* subnormal range: steps of 2^-9 */
        q = ldexp(1.0, -9);
    } else {
        e = (int)floor(log2(a));
        if (ldexp(1.0, e) > a) --e;     /* guard log2 rounding */
        if (ldexp(1.0, e + 1) <= a) ++e;
        q = ldexp(1.0, e - 3);
    }
    double m = nearbyint(a / q);        /* ties to even (default rounding mode) */
    double val = m * q;                 /* exact, at most 448 since a < 448 */
    if (val == 0.0) return sign;
    /* re-derive the code of the exactly representable value */
    if (val < ldexp(1.0, -6)) return sign | (uint8_t)(val / ldexp(1.0, -9));
    int ve = (int)floor(log2(val));
    if (ldexp(1.0, ve) > val) --ve;
    if (ldexp(1.0, ve + 1) <= val) ++ve;
    const int mant = (int)(val / ldexp(1.0, ve - 3)) - 8;
    return sign | (uint8_t)(((ve + 7) << 3) | mant);
}

/* scale code of a block whose largest magnitude is amax */
static uint8_t mx_scale_code(double amax) {
    if (amax == 0.0) return 0;
    int p = (int)floor(log2(amax));
    if (ldexp(1.0, p) > amax) --p;
    if (ldexp(1.0, p + 1) <= amax) ++p;
    int c = p - 8 + 127;
    return (uint8_t)(c < 0 ? 0 : c > 254 ? 254 : c);
}

/* quantise len values (len <= 32) of one block */
static void mx_quantize_block(const double* v, int len, uint8_t* q, uint8_t* s) {
    double amax = 0.0;
    for (int i = 0; i < len; ++i) amax = fmax(amax, fabs(v[i]));
    *s = mx_scale_code(amax);
    const double x = ldexp(1.0, (int)*s - 127);
    for (int i = 0; i < len; ++i) q[i] = e4m3_encode(v[i] / x);
}

/*
 * MXFP8 quantisation of a bf16 matrix [rows, K] along K: q uint8 [rows, K] (E4M3
 * codes), s uint8 [rows, K / 32] (UE8M0 codes).  K must be a multiple of 32.
 */
int oracle_mxfp8_quantize(int64_t rows, int K, const uint16_t* src, uint8_t* q, uint8_t* s) {
    if (rows < 0 || K <= 0 || K % 32) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double v[32];
        for (int b = 0; b < K / 32; ++b) {
            for (int i = 0; i < 32; ++i) v[i] = bf16_widen(src[r * K + b * 32 + i]);
            mx_quantize_block(v, 32, q + r * K + b * 32, s + r * (K / 32) + b);
        }
    }
    return ORACLE_OK;
}

/* one row of K elements: out[k] = E4M3(q[k]) * 2^(s[k / 32] - 127) */
static void mx_dequantize_row(int K, const uint8_t* q, const uint8_t* s, double* out) {
    for (int k = 0; k < K; ++k) out[k] = e4m3_decode(q[k]) * ldexp(1.0, (int)s[k / 32] - 127);
}

/* out[r, k] = E4M3(q[r, k]) * 2^(s[r, k / 32] - 127), in fp64 */
void oracle_mxfp8_dequantize(int64_t rows, int K, const uint8_t* q, const uint8_t* s, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) mx_dequantize_row(K, q + r * K, s + r * (K / 32), out + r * K);
}

/*
 * The expert FFN with MXFP8 operands, on an explicit list of grouped rows: the
 * gate/up GEMM on the dequantised x_perm row and weights (fp64), h = silu(g) * u
 * (fp64), h quantised to MXFP8 along I (blocks of 32, the same rule), then the
 * down GEMM on the dequantised h and W_down (fp64).
 *   xq/xs: x_perm [*, H] / [*, H/32];  wgq, wuq [n, I, H] with wgs, wus [n, I, H/32];
 *   wdq [n, H, I] with wds [n, H, I/32].
 *   h_in_q / h_in_s (optional, [nrows, I] / [nrows, I/32]): use this quantised h
 *   for the down GEMM instead of the oracle's own (to check a down GEMM alone).
 *   h_out (optional, fp64 [nrows, I]): h before quantisation;
 *   hq_out / hs_out (optional): the oracle's quantised h.
 * y: fp64 [nrows, H].  Rows outside every expert get y = 0.
 */
void oracle_expert_ffn_mxfp8_rowlist(int H, int I, int n, const uint8_t* xq, const uint8_t* xs,
                                     const int32_t* offsets, const uint8_t* wgq, const uint8_t* wgs,
                                     const uint8_t* wuq, const uint8_t* wus, const uint8_t* wdq, const uint8_t* wds,
                                     const int64_t* rows, int64_t nrows, const uint8_t* h_in_q,
                                     const uint8_t* h_in_s, double* h_out, uint8_t* hq_out, uint8_t* hs_out,
                                     double* y) {
#pragma omp parallel
    {
        double* xd = (double*)malloc(sizeof(double) * (size_t)H);
        double* w = (double*)malloc(sizeof(double) * (size_t)(H > I ? H : I));
        double* h = (double*)malloc(sizeof(double) * (size_t)I);
        double* hd = (double*)malloc(sizeof(double) * (size_t)I);
        uint8_t* hq = (uint8_t*)malloc((size_t)I);
        uint8_t* hs = (uint8_t*)malloc((size_t)I / 32 + 1);
#pragma omp for schedule(dynamic, 1)
        for (int64_t qi = 0; qi < nrows; ++qi) {
            const int64_t r = rows[qi];
            double* yr = y + qi * H;
            int e = -1;
            for (int c = 0; c < n; ++c)
                if (r >= offsets[c] && r < offsets[c + 1]) { e = c; break; }
            if (e < 0) {
                for (int j = 0; j < H; ++j) yr[j] = 0.0;
                continue;
            }
            mx_dequantize_row(H, xq + r * H, xs + r * (H / 32), xd);
            for (int i = 0; i < I; ++i) {
                const int64_t wr = (int64_t)e * I + i;
                double g = 0.0, u = 0.0;
                mx_dequantize_row(H, wgq + wr * H, wgs + wr * (H / 32), w);
                for (int j = 0; j < H; ++j) g += w[j] * xd[j];
                mx_dequantize_row(H, wuq + wr * H, wus + wr * (H / 32), w);
                for (int j = 0; j < H; ++j) u += w[j] * xd[j];
                h[i] = g / (1.0 + exp(-g)) * u;
            }
            for (int b = 0; b < I / 32; ++b) mx_quantize_block(h + b * 32, 32, hq + b * 32, hs + b);
            if (h_out) memcpy(h_out + qi * I, h, sizeof(double) * (size_t)I);
            if (hq_out) memcpy(hq_out + qi * I, hq, (size_t)I);
            if (hs_out) memcpy(hs_out + qi * (I / 32), hs, (size_t)I / 32);
            if (h_in_q)
                mx_dequantize_row(I, h_in_q + qi * I, h_in_s + qi * (I / 32), hd);
            else
                mx_dequantize_row(I, hq, hs, hd);
            for (int j = 0; j < H; ++j) {
                const int64_t wr = (int64_t)e * H + j;
                mx_dequantize_row(I, wdq + wr * I, wds + wr * (I / 32), w);
                double acc = 0.0;
                for (int i = 0; i < I; ++i) acc += w[i] * hd[i];
                yr[j] = acc;
            }
        }
        free(xd);
        free(w);
        free(h);
        free(hd);
        free(hq);
        free(hs);
    }
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
