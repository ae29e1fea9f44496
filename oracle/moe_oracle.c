/*
 * moe_oracle.c -- CPU oracle for the forward pass of one mixture-of-experts
 * layer: router, token dispatch, expert SwiGLU FFNs, weighted combine.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU path computes.  Only the test suite, the package
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or helper with the CUDA library, and it includes
 * nothing from it.
 *
 * Sources (Hugging Face Transformers documentation and the Ultra-Scale
 * Playbook):
 *   [EP]  "Expert parallelism", intro: a router sends every token to a few
 *         experts and gathers their results.
 *   [EP-add] "Expert parallelism", section "Adding an implementation": the
 *         expert call takes (hidden_states, top_k_index, top_k_weights) and
 *         returns the weighted expert output of every token; the experts run
 *         through experts_forward(tokens, expert_ids, weights).
 *   [EP-disp] "Expert parallelism", section "Token dispatch": each
 *         (token, expert) pair is sent to its expert, the experts run on what
 *         arrives, the results come back and are combined with the routing
 *         weights.
 *   [TP-pack] "Tensor parallelism for inference", section "Packed
 *         strategies": gate_up_proj has shape (num_experts, hidden, 2*f), is
 *         applied as hidden @ gate_up_proj and split with chunk(2, dim=-1)
 *         into (gate, up).
 * The router arithmetic (fp32 logits, softmax, top-k with the lower expert id
 * winning ties, renormalisation over the chosen k), the SwiGLU activation and
 * the stable expert-contiguous order are not printed on those pages; the
 * oracle takes the plainest reading: the definitions written out below.
 *
 * Precision: every sum and product here is in double.  Inputs arrive as the
 * exact float values of the (bf16 or fp32) tensors the GPU reads.  Router
 * logits are rounded once to float, because the method defines an fp32 logit
 * buffer and the selection is made on those fp32 values.
 *
 * Parity pins (what this file is checked against, outside itself): closed
 * forms for two-expert softmax and all-equal logits, a sort-based top-k and a
 * stable argsort for the permutation, the dense SwiGLU MLP for E=1,k=1
 * through library matmuls, the dense soft mixture for k=E without
 * renormalisation, a hand-worked SwiGLU fixture, and one-hot expert rows for
 * the combine (each output entry is then exactly one routing weight).  Every
 * function below is covered by at least one of them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Router logits [EP]: L[t][e] = sum_i x[t][i] * Wr[e][i] (+ bias[e]),
 * the router weight in nn.Linear layout (E rows of d).  The sum is taken in
 * double and rounded once to the fp32 logit the method defines.  bias may be
 * NULL (a per-expert additive logit offset; used for skewed routing).
 */
void oracle_router_logits(int64_t T, int32_t d, int32_t E, const float *x,
                          const float *Wr, const float *bias, float *logits)
{
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; ++t) {
        for (int32_t e = 0; e < E; ++e) {
            double s = 0.0;
            for (int32_t i = 0; i < d; ++i)
                s += (double)x[t * d + i] * (double)Wr[(int64_t)e * d + i];
            if (bias)
                s += (double)bias[e];
            logits[t * E + e] = (float)s;
        }
    }
}

/*
 * Rank order used by the selection: a larger logit comes first; equal logits
 * (+0.0 and -0.0 are equal) go to the lower expert id; a NaN ranks below
 * every number, and two NaNs again go to the lower id.
 */
static int ranks_before(float a, int32_t ia, float b, int32_t ib)
{
    int an = isnan(a), bn = isnan(b);
    if (an || bn) {
        if (an && bn)
            return ia < ib;
        return bn;
    }
    if (a > b)
        return 1;
    if (a < b)
        return 0;
    return ia < ib;
}

/*
 * Top-k routing on a GIVEN fp32 logit buffer [EP-add: top_k_index,
 * top_k_weights].  Slot j holds the j-th pick of k successive passes, each
 * taking the best not-yet-chosen expert under ranks_before().  The weights
 * come from the softmax over all E logits, p_e = exp(L_e - m) / Z with m the
 * largest logit; with renorm the chosen k are divided by their own sum.
 */
void oracle_topk(int64_t T, int32_t E, int32_t k, int32_t renorm,
                 const float *logits, int32_t *idx, double *w)
{
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; ++t) {
        const float *L = logits + t * E;
        unsigned char *chosen = (unsigned char *)calloc((size_t)E, 1);
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e) {
                if (chosen[e])
                    continue;
                if (best < 0 || ranks_before(L[e], e, L[best], best))
                    best = e;
            }
            chosen[best] = 1;
            idx[t * k + j] = best;
        }
        free(chosen);

        double m = -INFINITY;
        for (int32_t e = 0; e < E; ++e)
            if ((double)L[e] > m)
                m = (double)L[e];
        double Z = 0.0;
        for (int32_t e = 0; e < E; ++e)
            Z += exp((double)L[e] - m);
        double sel = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            double p = exp((double)L[idx[t * k + j]] - m) / Z;
            w[t * k + j] = p;
            sel += p;
        }
        if (renorm)
            for (int32_t j = 0; j < k; ++j)
                w[t * k + j] /= sel;
    }
}

/*
 * Token dispatch [EP-disp], single-device form: count the pairs sent to each
 * expert, take the exclusive prefix sum as each expert's first row, then
 * walk the pairs in (token, slot) order and hand each the next free row of
 * its expert.  pos[t*k+j] is the row of pair (t, j); src_token[row] = t.
 * Within an expert the rows are therefore in ascending token order.
 */
void oracle_dispatch(int64_t T, int32_t E, int32_t k, const int32_t *idx,
                     int32_t *counts, int32_t *offsets, int32_t *pos,
                     int32_t *src_token)
{
    int64_t P = T * k;
    for (int32_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t q = 0; q < P; ++q)
        counts[idx[q]] += 1;
    offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int32_t e = 0; e < E; ++e)
        cursor[e] = offsets[e];
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = idx[t * k + j];
            int32_t row = cursor[e]++;
            pos[t * k + j] = row;
            src_token[row] = (int32_t)t;
        }
    }
    free(cursor);
}

/*
 * One expert's SwiGLU FFN on one row [TP-pack, EP-add], on the input row
 * scaled by `scale` (1 unless the routing weights scale expert inputs):
 *   gu   = (scale * x) @ Wgu_e  (Wgu_e is d x 2f, row-major)
 *   gate = gu[0:f], up = gu[f:2f]          (chunk(2, dim=-1))
 *   h    = silu(gate) * up,  silu(z) = z / (1 + exp(-z))
 *   y    = h @ Wd_e             (Wd_e is f x d, row-major)
 * gu (2f) and h (f) are caller scratch; y has d entries.
 */
static void expert_ffn_row_scaled(int32_t d, int32_t f, const float *xrow,
                                  double scale, const float *Wgu_e,
                                  const float *Wd_e, double *gu, double *h,
                                  double *y)
{
    int64_t two_f = 2 * (int64_t)f;
    for (int64_t c = 0; c < two_f; ++c)
        gu[c] = 0.0;
    for (int32_t i = 0; i < d; ++i) {
        double xi = scale * (double)xrow[i];
        const float *wrow = Wgu_e + (int64_t)i * two_f;
        for (int64_t c = 0; c < two_f; ++c)
            gu[c] += xi * (double)wrow[c];
    }
    for (int32_t c = 0; c < f; ++c) {
        double g = gu[c], u = gu[f + c];
        h[c] = g / (1.0 + exp(-g)) * u;
    }
    for (int32_t c = 0; c < d; ++c)
        y[c] = 0.0;
    for (int32_t r = 0; r < f; ++r) {
        double hr = h[r];
        const float *wrow = Wd_e + (int64_t)r * d;
        for (int32_t c = 0; c < d; ++c)
            y[c] += hr * (double)wrow[c];
    }
}

void oracle_expert_ffn_row(int32_t d, int32_t f, const float *xrow,
                           const float *Wgu_e, const float *Wd_e, double *gu,
                           double *h, double *y)
{
    expert_ffn_row_scaled(d, f, xrow, 1.0, Wgu_e, Wd_e, gu, h, y);
}

/*
 * The same FFN on n independent rows [EP-add: experts_forward runs each
 * expert on the rows sent to it]: row r goes through expert expert[r] of the
 * given weight block (Wgu [ne][d][2f], Wd [ne][f][d]; expert[r] indexes that
 * block).  h is [n][f], y is [n][d].  Each row is exactly
 * oracle_expert_ffn_row; rows are spread over threads, nothing else changes.
 */
void oracle_expert_ffn_rows(int64_t n, int32_t d, int32_t f, const float *x,
                            const int32_t *expert, const float *Wgu,
                            const float *Wd, double *h, double *y)
{
    int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < n; ++r) {
        double *gu = (double *)malloc(sizeof(double) * 2 * (size_t)f);
        int64_t e = expert[r];
        expert_ffn_row_scaled(d, f, x + r * d, 1.0, Wgu + e * (int64_t)d * 2 * f,
                              Wd + e * (int64_t)f * d, gu, h + r * f, y + r * d);
        free(gu);
    }
}

/*
 * Layer output of selected tokens [EP-add, EP-disp]: for each listed token t,
 * out[n] = sum over slots j = 0..k-1, in slot order, of
 *   w[t][j] * FFN_{idx[t][j]}(x[t])        (scale_inputs == 0), or
 *   FFN_{idx[t][j]}(w[t][j] * x[t])        (scale_inputs != 0: the experts
 *                                            receive tokens already scaled
 *                                            by the router score [EP intro]).
 * Each (t, j) pair's expert row is exactly the row the dispatch would send,
 * so this is the combine written per token.  out is [ntok][d].
 */
void oracle_token_outputs(int64_t ntok, const int64_t *tokens, int32_t d,
                          int32_t k, int32_t f, const float *x,
                          const float *Wgu, const float *Wd,
                          const int32_t *idx, const double *w,
                          int32_t scale_inputs, double *out)
{
    int64_t n;
#pragma omp parallel for schedule(dynamic, 1)
    for (n = 0; n < ntok; ++n) {
        int64_t t = tokens[n];
        double *gu = (double *)malloc(sizeof(double) * 2 * (size_t)f);
        double *h = (double *)malloc(sizeof(double) * (size_t)f);
        double *y = (double *)malloc(sizeof(double) * (size_t)d);
        double *o = out + n * d;
        for (int32_t c = 0; c < d; ++c)
            o[c] = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            int64_t e = idx[t * k + j];
            double wj = w[t * k + j];
            expert_ffn_row_scaled(d, f, x + t * d, scale_inputs ? wj : 1.0,
                                  Wgu + e * (int64_t)d * 2 * f,
                                  Wd + e * (int64_t)f * d, gu, h, y);
            if (scale_inputs)
                wj = 1.0;
            for (int32_t c = 0; c < d; ++c)
                o[c] += wj * y[c];
        }
        free(gu);
        free(h);
        free(y);
    }
}

/*
 * Combine [EP-add: each token's weighted expert output; EP-disp: the expert
 * results come back and are combined with the routing weights]:
 *   out[t] = sum over slots j = 0..k-1, in slot order, of
 *            w[t][j] * y_perm[pos[t*k+j]]
 * (scale_inputs != 0: the weights were applied to the expert inputs, so the
 * rows are summed unweighted and w is not read).  y_perm [P][d], pos [P],
 * w [T][k], out [T][d].
 */
void oracle_combine(int64_t T, int32_t k, int32_t d, const double *y_perm,
                    const int32_t *pos, const double *w, int32_t scale_inputs,
                    double *out)
{
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; ++t) {
        double *o = out + t * d;
        for (int32_t c = 0; c < d; ++c)
            o[c] = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            const double *yr = y_perm + (int64_t)pos[t * k + j] * d;
            double wj = scale_inputs ? 1.0 : w[t * k + j];
            for (int32_t c = 0; c < d; ++c)
                o[c] += wj * yr[c];
        }
    }
}

/*
 * Whole layer, in the method's order [EP-disp]: logits, top-k, dispatch,
 * each expert on the rows sent to it (y_perm, row by row), then the combine
 * out[t] = sum_j w[t][j] * y_perm[pos[t][j]] in slot order.  With
 * scale_inputs the weight scales each expert's input row instead and the
 * combine sums the rows unweighted [EP intro: experts that receive tokens
 * already scaled by the router score].
 * Outputs: logits [T][E], idx/w [T][k], counts [E], offsets [E+1],
 * pos [T*k], src_token [T*k], out [T][d].
 */
void oracle_moe_forward(int64_t T, int32_t d, int32_t E, int32_t k, int32_t f,
                        int32_t renorm, int32_t scale_inputs, const float *x,
                        const float *Wr, const float *bias, const float *Wgu,
                        const float *Wd, float *logits, int32_t *idx,
                        double *w, int32_t *counts, int32_t *offsets,
                        int32_t *pos, int32_t *src_token, double *out)
{
    int64_t P = T * k;
    oracle_router_logits(T, d, E, x, Wr, bias, logits);
    oracle_topk(T, E, k, renorm, logits, idx, w);
    oracle_dispatch(T, E, k, idx, counts, offsets, pos, src_token);

    /* Expert id of each dispatched row: the e whose segment holds it, and the
     * routing weight the row carries (scale_inputs: applied to the input). */
    int32_t *row_expert = (int32_t *)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    double *row_scale = (double *)malloc(sizeof(double) * (size_t)(P > 0 ? P : 1));
    for (int32_t e = 0; e < E; ++e)
        for (int32_t r = offsets[e]; r < offsets[e + 1]; ++r)
            row_expert[r] = e;
    for (int64_t q = 0; q < P; ++q)
        row_scale[pos[q]] = scale_inputs ? w[q] : 1.0;

    double *y_perm = (double *)malloc(sizeof(double) * (size_t)(P > 0 ? P : 1) * (size_t)d);
    int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < P; ++r) {
        int64_t e = row_expert[r];
        int64_t t = src_token[r];
        double *gu = (double *)malloc(sizeof(double) * 2 * (size_t)f);
        double *h = (double *)malloc(sizeof(double) * (size_t)f);
        expert_ffn_row_scaled(d, f, x + t * d, row_scale[r],
                              Wgu + e * (int64_t)d * 2 * f,
                              Wd + e * (int64_t)f * d, gu, h, y_perm + r * d);
        free(gu);
        free(h);
    }

    oracle_combine(T, k, d, y_perm, pos, w, scale_inputs, out);
    free(y_perm);
    free(row_expert);
    free(row_scale);
}
