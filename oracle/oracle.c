/*
 * oracle.c -- float64 CPU reference for fused scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: it exists so that tests, the smoke check and the timed CPU
 * baseline of the benchmark can compare the CUDA library against the plain
 * definition of the operation.  It shares no code, header or table with the
 * CUDA library.
 *
 * What it computes (the textbook definition; the pages never write it out,
 * but every API they call is this operation: "Add torch scaled dot product
 * attention (FlashAttention)", title; "Significant Accuracy Difference
 * between Compiled and Eager Flex Attention", repro calling flex_attention
 * and torch.nn.functional.scaled_dot_product_attention):
 *
 *   s_ij  = scale * <q_i, k_j>                       for visible keys j
 *   LSE_i = log sum_j exp(s_ij)        (natural log, over the scaled scores)
 *   p_ij  = exp(s_ij - LSE_i)
 *   o_i   = sum_j p_ij v_j
 *
 * Visibility ("[PyTorch] fused CUDNN attention kernel not properly handling
 * strides", the window_size=(-1, 0) argument; "Significant Accuracy
 * Difference ...", sliding_window_causal mask_mod (q_idx >= kv_idx) &
 * (q_idx - kv_idx <= band)): key j is visible to query i iff
 *   (wl < 0 or j >= i - wl) and (wr < 0 or j <= i + wr) and 0 <= j < L_kv,
 * with i and j counted from 0 inside their own sequence (top-left aligned).
 * A row with no visible key gets o_i = 0 and LSE_i = -inf.
 *
 * Grouped heads ("[PyTorch] fused CUDNN attention ...", q_heads=16,
 * kv_heads=1, num_gqa_groups): query head h reads key/value head h / G with
 * G = Hq / Hkv.
 *
 * Packing ("[PyTorch] Add support for cuDNN FusedAttention + THD + CP",
 * the thd branch addressed by cu_seqlens): every tensor is given as rows of
 * tokens; sequence b owns query rows [cu_q[b], cu_q[b+1]) and key/value rows
 * [cu_kv[b], cu_kv[b+1]).  A dense batch is the special case
 * cu[b] = b * S.  Layouts (all contiguous, float64):
 *   q, o, dq : [Tq][Hq][D]      k, v, dk, dv : [Tkv][Hkv][D]
 *   lse, delta : [Tq][Hq]
 *
 * Backward (gradient of sum(dO * O) as in the repro's out.sum().backward(),
 * plus sum(dLSE * LSE) when an LSE gradient is given: the flex-attention
 * issue returns the LSE and merges through it, so a loss can reach the
 * scores through LSE as well as through O; d LSE_i / d s_ij = p_ij):
 *   dP_ij = <dO_i, v_j>
 *   r_i   = sum_j p_ij dP_ij          (the definitional softmax row term)
 *   dS_ij = p_ij (dP_ij - r_i + dLSE_i)
 *   dq_i  = scale * sum_j dS_ij k_j
 *   dk_j  = scale * sum_{h in group} sum_i dS_ij q_i
 *   dv_j  = sum_{h in group} sum_i p_ij dO_i
 *
 * LSE merge ("Significant Accuracy Difference ...", merge_attn): the two
 * partial results are weighted by exp(lse - max) and renormalised.  When
 * both sides are -inf (no visible key on either side) the merged row is
 * o = 0, lse = -inf instead of the NaN the formula would give.
 *
 * Merge backward: the derivative of that formula.  With w_k = e_k / (e1 + e2),
 * o = w1 o1 + w2 o2 and lse = m + log(e1 + e2):
 *   d o / d o_k = w_k,   d o / d lse_k = w_k (o_k - o),   d lse / d lse_k = w_k
 * so for upstream gradients dO, dLSE of the merged row:
 *   dO_k = w_k dO,   dLSE_k = w_k (<dO, o_k - o> + dLSE)
 * (both zero for a side whose lse is -inf).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Sequence that owns packed row t, by linear search over cu[0..nseq]. */
static int seq_of_row(int nseq, const int64_t *cu, int64_t t) {
    for (int b = 0; b < nseq; ++b)
        if (t >= cu[b] && t < cu[b + 1]) return b;
    return -1;
}

static int visible(int64_t i, int64_t j, int64_t len_kv, int wl, int wr) {
    if (j < 0 || j >= len_kv) return 0;
    if (wl >= 0 && j < i - wl) return 0;
    if (wr >= 0 && j > i + wr) return 0;
    return 1;
}

static double dot(const double *a, const double *b, int n) {
    double s = 0.0;
    for (int d = 0; d < n; ++d) s += a[d] * b[d];
    return s;
}

/* log-sum-exp of the scaled scores of query row (t, h); returns -inf when no
 * key is visible.  s must have room for len_kv doubles and receives s_ij
 * (garbage for invisible j). */
static double row_scores_lse(const double *qrow, const double *k, int64_t kv0,
                             int64_t len_kv, int Hkv, int hk, int D,
                             double scale, int64_t i, int wl, int wr,
                             double *s) {
    double m = -INFINITY;
    for (int64_t j = 0; j < len_kv; ++j) {
        if (!visible(i, j, len_kv, wl, wr)) continue;
        s[j] = scale * dot(qrow, k + ((kv0 + j) * Hkv + hk) * D, D);
        if (s[j] > m) m = s[j];
    }
    if (m == -INFINITY) return -INFINITY;
    double sum = 0.0;
    for (int64_t j = 0; j < len_kv; ++j)
        if (visible(i, j, len_kv, wl, wr)) sum += exp(s[j] - m);
    return m + log(sum);
}

static int64_t max_len(int nseq, const int64_t *cu) {
    int64_t mx = 1;
    for (int b = 0; b < nseq; ++b)
        if (cu[b + 1] - cu[b] > mx) mx = cu[b + 1] - cu[b];
    return mx;
}

/* Forward.  row_sel (optional, [Tq][Hq]) selects which (row, head) outputs to
 * compute; unselected outputs are left untouched. */
void oracle_attn_fwd(int nseq, const int64_t *cu_q, const int64_t *cu_kv,
                     int Hq, int Hkv, int D, const double *q, const double *k,
                     const double *v, double scale, int wl, int wr,
                     const uint8_t *row_sel, double *o, double *lse) {
    const int G = Hq / Hkv;
    const int64_t Tq = cu_q[nseq];
    const int64_t Lmax = max_len(nseq, cu_kv);
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Lmax);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < Tq * Hq; ++r) {
            if (row_sel && !row_sel[r]) continue;
            const int64_t t = r / Hq;
            const int h = (int)(r % Hq), hk = h / G;
            const int b = seq_of_row(nseq, cu_q, t);
            const int64_t i = t - cu_q[b], kv0 = cu_kv[b];
            const int64_t len_kv = cu_kv[b + 1] - kv0;
            const double *qrow = q + r * D;
            double *orow = o + r * D;
            const double L = row_scores_lse(qrow, k, kv0, len_kv, Hkv, hk, D,
                                            scale, i, wl, wr, s);
            for (int d = 0; d < D; ++d) orow[d] = 0.0;
            lse[r] = L;
            if (L == -INFINITY) continue;
            for (int64_t j = 0; j < len_kv; ++j) {
                if (!visible(i, j, len_kv, wl, wr)) continue;
                const double p = exp(s[j] - L);
                const double *vrow = v + ((kv0 + j) * Hkv + hk) * D;
                for (int d = 0; d < D; ++d) orow[d] += p * vrow[d];
            }
        }
        free(s);
    }
}

/* Backward.  dlse (optional, [Tq][Hq]) is the gradient of the loss with
 * respect to LSE (NULL: zero).  row_sel (optional, [Tq][Hq]) selects the dq
 * rows to compute, key_sel (optional, [Tkv][Hkv]) the dk/dv rows;
 * unselected outputs are left untouched.  lse_out and r_out (optional,
 * [Tq][Hq]) receive LSE_i and the row term r_i of every row that some
 * selected output depends on. */
void oracle_attn_bwd(int nseq, const int64_t *cu_q, const int64_t *cu_kv,
                     int Hq, int Hkv, int D, const double *q, const double *k,
                     const double *v, const double *dout, const double *dlse,
                     double scale, int wl, int wr, const uint8_t *row_sel,
                     const uint8_t *key_sel, double *dq, double *dk, double *dv,
                     double *lse_out, double *r_out) {
    const int G = Hq / Hkv;
    const int64_t Tq = cu_q[nseq], Tkv = cu_kv[nseq];
    const int64_t Lmax = max_len(nseq, cu_kv);

    /* Which (sequence, kv head) units have a selected dk/dv row. */
    uint8_t *unit = (uint8_t *)calloc((size_t)nseq * Hkv, 1);
    for (int64_t r = 0; r < Tkv * Hkv; ++r) {
        if (key_sel && !key_sel[r]) continue;
        const int b = seq_of_row(nseq, cu_kv, r / Hkv);
        if (b >= 0) unit[b * Hkv + (int)(r % Hkv)] = 1;
    }
    double *L = (double *)malloc(sizeof(double) * (size_t)(Tq * Hq));
    double *R = (double *)malloc(sizeof(double) * (size_t)(Tq * Hq));

    /* Pass 1: LSE_i and r_i = sum_j p_ij dP_ij for every needed row. */
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Lmax);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < Tq * Hq; ++r) {
            const int64_t t = r / Hq;
            const int h = (int)(r % Hq), hk = h / G;
            const int b = seq_of_row(nseq, cu_q, t);
            const int need = (row_sel ? row_sel[r] : 1) || unit[b * Hkv + hk];
            if (!need) continue;
            const int64_t i = t - cu_q[b], kv0 = cu_kv[b];
            const int64_t len_kv = cu_kv[b + 1] - kv0;
            L[r] = row_scores_lse(q + r * D, k, kv0, len_kv, Hkv, hk, D, scale,
                                  i, wl, wr, s);
            double acc = 0.0;
            if (L[r] != -INFINITY) {
                for (int64_t j = 0; j < len_kv; ++j) {
                    if (!visible(i, j, len_kv, wl, wr)) continue;
                    const double p = exp(s[j] - L[r]);
                    acc += p * dot(dout + r * D,
                                   v + ((kv0 + j) * Hkv + hk) * D, D);
                }
            }
            R[r] = acc;
            if (lse_out) lse_out[r] = L[r];
            if (r_out) r_out[r] = R[r];
        }
        free(s);
    }

    /* Pass 2: dq_i for selected rows. */
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < Tq * Hq; ++r) {
        if (row_sel && !row_sel[r]) continue;
        const int64_t t = r / Hq;
        const int h = (int)(r % Hq), hk = h / G;
        const int b = seq_of_row(nseq, cu_q, t);
        const int64_t i = t - cu_q[b], kv0 = cu_kv[b];
        const int64_t len_kv = cu_kv[b + 1] - kv0;
        double *dqrow = dq + r * D;
        for (int d = 0; d < D; ++d) dqrow[d] = 0.0;
        if (L[r] == -INFINITY) continue;
        for (int64_t j = 0; j < len_kv; ++j) {
            if (!visible(i, j, len_kv, wl, wr)) continue;
            const double *krow = k + ((kv0 + j) * Hkv + hk) * D;
            const double *vrow = v + ((kv0 + j) * Hkv + hk) * D;
            const double p = exp(scale * dot(q + r * D, krow, D) - L[r]);
            const double g = dlse ? dlse[r] : 0.0;
            const double dS = p * (dot(dout + r * D, vrow, D) - R[r] + g);
            for (int d = 0; d < D; ++d) dqrow[d] += scale * dS * krow[d];
        }
    }

    /* Pass 3: dk_j, dv_j for selected keys, summed over the query heads of
     * the group and over every query row that sees key j. */
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t rk = 0; rk < Tkv * Hkv; ++rk) {
        if (key_sel && !key_sel[rk]) continue;
        const int64_t tk = rk / Hkv;
        const int hk = (int)(rk % Hkv);
        const int b = seq_of_row(nseq, cu_kv, tk);
        double *dkrow = dk + rk * D, *dvrow = dv + rk * D;
        for (int d = 0; d < D; ++d) dkrow[d] = dvrow[d] = 0.0;
        if (b < 0) continue;
        const int64_t j = tk - cu_kv[b], len_kv = cu_kv[b + 1] - cu_kv[b];
        const double *krow = k + rk * D, *vrow = v + rk * D;
        for (int h = hk * G; h < (hk + 1) * G; ++h) {
            for (int64_t t = cu_q[b]; t < cu_q[b + 1]; ++t) {
                const int64_t i = t - cu_q[b], r = t * Hq + h;
                if (!visible(i, j, len_kv, wl, wr)) continue;
                const double p = exp(scale * dot(q + r * D, krow, D) - L[r]);
                const double g = dlse ? dlse[r] : 0.0;
                const double dS = p * (dot(dout + r * D, vrow, D) - R[r] + g);
                for (int d = 0; d < D; ++d) {
                    dkrow[d] += scale * dS * q[r * D + d];
                    dvrow[d] += p * dout[r * D + d];
                }
            }
        }
    }
    free(L);
    free(R);
    free(unit);
}

/* LSE merge of two partial attentions over disjoint key sets.
 * o1, o2, o : [n][D]; lse1, lse2, lse : [n]. */
void oracle_merge_lse(int64_t n, int D, const double *o1, const double *lse1,
                      const double *o2, const double *lse2, double *o,
                      double *lse) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        const double mx = lse1[r] > lse2[r] ? lse1[r] : lse2[r];
        if (mx == -INFINITY) {
            for (int d = 0; d < D; ++d) o[r * D + d] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        const double e1 = exp(lse1[r] - mx), e2 = exp(lse2[r] - mx);
        for (int d = 0; d < D; ++d)
            o[r * D + d] = (o1[r * D + d] * e1 + o2[r * D + d] * e2) / (e1 + e2);
        lse[r] = mx + log(e1 + e2);
    }
}

/* Backward of the LSE merge.  dout : [n][D] gradient of the merged o;
 * dlse (optional) : [n] gradient of the merged lse; outputs do1, do2 : [n][D]
 * and dlse1, dlse2 : [n]. */
void oracle_merge_lse_bwd(int64_t n, int D, const double *o1, const double *lse1,
                          const double *o2, const double *lse2,
                          const double *dout, const double *dlse, double *do1,
                          double *dlse1, double *do2, double *dlse2) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        const double mx = lse1[r] > lse2[r] ? lse1[r] : lse2[r];
        double w1 = 0.0, w2 = 0.0;
        if (mx != -INFINITY) {
            const double e1 = exp(lse1[r] - mx), e2 = exp(lse2[r] - mx);
            w1 = e1 / (e1 + e2);
            w2 = e2 / (e1 + e2);
        }
        double g1 = 0.0, g2 = 0.0;  /* <dO, o_k - o> */
        for (int d = 0; d < D; ++d) {
            const double o = w1 * o1[r * D + d] + w2 * o2[r * D + d];
            g1 += dout[r * D + d] * (o1[r * D + d] - o);
            g2 += dout[r * D + d] * (o2[r * D + d] - o);
            do1[r * D + d] = w1 * dout[r * D + d];
            do2[r * D + d] = w2 * dout[r * D + d];
        }
        const double g = dlse ? dlse[r] : 0.0;
        dlse1[r] = w1 * (g1 + g);
        dlse2[r] = w2 * (g2 + g);
    }
}

/* Number of OpenMP threads a parallel region uses (for the baseline's
 * "cores" field); 1 without OpenMP. */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
#else
int oracle_num_threads(void) { return 1; }
#endif
