/*
 * fa_oracle.c -- plain, slow, fp64 CPU oracle for exact scaled dot-product
 * attention (forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Every routine works on ONE sequence and ONE key/value head together with
 * the G query heads that read it (grouped-query attention), all in fp64:
 *
 *   q    [G][L][d]   query rows of the G query heads of the group
 *   k, v [L][d]      key / value rows of the shared key/value head
 *   dout [G][L][d]   upstream gradient dO
 *
 * Batching, packing (cu_seqlens) and the head grouping are unrolled by the
 * Python wrapper in this directory, which slices the device layouts into
 * these per-group arrays.
 *
 * Sources (page title, then section / equation):
 *  - "FlashAttention: How IO-Aware Tiling and Online Softmax Solved
 *    Transformer Memory Bottlenecks", section "Naive Attention Execution
 *    Profile": S = Q K^T, P = softmax(S), O = P V.
 *  - same page, section "2. Online Softmax Reduction": the max-subtracted
 *    softmax softmax(x)_i = e^{x_i - m} / sum_j e^{x_j - m}, m = max_j x_j,
 *    and the block recurrence for m^(j), l^(j), O_i^(j) and the final
 *    O_i = diag(l)^-1 O_i (used only by fa_oracle_fwd_tiled).
 *  - "Flash Attention -- Fast Memory-Efficient Exact Attention", section
 *    "Architecture Overview": the backward pass works from the saved output
 *    and the logsumexp statistics; "What Flash Attention Does": causal
 *    masking, variable-length sequences and GQA/MQA; "Key Features":
 *    sliding-window masks.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - scores carry an explicit softmax scale: S_ij = scale * q_i . k_j;
 *  - causal: key j is visible to query i iff j <= i (same sequence);
 *  - sliding window W > 0: additionally i - j < W (W keys including i);
 *  - logsumexp is the natural log: LSE_i = m_i + ln l_i;
 *  - a row with no visible key gets O_i = 0 and LSE_i = -inf and contributes
 *    no gradient;
 *  - backward (the pages give no formulas; this is the calculus of
 *    softmax): dV_j = sum_i P_ij dO_i, dP_ij = dO_i . v_j,
 *    D_i = dO_i . O_i, dS_ij = P_ij (dP_ij - D_i),
 *    dQ_i = scale sum_j dS_ij k_j, dK_j = scale sum_i dS_ij q_i,
 *    with dK and dV summed over the G query heads of the group.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Visible key range of query row i: keys j in [*lo, *hi] (empty if lo > hi). */
static void visible_range(int i, int L, int causal, int window, int* lo, int* hi) {
    int l = 0, h = L - 1;
    if (causal && i < h) h = i;
    if (window > 0 && i - window + 1 > l) l = i - window + 1;
    *lo = l;
    *hi = h;
}

static double dot(const double* a, const double* b, int d) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

/*
 * Row statistics of query row i of head g by the plain definition:
 * m = max_j S_ij, l = sum_j exp(S_ij - m) over the visible keys, and (if o is
 * not NULL) O_i = sum_j exp(S_ij - m) / l * v_j.  srow is scratch of size L.
 * Returns 0 if the row has no visible key (then m = -inf, l = 0, O = 0).
 */
static int row_forward(const double* qi, const double* k, const double* v, int L, int d,
                       int causal, int window, double scale, int i, double* srow,
                       double* m_out, double* l_out, double* o) {
    int lo, hi;
    visible_range(i, L, causal, window, &lo, &hi);
    if (o) memset(o, 0, sizeof(double) * (size_t)d);
    if (lo > hi) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return 0;
    }
    double m = -INFINITY;
    for (int j = lo; j <= hi; ++j) {
        srow[j] = scale * dot(qi, k + (size_t)j * d, d);
        if (srow[j] > m) m = srow[j];
    }
    double l = 0.0;
    for (int j = lo; j <= hi; ++j) l += exp(srow[j] - m);
    if (o) {
        for (int j = lo; j <= hi; ++j) {
            double p = exp(srow[j] - m) / l;
            const double* vj = v + (size_t)j * d;
            for (int c = 0; c < d; ++c) o[c] += p * vj[c];
        }
    }
    *m_out = m;
    *l_out = l;
    return 1;
}

/*
 * Forward pass.  rows == NULL computes every row (nrows must then equal L);
 * otherwise only the listed query rows.  Outputs: o [G][nrows][d],
 * lse [G][nrows].  Returns 0 on success, -1 on bad arguments.
 */
int fa_oracle_fwd(const double* q, const double* k, const double* v, int G, int L, int d,
                  int causal, int window, double scale, const int* rows, int nrows,
                  double* o, double* lse) {
    if (G <= 0 || L < 0 || d <= 0 || nrows < 0) return -1;
    if (!rows && nrows != L) return -1;
    long total = (long)G * nrows;
#pragma omp parallel
    {
        double* srow = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
#pragma omp for schedule(dynamic, 4)
        for (long t = 0; t < total; ++t) {
            int g = (int)(t / nrows), r = (int)(t % nrows);
            int i = rows ? rows[r] : r;
            double m, l;
            double* orow = o + ((size_t)g * nrows + r) * d;
            int any = row_forward(q + ((size_t)g * L + i) * d, k, v, L, d, causal, window, scale, i,
                                  srow, &m, &l, orow);
            lse[(size_t)g * nrows + r] = any ? m + log(l) : -INFINITY;
        }
        free(srow);
    }
    return 0;
}

/*
 * Forward pass by the block recurrence of the online softmax: query blocks of
 * Br rows, key/value blocks of Bc rows (ragged last blocks allowed).  Per
 * query block the running state (m, l, O) is updated block by block:
 *   m_new = max(m_old, rowmax(S_block))
 *   l     = exp(m_old - m_new) l + rowsum(exp(S_block - m_new))
 *   O     = diag(exp(m_old - m_new)) O + exp(S_block - m_new) V_block
 * and O = diag(l)^-1 O at the end.  Masked scores are -inf; a row whose
 * running max is still -inf skips the update (nothing visible yet).
 * Outputs o [G][L][d], lse [G][L].  This is a second, independent route to
 * the forward result, used to check the recurrence against the definition.
 */
int fa_oracle_fwd_tiled(const double* q, const double* k, const double* v, int G, int L, int d,
                        int causal, int window, double scale, int Br, int Bc, double* o,
                        double* lse) {
    if (G <= 0 || L < 0 || d <= 0 || Br <= 0 || Bc <= 0) return -1;
    int nqb = (L + Br - 1) / Br;
    long total = (long)G * nqb;
#pragma omp parallel
    {
        double* m = (double*)malloc(sizeof(double) * (size_t)Br);
        double* l = (double*)malloc(sizeof(double) * (size_t)Br);
        double* acc = (double*)malloc(sizeof(double) * (size_t)Br * d);
        double* s = (double*)malloc(sizeof(double) * (size_t)Br * Bc);
#pragma omp for schedule(dynamic, 1)
        for (long t = 0; t < total; ++t) {
            int g = (int)(t / nqb), qb = (int)(t % nqb);
            int i0 = qb * Br, rows = (L - i0 < Br) ? L - i0 : Br;
            for (int r = 0; r < rows; ++r) {
                m[r] = -INFINITY;
                l[r] = 0.0;
                for (int c = 0; c < d; ++c) acc[(size_t)r * d + c] = 0.0;
            }
            for (int j0 = 0; j0 < L; j0 += Bc) {
                int cols = (L - j0 < Bc) ? L - j0 : Bc;
                for (int r = 0; r < rows; ++r) {
                    int i = i0 + r, lo, hi;
                    visible_range(i, L, causal, window, &lo, &hi);
                    const double* qi = q + ((size_t)g * L + i) * d;
                    double mt = -INFINITY;
                    for (int cc = 0; cc < cols; ++cc) {
                        int j = j0 + cc;
                        double sv = (j >= lo && j <= hi) ? scale * dot(qi, k + (size_t)j * d, d)
                                                         : -INFINITY;
                        s[(size_t)r * Bc + cc] = sv;
                        if (sv > mt) mt = sv;
                    }
                    double mnew = m[r] > mt ? m[r] : mt;
                    if (mnew == -INFINITY) continue; /* nothing visible so far */
                    double alpha = exp(m[r] - mnew); /* exp(-inf) = 0 on the first hit */
                    double rs = 0.0;
                    double* ar = acc + (size_t)r * d;
                    for (int c = 0; c < d; ++c) ar[c] *= alpha;
                    for (int cc = 0; cc < cols; ++cc) {
                        double p = exp(s[(size_t)r * Bc + cc] - mnew);
                        rs += p;
                        if (p != 0.0) {
                            const double* vj = v + (size_t)(j0 + cc) * d;
                            for (int c = 0; c < d; ++c) ar[c] += p * vj[c];
                        }
                    }
                    l[r] = alpha * l[r] + rs;
                    m[r] = mnew;
                }
            }
            for (int r = 0; r < rows; ++r) {
                int i = i0 + r;
                double* orow = o + ((size_t)g * L + i) * d;
                if (l[r] > 0.0) {
                    for (int c = 0; c < d; ++c) orow[c] = acc[(size_t)r * d + c] / l[r];
                    lse[(size_t)g * L + i] = m[r] + log(l[r]);
                } else {
                    for (int c = 0; c < d; ++c) orow[c] = 0.0;
                    lse[(size_t)g * L + i] = -INFINITY;
                }
            }
        }
        free(m);
        free(l);
        free(acc);
        free(s);
    }
    return 0;
}

/*
 * Backward pass (analytic gradients of the loss <dO, O> with respect to
 * Q, K and V).  qrows/nq select the dQ rows to return (NULL: all, nq == L),
 * krows/nk the dK/dV rows (NULL: all, nk == L).  Outputs dq [G][nq][d],
 * dk [nk][d], dv [nk][d]; dk and dv are summed over the G query heads.
 * P is formed from the row max and normaliser (m, l) of the definition.
 */
int fa_oracle_bwd(const double* q, const double* k, const double* v, const double* dout, int G,
                  int L, int d, int causal, int window, double scale, const int* qrows, int nq,
                  const int* krows, int nk, double* dq, double* dk, double* dv) {
    if (G <= 0 || L < 0 || d <= 0 || nq < 0 || nk < 0) return -1;
    if ((!qrows && nq != L) || (!krows && nk != L)) return -1;
    size_t GL = (size_t)G * L;
    double* m = (double*)malloc(sizeof(double) * (GL ? GL : 1));
    double* l = (double*)malloc(sizeof(double) * (GL ? GL : 1));
    double* D = (double*)malloc(sizeof(double) * (GL ? GL : 1));
    if (!m || !l || !D) {
        free(m);
        free(l);
        free(D);
        return -2;
    }
    /* Pass 1: m_i, l_i and D_i = dO_i . O_i for every row of every head. */
#pragma omp parallel
    {
        double* srow = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double* orow = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
        for (long t = 0; t < (long)GL; ++t) {
            int g = (int)(t / L), i = (int)(t % L);
            row_forward(q + ((size_t)g * L + i) * d, k, v, L, d, causal, window, scale, i, srow,
                        &m[t], &l[t], orow);
            D[t] = dot(dout + ((size_t)g * L + i) * d, orow, d);
        }
        free(srow);
        free(orow);
    }
    /* Pass 2: dQ_i = scale * sum_j dS_ij k_j for the requested rows. */
#pragma omp parallel for schedule(dynamic, 4)
    for (long t = 0; t < (long)G * nq; ++t) {
        int g = (int)(t / nq), r = (int)(t % nq);
        int i = qrows ? qrows[r] : r;
        size_t gi = (size_t)g * L + i;
        double* out = dq + ((size_t)g * nq + r) * d;
        for (int c = 0; c < d; ++c) out[c] = 0.0;
        if (l[gi] == 0.0) continue;
        int lo, hi;
        visible_range(i, L, causal, window, &lo, &hi);
        const double* qi = q + gi * d;
        const double* doi = dout + gi * d;
        for (int j = lo; j <= hi; ++j) {
            double p = exp(scale * dot(qi, k + (size_t)j * d, d) - m[gi]) / l[gi];
            double dp = dot(doi, v + (size_t)j * d, d);
            double ds = p * (dp - D[gi]);
            const double* kj = k + (size_t)j * d;
            for (int c = 0; c < d; ++c) out[c] += scale * ds * kj[c];
        }
    }
    /* Pass 3: dV_j = sum_{g,i} P_ij dO_i and dK_j = scale * sum_{g,i} dS_ij q_i. */
#pragma omp parallel for schedule(dynamic, 4)
    for (long r = 0; r < (long)nk; ++r) {
        int j = krows ? krows[r] : (int)r;
        double* dkr = dk + (size_t)r * d;
        double* dvr = dv + (size_t)r * d;
        for (int c = 0; c < d; ++c) {
            dkr[c] = 0.0;
            dvr[c] = 0.0;
        }
        const double* kj = k + (size_t)j * d;
        const double* vj = v + (size_t)j * d;
        for (int g = 0; g < G; ++g) {
            for (int i = 0; i < L; ++i) {
                int lo, hi;
                visible_range(i, L, causal, window, &lo, &hi);
                if (j < lo || j > hi) continue;
                size_t gi = (size_t)g * L + i;
                const double* qi = q + gi * d;
                const double* doi = dout + gi * d;
                double p = exp(scale * dot(qi, kj, d) - m[gi]) / l[gi];
                double dp = dot(doi, vj, d);
                double ds = p * (dp - D[gi]);
                for (int c = 0; c < d; ++c) {
                    dvr[c] += p * doi[c];
                    dkr[c] += scale * ds * qi[c];
                }
            }
        }
    }
    free(m);
    free(l);
    free(D);
    return 0;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int fa_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
