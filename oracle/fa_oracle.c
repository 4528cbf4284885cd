/*
 * fa_oracle.c -- plain, slow, fp64 CPU oracle for exact attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header or constant
 * with the CUDA kernels.
 *
 * What it computes (all arithmetic in fp64, on the 16-bit input values
 * upcast exactly by the caller):
 *
 *   Exact attention, "flash-attn-triton" docs page, section "The argument"
 *   (ordinary attention: S = Q K^T / sqrt(d), softmax by rows, P V) and the
 *   FlashAttention note (narrativegoldmine), section "Key Mechanisms"
 *   (causal = lower-triangular mask).  With a caller-given scale:
 *       S_ij = scale * <q_i, k_j>,  j allowed iff (!causal || j <= i)
 *       m_i  = max_j S_ij,  l_i = sum_j exp(S_ij - m_i)
 *       P_ij = exp(S_ij - m_i) / l_i,  O_i = sum_j P_ij v_j
 *       L_i  = m_i + ln(l_i)        (natural-log logsumexp of scaled scores)
 *   Sliding window (window W > 0, causal only): key j is allowed for query i
 *   iff i - W < j <= i, the W most recent keys.  The docs page lists sliding
 *   windows among the features its kernels do not have yet ("Scope") and
 *   defines no convention; this causal band is the plain reading.
 *   A row with no allowed key (never produced by square causal masks) gets
 *   O_i = 0 and L_i = -inf: the tutorial page ("Start with a safe softmax")
 *   asks for fully masked rows to be handled but fixes no convention.
 *
 *   Backward: the docs page, section "Scope", says the backward rebuilds P
 *   from the saved L; the pages print no gradient formulas.  The oracle uses
 *   the plain chain rule of the definition above with upstream gradient dO:
 *       dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,
 *       dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
 *   (Pinned by finite differences in the tests.)
 *
 *   A separate, naive online-softmax oracle follows the per-tile update of
 *   the docs page, section "Tiling softmax is exact algebra", Fig. 3
 *   (running max m, running sum l, correction alpha = exp(m_old - m_new)
 *   applied to l and acc together, one divide after the loop), in base e or
 *   in base 2 with log2(e) folded into the scale.  A partial-state merge
 *   (tutorial page, "Softmax in pieces": merging two partial results) is
 *   exposed for the merge pins.
 *
 * Layout: Q, K, V, O, dO, dQ, dK, dV are dense row-major (B, H, N, d) fp64;
 * L and D are (B, H, N) fp64.  Heads and rows are independent: OpenMP runs over
 * (batch*head, query row) pairs, and for dK/dV over (batch*head, key row) pairs,
 * each output row written by exactly one thread.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double dot(const double* a, const double* b, int d)
{
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

static int n_allowed(int i, int N, int causal) { return causal ? (i + 1 < N ? i + 1 : N) : N; }
/* first allowed key of row i under a window of W keys (0: no window) */
static int win_start(int i, int window) { return (window > 0 && i - window + 1 > 0) ? i - window + 1 : 0; }

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Scores of row i against its allowed keys, then the softmax statistics.
 * s[0..nk) receives S_ij; returns m, writes l.  nk == 0 -> m = -inf, l = 0. */
static double row_scores(const double* qi, const double* k, int nk, int d, double scale,
                         double* s, double* l_out)
{
    double m = -INFINITY;
    for (int j = 0; j < nk; ++j) {
        s[j] = scale * dot(qi, k + (long)j * d, d);
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int j = 0; j < nk; ++j) l += exp(s[j] - m);
    *l_out = l;
    return m;
}

void oracle_fwd(const double* Q, const double* K, const double* V, double* O, double* L,
                int B, int H, int N, int d, int causal, double scale, int window)
{
    long BH = (long)B * H;
    /* every (batch, head, row) is independent */
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
#pragma omp for collapse(2) schedule(dynamic, 16)
        for (long bh = 0; bh < BH; ++bh) {
            for (int i = 0; i < N; ++i) {
                const double* q = Q + bh * N * d;
                const double* k = K + bh * N * d;
                const double* v = V + bh * N * d;
                double* o = O + bh * N * d;
                double* lse = L + bh * N;
                int j0 = win_start(i, window);
                int nk = n_allowed(i, N, causal) - j0;   /* keys j0 .. j0 + nk - 1 */
                double l;
                double m = row_scores(q + (long)i * d, k + (long)j0 * d, nk, d, scale, s, &l);
                double* oi = o + (long)i * d;
                for (int c = 0; c < d; ++c) oi[c] = 0.0;
                if (nk == 0) { lse[i] = -INFINITY; continue; }
                for (int j = 0; j < nk; ++j) {
                    double p = exp(s[j] - m) / l;
                    const double* vj = v + (long)(j0 + j) * d;
                    for (int c = 0; c < d; ++c) oi[c] += p * vj[c];
                }
                lse[i] = m + log(l);
            }
        }
        free(s);
    }
}

/* Backward in two passes over the same definition.
 * Pass 1, one query row i at a time: S_i., the softmax statistics (kept as the
 * logsumexp L_i), P_i., O_i, D_i = dO_i . O_i, dP_i. = dO_i V^T, dS_i., and
 * dQ_i = scale sum_j dS_ij k_j.
 * Pass 2, one key row j at a time: for every query i allowed to see key j,
 * P_ij = exp(S_ij - L_i), dP_ij = dO_i . v_j, dS_ij = P_ij (dP_ij - D_i);
 * dK_j = scale sum_i dS_ij q_i and dV_j = sum_i P_ij dO_i. */
void oracle_bwd(const double* Q, const double* K, const double* V, const double* dO,
                double* dQ, double* dK, double* dV, double* Dout,
                int B, int H, int N, int d, int causal, double scale, int window)
{
    long BH = (long)B * H;
    double* Lrow = (double*)malloc(sizeof(double) * (BH * N > 0 ? BH * N : 1));
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (N > 0 ? N : 1));
        double* oi = (double*)malloc(sizeof(double) * (d > 0 ? d : 1));
#pragma omp for collapse(2) schedule(dynamic, 16)
        for (long bh = 0; bh < BH; ++bh) {
            for (int i = 0; i < N; ++i) {
                const double* q = Q + bh * N * d;
                const double* k = K + bh * N * d;
                const double* v = V + bh * N * d;
                const double* dout = dO + bh * N * d;
                int j0 = win_start(i, window);
                int nk = n_allowed(i, N, causal) - j0;   /* keys j0 .. j0 + nk - 1 */
                const double* qi = q + (long)i * d;
                const double* doi = dout + (long)i * d;
                double* dqi = dQ + bh * N * d + (long)i * d;
                for (int c = 0; c < d; ++c) { dqi[c] = 0.0; oi[c] = 0.0; }
                if (nk == 0) { Dout[bh * N + i] = 0.0; Lrow[bh * N + i] = -INFINITY; continue; }
                double l;
                double m = row_scores(qi, k + (long)j0 * d, nk, d, scale, s, &l);
                Lrow[bh * N + i] = m + log(l);
                /* s[j] <- P_i,j0+j, and O_i = sum_j P_ij v_j */
                for (int j = 0; j < nk; ++j) {
                    s[j] = exp(s[j] - m) / l;
                    const double* vj = v + (long)(j0 + j) * d;
                    for (int c = 0; c < d; ++c) oi[c] += s[j] * vj[c];
                }
                double Di = dot(doi, oi, d);
                Dout[bh * N + i] = Di;
                for (int j = 0; j < nk; ++j) {
                    double dpij = dot(doi, v + (long)(j0 + j) * d, d);
                    double dsij = s[j] * (dpij - Di);
                    const double* kj = k + (long)(j0 + j) * d;
                    for (int c = 0; c < d; ++c) dqi[c] += scale * dsij * kj[c];
                }
            }
        }
        free(oi);
        free(s);
    }
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
    for (long bh = 0; bh < BH; ++bh) {
        for (int j = 0; j < N; ++j) {
            const double* q = Q + bh * N * d;
            const double* k = K + bh * N * d;
            const double* v = V + bh * N * d;
            const double* dout = dO + bh * N * d;
            const double* kj = k + (long)j * d;
            const double* vj = v + (long)j * d;
            double* dkj = dK + bh * N * d + (long)j * d;
            double* dvj = dV + bh * N * d + (long)j * d;
            for (int c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
            for (int i = causal ? j : 0; i < N; ++i) {
                if (window > 0 && i - j >= window) break;   /* key j left row i's window */
                const double* qi = q + (long)i * d;
                const double* doi = dout + (long)i * d;
                double pij = exp(scale * dot(qi, kj, d) - Lrow[bh * N + i]);
                double dpij = dot(doi, vj, d);
                double dsij = pij * (dpij - Dout[bh * N + i]);
                for (int c = 0; c < d; ++c) {
                    dkj[c] += scale * dsij * qi[c];
                    dvj[c] += pij * doi[c];
                }
            }
        }
    }
    free(Lrow);
}

/* ---- naive online-softmax oracle (Fig. 3 of the docs page) -------------- */

/* Partial state of one query row over keys [j0, j1): running max m, running
 * sum l of exp(s - m) and the undivided output acc (length d).  base2 != 0
 * works in base 2 with the scale already multiplied by log2(e), as the docs
 * page's Fig. 3 does; m is then in the log2 domain.  Tiles of size T walk the
 * range in order.  Returns m; l and acc are written. */
double oracle_row_partial(const double* qi, const double* K, const double* V, int d,
                          int i, int j0, int j1, int causal, double scale, int T, int base2,
                          double* l_out, double* acc)
{
    const double log2e = 1.4426950408889634073599246810019;
    double c = base2 ? scale * log2e : scale;
    double m = -INFINITY, l = 0.0;
    for (int t = 0; t < d; ++t) acc[t] = 0.0;
    if (T < 1) T = 1;
    double* s = (double*)malloc(sizeof(double) * T);
    for (int t0 = j0; t0 < j1; t0 += T) {
        int t1 = t0 + T < j1 ? t0 + T : j1;
        double mt = -INFINITY;
        for (int j = t0; j < t1; ++j) {
            int masked = causal && j > i;
            s[j - t0] = masked ? -INFINITY : c * dot(qi, K + (long)j * d, d);
            if (s[j - t0] > mt) mt = s[j - t0];
        }
        double m_new = mt > m ? mt : m;
        if (m_new == -INFINITY) continue;       /* nothing allowed seen yet */
        double alpha = base2 ? exp2(m - m_new) : exp(m - m_new);   /* m = -inf -> 0 */
        double psum = 0.0;
        for (int t = 0; t < d; ++t) acc[t] *= alpha;
        for (int j = t0; j < t1; ++j) {
            double p = base2 ? exp2(s[j - t0] - m_new) : exp(s[j - t0] - m_new);
            psum += p;
            if (p != 0.0) {
                const double* vj = V + (long)j * d;
                for (int t = 0; t < d; ++t) acc[t] += p * vj[t];
            }
        }
        l = l * alpha + psum;
        m = m_new;
    }
    free(s);
    *l_out = l;
    return m;
}

/* Merge two partial states of the same row (same domain).  exp(-inf - (-inf))
 * is taken as 0 so that an empty partial merges as the identity. */
double oracle_merge(double m1, double l1, const double* acc1,
                    double m2, double l2, const double* acc2,
                    int d, int base2, double* l_out, double* acc_out)
{
    double m = m1 > m2 ? m1 : m2;
    double a1, a2;
    if (m == -INFINITY) { a1 = 0.0; a2 = 0.0; }
    else {
        a1 = base2 ? exp2(m1 - m) : exp(m1 - m);
        a2 = base2 ? exp2(m2 - m) : exp(m2 - m);
    }
    for (int t = 0; t < d; ++t) acc_out[t] = a1 * acc1[t] + a2 * acc2[t];
    *l_out = a1 * l1 + a2 * l2;
    return m;
}

/* Whole forward by the online update with key tiles of size T (T need not
 * divide N).  Finishes with one divide per row and L = m + ln(l) (base e), or
 * L = (m + log2(l)) * ln(2) when the state is in base 2, so that L is the
 * natural-log logsumexp in both cases. */
void oracle_fwd_online(const double* Q, const double* K, const double* V, double* O, double* L,
                       int B, int H, int N, int d, int causal, double scale, int T, int base2)
{
    const double ln2 = 0.69314718055994530941723212145818;
    long BH = (long)B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < BH; ++bh) {
        const double* q = Q + bh * N * d;
        const double* k = K + bh * N * d;
        const double* v = V + bh * N * d;
        double* o = O + bh * N * d;
        double* lse = L + bh * N;
        for (int i = 0; i < N; ++i) {
            double l;
            double* oi = o + (long)i * d;
            double m = oracle_row_partial(q + (long)i * d, k, v, d, i, 0, N, causal, scale, T,
                                          base2, &l, oi);
            if (l == 0.0) {
                for (int t = 0; t < d; ++t) oi[t] = 0.0;
                lse[i] = -INFINITY;
                continue;
            }
            for (int t = 0; t < d; ++t) oi[t] /= l;
            lse[i] = base2 ? (m + log2(l)) * ln2 : m + log(l);
        }
    }
}
