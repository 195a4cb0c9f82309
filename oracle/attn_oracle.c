/*
 * CPU oracle for exact softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this file's library.  It shares no code, header,
 * table or helper with the CUDA path and never imports it.
 *
 * Everything is plain double-precision loops, written for a reader to check
 * against the defining passages by eye:
 *
 *   "The I/O Complexity of Attention" exposition (blog.aeilot.top,
 *   attention-io-complexity), section "Attention as a mathematical problem":
 *   for one head, Q, K, V are N x d; the score of query i against key j is the
 *   dot product q_i . k_j; softmax turns each row of scores into weights; the
 *   output row is the weighted average of the value rows, O = softmax(QK^T) V.
 *   The page drops the usual 1/sqrt(d); here a caller-given scale s multiplies
 *   every score before the softmax (s = 1 recovers the page's form).
 *
 *   Same page, section "Softmax without storing the score matrix": the
 *   stabilised online update over key blocks J with running max m, running sum
 *   l and running weighted sum u; the output is u / l.  The page notes that the
 *   streaming form evaluates the same function and only the rounding differs.
 *
 *   "On Fine-Grained I/O Complexity of Attention Backward Passes" summary
 *   (gist.science 2410.09397), "Problem Statement": the backward pass of the
 *   same attention.  The page prints no gradient formulas; the ones below are
 *   the plain chain rule of the forward definition.
 *
 * Conventions shared with the callers (not with the CUDA path):
 *   - every array is [nh][N][d] (or [nh][N]) contiguous, nh independent heads;
 *   - mask, when non-NULL, is an nb x nb byte array, nb = ceil(N/128), row-major,
 *     shared by all heads; mask[i/128][j/128] == 0 removes score (i, j) (its
 *     weight is exactly zero, as if the score were minus infinity);
 *   - a row whose every score is removed gets O = 0 and LSE = -inf, and passes
 *     no gradient.
 *   - LSE is the natural log of sum_j exp(S_ij) over the scaled scores S = s QK^T.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MASK_BLOCK 128

/*
 * Block mask of one head: score (i, j) is kept when mask[i/block][j/block] != 0
 * (an nb x nb byte array, nb = ceil(N/block)).  The plain entry points use
 * block 128 and one mask for every head; the *_m entry points take the block
 * side and the byte distance between consecutive heads' masks (0 = shared).
 */
typedef struct {
    const uint8_t *mask;  /* NULL: keep everything */
    int block;
    int nb;
} mask_view;

static int keep_v(const mask_view *mv, int i, int j)
{
    if (mv->mask == NULL) return 1;
    return mv->mask[(size_t)(i / mv->block) * mv->nb + (j / mv->block)] != 0;
}

static mask_view head_mask(const uint8_t *mask, int block, long long head_stride, int h, int N)
{
    mask_view mv;
    mv.block = block;
    mv.nb = (N + block - 1) / block;
    mv.mask = mask ? mask + (size_t)h * (size_t)head_stride : NULL;
    return mv;
}

static int keep(const uint8_t *mask, int nb, int i, int j)
{
    if (mask == NULL) return 1;
    return mask[(size_t)(i / ORACLE_MASK_BLOCK) * nb + (j / ORACLE_MASK_BLOCK)] != 0;
}

static int num_blocks(int N) { return (N + ORACLE_MASK_BLOCK - 1) / ORACLE_MASK_BLOCK; }

static double dot(const double *a, const double *b, int d)
{
    double acc = 0.0;
    for (int t = 0; t < d; ++t) acc += a[t] * b[t];
    return acc;
}

/* One row of scaled scores S_i. = s * q_i . k_j; removed entries are -inf.
 * Returns the exact row maximum (-inf when every entry is removed). */
static double score_row(const double *Q, const double *K, int N, int d, double s,
                        const uint8_t *mask, int nb, int i, double *srow)
{
    double mx = -INFINITY;
    for (int j = 0; j < N; ++j) {
        if (keep(mask, nb, i, j)) {
            srow[j] = s * dot(Q + (size_t)i * d, K + (size_t)j * d, d);
            if (srow[j] > mx) mx = srow[j];
        } else {
            srow[j] = -INFINITY;
        }
    }
    return mx;
}

/* Natural-log partition function of one score row, with the exact max. */
static double row_lse(const double *srow, int N, double mx)
{
    if (mx == -INFINITY) return -INFINITY;
    double z = 0.0;
    for (int j = 0; j < N; ++j) z += exp(srow[j] - mx);
    return mx + log(z);
}

/*
 * Forward, full-row evaluation ("Attention as a mathematical problem"):
 * S_i. = s q_i K^T, LSE_i = log sum_j e^{S_ij}, P_ij = e^{S_ij - LSE_i},
 * o_i = sum_j P_ij v_j.
 */
static void fwd_row(const double *Q, const double *K, const double *V, int N, int d,
                    double s, const uint8_t *mask, int nb, int i, double *srow,
                    double *o, double *lse)
{
    double mx = score_row(Q, K, N, d, s, mask, nb, i, srow);
    double L = row_lse(srow, N, mx);
    for (int t = 0; t < d; ++t) o[t] = 0.0;
    *lse = L;
    if (L == -INFINITY) return;
    for (int j = 0; j < N; ++j) {
        if (srow[j] == -INFINITY) continue;
        double p = exp(srow[j] - L);
        const double *vj = V + (size_t)j * d;
        for (int t = 0; t < d; ++t) o[t] += p * vj[t];
    }
}

void oracle_fwd_naive(int nh, int N, int d, double s, const uint8_t *mask,
                      const double *Q, const double *K, const double *V,
                      double *O, double *LSE)
{
    int nb = num_blocks(N);
#pragma omp parallel
    {
        double *srow = (double *)malloc((size_t)N * sizeof(double));
#pragma omp for collapse(2) schedule(dynamic, 16)
        for (int h = 0; h < nh; ++h)
            for (int i = 0; i < N; ++i) {
                size_t hb = (size_t)h * N * d;
                fwd_row(Q + hb, K + hb, V + hb, N, d, s, mask, nb, i, srow,
                        O + hb + (size_t)i * d, LSE + (size_t)h * N + i);
            }
        free(srow);
    }
}

/*
 * Forward for chosen rows only: out row r is head heads[r], query rows[r].
 * Same arithmetic as oracle_fwd_naive; used to check single outputs at sizes
 * where the whole tensor would take too long.
 */
void oracle_fwd_rows(int N, int d, double s, const uint8_t *mask,
                     const double *Q, const double *K, const double *V,
                     int nrows, const int *heads, const int *rows,
                     double *O_out, double *LSE_out)
{
    int nb = num_blocks(N);
#pragma omp parallel
    {
        double *srow = (double *)malloc((size_t)N * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nrows; ++r) {
            size_t hb = (size_t)heads[r] * N * d;
            fwd_row(Q + hb, K + hb, V + hb, N, d, s, mask, nb, rows[r], srow,
                    O_out + (size_t)r * d, LSE_out + r);
        }
        free(srow);
    }
}

/*
 * Forward by the stabilised online update ("Softmax without storing the score
 * matrix").  Keys are visited in blocks J_0, J_1, ... whose end indices are
 * ends[0] < ends[1] < ... = N.  For each block:
 *   m' = max(m, max_{j in J} S_ij)
 *   l  <- e^{m - m'} l + sum_{j in J} e^{S_ij - m'}
 *   u  <- e^{m - m'} u + sum_{j in J} e^{S_ij - m'} v_j
 * and at the end o = u / l.  LSE = m + log l (natural log).
 */
void oracle_fwd_stream(int nh, int N, int d, double s, const uint8_t *mask,
                       int nblocks, const int *ends,
                       const double *Q, const double *K, const double *V,
                       double *O, double *LSE)
{
    int nb = num_blocks(N);
#pragma omp parallel
    {
        double *sblk = (double *)malloc((size_t)N * sizeof(double));
        double *u = (double *)malloc((size_t)d * sizeof(double));
#pragma omp for collapse(2) schedule(dynamic, 16)
        for (int h = 0; h < nh; ++h)
            for (int i = 0; i < N; ++i) {
                size_t hb = (size_t)h * N * d;
                const double *Qh = Q + hb, *Kh = K + hb, *Vh = V + hb;
                double m = -INFINITY, l = 0.0;
                for (int t = 0; t < d; ++t) u[t] = 0.0;
                int start = 0;
                for (int b = 0; b < nblocks; ++b) {
                    int end = ends[b];
                    double mb = -INFINITY;
                    for (int j = start; j < end; ++j) {
                        if (keep(mask, nb, i, j)) {
                            sblk[j] = s * dot(Qh + (size_t)i * d, Kh + (size_t)j * d, d);
                            if (sblk[j] > mb) mb = sblk[j];
                        } else {
                            sblk[j] = -INFINITY;
                        }
                    }
                    double mnew = m > mb ? m : mb;
                    if (mnew != -INFINITY) {
                        double alpha = (m == -INFINITY) ? 0.0 : exp(m - mnew);
                        l *= alpha;
                        for (int t = 0; t < d; ++t) u[t] *= alpha;
                        for (int j = start; j < end; ++j) {
                            if (sblk[j] == -INFINITY) continue;
                            double p = exp(sblk[j] - mnew);
                            l += p;
                            const double *vj = Vh + (size_t)j * d;
                            for (int t = 0; t < d; ++t) u[t] += p * vj[t];
                        }
                        m = mnew;
                    }
                    start = end;
                }
                double *o = O + hb + (size_t)i * d;
                if (l > 0.0) {
                    for (int t = 0; t < d; ++t) o[t] = u[t] / l;
                    LSE[(size_t)h * N + i] = m + log(l);
                } else {
                    for (int t = 0; t < d; ++t) o[t] = 0.0;
                    LSE[(size_t)h * N + i] = -INFINITY;
                }
            }
        free(sblk);
        free(u);
    }
}

/*
 * Row quantities of the backward pass for query row i of one head:
 *   P_i. = e^{S_i. - LSE_i}   (LSE with the exact row max, as in the forward)
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_j P_ij dP_ij
 * prow/dprow receive P_i. and dP_i.; returns D_i and stores LSE_i.
 */
static double bwd_row(const double *Q, const double *K, const double *V, const double *dO,
                      int N, int d, double s, const uint8_t *mask, int nb, int i,
                      double *prow, double *dprow, double *lse_out)
{
    double mx = score_row(Q, K, N, d, s, mask, nb, i, prow);
    double L = row_lse(prow, N, mx);
    *lse_out = L;
    double D = 0.0;
    for (int j = 0; j < N; ++j) {
        if (L == -INFINITY || prow[j] == -INFINITY) {
            prow[j] = 0.0;
            dprow[j] = 0.0;
            continue;
        }
        prow[j] = exp(prow[j] - L);
        dprow[j] = dot(dO + (size_t)i * d, V + (size_t)j * d, d);
        D += prow[j] * dprow[j];
    }
    return D;
}

/*
 * Backward by the chain rule of O = softmax(s QK^T) V with upstream gradient dO:
 *   dV = P^T dO
 *   dP = dO V^T
 *   D_i = sum_j P_ij dP_ij
 *   dS = P o (dP - D 1^T)          (o: elementwise product)
 *   dQ = s dS K,   dK = s dS^T Q
 * Pass 1 walks query rows (LSE_i, D_i, dQ_i); pass 2 walks key rows (dK_j, dV_j),
 * recomputing P_ij and dS_ij from the stored LSE and D.  D and LSE are written
 * out when the pointers are non-NULL.
 */
void oracle_bwd_naive(int nh, int N, int d, double s, const uint8_t *mask,
                      const double *Q, const double *K, const double *V, const double *dO,
                      double *dQ, double *dK, double *dV, double *D_out, double *LSE_out)
{
    int nb = num_blocks(N);
    double *Dall = (double *)malloc((size_t)nh * N * sizeof(double));
    double *Lall = (double *)malloc((size_t)nh * N * sizeof(double));
#pragma omp parallel
    {
        double *prow = (double *)malloc((size_t)N * sizeof(double));
        double *dprow = (double *)malloc((size_t)N * sizeof(double));
#pragma omp for collapse(2) schedule(dynamic, 16)
        for (int h = 0; h < nh; ++h)
            for (int i = 0; i < N; ++i) {
                size_t hb = (size_t)h * N * d;
                const double *Qh = Q + hb, *Kh = K + hb, *Vh = V + hb, *dOh = dO + hb;
                double L;
                double D = bwd_row(Qh, Kh, Vh, dOh, N, d, s, mask, nb, i, prow, dprow, &L);
                Dall[(size_t)h * N + i] = D;
                Lall[(size_t)h * N + i] = L;
                double *dq = dQ + hb + (size_t)i * d;
                for (int t = 0; t < d; ++t) dq[t] = 0.0;
                for (int j = 0; j < N; ++j) {
                    double dS = prow[j] * (dprow[j] - D);
                    if (dS == 0.0) continue;
                    const double *kj = Kh + (size_t)j * d;
                    for (int t = 0; t < d; ++t) dq[t] += s * dS * kj[t];
                }
            }
#pragma omp for collapse(2) schedule(dynamic, 16)
        for (int h = 0; h < nh; ++h)
            for (int j = 0; j < N; ++j) {
                size_t hb = (size_t)h * N * d;
                const double *Qh = Q + hb, *Kh = K + hb, *Vh = V + hb, *dOh = dO + hb;
                double *dk = dK + hb + (size_t)j * d, *dv = dV + hb + (size_t)j * d;
                for (int t = 0; t < d; ++t) { dk[t] = 0.0; dv[t] = 0.0; }
                for (int i = 0; i < N; ++i) {
                    double L = Lall[(size_t)h * N + i];
                    if (L == -INFINITY || !keep(mask, nb, i, j)) continue;
                    double P = exp(s * dot(Qh + (size_t)i * d, Kh + (size_t)j * d, d) - L);
                    double dP = dot(dOh + (size_t)i * d, Vh + (size_t)j * d, d);
                    double dS = P * (dP - Dall[(size_t)h * N + i]);
                    const double *qi = Qh + (size_t)i * d, *doi = dOh + (size_t)i * d;
                    for (int t = 0; t < d; ++t) {
                        dv[t] += P * doi[t];
                        dk[t] += s * dS * qi[t];
                    }
                }
            }
        free(prow);
        free(dprow);
    }
    if (D_out) memcpy(D_out, Dall, (size_t)nh * N * sizeof(double));
    if (LSE_out) memcpy(LSE_out, Lall, (size_t)nh * N * sizeof(double));
    free(Dall);
    free(Lall);
}

/*
 * Backward for chosen outputs of one head (head offset already applied by the
 * caller): dQ for the query rows qrows[], and dK, dV for the key rows krows[].
 * dQ_i needs only row i; dK_j and dV_j need LSE_i and D_i of every row, so the
 * per-row pass runs over all N rows first.  Same arithmetic as oracle_bwd_naive.
 */
void oracle_bwd_rows(int N, int d, double s, const uint8_t *mask,
                     const double *Q, const double *K, const double *V, const double *dO,
                     int nq, const int *qrows, double *dQ_out,
                     int nk, const int *krows, double *dK_out, double *dV_out)
{
    int nb = num_blocks(N);
    double *Dall = (double *)malloc((size_t)N * sizeof(double));
    double *Lall = (double *)malloc((size_t)N * sizeof(double));
#pragma omp parallel
    {
        double *prow = (double *)malloc((size_t)N * sizeof(double));
        double *dprow = (double *)malloc((size_t)N * sizeof(double));
        int need_all = nk > 0;
#pragma omp for schedule(dynamic, 16)
        for (int i = 0; i < (need_all ? N : 0); ++i)
            Dall[i] = bwd_row(Q, K, V, dO, N, d, s, mask, nb, i, prow, dprow, &Lall[i]);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nq; ++r) {
            int i = qrows[r];
            double L;
            double D = bwd_row(Q, K, V, dO, N, d, s, mask, nb, i, prow, dprow, &L);
            double *dq = dQ_out + (size_t)r * d;
            for (int t = 0; t < d; ++t) dq[t] = 0.0;
            for (int j = 0; j < N; ++j) {
                double dS = prow[j] * (dprow[j] - D);
                if (dS == 0.0) continue;
                for (int t = 0; t < d; ++t) dq[t] += s * dS * K[(size_t)j * d + t];
            }
        }
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nk; ++r) {
            int j = krows[r];
            double *dk = dK_out + (size_t)r * d, *dv = dV_out + (size_t)r * d;
            for (int t = 0; t < d; ++t) { dk[t] = 0.0; dv[t] = 0.0; }
            for (int i = 0; i < N; ++i) {
                if (Lall[i] == -INFINITY || !keep(mask, nb, i, j)) continue;
                double P = exp(s * dot(Q + (size_t)i * d, K + (size_t)j * d, d) - Lall[i]);
                double dP = dot(dO + (size_t)i * d, V + (size_t)j * d, d);
                double dS = P * (dP - Dall[i]);
                for (int t = 0; t < d; ++t) {
                    dv[t] += P * dO[(size_t)i * d + t];
                    dk[t] += s * dS * Q[(size_t)i * d + t];
                }
            }
        }
        free(prow);
        free(dprow);
    }
    free(Dall);
    free(Lall);
}

/*
 * Rectangular forward: Nq queries against Nk keys per head, no mask
 * ("The I/O Complexity of Attention" exposition, end of "From a movement lower
 * bound to a performance upper bound": single-token decoding has query length
 * one and needs a rectangular account).  Same definition as the square case:
 * S_i. = s q_i K^T over the Nk keys, LSE_i = log sum_j e^{S_ij} with the exact
 * row max, o_i = sum_j e^{S_ij - LSE_i} v_j.
 * Q, O: [nh][Nq][d]; K, V: [nh][Nk][d]; LSE: [nh][Nq].
 */
void oracle_fwd_rect(int nh, int Nq, int Nk, int d, double s,
                     const double *Q, const double *K, const double *V,
                     double *O, double *LSE)
{
#pragma omp parallel
    {
        double *srow = (double *)malloc((size_t)Nk * sizeof(double));
#pragma omp for collapse(2) schedule(dynamic, 1)
        for (int h = 0; h < nh; ++h)
            for (int i = 0; i < Nq; ++i) {
                const double *q = Q + ((size_t)h * Nq + i) * d;
                const double *Kh = K + (size_t)h * Nk * d, *Vh = V + (size_t)h * Nk * d;
                double *o = O + ((size_t)h * Nq + i) * d;
                double mx = -INFINITY;
                for (int j = 0; j < Nk; ++j) {
                    srow[j] = s * dot(q, Kh + (size_t)j * d, d);
                    if (srow[j] > mx) mx = srow[j];
                }
                double L = row_lse(srow, Nk, mx);
                LSE[(size_t)h * Nq + i] = L;
                for (int t = 0; t < d; ++t) o[t] = 0.0;
                for (int j = 0; j < Nk; ++j) {
                    double p = exp(srow[j] - L);
                    const double *vj = Vh + (size_t)j * d;
                    for (int t = 0; t < d; ++t) o[t] += p * vj[t];
                }
            }
        free(srow);
    }
}

/*
 * Forward and backward with a general block mask (block side `block`, per-head
 * masks `head_stride` bytes apart).  Same definitions as oracle_fwd_naive and
 * oracle_bwd_naive; only the lookup of removed scores differs.
 */
static double score_row_m(const double *Q, const double *K, int N, int d, double s, const mask_view *mv, int i,
                          double *srow)
{
    double mx = -INFINITY;
    for (int j = 0; j < N; ++j) {
        if (keep_v(mv, i, j)) {
            srow[j] = s * dot(Q + (size_t)i * d, K + (size_t)j * d, d);
            if (srow[j] > mx) mx = srow[j];
        } else {
            srow[j] = -INFINITY;
        }
    }
    return mx;
}

void oracle_fwd_naive_m(int nh, int N, int d, double s, const uint8_t *mask, int block, long long head_stride,
                        const double *Q, const double *K, const double *V, double *O, double *LSE)
{
#pragma omp parallel
    {
        double *srow = (double *)malloc((size_t)N * sizeof(double));
#pragma omp for collapse(2) schedule(dynamic, 16)
        for (int h = 0; h < nh; ++h)
            for (int i = 0; i < N; ++i) {
                size_t hb = (size_t)h * N * d;
                mask_view mv = head_mask(mask, block, head_stride, h, N);
                double mx = score_row_m(Q + hb, K + hb, N, d, s, &mv, i, srow);
                double L = row_lse(srow, N, mx);
                double *o = O + hb + (size_t)i * d;
                for (int t = 0; t < d; ++t) o[t] = 0.0;
                LSE[(size_t)h * N + i] = L;
                if (L == -INFINITY) continue;
                for (int j = 0; j < N; ++j) {
                    if (srow[j] == -INFINITY) continue;
                    double p = exp(srow[j] - L);
                    const double *vj = V + hb + (size_t)j * d;
                    for (int t = 0; t < d; ++t) o[t] += p * vj[t];
                }
            }
        free(srow);
    }
}

void oracle_bwd_naive_m(int nh, int N, int d, double s, const uint8_t *mask, int block, long long head_stride,
                        const double *Q, const double *K, const double *V, const double *dO,
                        double *dQ, double *dK, double *dV)
{
    double *Dall = (double *)malloc((size_t)nh * N * sizeof(double));
    double *Lall = (double *)malloc((size_t)nh * N * sizeof(double));
#pragma omp parallel
    {
        double *prow = (double *)malloc((size_t)N * sizeof(double));
#pragma omp for collapse(2) schedule(dynamic, 16)
        for (int h = 0; h < nh; ++h)
            for (int i = 0; i < N; ++i) {
                size_t hb = (size_t)h * N * d;
                const double *Qh = Q + hb, *Kh = K + hb, *Vh = V + hb, *dOh = dO + hb;
                mask_view mv = head_mask(mask, block, head_stride, h, N);
                double mx = score_row_m(Qh, Kh, N, d, s, &mv, i, prow);
                double L = row_lse(prow, N, mx);
                double D = 0.0;
                double *dq = dQ + hb + (size_t)i * d;
                for (int t = 0; t < d; ++t) dq[t] = 0.0;
                Lall[(size_t)h * N + i] = L;
                if (L == -INFINITY) {
                    Dall[(size_t)h * N + i] = 0.0;
                    continue;
                }
                /* D_i = sum_j P_ij dP_ij */
                for (int j = 0; j < N; ++j) {
                    if (prow[j] == -INFINITY) continue;
                    D += exp(prow[j] - L) * dot(dOh + (size_t)i * d, Vh + (size_t)j * d, d);
                }
                Dall[(size_t)h * N + i] = D;
                for (int j = 0; j < N; ++j) {
                    if (prow[j] == -INFINITY) continue;
                    double P = exp(prow[j] - L);
                    double dS = P * (dot(dOh + (size_t)i * d, Vh + (size_t)j * d, d) - D);
                    for (int t = 0; t < d; ++t) dq[t] += s * dS * Kh[(size_t)j * d + t];
                }
            }
#pragma omp for collapse(2) schedule(dynamic, 16)
        for (int h = 0; h < nh; ++h)
            for (int j = 0; j < N; ++j) {
                size_t hb = (size_t)h * N * d;
                const double *Qh = Q + hb, *Kh = K + hb, *Vh = V + hb, *dOh = dO + hb;
                mask_view mv = head_mask(mask, block, head_stride, h, N);
                double *dk = dK + hb + (size_t)j * d, *dv = dV + hb + (size_t)j * d;
                for (int t = 0; t < d; ++t) { dk[t] = 0.0; dv[t] = 0.0; }
                for (int i = 0; i < N; ++i) {
                    double L = Lall[(size_t)h * N + i];
                    if (L == -INFINITY || !keep_v(&mv, i, j)) continue;
                    double P = exp(s * dot(Qh + (size_t)i * d, Kh + (size_t)j * d, d) - L);
                    double dS = P * (dot(dOh + (size_t)i * d, Vh + (size_t)j * d, d) - Dall[(size_t)h * N + i]);
                    for (int t = 0; t < d; ++t) {
                        dv[t] += P * dOh[(size_t)i * d + t];
                        dk[t] += s * dS * Qh[(size_t)i * d + t];
                    }
                }
            }
        free(prow);
    }
    free(Dall);
    free(Lall);
}

/* Number of OpenMP threads the oracle runs with (for reporting). */
int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
