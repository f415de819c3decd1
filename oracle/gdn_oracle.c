/*
 * GDN forward oracle: the gated delta rule applied token by token in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow definition that the
 * CUDA path is checked against.  It shares no code, header or table with the
 * CUDA library, and the library never calls it.
 *
 * What it computes (FlashQLA talk "Qwen系列模型线性注意力高性能优化实践", the
 * recurrent-form paragraph and the GDN paragraph: the state is updated once per
 * token through an update gate beta and a forget gate alpha):
 *
 *     S_t = S_{t-1} * alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = scale * S_t q_t                   (post-update state)
 *     alpha_t = exp(g_t)
 *
 * with S in R^{dv x dk}.  Row i of S only involves row i of S_{t-1} and v_t[i]:
 *
 *     s_i <- alpha_t (s_i - beta_t (s_i . k_t) k_t) + beta_t v_t[i] k_t
 *
 * so the rows are computed independently (and in parallel over OpenMP threads),
 * which is exact, not an approximation.
 *
 * Layouts (token-major, packed varlen): q, k [total_T, H, dk]; v, o
 * [total_T, H, dv]; g, beta [total_T, H]; s0, s_final [N, H, dk, dv] with
 * s[n][h][j][i] = S[i][j] (the state stored k-major, v fastest).  cu[n] is the
 * first token of sequence n, cu[N] = total_T.  s0 may be NULL (zero state).
 *
 * `mutation` plants one deliberate mistake (0 = none).  It exists only so the
 * pin tests can show that each pin catches a plausible error in this code:
 *   1  sign of the delta-rule correction flipped (+beta k k^T)
 *   2  output taken from the pre-update state S_{t-1}
 *   3  forget gate applied after the update instead of before
 *   4  beta dropped from the value write (writes v k^T, corrects with beta)
 *   5  state read transposed in the key product (S^T k instead of S k)
 *   6  output scale dropped
 *   7  alpha = exp(-g) (sign of the log gate flipped)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int gdn_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int j = 0; j < n; ++j) s += a[j] * b[j];
    return s;
}

/* Returns 0 on success, 1 on bad arguments, 2 on allocation failure. */
int gdn_oracle_fwd(const double *q, const double *k, const double *v,
                   const double *g, const double *beta, const double *s0,
                   const int64_t *cu, int n_seqs, int H, int dk, int dv,
                   double scale, int row_block, int nthreads, int mutation,
                   double *o, double *s_final)
{
    if (n_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || row_block <= 0) return 1;
    if (mutation == 5 && dk != dv) return 1;
    for (int n = 0; n < n_seqs; ++n)
        if (cu[n + 1] < cu[n]) return 1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const int nb = (dv + row_block - 1) / row_block;
    const long ntask = (long)n_seqs * H * nb;
    int failed = 0;

#pragma omp parallel
    {
        /* one row block of the state, plus a full dv x dk copy for mutation 5 */
        double *s = (double *)malloc(sizeof(double) * (size_t)dv * dk);
        double *sk_rows = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!s || !sk_rows) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long task = 0; task < ntask; ++task) {
            if (failed) continue;
            const int n = (int)(task / ((long)H * nb));
            const int rem = (int)(task % ((long)H * nb));
            const int h = rem / nb;
            int i0 = (rem % nb) * row_block;
            int i1 = i0 + row_block < dv ? i0 + row_block : dv;
            if (mutation == 5) { /* needs every row of the state */
                if (rem % nb != 0) continue;
                i0 = 0;
                i1 = dv;
            }
            const int nr = i1 - i0;
            /* initial state rows */
            for (int i = i0; i < i1; ++i)
                for (int j = 0; j < dk; ++j)
                    s[(size_t)(i - i0) * dk + j] =
                        s0 ? s0[(((size_t)n * H + h) * dk + j) * dv + i] : 0.0;

            for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
                const double *kt = k + ((size_t)t * H + h) * dk;
                const double *qt = q + ((size_t)t * H + h) * dk;
                const double *vt = v + ((size_t)t * H + h) * dv;
                const double gt = g[(size_t)t * H + h];
                const double bt = beta[(size_t)t * H + h];
                const double alpha = exp(mutation == 7 ? -gt : gt);
                double *ot = o + ((size_t)t * H + h) * dv;

                if (mutation == 5) {
                    /* (S^T k)_i = sum_j S[j][i] k[j]  (dk == dv) */
                    for (int i = 0; i < nr; ++i) {
                        double acc = 0.0;
                        for (int j = 0; j < dk; ++j) acc += s[(size_t)j * dk + i] * kt[j];
                        sk_rows[i] = acc;
                    }
                }
                for (int i = 0; i < nr; ++i) {
                    double *si = s + (size_t)i * dk;
                    if (mutation == 2) ot[i0 + i] = scale * dot(si, qt, dk);
                    const double sk = mutation == 5 ? sk_rows[i] : dot(si, kt, dk);
                    const double vi = vt[i0 + i];
                    switch (mutation) {
                    case 1:
                        for (int j = 0; j < dk; ++j)
                            si[j] = alpha * (si[j] + bt * sk * kt[j]) + bt * vi * kt[j];
                        break;
                    case 3:
                        for (int j = 0; j < dk; ++j)
                            si[j] = alpha * ((si[j] - bt * sk * kt[j]) + bt * vi * kt[j]);
                        break;
                    case 4:
                        for (int j = 0; j < dk; ++j)
                            si[j] = alpha * (si[j] - bt * sk * kt[j]) + vi * kt[j];
                        break;
                    default:
                        for (int j = 0; j < dk; ++j)
                            si[j] = alpha * (si[j] - bt * sk * kt[j]) + bt * vi * kt[j];
                        break;
                    }
                    if (mutation != 2)
                        ot[i0 + i] = (mutation == 6 ? 1.0 : scale) * dot(si, qt, dk);
                }
            }
            for (int i = i0; i < i1; ++i)
                for (int j = 0; j < dk; ++j)
                    s_final[(((size_t)n * H + h) * dk + j) * dv + i] = s[(size_t)(i - i0) * dk + j];
        }
        free(s);
        free(sk_rows);
    }
    return failed ? 2 : 0;
}
