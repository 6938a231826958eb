/*
 * FP64 CPU oracle for the scaled dot-product attention forward pass
 * (head dimension 256 on the pages; any D here).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * execute this file; only the test suite, the smoke check and the CPU legs
 * of the benchmark use it.  It shares no code, header, table or helper with
 * the CUDA path.
 *
 * What it computes: the "Xe2 Nbarrier Pipelining" page ("Proven Pattern:
 * SDP Kernel Split Barrier B") describes a flash-attention kernel for head
 * dimension 256: per block of keys it forms S = Q K^T, a softmax with a
 * running row maximum, a running row sum ("sum update") and a rescale of
 * the partial output ("compensation"), then accumulates P V.  That
 * streaming algorithm reaches, up to rounding, the plain definition of
 * attention, which is what this oracle writes out:
 *
 *     s_j  = scale * sum_{d=0}^{D-1} q_d * k_jd          (j = 0 .. Skv-1)
 *     m    = max_j s_j
 *     w_j  = exp(s_j - m)
 *     l    = sum_j w_j
 *     o_d  = (sum_j w_j * v_jd) / l
 *
 * for every batch b, head h and query row i, over the binary16 inputs
 * widened exactly to binary64.  Subtracting m changes nothing in exact
 * arithmetic (softmax is invariant to a common shift of its arguments) and
 * keeps exp() finite for large scores.  Sums run in increasing index order
 * from +0.0; there is no blocking and no streaming over key blocks.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/*
 * Q, K, V: binary64 arrays addressed as X[b*xs[0] + h*xs[1] + row*xs[2] + d]
 * (element strides for batch, head and row; d contiguous).
 * rows: the query rows to compute (nrows of them), or NULL for all Sq.
 * O: contiguous [B][H][nrows][D] (nrows = Sq when rows is NULL).
 * Returns 0, or -1 if scratch memory could not be allocated.
 */
int oracle_attention_f64(int64_t B, int64_t H, int64_t Sq, int64_t Skv, int64_t D,
                         const double *Q, const int64_t *qs,
                         const double *K, const int64_t *ks,
                         const double *V, const int64_t *vs,
                         double scale, const int64_t *rows, int64_t nrows,
                         double *O)
{
    const int64_t nr = rows ? nrows : Sq;
    const int64_t total = B * H * nr;
    int failed = 0;
    int64_t t;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : failed)
    for (t = 0; t < total; ++t) {
        const int64_t b = t / (H * nr);
        const int64_t h = (t / nr) % H;
        const int64_t r = t % nr;
        const int64_t i = rows ? rows[r] : r;
        const double *q = Q + b * qs[0] + h * qs[1] + i * qs[2];
        double *o = O + t * D;
        double *w = (double *)malloc((size_t)(Skv > 0 ? Skv : 1) * sizeof(double));
        if (!w) {
            failed = 1;
            continue;
        }
        /* scores */
        for (int64_t j = 0; j < Skv; ++j) {
            const double *k = K + b * ks[0] + h * ks[1] + j * ks[2];
            double s = 0.0;
            for (int64_t d = 0; d < D; ++d)
                s += q[d] * k[d];
            w[j] = scale * s;
        }
        /* softmax weights */
        double m = -INFINITY;
        for (int64_t j = 0; j < Skv; ++j)
            if (w[j] > m)
                m = w[j];
        double l = 0.0;
        for (int64_t j = 0; j < Skv; ++j) {
            w[j] = exp(w[j] - m);
            l += w[j];
        }
        /* weighted sum of value rows */
        for (int64_t d = 0; d < D; ++d)
            o[d] = 0.0;
        for (int64_t j = 0; j < Skv; ++j) {
            const double *v = V + b * vs[0] + h * vs[1] + j * vs[2];
            for (int64_t d = 0; d < D; ++d)
                o[d] += w[j] * v[d];
        }
        for (int64_t d = 0; d < D; ++d)
            o[d] /= l;
        free(w);
    }
    return failed ? -1 : 0;
}
