/*
 * tt_oracle.c -- float64 CPU oracle of the TT-EmbeddingBag hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code with the CUDA library.
 *
 * What it computes (TT-Rec / FBTT-Embedding pages):
 *   - the table of E rows and D = q1 q2 q3 columns is held as three TT cores
 *     G_k of shape [p_k][r_{k-1}][q_k][r_k], r_0 = r_3 = 1 (FBTT README,
 *     "Initialization": cores of size r_{k-1} x p_k x q_k x r_k; the slice
 *     index is moved first so that one slice is contiguous);
 *   - row i is the chain product of the slices G1[i1] G2[i2] G3[i3] with
 *     i = i1 p2 p3 + i2 p3 + i3 (FBTT README, "Software Cache": a row is
 *     computed from the cores by two consecutive matrix products), and column
 *     j = j1 q2 q3 + j2 q3 + j3 of the row is
 *        W[i][j] = sum_{a<r1} sum_{c<r2} G1[i1][0][j1][a] G2[i2][a][j2][c]
 *                                       G3[i3][c][j3][0];
 *   - bags are pooled like PyTorch's EmbeddingBag (FBTT README, opening
 *     paragraph; tensorflow/addons issue "EmbeddingBag and Product-Key Memory
 *     Layers": a gather followed by a weighted sum, never materialised):
 *        out[g] = sum_{n in bag g} s_n W[idx_n],  s_n = w_n (sum) or
 *        w_n / L_g (mean), w_n = 1 without per-sample weights, an empty bag
 *        gives a zero row;
 *   - the backward pass gives, for L = sum_g <out[g], grad_out[g]>, the
 *     gradient of every core element (FBTT README, "Software Cache": the
 *     gradient of each core is a chain of products in reversed order; here
 *     it is the definition written out):
 *        dG1[i1][0][j1][a] = sum_n sum_{j2,j3,c} g_n[j] G2[i2][a][j2][c] G3[i3][c][j3][0]
 *        dG2[i2][a][j2][c] = sum_n sum_{j1,j3}   g_n[j] G1[i1][0][j1][a] G3[i3][c][j3][0]
 *        dG3[i3][c][j3][0] = sum_n sum_{j1,j2,a} g_n[j] G1[i1][0][j1][a] G2[i2][a][j2][c]
 *     with g_n = s_n grad_out[bag(n)], each sum over the lookups n whose
 *     decoded slice index matches.
 *
 * Everything runs per lookup in the plain order: no de-duplication, no
 * sorting, no blocking.  Threads split only independent outputs (bags in the
 * forward pass, slices in the backward pass); each output is summed in the
 * same order whatever the thread count.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int64_t E;        /* number of rows */
    int64_t p[3];     /* row factorisation, p1 p2 p3 >= E */
    int64_t q[3];     /* column factorisation, q1 q2 q3 = D */
    int64_t r[2];     /* inner ranks r1, r2 */
    const double* G[3]; /* cores, [p_k][r_{k-1}][q_k][r_k] */
} tto_table;

enum { TTO_OK = 0, TTO_ERR_INDEX = 1, TTO_ERR_ARG = 2 };

int tto_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Mixed-radix decode of row i: i = i1 p2 p3 + i2 p3 + i3. */
static int decode_row(const tto_table* t, int64_t i, int64_t* i1, int64_t* i2, int64_t* i3) {
    if (i < 0 || i >= t->E) return TTO_ERR_INDEX;
    *i1 = i / (t->p[1] * t->p[2]);
    *i2 = (i / t->p[2]) % t->p[1];
    *i3 = i % t->p[2];
    return TTO_OK;
}

/* Bag of every lookup and the decoded slice indices, for the bit-exact checks. */
int tto_decode(const tto_table* tabs, int ntab, int64_t bags_per_table, int64_t nnz,
               const int64_t* idx, const int64_t* offsets, int64_t* i1, int64_t* i2,
               int64_t* i3, int64_t* bag) {
    int64_t nbags = bags_per_table * ntab;
    for (int64_t g = 0; g < nbags; ++g) {
        if (offsets[g] > offsets[g + 1]) return TTO_ERR_ARG;
        const tto_table* t = &tabs[g / bags_per_table];
        for (int64_t n = offsets[g]; n < offsets[g + 1]; ++n) {
            if (n < 0 || n >= nnz) return TTO_ERR_ARG;
            int rc = decode_row(t, idx[n], &i1[n], &i2[n], &i3[n]);
            if (rc) return rc;
            bag[n] = g;
        }
    }
    return TTO_OK;
}

/* Pooling scale of lookup n in bag g. */
static double pool_scale(const double* w, int mean, const int64_t* offsets, int64_t g, int64_t n) {
    double s = w ? w[n] : 1.0;
    if (mean) s /= (double)(offsets[g + 1] - offsets[g]);
    return s;
}

/* W[i][j] for one row, straight from the definition. */
static void tt_row(const tto_table* t, int64_t i1, int64_t i2, int64_t i3, double* row) {
    const int64_t q1 = t->q[0], q2 = t->q[1], q3 = t->q[2], r1 = t->r[0], r2 = t->r[1];
    const double* g1 = t->G[0] + i1 * (q1 * r1);      /* [1][q1][r1] */
    const double* g2 = t->G[1] + i2 * (r1 * q2 * r2); /* [r1][q2][r2] */
    const double* g3 = t->G[2] + i3 * (r2 * q3);      /* [r2][q3][1] */
    for (int64_t j1 = 0; j1 < q1; ++j1)
        for (int64_t j2 = 0; j2 < q2; ++j2)
            for (int64_t j3 = 0; j3 < q3; ++j3) {
                double acc = 0.0;
                for (int64_t a = 0; a < r1; ++a)
                    for (int64_t c = 0; c < r2; ++c)
                        acc += g1[j1 * r1 + a] * g2[(a * q2 + j2) * r2 + c] * g3[c * q3 + j3];
                row[(j1 * q2 + j2) * q3 + j3] = acc;
            }
}

/*
 * Forward pass.  Bags are ordered table-major (bag g belongs to table
 * g / bags_per_table).  With sel == NULL every bag is computed and out has
 * nbags rows; otherwise only the nsel listed bags, one output row each.
 * All tables must share D.
 */
int tto_forward(const tto_table* tabs, int ntab, int64_t bags_per_table, int64_t nnz,
                const int64_t* idx, const int64_t* offsets, const double* w, int mean,
                int64_t nsel, const int64_t* sel, double* out) {
    const int64_t D = tabs[0].q[0] * tabs[0].q[1] * tabs[0].q[2];
    const int64_t nbags = bags_per_table * ntab;
    const int64_t nout = sel ? nsel : nbags;
    for (int k = 0; k < ntab; ++k)
        if (tabs[k].q[0] * tabs[k].q[1] * tabs[k].q[2] != D) return TTO_ERR_ARG;
    int err = TTO_OK;
#pragma omp parallel
    {
        double* row = (double*)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 16) reduction(max : err)
        for (int64_t o = 0; o < nout; ++o) {
            int64_t g = sel ? sel[o] : o;
            double* y = out + o * D;
            for (int64_t j = 0; j < D; ++j) y[j] = 0.0;
            if (g < 0 || g >= nbags) { err = TTO_ERR_ARG; continue; }
            const tto_table* t = &tabs[g / bags_per_table];
            for (int64_t n = offsets[g]; n < offsets[g + 1]; ++n) {
                int64_t i1, i2, i3;
                if (n < 0 || n >= nnz || decode_row(t, idx[n], &i1, &i2, &i3)) { err = TTO_ERR_INDEX; break; }
                tt_row(t, i1, i2, i3, row);
                double s = pool_scale(w, mean, offsets, g, n);
                for (int64_t j = 0; j < D; ++j) y[j] += s * row[j];
            }
        }
        free(row);
    }
    return err;
}

/*
 * Gradient of core `core` (0, 1, 2) of table `table` for the listed slices.
 * dG receives nslice slices of r_{k-1} q_k r_k doubles each, in the core's
 * own [r_{k-1}][q_k][r_k] order.  For each slice the lookups are visited in
 * bag order, then position order, and only those whose slice index matches
 * contribute.
 */
int tto_backward_core(const tto_table* tabs, int ntab, int64_t bags_per_table, int64_t nnz,
                      const int64_t* idx, const int64_t* offsets, const double* w, int mean,
                      const double* grad_out, int table, int core, int64_t nslice,
                      const int64_t* slices, double* dG) {
    if (table < 0 || table >= ntab || core < 0 || core > 2) return TTO_ERR_ARG;
    const tto_table* t = &tabs[table];
    const int64_t q1 = t->q[0], q2 = t->q[1], q3 = t->q[2], r1 = t->r[0], r2 = t->r[1];
    const int64_t D = q1 * q2 * q3;
    const int64_t rk[4] = {1, r1, r2, 1};
    const int64_t ssz = rk[core] * t->q[core] * rk[core + 1];
    const int64_t g_lo = (int64_t)table * bags_per_table, g_hi = g_lo + bags_per_table;
    int err = TTO_OK;
    for (int64_t s = 0; s < nslice; ++s)
        if (slices[s] < 0 || slices[s] >= t->p[core]) return TTO_ERR_ARG;

#pragma omp parallel for schedule(dynamic, 1) reduction(max : err)
    for (int64_t s = 0; s < nslice; ++s) {
        double* d = dG + s * ssz;
        for (int64_t e = 0; e < ssz; ++e) d[e] = 0.0;
        for (int64_t g = g_lo; g < g_hi; ++g) {
            for (int64_t n = offsets[g]; n < offsets[g + 1]; ++n) {
                int64_t ii[3];
                if (n < 0 || n >= nnz || decode_row(t, idx[n], &ii[0], &ii[1], &ii[2])) { err = TTO_ERR_INDEX; continue; }
                if (ii[core] != slices[s]) continue;
                const double sn = pool_scale(w, mean, offsets, g, n);
                const double* go = grad_out + g * D;
                const double* g1 = t->G[0] + ii[0] * (q1 * r1);
                const double* g2 = t->G[1] + ii[1] * (r1 * q2 * r2);
                const double* g3 = t->G[2] + ii[2] * (r2 * q3);
                if (core == 0) {
                    for (int64_t j1 = 0; j1 < q1; ++j1)
                        for (int64_t a = 0; a < r1; ++a) {
                            double acc = 0.0;
                            for (int64_t j2 = 0; j2 < q2; ++j2)
                                for (int64_t j3 = 0; j3 < q3; ++j3)
                                    for (int64_t c = 0; c < r2; ++c)
                                        acc += go[(j1 * q2 + j2) * q3 + j3] * g2[(a * q2 + j2) * r2 + c] * g3[c * q3 + j3];
                            d[j1 * r1 + a] += sn * acc;
                        }
                } else if (core == 1) {
                    for (int64_t a = 0; a < r1; ++a)
                        for (int64_t j2 = 0; j2 < q2; ++j2)
                            for (int64_t c = 0; c < r2; ++c) {
                                double acc = 0.0;
                                for (int64_t j1 = 0; j1 < q1; ++j1)
                                    for (int64_t j3 = 0; j3 < q3; ++j3)
                                        acc += go[(j1 * q2 + j2) * q3 + j3] * g1[j1 * r1 + a] * g3[c * q3 + j3];
                                d[(a * q2 + j2) * r2 + c] += sn * acc;
                            }
                } else {
                    for (int64_t c = 0; c < r2; ++c)
                        for (int64_t j3 = 0; j3 < q3; ++j3) {
                            double acc = 0.0;
                            for (int64_t j1 = 0; j1 < q1; ++j1)
                                for (int64_t j2 = 0; j2 < q2; ++j2)
                                    for (int64_t a = 0; a < r1; ++a)
                                        acc += go[(j1 * q2 + j2) * q3 + j3] * g1[j1 * r1 + a] * g2[(a * q2 + j2) * r2 + c];
                            d[c * q3 + j3] += sn * acc;
                        }
                }
            }
        }
    }
    return err;
}
