/*
 * ck_oracle.c -- TEST INFRASTRUCTURE ONLY (the oracle).
 *
 * A plain, slow, fp64 CPU statement of the leaky-tanh recurrence over a fixed
 * sparse directed graph and of its hand-derived backward.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg use it; the CUDA library
 * never links, calls or includes anything from here, and this file shares no
 * code with it.
 *
 * What it follows (connectome-kernels page):
 *   - intro, the two update equations: proposal_i = tanh(sum_j W_ij h_j +
 *     drive_i + bias_i); h_i <- (1 - leak_i) h_i + leak_i * proposal_i,
 *     repeated `microsteps` times per input step;
 *   - intro: W is sparse with a fixed pattern, one scalar per edge, and the
 *     drive enters only at the designated input nodes;
 *   - "Use": edges are src[e] -> dst[e]; drives are [T, n_in, B]; state0 is
 *     [B, N]; the output is [T, B, N], the node states after each input step;
 *     gradients are taken with respect to edge values, leak, bias, drives and
 *     state0.
 *
 * Readings taken where the page leaves a step open:
 *   - W_ij h_j flows along an edge src=j -> dst=i, so W[dst][src] = w[e];
 *     repeated (src,dst) pairs add up.
 *   - All nodes update together: every node of a microstep reads the state
 *     left by the previous microstep.
 *   - The drive of input step t is added in every one of its microsteps; it is
 *     zero at nodes that are not input nodes.
 *   - out[t] is the state after the last microstep of input step t.
 *   - leak is used exactly as passed (a caller may squash it first).
 *   - The backward is the vector-Jacobian product of L = sum_t <dOut[t], out[t]>.
 *
 * Loops run over edges in the caller's edge order (coordinate lists), not in a
 * sorted or compressed layout.  Batch columns are independent sequences, so
 * the outer loop is over the batch index b.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define IDX3(a, b, c, B_, C_) (((int64_t)(a) * (B_) + (b)) * (C_) + (c))

/*
 * Forward over the whole window of T input steps x M microsteps.
 *   src, dst      [E]          edge endpoints, 0 <= src, dst < N
 *   w             [E]          edge values in the caller's order
 *   leak, bias    [N]
 *   input_nodes   [n_in]       distinct node ids; drive row k enters node input_nodes[k]
 *   drives        [T][n_in][B]
 *   state0        [B][N]
 * Outputs:
 *   out           [T][B][N]    state after the last microstep of each input step
 *   hprev         [S][B][N]    state entering microstep s (S = T*M); may be NULL
 *   pre           [S][B][N]    pre-activation a = W h + drive + bias of microstep s; may be NULL
 * Returns 0, or -1 when a work buffer cannot be allocated.
 */
int oracle_forward(int64_t N, int64_t E, const int64_t *src, const int64_t *dst,
                   const double *w, const double *leak, const double *bias,
                   int64_t n_in, const int64_t *input_nodes, const double *drives,
                   const double *state0, int64_t B, int64_t T, int64_t M,
                   double *out, double *hprev, double *pre)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)N);
    double *hn = (double *)malloc(sizeof(double) * (size_t)N);
    double *acc = (double *)malloc(sizeof(double) * (size_t)N);
    double *d = (double *)malloc(sizeof(double) * (size_t)N);
    if (!h || !hn || !acc || !d) {
        free(h); free(hn); free(acc); free(d);
        return -1;
    }
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t i = 0; i < N; ++i) h[i] = state0[b * N + i];
        for (int64_t t = 0; t < T; ++t) {
            /* drive vector of input step t for this batch column */
            for (int64_t i = 0; i < N; ++i) d[i] = 0.0;
            for (int64_t k = 0; k < n_in; ++k)
                d[input_nodes[k]] = drives[IDX3(t, k, b, n_in, B)];
            for (int64_t m = 0; m < M; ++m) {
                int64_t s = t * M + m;
                /* sum_j W_ij h_j over the edges, every edge reading the old h */
                for (int64_t i = 0; i < N; ++i) acc[i] = 0.0;
                for (int64_t e = 0; e < E; ++e) acc[dst[e]] += w[e] * h[src[e]];
                for (int64_t i = 0; i < N; ++i) {
                    double a = acc[i] + d[i] + bias[i];
                    double p = tanh(a);
                    if (hprev) hprev[IDX3(s, b, i, B, N)] = h[i];
                    if (pre) pre[IDX3(s, b, i, B, N)] = a;
                    hn[i] = (1.0 - leak[i]) * h[i] + leak[i] * p;
                }
                double *tmp = h; h = hn; hn = tmp;
            }
            for (int64_t i = 0; i < N; ++i) out[IDX3(t, b, i, B, N)] = h[i];
        }
    }
    free(h); free(hn); free(acc); free(d);
    return 0;
}

/*
 * Backward: the vector-Jacobian product of L = sum_t <dout[t], out[t]>,
 * derived by hand from the two update equations.  With G_s the gradient with
 * respect to the state after microstep s (including dout[t] when s is the last
 * microstep of step t), p_s = tanh(a_s) and h_{s-1} the state entering s:
 *   da_s     = G_s * leak * (1 - p_s^2)
 *   dleak   += G_s * (p_s - h_{s-1})          (summed over b and s)
 *   dbias   += da_s
 *   ddrives[t][k] += da_s[input_nodes[k]]     (every microstep of step t)
 *   dw[e]   += da_s[dst[e]] * h_{s-1}[src[e]]
 *   G_{s-1}  = G_s * (1 - leak) + W^T da_s    (W^T da: along each edge dst -> src)
 *   dstate0  = G_{-1}
 * hprev and pre are the buffers oracle_forward filled.  All outputs are
 * overwritten.  Returns 0, or -1 when a work buffer cannot be allocated.
 */
int oracle_backward(int64_t N, int64_t E, const int64_t *src, const int64_t *dst,
                    const double *w, const double *leak,
                    int64_t n_in, const int64_t *input_nodes,
                    int64_t B, int64_t T, int64_t M,
                    const double *hprev, const double *pre, const double *dout,
                    double *dw, double *dleak, double *dbias, double *ddrives,
                    double *dstate0)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)N);
    double *gn = (double *)malloc(sizeof(double) * (size_t)N);
    double *da = (double *)malloc(sizeof(double) * (size_t)N);
    if (!g || !gn || !da) {
        free(g); free(gn); free(da);
        return -1;
    }
    int64_t S = T * M;
    memset(dw, 0, sizeof(double) * (size_t)E);
    memset(dleak, 0, sizeof(double) * (size_t)N);
    memset(dbias, 0, sizeof(double) * (size_t)N);
    memset(ddrives, 0, sizeof(double) * (size_t)(T * n_in * B));
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t i = 0; i < N; ++i) g[i] = 0.0;
        for (int64_t s = S - 1; s >= 0; --s) {
            int64_t t = s / M, m = s % M;
            const double *hp = hprev + IDX3(s, b, 0, B, N);
            const double *a = pre + IDX3(s, b, 0, B, N);
            if (m == M - 1)
                for (int64_t i = 0; i < N; ++i) g[i] += dout[IDX3(t, b, i, B, N)];
            for (int64_t i = 0; i < N; ++i) {
                double p = tanh(a[i]);
                dleak[i] += g[i] * (p - hp[i]);
                da[i] = g[i] * leak[i] * (1.0 - p * p);
                dbias[i] += da[i];
            }
            for (int64_t k = 0; k < n_in; ++k)
                ddrives[IDX3(t, k, b, n_in, B)] += da[input_nodes[k]];
            for (int64_t e = 0; e < E; ++e) dw[e] += da[dst[e]] * hp[src[e]];
            for (int64_t i = 0; i < N; ++i) gn[i] = g[i] * (1.0 - leak[i]);
            for (int64_t e = 0; e < E; ++e) gn[src[e]] += w[e] * da[dst[e]];
            double *tmp = g; g = gn; gn = tmp;
        }
        for (int64_t i = 0; i < N; ++i) dstate0[b * N + i] = g[i];
    }
    free(g); free(gn); free(da);
    return 0;
}

/*
 * One whole training step (forward, then backward of L = sum_t <dout[t],
 * out[t]>) with the batch columns spread over `threads` OpenMP threads.
 * Each column is an independent sequence, so a column's forward and backward
 * are exactly the loops of oracle_forward / oracle_backward restricted to it;
 * this function only reorders the work by column to run columns in parallel.
 * Columns go to threads in contiguous blocks (static schedule); the gradients
 * shared by all columns (dw, dleak, dbias) are summed per thread in column
 * order and the per-thread sums are then added in thread order, so the
 * result is the same for every run with the same thread count and differs
 * from the single-thread functions only in the grouping of those sums.
 * Built without OpenMP it runs on one thread.  Outputs as oracle_forward and
 * oracle_backward (hprev and pre are not returned).  Returns 0, or -1 when a
 * work buffer cannot be allocated.
 */
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_threads_available(void)
{
#ifdef _OPENMP
    return omp_get_num_procs();
#else
    return 1;
#endif
}

int oracle_step_columns(int64_t N, int64_t E, const int64_t *src, const int64_t *dst,
                        const double *w, const double *leak, const double *bias,
                        int64_t n_in, const int64_t *input_nodes, const double *drives,
                        const double *state0, const double *dout, int64_t B, int64_t T,
                        int64_t M, int threads, double *out, double *dw, double *dleak,
                        double *dbias, double *ddrives, double *dstate0)
{
    const int64_t S = T * M;
    int nt = threads < 1 ? 1 : threads;
    if (nt > B) nt = (int)B;
#ifndef _OPENMP
    nt = 1;
#endif
    /* per-thread shared-parameter gradient sums: [nt][E + 2N] */
    const int64_t per = E + 2 * N;
    double *part = (double *)calloc((size_t)nt * (size_t)(per > 0 ? per : 1), sizeof(double));
    if (!part) return -1;
    int fail = 0;
#ifdef _OPENMP
#pragma omp parallel num_threads(nt)
#endif
    {
#ifdef _OPENMP
        const int tid = omp_get_thread_num();
#else
        const int tid = 0;
#endif
        const int64_t b0 = B * tid / nt, b1 = B * (tid + 1) / nt;
        double *h = (double *)malloc(sizeof(double) * (size_t)N);
        double *hn = (double *)malloc(sizeof(double) * (size_t)N);
        double *acc = (double *)malloc(sizeof(double) * (size_t)N);
        double *d = (double *)malloc(sizeof(double) * (size_t)N);
        double *hp_all = (double *)malloc(sizeof(double) * (size_t)(S * N));
        double *a_all = (double *)malloc(sizeof(double) * (size_t)(S * N));
        double *my_dw = part + (int64_t)tid * per;
        double *my_dl = my_dw + E, *my_db = my_dl + N;
        if (!h || !hn || !acc || !d || !hp_all || !a_all) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            fail = 1;
        } else {
            for (int64_t b = b0; b < b1; ++b) {
                /* forward of column b: oracle_forward's loops */
                for (int64_t i = 0; i < N; ++i) h[i] = state0[b * N + i];
                for (int64_t t = 0; t < T; ++t) {
                    for (int64_t i = 0; i < N; ++i) d[i] = 0.0;
                    for (int64_t k = 0; k < n_in; ++k)
                        d[input_nodes[k]] = drives[IDX3(t, k, b, n_in, B)];
                    for (int64_t m = 0; m < M; ++m) {
                        const int64_t s = t * M + m;
                        for (int64_t i = 0; i < N; ++i) acc[i] = 0.0;
                        for (int64_t e = 0; e < E; ++e) acc[dst[e]] += w[e] * h[src[e]];
                        for (int64_t i = 0; i < N; ++i) {
                            const double a = acc[i] + d[i] + bias[i];
                            hp_all[s * N + i] = h[i];
                            a_all[s * N + i] = a;
                            hn[i] = (1.0 - leak[i]) * h[i] + leak[i] * tanh(a);
                        }
                        double *tmp = h; h = hn; hn = tmp;
                    }
                    for (int64_t i = 0; i < N; ++i) out[IDX3(t, b, i, B, N)] = h[i];
                }
                /* backward of column b: oracle_backward's loops (h is g here,
                   hn is g', acc is da) */
                double *g = h, *gn = hn, *da = acc;
                for (int64_t i = 0; i < N; ++i) g[i] = 0.0;
                for (int64_t t = 0; t < T; ++t)
                    for (int64_t k = 0; k < n_in; ++k) ddrives[IDX3(t, k, b, n_in, B)] = 0.0;
                for (int64_t s = S - 1; s >= 0; --s) {
                    const int64_t t = s / M, m = s % M;
                    const double *hp = hp_all + s * N, *a = a_all + s * N;
                    if (m == M - 1)
                        for (int64_t i = 0; i < N; ++i) g[i] += dout[IDX3(t, b, i, B, N)];
                    for (int64_t i = 0; i < N; ++i) {
                        const double p = tanh(a[i]);
                        my_dl[i] += g[i] * (p - hp[i]);
                        da[i] = g[i] * leak[i] * (1.0 - p * p);
                        my_db[i] += da[i];
                    }
                    for (int64_t k = 0; k < n_in; ++k)
                        ddrives[IDX3(t, k, b, n_in, B)] += da[input_nodes[k]];
                    for (int64_t e = 0; e < E; ++e) my_dw[e] += da[dst[e]] * hp[src[e]];
                    for (int64_t i = 0; i < N; ++i) gn[i] = g[i] * (1.0 - leak[i]);
                    for (int64_t e = 0; e < E; ++e) gn[src[e]] += w[e] * da[dst[e]];
                    double *tmp = g; g = gn; gn = tmp;
                }
                for (int64_t i = 0; i < N; ++i) dstate0[b * N + i] = g[i];
                h = g; hn = gn;
            }
        }
        free(h); free(hn); free(acc); free(d); free(hp_all); free(a_all);
    }
    if (!fail) {
        /* fixed order: thread 0's sums, then thread 1's, ... */
        for (int64_t e = 0; e < E; ++e) dw[e] = 0.0;
        for (int64_t i = 0; i < N; ++i) dleak[i] = dbias[i] = 0.0;
        for (int t = 0; t < nt; ++t) {
            const double *p = part + (int64_t)t * per;
            for (int64_t e = 0; e < E; ++e) dw[e] += p[e];
            for (int64_t i = 0; i < N; ++i) {
                dleak[i] += p[E + i];
                dbias[i] += p[E + N + i];
            }
        }
    }
    free(part);
    return fail ? -1 : 0;
}
