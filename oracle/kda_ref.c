/*
 * fp64 CPU oracle for the KDA intra-chunk forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library or its CUDA kernels calls,
 * links or includes this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline arm do.  It shares no code with the GPU path.
 *
 * Definitions (bwd_intra page, module docstring and the diagonal/epilogue loops of
 * kda_cute_intra; the gated delta rule's intra-chunk forward).  Per unit (b, h, c),
 * with r, s the in-chunk rows [0, BT), d in [0, K) and E[r,s,d] = 2^(g[r,d]-g[s,d])
 * where g is the chunk-local cumulative log2 gate:
 *
 *   Aqk[r,s] = sum_d q[r,d] k[s,d] E[r,s,d]              for s <= r, else 0
 *   Akk[r,s] = beta[r] sum_d k[r,d] k[s,d] E[r,s,d]      for s <  r, else 0
 *   L        = sum dAqk * Aqk + sum dAkk * Akk
 *
 * and the backward returns dq, dk, dbeta, dg = dL/d(input), with dg taken with
 * respect to the log2 gate g exactly as passed (so d E / d g[r,d] = ln2 * E).
 *
 * The backward is the chain rule applied to every product term of L, one pair
 * (r, s) and one channel d at a time: each term's derivative is scattered to the
 * inputs that appear in it.  There is no blocking, no factorization and no
 * reordering beyond that; entries of dAqk above the diagonal and of dAkk on or
 * above it are outside the forward's support and are never read.
 *
 * Layout: every array is [B, T, H, X] row-major (X = K for q, k, g, dq, dk, dg;
 * X = BT for dAqk, dAkk, Aqk, Akk; X = 1 for beta, db).  All in fp64.
 * Outputs are fully overwritten.  nthreads <= 0 means "OpenMP default".
 * Return 0 on success, -1 on a bad argument.
 */
#include <math.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define LN2 0.69314718055994530941723212145817656807550013436025

static size_t row_index(int b, int t, int h, int T, int H) {
    return ((size_t)b * (size_t)T + (size_t)t) * (size_t)H + (size_t)h;
}

static int check_args(int B, int T, int H, int K, int BT) {
    if (B <= 0 || T <= 0 || H <= 0 || K <= 0 || BT <= 0) return -1;
    if (T % BT != 0) return -1;
    return 0;
}

int kda_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for one call: nthreads if positive, else every available one.  Given to each
   parallel region on its own, so one call's count never carries over to the next. */
static int call_threads(int nthreads) {
    return nthreads > 0 ? nthreads : kda_oracle_max_threads();
}

/* Forward: the two intra-chunk score matrices. */
int kda_intra_fwd_ref_f64(const double *q, const double *k, const double *g,
                          const double *beta, double *Aqk, double *Akk,
                          int B, int T, int H, int K, int BT, int nthreads) {
    if (check_args(B, T, H, K, BT)) return -1;
    const int nt = call_threads(nthreads);
    const int NT = T / BT;
    const long units = (long)B * H * NT;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (long u = 0; u < units; ++u) {
        const int h = (int)(u % H);
        const int c = (int)((u / H) % NT);
        const int b = (int)(u / ((long)H * NT));
        for (int r = 0; r < BT; ++r) {
            const size_t R = row_index(b, c * BT + r, h, T, H);
            for (int s = 0; s < BT; ++s) {
                const size_t S = row_index(b, c * BT + s, h, T, H);
                double sqk = 0.0, skk = 0.0;
                if (s <= r) {
                    for (int d = 0; d < K; ++d) {
                        const double E = exp2(g[R * K + d] - g[S * K + d]);
                        sqk += q[R * K + d] * k[S * K + d] * E;
                        skk += k[R * K + d] * k[S * K + d] * E;
                    }
                }
                Aqk[R * BT + s] = (s <= r) ? sqk : 0.0;
                Akk[R * BT + s] = (s < r) ? beta[R] * skk : 0.0;
            }
        }
    }
    return 0;
}

/* Backward: dq, dk, dbeta, dg of L = sum dAqk*Aqk + sum dAkk*Akk. */
int kda_intra_bwd_ref_f64(const double *q, const double *k, const double *g,
                          const double *beta, const double *dAqk, const double *dAkk,
                          double *dq, double *dk, double *db, double *dg,
                          int B, int T, int H, int K, int BT, int nthreads) {
    if (check_args(B, T, H, K, BT)) return -1;
    const int nt = call_threads(nthreads);
    const int NT = T / BT;
    const long units = (long)B * H * NT;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (long u = 0; u < units; ++u) {
        const int h = (int)(u % H);
        const int c = (int)((u / H) % NT);
        const int b = (int)(u / ((long)H * NT));
        /* zero this unit's outputs (units never overlap, so this is race-free) */
        for (int t = 0; t < BT; ++t) {
            const size_t Rt = row_index(b, c * BT + t, h, T, H);
            memset(dq + Rt * K, 0, sizeof(double) * (size_t)K);
            memset(dk + Rt * K, 0, sizeof(double) * (size_t)K);
            memset(dg + Rt * K, 0, sizeof(double) * (size_t)K);
            db[Rt] = 0.0;
        }
        for (int r = 0; r < BT; ++r) {
            const size_t R = row_index(b, c * BT + r, h, T, H);
            for (int s = 0; s <= r; ++s) {
                const size_t S = row_index(b, c * BT + s, h, T, H);
                const double aqk = dAqk[R * BT + s];
                const double akk = (s < r) ? dAkk[R * BT + s] : 0.0;
                for (int d = 0; d < K; ++d) {
                    const double qr = q[R * K + d], kr = k[R * K + d];
                    const double ks = k[S * K + d];
                    const double E = exp2(g[R * K + d] - g[S * K + d]);

                    /* term dAqk[r,s] * q[r,d] k[s,d] E[r,s,d] */
                    const double wq = aqk * qr * ks * E;
                    dq[R * K + d] += aqk * ks * E;
                    dk[S * K + d] += aqk * qr * E;
                    dg[R * K + d] += LN2 * wq;   /* E grows with g[r,d] */
                    dg[S * K + d] -= LN2 * wq;   /* E shrinks with g[s,d] */

                    if (s < r) {
                        /* term dAkk[r,s] * beta[r] k[r,d] k[s,d] E[r,s,d] */
                        const double wk = akk * beta[R] * kr * ks * E;
                        dk[R * K + d] += akk * beta[R] * ks * E;
                        dk[S * K + d] += akk * beta[R] * kr * E;
                        db[R] += akk * kr * ks * E;
                        dg[R * K + d] += LN2 * wk;
                        dg[S * K + d] -= LN2 * wk;
                    }
                }
            }
        }
    }
    return 0;
}
