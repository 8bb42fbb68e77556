/*
 * Float64 CPU oracle for the Mamba-2 chunked SSD forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header or constant
 * with the CUDA library.
 *
 * Source: "Accelerating Mamba-2 forward-pass kernels with CUDA Tile
 * (cuTile)" (Chinese translation, dbyun.net/article/14364):
 *   - section "Mamba-2 架构", recurrence  h_t = exp(A dt_t) h_{t-1} + dt_t B_t x_t^T,
 *     y_t = c_t^T h_t + D x_t;
 *   - section "Kernel 1": the within-chunk cumulative sum of A[h]*dt[t,h],
 *     scaled by log2(e);
 *   - section "Kernel 2: fwd_pass_state": every chunk's start state is the
 *     state before the chunk's first token (chunk 0 gets init_state), and
 *     the state after the last token is the final state.
 *
 * Readings taken where the pages are ambiguous (each is also listed in the
 * design notes):
 *   - y_t uses the state AFTER token t's update (inclusive); the
 *     "Mamba-2 架构" shorthand that writes h_{t-1} contradicts the
 *     expanded form and the causal mask i >= j of "Kernel 3".
 *   - The state is stored as h[p][s] (head dim P rows, state dim S
 *     columns), the orientation of the pages' hid_tile.
 *   - group(h) = h / (H / G): contiguous heads share B and C.
 *   - dt arrives already activated; nothing is applied to it here.
 *
 * Layouts (row-major, contiguous):
 *   x  [B,L,H,P]  dt [B,L,H]  A [H]  Bm, Cm [B,L,G,S]  D [H]
 *   init, final [B,H,P,S]     states [B,H,nc,P,S]      y [B,L,H,P]
 *   Gout [B,H,L]
 *
 * Parity of the product against this oracle is pinned by independent
 * checks in the test suite (brute-force quadratic form, chunked closed
 * form, linear-attention special case, hand-worked golden values and
 * invariants).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_LOG2E 1.4426950408889634073599246810019

/* Within-chunk cumulative sum of a = A[h]*dt, in log2 units ("Kernel 1").
 * The sum restarts at every multiple of T; it is not a global scan. */
int ssd_oracle_chunk_cumsum(int64_t B, int64_t L, int64_t H, int64_t T,
                            const double *dt, const double *A, double *Gout)
{
    if (B < 0 || L < 0 || H <= 0 || T <= 0 || !dt || !A || !Gout)
        return -1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h) {
            double run = 0.0;
            for (int64_t t = 0; t < L; ++t) {
                if (t % T == 0)
                    run = 0.0;
                run += A[h] * dt[(b * L + t) * H + h];
                Gout[(b * H + h) * L + t] = ORACLE_LOG2E * run;
            }
        }
    return 0;
}

/* Token-by-token recurrence ("Mamba-2 架构").  One (b, h) pair at a time:
 *
 *   for t in 0..L-1:
 *     if t % T == 0: states[c = t/T] = h        (chunk start state)
 *     h[p][s] = exp(A[h] dt[t]) h[p][s] + dt[t] x[t][p] B[t][s]
 *     y[t][p] = sum_s C[t][s] h[p][s] + D[h] x[t][p]
 *   final = h
 *
 * init may be NULL (zero state); final and states may be NULL (not
 * wanted).  nthreads <= 0 uses the OpenMP default. */
int ssd_oracle_fwd(int64_t B, int64_t L, int64_t H, int64_t P, int64_t S,
                   int64_t G, int64_t T,
                   const double *x, const double *dt, const double *A,
                   const double *Bm, const double *Cm, const double *D,
                   const double *init, double *y, double *final_state,
                   double *states, int nthreads)
{
    if (B < 0 || L < 0 || H <= 0 || P <= 0 || S <= 0 || G <= 0 || T <= 0)
        return -1;
    if (H % G != 0)
        return -1;
    if (!x || !dt || !A || !Bm || !Cm || !D || !y)
        return -1;
    const int64_t heads_per_group = H / G;
    const int64_t nc = (L + T - 1) / T;
    const int64_t pairs = B * H;
    int rc = 0;

#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t bh = 0; bh < pairs; ++bh) {
        const int64_t b = bh / H, h = bh % H;
        const int64_t g = h / heads_per_group;
        double *st = (double *)malloc((size_t)(P * S) * sizeof(double));
        if (!st) {
            rc = -2;
            continue;
        }
        if (init)
            memcpy(st, init + bh * P * S, (size_t)(P * S) * sizeof(double));
        else
            memset(st, 0, (size_t)(P * S) * sizeof(double));

        for (int64_t t = 0; t < L; ++t) {
            if (states && t % T == 0)
                memcpy(states + (bh * nc + t / T) * P * S, st,
                       (size_t)(P * S) * sizeof(double));
            const double dtv = dt[(b * L + t) * H + h];
            const double decay = exp(A[h] * dtv);
            const double *xt = x + ((b * L + t) * H + h) * P;
            const double *bt = Bm + ((b * L + t) * G + g) * S;
            const double *ct = Cm + ((b * L + t) * G + g) * S;
            double *yt = y + ((b * L + t) * H + h) * P;
            for (int64_t p = 0; p < P; ++p) {
                double *row = st + p * S;
                const double u = dtv * xt[p];
                double acc = 0.0;
                for (int64_t s = 0; s < S; ++s) {
                    row[s] = decay * row[s] + u * bt[s];
                    acc += ct[s] * row[s];
                }
                yt[p] = acc + D[h] * xt[p];
            }
        }
        if (final_state)
            memcpy(final_state + bh * P * S, st, (size_t)(P * S) * sizeof(double));
        free(st);
    }
    return rc;
}

/* Gradients of the token recurrence ("Mamba-2 架构") by its adjoint, for a
 * scalar loss whose gradients with respect to y and the final state are dy
 * and dfinal (dfinal may be NULL: zero).  Per (b, h), g = h / (H / G):
 *
 *   forward, keeping every state:  h_{-1} = init,
 *     a_t = exp(A dt_t),  h_t = a_t h_{t-1} + dt_t x_t B_t^T,  y_t = h_t C_t + D x_t
 *   backward, t = L-1 .. 0, with the adjoint state dh (P x S) = dfinal:
 *     dh    += dy_t C_t^T                         (y_t reads h_t)
 *     dC_t  += h_t^T dy_t                         (summed over the group's heads)
 *     dD    += dy_t . x_t
 *     dx_t   = D dy_t + dt_t dh B_t
 *     dB_t  += dt_t dh^T x_t                      (summed over the group's heads)
 *     da     = sum dh * h_{t-1}
 *     ddt_t  = x_t^T dh B_t + A a_t da
 *     dA    += dt_t a_t da
 *     dh     = a_t dh                             (to h_{t-1})
 *   dinit = dh  (if dinit is not NULL).
 *
 * Layouts as in ssd_oracle_fwd; dy like y, dfinal / dinit like init; dx like
 * x, ddt like dt, dA / dD [H], dB / dC like Bm / Cm.  Parallel over (b, g):
 * the heads of a group run in turn, so the group sums need no atomics.
 * Memory: (L + 1) P S doubles per thread (every state is kept). */
int ssd_oracle_bwd(int64_t B, int64_t L, int64_t H, int64_t P, int64_t S, int64_t G,
                   const double *x, const double *dt, const double *A,
                   const double *Bm, const double *Cm, const double *D,
                   const double *init, const double *dy, const double *dfinal,
                   double *dx, double *ddt, double *dA, double *dB, double *dC,
                   double *dD, double *dinit, int nthreads)
{
    if (B < 0 || L < 0 || H <= 0 || P <= 0 || S <= 0 || G <= 0 || H % G != 0)
        return -1;
    if (!x || !dt || !A || !Bm || !Cm || !D || !dy || !dx || !ddt || !dA || !dB || !dC || !dD)
        return -1;
    const int64_t hpg = H / G;
    const int64_t PS = P * S;
    memset(dB, 0, (size_t)(B * L * G * S) * sizeof(double));
    memset(dC, 0, (size_t)(B * L * G * S) * sizeof(double));
    /* per-(b, h) partial sums of dA and dD, reduced at the end in a fixed order */
    double *pA = (double *)calloc((size_t)(B * H), sizeof(double));
    double *pD = (double *)calloc((size_t)(B * H), sizeof(double));
    if (!pA || !pD) {
        free(pA);
        free(pD);
        return -2;
    }
    int rc = 0;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t bg = 0; bg < B * G; ++bg) {
        const int64_t b = bg / G, g = bg % G;
        double *traj = (double *)malloc((size_t)((L + 1) * PS) * sizeof(double));
        double *adj = (double *)malloc((size_t)PS * sizeof(double));
        if (!traj || !adj) {
            free(traj);
            free(adj);
            rc = -2;
            continue;
        }
        for (int64_t h = g * hpg; h < (g + 1) * hpg; ++h) {
            const int64_t bh = b * H + h;
            /* forward: traj[t + 1] = h_t, traj[0] = init */
            if (init)
                memcpy(traj, init + bh * PS, (size_t)PS * sizeof(double));
            else
                memset(traj, 0, (size_t)PS * sizeof(double));
            for (int64_t t = 0; t < L; ++t) {
                const double dtv = dt[(b * L + t) * H + h];
                const double a = exp(A[h] * dtv);
                const double *xt = x + ((b * L + t) * H + h) * P;
                const double *bt = Bm + ((b * L + t) * G + g) * S;
                const double *prev = traj + t * PS;
                double *cur = traj + (t + 1) * PS;
                for (int64_t p = 0; p < P; ++p)
                    for (int64_t s = 0; s < S; ++s)
                        cur[p * S + s] = a * prev[p * S + s] + dtv * xt[p] * bt[s];
            }
            /* backward */
            if (dfinal)
                memcpy(adj, dfinal + bh * PS, (size_t)PS * sizeof(double));
            else
                memset(adj, 0, (size_t)PS * sizeof(double));
            double sA = 0.0, sD = 0.0;
            for (int64_t t = L - 1; t >= 0; --t) {
                const double dtv = dt[(b * L + t) * H + h];
                const double a = exp(A[h] * dtv);
                const double *xt = x + ((b * L + t) * H + h) * P;
                const double *bt = Bm + ((b * L + t) * G + g) * S;
                const double *ct = Cm + ((b * L + t) * G + g) * S;
                const double *dyt = dy + ((b * L + t) * H + h) * P;
                const double *ht = traj + (t + 1) * PS;
                const double *hprev = traj + t * PS;
                double *dxt = dx + ((b * L + t) * H + h) * P;
                double *dbt = dB + ((b * L + t) * G + g) * S;
                double *dct = dC + ((b * L + t) * G + g) * S;
                for (int64_t p = 0; p < P; ++p)
                    for (int64_t s = 0; s < S; ++s)
                        adj[p * S + s] += dyt[p] * ct[s];
                for (int64_t s = 0; s < S; ++s) {
                    double acc = 0.0;
                    for (int64_t p = 0; p < P; ++p)
                        acc += ht[p * S + s] * dyt[p];
                    dct[s] += acc;
                }
                double ddirect = 0.0, da = 0.0;
                for (int64_t p = 0; p < P; ++p) {
                    sD += dyt[p] * xt[p];
                    double hb = 0.0;
                    for (int64_t s = 0; s < S; ++s) {
                        hb += adj[p * S + s] * bt[s];
                        da += adj[p * S + s] * hprev[p * S + s];
                    }
                    dxt[p] = D[h] * dyt[p] + dtv * hb;
                    ddirect += xt[p] * hb;
                }
                for (int64_t s = 0; s < S; ++s) {
                    double acc = 0.0;
                    for (int64_t p = 0; p < P; ++p)
                        acc += adj[p * S + s] * xt[p];
                    dbt[s] += dtv * acc;
                }
                ddt[(b * L + t) * H + h] = ddirect + A[h] * a * da;
                sA += dtv * a * da;
                for (int64_t k = 0; k < PS; ++k)
                    adj[k] *= a;
            }
            if (dinit)
                memcpy(dinit + bh * PS, adj, (size_t)PS * sizeof(double));
            pA[bh] = sA;
            pD[bh] = sD;
        }
        free(traj);
        free(adj);
    }
    for (int64_t h = 0; h < H; ++h) {
        double sa = 0.0, sd = 0.0;
        for (int64_t b = 0; b < B; ++b) {
            sa += pA[b * H + h];
            sd += pD[b * H + h];
        }
        dA[h] = sa;
        dD[h] = sd;
    }
    free(pA);
    free(pD);
    return rc;
}
