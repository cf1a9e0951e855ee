/*
 * oracle.c -- plain, slow, sequential fp64 reference of the selective scan
 * and of the Mamba-2 SSD scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library: it is the plain definition written out, one time step at a
 * time, in double precision, so that a reader can check it against the
 * equations by eye.
 *
 * Sources (page titles and sections):
 *  - "Mamba模型笔记" (sunyzhi55 study notes) §2.2: the discrete recurrence
 *    h_t = Abar h_{t-1} + Bbar x_t,  y_t = C h_t + D x_t.
 *  - same page §4.1 and §4.4: B, C and Delta depend on the input; one SSM per
 *    channel (diagonal A, one row of d_state values per channel).
 *  - same page §4.3: the gate branch; the gate is y * silu(z).
 *  - 0539edu paper talk §2.3: Abar = exp(Delta A), Bbar = Delta B, Cbar = C,
 *    Delta made positive by softplus.
 *  - 0539edu paper talk §4.1: the state is batch x d_inner x d_state and its
 *    size does not depend on the sequence length.
 *  - state-spaces/mamba README §4.3 and the study notes §5: Mamba-2 / SSD,
 *    multi-head with a scalar A per head and d_state 64..128.
 *
 *  - study notes §4.3 and the paper talk §3.1: the branch that feeds the SSM
 *    passes a short causal depthwise convolution (kernel width d_conv = 4)
 *    first; followed here by SiLU.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): softplus(x) = log(1 + e^x); A is given already negative and used as
 * is; the initial state is zero unless h0 is given; B and C are shared by all
 * channels of one batch row unless given per channel group (G groups of D/G
 * consecutive channels; G = D is one B, C per channel); the SSD dt is
 * already positive.
 *
 * What pins each function to something other than itself (CPU tests of the
 * oracle; no function here is left unpinned):
 *  - the selective scan: answers worked out by hand; the LTI special case
 *    against a directly evaluated causal convolution; the zero-step limit;
 *    brute-force unrolled products on short sequences; split invariance with
 *    the state carried; linearity and the zero cases.
 *  - its grouped form: brute-force sums per channel with the group's B and C,
 *    and equality with the shared form when all groups hold the same B, C.
 *  - the SSD scan: a hand-worked two-head case; equality with the selective
 *    scan given a scalar A per head; the dense quadratic (dual) form.
 *  - the causal convolution with SiLU: identity, delay and bias-only kernels
 *    and numpy's convolution.
 *  - the backward: central finite differences of the forward along random
 *    directions for every input.
 * A set of deliberately broken copies of this file (a dropped term, a wrong
 * sign, index or operand) is compiled by the tests, and each must fail one
 * of these pins.
 *
 * Parallelism: the optional OpenMP loop runs over independent (batch,
 * channel) or (batch, head) units only; every unit is computed by the same
 * sequential loop, so the result does not depend on the thread count.
 */
#include <math.h>
#include <stdlib.h>
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(x) = log(1 + exp(x)).  For x > 0 the identity
 * log(1 + e^x) = x + log(1 + e^-x) avoids overflowing exp; both branches are
 * the same real function. */
static double softplus_d(double x) {
    if (x > 0.0) return x + log1p(exp(-x));
    return log1p(exp(x));
}

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Selective scan (Mamba-1), one sequential loop per (batch row b, channel d).
 *
 *   u, delta, z, y : (Bsz, D, L), t fastest
 *   A              : (D, N)
 *   Bm, Cm         : (Bsz, G, N, L)  channel d reads group g = d / (D / G):
 *                    G = 1 is one B, C per batch row shared by all channels,
 *                    G = D one per channel
 *   Dv, delta_bias : (D)           (nullable: no skip / no bias)
 *   z              : nullable (no gate)
 *   h0             : (Bsz, D, N)   nullable (zero initial state)
 *   last_state     : (Bsz, D, N)   nullable (not written)
 *
 * For every t:
 *   dlt  = delta + delta_bias[d];  if softplus: dlt = softplus(dlt)
 *   h[n] = exp(dlt * A[d,n]) * h[n] + dlt * B[b,g,n,t] * u[b,d,t]
 *   out  = sum_n C[b,g,n,t] * h[n] + D[d] * u[b,d,t]
 *   if z: out = out * z / (1 + exp(-z))
 */
int oracle_selective_scan_grouped(int64_t Bsz, int64_t D, int64_t G, int64_t N, int64_t L,
                                  const double* u, const double* delta, const double* A,
                                  const double* Bm, const double* Cm, const double* Dv,
                                  const double* z, const double* delta_bias, int softplus,
                                  const double* h0, double* y, double* last_state,
                                  int nthreads) {
    if (Bsz < 0 || D < 0 || N < 1 || L < 0 || G < 1 || (D > 0 && D % G != 0)) return -1;
    int64_t units = Bsz * D;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t unit = 0; unit < units; ++unit) {
        int64_t b = unit / D, d = unit % D;
        int64_t g = d / (D / G);
        double* hp = (double*)malloc((size_t)N * sizeof(double));
        if (!hp) continue;
        for (int64_t n = 0; n < N; ++n)
            hp[n] = h0 ? h0[(b * D + d) * N + n] : 0.0;
        const double* ur = u + (b * D + d) * L;
        const double* dr = delta + (b * D + d) * L;
        const double* zr = z ? z + (b * D + d) * L : NULL;
        const double* Bg = Bm + (b * G + g) * N * L;  /* this channel's group */
        const double* Cg = Cm + (b * G + g) * N * L;
        double* yr = y + (b * D + d) * L;
        for (int64_t t = 0; t < L; ++t) {
            double dlt = dr[t] + (delta_bias ? delta_bias[d] : 0.0);
            if (softplus) dlt = softplus_d(dlt);
            double out = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double abar = exp(dlt * A[d * N + n]);
                double bbar = dlt * Bg[n * L + t];
                hp[n] = abar * hp[n] + bbar * ur[t];
                out += Cg[n * L + t] * hp[n];
            }
            if (Dv) out += Dv[d] * ur[t];
            if (zr) out = out * zr[t] / (1.0 + exp(-zr[t]));
            yr[t] = out;
        }
        if (last_state)
            for (int64_t n = 0; n < N; ++n) last_state[(b * D + d) * N + n] = hp[n];
        free(hp);
    }
    return 0;
}

/* The common case: one B and one C per batch row, (Bsz, N, L). */
int oracle_selective_scan(int64_t Bsz, int64_t D, int64_t N, int64_t L,
                          const double* u, const double* delta, const double* A,
                          const double* Bm, const double* Cm, const double* Dv,
                          const double* z, const double* delta_bias, int softplus,
                          const double* h0, double* y, double* last_state,
                          int nthreads) {
    return oracle_selective_scan_grouped(Bsz, D, 1, N, L, u, delta, A, Bm, Cm, Dv, z, delta_bias,
                                         softplus, h0, y, last_state, nthreads);
}

/*
 * Mamba-2 SSD scan, written as its recurrence, one sequential loop per
 * (batch row b, head h).  The chunk size of the fast algorithm does not enter
 * the definition, so it is not a parameter here.
 *
 *   x, y       : (Bsz, L, H, P)
 *   dt         : (Bsz, L, H)      already positive
 *   A_head     : (H)              scalar A per head
 *   Bm, Cm     : (Bsz, L, G, N)   head h reads group h / (H / G)
 *   Dv         : (H)              nullable
 *   h0         : (Bsz, H, P, N)   nullable (zero initial state)
 *   last_state : (Bsz, H, P, N)   nullable
 *
 * For every t:
 *   a          = exp(dt * A_h)
 *   S[p][n]    = a * S[p][n] + dt * x[p] * B[n]
 *   y[p]       = sum_n C[n] * S[p][n] + D_h * x[p]
 */
int oracle_ssd(int64_t Bsz, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N,
               const double* x, const double* dt, const double* A_head,
               const double* Bm, const double* Cm, const double* Dv,
               const double* h0, double* y, double* last_state, int nthreads) {
    if (Bsz < 0 || L < 0 || H < 1 || P < 1 || G < 1 || N < 1 || H % G != 0) return -1;
    int64_t units = Bsz * H;
    int64_t heads_per_group = H / G;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t unit = 0; unit < units; ++unit) {
        int64_t b = unit / H, hh = unit % H;
        int64_t g = hh / heads_per_group;
        double* S = (double*)malloc((size_t)(P * N) * sizeof(double));
        if (!S) continue;
        for (int64_t i = 0; i < P * N; ++i)
            S[i] = h0 ? h0[((b * H + hh) * P) * N + i] : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            double dtv = dt[(b * L + t) * H + hh];
            double a = exp(dtv * A_head[hh]);
            const double* xr = x + ((b * L + t) * H + hh) * P;
            const double* br = Bm + ((b * L + t) * G + g) * N;
            const double* cr = Cm + ((b * L + t) * G + g) * N;
            double* yr = y + ((b * L + t) * H + hh) * P;
            for (int64_t p = 0; p < P; ++p) {
                double out = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    S[p * N + n] = a * S[p * N + n] + dtv * xr[p] * br[n];
                    out += cr[n] * S[p * N + n];
                }
                if (Dv) out += Dv[hh] * xr[p];
                yr[p] = out;
            }
        }
        if (last_state)
            for (int64_t i = 0; i < P * N; ++i)
                last_state[((b * H + hh) * P) * N + i] = S[i];
        free(S);
    }
    return 0;
}

/*
 * Causal depthwise convolution over t followed by SiLU, one sequential loop per
 * (batch row b, channel d):
 *
 *   x, u : (Bsz, D, L), t fastest;  w : (D, W);  bias : (D) nullable
 *   pre  = bias[d] + sum_{k=0}^{W-1} w[d,k] * x[b,d,t - (W-1) + k]   (x = 0 before t = 0)
 *   u    = pre / (1 + exp(-pre))
 */
int oracle_causal_conv1d_silu(int64_t Bsz, int64_t D, int64_t L, int64_t W, const double* x,
                              const double* w, const double* bias, double* u, int nthreads) {
    if (Bsz < 0 || D < 0 || L < 0 || W < 1) return -1;
    int64_t units = Bsz * D;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t unit = 0; unit < units; ++unit) {
        int64_t d = unit % D;
        const double* xr = x + unit * L;
        double* ur = u + unit * L;
        for (int64_t t = 0; t < L; ++t) {
            double pre = bias ? bias[d] : 0.0;
            for (int64_t k = 0; k < W; ++k) {
                int64_t s = t - (W - 1) + k;
                if (s >= 0) pre += w[d * W + k] * xr[s];
            }
            ur[t] = pre / (1.0 + exp(-pre));
        }
    }
    return 0;
}

/*
 * Backward (reverse-mode derivative) of the selective scan above, one unit
 * (b, d) at a time, in two sweeps: forward to keep every state h_t, then
 * backward in t with the adjoint state g_n = dL/dh_t[n].  With out_t the
 * scan's output and dout_t the incoming gradient:
 *
 *   pre_t   = sum_n C[n,t] h_t[n] + D u_t            (output before the gate)
 *   dz_t    = dout_t * pre_t * silu'(z_t),  dpre_t = dout_t * silu(z_t)
 *   g_n     = C[n,t] dpre_t + abar_{t+1}[n] g_n      (adjoint, from t = L-1 down)
 *   dC[n,t] += dpre_t h_t[n]            dD += dpre_t u_t
 *   dB[n,t] += g_n dl_t u_t             du_t = D dpre_t + sum_n g_n dl_t B[n,t]
 *   dA[n]   += g_n h_{t-1}[n] abar_t[n] dl_t
 *   ddl_t   = sum_n g_n (h_{t-1}[n] abar_t[n] A[n] + B[n,t] u_t)
 *   ddelta_t = ddl_t * sigmoid(delta_t + bias)  (softplus' ; identity if off)
 *   dbias  += ddelta_t
 *
 * dB, dC are summed over all channels of a batch row (B and C are shared),
 * dA, dD, dbias over batch rows.  All output arrays are overwritten.
 */
int oracle_selective_scan_bwd(int64_t Bsz, int64_t D, int64_t N, int64_t L,
                              const double* u, const double* delta, const double* A,
                              const double* Bm, const double* Cm, const double* Dv,
                              const double* z, const double* delta_bias, int softplus,
                              const double* dout, double* du, double* ddelta, double* dA,
                              double* dB, double* dC, double* dD, double* dz,
                              double* ddelta_bias) {
    if (Bsz < 0 || D < 0 || N < 1 || L < 0) return -1;
    for (int64_t i = 0; i < D * N; ++i) dA[i] = 0.0;
    for (int64_t i = 0; i < Bsz * N * L; ++i) { dB[i] = 0.0; dC[i] = 0.0; }
    if (dD) for (int64_t i = 0; i < D; ++i) dD[i] = 0.0;
    if (ddelta_bias) for (int64_t i = 0; i < D; ++i) ddelta_bias[i] = 0.0;
    double* hs = (double*)malloc((size_t)((L + 1) * N) * sizeof(double));
    double* dls = (double*)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
    double* g = (double*)malloc((size_t)N * sizeof(double));
    if (!hs || !dls || !g) { free(hs); free(dls); free(g); return -2; }
    for (int64_t b = 0; b < Bsz; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            const double* ur = u + (b * D + d) * L;
            const double* dr = delta + (b * D + d) * L;
            const double* zr = z ? z + (b * D + d) * L : NULL;
            const double* gr = dout + (b * D + d) * L;
            /* forward sweep: h_0 .. h_L (hs[t+1] is the state after step t) */
            for (int64_t n = 0; n < N; ++n) hs[n] = 0.0;
            for (int64_t t = 0; t < L; ++t) {
                double dl = dr[t] + (delta_bias ? delta_bias[d] : 0.0);
                if (softplus) dl = softplus_d(dl);
                dls[t] = dl;
                for (int64_t n = 0; n < N; ++n)
                    hs[(t + 1) * N + n] = exp(dl * A[d * N + n]) * hs[t * N + n] +
                                          dl * Bm[(b * N + n) * L + t] * ur[t];
            }
            /* backward sweep */
            for (int64_t n = 0; n < N; ++n) g[n] = 0.0;
            for (int64_t t = L - 1; t >= 0; --t) {
                double dl = dls[t];
                double pre = (Dv ? Dv[d] * ur[t] : 0.0);
                for (int64_t n = 0; n < N; ++n) pre += Cm[(b * N + n) * L + t] * hs[(t + 1) * N + n];
                double dpre = gr[t];
                if (zr) {
                    double sg = 1.0 / (1.0 + exp(-zr[t]));
                    dpre = gr[t] * zr[t] * sg;
                    dz[(b * D + d) * L + t] = gr[t] * pre * (sg + zr[t] * sg * (1.0 - sg));
                }
                if (Dv) dD[d] += dpre * ur[t];
                double ddl = 0.0, dut = Dv ? Dv[d] * dpre : 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    double c = Cm[(b * N + n) * L + t], bb = Bm[(b * N + n) * L + t];
                    double abar = exp(dl * A[d * N + n]);
                    /* g_n currently holds abar_{t+1} g_{t+1}; add this step's readout */
                    g[n] += c * dpre;
                    dC[(b * N + n) * L + t] += dpre * hs[(t + 1) * N + n];
                    dB[(b * N + n) * L + t] += g[n] * dl * ur[t];
                    dut += g[n] * dl * bb;
                    dA[d * N + n] += g[n] * hs[t * N + n] * abar * dl;
                    ddl += g[n] * (hs[t * N + n] * abar * A[d * N + n] + bb * ur[t]);
                    g[n] *= abar; /* carry to step t-1 */
                }
                du[(b * D + d) * L + t] = dut;
                double x = dr[t] + (delta_bias ? delta_bias[d] : 0.0);
                double dx = softplus ? ddl / (1.0 + exp(-x)) : ddl;
                ddelta[(b * D + d) * L + t] = dx;
                if (ddelta_bias) ddelta_bias[d] += dx;
            }
        }
    }
    free(hs);
    free(dls);
    free(g);
    return 0;
}
