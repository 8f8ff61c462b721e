/*
 * oracle.c -- plain, slow, float64 CPU statement of the Mamba selective scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only tests/, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no header, helper or constant with the CUDA
 * library; every formula below is written out from the method text.
 *
 * Sources (page title, section):
 *   [FS]  "Mamba state space model" explainer (fsdata.site), §2.2 (ssm_step,
 *         zero initial state, negative diagonal A) and §3.2 (selective_step:
 *         dt = softplus(.), A_bar = exp(dt*A), B_bar = dt*B,
 *         h = A_bar*h + B_bar*x, y = C.h + D*x).
 *   [FG]  "Mamba: linear-time sequence modelling with selective state spaces"
 *         tutorial (freeguideonline), §2.2 (exact zero-order hold), §3.1 and
 *         §4.2 step 2 (B_k, C_k, Delta_k input dependent, Delta bias inside
 *         the softplus), §4.3 (every channel has its own N-wide state),
 *         §4.1 / §4.2 step 5 (output multiplied by the gate branch).
 *   [XW]  "Mamba: Linear-Time Sequence Modeling with Selective State Spaces"
 *         summary (ai.xwebgame.com), "running it in PyTorch" block: the gate
 *         is SiLU of the residual branch; the branch that feeds the scan is a
 *         depthwise causal Conv1d (kernel 4, padding 3, first L outputs)
 *         followed by SiLU.
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes): y_t reads the state *after* the update with token t; D*u is added
 * before the gate and the gate multiplies the whole output; with softplus off
 * Delta = Delta_raw + bias; a NULL D, bias, z or h0 means "absent" (0, 0, no
 * gate, zero state).
 *
 * Every function is sequential in t, in the order of the pages' step
 * function.  Parity status: pinned (LTI convolution, running sum, brute-force
 * unrolling, geometric closed form, hand-worked cases, invariants; the
 * convolution branch against numpy's convolution; the backward pass against
 * central differences of the forward) -- see the -m "not gpu" tests.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_DISC_SIMPLE 0 /* B_bar = dt * B                     ([FS] §3.2) */
#define ORACLE_DISC_ZOH 1    /* B_bar = (exp(dt*A) - 1) / A * B    ([FG] §2.2) */

/* softplus(x) = log(1 + e^x), written in the overflow-free form
 * max(x, 0) + log1p(exp(-|x|)).  [FS] §3.2: dt = softplus(...) so dt > 0. */
double oracle_softplus(double x) {
    double ax = fabs(x);
    return (x > 0.0 ? x : 0.0) + log1p(exp(-ax));
}

/* SiLU(z) = z * sigmoid(z) = z / (1 + e^-z)  ([XW] PyTorch block, nn.SiLU). */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* Discretised input weight for one (state n, step t).
 *   simple:  dt * B                        ([FS] §3.2, B_bar = dt * sB(x))
 *   ZOH:     (dA)^-1 (exp(dA) - 1) dt B    ([FG] §2.2) with diagonal A, i.e.
 *            (exp(dt*A) - 1) / A * B; as A -> 0 this tends to dt * B, which
 *            is what is used when A == 0 exactly. */
static double b_bar(int disc, double dt, double a, double bnt) {
    if (disc == ORACLE_DISC_ZOH && a != 0.0) return expm1(dt * a) / a * bnt;
    return dt * bnt;
}

/* One channel (b, d), forward in time over t = 0..L-1, or backward in time
 * over t = L-1..0 when reverse != 0 (the reverse SSM that is stacked for
 * bidirectional context, [FS] §7 pitfalls table).
 *   u, dt_raw, z, y : [L]          z may be NULL (no gate)
 *   Bm, Cm          : [N][L]       row n holds B_{t,n} / C_{t,n}
 *   A               : [N]          A_{d,n}
 *   h               : [N]          in: initial state, out: final state
 */
static void scan_channel(int64_t L, int64_t N, const double *u,
                         const double *dt_raw, const double *z,
                         const double *Bm, const double *Cm, const double *A,
                         double Dd, double bias, int softplus_flag, int disc,
                         int reverse, double *h, double *y) {
    for (int64_t i = 0; i < L; ++i) {
        int64_t t = reverse ? (L - 1 - i) : i;
        /* [FG] §4.2 step 2: Delta = softplus(Linear(u) + bias). */
        double dt = dt_raw[t] + bias;
        if (softplus_flag) dt = oracle_softplus(dt);
        /* [FS] §3.2: h_new = A_bar * h + B_bar * x, per state n. */
        for (int64_t n = 0; n < N; ++n) {
            double a_bar = exp(dt * A[n]);
            h[n] = a_bar * h[n] + b_bar(disc, dt, A[n], Bm[n * L + t]) * u[t];
        }
        /* [FS] §3.2: y = C . h_new + D * x. */
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) acc += Cm[n * L + t] * h[n];
        acc += Dd * u[t];
        /* [FG] §4.1: the SSM path is multiplied by SiLU(gate branch). */
        if (z) acc *= silu(z[t]);
        y[t] = acc;
    }
}

/* Full selective scan over [Bsz, Dch, L] inputs.
 *   u, dt_raw, z, y : [Bsz][Dch][L]
 *   Bm, Cm          : [Bsz][N][L]   shared by every channel of batch b
 *   A               : [Dch][N]
 *   Dv, bias        : [Dch]         may be NULL (taken as 0)
 *   h0              : [Bsz][Dch][N] may be NULL (zero initial state)
 *   last_state      : [Bsz][Dch][N] may be NULL
 * Channels are independent ([FG] §4.3), so the (b, d) loop may run on
 * several host threads; each channel is still the plain sequential loop. */
void oracle_selective_scan(const double *u, const double *dt_raw,
                           const double *A, const double *Bm, const double *Cm,
                           const double *Dv, const double *z,
                           const double *bias, int softplus_flag, int disc,
                           int reverse, const double *h0, double *y,
                           double *last_state, int64_t Bsz, int64_t Dch,
                           int64_t L, int64_t N) {
    int64_t nch = Bsz * Dch;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t c = 0; c < nch; ++c) {
        int64_t b = c / Dch, d = c % Dch;
        double h[4096];
        for (int64_t n = 0; n < N; ++n) h[n] = h0 ? h0[c * N + n] : 0.0;
        scan_channel(L, N, u + c * L, dt_raw + c * L, z ? z + c * L : NULL,
                     Bm + b * N * L, Cm + b * N * L, A + d * N,
                     Dv ? Dv[d] : 0.0, bias ? bias[d] : 0.0, softplus_flag,
                     disc, reverse, h, y + c * L);
        if (last_state)
            for (int64_t n = 0; n < N; ++n) last_state[c * N + n] = h[n];
    }
}

/* One-token recurrent step for every (b, d): the selective_step of [FS] §3.2
 * applied to a stored state ("inference carries only the fixed-size state",
 * [FS] §5 table).
 *   state  : [Bsz][Dch][N] in/out
 *   u, dt_raw, z, y : [Bsz][Dch]      z may be NULL
 *   Bm, Cm : [Bsz][N]
 *   A      : [Dch][N];  Dv, bias : [Dch] may be NULL */
void oracle_state_update(double *state, const double *u, const double *dt_raw,
                         const double *A, const double *Bm, const double *Cm,
                         const double *Dv, const double *z, const double *bias,
                         int softplus_flag, int disc, double *y, int64_t Bsz,
                         int64_t Dch, int64_t N) {
    int64_t nch = Bsz * Dch;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < nch; ++c) {
        int64_t b = c / Dch, d = c % Dch;
        /* A single step is scan_channel with L = 1; B and C rows of length 1
         * are the batch's N-vectors read with stride 1, so gather them. */
        double Bcol[4096], Ccol[4096];
        for (int64_t n = 0; n < N; ++n) {
            Bcol[n] = Bm[b * N + n];
            Ccol[n] = Cm[b * N + n];
        }
        scan_channel(1, N, u + c, dt_raw + c, z ? z + c : NULL, Bcol, Ccol,
                     A + d * N, Dv ? Dv[d] : 0.0, bias ? bias[d] : 0.0,
                     softplus_flag, disc, 0, state + c * N, y + c);
    }
}

/* Number of host threads the parallel loops above will use. */
/*
 * Gradient of the forward selective scan (simple discretisation, forward in
 * time, zero initial state) for an upstream gradient dy of y.  The pages
 * measure training throughput but print no backward pass; this is the chain
 * rule applied to the [FS] §3.2 step as written in scan_channel, one channel
 * at a time: a forward sweep that keeps every state h_t, then a sweep from
 * t = L-1 down to 0 carrying dh = dLoss/dh_t:
 *   g = SiLU(z_t) (1 without a gate),  dyh = dy_t * g,
 *   dz_t = dy_t * yhat_t * SiLU'(z_t),  SiLU'(z) = s (1 + z (1 - s)), s = sigmoid(z)
 *   dD += dyh u_t;  du_t = D dyh;  dC_{t,n} += dyh h_t[n];  dh[n] += dyh C_{t,n}
 *   with a = exp(dt A_n), h_t = a h_{t-1} + dt B_{t,n} u_t:
 *     dB_{t,n} += dh[n] dt u_t;  du_t += dh[n] dt B_{t,n}
 *     ddt += dh[n] (B_{t,n} u_t + A_n a h_{t-1}[n]);  dA_n += dh[n] dt a h_{t-1}[n]
 *     dh[n] *= a
 *   ddt_raw_t = ddt * sigmoid(dt_raw_t + bias) (softplus) or ddt;  dbias += ddt_raw_t
 * dA [Dch][N], dB, dC [Bsz][N][L], dD, dbias [Dch] are sums (zeroed here);
 * du, ddt_raw [Bsz][Dch][L] and dz (when z is given) are per element.  Runs
 * sequentially (the sums span channels).
 */
void oracle_selective_scan_bwd(const double *u, const double *dt_raw,
                               const double *A, const double *Bm,
                               const double *Cm, const double *Dv,
                               const double *z, const double *bias,
                               int softplus_flag, const double *dy, double *du,
                               double *ddt_raw, double *dA, double *dB,
                               double *dC, double *dD, double *dz,
                               double *dbias, double *work, int64_t Bsz,
                               int64_t Dch, int64_t L, int64_t N) {
    /* work: (L + 1) * N + 2 * L + N doubles */
    memset(dA, 0, sizeof(double) * Dch * N);
    memset(dB, 0, sizeof(double) * Bsz * N * L);
    memset(dC, 0, sizeof(double) * Bsz * N * L);
    if (dD) memset(dD, 0, sizeof(double) * Dch);
    if (dbias) memset(dbias, 0, sizeof(double) * Dch);
    double *hs = work;                  /* hs[(t + 1) * N + n] = h_t[n], hs[n] = 0 */
    double *dts = hs + (L + 1) * N;     /* Delta_t */
    double *yh = dts + L;               /* y before the gate */
    double *dh = yh + L;                /* N */
    for (int64_t c = 0; c < Bsz * Dch; ++c) {
        const int64_t b = c / Dch, d = c % Dch;
        const double *uc = u + c * L, *rc = dt_raw + c * L, *zc = z ? z + c * L : NULL;
        const double *Bb = Bm + b * N * L, *Cb = Cm + b * N * L, *Ad = A + d * N;
        const double Dd = Dv ? Dv[d] : 0.0, bs = bias ? bias[d] : 0.0;
        for (int64_t n = 0; n < N; ++n) hs[n] = 0.0;
        for (int64_t t = 0; t < L; ++t) {
            double dt = rc[t] + bs;
            if (softplus_flag) dt = oracle_softplus(dt);
            dts[t] = dt;
            double acc = Dd * uc[t];
            for (int64_t n = 0; n < N; ++n) {
                const double h = exp(dt * Ad[n]) * hs[t * N + n] + dt * Bb[n * L + t] * uc[t];
                hs[(t + 1) * N + n] = h;
                acc += Cb[n * L + t] * h;
            }
            yh[t] = acc;
        }
        for (int64_t n = 0; n < N; ++n) dh[n] = 0.0;
        for (int64_t t = L - 1; t >= 0; --t) {
            const double dt = dts[t];
            double g = 1.0;
            if (zc) {
                const double sg = 1.0 / (1.0 + exp(-zc[t]));
                g = zc[t] * sg;
                dz[c * L + t] = dy[c * L + t] * yh[t] * sg * (1.0 + zc[t] * (1.0 - sg));
            }
            const double dyh = dy[c * L + t] * g;
            if (dD) dD[d] += dyh * uc[t];
            double dut = Dd * dyh, ddt = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                dC[(b * N + n) * L + t] += dyh * hs[(t + 1) * N + n];
                dh[n] += dyh * Cb[n * L + t];
            }
            for (int64_t n = 0; n < N; ++n) {
                const double a = exp(dt * Ad[n]), hp = hs[t * N + n];
                dB[(b * N + n) * L + t] += dh[n] * dt * uc[t];
                dut += dh[n] * dt * Bb[n * L + t];
                ddt += dh[n] * (Bb[n * L + t] * uc[t] + Ad[n] * a * hp);
                dA[d * N + n] += dh[n] * dt * a * hp;
                dh[n] *= a;
            }
            du[c * L + t] = dut;
            const double draw = softplus_flag ? ddt / (1.0 + exp(-(rc[t] + bs))) : ddt;
            ddt_raw[c * L + t] = draw;
            if (dbias) dbias[d] += draw;
        }
    }
}

/*
 * Depthwise causal convolution of width W followed by SiLU, per row
 * r = b * Dch + d of x [nrows][L]:
 *   pre_t = bias_d + sum_{k=0}^{W-1} w[d][k] * x_{t-(W-1)+k}   (x_s = 0 for s < 0)
 *   u_t   = silu_flag ? pre_t / (1 + exp(-pre_t)) : pre_t
 * [XW] "running it in PyTorch" block: nn.Conv1d(d_inner, d_inner,
 * kernel_size=d_conv (4), groups=d_inner, padding=d_conv-1), keep the first L
 * outputs, then nn.SiLU -- the branch that feeds the selective scan ([FS] §4:
 * causal convolution before the scan).  bias may be NULL (0).
 */
void oracle_causal_conv1d(const double *x, const double *w, const double *bias,
                          int silu_flag, double *u, int64_t nrows, int64_t Dch,
                          int64_t L, int64_t W) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t d = r % Dch;
        const double *xr = x + r * L;
        for (int64_t t = 0; t < L; ++t) {
            double pre = bias ? bias[d] : 0.0;
            for (int64_t k = 0; k < W; ++k) {
                const int64_t s = t - (W - 1) + k;
                if (s >= 0) pre += w[d * W + k] * xr[s];
            }
            u[r * L + t] = silu_flag ? silu(pre) : pre;
        }
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
