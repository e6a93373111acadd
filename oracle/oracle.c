/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the Mamba selective scan (S6)
 * and the single-token selective state update.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA path.
 *
 * What it computes (sources are web pages on the subject; cited by page title
 * and section):
 *   - "Deep dive into Mamba: architecture and implementation of selective
 *     state-space models" (aiattnstudio.link/posts/mamba), section 4.4
 *     (complete selective scan) and section 5.2 (the block's selective scan):
 *     dA = exp(delta*A), dB*u = delta*B*u, sequential h = dA*h + dB*u starting
 *     from a zero fp32 state, y = sum_n C*h, y += D*u.
 *   - "State space models and Mamba" (metaphor-xennon.pages.dev), the
 *     MambaBlock listing: delta = softplus(.) of the dt projection (whose
 *     Linear carries a bias, here dt_bias), the same scan with
 *     y = einsum('bdn,bn->bd', h, C), then the gate y * silu(z).
 *   - zero-order hold (the `zoh` flag): "State space models and Mamba",
 *     section on discretisation (zero-order hold), and "Deep dive into Mamba"
 *     section 12 (summary of the core formulas) give, with Abar = exp(delta*A),
 *     Bbar = A^-1 (exp(delta*A) - I) B.  A is diagonal here, so per state
 *     Bbar_n = (exp(delta*A_n) - 1) / A_n * B_n, which tends to delta*B_n as
 *     delta*A_n -> 0 (and equals it when A_n = 0).
 *   - Mamba paper-presentation article (hnwysp.cn/news/102080), section 3.2:
 *     h_t = a_t*h_{t-1} + b_t is associative, so the sequence can be cut into
 *     segments, each run serially from a zero state, keeping the segment-end
 *     state and the segment's transfer coefficient, then merged by a prefix
 *     scan (oracle_scan_fwd_segmented).
 *
 * Readings taken where the pages are silent or disagree (each is listed in
 * the design notes):
 *   - dB = delta*B (the form all listings use) unless `zoh` asks for the
 *     zero-order-hold B above.
 *   - y_t sees u_t: h_t = dA_t*h_{t-1} + dB_t*u_t, y_t = C_t . h_t.
 *   - softplus is applied exactly once, to dt_raw + dt_bias; it is evaluated
 *     exactly (no large-x threshold).
 *   - the D skip and the gate are applied in full precision, gate after skip.
 *   - the initial state is zero unless h0 is given (h0 is an extension used
 *     for split prefill; NULL means zero).
 *
 * All arrays are row-major and contiguous, fp64:
 *   u, dt_raw, z, out : (batch, L, d_inner)
 *   B, C              : (batch, L, d_state)
 *   A                 : (d_inner, d_state)
 *   D, dt_bias        : (d_inner)              nullable -> 0 / no bias
 *   h0, last_state    : (batch, d_inner, d_state) nullable
 *   z                 : nullable -> no gate
 * Built with -O2, no fast-math, libm exp/log1p.  OpenMP over the independent
 * (batch, channel) pairs; nthreads <= 0 means the OpenMP default.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(x) = log(1 + e^x), written so that neither branch overflows. */
double oracle_softplus(double x) {
    if (x > 0.0) return x + log1p(exp(-x));
    return log1p(exp(x));
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
double oracle_silu(double z) {
    return z / (1.0 + exp(-z));
}

static int set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) return nthreads;
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Number of OpenMP threads a call with `nthreads` would use. */
int oracle_threads(int nthreads) { return set_threads(nthreads); }

/*
 * One channel (b, d) over the time range [t0, t1), starting from state h
 * (length d_state, updated in place).  Writes out[b, t, d] when out != NULL.
 * This is the body shared by every oracle entry point below; it is the
 * sequential recurrence of the listings, one time step after the other.
 */
static void scan_channel(const double* u, const double* dt_raw, const double* A,
                         const double* B, const double* C, const double* D,
                         const double* z, const double* dt_bias, double* out,
                         double* h, int64_t b, int64_t d, int64_t t0, int64_t t1,
                         int64_t L, int64_t d_inner, int64_t d_state, int zoh) {
    const double bias = dt_bias ? dt_bias[d] : 0.0;
    const double skip = D ? D[d] : 0.0;
    for (int64_t t = t0; t < t1; ++t) {
        const int64_t i = (b * L + t) * d_inner + d;      /* (b, t, d) */
        const int64_t r = (b * L + t) * d_state;          /* (b, t, :) */
        const double delta = oracle_softplus(dt_raw[i] + bias);
        const double ut = u[i];
        double y = 0.0;
        for (int64_t n = 0; n < d_state; ++n) {
            const double x = delta * A[d * d_state + n];
            const double dA = exp(x);
            /* input gain: delta (Euler) or (exp(x) - 1) / A_n = delta * expm1(x) / x (ZOH) */
            const double gain = zoh ? (x != 0.0 ? delta * (expm1(x) / x) : delta) : delta;
            const double dBu = gain * B[r + n] * ut;
            h[n] = dA * h[n] + dBu;
            y += C[r + n] * h[n];
        }
        y += skip * ut;
        if (z) y *= oracle_silu(z[i]);
        if (out) out[i] = y;
    }
}

/*
 * Selective scan forward: every output y[b, t, d] and the final state.
 * Returns 0, or -1 on a bad size.
 */
int oracle_scan_fwd(const double* u, const double* dt_raw, const double* A,
                    const double* B, const double* C, const double* D,
                    const double* z, const double* dt_bias, const double* h0,
                    double* out, double* last_state, int64_t batch, int64_t L,
                    int64_t d_inner, int64_t d_state, int zoh, int nthreads) {
    if (batch < 0 || L < 0 || d_inner < 0 || d_state < 1) return -1;
    const int64_t nch = batch * d_inner;
    const int nt = set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t c = 0; c < nch; ++c) {
        const int64_t b = c / d_inner, d = c % d_inner;
        double* h = (double*)malloc((size_t)d_state * sizeof(double));
        for (int64_t n = 0; n < d_state; ++n)
            h[n] = h0 ? h0[c * d_state + n] : 0.0;
        scan_channel(u, dt_raw, A, B, C, D, z, dt_bias, out, h, b, d, 0, L, L,
                     d_inner, d_state, zoh);
        if (last_state)
            memcpy(last_state + c * d_state, h, (size_t)d_state * sizeof(double));
        free(h);
    }
    return 0;
}

/*
 * Single-token decode step: the same update with L = 1, the state read from
 * and written back to `state` (batch, d_inner, d_state) in place.  Inputs u,
 * dt_raw, z, out are (batch, d_inner); B, C are (batch, d_state).
 */
int oracle_state_update(double* state, const double* u, const double* dt_raw,
                        const double* A, const double* B, const double* C,
                        const double* D, const double* z, const double* dt_bias,
                        double* out, int64_t batch, int64_t d_inner,
                        int64_t d_state, int zoh, int nthreads) {
    if (batch < 0 || d_inner < 0 || d_state < 1) return -1;
    const int64_t nch = batch * d_inner;
    const int nt = set_threads(nthreads);
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t c = 0; c < nch; ++c) {
        const int64_t b = c / d_inner, d = c % d_inner;
        scan_channel(u, dt_raw, A, B, C, D, z, dt_bias, out, state + c * d_state,
                     b, d, 0, 1, 1, d_inner, d_state, zoh);
    }
    return 0;
}

/*
 * Segmented form of the same scan (presentation article, section 3.2; the
 * chunk + recompute scheme of "Deep dive into Mamba" section 7.3):
 *   1. cut [0, L) into segments of `seg` steps;
 *   2. run each segment serially from a zero state, keeping its end state
 *      b_k and its transfer coefficient a_k = prod of dA over the segment;
 *   3. merge the segments in order with the associative combine
 *      (a1, b1) then (a2, b2)  ->  (a2*a1, a2*b1 + b2), which gives the
 *      state entering every segment;
 *   4. rerun every segment from its entering state to emit the outputs.
 * It must agree with oracle_scan_fwd up to fp64 rounding (Euler input
 * matrix, zero initial state).
 */
int oracle_scan_fwd_segmented(const double* u, const double* dt_raw,
                              const double* A, const double* B, const double* C,
                              const double* D, const double* z,
                              const double* dt_bias, double* out,
                              double* last_state, int64_t batch, int64_t L,
                              int64_t d_inner, int64_t d_state, int64_t seg,
                              int nthreads) {
    if (batch < 0 || L < 0 || d_inner < 0 || d_state < 1 || seg < 1) return -1;
    const int64_t nseg = (L + seg - 1) / seg;
    const int64_t nch = batch * d_inner;
    const int nt = set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t c = 0; c < nch; ++c) {
        const int64_t b = c / d_inner, d = c % d_inner;
        const double bias = dt_bias ? dt_bias[d] : 0.0;
        double* a_seg = (double*)calloc((size_t)(nseg * d_state) + 1, sizeof(double));
        double* b_seg = (double*)calloc((size_t)(nseg * d_state) + 1, sizeof(double));
        double* h = (double*)calloc((size_t)d_state, sizeof(double));
        /* step 2: per-segment summary from a zero state */
        for (int64_t k = 0; k < nseg; ++k) {
            const int64_t t0 = k * seg, t1 = (t0 + seg < L) ? t0 + seg : L;
            for (int64_t n = 0; n < d_state; ++n) {
                double a = 1.0, s = 0.0;
                for (int64_t t = t0; t < t1; ++t) {
                    const int64_t i = (b * L + t) * d_inner + d;
                    const int64_t r = (b * L + t) * d_state;
                    const double delta = oracle_softplus(dt_raw[i] + bias);
                    const double dA = exp(delta * A[d * d_state + n]);
                    s = dA * s + delta * B[r + n] * u[i];
                    a = dA * a;
                }
                a_seg[k * d_state + n] = a;
                b_seg[k * d_state + n] = s;
            }
        }
        /* step 3: in-order merge; h holds the state entering segment k */
        for (int64_t k = 0; k < nseg; ++k) {
            const int64_t t0 = k * seg, t1 = (t0 + seg < L) ? t0 + seg : L;
            double* hk = (double*)malloc((size_t)d_state * sizeof(double));
            memcpy(hk, h, (size_t)d_state * sizeof(double));
            /* step 4: rerun the segment from its entering state */
            scan_channel(u, dt_raw, A, B, C, D, z, dt_bias, out, hk, b, d, t0,
                         t1, L, d_inner, d_state, 0);
            free(hk);
            for (int64_t n = 0; n < d_state; ++n)
                h[n] = a_seg[k * d_state + n] * h[n] + b_seg[k * d_state + n];
        }
        if (last_state)
            memcpy(last_state + c * d_state, h, (size_t)d_state * sizeof(double));
        free(a_seg);
        free(b_seg);
        free(h);
    }
    return 0;
}

/*
 * Causal depthwise conv1d before the scan ("Deep dive into Mamba" section 3.2,
 * the block's Conv1d with kernel d_conv, padding d_conv - 1, one group per
 * channel, with bias; section 5.2 and the MambaBlock of "State space models
 * and Mamba": the first L outputs are kept, then SiLU).  PyTorch's Conv1d is a
 * cross-correlation, so with the left padding it reads, for output step t,
 * the inputs t-(d_conv-1) ... t:
 *     out[b,t,d] = bias[d] + sum_k w[d,k] * x[b, t - (d_conv-1) + k, d]
 *     out        = silu(out) when `silu` is set.
 * Inputs before t = 0 are zero, or, when state_in is given, the d_conv-1
 * inputs that preceded the sequence (state_in[b,d,j] is input step
 * j - (d_conv-1), oldest first).  state_out, when given, receives the last
 * d_conv-1 inputs in the same layout (the state a decode step continues
 * from).  x, out: (batch, L, d_inner); w: (d_inner, d_conv); bias (d_inner)
 * nullable; state_in, state_out: (batch, d_inner, d_conv-1) nullable.
 */
int oracle_causal_conv1d(const double* x, const double* w, const double* bias,
                         const double* state_in, double* out, double* state_out,
                         int64_t batch, int64_t L, int64_t d_inner, int64_t d_conv,
                         int silu, int nthreads) {
    if (batch < 0 || L < 0 || d_inner < 0 || d_conv < 1) return -1;
    const int64_t nch = batch * d_inner, H = d_conv - 1;
    const int nt = set_threads(nthreads);
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t c = 0; c < nch; ++c) {
        const int64_t b = c / d_inner, d = c % d_inner;
        /* the input at step s, for s in [-H, L) */
        #define XAT(s) ((s) >= 0 ? x[(b * L + (s)) * d_inner + d] \
                                 : (state_in ? state_in[c * H + H + (s)] : 0.0))
        for (int64_t t = 0; t < L; ++t) {
            double acc = bias ? bias[d] : 0.0;
            for (int64_t k = 0; k < d_conv; ++k)
                acc += w[d * d_conv + k] * XAT(t - H + k);
            out[(b * L + t) * d_inner + d] = silu ? oracle_silu(acc) : acc;
        }
        if (state_out)
            for (int64_t j = 0; j < H; ++j) state_out[c * H + j] = XAT(L - H + j);
        #undef XAT
    }
    return 0;
}

/*
 * One decode step of the same conv: the window is the d_conv-1 stored inputs
 * followed by x[b,d]; out[b,d] = (silu of) bias + sum_k w[d,k] * window[k];
 * then the state drops its oldest input and appends x (in place).
 * state: (batch, d_inner, d_conv-1); x, out: (batch, d_inner).
 */
int oracle_conv1d_update(double* state, const double* x, const double* w,
                         const double* bias, double* out, int64_t batch,
                         int64_t d_inner, int64_t d_conv, int silu, int nthreads) {
    if (batch < 0 || d_inner < 0 || d_conv < 1) return -1;
    const int64_t nch = batch * d_inner, H = d_conv - 1;
    const int nt = set_threads(nthreads);
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t c = 0; c < nch; ++c) {
        const int64_t d = c % d_inner;
        double* st = state + c * H;
        double acc = bias ? bias[d] : 0.0;
        for (int64_t k = 0; k < H; ++k) acc += w[d * d_conv + k] * st[k];
        acc += w[d * d_conv + H] * x[c];
        out[c] = silu ? oracle_silu(acc) : acc;
        for (int64_t k = 0; k + 1 < H; ++k) st[k] = st[k + 1];
        if (H > 0) st[H - 1] = x[c];
    }
    return 0;
}

/*
 * Mamba-3 exponential-trapezoid scan (the Mamba series article, section 2.1,
 * "exponential-trapezoidal discretisation"): the input term mixes the
 * previous and the current step's B*x with a data-dependent lambda in [0, 1]:
 *     h_t = exp(delta_t*A) h_{t-1} + (1 - lambda_t) delta_t B_{t-1} x_{t-1}
 *                                  + lambda_t delta_t B_t x_t
 * (x = u here; the formula as printed, without a decay on the t-1 term).  The
 * rest of the S6 step is unchanged: delta = softplus(dt + dt_bias),
 * y = C.h + D*u, gate.  B_{-1} x_{-1} is u_prev[b,d] * B_prev[b,n] when both
 * are given (the step before the sequence, for split prefill and decode),
 * zero otherwise.  lam: (batch, L, d_inner); u_prev: (batch, d_inner);
 * B_prev: (batch, d_state).
 */
static void trap_channel(const double* u, const double* dt_raw, const double* lam,
                         const double* A, const double* B, const double* C,
                         const double* D, const double* z, const double* dt_bias,
                         double* out, double* h, double* bx, int64_t b, int64_t d,
                         int64_t L, int64_t d_inner, int64_t d_state) {
    const double bias = dt_bias ? dt_bias[d] : 0.0;
    const double skip = D ? D[d] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
        const int64_t i = (b * L + t) * d_inner + d;
        const int64_t r = (b * L + t) * d_state;
        const double delta = oracle_softplus(dt_raw[i] + bias);
        const double lt = lam[i], ut = u[i];
        double y = 0.0;
        for (int64_t n = 0; n < d_state; ++n) {
            const double dA = exp(delta * A[d * d_state + n]);
            h[n] = dA * h[n] + (1.0 - lt) * delta * bx[n] + lt * delta * B[r + n] * ut;
            bx[n] = B[r + n] * ut;                           /* B_{t-1} x_{t-1} next */
            y += C[r + n] * h[n];
        }
        y += skip * ut;
        if (z) y *= oracle_silu(z[i]);
        if (out) out[i] = y;
    }
}

int oracle_scan_fwd_trap(const double* u, const double* dt_raw, const double* lam,
                         const double* A, const double* B, const double* C,
                         const double* D, const double* z, const double* dt_bias,
                         const double* h0, const double* u_prev, const double* B_prev,
                         double* out, double* last_state, int64_t batch, int64_t L,
                         int64_t d_inner, int64_t d_state, int nthreads) {
    if (batch < 0 || L < 0 || d_inner < 0 || d_state < 1) return -1;
    const int64_t nch = batch * d_inner;
    const int nt = set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t c = 0; c < nch; ++c) {
        const int64_t b = c / d_inner, d = c % d_inner;
        double* h = (double*)malloc((size_t)d_state * 2 * sizeof(double));
        double* bx = h + d_state;
        for (int64_t n = 0; n < d_state; ++n) {
            h[n] = h0 ? h0[c * d_state + n] : 0.0;
            bx[n] = (u_prev && B_prev) ? B_prev[b * d_state + n] * u_prev[c] : 0.0;
        }
        trap_channel(u, dt_raw, lam, A, B, C, D, z, dt_bias, out, h, bx, b, d, L,
                     d_inner, d_state);
        if (last_state)
            memcpy(last_state + c * d_state, h, (size_t)d_state * sizeof(double));
        free(h);
    }
    return 0;
}

/*
 * One decode token of the trapezoid scan: the state is read and written in
 * place; u_prev / B_prev are the previous token's u and B (nullable: zero).
 */
int oracle_state_update_trap(double* state, const double* u_prev, const double* B_prev,
                             const double* u, const double* dt_raw, const double* lam,
                             const double* A, const double* B, const double* C,
                             const double* D, const double* z, const double* dt_bias,
                             double* out, int64_t batch, int64_t d_inner,
                             int64_t d_state, int nthreads) {
    if (batch < 0 || d_inner < 0 || d_state < 1) return -1;
    const int64_t nch = batch * d_inner;
    const int nt = set_threads(nthreads);
#pragma omp parallel for schedule(static) num_threads(nt)
    for (int64_t c = 0; c < nch; ++c) {
        const int64_t b = c / d_inner, d = c % d_inner;
        double* bx = (double*)malloc((size_t)d_state * sizeof(double));
        for (int64_t n = 0; n < d_state; ++n)
            bx[n] = (u_prev && B_prev) ? B_prev[b * d_state + n] * u_prev[c] : 0.0;
        trap_channel(u, dt_raw, lam, A, B, C, D, z, dt_bias, out, state + c * d_state, bx,
                     b, d, 1, d_inner, d_state);
        free(bx);
    }
    return 0;
}

/*
 * Backward pass of the selective scan (Euler form): the gradients of a loss
 * J(out, last_state) with respect to every input, given dout = dJ/dout and
 * dlast = dJ/dlast_state (nullable: zero).  The pages say the backward
 * recomputes the states rather than storing them (the chunk + recompute
 * scheme of "Deep dive into Mamba" section 7.3; the Mamba series article,
 * section 3: a custom kernel differentiates the scan); this oracle simply
 * keeps every state of a channel and runs the adjoint recurrence backwards:
 *     dy_t  = dout_t * silu(z_t)              (dout_t without the gate)
 *     dh_t  = C_t dy_t + exp(delta_{t+1} A) dh_{t+1}      (dh_{L-1} += dlast)
 *     with a_t = exp(delta_t A), from h_t = a_t h_{t-1} + delta_t B_t u_t:
 *       dA      += dh_t h_{t-1} a_t delta_t
 *       ddelta_t = sum_n dh_t h_{t-1} a_t A + dh_t B_t u_t
 *       dB_t    += dh_t delta_t u_t        dC_t += dy_t h_t
 *       du_t     = dy_t D + sum_n dh_t delta_t B_t
 *     ddt_t = ddelta_t sigmoid(dt_t + dt_bias)  (softplus' = sigmoid)
 *     dz_t  = dout_t y_t silu'(z_t),  silu'(z) = s (1 + z (1 - s)), s = sigmoid(z)
 *     dD += dy_t u_t,  ddt_bias += ddt_t,  dh0 = a_0 dh_0.
 * Shapes as the forward; dA: (d_inner, d_state); dB, dC: (batch, L,
 * d_state); dD, ddt_bias: (d_inner); dh0: (batch, d_inner, d_state).  Every
 * output is overwritten.  Sequential (the parameter gradients are sums over
 * channels and steps).
 */
static double oracle_sigmoid(double x) {
    if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
    const double e = exp(x);
    return e / (1.0 + e);
}

int oracle_scan_bwd(const double* u, const double* dt_raw, const double* A,
                    const double* B, const double* C, const double* D,
                    const double* z, const double* dt_bias, const double* h0,
                    const double* dout, const double* dlast, double* du,
                    double* ddt, double* dA, double* dB, double* dC, double* dD,
                    double* dz, double* ddt_bias, double* dh0, int64_t batch,
                    int64_t L, int64_t d_inner, int64_t d_state) {
    if (batch < 0 || L < 0 || d_inner < 0 || d_state < 1) return -1;
    const int64_t N = d_state;
    memset(dA, 0, (size_t)(d_inner * N) * sizeof(double));
    memset(dB, 0, (size_t)(batch * L * N) * sizeof(double));
    memset(dC, 0, (size_t)(batch * L * N) * sizeof(double));
    memset(dD, 0, (size_t)d_inner * sizeof(double));
    memset(ddt_bias, 0, (size_t)d_inner * sizeof(double));
    double* hs = (double*)malloc((size_t)((L + 1) * N) * sizeof(double));
    double* ys = (double*)malloc((size_t)(L + 1) * sizeof(double));
    double* dh = (double*)malloc((size_t)N * sizeof(double));
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < d_inner; ++d) {
            const int64_t c = b * d_inner + d;
            const double bias = dt_bias ? dt_bias[d] : 0.0;
            const double skip = D ? D[d] : 0.0;
            /* forward, keeping h_{t} in hs[t + 1] and y_t (before the gate) */
            for (int64_t n = 0; n < N; ++n) hs[n] = h0 ? h0[c * N + n] : 0.0;
            for (int64_t t = 0; t < L; ++t) {
                const int64_t i = (b * L + t) * d_inner + d, r = (b * L + t) * N;
                const double delta = oracle_softplus(dt_raw[i] + bias);
                double y = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double a = exp(delta * A[d * N + n]);
                    hs[(t + 1) * N + n] = a * hs[t * N + n] + delta * B[r + n] * u[i];
                    y += C[r + n] * hs[(t + 1) * N + n];
                }
                ys[t] = y + skip * u[i];
            }
            /* backward */
            for (int64_t n = 0; n < N; ++n) dh[n] = dlast ? dlast[c * N + n] : 0.0;
            for (int64_t t = L - 1; t >= 0; --t) {
                const int64_t i = (b * L + t) * d_inner + d, r = (b * L + t) * N;
                const double x = dt_raw[i] + bias;
                const double delta = oracle_softplus(x);
                double dy = dout[i];
                if (z) {
                    const double s = oracle_sigmoid(z[i]);
                    dy = dout[i] * z[i] * s;
                    dz[i] = dout[i] * ys[t] * s * (1.0 + z[i] * (1.0 - s));
                }
                dD[d] += dy * u[i];
                double dui = dy * skip, ddelta = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double a = exp(delta * A[d * N + n]);
                    dh[n] += C[r + n] * dy;
                    dC[r + n] += dy * hs[(t + 1) * N + n];
                    const double da = dh[n] * hs[t * N + n];
                    dA[d * N + n] += da * a * delta;
                    ddelta += da * a * A[d * N + n] + dh[n] * B[r + n] * u[i];
                    dB[r + n] += dh[n] * delta * u[i];
                    dui += dh[n] * delta * B[r + n];
                    dh[n] *= a;
                }
                du[i] = dui;
                ddt[i] = ddelta * oracle_sigmoid(x);
                ddt_bias[d] += ddt[i];
            }
            if (dh0)
                for (int64_t n = 0; n < N; ++n) dh0[c * N + n] = dh[n];
        }
    }
    free(hs);
    free(ys);
    free(dh);
    return 0;
}
