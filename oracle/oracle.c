/*
 * Oracle for the selective scan — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the selective state space layer computes.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load this library; the product
 * path never does.  It shares no code, header or constant with the CUDA path.
 *
 * Sources (pages on "Mamba: Linear-Time Sequence Modeling with Selective State Spaces"):
 *  - continuous SSM h'(t) = A h(t) + B x(t), y(t) = C h(t) + D x(t), with D a skip connection:
 *    visual guide to Mamba and SSMs, section 2.2 ("What is a state space model?").
 *  - discretisation with a learnable step size Delta (zero-order hold): same guide, section 2.3.
 *    Its formula did not survive extraction; this oracle takes the reading
 *    Abar = exp(Delta * A), Bbar * x = Delta * B * x.
 *  - recurrence h_k = Abar h_{k-1} + Bbar x_k, y_k = C h_k: same guide, section 2.4.
 *  - selection: B, C and Delta vary with batch and position, A does not: same guide, section 3.2
 *    (and the news write-up's "selection mechanism" section).
 *  - exact zero-order hold (optional, flag zoh): the input is held constant over each step of
 *    length Delta (visual guide, section 2.3).  For a diagonal A the held-input solution of
 *    h' = A h + B x over one step gives Abar = exp(Delta A) and Bbar = (exp(Delta A) - 1) / A * B,
 *    which tends to Delta * B as A -> 0.
 *  - gradients (reverse mode, states recomputed rather than stored by the kernels; this oracle
 *    keeps them): visual guide, section 3.4 ("recomputation").  oracle_scan_bwd_rows applies the
 *    chain rule to the forward definition above, step by step in reverse time order.
 *  - Delta = softplus(delta + delta_bias) when softplus_flag is set, else delta + delta_bias;
 *    output gated by silu(z) = z * sigmoid(z), applied to C h + D x.  The pages leave the
 *    parametrisation of Delta and the gate open; these are the readings used throughout.
 *
 * Everything is evaluated in double precision, strictly in time order, one channel at a time,
 * with no reassociation.  Inputs stored as fp32 or bf16 are widened exactly to double.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2 /* inputs already in double (e.g. a convolution computed by this oracle) */

static double widen(const void* p, long long i, int dtype) {
    if (dtype == ORACLE_F64) return ((const double*)p)[i];
    if (dtype == ORACLE_BF16) {
        uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)p)[i];
}

/* softplus(x) = log(1 + e^x), written so that neither branch overflows. */
static double softplus(double x) {
    if (x > 0.0) return x + log1p(exp(-x));
    return log1p(exp(x));
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^{-z}). */
static double silu(double z) { return z / (1.0 + exp(-z)); }

static double step_size(double raw, double bias, int softplus_flag) {
    double d = raw + bias;
    return softplus_flag ? softplus(d) : d;
}

/* Factor k with Bbar * x = k * B * x.  Simplified reading: k = Delta.  Exact zero-order hold:
 * k = (exp(Delta a) - 1) / a, the integral of exp(a s) over s in [0, Delta]; k = Delta at a = 0. */
static double bbar_factor(double dt, double a, int zoh) {
    if (!zoh || a == 0.0) return dt;
    return expm1(dt * a) / a;
}

int oracle_version(void) { return 2; }

/*
 * Forward selective scan over a list of channels ("rows").
 *
 * Row i is channel (row_b[i], row_d[i]).  u_rows, delta_rows, z_rows hold that channel's inputs,
 * [nrows, seqlen] in in_dtype (fp32, bf16, or double: ORACLE_F64 takes values that are already
 * double, such as this oracle's own convolution output).  A [dim, dstate] fp32, D and delta_bias [dim] fp32 (either may be
 * NULL for zero); B, C [batch, dstate, seqlen] in in_dtype; z_rows may be NULL (no gate).
 * h0_rows [nrows, dstate] is the initial state (NULL = zero).
 * Outputs: y_rows [nrows, seqlen] and state_rows [nrows, dstate] (may be NULL), fp64.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_scan_rows_ex(long long nrows, const int* row_b, const int* row_d, int dim, int dstate,
                        long long seqlen, int in_dtype, const void* u_rows, const void* delta_rows,
                        const void* z_rows, const float* A, const float* D, const float* delta_bias,
                        const void* B, const void* C, int softplus_flag, int zoh,
                        const double* h0_rows, double* y_rows, double* state_rows, int nthreads) {
    if (nrows < 0 || dim <= 0 || dstate <= 0 || dstate > 256 || seqlen < 0) return -1;
    if (nrows > 0 && (!row_b || !row_d || !u_rows || !delta_rows || !A || !B || !C || !y_rows))
        return -1;
    if (in_dtype != ORACLE_F32 && in_dtype != ORACLE_BF16 && in_dtype != ORACLE_F64) return -1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long long i = 0; i < nrows; ++i) {
        const int b = row_b[i], d = row_d[i];
        double h[256];
        double a_n[256];
        const int N = dstate;
        for (int n = 0; n < N; ++n) h[n] = h0_rows ? h0_rows[i * dstate + n] : 0.0;
        const double Dd = D ? (double)D[d] : 0.0;
        const double bias = delta_bias ? (double)delta_bias[d] : 0.0;
        for (int n = 0; n < N; ++n) a_n[n] = (double)A[(long long)d * dstate + n];
        for (long long t = 0; t < seqlen; ++t) {
            const double x = widen(u_rows, i * seqlen + t, in_dtype);
            const double dt = step_size(widen(delta_rows, i * seqlen + t, in_dtype), bias, softplus_flag);
            double acc = 0.0;
            for (int n = 0; n < N; ++n) {
                const long long bc = ((long long)b * dstate + n) * seqlen + t;
                const double Abar = exp(dt * a_n[n]);
                const double Bbar_x = bbar_factor(dt, a_n[n], zoh) * widen(B, bc, in_dtype) * x;
                h[n] = Abar * h[n] + Bbar_x;
                acc += widen(C, bc, in_dtype) * h[n];
            }
            double y = acc + Dd * x;
            if (z_rows) y *= silu(widen(z_rows, i * seqlen + t, in_dtype));
            y_rows[i * seqlen + t] = y;
        }
        if (state_rows)
            for (int n = 0; n < N; ++n) state_rows[i * dstate + n] = h[n];
    }
    return 0;
}

/* The forward scan with the simplified discretisation Bbar = Delta * B (see oracle_scan_rows_ex). */
int oracle_scan_rows(long long nrows, const int* row_b, const int* row_d, int dim, int dstate,
                     long long seqlen, int in_dtype, const void* u_rows, const void* delta_rows,
                     const void* z_rows, const float* A, const float* D, const float* delta_bias,
                     const void* B, const void* C, int softplus_flag, const double* h0_rows,
                     double* y_rows, double* state_rows, int nthreads) {
    return oracle_scan_rows_ex(nrows, row_b, row_d, dim, dstate, seqlen, in_dtype, u_rows,
                               delta_rows, z_rows, A, D, delta_bias, B, C, softplus_flag, 0,
                               h0_rows, y_rows, state_rows, nthreads);
}

/*
 * One recurrent (decoding) step for a list of channels: the same body as one time step of the
 * scan, starting from the given state.  state_rows [nrows, dstate] fp64 is updated in place.
 * x_rows, delta_rows, z_rows [nrows] in in_dtype; B, C [batch, dstate] in in_dtype.
 * y_rows [nrows] fp64.  Constant work per token, no cache of past tokens (news write-up,
 * "architecture" section; visual guide section 1.4 on recurrent inference).
 */
int oracle_state_step_rows_ex(long long nrows, const int* row_b, const int* row_d, int dim,
                              int dstate, int in_dtype, double* state_rows, const void* x_rows,
                              const void* delta_rows, const void* z_rows, const float* A,
                              const float* D, const float* delta_bias, const void* B, const void* C,
                              int softplus_flag, int zoh, double* y_rows, int nthreads) {
    if (nrows < 0 || dim <= 0 || dstate <= 0 || dstate > 256) return -1;
    if (nrows > 0 && (!row_b || !row_d || !state_rows || !x_rows || !delta_rows || !A || !B || !C ||
                      !y_rows))
        return -1;
    if (in_dtype != ORACLE_F32 && in_dtype != ORACLE_BF16) return -1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (long long i = 0; i < nrows; ++i) {
        const int b = row_b[i], d = row_d[i];
        double* h = state_rows + i * dstate;
        const double x = widen(x_rows, i, in_dtype);
        const double bias = delta_bias ? (double)delta_bias[d] : 0.0;
        const double dt = step_size(widen(delta_rows, i, in_dtype), bias, softplus_flag);
        double acc = 0.0;
        for (int n = 0; n < dstate; ++n) {
            const long long bc = (long long)b * dstate + n;
            const double a = (double)A[(long long)d * dstate + n];
            const double Abar = exp(dt * a);
            h[n] = Abar * h[n] + bbar_factor(dt, a, zoh) * widen(B, bc, in_dtype) * x;
            acc += widen(C, bc, in_dtype) * h[n];
        }
        double y = acc + (D ? (double)D[d] : 0.0) * x;
        if (z_rows) y *= silu(widen(z_rows, i, in_dtype));
        y_rows[i] = y;
    }
    return 0;
}

/* One decoding step with the simplified discretisation Bbar = Delta * B. */
int oracle_state_step_rows(long long nrows, const int* row_b, const int* row_d, int dim, int dstate,
                           int in_dtype, double* state_rows, const void* x_rows,
                           const void* delta_rows, const void* z_rows, const float* A,
                           const float* D, const float* delta_bias, const void* B, const void* C,
                           int softplus_flag, double* y_rows, int nthreads) {
    return oracle_state_step_rows_ex(nrows, row_b, row_d, dim, dstate, in_dtype, state_rows, x_rows,
                                     delta_rows, z_rows, A, D, delta_bias, B, C, softplus_flag, 0,
                                     y_rows, nthreads);
}

/* d silu / dz = sigmoid(z) * (1 + z * (1 - sigmoid(z))). */
static double silu_grad(double z) {
    const double sg = 1.0 / (1.0 + exp(-z));
    return sg * (1.0 + z * (1.0 - sg));
}

/* d softplus / dx = sigmoid(x). */
static double softplus_grad(double x) { return 1.0 / (1.0 + exp(-x)); }

/*
 * Gradients of the forward scan for a list of channels, by reverse-mode differentiation of
 * oracle_scan_rows_ex's definition.  The loss is sum_t dy[t] * y[t] + sum_n dstate[n] * h_{L-1}[n]
 * per channel, so dy_rows [nrows, seqlen] and dstate_rows [nrows, dstate] (NULL = 0) are the
 * gradients arriving at y and at last_state.
 *
 * Inputs as for oracle_scan_rows_ex (in_dtype ORACLE_F64 included: inputs already in double, such
 * as this oracle's own convolution output).  Outputs, all fp64:
 *   per channel (overwritten): du_rows, ddelta_rows [nrows, seqlen]; dz_rows [nrows, seqlen]
 *     (only when z_rows is given; may be NULL); dh0_rows [nrows, dstate] (may be NULL);
 *   accumulated with += over the channels (the caller zeroes them): dA [dim, dstate],
 *     dD [dim], dbias [dim] (each may be NULL), dB, dC [batch, dstate, seqlen].
 * The forward states are kept in memory here; only the kernels recompute them.
 * Returns 0, -1 on a bad argument, -2 when memory runs out.
 */
int oracle_scan_bwd_rows(long long nrows, const int* row_b, const int* row_d, int batch, int dim,
                         int dstate, long long seqlen, int in_dtype, const void* u_rows,
                         const void* delta_rows, const void* z_rows, const float* A,
                         const float* D, const float* delta_bias, const void* B, const void* C,
                         int softplus_flag, int zoh, const double* h0_rows, const double* dy_rows,
                         const double* dstate_rows, double* du_rows, double* ddelta_rows,
                         double* dz_rows, double* dh0_rows, double* dA, double* dD, double* dbias,
                         double* dB, double* dC, int nthreads) {
    if (nrows < 0 || batch <= 0 || dim <= 0 || dstate <= 0 || dstate > 256 || seqlen < 0) return -1;
    if (nrows > 0 && (!row_b || !row_d || !u_rows || !delta_rows || !A || !B || !C || !dy_rows ||
                      !du_rows || !ddelta_rows || !dB || !dC))
        return -1;
    if (in_dtype != ORACLE_F32 && in_dtype != ORACLE_BF16 && in_dtype != ORACLE_F64) return -1;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long long i = 0; i < nrows; ++i) {
        const int b = row_b[i], d = row_d[i];
        const int N = dstate;
        const long long L = seqlen;
        /* hist[(t + 1) * N + n] = h_t[n], hist[0..N) = initial state */
        double* hist = (double*)malloc(sizeof(double) * (size_t)(L + 1) * (size_t)N);
        double* gB = (double*)calloc((size_t)N * (size_t)(L > 0 ? L : 1), sizeof(double));
        double* gC = (double*)calloc((size_t)N * (size_t)(L > 0 ? L : 1), sizeof(double));
        if (!hist || !gB || !gC) {
            free(hist); free(gB); free(gC);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
            continue;
        }
        double a_n[256], mu[256], gA[256];
        const double Dd = D ? (double)D[d] : 0.0;
        const double bias = delta_bias ? (double)delta_bias[d] : 0.0;
        for (int n = 0; n < N; ++n) {
            a_n[n] = (double)A[(long long)d * dstate + n];
            hist[n] = h0_rows ? h0_rows[i * dstate + n] : 0.0;
            mu[n] = dstate_rows ? dstate_rows[i * dstate + n] : 0.0;
            gA[n] = 0.0;
        }
        /* forward, keeping every state */
        for (long long t = 0; t < L; ++t) {
            const double x = widen(u_rows, i * L + t, in_dtype);
            const double dt = step_size(widen(delta_rows, i * L + t, in_dtype), bias, softplus_flag);
            for (int n = 0; n < N; ++n) {
                const long long bc = ((long long)b * dstate + n) * L + t;
                const double decay = exp(dt * a_n[n]);
                hist[(t + 1) * N + n] = decay * hist[t * N + n] +
                                        bbar_factor(dt, a_n[n], zoh) * widen(B, bc, in_dtype) * x;
            }
        }
        /* reverse: mu[n] is the gradient reaching h_t[n] from steps after t */
        double gD = 0.0, gbias = 0.0;
        for (long long t = L - 1; t >= 0; --t) {
            const double x = widen(u_rows, i * L + t, in_dtype);
            const double s = widen(delta_rows, i * L + t, in_dtype) + bias;
            const double dt = softplus_flag ? softplus(s) : s;
            const double* h_t = hist + (t + 1) * N;
            const double* h_prev = hist + t * N;
            double ypre = Dd * x;
            for (int n = 0; n < N; ++n)
                ypre += widen(C, ((long long)b * dstate + n) * L + t, in_dtype) * h_t[n];
            double gate = 1.0;
            if (z_rows) {
                const double zz = widen(z_rows, i * L + t, in_dtype);
                gate = silu(zz);
                if (dz_rows) dz_rows[i * L + t] = dy_rows[i * L + t] * ypre * silu_grad(zz);
            }
            const double e = dy_rows[i * L + t] * gate; /* gradient reaching C h + D x */
            double gx = e * Dd, gdt = 0.0;
            gD += e * x;
            for (int n = 0; n < N; ++n) {
                const long long bc = ((long long)b * dstate + n) * L + t;
                const double Bv = widen(B, bc, in_dtype);
                const double Cv = widen(C, bc, in_dtype);
                const double lam = mu[n] + e * Cv; /* total gradient reaching h_t[n] */
                const double decay = exp(dt * a_n[n]);
                const double k = bbar_factor(dt, a_n[n], zoh);
                /* h_t = decay * h_prev + k * B * x, decay = exp(dt * a), k as in bbar_factor */
                double dk_ddt = 1.0, dk_da = 0.0;
                if (zoh && a_n[n] != 0.0) {
                    dk_ddt = decay;
                    dk_da = (dt * a_n[n] * decay - expm1(dt * a_n[n])) / (a_n[n] * a_n[n]);
                } else if (zoh) {
                    dk_da = 0.5 * dt * dt;
                }
                gC[n * L + t] += e * h_t[n];
                gB[n * L + t] += lam * k * x;
                gx += lam * k * Bv;
                gdt += lam * (a_n[n] * decay * h_prev[n] + dk_ddt * Bv * x);
                gA[n] += lam * (dt * decay * h_prev[n] + dk_da * Bv * x);
                mu[n] = lam * decay;
            }
            const double gs = softplus_flag ? gdt * softplus_grad(s) : gdt;
            ddelta_rows[i * L + t] = gs;
            gbias += gs;
            du_rows[i * L + t] = gx;
        }
        if (dh0_rows)
            for (int n = 0; n < N; ++n) dh0_rows[i * dstate + n] = mu[n];
#ifdef _OPENMP
#pragma omp critical(oracle_bwd_accumulate)
#endif
        {
            for (int n = 0; n < N; ++n) {
                if (dA) dA[(long long)d * dstate + n] += gA[n];
                for (long long t = 0; t < L; ++t) {
                    dB[((long long)b * dstate + n) * L + t] += gB[n * L + t];
                    dC[((long long)b * dstate + n) * L + t] += gC[n * L + t];
                }
            }
            if (dD) dD[d] += gD;
            if (dbias) dbias[d] += gbias;
        }
        free(hist); free(gB); free(gC);
    }
    return failed ? -2 : 0;
}

/*
 * Causal depthwise convolution over time, the step the Mamba block applies to the expanded input
 * before the selective SSM (visual guide, section 3.5: a convolution in front of the SSM so that
 * tokens are not processed independently).  Per channel d, with kernel width K:
 *   u[t] = act(conv_bias[d] + sum_{k=0}^{K-1} w[d, k] * x[t - (K-1) + k])
 * where x at positions before 0 comes from x_prev (the K-1 inputs preceding the sequence, oldest
 * first) or is zero, and act is silu when act_silu is set, else the identity.  The width, the
 * "previous inputs" convention and the activation are readings: the pages do not give them.
 *
 * x_rows [nrows, seqlen] in in_dtype; w [dim, K], conv_bias [dim] (may be NULL) fp32;
 * x_prev_rows [nrows, K-1] fp64 or NULL; u_rows [nrows, seqlen] fp64 (output).
 */
int oracle_causal_conv_rows(long long nrows, const int* row_d, int dim, int K, long long seqlen, int in_dtype,
                            const void* x_rows, const float* w, const float* conv_bias, int act_silu,
                            const double* x_prev_rows, double* u_rows) {
    if (nrows < 0 || dim <= 0 || K <= 0 || K > 64 || seqlen < 0) return -1;
    if (nrows > 0 && (!row_d || !x_rows || !w || !u_rows)) return -1;
    if (in_dtype != ORACLE_F32 && in_dtype != ORACLE_BF16) return -1;
    for (long long i = 0; i < nrows; ++i) {
        const int d = row_d[i];
        for (long long t = 0; t < seqlen; ++t) {
            double acc = conv_bias ? (double)conv_bias[d] : 0.0;
            for (int k = 0; k < K; ++k) {
                const long long s = t - (K - 1) + k;  /* input position this tap reads */
                double xv = 0.0;
                if (s >= 0)
                    xv = widen(x_rows, i * seqlen + s, in_dtype);
                else if (x_prev_rows)
                    xv = x_prev_rows[i * (K - 1) + (K - 1) + s];
                acc += (double)w[(long long)d * K + k] * xv;
            }
            u_rows[i * seqlen + t] = act_silu ? silu(acc) : acc;
        }
    }
    return 0;
}
