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
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1

static double widen(const void* p, long long i, int dtype) {
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

int oracle_version(void) { return 1; }

/*
 * Forward selective scan over a list of channels ("rows").
 *
 * Row i is channel (row_b[i], row_d[i]).  u_rows, delta_rows, z_rows hold that channel's inputs,
 * [nrows, seqlen] in in_dtype.  A [dim, dstate] fp32, D and delta_bias [dim] fp32 (either may be
 * NULL for zero); B, C [batch, dstate, seqlen] in in_dtype; z_rows may be NULL (no gate).
 * h0_rows [nrows, dstate] is the initial state (NULL = zero).
 * Outputs: y_rows [nrows, seqlen] and state_rows [nrows, dstate] (may be NULL), fp64.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_scan_rows(long long nrows, const int* row_b, const int* row_d, int dim, int dstate,
                     long long seqlen, int in_dtype, const void* u_rows, const void* delta_rows,
                     const void* z_rows, const float* A, const float* D, const float* delta_bias,
                     const void* B, const void* C, int softplus_flag, const double* h0_rows,
                     double* y_rows, double* state_rows, int nthreads) {
    if (nrows < 0 || dim <= 0 || dstate <= 0 || dstate > 256 || seqlen < 0) return -1;
    if (nrows > 0 && (!row_b || !row_d || !u_rows || !delta_rows || !A || !B || !C || !y_rows))
        return -1;
    if (in_dtype != ORACLE_F32 && in_dtype != ORACLE_BF16) return -1;
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
                const double Bbar_x = dt * widen(B, bc, in_dtype) * x;
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

/*
 * One recurrent (decoding) step for a list of channels: the same body as one time step of the
 * scan, starting from the given state.  state_rows [nrows, dstate] fp64 is updated in place.
 * x_rows, delta_rows, z_rows [nrows] in in_dtype; B, C [batch, dstate] in in_dtype.
 * y_rows [nrows] fp64.  Constant work per token, no cache of past tokens (news write-up,
 * "architecture" section; visual guide section 1.4 on recurrent inference).
 */
int oracle_state_step_rows(long long nrows, const int* row_b, const int* row_d, int dim, int dstate,
                           int in_dtype, double* state_rows, const void* x_rows,
                           const void* delta_rows, const void* z_rows, const float* A,
                           const float* D, const float* delta_bias, const void* B, const void* C,
                           int softplus_flag, double* y_rows, int nthreads) {
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
            const double Abar = exp(dt * (double)A[(long long)d * dstate + n]);
            h[n] = Abar * h[n] + dt * widen(B, bc, in_dtype) * x;
            acc += widen(C, bc, in_dtype) * h[n];
        }
        double y = acc + (D ? (double)D[d] : 0.0) * x;
        if (z_rows) y *= silu(widen(z_rows, i, in_dtype));
        y_rows[i] = y;
    }
    return 0;
}
