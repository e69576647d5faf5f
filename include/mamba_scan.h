/*
 * mamba_scan.h — C ABI of the B300 (sm_103a) selective-scan library, libmambascan.so.
 *
 * The library implements the data-parallel core of the selective state space layer described in
 * "Mamba: Linear-Time Sequence Modeling with Selective State Spaces" (visual guide to Mamba and
 * SSMs, sections 2.2-2.4 and 3.2-3.4; news write-up, "selection mechanism" and "hardware-aware
 * algorithm" sections):
 *
 *   Delta_t = softplus(delta_t + delta_bias)   (or delta_t + delta_bias without the flag)
 *   Abar_t  = exp(Delta_t * A),   Bbar_t x_t = Delta_t * B_t * x_t          (discretisation, 2.3)
 *   h_t     = Abar_t (.) h_{t-1} + Bbar_t x_t                                (recurrence, 2.4)
 *   y_t     = (C_t . h_t + D * x_t) * silu(z_t)                              (readout + skip, 2.2)
 *
 * A is diagonal and real (one value per channel and state), B, C and Delta vary with batch and
 * position (selection, 3.2).  The discretisation, recurrence and readout run fused in one kernel
 * that keeps h on chip and never writes Abar or Bbar to memory (hardware-aware algorithm, 3.4).
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library keeps none of them
 *    after the call returns and allocates no persistent memory.  Layouts are dense row-major with
 *    the last index contiguous.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as void*; NULL = the
 *    legacy default stream).  Results are valid once the stream has reached that point.
 *  - Return value: MAMBA_OK (0) or a negative error code.  No entry point aborts, traps or exits;
 *    mamba_scan_last_error() gives a message for the calling thread's last failure.
 *  - Misaligned pointers and any sequence length are accepted: such calls take a slower load path.
 */
#ifndef MAMBA_SCAN_H
#define MAMBA_SCAN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MAMBA_SCAN_VERSION 2

/* storage type of u / delta / z / B / C / y (A, D, delta_bias and all states are always fp32) */
#define MAMBA_F32 0
#define MAMBA_BF16 1

#define MAMBA_OK 0
#define MAMBA_ERR_ARG (-1)     /* bad argument: NULL required pointer, bad size, dtype, aliasing */
#define MAMBA_ERR_CUDA (-2)    /* a CUDA call or kernel launch failed */
#define MAMBA_ERR_TIMEOUT (-3) /* a kernel gave up a bounded wait (see mamba_scan_device_status) */

#define MAMBA_MAX_DSTATE 64

/* How B is discretised (Abar = exp(Delta A) in both; visual guide section 2.3, zero-order hold):
 * MAMBA_DISC_SIMPLE: Bbar = Delta * B.  MAMBA_DISC_ZOH: Bbar = (exp(Delta A) - 1) / A * B, the
 * exact solution of h' = A h + B x with x held over the step (Delta * B where A == 0). */
#define MAMBA_DISC_SIMPLE 0
#define MAMBA_DISC_ZOH 1

typedef struct {
    int batch;          /* b  >= 1 */
    int dim;            /* d (channels, d_inner) >= 1 */
    int dstate;         /* N, 1 <= N <= MAMBA_MAX_DSTATE */
    long long seqlen;   /* L >= 0 (ignored by mamba_state_step) */
    int in_dtype;       /* MAMBA_F32 or MAMBA_BF16 */
} mamba_scan_shape;

/*
 * Forward selective scan from a zero initial state.
 *
 *   u, delta, z   [b, d, L]  in_dtype.  z == NULL: no gate (y = C.h + D x).
 *   A             [d, N]     fp32 (typically negative; Abar = exp(Delta A)).
 *   B, C          [b, N, L]  in_dtype, shared by all channels of a batch row.
 *   D             [d]        fp32 or NULL (= 0).
 *   delta_bias    [d]        fp32 or NULL (= 0).
 *   softplus_flag            nonzero: Delta = softplus(delta + bias); zero: Delta = delta + bias.
 *   y             [b, d, L]  in_dtype, written (bf16 by round-to-nearest-even).  Must not overlap
 *                            any input.
 *   last_state    [b, d, N]  fp32 or NULL: h after the last position (zeros when L == 0).
 *
 * Sequences with few channels (b*d small against the GPU) are split along L into segments that
 * exchange carries (prod Abar, end state) through stream-ordered scratch memory (cudaMallocAsync
 * on `stream`, freed on the same stream).  dstate <= 16: one kernel scans every segment at once
 * (the first from the initial state, the others from zero) and a second adds to each later
 * segment's outputs the decaying part of the state carried into it, dropping it once it has
 * decayed below 2^-40 of its size at the segment start (visual guide section 3.3, associativity
 * of the scan).  dstate > 16: a first kernel computes the carries and a second runs the fused
 * scan per segment from its folded carry.  With bf16 y, outputs a segment's correction reaches
 * are rounded twice (own part, then the sum).
 * Errors: MAMBA_ERR_ARG for bad arguments, MAMBA_ERR_CUDA if an allocation or launch fails.
 */
int mamba_scan_fwd(const mamba_scan_shape* s, const void* u, const void* delta, const float* A,
                   const void* B, const void* C, const float* D, const void* z,
                   const float* delta_bias, int softplus_flag, void* y, float* last_state,
                   void* stream);

/*
 * Forward selective scan from a given state: mamba_scan_fwd with the recurrence started from h0
 * instead of zero, so that a long prompt can be scanned in pieces and handed on to decoding
 * (recurrent inference carries only the state: news write-up, "architecture" section; visual
 * guide section 2.4).
 *
 *   h0            [b, d, N]  fp32 or NULL (= zero): h before position 0.  It may be the same
 *                            buffer as last_state (the call then advances that state in place);
 *                            partial overlap with last_state, or any overlap with y, is
 *                            MAMBA_ERR_ARG.
 *   With L == 0, last_state receives h0 (or zeros).  Everything else as for mamba_scan_fwd.
 */
int mamba_scan_fwd_state(const mamba_scan_shape* s, const void* u, const void* delta, const float* A,
                         const void* B, const void* C, const float* D, const void* z,
                         const float* delta_bias, int softplus_flag, const float* h0, void* y,
                         float* last_state, void* stream);

/*
 * mamba_scan_fwd_state with a choice of discretisation: MAMBA_DISC_SIMPLE (identical to
 * mamba_scan_fwd_state) or MAMBA_DISC_ZOH, the exact zero-order hold
 *   Bbar_t x_t = (exp(Delta_t A) - 1) / A * B_t x_t     (Delta_t B_t x_t where A == 0),
 * the discretisation the visual guide names in section 2.3 (the input held constant over each step
 * of length Delta).  Any other value is MAMBA_ERR_ARG.  Everything else as for mamba_scan_fwd_state.
 */
int mamba_scan_fwd_ex(const mamba_scan_shape* s, int discretization, const void* u, const void* delta,
                      const float* A, const void* B, const void* C, const float* D, const void* z,
                      const float* delta_bias, int softplus_flag, const float* h0, void* y,
                      float* last_state, void* stream);

/*
 * The block's causal depthwise convolution fused in front of the scan (visual guide section 3.5:
 * the Mamba block convolves the expanded input before the selective SSM).  Instead of u the call
 * takes the convolution's input x and computes, inside the scan kernel, per channel d
 *   u[t] = act(conv_bias[d] + sum_{k=0}^{conv_k-1} conv_w[d, k] * x[t - conv_k + 1 + k]),
 * act = silu when conv_silu is nonzero, else the identity; u is never written to memory.  It feeds
 * both the recurrence (Bbar u) and the skip term (D u).
 *
 *   x             [b, d, L]  in_dtype (takes the place of u).
 *   conv_w        [d, conv_k] fp32, 1 <= conv_k <= 4.   conv_bias [d] fp32 or NULL (= 0).
 *   conv_prev     [b, d, conv_k - 1] fp32 or NULL (= 0): the inputs x before position 0, oldest
 *                 first, for a sequence scanned in pieces (pass the previous piece's last
 *                 conv_k - 1 inputs, together with its last_state as h0).
 * Everything else as for mamba_scan_fwd_ex.
 */
int mamba_scan_fwd_conv(const mamba_scan_shape* s, int discretization, const void* x, const float* conv_w,
                        const float* conv_bias, int conv_k, int conv_silu, const float* conv_prev,
                        const void* delta, const float* A, const void* B, const void* C, const float* D,
                        const void* z, const float* delta_bias, int softplus_flag, const float* h0, void* y,
                        float* last_state, void* stream);

/*
 * One recurrent decoding step for every (batch, channel): constant work per token, no cache of
 * past tokens (news write-up, "architecture" section; visual guide section 1.4).
 *
 *   state         [b, d, N]  fp32, updated IN PLACE: h <- exp(Delta A) h + Delta B x.
 *   x, delta, z   [b, d]     in_dtype (z may be NULL).
 *   A [d, N], D [d], delta_bias [d]: as for mamba_scan_fwd.
 *   B, C          [b, N]     in_dtype.
 *   y             [b, d]     in_dtype, y = (C.h + D x) silu(z) with the updated h.
 * s->seqlen is ignored.  Errors as for mamba_scan_fwd.
 */
int mamba_state_step(const mamba_scan_shape* s, float* state, const void* x, const void* delta,
                     const float* A, const void* B, const void* C, const float* D, const void* z,
                     const float* delta_bias, int softplus_flag, void* y, void* stream);

/* mamba_state_step with a choice of discretisation (MAMBA_DISC_SIMPLE or MAMBA_DISC_ZOH, as for
 * mamba_scan_fwd_ex). */
int mamba_state_step_ex(const mamba_scan_shape* s, int discretization, float* state, const void* x,
                        const void* delta, const float* A, const void* B, const void* C, const float* D,
                        const void* z, const float* delta_bias, int softplus_flag, void* y, void* stream);

/*
 * Allocation-free variant of mamba_scan_fwd.  The pages describe nothing like it: it exists for
 * callers that must not have the library allocate device memory, for example a process that hands
 * all device memory to its own pool allocator up front, or one that runs under a fixed, audited
 * memory budget and forbids third-party code from calling the CUDA allocator.
 *
 * Arguments, layouts, results and errors are those of mamba_scan_fwd.  The only difference: when
 * the shape makes the library split the time axis into segments (few channels, long sequences),
 * the per-segment carries go to a fixed scratch array of MAMBA_NOALLOC_SCRATCH_BYTES that the
 * library holds in device memory on every GPU where it is loaded, until the process exits.  No
 * cudaMalloc, cudaMallocAsync, cudaFree or other allocating call is made.
 *  - A shape whose carries need more than MAMBA_NOALLOC_SCRATCH_BYTES, that is
 *    S * batch * dim * dstate * 8 bytes for S time segments when dstate <= 16 (S - 1 instead of
 *    S when dstate > 16), is rejected with MAMBA_ERR_ARG
 *    and a message stating both sizes; nothing is launched.  S follows from the shape and the SM
 *    count nSM of the device, and is at most max(1, seqlen / 256) (fp32) or seqlen / 512 (bf16):
 *      dstate <= 16: S = 1 unless batch * ceil(dim / 32) <= 2 * nSM; then
 *                    S <= ceil(4 * nSM / (batch * ceil(dim / 32))) + 1;
 *      dstate > 16:  S = 1 unless batch * ceil(dim / 8) < 5 * nSM; then
 *                    S = ceil(10 * nSM / (batch * ceil(dim / 8))).
 *    For example the million-token workload (batch 1, dim 1536, dstate 16) splits into at most
 *    14 segments on a 148-SM device, whose carries take at most 2.8 MB; batch 1, dim 32 takes
 *    4 KB per segment.
 *  - The first call on each device looks up the array's device address (cudaGetSymbolAddress)
 *    with that device current, then caches it under the unique id of the CUDA context that made
 *    the call; a call from another context, or after cudaDeviceReset, repeats the lookup.  Make
 *    the first call in each context before any stream capture.
 *  - All calls on a device share the one array and it keeps the last call's contents.  Every
 *    carry a call reads is written earlier in the same call, so nothing needs clearing.  Calls
 *    that can run at the same time on the GPU (for example on two streams with no ordering between
 *    them) race on it: order them on one stream or with events.
 */
#define MAMBA_NOALLOC_SCRATCH_BYTES (4u << 20)
int mamba_scan_fwd_noalloc(const mamba_scan_shape* s, const void* u, const void* delta, const float* A,
                           const void* B, const void* C, const float* D, const void* z,
                           const float* delta_bias, int softplus_flag, void* y, float* last_state,
                           void* stream);

/*
 * Forward pass of training: mamba_scan_fwd_ex that also writes the state before every 8-position
 * slot.  The hardware-aware algorithm keeps no state for the backward pass and recomputes them
 * there (visual guide section 3.4, "recomputation"); mamba_scan_bwd does so with a forward sweep
 * that writes exactly these one-in-eight states before its reverse sweep.  Writing them here
 * instead (8 bytes per channel and step, while the forward kernel is bound by arithmetic, not
 * HBM) lets mamba_scan_bwd_ckpt skip that sweep.
 *   ckpt          [b, ceil(L/8), d, 16] fp32 device memory, caller-owned, 16-byte aligned;
 *                 written for slots 1.. (slot 0 is h0), with the states past N as zero.  Must not
 *                 overlap any input or output.
 *   ckpt_written  host int: set to 1 when ckpt was written, 0 when it was not.  A sequence the
 *                 library splits along L (few channels, long sequences) gets no checkpoints, and
 *                 mamba_scan_bwd_ckpt then makes its own.  mamba_scan_fwd_train_ckpt_bytes
 *                 tells beforehand (0 bytes: none).
 * Everything else as for mamba_scan_fwd_ex (no fused convolution).  Errors: as mamba_scan_fwd_ex,
 * and MAMBA_ERR_ARG for a NULL ckpt or ckpt_written, dstate > 16, a misaligned or overlapping ckpt
 * (then nothing is launched, and ckpt_written, when not NULL, is 0).
 */
int mamba_scan_fwd_train(const mamba_scan_shape* s, int discretization, const void* u, const void* delta,
                         const float* A, const void* B, const void* C, const float* D, const void* z,
                         const float* delta_bias, int softplus_flag, const float* h0, void* y, float* last_state,
                         float* ckpt, int* ckpt_written, void* stream);

/*
 * Size in bytes of the checkpoints that mamba_scan_fwd_train writes for shape s on the current
 * device: b * ceil(L/8) * d * 16 * 4, or 0 when it would write none (dstate > 16, L = 0, or a
 * sequence the library splits along L).  Host-side only: no allocation and no launch.  The
 * answer holds while the device and the MAMBA_SCAN_* environment variables stay the same.
 *   bytes   written.
 * Errors: MAMBA_ERR_ARG (NULL pointer, bad shape).
 */
int mamba_scan_fwd_train_ckpt_bytes(const mamba_scan_shape* s, size_t* bytes);

/*
 * mamba_scan_bwd with the checkpoints of mamba_scan_fwd_train (same inputs, h0 and
 * discretization): when ckpt is non-NULL and the backward pass runs unsplit with dstate <= 16, it
 * skips its forward sweep and recomputes every slot from ckpt; otherwise ckpt is ignored.  ckpt
 * (16-byte aligned; MAMBA_ERR_ARG otherwise) must not overlap a gradient output.  Everything else
 * as for mamba_scan_bwd.
 */
int mamba_scan_bwd_ckpt(const mamba_scan_shape* s, int discretization, const void* u, const void* delta,
                        const float* A, const void* B, const void* C, const float* D, const void* z,
                        const float* delta_bias, int softplus_flag, const float* h0, const void* dy,
                        const float* dlast_state, const float* ckpt, void* du, void* ddelta, void* dz, float* dA,
                        float* dB, float* dC, float* dD, float* ddelta_bias, float* dh0, void* stream);

/*
 * Gradients of the forward scan (mamba_scan_fwd_state) for the loss
 *   sum(dy * y) + sum(dlast_state * last_state),
 * i.e. the backward pass of training.  The expanded states are not stored by the forward pass;
 * this call recomputes them (visual guide section 3.4, "recomputation"): a forward sweep keeps
 * one state checkpoint per 8 positions (stream-ordered scratch, cudaMallocAsync on `stream`,
 * b * ceil(L/8) * d * 64 bytes, freed on the same stream), and a reverse sweep recomputes each
 * 8-position slot from its checkpoint and walks it backwards.  States are handled in blocks of
 * 16, one kernel launch each.  When batch * ceil(d / 32) is at most 2 * nSM (few channels, e.g.
 * long sequences), the time axis is also split into segments that run at once (visual guide
 * section 3.3: the scan operator is associative, and both the state and its gradient are linear
 * recurrences): a carry launch gives each segment's (prod Abar, own end state), the full launch
 * runs every segment from its folded start state with no gradient arriving at its end, and a
 * correction launch adds, from each segment's end backwards, what the gradient carried in from
 * the later segments contributes, until it has decayed below 2^-40 of its size.  With several
 * blocks or segments the gradients of u, delta and z are summed in fp32 (in the outputs for fp32
 * storage; for bf16 in scratch of 2 or 3 * b * d * L * 4 bytes, converted at the end); segments
 * add nseg * b * d * N * 12 bytes of scratch.
 *
 *   discretization  MAMBA_DISC_SIMPLE or MAMBA_DISC_ZOH: the one the forward pass used.
 *   u .. h0         the forward inputs, as for mamba_scan_fwd_state (z, D, delta_bias, h0 may be
 *                   NULL with the same meaning); any dstate up to MAMBA_MAX_DSTATE.
 *   dy              [b, d, L]  in_dtype: gradient of the loss with respect to y.
 *   dlast_state     [b, d, N]  fp32 or NULL (= 0): gradient with respect to last_state.
 * Outputs (written; none may overlap an input or another output):
 *   du, ddelta      [b, d, L]  in_dtype (ddelta is the gradient with respect to the raw delta,
 *                              before bias and softplus).
 *   dz              [b, d, L]  in_dtype, or NULL (not computed; must be NULL when z is NULL).
 *   dA              [d, N]     fp32, summed over batch and positions.
 *   dB, dC          [b, N, L]  fp32, summed over channels.
 *   dD, ddelta_bias [d]        fp32 or NULL (not computed), summed over batch and positions.
 *   dh0             [b, d, N]  fp32 or NULL: gradient with respect to h0.
 * With L == 0 only dA, dD, ddelta_bias (zeros) and dh0 (= dlast_state, or zeros) are written and
 * the per-position pointers may be NULL.  The sums over channels and batch rows are accumulated
 * with atomics, so their rounding (not their value) can differ between runs.
 * Errors: MAMBA_ERR_ARG, MAMBA_ERR_CUDA.
 */
int mamba_scan_bwd(const mamba_scan_shape* s, int discretization, const void* u, const void* delta,
                   const float* A, const void* B, const void* C, const float* D, const void* z,
                   const float* delta_bias, int softplus_flag, const float* h0, const void* dy,
                   const float* dlast_state, void* du, void* ddelta, void* dz, float* dA, float* dB,
                   float* dC, float* dD, float* ddelta_bias, float* dh0, void* stream);

/*
 * Gradients of the forward scan with the block's causal convolution in front of it
 * (mamba_scan_fwd_conv) for the loss sum(dy * y) + sum(dlast_state * last_state): the backward pass
 * of training the convolution and the selective SSM together (visual guide sections 3.4 and 3.5).
 * Steps, all on `stream`: u = act(conv(x)) is recomputed into stream-ordered scratch
 * (cudaMallocAsync, 2 * b * d * L * sizeof(in_dtype) bytes with du, freed on the same stream);
 * the scan's backward pass (as mamba_scan_bwd) gives du; a convolution kernel takes du back
 * through the activation and the taps.
 *
 *   discretization, x, conv_w, conv_bias, conv_k, conv_silu, conv_prev, delta .. h0:
 *                   the forward inputs, as for mamba_scan_fwd_conv.
 *   dy, dlast_state as for mamba_scan_bwd.
 * Outputs (written; dx must not overlap an input or another output):
 *   dx              [b, d, L]  in_dtype: gradient with respect to the convolution's input x.
 *   ddelta, dz, dA, dB, dC, dD, ddelta_bias, dh0: as for mamba_scan_bwd.
 *   dconv_w         [d, conv_k] fp32 or NULL, summed over batch and positions.
 *   dconv_bias      [d] fp32 or NULL, summed over batch and positions (also when conv_bias is NULL).
 *   dconv_prev      [b, d, conv_k - 1] fp32 or NULL: gradient with respect to the inputs before
 *                   position 0 (conv_prev, or the zeros that stand for it when it is NULL); zeros
 *                   when L == 0.
 * With bf16 storage, u and du pass through bf16 scratch (the forward kept u in fp32 registers).
 * The per-channel sums use atomics, so their rounding (not their value) can differ between runs.
 * Errors: MAMBA_ERR_ARG, MAMBA_ERR_CUDA.
 */
int mamba_scan_bwd_conv(const mamba_scan_shape* s, int discretization, const void* x, const float* conv_w,
                        const float* conv_bias, int conv_k, int conv_silu, const float* conv_prev,
                        const void* delta, const float* A, const void* B, const void* C, const float* D,
                        const void* z, const float* delta_bias, int softplus_flag, const float* h0,
                        const void* dy, const float* dlast_state, void* dx, void* ddelta, void* dz, float* dA,
                        float* dB, float* dC, float* dD, float* ddelta_bias, float* dconv_w, float* dconv_bias,
                        float* dconv_prev, float* dh0, void* stream);

/* Message describing the calling thread's most recent failure ("" if none). */
const char* mamba_scan_last_error(void);

/* MAMBA_SCAN_VERSION of the loaded library. */
int mamba_scan_version(void);

/* Number of kernels this library has launched in this process so far (all threads, all devices);
 * lets a caller count the GPU work behind a sequence of calls. */
long long mamba_scan_launch_count(void);

/*
 * Synchronises `stream`, then reads and clears the library's device status word on the current
 * device.  Returns MAMBA_OK, MAMBA_ERR_TIMEOUT if any kernel since the last call abandoned a
 * bounded wait on an asynchronous copy (its outputs are then invalid), or MAMBA_ERR_CUDA.
 */
int mamba_scan_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_SCAN_H */
