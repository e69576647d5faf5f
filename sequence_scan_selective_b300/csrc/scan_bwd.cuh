// Backward pass of the selective scan, with the states recomputed instead of stored.
//
// The forward pass keeps the expanded state h[b, d, n, t] in registers and never writes it (visual
// guide to Mamba and SSMs, section 3.4, kernel fusion); the backward pass needs it, and the guide's
// answer (same section, "recomputation") is to recompute it from what is cheap to keep.  Here that
// is one checkpoint of the state per 8 steps (written by a forward sweep, half the size of u in
// fp32 at N = 16), from which each 8-step slot is recomputed into registers and then walked in
// reverse.  (8 rather than 16 steps: the slot's states then fit in 128 registers per thread, and
// four CTAs share an SM.)
//
// With a_t = exp(Delta_t A), h_t = a_t h_{t-1} + Delta_t B_t x_t, ypre_t = C_t h_t + D x_t and
// y_t = ypre_t silu(z_t), the reverse walk carries mu_t = dL/dh_t from the later steps:
//   e_t      = dy_t silu(z_t)                        gradient reaching ypre_t
//   lam_t    = mu_t + e_t C_t                         total gradient reaching h_t
//   dC_t    += e_t h_t,  dB_t += lam_t Delta_t x_t    (summed over the channels of a batch row)
//   dDelta_t = sum_n lam_t (A a_t h_{t-1} + B_t x_t)  (a_t h_{t-1} = h_t - Delta_t B_t x_t)
//   dx_t     = Delta_t sum_n lam_t B_t + D e_t,   dA += lam_t a_t h_{t-1} Delta_t
//   mu_{t-1} = a_t lam_t
// then ddelta = dDelta * sigmoid(delta + bias) (softplus) and dz = dy ypre silu'(z).
//
// Work layout: a CTA of 4 warps owns 32 channels of one batch row for the whole sequence; a warp
// owns 8 channels, lane (c = lane % 8, g = lane / 8) holds states nb+4g .. nb+4g+3 of channel c,
// where nb is the first state of the launch's block of 16 (N > 16 runs one launch per block, in
// order: the states are independent of one another, and the per-(channel, step) gradients, which
// sum over all states, are accumulated in fp32 across the launches).
// Tiles of 16 steps of u, delta, z, dy (per channel) and B, C (per batch row) are staged in shared
// memory by cp.async, double-buffered.  The sums over channels (dB, dC) are reduced across the 8
// channel lanes of a warp by a shuffle reduce-scatter, across the 4 warps in shared memory, and
// across CTAs of the same batch row with vector atomics; the sums over states (dDelta, dx, ypre)
// across the 4 state lanes of a channel by a second reduce-scatter.
#pragma once
#include <stdint.h>

#include "ptx.cuh"
#include "common.cuh"

namespace mscan {

struct BwdArgs {
    const void* u;      // [b, d, L] TIn
    const void* delta;  // [b, d, L] TIn
    const void* z;      // [b, d, L] TIn or null (no gate)
    const void* dy;     // [b, d, L] TIn
    const void* B;      // [b, N, L] TIn
    const void* C;      // [b, N, L] TIn
    const float* A;     // [d, N]
    const float* D;     // [d] or null
    const float* bias;  // [d] or null
    const float* h0;    // [b, d, N] or null (zero initial state)
    const float* dlast; // [b, d, N] or null (no gradient at last_state)
    void* du;           // [b, d, L] TIn
    void* ddelta;       // [b, d, L] TIn
    void* dz;           // [b, d, L] TIn or null
    float* dA;          // [d, N], accumulated (zeroed by the host)
    float* dB;          // [b, N, L], accumulated (zeroed by the host)
    float* dC;          // [b, N, L], accumulated (zeroed by the host)
    float* dD;          // [d] or null, accumulated
    float* dbias;       // [d] or null, accumulated
    float* dh0;         // [b, d, N] or null
    float* ckpt;        // [b, nslot, d, 16] state before each slot of kSlot steps (slot 0 unused)
    int batch, dim, dstate;
    long long L;
    int ntile, nslot;
    int softplus;
    // State block: this launch handles states nb .. nb + 15 (N > 16 takes ceil(N / 16) launches,
    // in order).  Then the per-(channel, step) gradients, whose sums over states span all blocks,
    // are added into fp32 accumulators acc_du, acc_dd, acc_dz [b, d, L] (the first block writes
    // them); a final pass converts them.  With acc_du == null (N <= 16) they are stored directly.
    int nb;
    float* acc_du;
    float* acc_dd;
    float* acc_dz;
    // Split time axis: segment blockIdx.z covers tiles [z * seg_tiles, (z + 1) * seg_tiles).
    // carry [nseg][b][d][N]: (prod Abar over the segment, end state from the segment's own start:
    // the initial state for segment 0, zero for the others); mu_local [nseg][b][d][N]: dL/dh at
    // the segment's start from its own reverse walk (no gradient carried in from later segments).
    int nseg, seg_tiles;
    float2* carry;
    float* mu_local;
    // nonzero: ckpt holds the forward pass's checkpoints already (unsplit, N <= 16), so the full
    // launch skips its forward sweep
    int ck_given;
};

namespace bwd {

// Hint: bring the line holding p into L2 (no register, no completion to wait for).
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kCh = kWarps * 8;  // channels per CTA
constexpr int kT = 16;           // steps per tile
constexpr int kSPL = kT / 4;     // steps per lane in the per-(channel, step) phases
constexpr int kSlot = 8;         // steps per recomputed slot (its states live in registers)
constexpr int kSlots = kT / kSlot;
constexpr int kNS = 16;          // state capacity (lanes per channel x 4)
constexpr int kPad = kT + 1;     // padded row (floats) of the per-channel sums r[k][c][t]
constexpr int kPartPitch = 33;   // padded row (floats) of the dB/dC partials part[t][32 columns]
constexpr int kBcqPitch = 36;    // floats per step in the B/C step buffer (padded)
constexpr float kDropBelow = 9.094947017729282e-13f;  // 2^-40

// Launch modes of scan_bwd_kernel.
//  kFull:  forward sweep (checkpoints) + reverse walk of the segment, from the state carried into
//          it; gradient at the segment's end: dlast for the last segment, else zero.
//  kCarry: forward sweep of the segment from its own start only, writing its carry.
//  kCorr:  reverse walk of a segment from its end with mu = the gradient carried in from the later
//          segments and no output gradient (dy = 0), adding what that gradient contributes; it stops
//          once mu has decayed below 2^-40 of its size at the segment's end.
constexpr int kFull = 0, kCarry = 1, kCorr = 2;

template <typename TIn>
struct Layout {
    static constexpr int ROW = kT * (int)sizeof(TIn) + 16;  // bytes per staged row (padded)
    static constexpr int CHUNKS = kT * (int)sizeof(TIn) / 16;  // 16-byte pieces per row
    // one stage: u, delta, z, dy rows of the CTA's channels, then B and C rows
    static constexpr int OFF_U = 0;
    static constexpr int OFF_DL = OFF_U + kCh * ROW;
    static constexpr int OFF_Z = OFF_DL + kCh * ROW;
    static constexpr int OFF_DY = OFF_Z + kCh * ROW;
    static constexpr int OFF_B = OFF_DY + kCh * ROW;
    static constexpr int OFF_C = OFF_B + kNS * ROW;
    static constexpr int STAGE = OFF_C + kNS * ROW;
    // after the two stages: B/C per step (bcq[t][0..15] = B, [16..31] = C), per-warp step data
    // q[t][c] = (Delta, Delta x, e, x), per-warp per-channel sums r[k][c][t] (k: dDelta, sum of
    // lam B, sum of C h), per-warp dB/dC partials part[t][kind * 16 + n] (kind 0: dC, 1: dB)
    static constexpr int OFF_BCQ = 2 * STAGE;
    static constexpr int OFF_Q = OFF_BCQ + kT * kBcqPitch * 4;
    static constexpr int OFF_R = OFF_Q + kWarps * kT * 8 * 16;
    static constexpr int OFF_PART = OFF_R + kWarps * 3 * 8 * kPad * 4;
    static constexpr int BYTES = OFF_PART + kWarps * kT * kPartPitch * 4;
};

// v[0..7] held by every lane; returns, in the lane with (lane & 7) == k, the sum of v[k] over the
// 8 lanes that differ from it in bits 0-2.  Seven shuffles instead of 24 for a plain butterfly.
__device__ __forceinline__ float reduce_scatter8(const float (&v)[8], int lane) {
    const bool b2 = lane & 4, b1 = lane & 2, b0 = lane & 1;
    float w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float send = b2 ? v[j] : v[j + 4];
        const float keep = b2 ? v[j + 4] : v[j];
        w[j] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float x[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float send = b1 ? w[j] : w[j + 2];
        const float keep = b1 ? w[j + 2] : w[j];
        x[j] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const float send = b0 ? x[0] : x[1];
    const float keep = b0 ? x[1] : x[0];
    return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

// (v0, v1, v2) held by every lane; returns, in the lane with ((lane >> 3) & 3) == k < 3, the sum
// of v_k over the 4 lanes that differ from it in bits 3-4 (the state lanes of one channel).
__device__ __forceinline__ float reduce_scatter3(float v0, float v1, float v2, int lane) {
    const bool b4 = lane & 16, b3 = lane & 8;
    const float s0 = b4 ? v0 : v2, k0 = b4 ? v2 : v0;
    const float s1 = b4 ? v1 : 0.f, k1 = b4 ? 0.f : v1;
    const float w0 = k0 + __shfl_xor_sync(0xffffffffu, s0, 16);
    const float w1 = k1 + __shfl_xor_sync(0xffffffffu, s1, 16);
    const float send = b3 ? w0 : w1;
    const float keep = b3 ? w1 : w0;
    return keep + __shfl_xor_sync(0xffffffffu, send, 8);
}


// Stage tile k (steps 32k .. 32k+31) of the CTA's channel rows (u, delta; z and dy when `full`) and
// of B (and C when `full`) rows nb .. min(nb + 16, N) - 1 (the state block).  Positions past L or past the last channel read as zero.
// VEC: 16-byte cp.async pieces (rows 16-byte aligned, L * sizeof(TIn) a multiple of 16), left in
// flight; otherwise plain element loads, complete on return.
template <typename TIn, bool VEC>
__device__ __forceinline__ void load_tile(uint8_t* st, const BwdArgs& a, int b, int d0, int k, bool full) {
    using Lt = Layout<TIn>;
    constexpr int EPC = 16 / (int)sizeof(TIn);  // elements per 16-byte piece
    const long long t0 = (long long)k * kT;
    const int tid = threadIdx.x;
    const int nch_t = full ? 4 : 2;
    const int nbc_t = full ? 2 : 1;
    // the four channel tensors sit back to back in a stage: u, delta, z, dy
    auto chsrc = [&](int tens) -> const void* { return tens == 0 ? a.u : tens == 1 ? a.delta : tens == 2 ? a.z : a.dy; };
    auto choff = [](int tens) { return Lt::OFF_U + tens * kCh * Lt::ROW; };
    if (VEC) {
        constexpr int per = kCh * Lt::CHUNKS;
        for (int i = tid; i < nch_t * per; i += kThreads) {
            const int tens = i / per, rem = i - tens * per;
            const int row = rem / Lt::CHUNKS, piece = rem - row * Lt::CHUNKS;
            if (!chsrc(tens)) continue;
            const int d = d0 + row;
            const long long e0 = t0 + piece * EPC;
            const bool ok = d < a.dim && e0 < a.L;
            const TIn* p = static_cast<const TIn*>(chsrc(tens)) +
                           (ok ? ((long long)b * a.dim + d) * a.L + e0 : 0);
            cp_async16(st + choff(tens) + row * Lt::ROW + piece * 16, p, ok ? 16u : 0u);
        }
        const int nrow = min(kNS, a.dstate - a.nb);  // this block's states
        const int perb = nrow * Lt::CHUNKS;
        for (int i = tid; i < nbc_t * perb; i += kThreads) {
            const int tens = i / perb, rem = i - tens * perb;
            const int n = rem / Lt::CHUNKS, piece = rem - n * Lt::CHUNKS;
            const long long e0 = t0 + piece * EPC;
            const bool ok = e0 < a.L;
            const TIn* p = static_cast<const TIn*>(tens ? a.C : a.B) +
                           (ok ? ((long long)b * a.dstate + a.nb + n) * a.L + e0 : 0);
            cp_async16(st + (tens ? Lt::OFF_C : Lt::OFF_B) + n * Lt::ROW + piece * 16, p, ok ? 16u : 0u);
        }
        cp_async_commit();
    } else {
        constexpr int per = kCh * kT;
        for (int i = tid; i < nch_t * per; i += kThreads) {
            const int tens = i / per, rem = i - tens * per;
            const int row = rem / kT, t = rem - row * kT;
            if (!chsrc(tens)) continue;
            const int d = d0 + row;
            const long long e = t0 + t;
            TIn v{};
            if (d < a.dim && e < a.L) v = static_cast<const TIn*>(chsrc(tens))[((long long)b * a.dim + d) * a.L + e];
            reinterpret_cast<TIn*>(st + choff(tens) + row * Lt::ROW)[t] = v;
        }
        const int nrow = min(kNS, a.dstate - a.nb);
        const int perb = nrow * kT;
        for (int i = tid; i < nbc_t * perb; i += kThreads) {
            const int tens = i / perb, rem = i - tens * perb;
            const int n = rem / kT, t = rem - n * kT;
            const long long e = t0 + t;
            TIn v{};
            if (e < a.L) v = static_cast<const TIn*>(tens ? a.C : a.B)[((long long)b * a.dstate + a.nb + n) * a.L + e];
            reinterpret_cast<TIn*>(st + (tens ? Lt::OFF_C : Lt::OFF_B) + n * Lt::ROW)[t] = v;
        }
    }
}

// kSPL consecutive staged elements (steps kSPL*g ..) of one row, widened to fp32.
template <typename TIn>
__device__ __forceinline__ void row_steps(const uint8_t* row, int g, float (&v)[kSPL]) {
    static_assert(kSPL == 4 || kSPL == 8, "vector widths");
    if constexpr (sizeof(TIn) == 4) {
#pragma unroll
        for (int i = 0; i < kSPL / 4; ++i) {
            const float4 p = reinterpret_cast<const float4*>(row)[(kSPL / 4) * g + i];
            v[4 * i] = p.x; v[4 * i + 1] = p.y; v[4 * i + 2] = p.z; v[4 * i + 3] = p.w;
        }
    } else if constexpr (kSPL == 4) {
        const uint2 p = reinterpret_cast<const uint2*>(row)[g];
        v[0] = __uint_as_float(p.x << 16); v[1] = __uint_as_float(p.x & 0xffff0000u);
        v[2] = __uint_as_float(p.y << 16); v[3] = __uint_as_float(p.y & 0xffff0000u);
    } else {
        const uint4 p = reinterpret_cast<const uint4*>(row)[g];
        const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
}

// Store kSPL consecutive outputs of one row at steps tg0 .. (those below L).
template <typename TIn, bool VEC>
__device__ __forceinline__ void store_steps(TIn* p, long long tg0, long long L, const float (&v)[kSPL]) {
    if (VEC && tg0 + kSPL <= L) {
        if constexpr (sizeof(TIn) == 4) {
#pragma unroll
            for (int i = 0; i < kSPL / 4; ++i)
                reinterpret_cast<float4*>(p)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        } else if constexpr (kSPL == 4) {
            reinterpret_cast<uint2*>(p)[0] = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
        } else {
            reinterpret_cast<uint4*>(p)[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                        pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
        }
    } else {
#pragma unroll
        for (int j = 0; j < kSPL; ++j)
            if (tg0 + j < L) store_out<TIn>(p + j, v[j]);
    }
}

}  // namespace bwd

// MINB: CTAs per SM the register budget is cut for (4: 128 registers a thread; 3: 168).  With 3,
// the simplified discretisation keeps each step's Abar from the slot's recomputation for the
// reverse walk instead of computing it again (2 ex2 and a packed multiply per state pair and step
// fewer, 32 more registers); it suits grids of at most 3 CTAs per SM.
template <typename TIn, bool VEC, bool ZOH, int MODE, int MINB = 4>
__global__ void __launch_bounds__(bwd::kThreads, MINB) scan_bwd_kernel(const BwdArgs a) {
    using namespace bwd;
    constexpr bool KEEP = MINB < 4 && !ZOH && MODE != kCarry;
    using Lt = bwd::Layout<TIn>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = lane & 7, g = lane >> 3;  // channel lane and state group (also step group)
    const int b = blockIdx.y;
    const int seg = blockIdx.z;                           // segment of the time axis
    const int k_begin = seg * a.seg_tiles;                // its tiles
    const int k_end = min(a.ntile, k_begin + a.seg_tiles);
    const int d0 = blockIdx.x * kCh;
    const int row = warp * 8 + c;  // the lane's channel within the CTA
    const int d = d0 + row;
    const bool dvalid = d < a.dim;
    const int N = a.dstate;
    const bool gate = a.z != nullptr;

    float* bcq = reinterpret_cast<float*>(smem + Lt::OFF_BCQ);
    float4* q = reinterpret_cast<float4*>(smem + Lt::OFF_Q) + warp * kT * 8;        // [t][c]
    float* R = reinterpret_cast<float*>(smem + Lt::OFF_R) + warp * 3 * 8 * kPad;     // [k][c][t]
    float* part = reinterpret_cast<float*>(smem + Lt::OFF_PART) + warp * kT * kPartPitch;  // [t][col]

    // B/C rows of states past N stay zero in both stages: their states never move
    for (int i = tid; i < 2 * 2 * kNS * Lt::ROW / 16; i += kThreads) {
        const int stg = i / (2 * kNS * Lt::ROW / 16), rem = i - stg * (2 * kNS * Lt::ROW / 16);
        reinterpret_cast<uint4*>(smem + stg * Lt::STAGE + Lt::OFF_B)[rem] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();

    // per-state constants of the lane's 4 states, as pairs (states 4g+2p, 4g+2p+1) for the
    // packed f32x2 arithmetic; el(arr, j) is state 4g+j
    float2 Aj[2], A2[2], invA[2];
    auto el = [](float2* v, int j) -> float& { return (j & 1) ? v[j >> 1].y : v[j >> 1].x; };
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = a.nb + 4 * g + j;  // state (this block's 4g + j)
        el(Aj, j) = (dvalid && n < N) ? a.A[(long long)d * N + n] : 0.f;
        el(A2, j) = el(Aj, j) * kLog2e;
        el(invA, j) = 1.f / el(Aj, j);  // hold only; infinite at A = 0, where the series branch is taken
    }
    // Bbar x / (B x): Delta, or the hold's (exp(Delta A) - 1) / A (series for small |Delta A|)
    auto kfac = [&](float dt, float X, float abar, int j) -> float {
        if (!ZOH) return dt;
        return fabsf(X) < kZohSeriesLimit ? dt * zoh_phi(X) : (abar - 1.f) * el(invA, j);
    };
    const float bias_c = (dvalid && a.bias) ? a.bias[d] : 0.f;
    const float D_once = (dvalid && a.D && a.nb == 0) ? a.D[d] : 0.f;  // the skip term, first state block only
    const long long chrow = ((long long)b * a.dim + d) * a.L;  // start of the channel's rows

    // state before the segment: the initial state (segment 0); in a full launch of a later
    // segment, segment 0's end state folded with the carries of segments 1 .. seg-1; from zero in
    // a carry launch
    const long long cstride = (long long)a.batch * a.dim * N;  // one segment's carries
    float h0v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = a.nb + 4 * g + j;  // state (this block's 4g + j)
        const bool sv = dvalid && n < N;
        float hv = 0.f;
        if (seg == 0) {
            hv = (a.h0 && sv) ? a.h0[((long long)b * a.dim + d) * N + n] : 0.f;
        } else if (MODE == kFull && sv) {
            const float2* cr = a.carry + ((long long)b * a.dim + d) * N + n;
            hv = cr[0].y;
            for (int q2 = 1; q2 < seg; ++q2) hv = fmaf(cr[q2 * cstride].x, hv, cr[q2 * cstride].y);
        }
        h0v[j] = hv;
    }
    float* ck = a.ckpt ? a.ckpt + (((long long)b * a.nslot) * a.dim + d) * kNS + 4 * g : nullptr;
    const long long ckstride = (long long)a.dim * kNS;  // floats between consecutive slots

    // Phase A: per (channel, step) quantities of tile k for this lane's channel c, steps
    // kSPL*g .. kSPL*g + kSPL-1.
    auto phase_a = [&](const uint8_t* st, int k, bool full) {
        const long long t0 = (long long)k * kT;
        float dl[kSPL], uu[kSPL], zz[kSPL], dyv[kSPL];
        row_steps<TIn>(st + Lt::OFF_DL + row * Lt::ROW, g, dl);
        row_steps<TIn>(st + Lt::OFF_U + row * Lt::ROW, g, uu);
        if (full) {
            row_steps<TIn>(st + Lt::OFF_DY + row * Lt::ROW, g, dyv);
            if (gate) row_steps<TIn>(st + Lt::OFF_Z + row * Lt::ROW, g, zz);
        }
#pragma unroll
        for (int j = 0; j < kSPL; j += 2) {
            float2 s2 = make_float2(dl[j] + bias_c, dl[j + 1] + bias_c);
            if (a.softplus) s2 = softplus2(s2);
            const float sv[2] = {s2.x, s2.y};
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int t = kSPL * g + j + i;
                const bool ok = dvalid && t0 + t < a.L;
                const float dt = ok ? sv[i] : 0.f;
                const float x = ok ? uu[j + i] : 0.f;
                float e = 0.f;
                if (full && ok) e = gate ? dyv[j + i] * silu_f(zz[j + i]) : dyv[j + i];
                q[t * 8 + c] = make_float4(dt, dt * x, e, x);
            }
        }
    };

    // B and C of the tile, one step per row of bcq: item (t, kind, quad) moves 4 states of B
    // (kind 0) or C (kind 1) at step t.  (C is stale and unused in the forward sweep.)
    auto transpose_bc = [&](const uint8_t* st) {
        constexpr int RW = Lt::ROW / (int)sizeof(TIn);
#pragma unroll
        for (int r = 0; r < kT * 8 / kThreads; ++r) {
            const int it = tid + r * kThreads;
            const int t = it % kT, grp = it / kT;
            const int kind = grp >> 2, n0 = 4 * (grp & 3);
            const TIn* S = reinterpret_cast<const TIn*>(st + (kind ? Lt::OFF_C : Lt::OFF_B));
            const float4 v = make_float4(In<TIn>::to_f32(S[(n0 + 0) * RW + t]), In<TIn>::to_f32(S[(n0 + 1) * RW + t]),
                                         In<TIn>::to_f32(S[(n0 + 2) * RW + t]), In<TIn>::to_f32(S[(n0 + 3) * RW + t]));
            *reinterpret_cast<float4*>(bcq + t * kBcqPitch + 16 * kind + n0) = v;
        }
    };

    // one step of the lane's 4 states: h <- Abar h + Bbar x (packed pairs for the simplified B);
    // abar_out, when given, receives the step's Abar pairs
    auto advance = [&](float2 (&h)[2], const float4& qq, const float4& bq, float2* abar_out = nullptr) {
        const float2 bp[2] = {make_float2(bq.x, bq.y), make_float2(bq.z, bq.w)};
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const float2 X = fmul2(make_float2(qq.x, qq.x), A2[p]);
            const float2 ab = make_float2(ex2_approx(X.x), ex2_approx(X.y));
            if (abar_out != nullptr) abar_out[p] = ab;
            if constexpr (!ZOH) {
                h[p] = ffma2(ab, h[p], fmul2(make_float2(qq.y, qq.y), bp[p]));
            } else {
                const float kx0 = kfac(qq.x, X.x, ab.x, 2 * p) * qq.w, kx1 = kfac(qq.x, X.y, ab.y, 2 * p + 1) * qq.w;
                h[p] = ffma2(ab, h[p], fmul2(make_float2(kx0, kx1), bp[p]));
            }
        }
    };

    // ---------------------------------------------------------------- forward sweep: checkpoints
    if (MODE == kCarry || (MODE == kFull && a.nslot > 1 && !a.ck_given)) {
        float2 h[2] = {make_float2(h0v[0], h0v[1]), make_float2(h0v[2], h0v[3])};
        float sumdt = 0.f;  // carry launch: sum of Delta over the segment
        if (VEC) load_tile<TIn, VEC>(smem + (k_begin & 1) * Lt::STAGE, a, b, d0, k_begin, false);
        for (int k = k_begin; k < k_end; ++k) {
            uint8_t* st = smem + (k & 1) * Lt::STAGE;
            if (VEC) {
                if (k + 1 < k_end) {
                    load_tile<TIn, VEC>(smem + ((k + 1) & 1) * Lt::STAGE, a, b, d0, k + 1, false);
                    cp_async_wait<1>();
                } else {
                    cp_async_wait<0>();
                }
            } else {
                load_tile<TIn, VEC>(st, a, b, d0, k, false);
            }
            __syncthreads();
            transpose_bc(st);
            phase_a(st, k, false);
            __syncthreads();
#pragma unroll 1
            for (int s = 0; s < kSlots; ++s) {
                const int gs = kSlots * k + s;
                if (gs >= a.nslot) break;
                if (MODE == kFull && gs >= 1 && dvalid)
                    *reinterpret_cast<float4*>(ck + gs * ckstride) = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
#pragma unroll
                for (int i = 0; i < bwd::kSlot; ++i) {
                    const int t = s * bwd::kSlot + i;
                    const float4 qq = q[t * 8 + c];
                    const float4 bq = *reinterpret_cast<const float4*>(bcq + t * kBcqPitch + 4 * g);
                    advance(h, qq, bq);
                    if (MODE == kCarry) sumdt += qq.x;
                }
            }
            __syncthreads();
        }
        if constexpr (MODE == kCarry) {
            // (prod Abar = 2^(A log2(e) sum Delta), end state from the segment's own start)
            if (dvalid) {
                float2* cw = a.carry + (long long)seg * cstride + ((long long)b * a.dim + d) * N;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n = a.nb + 4 * g + j;
                    if (n < N) cw[n] = make_float2(ex2_approx(el(A2, j) * sumdt), el(h, j));
                }
            }
            return;
        }
    }
    // ---------------------------------------------------------------- reverse sweep
    // mu = dL/dh at the segment's end: dlast for the last segment; in a full launch of an earlier
    // segment zero (its own part only); in a correction launch the gradient carried in from the
    // later segments, folded back from the last one (whose own walk started from dlast, so that its
    // mu_local is already its whole start gradient): mu_end(s) = mu_start(s+1) with
    // mu_start(S-1) = mu_local(S-1) and mu_start(q) = mu_local(q) + P(q) mu_start(q+1)
    float2 mu[2], dAacc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    float thr = 0.f;  // correction launch: stop once every |mu| is at most this
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = a.nb + 4 * g + j;  // state (this block's 4g + j)
        const bool sv = dvalid && n < N;
        const long long sn = ((long long)b * a.dim + d) * N + n;
        float m = (a.dlast && sv) ? a.dlast[sn] : 0.f;
        if (MODE == kFull && seg != a.nseg - 1) m = 0.f;
        if (MODE == kCorr && sv) {
            m = a.mu_local[(a.nseg - 1) * cstride + sn];
            for (int q2 = a.nseg - 2; q2 > seg; --q2) m = fmaf(a.carry[q2 * cstride + sn].x, m, a.mu_local[q2 * cstride + sn]);
            // gradient at the initial state: segment 0's own part plus what reaches it through
            // the whole of segment 0
            if (seg == 0 && a.dh0) a.dh0[sn] = fmaf(a.carry[sn].x, m, a.mu_local[sn]);
        }
        el(mu, j) = m;
        thr = fmaxf(thr, fabsf(m));
    }
    thr = thr <= 3.4028234663852886e38f ? thr * kDropBelow : 0.f;  // (an infinite or NaN gradient is never dropped)
    float dD_acc = 0.f, dbias_acc = 0.f;
    const int col = (c >> 2) * 16 + 4 * g + (c & 3);  // this lane's dC/dB column after the scatter
    // The checkpoints of the next tile's slots are prefetched into L2 one tile ahead, so that
    // each slot's recomputation starts from an L2 hit rather than waiting on HBM.
    auto prefetch_ck = [&](int k) {
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
            const int gs = kSlots * k + s;
            if (dvalid && gs >= 1 && gs < a.nslot) prefetch_l2(ck + gs * ckstride);
        }
    };
    prefetch_ck(k_end - 1);
    if (VEC) load_tile<TIn, VEC>(smem + ((k_end - 1) & 1) * Lt::STAGE, a, b, d0, k_end - 1, true);
#pragma unroll 1
    for (int k = k_end - 1; k >= k_begin; --k) {
        uint8_t* st = smem + (k & 1) * Lt::STAGE;
        const long long t0 = (long long)k * kT;
        if (k > k_begin) prefetch_ck(k - 1);
        if (VEC) {
            if (k > k_begin) {
                load_tile<TIn, VEC>(smem + ((k - 1) & 1) * Lt::STAGE, a, b, d0, k - 1, true);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
        } else {
            load_tile<TIn, VEC>(st, a, b, d0, k, true);
        }
        __syncthreads();
        transpose_bc(st);
        phase_a(st, k, MODE != kCorr);  // a correction sees no output gradient: e = 0
        __syncthreads();

#pragma unroll 1
        for (int s = kSlots - 1; s >= 0; --s) {
            const int gs = kSlots * k + s;
            if (gs >= a.nslot) continue;  // wholly past L: nothing moves there
            float2 h[2];
            if (gs == 0) {
                h[0] = make_float2(h0v[0], h0v[1]);
                h[1] = make_float2(h0v[2], h0v[3]);
            } else {
                const float4 v = dvalid ? *reinterpret_cast<const float4*>(ck + gs * ckstride) : make_float4(0.f, 0.f, 0.f, 0.f);
                h[0] = make_float2(v.x, v.y);
                h[1] = make_float2(v.z, v.w);
            }
            // recompute the slot's states (and, KEEP, their Abar)
            float2 hist[bwd::kSlot][2];
            float2 abk[KEEP ? bwd::kSlot : 1][2];
#pragma unroll
            for (int i = 0; i < bwd::kSlot; ++i) {
                const int t = s * bwd::kSlot + i;
                advance(h, q[t * 8 + c], *reinterpret_cast<const float4*>(bcq + t * kBcqPitch + 4 * g),
                        KEEP ? abk[KEEP ? i : 0] : nullptr);
                hist[i][0] = h[0];
                hist[i][1] = h[1];
            }
            // walk the slot in reverse
#pragma unroll
            for (int i = bwd::kSlot - 1; i >= 0; --i) {
                const int t = s * bwd::kSlot + i;
                const float4 qq = q[t * 8 + c];  // (Delta, Delta x, e, x)
                const float4 bq = *reinterpret_cast<const float4*>(bcq + t * kBcqPitch + 4 * g);
                const float4 cq = *reinterpret_cast<const float4*>(bcq + t * kBcqPitch + 16 + 4 * g);
                const float bv[4] = {bq.x, bq.y, bq.z, bq.w};
                const float cv[4] = {cq.x, cq.y, cq.z, cq.w};
                float v[8];
                float sdt = 0.f, sub = 0.f, sch = 0.f;
                if constexpr (!ZOH) {
                    // state pairs in packed f32x2 arithmetic
                    const float2 dq = make_float2(qq.x, qq.x), dxq = make_float2(qq.y, qq.y);
                    const float2 eq = make_float2(qq.z, qq.z), xq = make_float2(qq.w, qq.w);
                    const float2 ndxq = make_float2(-qq.y, -qq.y);
                    const float2 bp[2] = {make_float2(bq.x, bq.y), make_float2(bq.z, bq.w)};
                    const float2 cp[2] = {make_float2(cq.x, cq.y), make_float2(cq.z, cq.w)};
                    float2 sdt2 = make_float2(0.f, 0.f), sub2 = sdt2, sch2 = sdt2;
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        const float2 ht = hist[i][p];
                        float2 ab;
                        if constexpr (KEEP) {
                            ab = abk[i][p];
                        } else {
                            const float2 X = fmul2(dq, A2[p]);
                            ab = make_float2(ex2_approx(X.x), ex2_approx(X.y));
                        }
                        const float2 lam = ffma2(eq, cp[p], mu[p]);
                        sch2 = ffma2(cp[p], ht, sch2);
                        const float2 vc = fmul2(eq, ht);
                        const float2 ah = ffma2(ndxq, bp[p], ht);  // a_t h_{t-1}
                        const float2 vb = fmul2(lam, dxq);
                        v[2 * p] = vc.x; v[2 * p + 1] = vc.y;
                        v[4 + 2 * p] = vb.x; v[5 + 2 * p] = vb.y;
                        sub2 = ffma2(lam, bp[p], sub2);
                        sdt2 = ffma2(lam, ffma2(Aj[p], ah, fmul2(bp[p], xq)), sdt2);
                        dAacc[p] = ffma2(fmul2(lam, ah), dq, dAacc[p]);
                        mu[p] = fmul2(ab, lam);
                    }
                    sdt = sdt2.x + sdt2.y;
                    sub = sub2.x + sub2.y;
                    sch = sch2.x + sch2.y;
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float ht = el(hist[i], j);
                        const float X = qq.x * el(A2, j), ab = ex2_approx(X);
                        const float lam = fmaf(qq.z, cv[j], el(mu, j));
                        sch = fmaf(cv[j], ht, sch);
                        v[j] = qq.z * ht;
                        // h_t = a h_{t-1} + k B x: dk/dDelta = a, dk/dA = Delta^2 psi(Delta A)
                        const float kf = kfac(qq.x, X, ab, j);
                        const float bxs = bv[j] * qq.w;  // B x
                        const float ah = fmaf(-kf, bxs, ht);
                        const float dkdA = fabsf(X) < kZohSeriesLimit ? qq.x * qq.x * zoh_psi(X)
                                                                      : (qq.x * ab - kf) * el(invA, j);
                        v[4 + j] = lam * kf * qq.w;
                        sub = fmaf(lam * kf, bv[j], sub);
                        sdt = fmaf(lam, fmaf(el(Aj, j), ah, ab * bxs), sdt);
                        el(dAacc, j) = fmaf(lam, fmaf(qq.x, ah, dkdA * bxs), el(dAacc, j));
                        el(mu, j) = ab * lam;
                    }
                }
                part[t * kPartPitch + col] = reduce_scatter8(v, lane);
                const float r3 = reduce_scatter3(sdt, sub, sch, lane);
                if (g < 3) R[(g * 8 + c) * kPad + t] = r3;
            }
        }
        __syncwarp();

        // Phase C: per (channel, step) gradients for channel c, steps kSPL*g .. of the tile
        {
            float dl[kSPL], zz[kSPL], dyv[kSPL], o_du[kSPL], o_dd[kSPL], o_dz[kSPL];
            row_steps<TIn>(st + Lt::OFF_DL + row * Lt::ROW, g, dl);
            row_steps<TIn>(st + Lt::OFF_DY + row * Lt::ROW, g, dyv);
            if (gate) row_steps<TIn>(st + Lt::OFF_Z + row * Lt::ROW, g, zz);
#pragma unroll
            for (int j = 0; j < kSPL; ++j) {
                const int t = kSPL * g + j;
                const bool ok = dvalid && t0 + t < a.L;
                const float4 qq = q[t * 8 + c];
                const float sdt = R[(0 * 8 + c) * kPad + t];
                const float sub = R[(1 * 8 + c) * kPad + t];
                const float sch = R[(2 * 8 + c) * kPad + t];
                const float sarg = dl[j] + bias_c;
                const float gdt = a.softplus ? sdt * sigmoid_approx(sarg) : sdt;
                o_dd[j] = gdt;
                // the skip term D x belongs to no state: only the first state block adds it
                o_du[j] = fmaf(sub, ZOH ? 1.f : qq.x, qq.z * D_once);  // the hold's k already holds Delta
                if (gate) {
                    const float sg = sigmoid_approx(zz[j]);
                    const float ypre = fmaf(D_once, qq.w, sch);
                    o_dz[j] = dyv[j] * ypre * sg * fmaf(zz[j], 1.f - sg, 1.f);
                }
                if (ok) {
                    dD_acc = fmaf(qq.z, qq.w, dD_acc);
                    dbias_acc += gdt;
                }
            }
            if (dvalid) {
                const long long tg0 = t0 + kSPL * g, off = chrow + tg0;
                if (a.acc_du != nullptr) {  // state blocks or segments: add into the fp32 accumulators
                    const bool first = MODE == kFull && a.nb == 0;
#pragma unroll
                    for (int j = 0; j < kSPL; ++j) {
                        if (tg0 + j >= a.L) break;
                        a.acc_du[off + j] = (first ? 0.f : a.acc_du[off + j]) + o_du[j];
                        a.acc_dd[off + j] = (first ? 0.f : a.acc_dd[off + j]) + o_dd[j];
                        if (MODE == kFull && gate && a.acc_dz)
                            a.acc_dz[off + j] = (first ? 0.f : a.acc_dz[off + j]) + o_dz[j];
                    }
                } else {
                    store_steps<TIn, VEC>(static_cast<TIn*>(a.du) + off, tg0, a.L, o_du);
                    store_steps<TIn, VEC>(static_cast<TIn*>(a.ddelta) + off, tg0, a.L, o_dd);
                    if (gate && a.dz) store_steps<TIn, VEC>(static_cast<TIn*>(a.dz) + off, tg0, a.L, o_dz);
                }
            }
        }
        __syncthreads();

        // dB, dC of the tile: sum the 4 warps' partials, one atomic per 4 steps per CTA
        {
            const float* P = reinterpret_cast<const float*>(smem + Lt::OFF_PART);
#pragma unroll
            for (int rep = 0; rep < kT * 8 / kThreads; ++rep) {
                const int gi = tid + rep * kThreads;  // 32 columns x kT/4 groups of 4 steps
                const int colr = gi / (kT / 4), tq = gi % (kT / 4);
                const int kind = colr >> 4, n = a.nb + (colr & 15);
                if (n < N && (MODE != kCorr || kind == 1)) {  // a correction changes dB only
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int w = 0; w < kWarps; ++w)
#pragma unroll
                        for (int tt = 0; tt < 4; ++tt) acc[tt] += P[w * kT * kPartPitch + (tq * 4 + tt) * kPartPitch + colr];
                    const long long tg = t0 + tq * 4;
                    float* dst = (kind ? a.dB : a.dC) + ((long long)b * N + n) * a.L + tg;
                    if (VEC) {
                        if (tg < a.L) red_add_v4(dst, make_float4(acc[0], acc[1], acc[2], acc[3]));
                    } else {
#pragma unroll
                        for (int tt = 0; tt < 4; ++tt)
                            if (tg + tt < a.L) atomicAdd(dst + tt, acc[tt]);
                    }
                }
            }
        }
        if constexpr (MODE == kCorr) {
            // stop once the carried-in gradient has decayed in every lane of the CTA (the copies
            // of the next tile are still in flight: let them land first)
            bool small = true;
#pragma unroll
            for (int j = 0; j < 4; ++j) small = small && fabsf(el(mu, j)) <= thr;
            if (__syncthreads_and(small)) {
                if (VEC) cp_async_wait<0>();
                break;
            }
        } else {
            __syncthreads();
        }
    }

    // ---------------------------------------------------------------- per-channel results
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = a.nb + 4 * g + j;  // state (this block's 4g + j)
        if (dvalid && n < N) {
            atomicAdd(a.dA + (long long)d * N + n, el(dAacc, j));
            // gradient at the segment's start: the initial state's gradient when the time axis
            // is not split; with a split, this segment's own part (the correction launch of
            // segment 0 combines them)
            const long long sn = ((long long)b * a.dim + d) * N + n;
            if (MODE == kFull && a.nseg > 1) a.mu_local[(long long)seg * cstride + sn] = el(mu, j);
            else if (MODE == kFull && a.dh0) a.dh0[sn] = el(mu, j);
        }
    }
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, 8);
    dD_acc += __shfl_xor_sync(0xffffffffu, dD_acc, 16);
    dbias_acc += __shfl_xor_sync(0xffffffffu, dbias_acc, 8);
    dbias_acc += __shfl_xor_sync(0xffffffffu, dbias_acc, 16);
    if (dvalid && g == 0) {
        if (MODE == kFull && a.dD && a.nb == 0) atomicAdd(a.dD + d, dD_acc);
        if (a.dbias) atomicAdd(a.dbias + d, dbias_acc);
    }
}

// fp32 accumulators of the state-block launches -> the per-(channel, step) gradients in the
// storage type.
template <typename TIn>
__global__ void __launch_bounds__(256) bwd_finish_kernel(const BwdArgs a, long long n) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        store_out<TIn>(static_cast<TIn*>(a.du) + i, a.acc_du[i]);
        store_out<TIn>(static_cast<TIn*>(a.ddelta) + i, a.acc_dd[i]);
        if (a.acc_dz != nullptr) store_out<TIn>(static_cast<TIn*>(a.dz) + i, a.acc_dz[i]);
    }
}

}  // namespace mscan
