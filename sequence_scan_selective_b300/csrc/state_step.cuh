// Recurrent decoding step: one token for every (batch, channel), state updated in place.
//
// Recurrent form of the discretised SSM (visual guide to Mamba and SSMs, section 2.4) used for
// autoregressive inference with constant work per token (news write-up, "architecture" section):
//   h <- exp(Delta A) h + Delta B x,   y = (C.h + D x) silu(z)
// (with the exact zero-order hold, Delta B x becomes (exp(Delta A) - 1) / A * B x).
//
// The fp32 state [b, d, N] dominates the traffic (read + write).  Each thread owns Q = min(N, 8)
// consecutive states of one channel (S = ceil(N / Q) threads per channel, next to each other in
// the warp) and moves them with 128-bit loads and stores, for several batch rows at once; A[d, n..]
// arrives with 128-bit loads as well, once for those rows, and B[b, :], C[b, :] -- the same for
// every channel of a batch row -- are widened once per block into shared memory.  The S threads of
// a channel each form Delta and the gate themselves (a few dozen operations, cheaper than an
// exchange) and combine their partial C.h with shuffles.
#pragma once
#include <stdint.h>

#include "ptx.cuh"
#include "common.cuh"

namespace mscan {

struct StepArgs {
    float* state;
    const void* x;
    const void* delta;
    const void* z;
    const void* B;
    const void* C;
    const float* A;
    const float* D;
    const float* bias;
    void* y;
    int batch, dim, dstate;
    int softplus;
    int zoh;  // nonzero: exact zero-order hold for B
};

constexpr int kStepRows = 4;  // batch rows per thread (decode step)

// VEC: N is a multiple of Q (= 8, or 4 for N = 4) and every row is aligned for vector access;
// otherwise element-wise accesses with bounds checks on the state index.
//
// Thread (channel d, state group q) walks kStepRows batch rows of the same channel: A[d, ...],
// the bias and D are loaded once and reused, and the rows' state loads are independent, so each
// thread keeps several 128-bit loads in flight.  Block = 256 / S channels x kStepRows rows.
template <typename TIn, int NP, bool VEC>
__global__ void __launch_bounds__(256, 3) state_step_kernel(const StepArgs a) {
    constexpr int Q = NP < 8 ? NP : 8;   // states per thread
    constexpr int S = NP / Q;            // threads per channel
    static_assert(Q % 4 == 0 && 32 % S == 0, "a channel's threads must sit in one warp");
    const int d = blockIdx.x * (256 / S) + (int)threadIdx.x / S;
    const int q = (int)threadIdx.x % S;
    const int b0 = blockIdx.y * kStepRows;
    const bool valid = d < a.dim;
    const int N = a.dstate;
    const int n0 = q * Q;
    // B, C of the block's batch rows (the same for all its channels), widened once into shared memory
    __shared__ __align__(16) float Bs[kStepRows][NP], Cs[kStepRows][NP];
    for (int i = threadIdx.x; i < kStepRows * NP; i += blockDim.x) {
        const int r = i / NP, n = i % NP, b = b0 + r;
        const bool in = b < a.batch && n < N;
        const long long off = (long long)b * N + n;
        Bs[r][n] = in ? In<TIn>::to_f32(static_cast<const TIn*>(a.B)[off]) : 0.f;
        Cs[r][n] = in ? In<TIn>::to_f32(static_cast<const TIn*>(a.C)[off]) : 0.f;
    }
    __syncthreads();
    float Av[Q];
#pragma unroll
    for (int i = 0; i < Q; ++i) Av[i] = 0.f;
    float bias = 0.f, Dd = 0.f;
    if (valid) {
        const float* Ap = a.A + (long long)d * N + n0;
        if (VEC) {
#pragma unroll
            for (int i = 0; i < Q; i += 4) {
                const float4 w = __ldg(reinterpret_cast<const float4*>(Ap + i));
                Av[i] = w.x; Av[i + 1] = w.y; Av[i + 2] = w.z; Av[i + 3] = w.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < Q; ++i) Av[i] = (n0 + i < N) ? Ap[i] : 0.f;
        }
        bias = a.bias ? a.bias[d] : 0.f;
        Dd = a.D ? a.D[d] : 0.f;
    }
    // all rows' loads first (the stores of one row could alias the next row's loads in the
    // compiler's view, so it would not move them ahead by itself), then the updates
    const int nr = min(kStepRows, a.batch - b0);
    float hv[kStepRows][Q], xv[kStepRows], dv[kStepRows], zv[kStepRows];
#pragma unroll
    for (int r = 0; r < kStepRows; ++r) {
        const int b = b0 + (r < nr ? r : 0);
        const long long ch = (long long)b * a.dim + (valid ? d : 0);
        const float* hp = a.state + ch * N + n0;
        xv[r] = In<TIn>::to_f32(static_cast<const TIn*>(a.x)[ch]);
        dv[r] = In<TIn>::to_f32(static_cast<const TIn*>(a.delta)[ch]);
        zv[r] = a.z ? In<TIn>::to_f32(static_cast<const TIn*>(a.z)[ch]) : 0.f;
        if (VEC) {
#pragma unroll
            for (int i = 0; i < Q; i += 4) {
                const float4 v = *reinterpret_cast<const float4*>(hp + i);
                hv[r][i] = v.x; hv[r][i + 1] = v.y; hv[r][i + 2] = v.z; hv[r][i + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < Q; ++i) hv[r][i] = (n0 + i < N) ? hp[i] : 0.f;
        }
    }
#pragma unroll
    for (int r = 0; r < kStepRows; ++r) {
        if (r >= nr) break;  // uniform over the block
        const long long ch = (long long)(b0 + r) * a.dim + d;
        float dt = dv[r] + bias;
        const float sp = softplus1(dt);
        dt = a.softplus ? sp : dt;
        const float du = dt * xv[r];
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < Q; ++i) {
            const float xe = dt * (Av[i] * kLog2e);
            const float abar = ex2_approx(xe);
            float bx = du;  // Bbar x / B
            if (a.zoh) bx = fabsf(xe) < kZohSeriesLimit ? du * zoh_phi(xe) : (abar - 1.f) * (xv[r] / Av[i]);
            hv[r][i] = fmaf(abar, hv[r][i], bx * Bs[r][n0 + i]);
            part = fmaf(Cs[r][n0 + i], hv[r][i], part);
        }
        if (valid) {
            float* hp = a.state + ch * N + n0;
            if (VEC) {
#pragma unroll
                for (int i = 0; i < Q; i += 4)
                    *reinterpret_cast<float4*>(hp + i) = make_float4(hv[r][i], hv[r][i + 1], hv[r][i + 2], hv[r][i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < Q; ++i)
                    if (n0 + i < N) hp[i] = hv[r][i];
            }
        }
#pragma unroll
        for (int m = S / 2; m >= 1; m /= 2) part += __shfl_xor_sync(0xffffffffu, part, m);
        if (valid && q == 0) {
            float yv = fmaf(Dd, xv[r], part);
            if (a.z) yv *= silu_f(zv[r]);
            store_out<TIn>(static_cast<TIn*>(a.y) + ch, yv);
        }
    }
}

}  // namespace mscan
