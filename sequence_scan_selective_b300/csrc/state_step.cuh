// Recurrent decoding step: one token for every (batch, channel), state updated in place.
//
// Recurrent form of the discretised SSM (visual guide to Mamba and SSMs, section 2.4) used for
// autoregressive inference with constant work per token (news write-up, "architecture" section):
//   h <- exp(Delta A) h + Delta B x,   y = (C.h + D x) silu(z)
// (with the exact zero-order hold, Delta B x becomes (exp(Delta A) - 1) / A * B x).
// The state [b, d, N] fp32 dominates the traffic (read + write); each thread owns 4 consecutive
// states of one channel so that a warp streams 512 contiguous bytes of state per 128-bit access,
// and the NP/4 lanes of a channel combine their partial C.h with warp shuffles.
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

template <typename TIn, int NP, bool VEC4>
__global__ void __launch_bounds__(256) state_step_kernel(const StepArgs a) {
    constexpr int Q = 4;        // states per thread
    constexpr int S = NP / Q;   // lanes per channel
    static_assert(32 % S == 0, "a channel's lanes must sit in one warp");
    const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long ch = gt / S;
    const int q = (int)(gt % S);
    const long long nch = (long long)a.batch * a.dim;
    const bool valid = ch < nch;
    const int N = a.dstate;
    float part = 0.f;
    float xv = 0.f;
    int d = 0;
    if (valid) {
        const int b = (int)(ch / a.dim);
        d = (int)(ch % a.dim);
        const TIn* X = static_cast<const TIn*>(a.x);
        const TIn* Dl = static_cast<const TIn*>(a.delta);
        xv = In<TIn>::to_f32(X[ch]);
        float dt = In<TIn>::to_f32(Dl[ch]) + (a.bias ? a.bias[d] : 0.f);
        if (a.softplus) dt = softplus1(dt);
        const float du = dt * xv;
        const TIn* Bp = static_cast<const TIn*>(a.B) + (long long)b * N;
        const TIn* Cp = static_cast<const TIn*>(a.C) + (long long)b * N;
        const float* Ap = a.A + (long long)d * N;
        float* hp = a.state + ch * N + q * Q;
        const int n0 = q * Q;
        float hv[Q];
        if (VEC4) {
            const float4 v = *reinterpret_cast<const float4*>(hp);
            hv[0] = v.x; hv[1] = v.y; hv[2] = v.z; hv[3] = v.w;
        } else {
#pragma unroll
            for (int i = 0; i < Q; ++i) hv[i] = (n0 + i < N) ? hp[i] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < Q; ++i) {
            const int n = n0 + i;
            if (VEC4 || n < N) {
                const float xe = dt * (Ap[n] * kLog2e);
                const float abar = ex2_approx(xe);
                float bx = du;  // Bbar x / B
                if (a.zoh) bx = fabsf(xe) < kZohSeriesLimit ? du * zoh_phi(xe) : (abar - 1.f) * (xv / Ap[n]);
                hv[i] = fmaf(abar, hv[i], bx * In<TIn>::to_f32(Bp[n]));
                part = fmaf(In<TIn>::to_f32(Cp[n]), hv[i], part);
            }
        }
        if (VEC4) {
            *reinterpret_cast<float4*>(hp) = make_float4(hv[0], hv[1], hv[2], hv[3]);
        } else {
#pragma unroll
            for (int i = 0; i < Q; ++i)
                if (n0 + i < N) hp[i] = hv[i];
        }
    }
#pragma unroll
    for (int m = S / 2; m >= 1; m /= 2) part += __shfl_xor_sync(0xffffffffu, part, m);
    if (valid && q == 0) {
        float yv = fmaf(a.D ? a.D[d] : 0.f, xv, part);
        if (a.z) yv *= silu_f(In<TIn>::to_f32(static_cast<const TIn*>(a.z)[ch]));
        store_out<TIn>(static_cast<TIn*>(a.y) + ch, yv);
    }
}

}  // namespace mscan
