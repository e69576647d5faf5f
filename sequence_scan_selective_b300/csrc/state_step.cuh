// Recurrent decoding step: one token for every (batch, channel), state updated in place.
//
// Recurrent form of the discretised SSM (visual guide to Mamba and SSMs, section 2.4) used for
// autoregressive inference with constant work per token (news write-up, "architecture" section):
//   h <- exp(Delta A) h + Delta B x,   y = (C.h + D x) silu(z)
// (with the exact zero-order hold, Delta B x becomes (exp(Delta A) - 1) / A * B x).
//
// The fp32 state [b, d, N] dominates the traffic (read + write).  Each thread owns Q = min(N, 8)
// consecutive states of one channel (S = ceil(N / Q) threads per channel, next to each other in
// the warp) and moves them with 128-bit loads and stores; A[d, n..] arrives with 128-bit loads as
// well, and B[b, n..], C[b, n..] -- the same for every channel of a batch row, so one broadcast
// transaction per warp -- with 64-bit (bf16) or 128-bit (fp32) loads.  The S threads of a
// channel each form Delta and the gate themselves (a few dozen operations, cheaper than an
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

// 4 consecutive inputs at p (16-byte aligned for fp32, 8-byte aligned for bf16) -> fp32
template <typename TIn>
__device__ __forceinline__ void load4(const TIn* p, float* v);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float* v) {
    const float4 q = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
template <>
__device__ __forceinline__ void load4<uint16_t>(const uint16_t* p, float* v) {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
    v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xffff0000u);
}

// VEC: N is a multiple of Q (= 8, or 4 for N = 4) and every row is aligned for vector access;
// otherwise element-wise accesses with bounds checks on the state index.
template <typename TIn, int NP, bool VEC>
__global__ void __launch_bounds__(256) state_step_kernel(const StepArgs a) {
    constexpr int Q = NP < 8 ? NP : 8;   // states per thread
    constexpr int S = NP / Q;            // threads per channel
    static_assert(Q % 4 == 0 && 32 % S == 0, "a channel's threads must sit in one warp");
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
        xv = In<TIn>::to_f32(static_cast<const TIn*>(a.x)[ch]);
        float dt = In<TIn>::to_f32(static_cast<const TIn*>(a.delta)[ch]) + (a.bias ? a.bias[d] : 0.f);
        if (a.softplus) dt = softplus1(dt);
        const float du = dt * xv;
        const int n0 = q * Q;
        const TIn* Bp = static_cast<const TIn*>(a.B) + (long long)b * N + n0;
        const TIn* Cp = static_cast<const TIn*>(a.C) + (long long)b * N + n0;
        const float* Ap = a.A + (long long)d * N + n0;
        float* hp = a.state + ch * N + n0;
        float hv[Q], Av[Q], Bv[Q], Cv[Q];
        if (VEC) {
#pragma unroll
            for (int i = 0; i < Q; i += 4) {
                const float4 v = *reinterpret_cast<const float4*>(hp + i);
                hv[i] = v.x; hv[i + 1] = v.y; hv[i + 2] = v.z; hv[i + 3] = v.w;
                const float4 w = __ldg(reinterpret_cast<const float4*>(Ap + i));
                Av[i] = w.x; Av[i + 1] = w.y; Av[i + 2] = w.z; Av[i + 3] = w.w;
                load4<TIn>(Bp + i, Bv + i);
                load4<TIn>(Cp + i, Cv + i);
            }
        } else {
#pragma unroll
            for (int i = 0; i < Q; ++i) {
                const bool in = n0 + i < N;
                hv[i] = in ? hp[i] : 0.f;
                Av[i] = in ? Ap[i] : 0.f;
                Bv[i] = in ? In<TIn>::to_f32(Bp[i]) : 0.f;
                Cv[i] = in ? In<TIn>::to_f32(Cp[i]) : 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < Q; ++i) {
            const float xe = dt * (Av[i] * kLog2e);
            const float abar = ex2_approx(xe);
            float bx = du;  // Bbar x / B
            if (a.zoh) bx = fabsf(xe) < kZohSeriesLimit ? du * zoh_phi(xe) : (abar - 1.f) * (xv / Av[i]);
            hv[i] = fmaf(abar, hv[i], bx * Bv[i]);
            part = fmaf(Cv[i], hv[i], part);
        }
        if (VEC) {
#pragma unroll
            for (int i = 0; i < Q; i += 4)
                *reinterpret_cast<float4*>(hp + i) = make_float4(hv[i], hv[i + 1], hv[i + 2], hv[i + 3]);
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
