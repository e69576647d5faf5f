// Element access, step-size map and gate shared by the scan and decode kernels.
//
// The step-size map and the gate are the per-element parts of the selective SSM (visual guide to
// Mamba and SSMs, sections 2.3 and 3.2; the gate multiplies the SSM output by silu(z)):
//   Delta = softplus(delta + delta_bias)   (or delta + delta_bias)
//   gate  = silu(z) = z * sigmoid(z)
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace mscan {

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s bound on any wait inside a kernel

// Nonzero: some kernel abandoned a bounded wait.  One copy per translation unit (each compiles to
// its own module); the host reads every unit's copy.
static __device__ int g_status;

// ------------------------------------------------------------------------------ element access
// Inputs are fp32 or bf16 (held as uint16_t bit patterns); arithmetic is always fp32.
template <typename TIn>
struct In;
template <>
struct In<float> {
    __device__ static __forceinline__ float to_f32(float x) { return x; }
};
template <>
struct In<uint16_t> {
    __device__ static __forceinline__ float to_f32(uint16_t x) { return bf16_bits_to_f32(x); }
};

template <typename TIn>
__device__ __forceinline__ void store_out(TIn* p, float v);
template <>
__device__ __forceinline__ void store_out<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_out<uint16_t>(uint16_t* p, float v) {
    *p = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xffffu);
}

// ------------------------------------------------------------------------------ step size, gate
// softplus(x) = max(x, 0) + log1p(e) with e = exp(-|x|) in (0, 1].  log1p(e) = e * P(e), P the
// degree-6 Chebyshev interpolant of log1p(e)/e on [0, 1] in monomial form (gen_softplus_poly.py
// derives the coefficients; fp32 relative error of the log1p term below 1.6e-6).  No threshold
// is needed: the form is exact in structure for every x, and NaN propagates through e.
__device__ __forceinline__ float2 softplus2(float2 x) {
    const float2 e = make_float2(ex2_approx(-fabsf(x.x) * kLog2e), ex2_approx(-fabsf(x.y) * kLog2e));
    float2 p = make_float2(0.013874484f, 0.013874484f);
    p = ffma2(p, e, make_float2(-0.06559031f, -0.06559031f));
    p = ffma2(p, e, make_float2(0.14829414f, 0.14829414f));
    p = ffma2(p, e, make_float2(-0.2345452f, -0.2345452f));
    p = ffma2(p, e, make_float2(0.33097526f, 0.33097526f));
    p = ffma2(p, e, make_float2(-0.499859f, -0.499859f));
    p = ffma2(p, e, make_float2(0.99999857f, 0.99999857f));
    return ffma2(e, p, make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)));
}

__device__ __forceinline__ float softplus1(float x) { return softplus2(make_float2(x, x)).x; }

// silu(z) = z / (1 + e^-z)
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.f + ex2_approx(-z * kLog2e)); }

__device__ __forceinline__ float sigmoid_approx(float x) { return rcp_approx(1.f + ex2_approx(-x * kLog2e)); }

__device__ __forceinline__ float2 silu2(float2 z) {
    const float2 e = make_float2(ex2_approx(-z.x * kLog2e), ex2_approx(-z.y * kLog2e));
    const float2 den = fadd2(e, make_float2(1.f, 1.f));
    return fmul2(z, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
}

// ------------------------------------------------------------------------------ zero-order hold
// The hold's factor (e^x - 1) / x and, for gradients, its derivative companion
// (x e^x - (e^x - 1)) / x^2, as Taylor series for small |x|.  The argument is given in base-2
// units, X = x log2(e) (the exponent the kernels already form for exp2), so the coefficients are
// ln2^k / (k+1)! and k ln2^(k-1) / (k+1)!; the series are used for |x| < 1/4, where six terms leave
// a relative error below 5e-8.
constexpr double kLn2d = 0.6931471805599453;
constexpr float kZohSeriesLimit = (float)(0.25 * 1.4426950408889634);  // |X| bound for the series

__device__ __forceinline__ float2 zoh_phi2(float2 X) {
    constexpr double l = kLn2d;
    const float2 c5 = make_float2((float)(l * l * l * l * l / 720.0), (float)(l * l * l * l * l / 720.0));
    float2 p = ffma2(c5, X, make_float2((float)(l * l * l * l / 120.0), (float)(l * l * l * l / 120.0)));
    p = ffma2(p, X, make_float2((float)(l * l * l / 24.0), (float)(l * l * l / 24.0)));
    p = ffma2(p, X, make_float2((float)(l * l / 6.0), (float)(l * l / 6.0)));
    p = ffma2(p, X, make_float2((float)(l / 2.0), (float)(l / 2.0)));
    return ffma2(p, X, make_float2(1.f, 1.f));
}

__device__ __forceinline__ float zoh_phi(float X) { return zoh_phi2(make_float2(X, X)).x; }

// psi(x) = (x e^x - (e^x - 1)) / x^2 = sum_{k>=1} k x^(k-1) / (k+1)!, argument in base-2 units.
__device__ __forceinline__ float zoh_psi(float X) {
    constexpr double l = kLn2d;
    float p = (float)(6.0 * l * l * l * l * l / 5040.0);
    p = fmaf(p, X, (float)(5.0 * l * l * l * l / 720.0));
    p = fmaf(p, X, (float)(4.0 * l * l * l / 120.0));
    p = fmaf(p, X, (float)(3.0 * l * l / 24.0));
    p = fmaf(p, X, (float)(2.0 * l / 6.0));
    return fmaf(p, X, 0.5f);
}

}  // namespace mscan
