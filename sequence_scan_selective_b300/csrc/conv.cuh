// Causal depthwise convolution in front of the scan, as separate kernels for the backward pass of
// the fused block (the forward pass fuses it into the scan kernels).
//
// The Mamba block convolves the expanded input over time before the selective SSM (visual guide
// to Mamba and SSMs, section 3.5):
//   pre[t] = conv_bias[d] + sum_{k<K} w[d, k] x[t-(K-1)+k],   u[t] = silu(pre[t]) (or pre[t]),
// with x before position 0 taken from conv_prev [b, d, K-1] (oldest first) or zero.
//  * conv_fwd_kernel materialises u for the backward pass's recomputation, with the same
//    arithmetic, in the same order, as the fused forward kernels (taps right-aligned in a 4-tap
//    window, fmaf from the oldest input, silu as z * sigmoid(z)), so fp32 u matches theirs bit for
//    bit.
//  * conv_bwd_kernel takes du (the gradient reaching u) back through the convolution:
//      dpre[t] = du[t] silu'(pre[t]),  silu'(p) = s(p) (1 + p (1 - s(p))), s the logistic,
//      dx[j]   = sum_k w[k] dpre[j + (K-1) - k],
//      dw[k]  += sum_t dpre[t] x[t-(K-1)+k],   dbias += sum_t dpre[t],
//    and the gradient of the K-1 inputs before position 0 (dconv_prev).
// A CTA owns kConvTile positions of one (batch row, channel): it stages that tile of x (with the
// 3 inputs before it and, backward, 3 after) and of du once in shared memory with coalesced
// loads, and every tap reads from there; the sums over positions go to the per-channel gradients
// with one atomic per tap per CTA.
#pragma once
#include <stdint.h>

#include "common.cuh"

namespace mscan {

struct ConvArgs {
    const void* x;          // [b, d, L] TIn
    const float* w;         // [d, K]
    const float* bias;      // [d] or null
    const float* prev;      // [b, d, K-1] or null (zeros)
    void* u;                // forward: [b, d, L] TIn, written
    const void* du;         // backward: [b, d, L] TIn
    void* dx;               // backward: [b, d, L] TIn, written
    float* dw;              // backward: [d, K], accumulated (zeroed by the host) or null
    float* dbias;           // backward: [d], accumulated (zeroed by the host) or null
    float* dprev;           // backward: [b, d, K-1], written, or null
    int batch, dim, K, silu;
    long long L;
    long long ntile;        // position tiles per row: the grid is rows x ntile CTAs
};

constexpr int kConvThreads = 256;
constexpr int kConvTile = 1024;  // positions per CTA

// Input position p of row `row` (p < 0: the inputs before the sequence).
template <typename TIn>
__device__ __forceinline__ float conv_x(const ConvArgs& a, long long row, long long p) {
    if (p >= 0) return In<TIn>::to_f32(static_cast<const TIn*>(a.x)[row * a.L + p]);
    if (a.prev != nullptr && p >= -(a.K - 1)) return a.prev[row * (a.K - 1) + (a.K - 1) + p];
    return 0.f;
}

// dst[i] = x at position t0 - 3 + i for i < n (0 past L): every load of the thread is issued
// before the first store, so that each thread keeps several loads in flight.
template <typename TIn, int MAXN>
__device__ __forceinline__ void stage_x(float* dst, const ConvArgs& a, long long row, long long t0, int n) {
    constexpr int PER = (MAXN + kConvThreads - 1) / kConvThreads;
    float v[PER];
#pragma unroll
    for (int r = 0; r < PER; ++r) {
        const int i = (int)threadIdx.x + r * kConvThreads;
        const long long p = t0 - 3 + i;
        v[r] = (i < n && p < a.L) ? conv_x<TIn>(a, row, p) : 0.f;
    }
#pragma unroll
    for (int r = 0; r < PER; ++r) {
        const int i = (int)threadIdx.x + r * kConvThreads;
        if (i < n) dst[i] = v[r];
    }
}

template <typename TIn>
__global__ void __launch_bounds__(kConvThreads) conv_fwd_kernel(const ConvArgs a) {
    __shared__ float xs[kConvTile + 3];  // x at t0 - 3 .. t0 + kConvTile - 1
    const long long row = (long long)blockIdx.x / a.ntile;  // b * dim + d
    const long long tile = (long long)blockIdx.x % a.ntile;
    const int d = (int)(row % a.dim);
    float w4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (q >= 4 - a.K) w4[q] = a.w[(long long)d * a.K + q - (4 - a.K)];
    const float cb = a.bias != nullptr ? a.bias[d] : 0.f;
    const long long t0 = tile * kConvTile;
    stage_x<TIn, kConvTile + 3>(xs, a, row, t0, kConvTile + 3);
    __syncthreads();
    for (int i = threadIdx.x; i < kConvTile; i += kConvThreads) {
        const long long t = t0 + i;
        if (t >= a.L) break;
        // pre[t]: the taps right-aligned in a 4-tap window, summed from the oldest input (the
        // order of the fused forward kernels); xs[i + q] is x[t - 3 + q]
        float p = cb;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (q >= 4 - a.K) p = fmaf(w4[q], xs[i + q], p);
        store_out<TIn>(static_cast<TIn*>(a.u) + row * a.L + t, a.silu ? p * sigmoid_approx(p) : p);
    }
}

template <typename TIn>
__global__ void __launch_bounds__(kConvThreads) conv_bwd_kernel(const ConvArgs a) {
    __shared__ float xs[kConvTile + 6];      // x at t0 - 3 .. t0 + kConvTile + 2
    __shared__ float dpre_s[kConvTile + 3];  // dpre at t0 .. t0 + kConvTile + 2
    __shared__ float red[kConvThreads / 32][5];
    const long long row = (long long)blockIdx.x / a.ntile;
    const long long tile = (long long)blockIdx.x % a.ntile;
    const int d = (int)(row % a.dim);
    const int K = a.K;
    float w4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (q >= 4 - K) w4[q] = a.w[(long long)d * K + q - (4 - K)];
    const float cb = a.bias != nullptr ? a.bias[d] : 0.f;
    const long long t0 = tile * kConvTile;
    const TIn* du = static_cast<const TIn*>(a.du) + row * a.L;
    {
        constexpr int PER = (kConvTile + 3 + kConvThreads - 1) / kConvThreads;
        float g[PER];
#pragma unroll
        for (int r = 0; r < PER; ++r) {  // du loads issued first, then the x tile's
            const int i = (int)threadIdx.x + r * kConvThreads;
            g[r] = (i < kConvTile + 3 && t0 + i < a.L) ? In<TIn>::to_f32(du[t0 + i]) : 0.f;
        }
        stage_x<TIn, kConvTile + 6>(xs, a, row, t0, kConvTile + 6);
#pragma unroll
        for (int r = 0; r < PER; ++r) {
            const int i = (int)threadIdx.x + r * kConvThreads;
            if (i < kConvTile + 3) dpre_s[i] = g[r];
        }
    }
    __syncthreads();
    // dpre over the tile and the K-1 positions after it (they reach the tile's last inputs)
    for (int i = threadIdx.x; i < kConvTile + 3; i += kConvThreads) {
        if (!a.silu || t0 + i >= a.L) continue;  // identity activation: dpre = du (zero past L)
        float p = cb;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (q >= 4 - K) p = fmaf(w4[q], xs[i + q], p);
        const float sg = sigmoid_approx(p);
        dpre_s[i] = dpre_s[i] * sg * fmaf(p, 1.f - sg, 1.f);
    }
    __syncthreads();

    // dx of the tile's inputs, and this thread's share of the tap and bias sums
    float sw[4] = {0.f, 0.f, 0.f, 0.f}, sb = 0.f;
    for (int i = threadIdx.x; i < kConvTile; i += kConvThreads) {
        const long long j = t0 + i;
        if (j >= a.L) break;
        // input j feeds outputs j + (K-1) - k through tap k: w4[q] with q = k + 4 - K
        float g = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (q >= 4 - K) g = fmaf(w4[q], dpre_s[i + 3 - q], g);
        store_out<TIn>(static_cast<TIn*>(a.dx) + row * a.L + j, g);
        const float gp = dpre_s[i];  // dpre at t = j
        sb += gp;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (q >= 4 - K) sw[q] = fmaf(gp, xs[i + q], sw[q]);  // x[j - 3 + q]
    }
    // inputs before position 0: the first tile's CTA
    if (tile == 0 && a.dprev != nullptr && threadIdx.x < K - 1) {
        const int pidx = threadIdx.x;         // 0 .. K-2, position pidx - (K-1)
        const long long j = pidx - (K - 1);
        float g = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const long long t = j + 3 - q;     // output reached through tap q
            if (q >= 4 - K && t >= 0 && t < a.L) g = fmaf(w4[q], dpre_s[t], g);
        }
        a.dprev[row * (K - 1) + pidx] = g;
    }
    // CTA sums of the 4 tap slots and the bias, then one atomic each
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    float v[5] = {sw[0], sw[1], sw[2], sw[3], sb};
#pragma unroll
    for (int m = 16; m >= 1; m /= 2)
#pragma unroll
        for (int i = 0; i < 5; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], m);
    if (lane == 0)
#pragma unroll
        for (int i = 0; i < 5; ++i) red[wid][i] = v[i];
    __syncthreads();
    if (threadIdx.x < 5) {
        float s = 0.f;
        for (int w = 0; w < kConvThreads / 32; ++w) s += red[w][threadIdx.x];
        const int q = threadIdx.x;
        if (q < 4) {
            if (q >= 4 - K && a.dw != nullptr) atomicAdd(a.dw + (long long)d * K + q - (4 - K), s);
        } else if (a.dbias != nullptr) {
            atomicAdd(a.dbias + d, s);
        }
    }
}

}  // namespace mscan
