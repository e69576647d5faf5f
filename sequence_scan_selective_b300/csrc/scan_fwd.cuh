// Fused selective-scan forward kernel: discretisation + diagonal recurrence + readout + skip + gate.
//
// Follows the hardware-aware design described for Mamba's selective SSM (visual guide to Mamba and
// SSMs, section 3.4; news write-up, "hardware-aware algorithm"): the step-size map, the
// discretisation Abar = exp(Delta A) / Bbar x = Delta B x, the recurrence and the multiplication by C
// run in one kernel; the expanded state h [b, d, N, L] and Abar, Bbar never leave the chip.
//
// B300 mapping (warp-specialised)
//  * A CTA owns CH = 32 channels of one batch row and walks its time range in chunks of TC steps.
//  * One helper warp (lane = channel) moves data and does the per-element work:
//      - issues TMA loads (cp.async.bulk.tensor, 64-byte swizzle) of u, delta, z [CH x TC] and
//        B, C [N x TC] into an NSTAGE-deep ring guarded by mbarriers;
//      - produce: per slot of U = 8 steps, turns (delta, u) into (Delta, Delta, Delta*u, Delta*u)
//        fp32 quads (softplus + bias), B and C into (B_n, B_n+1, C_n, C_n+1) quads per step, and
//        z, u into (D*u, silu(z)) pairs, all in a ring of R slot buffers;
//      - post: sums the scan threads' partial C.h of a slot, applies the skip term and the gate,
//        writes the output tile (same swizzle) and sends each finished chunk to y by TMA store.
//  * Scan warps: each thread holds G states of one channel in registers and advances them
//    sequentially in time with packed fp32x2 arithmetic (MUFU ex2 for Abar); S = NP/G threads
//    share a channel and leave their partial sums per step in the slot.  They never touch global
//    memory in the loop and synchronise with the helper only through the slot mbarriers.
//  * Few channels (long sequences): the time axis is split into segments.  An AGG launch computes
//    each segment's carry (prod Abar = exp(A * sum Delta), h_end from zero); the full launch folds
//    the carries of the preceding segments into its initial state (the scan operator is
//    associative; guide section 3.3).
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "ptx.cuh"

namespace mscan {

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s bound on any wait

__device__ int g_status;  // nonzero: some kernel abandoned a bounded wait

struct FwdArgs {
    const void* u;
    const void* delta;
    const void* z;
    const void* B;
    const void* C;
    const float* A;
    const float* D;
    const float* bias;
    void* y;
    float* last_state;
    float2* agg;  // [nseg-1][batch][dim][dstate] (prod Abar, h_end)
    int batch, dim, dstate;
    long long L;
    long long seg_len;  // multiple of TC
    int nseg;
    int softplus;
    int has_z;
};

// ------------------------------------------------------------------------------ element access
template <typename TIn>
struct In;
template <>
struct In<float> {
    __device__ static __forceinline__ float to_f32(float x) { return x; }
    // 8 consecutive values from two 16-byte chunks
    __device__ static __forceinline__ void unpack8(const uint4& a, const uint4& b, float* v) {
        v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
        v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y); v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
    }
    __device__ static __forceinline__ void pack8(const float* v, uint4& a, uint4& b) {
        a = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
        b = make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]), __float_as_uint(v[6]), __float_as_uint(v[7]));
    }
};
template <>
struct In<uint16_t> {
    __device__ static __forceinline__ float to_f32(uint16_t x) { return bf16_bits_to_f32(x); }
    __device__ static __forceinline__ void unpack8(const uint4& a, const uint4&, float* v) {
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static __forceinline__ void pack8(const float* v, uint4& a, uint4&) {
        a = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                       pack_bf16x2(v[6], v[7]));
    }
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
// softplus(x) = max(x, 0) + log1p(e), e = exp(-|x|) in (0, 1]; log1p(e) = e * P(e) with P the
// degree-8 Chebyshev interpolant of log1p(e)/e on [0, 1] (coefficients from gen_softplus_poly.py;
// fp32 relative error of the log1p term below 3e-7).  NaN propagates through e.
__device__ __forceinline__ float2 softplus2(float2 x) {
    const float2 e = make_float2(ex2_approx(-fabsf(x.x) * kLog2e), ex2_approx(-fabsf(x.y) * kLog2e));
    float2 p = make_float2(0.005126102f, 0.005126102f);
    p = ffma2(p, e, make_float2(-0.029074065f, -0.029074065f));
    p = ffma2(p, e, make_float2(0.07751609f, 0.07751609f));
    p = ffma2(p, e, make_float2(-0.13602248f, -0.13602248f));
    p = ffma2(p, e, make_float2(0.19076881f, 0.19076881f));
    p = ffma2(p, e, make_float2(-0.24835399f, -0.24835399f));
    p = ffma2(p, e, make_float2(0.3331812f, 0.3331812f));
    p = ffma2(p, e, make_float2(-0.49999446f, -0.49999446f));
    p = ffma2(p, e, make_float2(0.99999994f, 0.99999994f));
    return ffma2(e, p, make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)));
}

__device__ __forceinline__ float softplus1(float x) { return softplus2(make_float2(x, x)).x; }

// silu(z) = z * sigmoid(z) = z / (1 + e^-z)
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.f + ex2_approx(-z * kLog2e)); }

// ------------------------------------------------------------------------------ smem geometry
// Tiles of u, delta, z and y are [CH rows][TC cols] with 64-byte rows stored with the TMA 64-byte
// swizzle: the 16-byte chunk index (address bits 4-5) is XORed with address bits 7-8.  Rows are
// read and written whole by one helper lane each, so 8 lanes touching the same logical chunk of 8
// consecutive rows hit 8 different bank groups.
__device__ __forceinline__ uint32_t swz64(uint32_t off) { return off ^ (((off >> 7) & 3u) << 4); }

template <typename TIn, int NP, int G, int CH, int TC, int NS>
struct FwdSmem {
    static constexpr int S = NP / G;
    static constexpr int U = 8;                                  // steps per slot
    static constexpr int R = 2;                                  // slots in the ring
    static constexpr int kRow = TC * (int)sizeof(TIn);           // bytes per tile row (64)
    static constexpr int kTile = CH * kRow;                      // one u/delta/z tile
    static constexpr int kBC = NP * kRow;                        // one B or C tile (N <= NP rows)
    static constexpr int kStage = (3 * kTile + 2 * kBC + 1023) / 1024 * 1024;
    static constexpr int kQPitch = U * 16 + 16;                  // (Dt,Dt,Du,Du) quads per channel
    static constexpr int kBCPitch = NP * 8 + 16;                 // (B,B,C,C) quads per step
    static constexpr int kYPitch = U * 4 + 16;                   // partial sums per scan thread
    static constexpr int kZPitch = U * 8 + 16;                   // (D u, silu z) per channel
    static constexpr int kSlotQ = CH * kQPitch;
    static constexpr int kSlotBC = U * kBCPitch;
    static constexpr int kSlotY = CH * S * kYPitch;
    static constexpr int kSlotZ = CH * kZPitch;
    static constexpr int kSlot = kSlotQ + kSlotBC + kSlotY + kSlotZ;
    static constexpr int kOffSlots = NS * kStage;
    static constexpr int kOffOut = (kOffSlots + R * kSlot + 1023) / 1024 * 1024;  // 2 output tiles
    static constexpr int kOffBar = kOffOut + 2 * kTile;
    static constexpr int kBars = NS + 2 * R;
    static constexpr int kBytes = kOffBar + kBars * 8;
    static_assert(kRow == 64, "tile rows must be 64 bytes (64-byte TMA swizzle)");
    static_assert(kSlot % 16 == 0 && kTile % 1024 == 0, "alignment");
};

template <typename TIn, int NP, int G, int CH, int TC, int NSTAGE, bool TMA, bool AGG>
__global__ void __launch_bounds__(CH*(NP / G) + 32, 1)
    scan_fwd_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap tm_u,
                    const __grid_constant__ CUtensorMap tm_d, const __grid_constant__ CUtensorMap tm_z,
                    const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_C,
                    const __grid_constant__ CUtensorMap tm_y) {
    using SM = FwdSmem<TIn, NP, G, CH, TC, NSTAGE>;
    constexpr int S = SM::S;         // scan threads per channel
    constexpr int NSCAN = CH * S;    // scan threads (warps 0 .. NSCAN/32-1); the last warp helps
    constexpr int U = SM::U;
    constexpr int R = SM::R;
    constexpr int NS = NSTAGE;
    constexpr int SPC = TC / U;      // slots per chunk
    constexpr int VPR = U * (int)sizeof(TIn) / 16;  // 16-byte chunks per slot row (1 bf16, 2 fp32)
    static_assert(CH == 32, "one helper warp: lane = channel");
    static_assert(G % 2 == 0 && 32 % S == 0 && NSCAN % 32 == 0 && TC % U == 0 && NS >= 2, "shape");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // swizzled TMA tiles need 1024-byte alignment; the launch reserves 1 KB of slack for this
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* tma_full = reinterpret_cast<uint64_t*>(smem + SM::kOffBar);
    uint64_t* full = tma_full + NS;
    uint64_t* done = full + R;

    const int tid = threadIdx.x;
    const int d0 = blockIdx.x * CH;
    const int b = blockIdx.y;
    const int seg = blockIdx.z;
    const int N = a.dstate;
    const long long t_begin = (long long)seg * a.seg_len;
    const long long t_end = min(a.L, t_begin + a.seg_len);
    const int nchunks = (int)((t_end - t_begin + TC - 1) / TC);
    const int nslots = (int)((t_end - t_begin + U - 1) / U);
    const bool has_z = !AGG && a.has_z;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&tma_full[s], 1);
        for (int r = 0; r < R; ++r) {
            mbar_init(&full[r], 32);
            mbar_init(&done[r], NSCAN);
        }
        mbar_fence_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    if (tid >= NSCAN) {
        // =============================================================== helper warp (lane = channel)
        const int lane = tid - NSCAN;
        const int dch = d0 + lane;
        const bool cvalid = dch < a.dim;
        const float bias = (a.bias != nullptr && cvalid) ? a.bias[dch] : 0.f;
        const float Dd = (!AGG && a.D != nullptr && cvalid) ? a.D[dch] : 0.f;
        const uint32_t tile_bytes = (uint32_t)SM::kTile;
        const uint32_t bc_bytes = (uint32_t)(N * SM::kRow);
        const uint32_t stage_tx = (AGG ? 2u : (has_z ? 3u : 2u)) * tile_bytes + (AGG ? 1u : 2u) * bc_bytes;

        auto issue_loads = [&](int k) {  // chunk k -> stage k % NS (lane 0 only)
            unsigned char* st = smem + (k % NS) * SM::kStage;
            const int t0 = (int)(t_begin + (long long)k * TC);
            uint64_t* bar = &tma_full[k % NS];
            mbar_arrive_expect_tx(bar, stage_tx);
            tma_load_3d(st, &tm_u, bar, t0, d0, b);
            tma_load_3d(st + SM::kTile, &tm_d, bar, t0, d0, b);
            if (has_z) tma_load_3d(st + 2 * SM::kTile, &tm_z, bar, t0, d0, b);
            tma_load_3d(st + 3 * SM::kTile, &tm_B, bar, t0, 0, b);
            if (!AGG) tma_load_3d(st + 3 * SM::kTile + SM::kBC, &tm_C, bar, t0, 0, b);
        };
        // plain-load fallback (unaligned shapes): same swizzled layout, one row per lane
        auto plain_load = [&](int k) {
            unsigned char* st = smem + (k % NS) * SM::kStage;
            const long long t0 = t_begin + (long long)k * TC;
            const int tv = (int)min((long long)TC, t_end - t0);
            const TIn* src[3] = {static_cast<const TIn*>(a.u), static_cast<const TIn*>(a.delta),
                                 static_cast<const TIn*>(a.z)};
            for (int m = 0; m < (has_z ? 3 : 2); ++m) {
                unsigned char* tile = st + m * SM::kTile;
                for (int t = 0; t < TC; ++t) {
                    TIn v = TIn(0);
                    if (cvalid && t < tv) v = src[m][((long long)b * a.dim + dch) * a.L + t0 + t];
                    *reinterpret_cast<TIn*>(tile + swz64(lane * SM::kRow + t * (int)sizeof(TIn))) = v;
                }
            }
            for (int m = 0; m < (AGG ? 1 : 2); ++m) {
                const TIn* gsrc = static_cast<const TIn*>(m == 0 ? a.B : a.C);
                TIn* tile = reinterpret_cast<TIn*>(st + 3 * SM::kTile + m * SM::kBC);
                for (int j = lane; j < N * TC; j += 32) {
                    const int n = j / TC, t = j % TC;
                    tile[j] = t < tv ? gsrc[((long long)b * N + n) * a.L + t0 + t] : TIn(0);
                }
            }
            __syncwarp();
        };

        if (TMA && lane == 0)
            for (int k = 0; k < NS && k < nchunks; ++k) issue_loads(k);

        bool ok = true;
        // post: finish slot i (its partial sums are complete) -> output tile
        auto post = [&](int i) {
            const int r = i % R;
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(&done[r], (uint32_t)((i / R) & 1), kWaitLimitNs));
            if (!ok) return;
            const int k = i / SPC, j = i % SPC;
            unsigned char* slot = smem + SM::kOffSlots + r * SM::kSlot;
            const unsigned char* yp = slot + SM::kSlotQ + SM::kSlotBC;
            const float2* zz = reinterpret_cast<const float2*>(slot + SM::kSlotQ + SM::kSlotBC + SM::kSlotY + lane * SM::kZPitch);
            float y[U];
#pragma unroll
            for (int q = 0; q < U; q += 4) {
                float4 acc = *reinterpret_cast<const float4*>(yp + (lane * S) * SM::kYPitch + q * 4);
#pragma unroll
                for (int gg = 1; gg < S; ++gg) {
                    const float4 v = *reinterpret_cast<const float4*>(yp + (lane * S + gg) * SM::kYPitch + q * 4);
                    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
                }
                const float4 z01 = *reinterpret_cast<const float4*>(zz + q);
                const float4 z23 = *reinterpret_cast<const float4*>(zz + q + 2);
                y[q] = (acc.x + z01.x) * z01.y;
                y[q + 1] = (acc.y + z01.z) * z01.w;
                y[q + 2] = (acc.z + z23.x) * z23.y;
                y[q + 3] = (acc.w + z23.z) * z23.w;
            }
            unsigned char* out = smem + SM::kOffOut + (k & 1) * SM::kTile;
            uint4 c0, c1;
            In<TIn>::pack8(y, c0, c1);
            const uint32_t off = lane * SM::kRow + j * U * (int)sizeof(TIn);
            *reinterpret_cast<uint4*>(out + swz64(off)) = c0;
            if (VPR == 2) *reinterpret_cast<uint4*>(out + swz64(off + 16)) = c1;
            if (j == SPC - 1 || i == nslots - 1) {
                const long long t0 = t_begin + (long long)k * TC;
                if (TMA) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&tm_y, out, (int)t0, d0, b);
                        bulk_commit();
                        bulk_wait_read<1>();  // the other output tile may be overwritten next
                    }
                    __syncwarp();
                } else {
                    const int tv = (int)min((long long)TC, t_end - t0);
                    TIn* gy = static_cast<TIn*>(a.y);
                    if (cvalid)
                        for (int t = 0; t < tv; ++t)
                            gy[((long long)b * a.dim + dch) * a.L + t0 + t] =
                                *reinterpret_cast<const TIn*>(out + swz64(lane * SM::kRow + t * (int)sizeof(TIn)));
                }
            }
        };
        // produce: slot i's operands from the staged tiles
        auto produce = [&](int i) {
            const int r = i % R;
            const int k = i / SPC, j = i % SPC;
            if (j == 0) {
                if (TMA) {
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(&tma_full[k % NS], (uint32_t)((k / NS) & 1), kWaitLimitNs));
                    if (!ok) return;
                } else {
                    plain_load(k);
                }
            }
            const unsigned char* st = smem + (k % NS) * SM::kStage;
            unsigned char* slot = smem + SM::kOffSlots + r * SM::kSlot;
            const long long t0 = t_begin + (long long)k * TC + j * U;
            const int tv = (int)min((long long)U, t_end - t0);
            const uint32_t off = lane * SM::kRow + j * U * (int)sizeof(TIn);
            float uv[U], dv[U];
            {
                const uint4 u0 = *reinterpret_cast<const uint4*>(st + swz64(off));
                const uint4 u1 = VPR == 2 ? *reinterpret_cast<const uint4*>(st + swz64(off + 16)) : u0;
                const uint4 e0 = *reinterpret_cast<const uint4*>(st + SM::kTile + swz64(off));
                const uint4 e1 = VPR == 2 ? *reinterpret_cast<const uint4*>(st + SM::kTile + swz64(off + 16)) : e0;
                In<TIn>::unpack8(u0, u1, uv);
                In<TIn>::unpack8(e0, e1, dv);
            }
            float4* q = reinterpret_cast<float4*>(slot + lane * SM::kQPitch);
#pragma unroll
            for (int t = 0; t < U; t += 2) {
                float2 dt = make_float2(dv[t] + bias, dv[t + 1] + bias);
                if (a.softplus) dt = softplus2(dt);
                if (t >= tv) dt.x = 0.f;
                if (t + 1 >= tv) dt.y = 0.f;
                const float2 du = fmul2(dt, make_float2(uv[t], uv[t + 1]));
                q[t] = make_float4(dt.x, dt.x, du.x, du.x);
                q[t + 1] = make_float4(dt.y, dt.y, du.y, du.y);
            }
            if (!AGG) {
                float zv[U];
                if (has_z) {
                    const uint4 z0 = *reinterpret_cast<const uint4*>(st + 2 * SM::kTile + swz64(off));
                    const uint4 z1 = VPR == 2 ? *reinterpret_cast<const uint4*>(st + 2 * SM::kTile + swz64(off + 16)) : z0;
                    In<TIn>::unpack8(z0, z1, zv);
                }
                float4* zz = reinterpret_cast<float4*>(slot + SM::kSlotQ + SM::kSlotBC + SM::kSlotY + lane * SM::kZPitch);
#pragma unroll
                for (int t = 0; t < U; t += 2) {
                    const float g0 = has_z ? silu_f(zv[t]) : 1.f;
                    const float g1 = has_z ? silu_f(zv[t + 1]) : 1.f;
                    zz[t / 2] = make_float4(Dd * uv[t], g0, Dd * uv[t + 1], g1);
                }
            }
            // B, C of the slot's steps as fp32 quads; states >= N are zero
            const TIn* tB = reinterpret_cast<const TIn*>(st + 3 * SM::kTile);
            const TIn* tC = reinterpret_cast<const TIn*>(st + 3 * SM::kTile + SM::kBC);
            unsigned char* bcq = slot + SM::kSlotQ;
#pragma unroll
            for (int e = lane; e < U * (NP / 2); e += 32) {
                const int t = e % U, p = e / U;
                const int n0 = 2 * p, n1 = n0 + 1, tt = j * U + t;
                float4 w;
                w.x = n0 < N ? In<TIn>::to_f32(tB[n0 * TC + tt]) : 0.f;
                w.y = n1 < N ? In<TIn>::to_f32(tB[n1 * TC + tt]) : 0.f;
                w.z = (!AGG && n0 < N) ? In<TIn>::to_f32(tC[n0 * TC + tt]) : 0.f;
                w.w = (!AGG && n1 < N) ? In<TIn>::to_f32(tC[n1 * TC + tt]) : 0.f;
                *reinterpret_cast<float4*>(bcq + t * SM::kBCPitch + p * 16) = w;
            }
            mbar_arrive(&full[r]);
            if (j == SPC - 1) {
                // every lane has read stage k: refill it with chunk k + NS
                __syncwarp();
                if (TMA && lane == 0 && k + NS < nchunks) issue_loads(k + NS);
            }
        };

        for (int i = 0; i < nslots + R && ok; ++i) {
            if (i >= R) {
                if (AGG) {  // slot free once the scan threads are done with it
                    const int r = (i - R) % R;
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(&done[r], (uint32_t)(((i - R) / R) & 1), kWaitLimitNs));
                } else {
                    post(i - R);
                }
                if (!ok) break;
            }
            if (i < nslots) produce(i);
        }
        if (TMA && !AGG && lane == 0) bulk_wait_all<0>();
        if (!ok && lane == 0) atomicExch(&g_status, 1);
        return;
    }

    // =================================================================== scan threads
    const int c = tid / S;
    const int g = tid % S;
    const int dch = d0 + c;
    const bool cvalid = dch < a.dim;
    float2 A2[G / 2];
    float2 h[G / 2];
#pragma unroll
    for (int p = 0; p < G / 2; ++p) {
        const int n0 = g * G + 2 * p, n1 = n0 + 1;
        A2[p].x = (cvalid && n0 < N) ? a.A[(long long)dch * N + n0] * kLog2e : 0.f;
        A2[p].y = (cvalid && n1 < N) ? a.A[(long long)dch * N + n1] * kLog2e : 0.f;
        h[p] = make_float2(0.f, 0.f);
    }
    if (seg > 0 && cvalid) {
        // fold the carries of segments 0..seg-1 in order: h <- prodAbar * h + h_end
        for (int q = 0; q < seg; ++q) {
            const float2* ag = a.agg + (((long long)q * a.batch + b) * a.dim + dch) * N;
#pragma unroll
            for (int p = 0; p < G / 2; ++p) {
                const int n0 = g * G + 2 * p, n1 = n0 + 1;
                if (n0 < N) { const float2 v = ag[n0]; h[p].x = fmaf(v.x, h[p].x, v.y); }
                if (n1 < N) { const float2 v = ag[n1]; h[p].y = fmaf(v.x, h[p].y, v.y); }
            }
        }
    }
    float sumdt = 0.f;
    bool ok = true;
    for (int i = 0; i < nslots; ++i) {
        const int r = i % R;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[r], (uint32_t)((i / R) & 1), kWaitLimitNs));
        if (!ok) break;
        unsigned char* slot = smem + SM::kOffSlots + r * SM::kSlot;
        const float4* qrow = reinterpret_cast<const float4*>(slot + c * SM::kQPitch);
        const float4* bcg = reinterpret_cast<const float4*>(slot + SM::kSlotQ) + g * (G / 2);
        constexpr int kBCQ = SM::kBCPitch / 16;
        float yp[U];
#pragma unroll
        for (int t = 0; t < U; ++t) {
            const float4 q = qrow[t];  // (Delta, Delta, Delta*u, Delta*u)
            float2 y0 = make_float2(0.f, 0.f), y1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int p = 0; p < G / 2; ++p) {
                const float4 w = bcg[t * kBCQ + p];
                const float2 x = fmul2(make_float2(q.x, q.y), A2[p]);
                const float2 abar = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                const float2 bx = fmul2(make_float2(q.z, q.w), make_float2(w.x, w.y));
                h[p] = ffma2(abar, h[p], bx);
                if (!AGG) {
                    if (p & 1) y1 = ffma2(make_float2(w.z, w.w), h[p], y1);
                    else       y0 = ffma2(make_float2(w.z, w.w), h[p], y0);
                }
            }
            if (AGG) sumdt += q.x;
            const float2 ys = fadd2(y0, y1);
            yp[t] = ys.x + ys.y;
        }
        if (!AGG) {
            float4* yd = reinterpret_cast<float4*>(slot + SM::kSlotQ + SM::kSlotBC + tid * SM::kYPitch);
            yd[0] = make_float4(yp[0], yp[1], yp[2], yp[3]);
            yd[1] = make_float4(yp[4], yp[5], yp[6], yp[7]);
        }
        mbar_arrive(&done[r]);
    }
    if (!ok) {
        if (tid == 0) atomicExch(&g_status, 1);
        return;
    }
    if (AGG) {
        if (cvalid) {
            float2* ag = a.agg + (((long long)seg * a.batch + b) * a.dim + dch) * N;
#pragma unroll
            for (int p = 0; p < G / 2; ++p) {
                const int n0 = g * G + 2 * p, n1 = n0 + 1;
                if (n0 < N) ag[n0] = make_float2(ex2_approx(A2[p].x * sumdt), h[p].x);
                if (n1 < N) ag[n1] = make_float2(ex2_approx(A2[p].y * sumdt), h[p].y);
            }
        }
    } else if (a.last_state != nullptr && cvalid && seg == a.nseg - 1) {
        float* ls = a.last_state + ((long long)b * a.dim + dch) * N;
#pragma unroll
        for (int p = 0; p < G / 2; ++p) {
            const int n0 = g * G + 2 * p, n1 = n0 + 1;
            if (n0 < N) ls[n0] = h[p].x;
            if (n1 < N) ls[n1] = h[p].y;
        }
    }
}

}  // namespace mscan
