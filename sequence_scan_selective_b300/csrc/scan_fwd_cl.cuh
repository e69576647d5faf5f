// Fused selective-scan forward kernel with one channel per lane: step-size map + discretisation +
// diagonal recurrence + readout + skip + gate, all NP <= 16 states of a channel in the registers
// of one thread.
//
// Same method as scan_fwd_kernel (visual guide to Mamba and SSMs, section 3.4: Abar = exp(Delta A)
// and Bbar x = Delta B x are formed on chip, h_t = Abar_t h_{t-1} + Bbar_t x_t runs there, only
// y = (C h + D x) silu(z) and the final state leave the SM), with a lane layout chosen for the
// B300 SM's pipes:
//  * Lane = channel.  A lane owns every state of its channel, so the per-element work (softplus
//    step size, Delta x, D x, silu gate) is done once, by the lane that needs it, and the readout
//    C.h is summed in registers: no exchange between lanes at all.
//  * B and C are the same for every channel of a batch row, so all 32 lanes of a warp read the
//    same (B_n, B_n+1, C_n, C_n+1) quad at each step: a broadcast 16-byte shared-memory load,
//    which the SM serves at about one per clock.  The producer warp builds the quads once per
//    chunk for all consumer warps (converting bf16 to fp32 on the way).
//  * Per state pair and step: one packed f32x2 multiply for Delta A log2(e), two MUFU ex2, one
//    f32x2 multiply for (Delta x) B, one f32x2 FMA for h, one f32x2 FMA for C.h.  The packed
//    forms keep the FP32 pipe and the MUFU pipe busy together.
//  * u, delta, z arrive by TMA as [32 * warps, TC] tiles (128-byte swizzle); y leaves by TMA
//    store from a per-warp staging tile in the same layout.
//  * Few channels (long sequences): the time axis is split into segments that all run at once
//    (LOCAL): segment 0 from the initial state, every later one from zero.  Each writes its
//    outputs and its carry (prod Abar, h_end); scan_fix_kernel then adds to each later segment's
//    outputs the part of the state carried in from before it, which decays from the segment's
//    start on (the scan operator is associative and the recurrence linear in h: guide section
//    3.3).
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "scan_fwd.cuh"

namespace mscan {
namespace cl {

constexpr int kRowBytes = 128;     // bytes per tile row (one chunk of one channel)

// A work unit is 32 channels of one batch row, one per lane of a consumer warp; a CTA holds up
// to 4 consumer warps, one per SM sub-partition.
struct Lanes {
    static constexpr int CPW = 32;                       // channels per warp (work unit)
    static constexpr int MAX_WARPS = 4;                  // consumer warps per CTA
    static constexpr int YTILE = CPW * kRowBytes;        // one warp's y staging tile
};

template <int NP>
struct Quads {
    static constexpr int PAIRS = NP / 2;
    static constexpr int PITCH = PAIRS * 16 + 16;  // bytes per step (padded: conflict-free stores)
};

// BLK consecutive elements at byte `byte` of row `row` of a 128-byte-swizzled tile -> fp32
// (BLK = 4 for fp32, 8 for bf16: one 16-byte read)
template <typename TIn>
__device__ __forceinline__ void tile_load16(const unsigned char* tile, int row, int byte, float* v);
template <>
__device__ __forceinline__ void tile_load16<float>(const unsigned char* tile, int row, int byte, float* v) {
    const float4 q = *reinterpret_cast<const float4*>(tile + swz128(row, byte));
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
template <>
__device__ __forceinline__ void tile_load16<uint16_t>(const unsigned char* tile, int row, int byte, float* v) {
    const uint4 q = *reinterpret_cast<const uint4*>(tile + swz128(row, byte));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// BLK outputs -> 16 bytes at byte `byte` of row `row` of a 128-byte-swizzled tile
template <typename TIn>
__device__ __forceinline__ void tile_store16(unsigned char* tile, int row, int byte, const float* v);
template <>
__device__ __forceinline__ void tile_store16<float>(unsigned char* tile, int row, int byte, const float* v) {
    *reinterpret_cast<float4*>(tile + swz128(row, byte)) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void tile_store16<uint16_t>(unsigned char* tile, int row, int byte, const float* v) {
    *reinterpret_cast<uint4*>(tile + swz128(row, byte)) =
        make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

}  // namespace cl

// Shared memory (offsets in FwdArgs): NS stages of [u | delta | z tiles (wmax * 32 rows of 128 B
// each) | B, C tiles (NP rows of 128 B) | quads (TC steps x PITCH)], then the y staging tiles
// (2 per consumer warp), then 3 NS + 1 mbarriers.
//
// MODE bit 0: exact zero-order hold, Bbar x = k B x with k = (exp(Delta A) - 1) / A (guide
// section 2.3; k evaluated as in scan_fwd_kernel's phase_b_zoh).  MODE bit 1: causal depthwise
// convolution in front of the scan (guide section 3.5): the u tile then holds the block input x,
// and the lane forms u[t] = act(conv_bias + sum_k conv_w[k] x[t-K+1+k]) itself, keeping the last
// three inputs of its channel in registers from block to block.
template <typename TIn, int NP, bool TMA, bool LOCAL, int MODE>
__global__ void __launch_bounds__(32 * (cl::Lanes::MAX_WARPS + 1), 1)
    scan_fwd_cl_kernel(const FwdArgs a, const __grid_constant__ FwdMaps maps) {
    constexpr int TC = Chunk<TIn>::TC;
    constexpr int ES = (int)sizeof(TIn);
    constexpr int BLK = 16 / ES;  // steps per 16-byte tile read
    constexpr int NPAIR = NP / 2;
    constexpr int QPITCH = cl::Quads<NP>::PITCH;
    constexpr int CPW = cl::Lanes::CPW;
    constexpr int PL = NPAIR;                  // state pairs per lane
    constexpr int TILE = CPW * cl::kRowBytes;  // one warp's rows of one input tile
    constexpr bool ZOH = (MODE & 1) != 0;
    constexpr bool CONV = (MODE & 2) != 0;
    constexpr bool CKPT = (MODE & 4) != 0;  // forward pass of training: state checkpoints
    static_assert(!CKPT || (!LOCAL && !CONV), "checkpoints: unsplit time axis, no fused convolution");
    const bool has_z = a.z != nullptr;
    const bool softplus = a.softplus != 0;
    static_assert(NP % 2 == 0 && NP <= 16, "shape");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int NS = a.nstage;
    const int W = a.wmax;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.bar_off);
    uint64_t* qready = full + NS;
    uint64_t* empty = qready + NS;
    uint64_t* never = empty + NS;  // nothing ever arrives here (test knob)

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int kc = a.kcta;
    const int rrow = blockIdx.x / kc, ci = blockIdx.x % kc;
    const int seg = rrow / a.batch;
    const int b = rrow % a.batch;
    const int u0 = (int)((long long)ci * a.upr / kc);
    const int u1 = (int)((long long)(ci + 1) * a.upr / kc);
    const int nunits = u1 - u0;
    const int N = a.dstate;
    const long long t_begin = (long long)seg * a.seg_len;
    const long long t_end = min(a.L, t_begin + a.seg_len);
    const int nchunks = (int)((t_end - t_begin + TC - 1) / TC);

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&qready[s], 32);
            mbar_init(&empty[s], 32 * nunits);
        }
        mbar_init(never, 1);
        mbar_fence_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    if (wid == W) {
        // ================================================================== producer warp
        const int mi = nunits == a.wlo ? 0 : 1;
        const uint32_t tx = (uint32_t)(nunits * TILE * (has_z ? 3 : 2) + 2 * N * cl::kRowBytes);
        auto issue = [&](int k) {  // lane 0: TMA loads of chunk k into stage k % NS
            const int s = k % NS;
            unsigned char* st = smem + s * a.stage_bytes;
            const int t0 = (int)(t_begin + (long long)k * TC);
            mbar_arrive_expect_tx(&full[s], tx);
            const int r0 = u0 * CPW;
            tma_load_3d(st, &maps.u[mi], &full[s], t0, r0, b);
            tma_load_3d(st + W * TILE, &maps.d[mi], &full[s], t0, r0, b);
            if (has_z) tma_load_3d(st + 2 * W * TILE, &maps.z[mi], &full[s], t0, r0, b);
            tma_load_3d(st + a.bc_off, &maps.B, &full[s], t0, 0, b);
            tma_load_3d(st + a.bc_off + NP * cl::kRowBytes, &maps.C, &full[s], t0, 0, b);
        };
        // chunk k's B, C as (B_n, B_n+1, C_n, C_n+1) quads per step; lane handles steps lane + 32 i
        auto build_quads = [&](int k) {
            unsigned char* st = smem + (k % NS) * a.stage_bytes;
            const unsigned char* tB = st + a.bc_off;
            const unsigned char* tC = tB + NP * cl::kRowBytes;
#pragma unroll
            for (int i = 0; i < TC / 32; ++i) {
                const int t = lane + 32 * i;
                float bv[NP], cv[NP];
#pragma unroll
                for (int n = 0; n < NP; ++n) {
                    bv[n] = 0.f;
                    cv[n] = 0.f;
                    if (n < N) {
                        if (TMA) {
                            if constexpr (ES == 4) {
                                bv[n] = *reinterpret_cast<const float*>(tB + swz128(n, t * 4));
                                cv[n] = *reinterpret_cast<const float*>(tC + swz128(n, t * 4));
                            } else {
                                bv[n] = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(tB + swz128(n, t * 2)));
                                cv[n] = bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(tC + swz128(n, t * 2)));
                            }
                        } else {
                            const long long tg = t_begin + (long long)k * TC + t;
                            if (tg < t_end) {
                                const long long off = ((long long)b * N + n) * a.L + tg;
                                bv[n] = In<TIn>::to_f32(static_cast<const TIn*>(a.B)[off]);
                                cv[n] = In<TIn>::to_f32(static_cast<const TIn*>(a.C)[off]);
                            }
                        }
                    }
                }
                float4* qd = reinterpret_cast<float4*>(st + a.quad_off + t * QPITCH);
#pragma unroll
                for (int p = 0; p < NPAIR; ++p) qd[p] = make_float4(bv[2 * p], bv[2 * p + 1], cv[2 * p], cv[2 * p + 1]);
            }
        };

        bool ok = true;
        int issued = 0, landed = 0;  // chunks whose loads were issued / observed complete
        if (TMA) {
            issued = min(NS, nchunks);
            if (lane == 0)
                for (int k = 0; k < issued; ++k) issue(k);
        }
        for (int k = 0; k < nchunks && ok; ++k) {
            const int s = k % NS;
            if (TMA) {
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (uint32_t)((k / NS) & 1), kWaitLimitNs));
                if (!ok) break;
                landed = k + 1;
            } else if (k >= NS) {
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&empty[s], (uint32_t)((k / NS - 1) & 1), a.wait_ns));
                if (!ok) break;
            }
            build_quads(k);
            mbar_arrive(&qready[s]);
            // refill the stage of chunk k-1 with chunk k-1+NS once every consumer has left it
            if (TMA && k >= 1 && k - 1 + NS < nchunks) {
                const int sp = (k - 1) % NS;
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&empty[sp], (uint32_t)(((k - 1) / NS) & 1), a.wait_ns));
                if (!ok) break;
                if (lane == 0) issue(k - 1 + NS);
                ++issued;
            }
        }
        if (!ok) {
            if (lane == 0) atomicExch(&g_status, 1);
            // let the copies still in flight land before the CTA can exit
            for (int k = landed; k < issued; ++k)
                if (!mbar_wait_bounded(&full[k % NS], (uint32_t)((k / NS) & 1), kWaitLimitNs)) break;
        }
        return;
    }
    if (wid >= nunits) return;

    // ====================================================================== consumer warps
    const int c = lane;  // channel within the unit
    const int dch = (u0 + wid) * CPW + c;
    const bool cvalid = dch < a.dim;
    const long long row = (long long)b * a.dim + (cvalid ? dch : 0);
    const float bias = (cvalid && a.bias != nullptr) ? a.bias[dch] : 0.f;
    const float Dd = (cvalid && a.D != nullptr) ? a.D[dch] : 0.f;
    const int trow = wid * CPW + c;  // this lane's row in the CTA's u, delta, z tiles

    // the lane's states, as pairs (2p, 2p + 1)
    float2 A2[PL], h[PL], invA[ZOH ? PL : 1];
    // segment 0 starts from the initial state, later segments (LOCAL) from zero
    const float* h0 = (seg == 0 && cvalid && a.h0 != nullptr) ? a.h0 + row * N : nullptr;
#pragma unroll
    for (int p = 0; p < PL; ++p) {
        const int n0 = 2 * p, n1 = n0 + 1;
        const float a0 = (cvalid && n0 < N) ? a.A[(long long)dch * N + n0] : 0.f;
        const float a1 = (cvalid && n1 < N) ? a.A[(long long)dch * N + n1] : 0.f;
        A2[p] = make_float2(a0 * kLog2e, a1 * kLog2e);
        h[p] = make_float2((h0 && n0 < N) ? h0[n0] : 0.f, (h0 && n1 < N) ? h0[n1] : 0.f);
        // 1/A for the hold (infinite at A = 0 or a padding state: that lane of k then always takes
        // the series branch; the other branch's value is discarded)
        if constexpr (ZOH) invA[p] = make_float2(1.f / a0, 1.f / a1);
    }
    // convolution: taps right-aligned in a 4-tap window (unused taps zero), bias, and the three
    // inputs before the segment (from x itself, or conv_prev before position 0, else zero)
    float w4[4] = {0.f, 0.f, 0.f, 0.f}, cbias = 0.f, xh[3] = {0.f, 0.f, 0.f};
    if (CONV && cvalid) {
        const int K = a.conv_k;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (q >= 4 - K) w4[q] = a.conv_w[(long long)dch * K + q - (4 - K)];
        cbias = a.conv_bias != nullptr ? a.conv_bias[dch] : 0.f;
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const long long pos = t_begin - 3 + q;
            if (pos >= 0)
                xh[q] = In<TIn>::to_f32(static_cast<const TIn*>(a.u)[row * a.L + pos]);
            else if (a.conv_prev != nullptr && pos >= -(K - 1))
                xh[q] = a.conv_prev[row * (K - 1) + (K - 1) + pos];
        }
    }

    constexpr int YTILE = cl::Lanes::YTILE;
    unsigned char* ystage = smem + a.scratch_off + wid * 2 * YTILE;
    float sumdt = 0.f;
    bool ok = true;
    if (a.test_stall) ok = __all_sync(0xffffffffu, mbar_wait_bounded(never, 0u, a.wait_ns));

#pragma unroll 1
    for (int k = 0; k < nchunks && ok; ++k) {
        const int s = k % NS;
        if (TMA) ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (uint32_t)((k / NS) & 1), a.wait_ns));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(&qready[s], (uint32_t)((k / NS) & 1), a.wait_ns));
        if (!ok) break;
        const unsigned char* st = smem + s * a.stage_bytes;
        const unsigned char* qbase = st + a.quad_off;
        unsigned char* ybuf = ystage + (k & 1) * YTILE;
        if (TMA && k >= 2) {  // the store issued from this buffer two chunks ago has read it
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
        }
        const long long tc0 = t_begin + (long long)k * TC;

        // Per-element work of block blk: Delta, Delta*u, u, D*u and the gate, as pairs of steps.
        struct Elem {
            float2 dt[BLK / 2], du[BLK / 2], skip[BLK / 2], gate[BLK / 2];
            float uv[BLK];
        };
        auto elem = [&](int blk, Elem& e) {
            const long long to = tc0 + blk * BLK;  // first step of this block
            float dv[BLK], uv[BLK], zv[BLK];
            if (TMA) {
                cl::tile_load16<TIn>(st + W * TILE, trow, blk * 16, dv);
                cl::tile_load16<TIn>(st, trow, blk * 16, uv);
                // read unconditionally (without z the slot holds stale data, and the gate selects 1)
                cl::tile_load16<TIn>(st + 2 * W * TILE, trow, blk * 16, zv);
            } else {
                const TIn* gd = static_cast<const TIn*>(a.delta) + row * a.L;
                const TIn* gu = static_cast<const TIn*>(a.u) + row * a.L;
                const TIn* gz = static_cast<const TIn*>(a.z) + row * a.L;
#pragma unroll
                for (int j = 0; j < BLK; ++j) {
                    const bool in = cvalid && to + j < t_end;
                    dv[j] = in ? In<TIn>::to_f32(gd[to + j]) : 0.f;
                    uv[j] = in ? In<TIn>::to_f32(gu[to + j]) : 0.f;
                    zv[j] = (in && has_z) ? In<TIn>::to_f32(gz[to + j]) : 0.f;
                }
            }
            if constexpr (CONV) {  // uv holds x: form the convolution outputs of the block
                float xw[BLK + 3];
                xw[0] = xh[0]; xw[1] = xh[1]; xw[2] = xh[2];
#pragma unroll
                for (int j = 0; j < BLK; ++j) xw[3 + j] = uv[j];
#pragma unroll
                for (int j = 0; j < BLK; ++j) {
                    float acc = cbias;
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc = fmaf(w4[q], xw[j + q], acc);
                    uv[j] = a.conv_silu ? acc * sigmoid_approx(acc) : acc;
                }
                xh[0] = xw[BLK]; xh[1] = xw[BLK + 1]; xh[2] = xw[BLK + 2];
            }
            // per-element work of the block: Delta, Delta*u, D*u, gate
#pragma unroll
            for (int j = 0; j < BLK / 2; ++j) {
                // straight-line code (selects, no branches) keeps the block one basic block
                float2 d2 = make_float2(dv[2 * j] + bias, dv[2 * j + 1] + bias);
                const float2 sp2 = softplus2(d2);
                d2 = make_float2(softplus ? sp2.x : d2.x, softplus ? sp2.y : d2.y);
                // steps past the end (or past this segment) leave h unchanged
                if (to + 2 * j >= t_end) d2.x = 0.f;
                if (to + 2 * j + 1 >= t_end) d2.y = 0.f;
                e.dt[j] = d2;
                const float2 u2 = make_float2(uv[2 * j], uv[2 * j + 1]);
                e.du[j] = fmul2(d2, u2);
                e.skip[j] = fmul2(make_float2(Dd, Dd), u2);
                const float2 sg = silu2(make_float2(zv[2 * j], zv[2 * j + 1]));
                e.gate[j] = make_float2(has_z ? sg.x : 1.f, has_z ? sg.y : 1.f);
            }
#pragma unroll
            for (int j = 0; j < BLK; ++j) e.uv[j] = uv[j];
        };
        // The recurrence through block blk's steps, then its outputs.
        auto recur = [&](int blk, const Elem& e) {
            const long long to = tc0 + blk * BLK;
            const float2* dt = e.dt;
            const float2* du = e.du;
            const float2* skip = e.skip;
            const float2* gate = e.gate;
            const float* uv = e.uv;
            float yv[BLK];
#pragma unroll
            for (int j = 0; j < BLK; ++j) {
                const float dq = (j & 1) ? dt[j / 2].y : dt[j / 2].x;
                const float duq = (j & 1) ? du[j / 2].y : du[j / 2].x;
                const float uq = uv[j];
                const float4* qrow = reinterpret_cast<const float4*>(qbase + (blk * BLK + j) * QPITCH);
                float2 ya = make_float2(0.f, 0.f);
#pragma unroll
                for (int p = 0; p < PL; ++p) {
                    const float4 w = qrow[p];  // (B_n, B_n+1, C_n, C_n+1), the same for every lane of a state group
                    const float2 x = fmul2(make_float2(dq, dq), A2[p]);
                    const float2 abar = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    if constexpr (ZOH) {
                        // k B u with k = (Abar - 1) / A where |Delta A| >= 1/4, else the series
                        // Delta phi(Delta A) (there Abar - 1 would cancel)
                        const float2 ser = fmul2(zoh_phi2(x), make_float2(duq, duq));
                        const float2 big = fmul2(fadd2(abar, make_float2(-1.f, -1.f)), fmul2(invA[p], make_float2(uq, uq)));
                        const float2 kx = make_float2(fabsf(x.x) < kZohSeriesLimit ? ser.x : big.x,
                                                      fabsf(x.y) < kZohSeriesLimit ? ser.y : big.y);
                        h[p] = ffma2(abar, h[p], fmul2(kx, make_float2(w.x, w.y)));
                    } else {
                        const float2 bx = fmul2(make_float2(duq, duq), make_float2(w.x, w.y));
                        h[p] = ffma2(abar, h[p], bx);
                    }
                    ya = ffma2(make_float2(w.z, w.w), h[p], ya);
                }
                if (LOCAL) sumdt += dq;
                yv[j] = ya.x + ya.y;
            }
            float yo[BLK];
#pragma unroll
            for (int j = 0; j < BLK / 2; ++j) {
                const float2 y2 = fmul2(fadd2(make_float2(yv[2 * j], yv[2 * j + 1]), skip[j]), gate[j]);
                yo[2 * j] = y2.x;
                yo[2 * j + 1] = y2.y;
            }
            if (TMA) {
                cl::tile_store16<TIn>(ybuf, c, blk * 16, yo);
            } else if (cvalid) {
                TIn* gy = static_cast<TIn*>(a.y) + row * a.L;
#pragma unroll
                for (int j = 0; j < BLK; ++j)
                    if (to + j < t_end) store_out<TIn>(gy + to + j, yo[j]);
            }
        };

#pragma unroll 1
        for (int blk = 0; blk < TC / BLK; ++blk) {
            Elem e;
            elem(blk, e);
            recur(blk, e);
            if constexpr (CKPT) {
                // after every 8 steps: the state before the next 8-step slot, all 16 positions
                // (those past NP as zero), in the backward pass's checkpoint layout
                const long long tt = tc0 + (long long)(blk + 1) * BLK;
                const long long sl8 = tt / 8;
                if ((((blk + 1) * BLK) % 8) == 0 && cvalid && sl8 < a.ck_nslot) {
                    float4* dst = reinterpret_cast<float4*>(a.ckpt + ((b * (long long)a.ck_nslot + sl8) * a.dim + dch) * 16);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        constexpr int last = PL - 1;
                        const int p0 = 2 * q4 < last ? 2 * q4 : last, p1 = 2 * q4 + 1 < last ? 2 * q4 + 1 : last;
                        dst[q4] = 2 * q4 + 1 < PL ? make_float4(h[p0].x, h[p0].y, h[p1].x, h[p1].y)
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            }
        }
        __syncwarp();
        mbar_arrive(&empty[s]);
        if (TMA) {
            // the warp's y tile of this chunk -> global (rows past dim and columns past L clipped)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(&maps.y, ybuf, (int)tc0, (u0 + wid) * CPW, b);
                bulk_commit();
            }
        }
    }
    if (TMA && lane == 0) bulk_wait_all<0>();  // stores complete before the CTA can exit
    __syncwarp();
    if (!ok) {
        if (lane == 0) atomicExch(&g_status, 1);
        return;
    }
    if (!cvalid) return;
    if (LOCAL) {
        // this segment's carry: (prod Abar = 2^(A log2(e) sum Delta), end state from its own start)
        float2* ag = a.agg + (((long long)seg * a.batch + b) * a.dim + dch) * N;
#pragma unroll
        for (int p = 0; p < PL; ++p) {
            const int n0 = 2 * p, n1 = n0 + 1;
            if (n0 < N) ag[n0] = make_float2(ex2_approx(A2[p].x * sumdt), h[p].x);
            if (n1 < N) ag[n1] = make_float2(ex2_approx(A2[p].y * sumdt), h[p].y);
        }
    } else if (a.last_state != nullptr) {
        float* ls = a.last_state + row * N;
#pragma unroll
        for (int p = 0; p < PL; ++p) {
            const int n0 = 2 * p, n1 = n0 + 1;
            if (n0 < N) ls[n0] = h[p].x;
            if (n1 < N) ls[n1] = h[p].y;
        }
    }
}

}  // namespace mscan
