// Second launch of a split time axis for the channel-per-lane forward scan: adds to each segment's
// outputs the part of the state carried in from the segments before it.
//
// With the time axis cut into segments, scan_fwd_cl_kernel (LOCAL) runs segment 0 from the
// initial state and every later segment s from a zero state, all at once.  The recurrence
// h_t = Abar_t h_{t-1} + Bbar_t x_t is linear in h, so inside segment s the true state is the
// segment's own state plus the state h_in it starts from, decayed step by step:
//   h_t = h_t(own) + G_t,   G_t = Abar_t G_{t-1},   G_{start-1} = h_in,
// and the true output adds (C_t . G_t) silu(z_t) to the segment's own output (visual guide to Mamba
// and SSMs, section 3.3: the scan operator (a2, b2) o (a1, b1) = (a1 a2, a2 b1 + b2) is
// associative, so per-segment results combine in any grouping).  h_in is the fold of the carries
// (prod Abar, own end state) that the first launch wrote: segment 0's end state (already from the
// initial state), then h <- prod Abar * h + h_end for segments 1 .. s-1.
//
// One warp per (segment s > 0, batch row, 32 channels), lane = channel with all NP states in
// registers, as in the forward kernel.  The warp walks its segment chunk by chunk: delta, z, y and
// C tiles arrive by TMA into a ring of stages, the lane adds its channel's correction to the y tile
// in place, and a TMA store writes the tile back.  Only Delta and C enter; B and u do not.
//
// With A < 0, G decays geometrically, and the walk stops after the first chunk at whose end every
// |G_n| of every lane of the warp is at most 2^-40 times the largest |h_in,n| of its lane: what is
// left is far below the fp32 resolution of the outputs it could still reach.  Without decay
// (A >= 0, or Delta = 0 throughout) the walk covers the whole segment.  The warp of the last
// segment also writes the final state, prod Abar * h_in + h_end.
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "scan_fwd.cuh"
#include "scan_fwd_cl.cuh"

namespace mscan {
namespace fix {

constexpr int kStages = 3;
constexpr int kTile = 32 * cl::kRowBytes;  // one [32 channels, one chunk] tile
constexpr float kDropBelow = 9.094947017729282e-13f;  // 2^-40

// Stage: [delta tile | z tile | y tile | C tile (N rows of 128 bytes)], 1024-byte aligned for the
// 128-byte swizzle; then kStages mbarriers.
template <int NP>
struct Layout {
    static constexpr int STAGE = (3 * kTile + NP * cl::kRowBytes + 1023) / 1024 * 1024;
    static constexpr int SMEM = kStages * STAGE + kStages * 8 + 1024;
};

}  // namespace fix

// delta, z, y: box [TC, 32 channels] over [L, dim, batch]; C: box [TC, N] over [L, N, batch].
struct FixMaps {
    CUtensorMap d, z, y, C;
};

template <typename TIn, int NP, bool TMA>
__global__ void __launch_bounds__(32) scan_fix_kernel(const FwdArgs a, const __grid_constant__ FixMaps maps) {
    constexpr int TC = Chunk<TIn>::TC;
    constexpr int ES = (int)sizeof(TIn);
    constexpr int BLK = 16 / ES;  // steps per 16-byte tile read
    constexpr int NPAIR = NP / 2;
    constexpr int NS = fix::kStages;
    constexpr int STAGE = fix::Layout<NP>::STAGE;
    constexpr int TILE = fix::kTile;
    static_assert(NP % 2 == 0 && NP <= 16, "shape");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * STAGE);

    const int lane = threadIdx.x;
    const long long item = blockIdx.x;
    const int unit = (int)(item % a.upr);
    const int b = (int)((item / a.upr) % a.batch);
    const int seg = 1 + (int)(item / ((long long)a.upr * a.batch));
    const int N = a.dstate;
    const int dch = unit * 32 + lane;
    const bool cvalid = dch < a.dim;
    const long long row = (long long)b * a.dim + (cvalid ? dch : 0);
    const long long t_begin = (long long)seg * a.seg_len;
    const long long t_end = min(a.L, t_begin + a.seg_len);
    const int nchunks = (int)((t_end - t_begin + TC - 1) / TC);
    const bool has_z = a.z != nullptr;
    const bool softplus = a.softplus != 0;
    const float bias = (cvalid && a.bias != nullptr) ? a.bias[dch] : 0.f;

    // h_in: segment 0's end state, then the carries of segments 1 .. seg-1
    const long long cstride = (long long)a.batch * a.dim * N;  // one segment's carries
    const float2* cr = a.agg + row * N;
    float2 A2[NPAIR], G[NPAIR];
#pragma unroll
    for (int p = 0; p < NPAIR; ++p) {
        const int n0 = 2 * p, n1 = n0 + 1;
        const bool v0 = cvalid && n0 < N, v1 = cvalid && n1 < N;
        A2[p] = make_float2(v0 ? a.A[(long long)dch * N + n0] * kLog2e : 0.f, v1 ? a.A[(long long)dch * N + n1] * kLog2e : 0.f);
        G[p] = make_float2(v0 ? cr[n0].y : 0.f, v1 ? cr[n1].y : 0.f);
    }
    for (int q = 1; q < seg; ++q) {
        const float2* c = cr + q * cstride;
#pragma unroll
        for (int p = 0; p < NPAIR; ++p) {
            const int n0 = 2 * p, n1 = n0 + 1;
            if (cvalid && n0 < N) { const float2 v = c[n0]; G[p].x = fmaf(v.x, G[p].x, v.y); }
            if (cvalid && n1 < N) { const float2 v = c[n1]; G[p].y = fmaf(v.x, G[p].y, v.y); }
        }
    }
    if (seg == a.nseg - 1 && a.last_state != nullptr && cvalid) {
        const float2* c = cr + seg * cstride;
        float* ls = a.last_state + row * N;
#pragma unroll
        for (int p = 0; p < NPAIR; ++p) {
            const int n0 = 2 * p, n1 = n0 + 1;
            if (n0 < N) { const float2 v = c[n0]; ls[n0] = fmaf(v.x, G[p].x, v.y); }
            if (n1 < N) { const float2 v = c[n1]; ls[n1] = fmaf(v.x, G[p].y, v.y); }
        }
    }
    // drop threshold (an infinite or NaN carry is never dropped)
    float hmax = 0.f;
#pragma unroll
    for (int p = 0; p < NPAIR; ++p) hmax = fmaxf(hmax, fmaxf(fabsf(G[p].x), fabsf(G[p].y)));
    const float thr = hmax <= 3.4028234663852886e38f ? hmax * fix::kDropBelow : 0.f;

    if (TMA && lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
        mbar_fence_init();
        fence_proxy_async_smem();
    }
    __syncwarp();
    const uint32_t tx = (uint32_t)((has_z ? 3 : 2) * TILE + N * cl::kRowBytes);
    auto issue = [&](int k) {  // lane 0: chunk k into stage k % NS
        unsigned char* st = smem + (k % NS) * STAGE;
        const int t0 = (int)(t_begin + (long long)k * TC);
        mbar_arrive_expect_tx(&full[k % NS], tx);
        tma_load_3d(st, &maps.d, &full[k % NS], t0, unit * 32, b);
        if (has_z) tma_load_3d(st + TILE, &maps.z, &full[k % NS], t0, unit * 32, b);
        tma_load_3d(st + 2 * TILE, &maps.y, &full[k % NS], t0, unit * 32, b);
        tma_load_3d(st + 3 * TILE, &maps.C, &full[k % NS], t0, 0, b);
    };
    int issued = 0, landed = 0;
    if (TMA) {
        issued = min(NS, nchunks);
        if (lane == 0)
            for (int k = 0; k < issued; ++k) issue(k);
    }

    bool ok = true;
#pragma unroll 1
    for (int k = 0; k < nchunks && ok; ++k) {
        const int s = k % NS;
        if (TMA) {
            ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (uint32_t)((k / NS) & 1), kWaitLimitNs));
            if (!ok) break;
            landed = k + 1;
        }
        unsigned char* st = smem + s * STAGE;
        const unsigned char* tC = st + 3 * TILE;
        const long long tc0 = t_begin + (long long)k * TC;
#pragma unroll 1
        for (int blk = 0; blk < TC / BLK; ++blk) {
            const long long to = tc0 + blk * BLK;
            float dv[BLK], zv[BLK], yv[BLK];
            if (TMA) {
                cl::tile_load16<TIn>(st, lane, blk * 16, dv);
                // read unconditionally (without z the slot holds stale data, and the gate selects 1)
                cl::tile_load16<TIn>(st + TILE, lane, blk * 16, zv);
                cl::tile_load16<TIn>(st + 2 * TILE, lane, blk * 16, yv);
            } else {
                const TIn* gd = static_cast<const TIn*>(a.delta) + row * a.L;
                const TIn* gz = static_cast<const TIn*>(a.z) + row * a.L;
                const TIn* gy = static_cast<const TIn*>(a.y) + row * a.L;
#pragma unroll
                for (int j = 0; j < BLK; ++j) {
                    const bool in = cvalid && to + j < t_end;
                    dv[j] = in ? In<TIn>::to_f32(gd[to + j]) : 0.f;
                    zv[j] = (in && has_z) ? In<TIn>::to_f32(gz[to + j]) : 0.f;
                    yv[j] = in ? In<TIn>::to_f32(gy[to + j]) : 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < BLK; ++j) {
                float dt = dv[j] + bias;
                const float sp = softplus1(dt);
                dt = softplus ? sp : dt;
                dt = to + j < t_end ? dt : 0.f;  // steps past the end leave G unchanged
                const float gate = has_z ? silu_f(zv[j]) : 1.f;
                const int col = blk * BLK + j;  // step within the chunk
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int p = 0; p < NPAIR; ++p) {
                    float2 cv;
                    if (TMA) {
                        // rows of the C tile past N were never written: select zero there
                        if constexpr (ES == 4) {
                            cv = make_float2(*reinterpret_cast<const float*>(tC + swz128(2 * p, col * 4)),
                                             *reinterpret_cast<const float*>(tC + swz128(2 * p + 1, col * 4)));
                        } else {
                            cv = make_float2(bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(tC + swz128(2 * p, col * 2))),
                                             bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(tC + swz128(2 * p + 1, col * 2))));
                        }
                        cv = make_float2(2 * p < N ? cv.x : 0.f, 2 * p + 1 < N ? cv.y : 0.f);
                    } else {
                        const bool in = to + j < t_end;
                        const TIn* gc = static_cast<const TIn*>(a.C) + (long long)b * N * a.L + to + j;
                        cv = make_float2((in && 2 * p < N) ? In<TIn>::to_f32(gc[(long long)(2 * p) * a.L]) : 0.f,
                                         (in && 2 * p + 1 < N) ? In<TIn>::to_f32(gc[(long long)(2 * p + 1) * a.L]) : 0.f);
                    }
                    const float2 x = fmul2(make_float2(dt, dt), A2[p]);
                    G[p] = fmul2(make_float2(ex2_approx(x.x), ex2_approx(x.y)), G[p]);
                    acc = ffma2(cv, G[p], acc);
                }
                yv[j] = fmaf(acc.x + acc.y, gate, yv[j]);
            }
            if (TMA) {
                cl::tile_store16<TIn>(st + 2 * TILE, lane, blk * 16, yv);
            } else if (cvalid) {
                TIn* gy = static_cast<TIn*>(a.y) + row * a.L;
#pragma unroll
                for (int j = 0; j < BLK; ++j)
                    if (to + j < t_end) store_out<TIn>(gy + to + j, yv[j]);
            }
        }
        if (TMA) {
            // the corrected y tile -> global (rows past dim and columns past L clipped)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(&maps.y, st + 2 * TILE, (int)tc0, unit * 32, b);
                bulk_commit();
            }
        }
        bool alive = false;
#pragma unroll
        for (int p = 0; p < NPAIR; ++p) alive = alive || !(fabsf(G[p].x) <= thr) || !(fabsf(G[p].y) <= thr);
        if (!__any_sync(0xffffffffu, alive)) break;
        if (TMA && k + NS < nchunks) {
            // refill this stage once the store has read its y tile
            if (lane == 0) {
                bulk_wait_read<0>();
                issue(k + NS);
            }
            ++issued;
        }
    }
    if (TMA && lane == 0) {
        // copies still in flight land, and stores complete, before the CTA can exit
        for (int k = landed; k < issued; ++k)
            if (!mbar_wait_bounded(&full[k % NS], (uint32_t)((k / NS) & 1), kWaitLimitNs)) {
                ok = false;
                break;
            }
        bulk_wait_all<0>();
    }
    if (!ok && lane == 0) atomicExch(&g_status, 1);
}

}  // namespace mscan
