// Fused selective-scan forward kernel for N <= 16 with the B/C operands in tensor memory.
//
// Same computation and work split as scan_fwd_kernel (step size, discretisation, recurrence,
// readout, skip, gate; one warp per 8 channels, 4 lanes per channel, G = 4 states per lane), but
// the per-step B/C operands reach the lanes through tensor memory instead of shared memory:
//  * Every lane needs (B_n, B_n+1, C_n, C_n+1) of its state pairs at every step.  Read from shared
//    memory, these 16-byte vectors were the largest stream through the SM's shared-memory pipe
//    (two 128-bit loads per lane per step) and bounded the whole kernel.
//  * The producer warp writes, for each 32-step segment, one 128-byte "core matrix" per 4-column
//    group (the quads of the 4 state groups, twice) and issues one tcgen05.cp.128x256b per step
//    (8 columns: the two groups of that step as the two K-halves, stride 0 between 8-row core
//    matrices), which fills every 8-lane group of all 128 TMEM lanes with the same pattern.  TMEM
//    lane 4c + g then holds the quads of state group g for every step: 8 columns per step, 256
//    columns per segment, two segments in flight (512 columns).
//  * Measured on B300 this variant is not faster than the shared-memory kernel: TMEM is per-lane
//    storage, so the broadcast writes 128 KB per segment (every lane its own copy), and the copies
//    plus their synchronisation cost about as much as the shared-memory reads they replace.  It is
//    kept as a tested alternative (MAMBA_SCAN_TMEM=1).
//  * Consumer lanes read their operands with tcgen05.ld (32 columns = 4 steps per load); shared
//    memory now carries only the (Delta, Delta, Delta*u, Delta*u) quads and the partial sums of
//    C.h.
// Lane mapping in the recurrence: lane = 4c + g (channel c of the warp's 8, state group g).
// Synchronisation: full/empty mbarriers for the TMA ring (as in scan_fwd_kernel), and
// tm_full/tm_empty for the two TMEM segments (tcgen05.commit arrives on tm_full once a segment's
// copies have landed; every consumer lane arrives on tm_empty after its last load of a segment).
// All waits are bounded; TMEM is allocated and released by the producer warp around CTA barriers.
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "scan_fwd.cuh"

namespace mscan {

constexpr int kTmSeg = 32;                                   // steps per TMEM segment
constexpr int kTmCols = 512;                                 // 2 segments x 32 steps x 8 columns
constexpr int kQPitchT = 18 * 16;                            // bytes per channel row of Delta quads
constexpr int kQBufT = kUnitCh * kQPitchT;                   // one Delta-quad buffer (8 channels)
constexpr int kYPitchT = kSlot * 4 + 16;                     // bytes per (channel, lane group) row of partials
constexpr int kWarpScratchT = 2 * kQBufT + 32 * kYPitchT;    // 7168 bytes
constexpr int kSrcBytes = 2 * kTmSeg * 128;                  // one segment's copy source: 64 x 128 B

// Slot of step t's Delta quad in a channel row.  Phase A lane (c, g) writes steps 4g..4g+3 of
// channel c; with 18-chunk rows and this slot map, the 8 lanes of a quarter-warp (channels c, c+1,
// groups 0..3) hit 8 different bank groups.
__device__ __forceinline__ int qslot(int t) { return t + (t >> 3); }

template <typename TIn, bool TMA, bool AGG, bool SOFTPLUS, bool GATE>
__global__ void __launch_bounds__(kMaxThreads, 1)
    scan_fwd_tm_kernel(const FwdArgs a, const __grid_constant__ FwdMaps maps) {
    constexpr int NP = 16;
    constexpr int G = 4;
    constexpr int NPAIR = NP / 2;
    constexpr int TC = Chunk<TIn>::TC;
    constexpr int SPC = Chunk<TIn>::SPC;
    constexpr int ES = (int)sizeof(TIn);
    constexpr int SEGS_PER_CHUNK = TC / kTmSeg;
    constexpr bool has_z = !AGG && GATE;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int NS = a.nstage;
    const int W = a.wmax;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.bar_off);
    uint64_t* empty = full + NS;
    uint64_t* tm_full = empty + NS;
    uint64_t* tm_empty = tm_full + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(tm_empty + 2);

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
    const int nsegs = (int)((t_end - t_begin + kTmSeg - 1) / kTmSeg);
    const int nslots = (int)((t_end - t_begin + kSlot - 1) / kSlot);

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 32 * nunits);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&tm_full[s], 1);
            mbar_init(&tm_empty[s], 32 * nunits);
        }
        mbar_fence_init();
        fence_proxy_async_smem();
    }
    if (wid == W) tmem_alloc(tslot, kTmCols);
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tbase = *tslot;

    bool ok = true;
    if (wid == W) {
        // ================================================================== producer warp
        const int mi = nunits == a.wlo ? 0 : 1;
        const uint32_t tx = (uint32_t)(nunits * kUnitCh * 128 * (has_z ? 3 : 2) + (AGG ? 1 : 2) * N * 128);
        auto issue = [&](int k) {  // lane 0: TMA loads of chunk k into stage k % NS
            const int s = k % NS;
            unsigned char* st = smem + s * a.stage_bytes;
            const int t0 = (int)(t_begin + (long long)k * TC);
            mbar_arrive_expect_tx(&full[s], tx);
            const int r0 = u0 * kUnitCh;
            tma_load_3d(st, &maps.u[mi], &full[s], t0, r0, b);
            tma_load_3d(st + W * 1024, &maps.d[mi], &full[s], t0, r0, b);
            if (has_z) tma_load_3d(st + 2 * W * 1024, &maps.z[mi], &full[s], t0, r0, b);
            tma_load_3d(st + a.bc_off, &maps.B, &full[s], t0, 0, b);
            if (!AGG) tma_load_3d(st + a.bc_off + NP * 128, &maps.C, &full[s], t0, 0, b);
        };
        // Copy source of segment m (steps [32m, 32m+32) of this range): column group j = 2t + p
        // holds, in rows 0-3 and again 4-7, the quads (B_n, B_n+1, C_n, C_n+1), n = 4g + 2p, of
        // state groups g = 0..3 at step t.
        auto build_source = [&](int m, unsigned char* src) {
            const int k = m / SEGS_PER_CHUNK;
            const int o = (m % SEGS_PER_CHUNK) * kTmSeg;  // first step of the segment within chunk k
            const unsigned char* st = smem + (k % NS) * a.stage_bytes;
            for (int item = lane; item < NPAIR * (kTmSeg / 4); item += 32) {
                const int P = item & (NPAIR - 1), tq = item / NPAIR;
                const int n0 = 2 * P, n1 = n0 + 1;
                float b0[4] = {0.f, 0.f, 0.f, 0.f}, b1[4] = {0.f, 0.f, 0.f, 0.f};
                float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
                if (TMA) {
                    const unsigned char* tB = st + a.bc_off;
                    const unsigned char* tC = tB + NP * 128;
                    const int byte = (o + 4 * tq) * ES;
                    if (n0 < N) { tile_load4<TIn>(tB, n0, byte, b0); if (!AGG) tile_load4<TIn>(tC, n0, byte, c0); }
                    if (n1 < N) { tile_load4<TIn>(tB, n1, byte, b1); if (!AGG) tile_load4<TIn>(tC, n1, byte, c1); }
                } else {
                    const TIn* gB = static_cast<const TIn*>(a.B);
                    const TIn* gC = static_cast<const TIn*>(a.C);
                    const long long tb = t_begin + (long long)m * kTmSeg + 4 * tq;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (tb + i >= t_end) break;
                        if (n0 < N) {
                            b0[i] = In<TIn>::to_f32(gB[((long long)b * N + n0) * a.L + tb + i]);
                            if (!AGG) c0[i] = In<TIn>::to_f32(gC[((long long)b * N + n0) * a.L + tb + i]);
                        }
                        if (n1 < N) {
                            b1[i] = In<TIn>::to_f32(gB[((long long)b * N + n1) * a.L + tb + i]);
                            if (!AGG) c1[i] = In<TIn>::to_f32(gC[((long long)b * N + n1) * a.L + tb + i]);
                        }
                    }
                }
                const int g = P >> 1, p = P & 1;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float4* cm = reinterpret_cast<float4*>(src + (2 * (4 * tq + i) + p) * 128);
                    const float4 q = make_float4(b0[i], b1[i], c0[i], c1[i]);
                    cm[g] = q;
                    cm[g + 4] = q;
                }
            }
        };

        int issued = 0, landed = 0, committed = -1;
        if (TMA) {
            issued = min(NS, nchunks);
            if (lane == 0)
                for (int k = 0; k < issued; ++k) issue(k);
        }
        for (int k = 0; k < nchunks && ok; ++k) {
            if (TMA) {
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[k % NS], (uint32_t)((k / NS) & 1), kWaitLimitNs));
                if (!ok) break;
                landed = k + 1;
            }
            for (int hs = 0; hs < SEGS_PER_CHUNK && ok; ++hs) {
                const int m = k * SEGS_PER_CHUNK + hs;
                if (m >= nsegs) break;
                const int tb = m & 1;
                if (m >= 2) {  // consumers are done with segment m-2 (same TMEM columns, same source)
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait_bounded(&tm_empty[tb], (uint32_t)(((m >> 1) - 1) & 1), kWaitLimitNs));
                    if (!ok) break;
                }
                unsigned char* src = smem + a.src_off + tb * kSrcBytes;
                build_source(m, src);
                fence_proxy_async_smem();  // generic-proxy writes -> visible to tcgen05.cp
                __syncwarp();
                if (lane == 0) {
                    const uint32_t sbase = smem_u32(src);
                    const uint32_t tcol = tbase + (uint32_t)(tb * 256);
#pragma unroll 4
                    for (int t = 0; t < kTmSeg; ++t) tmem_cp_128x256b(tcol + 8 * t, smem_desc(sbase + t * 256, 128, 0));
                    tmem_commit(&tm_full[tb]);
                }
                committed = m;
                __syncwarp();
            }
            if (!ok) break;
            // refill the stage of chunk k-1 with chunk k-1+NS once every consumer has left it
            if (TMA && k >= 1 && k - 1 + NS < nchunks) {
                const int sp = (k - 1) % NS;
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&empty[sp], (uint32_t)(((k - 1) / NS) & 1), kWaitLimitNs));
                if (!ok) break;
                if (lane == 0) issue(k - 1 + NS);
                ++issued;
            }
        }
        if (!ok) {
            // let the copies still in flight land before TMEM and shared memory are released
            for (int k = landed; k < issued; ++k)
                if (!mbar_wait_bounded(&full[k % NS], (uint32_t)((k / NS) & 1), kWaitLimitNs)) break;
            if (committed >= 0)
                mbar_wait_bounded(&tm_full[committed & 1], (uint32_t)((committed >> 1) & 1), kWaitLimitNs);
        }
    } else if (wid < nunits) {
        // ================================================================== consumer warps
        const int c = lane >> 2;  // channel within the unit
        const int g = lane & 3;   // state group: states 4g .. 4g+3
        const int dch = (u0 + wid) * kUnitCh + c;
        const bool cvalid = dch < a.dim;
        const long long row = (long long)b * a.dim + (cvalid ? dch : 0);
        const float bias = (cvalid && a.bias != nullptr) ? a.bias[dch] : 0.f;
        const float Dd = (!AGG && cvalid && a.D != nullptr) ? a.D[dch] : 0.f;

        f2p A2[G / 2];  // A * log2(e) of the lane's state pairs
        f2p h[G / 2];   // the lane's states, as packed pairs
        const float* hin = (!AGG && cvalid && a.h0 != nullptr) ? a.h0 + row * N : nullptr;
#pragma unroll
        for (int p = 0; p < G / 2; ++p) {
            const int n0 = g * G + 2 * p, n1 = n0 + 1;
            float h0 = (hin && n0 < N) ? hin[n0] : 0.f, h1 = (hin && n1 < N) ? hin[n1] : 0.f;
            if (!AGG && seg > 0 && cvalid) {
                // fold the carries of segments 0 .. seg-1 in order: h <- prod Abar * h + h_end
                for (int q = 0; q < seg; ++q) {
                    const float2* ag = a.agg + (((long long)q * a.batch + b) * a.dim + dch) * N;
                    if (n0 < N) { const float2 v = ag[n0]; h0 = fmaf(v.x, h0, v.y); }
                    if (n1 < N) { const float2 v = ag[n1]; h1 = fmaf(v.x, h1, v.y); }
                }
            }
            A2[p] = ppack((cvalid && n0 < N) ? a.A[(long long)dch * N + n0] * kLog2e : 0.f,
                          (cvalid && n1 < N) ? a.A[(long long)dch * N + n1] * kLog2e : 0.f);
            h[p] = ppack(h0, h1);
        }

        unsigned char* wsq = smem + a.scratch_off + wid * kWarpScratchT;
        unsigned char* wsy = wsq + 2 * kQBufT;
        const uint32_t tlane = tbase + ((uint32_t)(32 * (wid & 3)) << 16);  // this warp's TMEM lanes
        float sumdt = 0.f;

        auto wait_tiles = [&](int k) -> bool {
            if (!TMA) return true;
            return __all_sync(0xffffffffu, mbar_wait_bounded(&full[k % NS], (uint32_t)((k / NS) & 1), kWaitLimitNs));
        };

        // Phase A of slot i: Delta, Delta*u of steps 4g..4g+3 of channel c -> quads; D*u and gate.
        auto phase_a = [&](int i, float2& skip01, float2& skip23, float2& gate01, float2& gate23) {
            const int k = i / SPC, sl = i % SPC;
            const long long to = t_begin + (long long)i * kSlot + g * kOwned;
            const unsigned char* st = smem + (k % NS) * a.stage_bytes;
            float dv[4], uv[4], zv[4];
            if (TMA) {
                const int byte = (sl * kSlot + g * kOwned) * ES;
                tile_load4<TIn>(st + (W + wid) * 1024, c, byte, dv);
                tile_load4<TIn>(st + wid * 1024, c, byte, uv);
                if (has_z) tile_load4<TIn>(st + (2 * W + wid) * 1024, c, byte, zv);
            } else {
                const TIn* gd = static_cast<const TIn*>(a.delta) + row * a.L;
                const TIn* gu = static_cast<const TIn*>(a.u) + row * a.L;
                const TIn* gz = static_cast<const TIn*>(a.z) + row * a.L;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = cvalid && to + j < t_end;
                    dv[j] = in ? In<TIn>::to_f32(gd[to + j]) : 0.f;
                    uv[j] = in ? In<TIn>::to_f32(gu[to + j]) : 0.f;
                    zv[j] = (in && has_z) ? In<TIn>::to_f32(gz[to + j]) : 0.f;
                }
            }
            float2 dt01 = make_float2(dv[0] + bias, dv[1] + bias);
            float2 dt23 = make_float2(dv[2] + bias, dv[3] + bias);
            if (SOFTPLUS) {
                dt01 = softplus2(dt01);
                dt23 = softplus2(dt23);
            }
            if (to + 4 > t_end) {  // steps past the end (or past this segment) leave h unchanged
                const long long nv = t_end - to;
                if (nv < 1) dt01.x = 0.f;
                if (nv < 2) dt01.y = 0.f;
                if (nv < 3) dt23.x = 0.f;
                dt23.y = 0.f;
            }
            const float2 du01 = fmul2(dt01, make_float2(uv[0], uv[1]));
            const float2 du23 = fmul2(dt23, make_float2(uv[2], uv[3]));
            float4* qw = reinterpret_cast<float4*>(wsq + (i & 1) * kQBufT + c * kQPitchT);
            qw[qslot(4 * g + 0)] = make_float4(dt01.x, dt01.x, du01.x, du01.x);
            qw[qslot(4 * g + 1)] = make_float4(dt01.y, dt01.y, du01.y, du01.y);
            qw[qslot(4 * g + 2)] = make_float4(dt23.x, dt23.x, du23.x, du23.x);
            qw[qslot(4 * g + 3)] = make_float4(dt23.y, dt23.y, du23.y, du23.y);
            if (!AGG) {
                skip01 = fmul2(make_float2(Dd, Dd), make_float2(uv[0], uv[1]));
                skip23 = fmul2(make_float2(Dd, Dd), make_float2(uv[2], uv[3]));
                if (has_z) {
                    gate01 = silu2(make_float2(zv[0], zv[1]));
                    gate23 = silu2(make_float2(zv[2], zv[3]));
                } else {
                    gate01 = gate23 = make_float2(1.f, 1.f);
                }
            }
        };

        // one step: (Delta, Delta | Delta*u, Delta*u) from shared memory; the lane's pairs
        // (B_n, B_n+1), (C_n, C_n+1) for its two state pairs from TMEM registers w[0..3]
        auto step = [&](const ulonglong2* qrow, int t, const f2p* w, float* yp) {
            const ulonglong2 q = qrow[qslot(t)];
            if (AGG) sumdt += plo(q.x);
            f2p ya;
#pragma unroll
            for (int p = 0; p < G / 2; ++p) {
                const f2p abar = pex2(pmul(q.x, A2[p]));
                const f2p bx = pmul(q.y, w[2 * p]);
                h[p] = pfma(abar, h[p], bx);
                if (!AGG) ya = p == 0 ? pmul(w[2 * p + 1], h[p]) : pfma(w[2 * p + 1], h[p], ya);
            }
            if (!AGG) yp[t] = psum(ya);
        };

        // Phase B of slot i: 16 steps; B/C pairs arrive 4 steps (32 columns) per TMEM load.
        auto phase_b = [&](int i, float* yp) {
            const int m = i >> 1;
            const uint32_t tcol = tlane + (uint32_t)((m & 1) * 256 + (i & 1) * 128);
            const ulonglong2* qrow = reinterpret_cast<const ulonglong2*>(wsq + (i & 1) * kQBufT + c * kQPitchT);
#pragma unroll
            for (int tq = 0; tq < kSlot / 4; ++tq) {
                f2p w[16];
                tmem_ld32_pairs(tcol + 32 * tq, w);
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) step(qrow, 4 * tq + tt, w + 4 * tt, yp);
            }
        };

        // Phase C of slot i: the 4 lanes' partials of steps 4g..4g+3 of channel c, skip, gate, store.
        auto phase_c = [&](int i, float2 skip01, float2 skip23, float2 gate01, float2 gate23) {
            const long long to = t_begin + (long long)i * kSlot + g * kOwned;
            float4 acc = *reinterpret_cast<const float4*>(wsy + (4 * c) * kYPitchT + g * 16);
#pragma unroll
            for (int gg = 1; gg < kLanesPerCh; ++gg) {
                const float4 v = *reinterpret_cast<const float4*>(wsy + (4 * c + gg) * kYPitchT + g * 16);
                const float2 lo = fadd2(make_float2(acc.x, acc.y), make_float2(v.x, v.y));
                const float2 hi = fadd2(make_float2(acc.z, acc.w), make_float2(v.z, v.w));
                acc = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
            const float2 y01 = fmul2(fadd2(make_float2(acc.x, acc.y), skip01), gate01);
            const float2 y23 = fmul2(fadd2(make_float2(acc.z, acc.w), skip23), gate23);
            const float yv[4] = {y01.x, y01.y, y23.x, y23.y};
            TIn* gy = static_cast<TIn*>(a.y) + row * a.L + to;
            if (TMA && to + 4 <= t_end) {
                if (cvalid) store4<TIn>(gy, yv);
            } else if (cvalid) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (to + j < t_end) store_out<TIn>(gy + j, yv[j]);
            }
        };

        float2 sk01 = make_float2(0.f, 0.f), sk23 = sk01, gt01 = sk01, gt23 = sk01;
        ok = wait_tiles(0);
        if (ok) phase_a(0, sk01, sk23, gt01, gt23);
        __syncwarp();
#pragma unroll 1
        for (int i = 0; i < nslots && ok; ++i) {
            const int k = i / SPC, sl = i % SPC, m = i >> 1;
            const bool next = i + 1 < nslots;
            if ((i & 1) == 0) {
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&tm_full[m & 1], (uint32_t)((m >> 1) & 1), kWaitLimitNs));
                tmem_fence_after_sync();
            }
            if (ok && next && sl == SPC - 1) ok = wait_tiles(k + 1);
            if (!ok) break;
            float2 nk01 = make_float2(0.f, 0.f), nk23 = nk01, nt01 = nk01, nt23 = nk01;
            if (next) phase_a(i + 1, nk01, nk23, nt01, nt23);
            float yp[kSlot];
            phase_b(i, yp);
            if ((i & 1) == 1 || !next) {  // this lane's last TMEM load of segment m is complete
                tmem_fence_before_sync();
                mbar_arrive(&tm_empty[m & 1]);
            }
            __syncwarp();
            if (sl == SPC - 1 || !next) mbar_arrive(&empty[k % NS]);  // done with chunk k's stage
            if (!AGG) {
                float4* yw = reinterpret_cast<float4*>(wsy + (4 * c + g) * kYPitchT);
#pragma unroll
                for (int j = 0; j < kSlot / 4; ++j)
                    yw[j] = make_float4(yp[4 * j], yp[4 * j + 1], yp[4 * j + 2], yp[4 * j + 3]);
            }
            __syncwarp();
            if (!AGG) phase_c(i, sk01, sk23, gt01, gt23);
            sk01 = nk01; sk23 = nk23; gt01 = nt01; gt23 = nt23;
        }
        if (ok && cvalid) {
            if (AGG) {
                float2* ag = a.agg + (((long long)seg * a.batch + b) * a.dim + dch) * N;
#pragma unroll
                for (int p = 0; p < G / 2; ++p) {
                    const int n0 = g * G + 2 * p, n1 = n0 + 1;
                    if (n0 < N) ag[n0] = make_float2(ex2_approx(plo(A2[p]) * sumdt), plo(h[p]));
                    if (n1 < N) ag[n1] = make_float2(ex2_approx(phi(A2[p]) * sumdt), phi(h[p]));
                }
            } else if (a.last_state != nullptr && seg == a.nseg - 1) {
                float* ls = a.last_state + row * N;
#pragma unroll
                for (int p = 0; p < G / 2; ++p) {
                    const int n0 = g * G + 2 * p, n1 = n0 + 1;
                    if (n0 < N) ls[n0] = plo(h[p]);
                    if (n1 < N) ls[n1] = phi(h[p]);
                }
            }
        }
    }
    if (!ok && lane == 0) atomicExch(&g_status, 1);
    // every TMEM load and copy of this CTA is complete before the columns are released
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (wid == W) tmem_dealloc(tbase, kTmCols);
}

}  // namespace mscan
