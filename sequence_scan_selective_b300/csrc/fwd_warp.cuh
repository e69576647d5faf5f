// Forward scan, four-lanes-per-channel kernel (any N <= 64; also the exact hold and the fused
// convolution): planner, TMA descriptors and launches of scan_fwd_kernel.  Included by one
// translation unit per input type (fwd_warp_f32.cu, fwd_warp_bf16.cu), which instantiates
// fwd_warp_run_t and fwd_warp_status_t for that type.
#pragma once
#include <cstring>

#include "host.cuh"
#include "fwd_common.cuh"
#include "scan_fwd.cuh"

namespace mscan {

// Work split of scan_fwd_kernel.  Units (8 channels of one batch row, one consumer warp each) are
// the grain.  The time axis is split into segments only when the units alone cannot give every SM
// several warps (a split costs one extra pass over delta, u and B for all but the last segment).
// Each (segment, batch row) gets kcta CTAs with an even share of its units, so that the grid is
// about one CTA per SM and the per-SM work differs by at most one unit.
template <typename TIn, int NP>
static int plan_warp(const mamba_scan_shape* s, int nsm, FwdPlan& p) {
    constexpr int TC = Chunk<TIn>::TC;
    constexpr int CPW = kUnitCh;    // channels per work unit
    constexpr int UB = CPW * 128;   // u/delta/z tile bytes per unit and chunk
    const long long L = s->seqlen;
    p.upr = (s->dim + CPW - 1) / CPW;
    const long long units = (long long)s->batch * p.upr;
    long long want = env_int("MAMBA_SCAN_NSEG", 0);
    if (want <= 0) {
        want = 1;
        const long long target = (long long)nsm * 10;  // consumer warps that keep every SM busy
        if (units * 2 < target) want = (target + units - 1) / units;
    }
    long long maxseg = L / (8LL * TC);
    if (maxseg < 1) maxseg = 1;
    if (want > maxseg) want = maxseg;
    if (want > 4096) want = 4096;
    p.nseg = 1;
    p.seg_len = L;
    if (want > 1) {
        long long seg = (L + want - 1) / want;
        seg = (seg + TC - 1) / TC * TC;
        p.seg_len = seg;
        p.nseg = (int)((L + seg - 1) / seg);
    }
    const long long rows = (long long)s->batch * p.nseg;
    // shared memory: NS stages of [u | delta | z tiles (1 KB per unit each) | B, C tiles | quads],
    // then per-warp scratch, then 3 NS mbarriers.  Consumer warps per CTA are capped so that two
    // stages fit.
    const int bc_bytes = 2 * NP * 128, quad_bytes = TC * (NP / 2) * 16;
    const int wscratch = kWarpScratch;
    auto stage_of = [&](int w) { return (3 * w * UB + bc_bytes + quad_bytes + 1023) / 1024 * 1024; };
    auto smem_of = [&](int w, int ns) { return ns * stage_of(w) + w * wscratch + 3 * ns * 8 + 1024; };
    int wcap = kMaxConsumerWarps;
    while (wcap > 1 && smem_of(wcap, 2) > kSmemLimit) --wcap;
    const int wforce = env_int("MAMBA_SCAN_WMAX", 0);
    if (wforce > wcap) return fail(MAMBA_ERR_ARG, "MAMBA_SCAN_WMAX above %d", wcap);
    long long k;
    if (wforce > 0) {
        k = (p.upr + wforce - 1) / wforce;
    } else {
        k = rows >= nsm ? 1 : nsm / rows;
        if (k > p.upr) k = p.upr;
        if ((p.upr + k - 1) / k > wcap) k = (p.upr + wcap - 1) / wcap;
    }
    if (k < 1) k = 1;
    p.kcta = (int)k;
    p.wmax = (int)((p.upr + k - 1) / k);
    p.wlo = p.upr / p.kcta;
    if (rows * k > 0x7fffffffLL) return fail(MAMBA_ERR_ARG, "grid too large");

    p.bc_off = 3 * p.wmax * UB;
    p.quad_off = p.bc_off + bc_bytes;
    p.stage_bytes = stage_of(p.wmax);
    int ns = env_int("MAMBA_SCAN_STAGES", 4);
    if (ns < 2) ns = 2;
    while (ns > 2 && smem_of(p.wmax, ns) > kSmemLimit) --ns;
    p.nstage = ns;
    p.scratch_off = ns * p.stage_bytes;
    p.src_off = p.scratch_off + p.wmax * wscratch;
    p.bar_off = p.src_off;
    p.smem_bytes = smem_of(p.wmax, ns);
    if (p.smem_bytes > kSmemLimit) return fail(MAMBA_ERR_ARG, "tiling needs %d bytes of shared memory", p.smem_bytes);
    return MAMBA_OK;
}

template <typename TIn, int NP, bool TMA, bool AGG, bool SP, bool GATE, bool CKPT = false>
static int launch_fwd_one(const FwdArgs& a, const FwdMaps& maps, unsigned grid, int smem_bytes, cudaStream_t st) {
    static AttrCache attr;
    auto kern = scan_fwd_kernel<TIn, NP, 4, TMA, AGG, SP, GATE, CKPT>;
    int rc = allow_smem(kern, attr);
    if (rc) return rc;
    kern<<<grid, 32 * (a.wmax + 1), smem_bytes, st>>>(a, maps);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "forward scan kernel launch");
    return MAMBA_OK;
}

// Selects the instantiation for the runtime flags (data path, softplus, gate).
template <typename TIn, int NP, bool AGG>
static int launch_fwd(const FwdArgs& a, const FwdMaps& maps, unsigned grid, int smem_bytes, bool tma, bool sp,
                      bool gate, cudaStream_t st) {
    if constexpr (AGG) {  // the aggregate pass reads no z
        if (tma) return sp ? launch_fwd_one<TIn, NP, true, true, true, false>(a, maps, grid, smem_bytes, st)
                           : launch_fwd_one<TIn, NP, true, true, false, false>(a, maps, grid, smem_bytes, st);
        return sp ? launch_fwd_one<TIn, NP, false, true, true, false>(a, maps, grid, smem_bytes, st)
                  : launch_fwd_one<TIn, NP, false, true, false, false>(a, maps, grid, smem_bytes, st);
    } else {
        if constexpr (NP == 16) {
            if (a.ckpt != nullptr) {  // forward pass of training: also the state checkpoints
                if (tma) {
                    if (sp) return gate ? launch_fwd_one<TIn, NP, true, false, true, true, true>(a, maps, grid, smem_bytes, st)
                                        : launch_fwd_one<TIn, NP, true, false, true, false, true>(a, maps, grid, smem_bytes, st);
                    return gate ? launch_fwd_one<TIn, NP, true, false, false, true, true>(a, maps, grid, smem_bytes, st)
                                : launch_fwd_one<TIn, NP, true, false, false, false, true>(a, maps, grid, smem_bytes, st);
                }
                if (sp) return gate ? launch_fwd_one<TIn, NP, false, false, true, true, true>(a, maps, grid, smem_bytes, st)
                                    : launch_fwd_one<TIn, NP, false, false, true, false, true>(a, maps, grid, smem_bytes, st);
                return gate ? launch_fwd_one<TIn, NP, false, false, false, true, true>(a, maps, grid, smem_bytes, st)
                            : launch_fwd_one<TIn, NP, false, false, false, false, true>(a, maps, grid, smem_bytes, st);
            }
        }
        if (tma) {
            if (sp) return gate ? launch_fwd_one<TIn, NP, true, false, true, true>(a, maps, grid, smem_bytes, st)
                                : launch_fwd_one<TIn, NP, true, false, true, false>(a, maps, grid, smem_bytes, st);
            return gate ? launch_fwd_one<TIn, NP, true, false, false, true>(a, maps, grid, smem_bytes, st)
                        : launch_fwd_one<TIn, NP, true, false, false, false>(a, maps, grid, smem_bytes, st);
        }
        if (sp) return gate ? launch_fwd_one<TIn, NP, false, false, true, true>(a, maps, grid, smem_bytes, st)
                            : launch_fwd_one<TIn, NP, false, false, true, false>(a, maps, grid, smem_bytes, st);
        return gate ? launch_fwd_one<TIn, NP, false, false, false, true>(a, maps, grid, smem_bytes, st)
                    : launch_fwd_one<TIn, NP, false, false, false, false>(a, maps, grid, smem_bytes, st);
    }
}

// Plans and launches the scan.  Split time axis: an aggregate launch writes the carries of all
// but the last segment, and the full launch folds the carries of earlier segments into each
// segment's initial state.  An initial state that shares memory with last_state is copied first
// (the last segment writes last_state while CTAs of earlier segments may still read it).
template <typename TIn, int NP>
static int run(const mamba_scan_shape* s, FwdArgs a, bool softplus, bool gate, float2* scratch, size_t cap,
               cudaStream_t st) {
    constexpr int TC = Chunk<TIn>::TC;
    const int esize = (int)sizeof(TIn);
    const long long L = s->seqlen;
    FwdPlan p;
    int rc = plan_warp<TIn, NP>(s, sm_count(), p);
    if (rc) return rc;
    const bool tma = fwd_tma_ok(a, L, esize);
    FwdMaps maps;
    memset(&maps, 0, sizeof maps);
    if (tma && !fwd_maps(maps, a, s, p, esize, TC, kUnitCh, false)) return fail(MAMBA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    fwd_apply_plan(a, p, softplus);
    if (p.nseg == 1) {
        if (a.ck_written) *a.ck_written = (a.ckpt != nullptr && NP == 16) ? 1 : 0;
        const unsigned grid = (unsigned)((long long)s->batch * p.kcta);
        return launch_fwd<TIn, NP, false>(a, maps, grid, p.smem_bytes, tma, softplus, gate, st);
    }
    a.ckpt = nullptr;  // checkpoints are written only with an unsplit time axis
    if (a.ck_written) *a.ck_written = 0;
    const size_t nstate = (size_t)s->batch * s->dim * s->dstate;
    const size_t bytes = (size_t)(p.nseg - 1) * nstate * sizeof(float2);
    const bool copy_h0 = a.h0 != nullptr && overlaps(a.h0, nstate * 4, a.last_state, nstate * 4);
    bool owned = false;
    rc = carries_get(bytes, copy_h0 ? nstate * sizeof(float) : 0, scratch, cap, p.nseg, st, &a.agg, &owned);
    if (rc) return rc;
    if (copy_h0) {
        float* hcopy = reinterpret_cast<float*>(reinterpret_cast<char*>(a.agg) + bytes);
        cudaError_t e = cudaMemcpyAsync(hcopy, a.h0, nstate * sizeof(float), cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) rc = cuda_fail(e, "cudaMemcpyAsync (initial state)");
        a.h0 = hcopy;
    }
    if (rc == MAMBA_OK) {
        const unsigned g1 = (unsigned)((long long)s->batch * (p.nseg - 1) * p.kcta);
        rc = launch_fwd<TIn, NP, true>(a, maps, g1, p.smem_bytes, tma, softplus, gate, st);
    }
    if (rc == MAMBA_OK) {
        const unsigned grid = (unsigned)((long long)s->batch * p.nseg * p.kcta);
        rc = launch_fwd<TIn, NP, false>(a, maps, grid, p.smem_bytes, tma, softplus, gate, st);
    }
    if (owned) {
        cudaError_t e = cudaFreeAsync(a.agg, st);
        if (e != cudaSuccess && rc == MAMBA_OK) rc = cuda_fail(e, "cudaFreeAsync (segment carries)");
    }
    return rc;
}

template <typename TIn>
int fwd_warp_run_t(const mamba_scan_shape* s, const FwdArgs& a, bool softplus, bool gate, float2* scratch,
                   size_t cap, cudaStream_t st) {
    if (s->dstate <= 16) return run<TIn, 16>(s, a, softplus, gate, scratch, cap, st);
    if (s->dstate <= 32) return run<TIn, 32>(s, a, softplus, gate, scratch, cap, st);
    return run<TIn, 64>(s, a, softplus, gate, scratch, cap, st);
}

template <typename TIn>
int fwd_warp_status_t(bool clear) {
    return read_status(g_status, clear);
}

}  // namespace mscan
