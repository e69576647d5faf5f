// Forward scan, channel-per-lane kernel (N <= 16): planner, TMA descriptors and launches of
// scan_fwd_cl_kernel, and for a split time axis the second launch, scan_fix_kernel.  Included by
// one translation unit per input type (fwd_lane_f32.cu, fwd_lane_bf16.cu), which instantiates
// fwd_lane_run_t and fwd_lane_status_t for that type.
#pragma once
#include <cstring>

#include "host.cuh"
#include "fwd_common.cuh"
#include "scan_fwd_cl.cuh"
#include "scan_fix.cuh"

namespace mscan {


// Segments and CTAs for the channel-per-lane kernel.  A CTA runs one (segment, batch row) range of
// at most wcap units, every warp on its own SM sub-partition, so a launch takes about
// waves * segment length; a split adds the fix-up launch, which walks each later segment until
// the carried-in state has decayed (modelled as kFixSteps steps, at most the segment).  The
// segment count minimises that estimate.
constexpr long long kFixSteps = 4096;

template <typename TIn, int NP>
static int plan_cl(const mamba_scan_shape* s, int nsm, FwdPlan& p) {
    constexpr int TC = Chunk<TIn>::TC;
    constexpr int CPW = cl::Lanes::CPW;
    constexpr int TILE = CPW * cl::kRowBytes;
    constexpr int YTILE = cl::Lanes::YTILE;
    const long long L = s->seqlen;
    p.upr = (s->dim + CPW - 1) / CPW;
    auto stage_of = [&](int w) { return round_up(3 * w * TILE + 2 * NP * cl::kRowBytes + TC * cl::Quads<NP>::PITCH, 1024); };
    auto smem_of = [&](int w, int ns) { return ns * stage_of(w) + w * 2 * YTILE + (3 * ns + 1) * 8 + 1024; };
    int wcap = cl::Lanes::MAX_WARPS;
    while (wcap > 1 && smem_of(wcap, 2) > kSmemLimit) --wcap;
    const int wforce = env_int("MAMBA_SCAN_WMAX", 0);
    if (wforce > wcap) return fail(MAMBA_ERR_ARG, "MAMBA_SCAN_WMAX above %d", wcap);
    const int wlim = wforce > 0 ? wforce : wcap;
    auto kcta_of = [&](long long rows) {
        long long k = wforce > 0 ? (p.upr + wforce - 1) / wforce : (rows >= nsm ? 1 : nsm / rows);
        if (k > p.upr) k = p.upr;
        const long long kmin = (p.upr + wlim - 1) / wlim;
        if (k < kmin) k = kmin;
        return k < 1 ? 1LL : k;
    };
    long long maxseg = L / (8LL * TC);
    if (maxseg < 1) maxseg = 1;
    if (maxseg > 4096) maxseg = 4096;
    // the time axis is split only when the units fill at most half of the 4 * nsm sub-partitions,
    // into at most ceil(4 * nsm / units) + 1 segments (a bound callers of the allocation-free entry
    // point can compute)
    const long long units = (long long)s->batch * p.upr, slots = 4LL * nsm;
    const long long smax = units * 2 <= slots ? (slots + units - 1) / units + 1 : 1;
    long long best = 1;
    const long long want = env_int("MAMBA_SCAN_NSEG", 0);
    if (want > 0) {
        best = want < maxseg ? want : maxseg;
    } else {
        double best_cost = 0.0;
        for (long long ns = 1; ns <= maxseg && ns <= smax; ++ns) {
            const long long seg = (L + ns - 1) / ns;
            const long long segr = (seg + TC - 1) / TC * TC;
            const long long nseg = (L + segr - 1) / segr;
            if (nseg != ns) continue;
            const long long k = kcta_of((long long)s->batch * ns);
            const long long waves = ((long long)s->batch * ns * k + nsm - 1) / nsm;
            double cost = (double)waves * segr;
            if (ns > 1) cost += (double)(segr < kFixSteps ? segr : kFixSteps);
            if (ns == 1 || cost < best_cost * 0.98) {
                best_cost = cost;
                best = ns;
            }
        }
    }
    p.nseg = 1;
    p.seg_len = L;
    if (best > 1) {
        long long seg = (L + best - 1) / best;
        seg = (seg + TC - 1) / TC * TC;
        p.seg_len = seg;
        p.nseg = (int)((L + seg - 1) / seg);
    }
    const long long rows = (long long)s->batch * p.nseg;
    const long long k = kcta_of(rows);
    p.kcta = (int)k;
    p.wmax = (int)((p.upr + k - 1) / k);
    p.wlo = p.upr / p.kcta;
    if (rows * k > 0x7fffffffLL) return fail(MAMBA_ERR_ARG, "grid too large");
    p.bc_off = 3 * p.wmax * TILE;
    p.quad_off = p.bc_off + 2 * NP * cl::kRowBytes;
    p.stage_bytes = stage_of(p.wmax);
    int ns = env_int("MAMBA_SCAN_STAGES", 4);
    if (ns < 2) ns = 2;
    while (ns > 2 && smem_of(p.wmax, ns) > kSmemLimit) --ns;
    p.nstage = ns;
    p.scratch_off = ns * p.stage_bytes;  // y staging tiles
    p.src_off = p.scratch_off + p.wmax * 2 * YTILE;
    p.bar_off = p.src_off;
    p.smem_bytes = smem_of(p.wmax, ns);
    if (p.smem_bytes > kSmemLimit) return fail(MAMBA_ERR_ARG, "tiling needs %d bytes of shared memory", p.smem_bytes);
    return MAMBA_OK;
}

static int launch_kernel(void (*kern)(const FwdArgs, const FwdMaps), AttrCache& attr, const FwdArgs& a,
                         const FwdMaps& maps, unsigned grid, int smem_bytes, cudaStream_t st) {
    int rc = allow_smem(kern, attr);
    if (rc) return rc;
    kern<<<grid, 32 * (a.wmax + 1), smem_bytes, st>>>(a, maps);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "forward scan kernel launch");
    return MAMBA_OK;
}

// Channel-per-lane kernel: data path and discretisation / convolution mode are template
// parameters; softplus and the gate are runtime flags.
template <typename TIn, int NP, bool TMA, bool LOCAL, int MODE>
static int launch_cl_one(const FwdArgs& a, const FwdMaps& maps, unsigned grid, int smem_bytes, cudaStream_t st) {
    static AttrCache attr;
    return launch_kernel(scan_fwd_cl_kernel<TIn, NP, TMA, LOCAL, MODE>, attr, a, maps, grid, smem_bytes, st);
}

template <typename TIn, int NP, bool LOCAL>
static int launch_cl(const FwdArgs& a, const FwdMaps& maps, unsigned grid, int smem_bytes, bool tma, int mode,
                     cudaStream_t st) {
    switch (mode) {
        case 0: return tma ? launch_cl_one<TIn, NP, true, LOCAL, 0>(a, maps, grid, smem_bytes, st)
                           : launch_cl_one<TIn, NP, false, LOCAL, 0>(a, maps, grid, smem_bytes, st);
        case 1: return tma ? launch_cl_one<TIn, NP, true, LOCAL, 1>(a, maps, grid, smem_bytes, st)
                           : launch_cl_one<TIn, NP, false, LOCAL, 1>(a, maps, grid, smem_bytes, st);
        case 2: return tma ? launch_cl_one<TIn, NP, true, LOCAL, 2>(a, maps, grid, smem_bytes, st)
                           : launch_cl_one<TIn, NP, false, LOCAL, 2>(a, maps, grid, smem_bytes, st);
        case 3: return tma ? launch_cl_one<TIn, NP, true, LOCAL, 3>(a, maps, grid, smem_bytes, st)
                           : launch_cl_one<TIn, NP, false, LOCAL, 3>(a, maps, grid, smem_bytes, st);
        default:
            if constexpr (!LOCAL) {  // modes 4, 5: forward pass of training (checkpoints), no convolution
                if (mode == 4)
                    return tma ? launch_cl_one<TIn, NP, true, false, 4>(a, maps, grid, smem_bytes, st)
                               : launch_cl_one<TIn, NP, false, false, 4>(a, maps, grid, smem_bytes, st);
                if (mode == 5)
                    return tma ? launch_cl_one<TIn, NP, true, false, 5>(a, maps, grid, smem_bytes, st)
                               : launch_cl_one<TIn, NP, false, false, 5>(a, maps, grid, smem_bytes, st);
            }
            return fail(MAMBA_ERR_ARG, "internal: forward mode %d", mode);
    }
}

// The second launch of a split time axis (channel-per-lane kernel): one warp per (segment > 0,
// batch row, 32 channels).
template <typename TIn, int NP>
static int launch_fix(const FwdArgs& a, const FixMaps& maps, bool tma, cudaStream_t st) {
    static AttrCache attr[2];
    auto kern = tma ? scan_fix_kernel<TIn, NP, true> : scan_fix_kernel<TIn, NP, false>;
    int rc = allow_smem(kern, attr[tma ? 1 : 0]);
    if (rc) return rc;
    const long long items = (long long)(a.nseg - 1) * a.batch * a.upr;
    if (items > 0x7fffffffLL) return fail(MAMBA_ERR_ARG, "grid too large");
    kern<<<(unsigned)items, 32, fix::Layout<NP>::SMEM, st>>>(a, maps);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "split-scan fix-up kernel launch");
    return MAMBA_OK;
}

// Plans and launches the scan.  Split time axis: every segment runs at once (segment 0 from the
// initial state, the others from zero) and writes its carry; scan_fix_kernel then folds the
// carries and adds the carried-in part to the later segments' outputs.  The first launch reads
// the initial state and the second writes last_state, so the two may be one buffer.
template <typename TIn, int NP>
static int run(const mamba_scan_shape* s, FwdArgs a, bool softplus, float2* scratch, size_t cap, cudaStream_t st) {
    constexpr int TC = Chunk<TIn>::TC;
    constexpr int CPW = cl::Lanes::CPW;
    const int esize = (int)sizeof(TIn);
    const long long L = s->seqlen;
    FwdPlan p;
    int rc = plan_cl<TIn, NP>(s, sm_count(), p);
    if (rc) return rc;
    const bool tma = fwd_tma_ok(a, L, esize);
    FwdMaps maps;
    memset(&maps, 0, sizeof maps);
    if (tma && !fwd_maps(maps, a, s, p, esize, TC, CPW, true)) return fail(MAMBA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    fwd_apply_plan(a, p, softplus);
    // test knob (read here on the host): a 1 ms limit for waits on other warps, and consumer
    // warps that wait on a barrier nothing arrives on
    if (env_int("MAMBA_SCAN_TEST_STALL", 0) != 0) {
        a.wait_ns = 1000000ull;
        a.test_stall = 1;
    }
    // checkpoints for the backward pass: only with an unsplit time axis and no fused convolution
    const bool ckpt = a.ckpt != nullptr && p.nseg == 1 && a.conv_w == nullptr;
    if (a.ck_written) *a.ck_written = ckpt ? 1 : 0;
    if (!ckpt) a.ckpt = nullptr;
    const int mode = (a.zoh ? 1 : 0) | (a.conv_w != nullptr ? 2 : 0) | (ckpt ? 4 : 0);
    if (p.nseg == 1) {
        const unsigned grid = (unsigned)((long long)s->batch * p.kcta);
        return launch_cl<TIn, NP, false>(a, maps, grid, p.smem_bytes, tma, mode, st);
    }
    const size_t nstate = (size_t)s->batch * s->dim * s->dstate;
    bool owned = false;
    rc = carries_get((size_t)p.nseg * nstate * sizeof(float2), 0, scratch, cap, p.nseg, st, &a.agg, &owned);
    if (rc) return rc;
    const unsigned grid = (unsigned)((long long)s->batch * p.nseg * p.kcta);
    rc = launch_cl<TIn, NP, true>(a, maps, grid, p.smem_bytes, tma, mode, st);
    if (rc == MAMBA_OK) {
        FixMaps fm;
        memset(&fm, 0, sizeof fm);
        if (tma) {
            const bool ok = encode_3d(&fm.d, a.delta, esize, L, s->dim, s->batch, TC, 32) &&
                            encode_3d(&fm.z, a.z ? a.z : a.delta, esize, L, s->dim, s->batch, TC, 32);
            if (!ok) rc = fail(MAMBA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
            fm.y = maps.y;
            fm.C = maps.C;
        }
        if (rc == MAMBA_OK) rc = launch_fix<TIn, NP>(a, fm, tma, st);
    }
    if (owned) {
        cudaError_t e = cudaFreeAsync(a.agg, st);
        if (e != cudaSuccess && rc == MAMBA_OK) rc = cuda_fail(e, "cudaFreeAsync (segment carries)");
    }
    return rc;
}

template <typename TIn>
int fwd_lane_run_t(const mamba_scan_shape* s, const FwdArgs& a, bool softplus, float2* scratch, size_t cap,
                   cudaStream_t st) {
    if (s->dstate > 16) return fail(MAMBA_ERR_ARG, "the channel-per-lane kernel takes N <= 16");
    if (s->dstate <= 8) return run<TIn, 8>(s, a, softplus, scratch, cap, st);
    return run<TIn, 16>(s, a, softplus, scratch, cap, st);
}

template <typename TIn>
int fwd_lane_status_t(bool clear) {
    return read_status(g_status, clear);
}

}  // namespace mscan
