// Host-side plan format and set-up shared by the two forward kernels' launch code (fwd_lane.cu,
// fwd_warp.cu).
//
// Both kernels take the same plan: work units (a warp's channels of one batch row) spread over
// CTAs of about one per SM, an optional split of the time axis into segments, and an NS-deep ring
// of shared-memory stages fed by TMA.
//  * scan_fwd_cl_kernel (channel per lane, N <= 16): work unit = 32 channels;
//  * scan_fwd_kernel (4 lanes per channel, any N <= 64): work unit = 8 channels.
#pragma once
#include <cstring>

#include "host.cuh"
#include "scan_fwd.cuh"

namespace mscan {

struct FwdPlan {
    int nseg;
    long long seg_len;
    int upr, kcta, wmax, wlo, nstage;
    int stage_bytes, bc_off, quad_off, scratch_off, src_off, bar_off, smem_bytes;
};

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// TMA needs 16-byte aligned rows and bases (and a driver entry point); MAMBA_SCAN_NO_TMA=1 forces
// the plain-load path (tests).
inline bool fwd_tma_ok(const FwdArgs& a, long long L, int esize) {
    return encode_fn() != nullptr && (L * esize) % 16 == 0 && aligned16(a.u) && aligned16(a.delta) &&
           aligned16(a.B) && aligned16(a.C) && aligned16(a.y) && (a.z == nullptr || aligned16(a.z)) &&
           L < (1LL << 31) && getenv("MAMBA_SCAN_NO_TMA") == nullptr;
}

// Maps of u, delta, z (box heights of wlo and wlo + 1 units of cpw channels), B, C (box [N, TC])
// and, when with_y, y (box [cpw, TC]).
inline bool fwd_maps(FwdMaps& maps, const FwdArgs& a, const mamba_scan_shape* s, const FwdPlan& p, int esize,
                     int tc, int cpw, bool with_y) {
    memset(&maps, 0, sizeof maps);
    const long long L = s->seqlen;
    const void* zb = a.z ? a.z : a.u;
    const void* src[3] = {a.u, a.delta, zb};
    CUtensorMap* dst[3] = {maps.u, maps.d, maps.z};
    bool ok = true;
    for (int m = 0; m < 3 && ok; ++m)
        for (int w = 0; w < 2 && ok; ++w) {
            const int rowsbox = cpw * (w == 0 ? (p.wlo > 0 ? p.wlo : 1) : p.wlo + 1);
            ok = encode_3d(&dst[m][w], src[m], esize, L, s->dim, s->batch, tc, rowsbox > 256 ? 256 : rowsbox);
        }
    ok = ok && encode_3d(&maps.B, a.B, esize, L, s->dstate, s->batch, tc, s->dstate) &&
         encode_3d(&maps.C, a.C, esize, L, s->dstate, s->batch, tc, s->dstate);
    if (with_y) ok = ok && encode_3d(&maps.y, a.y, esize, L, s->dim, s->batch, tc, cpw);
    return ok;
}

// Copies the plan into the kernel arguments; full wait limits, no test knob.
inline void fwd_apply_plan(FwdArgs& a, const FwdPlan& p, bool softplus) {
    a.nseg = p.nseg;
    a.seg_len = p.seg_len;
    a.upr = p.upr;
    a.kcta = p.kcta;
    a.wmax = p.wmax;
    a.wlo = p.wlo;
    a.nstage = p.nstage;
    a.stage_bytes = p.stage_bytes;
    a.bc_off = p.bc_off;
    a.quad_off = p.quad_off;
    a.scratch_off = p.scratch_off;
    a.src_off = p.src_off;
    a.bar_off = p.bar_off;
    a.agg = nullptr;
    a.wait_ns = kWaitLimitNs;
    a.test_stall = 0;
    a.softplus = softplus ? 1 : 0;
}

// Segment carries of `bytes` bytes (plus `extra` bytes after them) in the caller's fixed scratch,
// or from cudaMallocAsync on st (then *owned is set and the caller frees them on st).
inline int carries_get(size_t bytes, size_t extra, float2* scratch, size_t cap, int nseg, cudaStream_t st,
                       float2** out, bool* owned) {
    *owned = false;
    if (scratch != nullptr) {
        if (extra != 0) return fail(MAMBA_ERR_ARG, "internal: initial state with fixed scratch");
        if (bytes > cap)
            return fail(MAMBA_ERR_ARG, "this shape splits the sequence into %d segments whose carries need %zu bytes "
                        "of scratch; the fixed scratch holds %zu bytes", nseg, bytes, cap);
        *out = scratch;
        return MAMBA_OK;
    }
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(out), bytes + extra, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync (segment carries)");
    *owned = true;
    return MAMBA_OK;
}

}  // namespace mscan
