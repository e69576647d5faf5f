// Host side of libmambascan.so: argument checks, launch selection, TMA descriptors and the C ABI
// declared in include/mamba_scan.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "mamba_scan.h"
#include "common.cuh"
#include "scan_fwd.cuh"
#include "scan_fwd_cl.cuh"
#include "scan_fix.cuh"
#include "scan_bwd.cuh"
#include "state_step.cuh"

namespace mscan {

static thread_local std::string t_err;
static std::atomic<long long> g_launches{0};

static int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_err = buf;
    return code;
}

static int cuda_fail(cudaError_t e, const char* what) {
    return fail(MAMBA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------------------- TMA descriptors
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D map over a dense [d2][d1][d0] tensor (d0 contiguous), box [b1 rows x b0 cols], 128-byte
// swizzle (b0 * esize must be 128).
static bool encode_3d(CUtensorMap* m, const void* base, int esize, long long d0, long long d1, long long d2,
                      int b0, int b1) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)(d0 * esize), (cuuint64_t)(d0 * d1 * esize)};
    cuuint32_t box[3] = {(cuuint32_t)b0, (cuuint32_t)b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int env_int(const char* name, int dflt) {
    const char* v = getenv(name);
    return (v && *v) ? atoi(v) : dflt;
}

static bool overlaps(const void* a, size_t na, const void* b, size_t nb);

// ---------------------------------------------------------------------------- forward plan
constexpr int kSmemLimit = 227 * 1024;

struct FwdPlan {
    int nseg;
    long long seg_len;
    int upr, kcta, wmax, wlo, nstage;
    int stage_bytes, bc_off, quad_off, scratch_off, src_off, bar_off, smem_bytes;
};

// Two forward kernels share the plan format and the split of the time axis:
//  * scan_fwd_cl_kernel (channel per lane, N <= 16): work unit = 32 channels of one batch row,
//    one consumer warp each, at most cl::kMaxWarps per CTA (one per SM sub-partition);
//  * scan_fwd_kernel (4 lanes per channel, any N <= 64, also the exact hold and the fused
//    convolution): work unit = 8 channels of one batch row.
enum class FwdKernel { kChannelLane, kWarp };

static int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Segments and CTAs for the channel-per-lane kernel.  A CTA runs one (segment, batch row) range of
// at most wcap units, every warp on its own SM sub-partition, so a launch takes about
// waves * segment length; a split adds the fix-up launch, which walks each later segment until
// the carried-in state has decayed (modelled as kFixSteps steps, at most the segment).  The
// segment count minimises that estimate.
constexpr long long kFixSteps = 4096;

template <typename TIn, int NP, int LPC>
static int plan_cl(const mamba_scan_shape* s, int nsm, FwdPlan& p) {
    constexpr int TC = Chunk<TIn>::TC;
    constexpr int CPW = cl::Lanes<LPC>::CPW;
    constexpr int TILE = CPW * cl::kRowBytes;
    constexpr int YTILE = cl::Lanes<LPC>::YTILE;
    const long long L = s->seqlen;
    p.upr = (s->dim + CPW - 1) / CPW;
    auto stage_of = [&](int w) { return round_up(3 * w * TILE + 2 * NP * cl::kRowBytes + TC * cl::Quads<NP>::PITCH, 1024); };
    auto smem_of = [&](int w, int ns) { return ns * stage_of(w) + w * 2 * YTILE + (3 * ns + 1) * 8 + 1024; };
    int wcap = cl::Lanes<LPC>::MAX_WARPS;
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

// Raises a kernel's dynamic shared memory limit once per CUDA context (the attribute belongs to
// the function in one context; setting it on every call costs tens of microseconds of host time).
// Unique id of the CUDA context current on this thread (0 if none is current or the driver
// entry points are missing).  Ids are never reused within a process, so an id stays tied to one
// context even after cudaDeviceReset replaces the primary context at the same address.
static unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

struct AttrCache {
    std::atomic<unsigned long long> ctx[8] = {};
};

template <typename K>
static int allow_smem(K kern, AttrCache& cache) {
    const unsigned long long id = current_context_id();
    if (id != 0)
        for (auto& c : cache.ctx)
            if (c.load(std::memory_order_acquire) == id) return MAMBA_OK;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    if (id != 0) cache.ctx[id % 8].store(id, std::memory_order_release);
    return MAMBA_OK;
}

static int launch_kernel(void (*kern)(const FwdArgs, const FwdMaps), AttrCache& attr, const FwdArgs& a,
                         const FwdMaps& maps, unsigned grid, int smem_bytes, cudaStream_t st) {
    int rc = allow_smem(kern, attr);
    if (rc) return rc;
    kern<<<grid, 32 * (a.wmax + 1), smem_bytes, st>>>(a, maps);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "forward scan kernel launch");
    return MAMBA_OK;
}

// Channel-per-lane kernel: data path and discretisation / convolution mode are template
// parameters; softplus and the gate are runtime flags.
template <typename TIn, int NP, int LPC, bool TMA, bool LOCAL, int MODE>
static int launch_cl_one(const FwdArgs& a, const FwdMaps& maps, unsigned grid, int smem_bytes, cudaStream_t st) {
    static AttrCache attr;
    return launch_kernel(scan_fwd_cl_kernel<TIn, NP, LPC, TMA, LOCAL, MODE>, attr, a, maps, grid, smem_bytes, st);
}

template <typename TIn, int NP, int LPC, bool LOCAL>
static int launch_cl(const FwdArgs& a, const FwdMaps& maps, unsigned grid, int smem_bytes, bool tma, int mode,
                     cudaStream_t st) {
    switch (mode) {
        case 0: return tma ? launch_cl_one<TIn, NP, LPC, true, LOCAL, 0>(a, maps, grid, smem_bytes, st)
                           : launch_cl_one<TIn, NP, LPC, false, LOCAL, 0>(a, maps, grid, smem_bytes, st);
        case 1: return tma ? launch_cl_one<TIn, NP, LPC, true, LOCAL, 1>(a, maps, grid, smem_bytes, st)
                           : launch_cl_one<TIn, NP, LPC, false, LOCAL, 1>(a, maps, grid, smem_bytes, st);
        case 2: return tma ? launch_cl_one<TIn, NP, LPC, true, LOCAL, 2>(a, maps, grid, smem_bytes, st)
                           : launch_cl_one<TIn, NP, LPC, false, LOCAL, 2>(a, maps, grid, smem_bytes, st);
        default: return tma ? launch_cl_one<TIn, NP, LPC, true, LOCAL, 3>(a, maps, grid, smem_bytes, st)
                            : launch_cl_one<TIn, NP, LPC, false, LOCAL, 3>(a, maps, grid, smem_bytes, st);
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
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "split-scan fix-up kernel launch");
    return MAMBA_OK;
}

template <FwdKernel KIND, typename TIn, int NP, bool TMA, bool AGG, bool SP, bool GATE>
static int launch_fwd_one(const FwdArgs& a, const FwdMaps& maps, unsigned grid, int smem_bytes, cudaStream_t st) {
    static AttrCache attr;
    auto kern = scan_fwd_kernel<TIn, NP, 4, TMA, AGG, SP, GATE>;
    int rc = allow_smem(kern, attr);
    if (rc) return rc;
    kern<<<grid, 32 * (a.wmax + 1), smem_bytes, st>>>(a, maps);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "forward scan kernel launch");
    return MAMBA_OK;
}

// Selects the instantiation for the runtime flags (data path, softplus, gate).
template <FwdKernel KIND, typename TIn, int NP, bool AGG>
static int launch_fwd(const FwdArgs& a, const FwdMaps& maps, unsigned grid, int smem_bytes, bool tma, bool sp,
                      bool gate, cudaStream_t st) {
    if constexpr (AGG) {  // the aggregate pass reads no z
        if (tma) return sp ? launch_fwd_one<KIND, TIn, NP, true, true, true, false>(a, maps, grid, smem_bytes, st)
                           : launch_fwd_one<KIND, TIn, NP, true, true, false, false>(a, maps, grid, smem_bytes, st);
        return sp ? launch_fwd_one<KIND, TIn, NP, false, true, true, false>(a, maps, grid, smem_bytes, st)
                  : launch_fwd_one<KIND, TIn, NP, false, true, false, false>(a, maps, grid, smem_bytes, st);
    } else {
        if (tma) {
            if (sp) return gate ? launch_fwd_one<KIND, TIn, NP, true, false, true, true>(a, maps, grid, smem_bytes, st)
                                : launch_fwd_one<KIND, TIn, NP, true, false, true, false>(a, maps, grid, smem_bytes, st);
            return gate ? launch_fwd_one<KIND, TIn, NP, true, false, false, true>(a, maps, grid, smem_bytes, st)
                        : launch_fwd_one<KIND, TIn, NP, true, false, false, false>(a, maps, grid, smem_bytes, st);
        }
        if (sp) return gate ? launch_fwd_one<KIND, TIn, NP, false, false, true, true>(a, maps, grid, smem_bytes, st)
                            : launch_fwd_one<KIND, TIn, NP, false, false, true, false>(a, maps, grid, smem_bytes, st);
        return gate ? launch_fwd_one<KIND, TIn, NP, false, false, false, true>(a, maps, grid, smem_bytes, st)
                    : launch_fwd_one<KIND, TIn, NP, false, false, false, false>(a, maps, grid, smem_bytes, st);
    }
}

// `scratch`/`scratch_cap`: when scratch is non-NULL the segment carries live there (no allocation);
// otherwise they come from cudaMallocAsync on `st`.
template <FwdKernel KIND, typename TIn, int NP, int LPC = 1>
static int fwd_run(const mamba_scan_shape* s, FwdArgs a, bool softplus, bool gate, float2* scratch,
                   size_t scratch_cap, cudaStream_t st) {
    constexpr int TC = Chunk<TIn>::TC;
    constexpr int CPW = KIND == FwdKernel::kChannelLane ? cl::Lanes<LPC>::CPW : kUnitCh;  // channels per work unit
    const int esize = (int)sizeof(TIn);
    const long long L = s->seqlen;

    int dev = 0, nsm = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);

    FwdPlan p;
    int rc;
    if constexpr (KIND == FwdKernel::kChannelLane)
        rc = plan_cl<TIn, NP, LPC>(s, nsm, p);
    else
        rc = plan_warp<TIn, NP>(s, nsm, p);
    if (rc) return rc;

    const bool tma_ok = encode_fn() != nullptr && (L * esize) % 16 == 0 && aligned16(a.u) && aligned16(a.delta) &&
                        aligned16(a.B) && aligned16(a.C) && aligned16(a.y) && (a.z == nullptr || aligned16(a.z)) &&
                        L < (1LL << 31) && getenv("MAMBA_SCAN_NO_TMA") == nullptr;
    FwdMaps maps;
    memset(&maps, 0, sizeof maps);
    if (tma_ok) {
        const void* zb = a.z ? a.z : a.u;
        const void* src[3] = {a.u, a.delta, zb};
        CUtensorMap* dst[3] = {maps.u, maps.d, maps.z};
        bool ok = true;
        for (int m = 0; m < 3 && ok; ++m)
            for (int w = 0; w < 2 && ok; ++w) {
                const int rowsbox = CPW * (w == 0 ? (p.wlo > 0 ? p.wlo : 1) : p.wlo + 1);
                ok = encode_3d(&dst[m][w], src[m], esize, L, s->dim, s->batch, TC, rowsbox > 256 ? 256 : rowsbox);
            }
        ok = ok && encode_3d(&maps.B, a.B, esize, L, s->dstate, s->batch, TC, s->dstate) &&
             encode_3d(&maps.C, a.C, esize, L, s->dstate, s->batch, TC, s->dstate);
        if (KIND != FwdKernel::kWarp) ok = ok && encode_3d(&maps.y, a.y, esize, L, s->dim, s->batch, TC, CPW);
        if (!ok) return fail(MAMBA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    }

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
    // bounded waits: the full limit, or (test knob, read here on the host) a 1 ms limit for waits
    // on other warps together with consumer warps that wait on a barrier nothing arrives on
    a.wait_ns = kWaitLimitNs;
    a.test_stall = 0;
    a.softplus = softplus ? 1 : 0;
    const int mode = (a.zoh ? 1 : 0) | (a.conv_w != nullptr ? 2 : 0);
    if (KIND != FwdKernel::kWarp && env_int("MAMBA_SCAN_TEST_STALL", 0) != 0) {
        a.wait_ns = 1000000ull;
        a.test_stall = 1;
    }

    // Split time axis.  Channel-per-lane kernel: every segment runs at once (segment 0 from the
    // initial state, the others from zero) and writes its carry; scan_fix_kernel then folds the
    // carries and adds the carried-in part to the later segments' outputs.  scan_fwd_kernel: an
    // aggregate launch writes the carries of all but the last segment, and the full launch folds
    // them into each segment's initial state.
    constexpr bool kLocal = KIND == FwdKernel::kChannelLane;
    bool owned = false;
    if (p.nseg > 1) {
        const size_t nstate = (size_t)s->batch * s->dim * s->dstate;
        const size_t bytes = (size_t)(kLocal ? p.nseg : p.nseg - 1) * nstate * sizeof(float2);
        // scan_fwd_kernel: an initial state that shares memory with last_state is copied first
        // (the last segment writes last_state while CTAs of earlier segments may still be reading
        // the initial state).  The channel-per-lane split reads the initial state in its first
        // launch and writes last_state in its second.
        const bool copy_h0 = !kLocal && a.h0 != nullptr && overlaps(a.h0, nstate * 4, a.last_state, nstate * 4);
        const size_t total = bytes + (copy_h0 ? nstate * sizeof(float) : 0);
        if (copy_h0 && scratch != nullptr) return fail(MAMBA_ERR_ARG, "internal: initial state with fixed scratch");
        if (scratch != nullptr) {
            if (bytes > scratch_cap)
                return fail(MAMBA_ERR_ARG, "this shape splits the sequence into %d segments whose carries need %zu bytes "
                            "of scratch; the fixed scratch holds %zu bytes", p.nseg, bytes, scratch_cap);
            a.agg = scratch;
        } else {
            cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&a.agg), total, st);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync (segment carries)");
            owned = true;
            if (copy_h0) {
                float* hcopy = reinterpret_cast<float*>(reinterpret_cast<char*>(a.agg) + bytes);
                e = cudaMemcpyAsync(hcopy, a.h0, nstate * sizeof(float), cudaMemcpyDeviceToDevice, st);
                if (e != cudaSuccess) {
                    cudaFreeAsync(a.agg, st);
                    return cuda_fail(e, "cudaMemcpyAsync (initial state)");
                }
                a.h0 = hcopy;
            }
        }
        const unsigned grid = (unsigned)((long long)s->batch * p.nseg * p.kcta);
        if constexpr (kLocal) {
            rc = launch_cl<TIn, NP, LPC, true>(a, maps, grid, p.smem_bytes, tma_ok, mode, st);
            if (rc == MAMBA_OK) {
                FixMaps fm;
                memset(&fm, 0, sizeof fm);
                if (tma_ok) {
                    bool ok = encode_3d(&fm.d, a.delta, esize, L, s->dim, s->batch, TC, 32) &&
                              encode_3d(&fm.z, a.z ? a.z : a.delta, esize, L, s->dim, s->batch, TC, 32);
                    if (!ok) rc = fail(MAMBA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
                    fm.y = maps.y;
                    fm.C = maps.C;
                }
                if (rc == MAMBA_OK) rc = launch_fix<TIn, NP>(a, fm, tma_ok, st);
            }
        } else {
            const unsigned g1 = (unsigned)((long long)s->batch * (p.nseg - 1) * p.kcta);
            rc = launch_fwd<KIND, TIn, NP, true>(a, maps, g1, p.smem_bytes, tma_ok, softplus, gate, st);
            if (rc == MAMBA_OK)
                rc = launch_fwd<KIND, TIn, NP, false>(a, maps, grid, p.smem_bytes, tma_ok, softplus, gate, st);
        }
    } else {
        const unsigned grid = (unsigned)((long long)s->batch * p.kcta);
        if constexpr (kLocal)
            rc = launch_cl<TIn, NP, LPC, false>(a, maps, grid, p.smem_bytes, tma_ok, mode, st);
        else
            rc = launch_fwd<KIND, TIn, NP, false>(a, maps, grid, p.smem_bytes, tma_ok, softplus, gate, st);
    }
    if (owned) {
        cudaError_t e = cudaFreeAsync(a.agg, st);
        if (e != cudaSuccess && rc == MAMBA_OK) rc = cuda_fail(e, "cudaFreeAsync (segment carries)");
    }
    return rc;
}

// Kernel choice for N <= 16.  Both kernels are limited by one warp's arithmetic per SM
// sub-partition, so the one whose work units fill the 4 * nsm sub-partitions better in its last
// wave wins; per filled sub-partition the channel-per-lane kernel is about 7 % faster (measured on
// the Mamba-130M and 1.4B layer shapes).  Shapes with too few channels for half the
// sub-partitions split the time axis, which the channel-per-lane kernel plans to fill the GPU.
static bool prefer_lane_kernel(const mamba_scan_shape* s, int nsm) {
    const long long slots = 4LL * nsm;
    const long long lane_units = (long long)s->batch * ((s->dim + 31) / 32);
    if (lane_units * 2 <= slots) return true;
    const long long warp_units = (long long)s->batch * ((s->dim + kUnitCh - 1) / kUnitCh);
    auto fill = [&](long long u) { return (double)u / (double)(slots * ((u + slots - 1) / slots)); };
    return 1.07 * fill(lane_units) >= fill(warp_units);
}

// The channel-per-lane kernel for N <= 16 where it fills the GPU (prefer_lane_kernel),
// scan_fwd_kernel otherwise.  MAMBA_SCAN_KERNEL=warp or =lane forces one (tests, benchmarks).
template <typename TIn, int NP>
static int fwd_dispatch(const mamba_scan_shape* s, const FwdArgs& a, bool softplus, bool gate, float2* scratch,
                        size_t scratch_cap, cudaStream_t st) {
    const char* force = getenv("MAMBA_SCAN_KERNEL");
    const bool lane_ok = NP <= 16;
    bool use_lane = false;
    if (lane_ok) {
        int dev = 0, nsm = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        use_lane = prefer_lane_kernel(s, nsm);
    }
    if (force && strcmp(force, "warp") == 0) use_lane = false;
    if (force && strcmp(force, "lane") == 0) {
        if (!lane_ok) return fail(MAMBA_ERR_ARG, "MAMBA_SCAN_KERNEL=lane: the channel-per-lane kernel takes N <= 16");
        use_lane = true;
    }
    if constexpr (NP <= 16) {
        if (use_lane) {
            if (s->dstate <= 8) return fwd_run<FwdKernel::kChannelLane, TIn, 8, 1>(s, a, softplus, gate, scratch, scratch_cap, st);
            return fwd_run<FwdKernel::kChannelLane, TIn, 16, 1>(s, a, softplus, gate, scratch, scratch_cap, st);
        }
    }
    return fwd_run<FwdKernel::kWarp, TIn, NP>(s, a, softplus, gate, scratch, scratch_cap, st);
}

// ---------------------------------------------------------------------------- checks
static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

static int check_shape(const mamba_scan_shape* s, bool need_len) {
    if (!s) return fail(MAMBA_ERR_ARG, "shape is NULL");
    if (s->batch <= 0 || s->dim <= 0) return fail(MAMBA_ERR_ARG, "batch and dim must be positive");
    if (s->dstate <= 0 || s->dstate > MAMBA_MAX_DSTATE)
        return fail(MAMBA_ERR_ARG, "dstate must be in [1, %d]", MAMBA_MAX_DSTATE);
    if (need_len && s->seqlen < 0) return fail(MAMBA_ERR_ARG, "seqlen must be >= 0");
    if (s->in_dtype != MAMBA_F32 && s->in_dtype != MAMBA_BF16)
        return fail(MAMBA_ERR_ARG, "in_dtype must be MAMBA_F32 or MAMBA_BF16");
    return MAMBA_OK;
}

template <typename TIn, int NP>
static int step_dispatch(const StepArgs& a, cudaStream_t st) {
    constexpr int S = NP / (NP < 8 ? NP : 8);  // threads per channel (state_step_kernel)
    const int bs = 256;
    const long long gx = ((long long)a.dim * S + bs - 1) / bs;  // blocks over channels
    const long long gy = ((long long)a.batch + kStepRows - 1) / kStepRows;
    if (gx > 0x7fffffffLL || gy > 65535) return fail(MAMBA_ERR_ARG, "too many channels or batch rows");
    const dim3 grid((unsigned)gx, (unsigned)gy);
    // vector accesses: whole rows of NP states, 16-byte aligned state and A rows
    const bool vec4 = (a.dstate == NP) && aligned16(a.state) && aligned16(a.A);
    if (vec4)
        state_step_kernel<TIn, NP, true><<<grid, bs, 0, st>>>(a);
    else
        state_step_kernel<TIn, NP, false><<<grid, bs, 0, st>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "state_step_kernel launch");
    return MAMBA_OK;
}

template <typename TIn, bool ZOH>
static int bwd_launch(const BwdArgs& a, bool vec, cudaStream_t st) {
    static AttrCache attr_vec, attr_scalar;
    auto kern = vec ? scan_bwd_kernel<TIn, true, ZOH> : scan_bwd_kernel<TIn, false, ZOH>;
    int rc = allow_smem(kern, vec ? attr_vec : attr_scalar);
    if (rc) return rc;
    const dim3 grid((unsigned)((a.dim + bwd::kCh - 1) / bwd::kCh), (unsigned)a.batch);
    kern<<<grid, bwd::kThreads, bwd::Layout<TIn>::BYTES, st>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "scan_bwd_kernel launch");
    return MAMBA_OK;
}

}  // namespace mscan

using namespace mscan;

struct ConvSpec {
    const float* w = nullptr;
    const float* bias = nullptr;
    const float* prev = nullptr;
    int k = 0;
    int silu = 0;
};

static int scan_fwd_impl(const mamba_scan_shape* s, const void* u, const void* delta, const float* A, const void* B,
                         const void* C, const float* D, const void* z, const float* delta_bias, int softplus_flag,
                         const float* h0, void* y, float* last_state, float2* scratch, size_t scratch_cap,
                         void* stream, int discretization = MAMBA_DISC_SIMPLE, ConvSpec conv = ConvSpec()) {
    t_err.clear();
    int rc = check_shape(s, true);
    if (rc) return rc;
    if (discretization != MAMBA_DISC_SIMPLE && discretization != MAMBA_DISC_ZOH)
        return fail(MAMBA_ERR_ARG, "unknown discretization %d", discretization);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long chans = (long long)s->batch * s->dim;
    if (s->seqlen == 0) {
        if (last_state) {
            const size_t nb = (size_t)chans * s->dstate * sizeof(float);
            cudaError_t e = h0 ? (h0 == last_state ? cudaSuccess
                                                   : cudaMemcpyAsync(last_state, h0, nb, cudaMemcpyDeviceToDevice, st))
                               : cudaMemsetAsync(last_state, 0, nb, st);
            if (e != cudaSuccess) return cuda_fail(e, "last_state for an empty sequence");
        }
        return MAMBA_OK;
    }
    if (!u || !delta || !A || !B || !C || !y) return fail(MAMBA_ERR_ARG, "u, delta, A, B, C and y are required");
    if (s->seqlen > (1LL << 40)) return fail(MAMBA_ERR_ARG, "seqlen too large");
    const size_t es = s->in_dtype == MAMBA_F32 ? 4 : 2;
    const size_t nx = (size_t)chans * s->seqlen * es;
    const size_t nbc = (size_t)s->batch * s->dstate * s->seqlen * es;
    if (overlaps(y, nx, u, nx) || overlaps(y, nx, delta, nx) || overlaps(y, nx, z, nx) || overlaps(y, nx, B, nbc) ||
        overlaps(y, nx, C, nbc) || overlaps(y, nx, last_state, (size_t)chans * s->dstate * 4) ||
        overlaps(y, nx, h0, (size_t)chans * s->dstate * 4))
        return fail(MAMBA_ERR_ARG, "y overlaps an input or last_state");
    if (h0 && last_state && h0 != last_state &&
        overlaps(h0, (size_t)chans * s->dstate * 4, last_state, (size_t)chans * s->dstate * 4))
        return fail(MAMBA_ERR_ARG, "h0 and last_state must be the same buffer or not overlap");
    FwdArgs a{};
    a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C;
    a.A = A; a.D = D; a.bias = delta_bias;
    a.y = y; a.last_state = last_state; a.h0 = h0;
    a.batch = s->batch; a.dim = s->dim; a.dstate = s->dstate;
    a.L = s->seqlen;
    a.zoh = discretization == MAMBA_DISC_ZOH;
    a.conv_w = conv.w; a.conv_bias = conv.bias; a.conv_prev = conv.prev;
    a.conv_k = conv.k; a.conv_silu = conv.silu;
    const bool sp = softplus_flag != 0, gate = z != nullptr;
    const bool bf = s->in_dtype == MAMBA_BF16;
    if (s->dstate <= 16)
        return bf ? fwd_dispatch<uint16_t, 16>(s, a, sp, gate, scratch, scratch_cap, st) : fwd_dispatch<float, 16>(s, a, sp, gate, scratch, scratch_cap, st);
    if (s->dstate <= 32)
        return bf ? fwd_dispatch<uint16_t, 32>(s, a, sp, gate, scratch, scratch_cap, st) : fwd_dispatch<float, 32>(s, a, sp, gate, scratch, scratch_cap, st);
    return bf ? fwd_dispatch<uint16_t, 64>(s, a, sp, gate, scratch, scratch_cap, st) : fwd_dispatch<float, 64>(s, a, sp, gate, scratch, scratch_cap, st);
}

extern "C" int mamba_scan_fwd(const mamba_scan_shape* s, const void* u, const void* delta, const float* A,
                              const void* B, const void* C, const float* D, const void* z,
                              const float* delta_bias, int softplus_flag, void* y, float* last_state,
                              void* stream) {
    return scan_fwd_impl(s, u, delta, A, B, C, D, z, delta_bias, softplus_flag, nullptr, y, last_state, nullptr, 0,
                         stream);
}

extern "C" int mamba_scan_fwd_state(const mamba_scan_shape* s, const void* u, const void* delta, const float* A,
                                    const void* B, const void* C, const float* D, const void* z,
                                    const float* delta_bias, int softplus_flag, const float* h0, void* y,
                                    float* last_state, void* stream) {
    return scan_fwd_impl(s, u, delta, A, B, C, D, z, delta_bias, softplus_flag, h0, y, last_state, nullptr, 0,
                         stream);
}

extern "C" int mamba_scan_fwd_ex(const mamba_scan_shape* s, int discretization, const void* u, const void* delta,
                                 const float* A, const void* B, const void* C, const float* D, const void* z,
                                 const float* delta_bias, int softplus_flag, const float* h0, void* y,
                                 float* last_state, void* stream) {
    return scan_fwd_impl(s, u, delta, A, B, C, D, z, delta_bias, softplus_flag, h0, y, last_state, nullptr, 0,
                         stream, discretization);
}

extern "C" int mamba_scan_fwd_conv(const mamba_scan_shape* s, int discretization, const void* x, const float* conv_w,
                                   const float* conv_bias, int conv_k, int conv_silu, const float* conv_prev,
                                   const void* delta, const float* A, const void* B, const void* C, const float* D,
                                   const void* z, const float* delta_bias, int softplus_flag, const float* h0,
                                   void* y, float* last_state, void* stream) {
    t_err.clear();
    if (!conv_w) return fail(MAMBA_ERR_ARG, "conv_w is required");
    if (conv_k < 1 || conv_k > 4) return fail(MAMBA_ERR_ARG, "conv_k must be in [1, 4]");
    ConvSpec cs;
    cs.w = conv_w; cs.bias = conv_bias; cs.prev = conv_prev; cs.k = conv_k; cs.silu = conv_silu != 0;
    return scan_fwd_impl(s, x, delta, A, B, C, D, z, delta_bias, softplus_flag, h0, y, last_state, nullptr, 0, stream,
                         discretization, cs);
}

// ---------------------------------------------------------------------------- allocation-free variant
// Scratch of mamba_scan_fwd_noalloc: the segment carries of a split time axis.  A file-scope
// device array, so it exists on every device that loads this library, from module load to exit.
static __device__ __align__(256) float2 g_noalloc_scratch[MAMBA_NOALLOC_SCRATCH_BYTES / sizeof(float2)];

// Device address of g_noalloc_scratch in the CUDA context current on this thread.  In host code
// the symbol is only a host-side stand-in, so its device address is looked up with
// cudaGetSymbolAddress the first time a context calls (the set-up of that device in that
// context) and cached under the context's unique id; a reset device or another context (driver
// API) gets a fresh lookup instead of a stale address.
static int noalloc_scratch(float2** out) {
    static std::mutex mu;
    struct Entry {
        unsigned long long ctx;
        float2* addr;
    };
    static Entry cache[256] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 256) return fail(MAMBA_ERR_ARG, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);
    unsigned long long ctx = current_context_id();
    if (ctx != 0 && cache[dev].ctx == ctx && cache[dev].addr != nullptr) {
        *out = cache[dev].addr;
        return MAMBA_OK;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the device's context current if needed
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    if (ctx == 0) ctx = current_context_id();
    cache[dev].ctx = ctx;  // 0 (no id available) never matches, so the lookup then repeats
    cache[dev].addr = static_cast<float2*>(p);
    *out = cache[dev].addr;
    return MAMBA_OK;
}

extern "C" int mamba_scan_fwd_noalloc(const mamba_scan_shape* s, const void* u, const void* delta, const float* A,
                                      const void* B, const void* C, const float* D, const void* z,
                                      const float* delta_bias, int softplus_flag, void* y, float* last_state,
                                      void* stream) {
    t_err.clear();
    int rc = check_shape(s, true);
    if (rc) return rc;
    float2* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    return scan_fwd_impl(s, u, delta, A, B, C, D, z, delta_bias, softplus_flag, nullptr, y, last_state, scratch,
                         (size_t)MAMBA_NOALLOC_SCRATCH_BYTES, stream);
}

static int state_step_impl(const mamba_scan_shape* s, int discretization, float* state, const void* x,
                           const void* delta, const float* A, const void* B, const void* C, const float* D,
                           const void* z, const float* delta_bias, int softplus_flag, void* y, void* stream) {
    t_err.clear();
    int rc = check_shape(s, false);
    if (rc) return rc;
    if (discretization != MAMBA_DISC_SIMPLE && discretization != MAMBA_DISC_ZOH)
        return fail(MAMBA_ERR_ARG, "unknown discretization %d", discretization);
    if (!state || !x || !delta || !A || !B || !C || !y)
        return fail(MAMBA_ERR_ARG, "state, x, delta, A, B, C and y are required");
    const long long chans = (long long)s->batch * s->dim;
    const size_t es = s->in_dtype == MAMBA_F32 ? 4 : 2;
    const size_t ny = (size_t)chans * es;
    const size_t ns = (size_t)chans * s->dstate * 4;
    if (overlaps(y, ny, state, ns) || overlaps(y, ny, x, ny) || overlaps(y, ny, delta, ny) || overlaps(y, ny, z, ny))
        return fail(MAMBA_ERR_ARG, "y overlaps the state or an input");
    StepArgs a{};
    a.state = state; a.x = x; a.delta = delta; a.z = z; a.B = B; a.C = C;
    a.A = A; a.D = D; a.bias = delta_bias; a.y = y;
    a.batch = s->batch; a.dim = s->dim; a.dstate = s->dstate;
    a.softplus = softplus_flag != 0;
    a.zoh = discretization == MAMBA_DISC_ZOH;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool bf = s->in_dtype == MAMBA_BF16;
    if (s->dstate <= 4) return bf ? step_dispatch<uint16_t, 4>(a, st) : step_dispatch<float, 4>(a, st);
    if (s->dstate <= 16) return bf ? step_dispatch<uint16_t, 16>(a, st) : step_dispatch<float, 16>(a, st);
    if (s->dstate <= 32) return bf ? step_dispatch<uint16_t, 32>(a, st) : step_dispatch<float, 32>(a, st);
    return bf ? step_dispatch<uint16_t, 64>(a, st) : step_dispatch<float, 64>(a, st);
}

extern "C" int mamba_state_step(const mamba_scan_shape* s, float* state, const void* x, const void* delta,
                                const float* A, const void* B, const void* C, const float* D, const void* z,
                                const float* delta_bias, int softplus_flag, void* y, void* stream) {
    return state_step_impl(s, MAMBA_DISC_SIMPLE, state, x, delta, A, B, C, D, z, delta_bias, softplus_flag, y,
                           stream);
}

extern "C" int mamba_state_step_ex(const mamba_scan_shape* s, int discretization, float* state, const void* x,
                                   const void* delta, const float* A, const void* B, const void* C, const float* D,
                                   const void* z, const float* delta_bias, int softplus_flag, void* y,
                                   void* stream) {
    return state_step_impl(s, discretization, state, x, delta, A, B, C, D, z, delta_bias, softplus_flag, y, stream);
}

extern "C" int mamba_scan_bwd(const mamba_scan_shape* s, int discretization, const void* u, const void* delta,
                              const float* A, const void* B, const void* C, const float* D, const void* z,
                              const float* delta_bias, int softplus_flag, const float* h0, const void* dy,
                              const float* dlast_state, void* du, void* ddelta, void* dz, float* dA, float* dB,
                              float* dC, float* dD, float* ddelta_bias, float* dh0, void* stream) {
    t_err.clear();
    int rc = check_shape(s, true);
    if (rc) return rc;
    if (discretization != MAMBA_DISC_SIMPLE && discretization != MAMBA_DISC_ZOH)
        return fail(MAMBA_ERR_ARG, "unknown discretization %d", discretization);
    if (s->dstate > 16) return fail(MAMBA_ERR_ARG, "the backward pass supports dstate <= 16");
    if (s->batch > 65535) return fail(MAMBA_ERR_ARG, "the backward pass supports batch <= 65535");
    if (s->seqlen > (1LL << 34)) return fail(MAMBA_ERR_ARG, "seqlen too large");
    if (!A || !dA) return fail(MAMBA_ERR_ARG, "A and dA are required");
    if (dz && !z) return fail(MAMBA_ERR_ARG, "dz given without z");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long chans = (long long)s->batch * s->dim;
    const long long L = s->seqlen;
    const int N = s->dstate;
    const size_t es = s->in_dtype == MAMBA_F32 ? 4 : 2;
    const size_t nx = (size_t)chans * L * es, nbc4 = (size_t)s->batch * N * L * 4, ns = (size_t)chans * N * 4;
    cudaError_t e = cudaMemsetAsync(dA, 0, (size_t)s->dim * N * 4, st);
    if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, (size_t)s->dim * 4, st);
    if (e == cudaSuccess && ddelta_bias) e = cudaMemsetAsync(ddelta_bias, 0, (size_t)s->dim * 4, st);
    if (e != cudaSuccess) return cuda_fail(e, "zeroing parameter gradients");
    if (L == 0) {  // nothing reaches the inputs; the state's gradient passes straight through
        if (dh0) {
            e = dlast_state ? (dlast_state == dh0 ? cudaSuccess
                                                  : cudaMemcpyAsync(dh0, dlast_state, ns, cudaMemcpyDeviceToDevice, st))
                            : cudaMemsetAsync(dh0, 0, ns, st);
            if (e != cudaSuccess) return cuda_fail(e, "dh0 for an empty sequence");
        }
        return MAMBA_OK;
    }
    if (!u || !delta || !B || !C || !dy || !du || !ddelta || !dB || !dC)
        return fail(MAMBA_ERR_ARG, "u, delta, B, C, dy, du, ddelta, dB and dC are required");
    const void* ins[] = {u, delta, z, dy};
    const void* outs[] = {du, ddelta, dz};
    for (const void* o : outs)
        for (const void* i : ins)
            if (overlaps(o, nx, i, nx)) return fail(MAMBA_ERR_ARG, "a gradient output overlaps an input");
    if (overlaps(du, nx, ddelta, nx) || overlaps(du, nx, dz, nx) || overlaps(ddelta, nx, dz, nx) ||
        overlaps(dB, nbc4, dC, nbc4) || overlaps(dB, nbc4, B, nbc4 * es / 4) || overlaps(dC, nbc4, C, nbc4 * es / 4))
        return fail(MAMBA_ERR_ARG, "gradient outputs overlap");
    e = cudaMemsetAsync(dB, 0, nbc4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dC, 0, nbc4, st);
    if (e != cudaSuccess) return cuda_fail(e, "zeroing dB/dC");

    BwdArgs a{};
    a.u = u; a.delta = delta; a.z = z; a.dy = dy; a.B = B; a.C = C;
    a.A = A; a.D = D; a.bias = delta_bias; a.h0 = h0; a.dlast = dlast_state;
    a.du = du; a.ddelta = ddelta; a.dz = dz;
    a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD; a.dbias = ddelta_bias; a.dh0 = dh0;
    a.batch = s->batch; a.dim = s->dim; a.dstate = N; a.L = L;
    a.ntile = (int)((L + bwd::kT - 1) / bwd::kT);
    a.nslot = (int)((L + bwd::kSlot - 1) / bwd::kSlot);
    a.softplus = softplus_flag != 0;
    const bool vec = (L * (long long)es) % 16 == 0 && aligned16(u) && aligned16(delta) && aligned16(dy) &&
                     aligned16(B) && aligned16(C) && aligned16(du) && aligned16(ddelta) && aligned16(dB) &&
                     aligned16(dC) && (!z || aligned16(z)) && (!dz || aligned16(dz));
    float* ckpt = nullptr;
    if (a.nslot > 1) {
        const size_t nck = (size_t)s->batch * a.nslot * s->dim * bwd::kNS * sizeof(float);
        e = cudaMallocAsync(reinterpret_cast<void**>(&ckpt), nck, st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(state checkpoints)");
    }
    a.ckpt = ckpt;
    const bool zoh = discretization == MAMBA_DISC_ZOH;
    if (s->in_dtype == MAMBA_BF16)
        rc = zoh ? bwd_launch<uint16_t, true>(a, vec, st) : bwd_launch<uint16_t, false>(a, vec, st);
    else
        rc = zoh ? bwd_launch<float, true>(a, vec, st) : bwd_launch<float, false>(a, vec, st);
    if (ckpt) {
        e = cudaFreeAsync(ckpt, st);
        if (rc == MAMBA_OK && e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(state checkpoints)");
    }
    return rc;
}

extern "C" const char* mamba_scan_last_error(void) { return t_err.c_str(); }

extern "C" int mamba_scan_version(void) { return MAMBA_SCAN_VERSION; }

extern "C" long long mamba_scan_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int mamba_scan_device_status(void* stream) {
    t_err.clear();
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_status, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e, "read device status");
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_status, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e, "clear device status");
        return fail(MAMBA_ERR_TIMEOUT, "a kernel abandoned a bounded wait for an asynchronous copy");
    }
    return MAMBA_OK;
}
