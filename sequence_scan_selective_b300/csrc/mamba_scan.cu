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
#include "scan_fwd.cuh"
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

// 3-D map over a dense [d2][d1][d0] tensor (d0 contiguous) with box [b1 rows x b0 cols].
static bool encode_3d(CUtensorMap* m, const void* base, int esize, long long d0, long long d1, long long d2,
                      int b0, int b1, bool swizzle64) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
    cuuint64_t strides[2] = {(cuuint64_t)(d0 * esize), (cuuint64_t)(d0 * d1 * esize)};
    cuuint32_t box[3] = {(cuuint32_t)b0, (cuuint32_t)b1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------- forward launch
template <typename TIn, int NP, int G, int CH, int TC, int NSTAGE, bool TMA, bool AGG>
static int launch_fwd_one(const FwdArgs& a, dim3 grid, const CUtensorMap* maps, cudaStream_t st) {
    using SM = FwdSmem<TIn, NP, G, CH, TC, NSTAGE>;
    auto kern = scan_fwd_kernel<TIn, NP, G, CH, TC, NSTAGE, TMA, AGG>;
    const int smem_bytes = SM::kBytes + 1024;  // slack to align the swizzled tiles
    static bool attr_set = false;              // benign race: every caller sets the same value
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        attr_set = true;
    }
    kern<<<grid, CH * (NP / G) + 32, smem_bytes, st>>>(a, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5]);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "scan_fwd_kernel launch");
    return MAMBA_OK;
}

struct FwdPlan {
    int nseg;
    long long seg_len;
};

// Split the time axis only when the channels alone cannot fill the GPU: a split costs one extra
// pass over delta, u and B for all but the last segment.
static FwdPlan plan_split(long long channels, int threads_per_channel, long long L, int TC, int nsm) {
    FwdPlan p{1, L};
    const char* force = getenv("MAMBA_SCAN_NSEG");
    long long want = 1;
    if (force && atoi(force) > 0) {
        want = atoi(force);
    } else {
        const long long target = (long long)nsm * 192;  // scan threads that keep every SM busy
        const long long have = channels * threads_per_channel;
        if (have < target / 2) want = (target + have - 1) / have;
    }
    const long long min_seg = 16LL * TC;
    long long maxseg = L / min_seg;
    if (maxseg < 1) maxseg = 1;
    if (want > maxseg) want = maxseg;
    if (want > 4096) want = 4096;
    if (want <= 1) return p;
    long long seg = (L + want - 1) / want;
    seg = (seg + TC - 1) / TC * TC;
    p.seg_len = seg;
    p.nseg = (int)((L + seg - 1) / seg);
    return p;
}

// One tiling of the forward kernel: G states per thread, CH channels per CTA, TC steps per chunk,
// NSTAGE-deep TMA ring.
template <typename TIn, int NP, int G, int CH, int TC, int NSTAGE>
static int fwd_run(const mamba_scan_shape* s, FwdArgs a, cudaStream_t st) {
    constexpr int S = NP / G;
    const int esize = (int)sizeof(TIn);
    const long long L = s->seqlen;

    int dev = 0, nsm = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);

    const bool tma_ok = encode_fn() != nullptr && (L * esize) % 16 == 0 && aligned16(a.u) && aligned16(a.delta) &&
                        aligned16(a.B) && aligned16(a.C) && aligned16(a.y) && (a.z == nullptr || aligned16(a.z)) &&
                        L < (1LL << 31) && getenv("MAMBA_SCAN_NO_TMA") == nullptr;
    CUtensorMap maps[6];
    memset(maps, 0, sizeof maps);
    if (tma_ok) {
        const void* zb = a.z ? a.z : a.u;
        bool ok = encode_3d(&maps[0], a.u, esize, L, s->dim, s->batch, TC, CH, true) &&
                  encode_3d(&maps[1], a.delta, esize, L, s->dim, s->batch, TC, CH, true) &&
                  encode_3d(&maps[2], zb, esize, L, s->dim, s->batch, TC, CH, true) &&
                  encode_3d(&maps[3], a.B, esize, L, s->dstate, s->batch, TC, s->dstate, false) &&
                  encode_3d(&maps[4], a.C, esize, L, s->dstate, s->batch, TC, s->dstate, false) &&
                  encode_3d(&maps[5], a.y, esize, L, s->dim, s->batch, TC, CH, true);
        if (!ok) return fail(MAMBA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    }

    const long long nblk = (s->dim + CH - 1) / CH;
    const FwdPlan plan = plan_split((long long)s->batch * s->dim, S, L, TC, nsm);
    a.nseg = plan.nseg;
    a.seg_len = plan.seg_len;
    a.agg = nullptr;
    if (plan.nseg > 65535 || s->batch > 65535) return fail(MAMBA_ERR_ARG, "grid too large");

    int rc = MAMBA_OK;
    if (plan.nseg > 1) {
        const size_t bytes = (size_t)(plan.nseg - 1) * s->batch * s->dim * s->dstate * sizeof(float2);
        cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&a.agg), bytes, st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync (segment carries)");
        dim3 g1((unsigned)nblk, (unsigned)s->batch, (unsigned)(plan.nseg - 1));
        rc = tma_ok ? launch_fwd_one<TIn, NP, G, CH, TC, NSTAGE, true, true>(a, g1, maps, st)
                    : launch_fwd_one<TIn, NP, G, CH, TC, NSTAGE, false, true>(a, g1, maps, st);
    }
    if (rc == MAMBA_OK) {
        dim3 g2((unsigned)nblk, (unsigned)s->batch, (unsigned)plan.nseg);
        rc = tma_ok ? launch_fwd_one<TIn, NP, G, CH, TC, NSTAGE, true, false>(a, g2, maps, st)
                    : launch_fwd_one<TIn, NP, G, CH, TC, NSTAGE, false, false>(a, g2, maps, st);
    }
    if (a.agg) {
        cudaError_t e = cudaFreeAsync(a.agg, st);
        if (e != cudaSuccess && rc == MAMBA_OK) rc = cuda_fail(e, "cudaFreeAsync (segment carries)");
    }
    return rc;
}

static int variant() {
    const char* v = getenv("MAMBA_SCAN_VARIANT");
    return v ? atoi(v) : 0;
}

template <typename TIn, int NP>
static int fwd_dispatch(const mamba_scan_shape* s, const FwdArgs& a, cudaStream_t st) {
    // 64-byte tile rows: 32 bf16 or 16 fp32 steps per chunk
    constexpr int TC = sizeof(TIn) == 2 ? 32 : 16;
    constexpr int NSTAGE = sizeof(TIn) == 2 ? 3 : 4;
    if constexpr (NP == 16) {
        if (variant() == 1) return fwd_run<TIn, 16, 4, 32, TC, NSTAGE>(s, a, st);
    }
    return fwd_run<TIn, NP, 8, 32, TC, NSTAGE>(s, a, st);
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
    constexpr int S = NP / 4;
    const long long threads = (long long)a.batch * a.dim * S;
    const int bs = 256;
    const long long blocks = (threads + bs - 1) / bs;
    if (blocks > 0x7fffffffLL) return fail(MAMBA_ERR_ARG, "too many channels");
    const bool vec4 = (a.dstate == NP) && aligned16(a.state);
    if (vec4)
        state_step_kernel<TIn, NP, true><<<(unsigned)blocks, bs, 0, st>>>(a);
    else
        state_step_kernel<TIn, NP, false><<<(unsigned)blocks, bs, 0, st>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "state_step_kernel launch");
    return MAMBA_OK;
}

}  // namespace mscan

using namespace mscan;

extern "C" int mamba_scan_fwd(const mamba_scan_shape* s, const void* u, const void* delta, const float* A,
                              const void* B, const void* C, const float* D, const void* z,
                              const float* delta_bias, int softplus_flag, void* y, float* last_state,
                              void* stream) {
    t_err.clear();
    int rc = check_shape(s, true);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long chans = (long long)s->batch * s->dim;
    if (s->seqlen == 0) {
        if (last_state) {
            cudaError_t e = cudaMemsetAsync(last_state, 0, (size_t)chans * s->dstate * sizeof(float), st);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(last_state)");
        }
        return MAMBA_OK;
    }
    if (!u || !delta || !A || !B || !C || !y) return fail(MAMBA_ERR_ARG, "u, delta, A, B, C and y are required");
    if (s->seqlen > (1LL << 40)) return fail(MAMBA_ERR_ARG, "seqlen too large");
    const size_t es = s->in_dtype == MAMBA_F32 ? 4 : 2;
    const size_t nx = (size_t)chans * s->seqlen * es;
    const size_t nbc = (size_t)s->batch * s->dstate * s->seqlen * es;
    if (overlaps(y, nx, u, nx) || overlaps(y, nx, delta, nx) || overlaps(y, nx, z, nx) || overlaps(y, nx, B, nbc) ||
        overlaps(y, nx, C, nbc) || overlaps(y, nx, last_state, (size_t)chans * s->dstate * 4))
        return fail(MAMBA_ERR_ARG, "y overlaps an input or last_state");
    FwdArgs a{};
    a.u = u; a.delta = delta; a.z = z; a.B = B; a.C = C;
    a.A = A; a.D = D; a.bias = delta_bias;
    a.y = y; a.last_state = last_state;
    a.batch = s->batch; a.dim = s->dim; a.dstate = s->dstate;
    a.L = s->seqlen;
    a.softplus = softplus_flag != 0;
    a.has_z = z != nullptr;
    const bool bf = s->in_dtype == MAMBA_BF16;
    if (s->dstate <= 16) return bf ? fwd_dispatch<uint16_t, 16>(s, a, st) : fwd_dispatch<float, 16>(s, a, st);
    if (s->dstate <= 32) return bf ? fwd_dispatch<uint16_t, 32>(s, a, st) : fwd_dispatch<float, 32>(s, a, st);
    return bf ? fwd_dispatch<uint16_t, 64>(s, a, st) : fwd_dispatch<float, 64>(s, a, st);
}

extern "C" int mamba_state_step(const mamba_scan_shape* s, float* state, const void* x, const void* delta,
                                const float* A, const void* B, const void* C, const float* D, const void* z,
                                const float* delta_bias, int softplus_flag, void* y, void* stream) {
    t_err.clear();
    int rc = check_shape(s, false);
    if (rc) return rc;
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
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool bf = s->in_dtype == MAMBA_BF16;
    if (s->dstate <= 4) return bf ? step_dispatch<uint16_t, 4>(a, st) : step_dispatch<float, 4>(a, st);
    if (s->dstate <= 16) return bf ? step_dispatch<uint16_t, 16>(a, st) : step_dispatch<float, 16>(a, st);
    if (s->dstate <= 32) return bf ? step_dispatch<uint16_t, 32>(a, st) : step_dispatch<float, 32>(a, st);
    return bf ? step_dispatch<uint16_t, 64>(a, st) : step_dispatch<float, 64>(a, st);
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
