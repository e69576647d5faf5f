// Host side of libmambascan.so: the C ABI declared in include/mamba_scan.h, argument checks, the
// choice between the two forward kernels, and the helpers shared by the kernel units (host.cuh).
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
#include "host.cuh"
#include "scan_fwd.cuh"
#include "scan_bwd.cuh"
#include "state_step.cuh"
#include "conv.cuh"

namespace mscan {

static thread_local std::string t_err;
static std::atomic<long long> g_launches{0};

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) { return fail(MAMBA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e)); }

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int sm_count() {
    int dev = 0, nsm = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    return nsm;
}

int env_int(const char* name, int dflt) {
    const char* v = getenv(name);
    return (v && *v) ? atoi(v) : dflt;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

// ---------------------------------------------------------------------------- TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

bool encode_3d(CUtensorMap* m, const void* base, int esize, long long d0, long long d1, long long d2, int b0,
               int b1) {
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

// the function in one context; setting it on every call costs tens of microseconds of host time).
// Unique id of the CUDA context current on this thread (0 if none is current or the driver
// entry points are missing).  Ids are never reused within a process, so an id stays tied to one
// context even after cudaDeviceReset replaces the primary context at the same address.
unsigned long long current_context_id() {
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


// ---------------------------------------------------------------------------- forward kernel choice
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
static int choose_lane_kernel(const mamba_scan_shape* s, bool* use_lane) {
    const char* force = getenv("MAMBA_SCAN_KERNEL");
    const bool lane_ok = s->dstate <= 16;
    *use_lane = lane_ok && prefer_lane_kernel(s, sm_count());
    if (force && strcmp(force, "warp") == 0) *use_lane = false;
    if (force && strcmp(force, "lane") == 0) {
        if (!lane_ok) return fail(MAMBA_ERR_ARG, "MAMBA_SCAN_KERNEL=lane: the channel-per-lane kernel takes N <= 16");
        *use_lane = true;
    }
    return MAMBA_OK;
}

static int fwd_dispatch(const mamba_scan_shape* s, const FwdArgs& a, bool softplus, bool gate, float2* scratch,
                        size_t scratch_cap, cudaStream_t st) {
    bool use_lane = false;
    const int rc = choose_lane_kernel(s, &use_lane);
    if (rc) return rc;
    const bool bf = s->in_dtype == MAMBA_BF16;
    if (use_lane)
        return bf ? fwd_lane_run_t<uint16_t>(s, a, softplus, scratch, scratch_cap, st)
                  : fwd_lane_run_t<float>(s, a, softplus, scratch, scratch_cap, st);
    return bf ? fwd_warp_run_t<uint16_t>(s, a, softplus, gate, scratch, scratch_cap, st)
              : fwd_warp_run_t<float>(s, a, softplus, gate, scratch, scratch_cap, st);
}

// ---------------------------------------------------------------------------- checks
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

}  // namespace mscan

using namespace mscan;

struct ConvSpec {
    const float* w = nullptr;
    const float* bias = nullptr;
    const float* prev = nullptr;
    int k = 0;
    int silu = 0;
};

struct CkptSpec {
    float* ckpt = nullptr;     // forward pass of training: state checkpoints, or NULL
    int* written = nullptr;    // set to 1 when they were written
};

static int scan_fwd_impl(const mamba_scan_shape* s, const void* u, const void* delta, const float* A, const void* B,
                         const void* C, const float* D, const void* z, const float* delta_bias, int softplus_flag,
                         const float* h0, void* y, float* last_state, float2* scratch, size_t scratch_cap,
                         void* stream, int discretization = MAMBA_DISC_SIMPLE, ConvSpec conv = ConvSpec(),
                         CkptSpec ck = CkptSpec()) {
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
    a.ckpt = ck.ckpt;
    a.ck_nslot = (int)((s->seqlen + 7) / 8);
    a.ck_written = ck.written;
    return fwd_dispatch(s, a, softplus_flag != 0, z != nullptr, scratch, scratch_cap, st);
}

extern "C" int mamba_scan_fwd_train_ckpt_bytes(const mamba_scan_shape* s, size_t* bytes) {
    t_err.clear();
    if (!bytes) return fail(MAMBA_ERR_ARG, "bytes is NULL");
    *bytes = 0;
    int rc = check_shape(s, true);
    if (rc) return rc;
    if (s->dstate > 16 || s->seqlen == 0) return MAMBA_OK;
    bool lane = false;
    rc = choose_lane_kernel(s, &lane);
    if (rc) return rc;
    const bool bf = s->in_dtype == MAMBA_BF16;
    const int nseg = lane ? (bf ? fwd_lane_nseg_t<uint16_t>(s) : fwd_lane_nseg_t<float>(s))
                          : (bf ? fwd_warp_nseg_t<uint16_t>(s) : fwd_warp_nseg_t<float>(s));
    if (nseg < 0) return nseg;
    if (nseg == 1) *bytes = (size_t)s->batch * (size_t)((s->seqlen + 7) / 8) * s->dim * 16 * sizeof(float);
    return MAMBA_OK;
}

extern "C" int mamba_scan_fwd_train(const mamba_scan_shape* s, int discretization, const void* u, const void* delta,
                                    const float* A, const void* B, const void* C, const float* D, const void* z,
                                    const float* delta_bias, int softplus_flag, const float* h0, void* y,
                                    float* last_state, float* ckpt, int* ckpt_written, void* stream) {
    t_err.clear();
    if (ckpt_written) *ckpt_written = 0;
    int rc = check_shape(s, true);
    if (rc) return rc;
    if (!ckpt || !ckpt_written) return fail(MAMBA_ERR_ARG, "ckpt and ckpt_written are required");
    if (!aligned16(ckpt)) return fail(MAMBA_ERR_ARG, "ckpt must be 16-byte aligned");
    if (s->dstate > 16) return fail(MAMBA_ERR_ARG, "checkpoints are kept for dstate <= 16");
    const long long chans = (long long)s->batch * s->dim;
    const size_t es = s->in_dtype == MAMBA_F32 ? 4 : 2;
    const size_t nx = (size_t)chans * s->seqlen * es, nbc = (size_t)s->batch * s->dstate * s->seqlen * es;
    const size_t nck = (size_t)chans * ((s->seqlen + 7) / 8) * 16 * sizeof(float);
    if (overlaps(ckpt, nck, u, nx) || overlaps(ckpt, nck, delta, nx) || overlaps(ckpt, nck, z, nx) ||
        overlaps(ckpt, nck, y, nx) || overlaps(ckpt, nck, B, nbc) || overlaps(ckpt, nck, C, nbc) ||
        overlaps(ckpt, nck, last_state, (size_t)chans * s->dstate * 4) || overlaps(ckpt, nck, h0, (size_t)chans * s->dstate * 4))
        return fail(MAMBA_ERR_ARG, "ckpt overlaps an input or an output");
    CkptSpec ck;
    ck.ckpt = ckpt;
    ck.written = ckpt_written;
    return scan_fwd_impl(s, u, delta, A, B, C, D, z, delta_bias, softplus_flag, h0, y, last_state, nullptr, 0, stream,
                         discretization, ConvSpec(), ck);
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
    return step_run(a, s->in_dtype, static_cast<cudaStream_t>(stream));
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

static int scan_bwd_impl(const mamba_scan_shape* s, int discretization, const void* u, const void* delta,
                         const float* A, const void* B, const void* C, const float* D, const void* z,
                         const float* delta_bias, int softplus_flag, const float* h0, const void* dy,
                         const float* dlast_state, void* du, void* ddelta, void* dz, float* dA, float* dB, float* dC,
                         float* dD, float* ddelta_bias, float* dh0, void* stream, const float* ckpt_in = nullptr) {
    int rc = check_shape(s, true);
    if (rc) return rc;
    if (discretization != MAMBA_DISC_SIMPLE && discretization != MAMBA_DISC_ZOH)
        return fail(MAMBA_ERR_ARG, "unknown discretization %d", discretization);
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
    // Split of the time axis, when the CTAs (batch x ceil(dim / 32)) fill at most half of four per
    // SM: segments of at least kBwdMinSegTiles tiles, about four CTAs per SM.  MAMBA_SCAN_BWD_NSEG
    // forces a count (tests).
    constexpr long long kBwdMinSegTiles = 512;
    const long long nsm = sm_count();
    const long long ctas = (long long)s->batch * ((s->dim + bwd::kCh - 1) / bwd::kCh);
    long long S = 1;
    const int want = env_int("MAMBA_SCAN_BWD_NSEG", 0);
    if (want > 0) {
        S = want < a.ntile ? want : a.ntile;
    } else if (ctas * 2 <= 4 * nsm) {
        S = 4 * nsm / ctas;
        const long long smax = a.ntile / kBwdMinSegTiles;
        if (S > smax) S = smax;
    }
    if (S > 4096) S = 4096;
    if (S < 1) S = 1;
    a.seg_tiles = (int)((a.ntile + S - 1) / S);
    a.nseg = (a.ntile + a.seg_tiles - 1) / a.seg_tiles;
    // scratch: the state checkpoints of one block of 16 states (reused by the blocks in turn);
    // with several blocks or segments, fp32 accumulators of du, ddelta (and dz) (for fp32
    // storage the outputs themselves); with segments, their carries and local start gradients
    // checkpoints from the forward pass of training replace the forward sweep (unsplit, N <= 16)
    const bool use_ck = ckpt_in != nullptr && a.nseg == 1 && N <= bwd::kNS && a.nslot > 1;
    a.ck_given = use_ck ? 1 : 0;
    const size_t nck = (a.nslot > 1 && !use_ck) ? (size_t)s->batch * a.nslot * s->dim * bwd::kNS * sizeof(float) : 0;
    const bool accumulate = N > bwd::kNS || a.nseg > 1;
    const size_t nacc = accumulate && s->in_dtype == MAMBA_BF16 ? (size_t)chans * L * sizeof(float) : 0;
    const int nacc_t = dz ? 3 : 2;
    const size_t nstate = (size_t)chans * N;
    const size_t nseg_b = a.nseg > 1 ? (size_t)a.nseg * nstate * (sizeof(float2) + sizeof(float)) : 0;
    char* scratch = nullptr;
    if (nck + nacc * nacc_t + nseg_b > 0) {
        e = cudaMallocAsync(reinterpret_cast<void**>(&scratch), nck + nacc * nacc_t + nseg_b, st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(state checkpoints)");
    }
    a.ckpt = use_ck ? const_cast<float*>(ckpt_in) : nck ? reinterpret_cast<float*>(scratch) : nullptr;
    if (nacc) {
        a.acc_du = reinterpret_cast<float*>(scratch + nck);
        a.acc_dd = reinterpret_cast<float*>(scratch + nck + nacc);
        a.acc_dz = dz ? reinterpret_cast<float*>(scratch + nck + 2 * nacc) : nullptr;
    } else if (accumulate) {  // fp32 storage: accumulate in the outputs
        a.acc_du = static_cast<float*>(du);
        a.acc_dd = static_cast<float*>(ddelta);
        a.acc_dz = static_cast<float*>(dz);
    }
    if (nseg_b) {
        a.carry = reinterpret_cast<float2*>(scratch + nck + nacc * nacc_t);
        a.mu_local = reinterpret_cast<float*>(scratch + nck + nacc * nacc_t + (size_t)a.nseg * nstate * sizeof(float2));
    }
    const bool zoh = discretization == MAMBA_DISC_ZOH;
    rc = bwd_run(a, s->in_dtype, zoh, vec, st);
    if (scratch) {
        e = cudaFreeAsync(scratch, st);
        if (rc == MAMBA_OK && e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(state checkpoints)");
    }
    return rc;
}

extern "C" int mamba_scan_bwd(const mamba_scan_shape* s, int discretization, const void* u, const void* delta,
                              const float* A, const void* B, const void* C, const float* D, const void* z,
                              const float* delta_bias, int softplus_flag, const float* h0, const void* dy,
                              const float* dlast_state, void* du, void* ddelta, void* dz, float* dA, float* dB,
                              float* dC, float* dD, float* ddelta_bias, float* dh0, void* stream) {
    t_err.clear();
    return scan_bwd_impl(s, discretization, u, delta, A, B, C, D, z, delta_bias, softplus_flag, h0, dy, dlast_state,
                         du, ddelta, dz, dA, dB, dC, dD, ddelta_bias, dh0, stream);
}

extern "C" int mamba_scan_bwd_ckpt(const mamba_scan_shape* s, int discretization, const void* u, const void* delta,
                                   const float* A, const void* B, const void* C, const float* D, const void* z,
                                   const float* delta_bias, int softplus_flag, const float* h0, const void* dy,
                                   const float* dlast_state, const float* ckpt, void* du, void* ddelta, void* dz,
                                   float* dA, float* dB, float* dC, float* dD, float* ddelta_bias, float* dh0,
                                   void* stream) {
    t_err.clear();
    if (ckpt && !aligned16(ckpt)) return fail(MAMBA_ERR_ARG, "ckpt must be 16-byte aligned");
    if (s && ckpt && s->seqlen > 0) {
        const long long chans = (long long)s->batch * s->dim;
        const size_t es = s->in_dtype == MAMBA_F32 ? 4 : 2;
        const size_t nx = (size_t)chans * s->seqlen * es, nbc4 = (size_t)s->batch * s->dstate * s->seqlen * 4;
        const size_t nck = (size_t)chans * ((s->seqlen + 7) / 8) * 16 * sizeof(float);
        if (overlaps(ckpt, nck, du, nx) || overlaps(ckpt, nck, ddelta, nx) || overlaps(ckpt, nck, dz, nx) ||
            overlaps(ckpt, nck, dB, nbc4) || overlaps(ckpt, nck, dC, nbc4))
            return fail(MAMBA_ERR_ARG, "ckpt overlaps a gradient output");
    }
    return scan_bwd_impl(s, discretization, u, delta, A, B, C, D, z, delta_bias, softplus_flag, h0, dy, dlast_state,
                         du, ddelta, dz, dA, dB, dC, dD, ddelta_bias, dh0, stream, ckpt);
}

extern "C" int mamba_scan_bwd_conv(const mamba_scan_shape* s, int discretization, const void* x, const float* conv_w,
                                   const float* conv_bias, int conv_k, int conv_silu, const float* conv_prev,
                                   const void* delta, const float* A, const void* B, const void* C, const float* D,
                                   const void* z, const float* delta_bias, int softplus_flag, const float* h0,
                                   const void* dy, const float* dlast_state, void* dx, void* ddelta, void* dz,
                                   float* dA, float* dB, float* dC, float* dD, float* ddelta_bias, float* dconv_w,
                                   float* dconv_bias, float* dconv_prev, float* dh0, void* stream) {
    t_err.clear();
    int rc = check_shape(s, true);
    if (rc) return rc;
    if (!conv_w) return fail(MAMBA_ERR_ARG, "conv_w is required");
    if (conv_k < 1 || conv_k > 4) return fail(MAMBA_ERR_ARG, "conv_k must be in [1, 4]");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long chans = (long long)s->batch * s->dim;
    const long long L = s->seqlen;
    const size_t es = s->in_dtype == MAMBA_F32 ? 4 : 2;
    const size_t nx = (size_t)chans * L * es;
    cudaError_t e = cudaSuccess;
    if (dconv_w) e = cudaMemsetAsync(dconv_w, 0, (size_t)s->dim * conv_k * sizeof(float), st);
    if (e == cudaSuccess && dconv_bias) e = cudaMemsetAsync(dconv_bias, 0, (size_t)s->dim * sizeof(float), st);
    if (e == cudaSuccess && dconv_prev && conv_k > 1)
        e = cudaMemsetAsync(dconv_prev, 0, (size_t)chans * (conv_k - 1) * sizeof(float), st);
    if (e != cudaSuccess) return cuda_fail(e, "zeroing convolution gradients");
    if (L == 0)  // nothing reaches the convolution; the scan's own gradients as for an empty sequence
        return scan_bwd_impl(s, discretization, nullptr, nullptr, A, B, C, D, z, delta_bias, softplus_flag, h0, dy,
                             dlast_state, nullptr, nullptr, nullptr, dA, dB, dC, dD, ddelta_bias, dh0, stream);
    if (!x || !dx) return fail(MAMBA_ERR_ARG, "x and dx are required");
    const void* ins[] = {x, delta, z, dy};
    for (const void* i : ins)
        if (overlaps(dx, nx, i, nx)) return fail(MAMBA_ERR_ARG, "dx overlaps an input");
    if (overlaps(dx, nx, ddelta, nx) || overlaps(dx, nx, dz, nx))
        return fail(MAMBA_ERR_ARG, "gradient outputs overlap");
    // u = conv(x) for the recomputation, and du, in stream-ordered scratch
    char* tmp = nullptr;
    e = cudaMallocAsync(reinterpret_cast<void**>(&tmp), 2 * nx, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync (convolution output and its gradient)");
    ConvArgs ca{};
    ca.x = x; ca.w = conv_w; ca.bias = conv_bias; ca.prev = conv_prev;
    ca.u = tmp; ca.du = tmp + nx; ca.dx = dx; ca.dw = dconv_w; ca.dbias = dconv_bias;
    ca.dprev = conv_k > 1 ? dconv_prev : nullptr;
    ca.batch = s->batch; ca.dim = s->dim; ca.K = conv_k; ca.silu = conv_silu != 0; ca.L = L;
    rc = conv_run(ca, s->in_dtype, false, st);
    if (rc == MAMBA_OK)
        rc = scan_bwd_impl(s, discretization, tmp, delta, A, B, C, D, z, delta_bias, softplus_flag, h0, dy, dlast_state,
                           tmp + nx, ddelta, dz, dA, dB, dC, dD, ddelta_bias, dh0, stream);
    if (rc == MAMBA_OK) rc = conv_run(ca, s->in_dtype, true, st);
    e = cudaFreeAsync(tmp, st);
    if (rc == MAMBA_OK && e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync (convolution scratch)");
    return rc;
}

extern "C" const char* mamba_scan_last_error(void) { return t_err.c_str(); }

extern "C" int mamba_scan_version(void) { return MAMBA_SCAN_VERSION; }

extern "C" long long mamba_scan_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int mamba_scan_device_status(void* stream) {
    t_err.clear();
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    // the forward units hold the kernels with bounded waits; each unit has its own status word
    const int v[4] = {fwd_lane_status_t<float>(true), fwd_lane_status_t<uint16_t>(true),
                      fwd_warp_status_t<float>(true), fwd_warp_status_t<uint16_t>(true)};
    bool timed_out = false;
    for (int x : v) {
        if (x < 0) return fail(MAMBA_ERR_CUDA, "reading the device status word failed");
        timed_out = timed_out || x != 0;
    }
    if (timed_out) return fail(MAMBA_ERR_TIMEOUT, "a kernel abandoned a bounded wait for an asynchronous copy");
    return MAMBA_OK;
}
