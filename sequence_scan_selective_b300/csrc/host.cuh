// Host-side helpers shared by the library's translation units, and the entry points each unit
// exports to the C ABI in mamba_scan.cu.
//
// Units: mamba_scan.cu (C ABI, argument checks, kernel choice), fwd_lane_{f32,bf16}.cu
// (channel-per-lane forward scan and its split-sequence second launch), fwd_warp_{f32,bf16}.cu
// (four-lanes-per-channel forward scan), fwd_plan.cu (the forward planners' segment counts,
// host-side), bwd.cu (backward pass), conv.cu (causal convolution for the block's backward pass),
// step.cu (decoding step).  Each compiles to its own device module.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>

#include "mamba_scan.h"

namespace mscan {

struct FwdArgs;
struct StepArgs;
struct BwdArgs;
struct ConvArgs;

// ---------------------------------------------------------------------------- errors, counters
int fail(int code, const char* fmt, ...);           // records the message; returns code
int cuda_fail(cudaError_t e, const char* what);     // MAMBA_ERR_CUDA with the CUDA error text
void count_launch();                                // one of this library's kernels was launched

// ---------------------------------------------------------------------------- device and memory
int sm_count();                                     // SMs of the current device
unsigned long long current_context_id();            // unique id of the current context (0: none)
int env_int(const char* name, int dflt);
bool overlaps(const void* a, size_t na, const void* b, size_t nb);
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------- TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();      // NULL when the driver lacks the entry point
// 3-D map over a dense [d2][d1][d0] tensor (d0 contiguous), box [b1 rows x b0 cols], 128-byte
// swizzle (b0 * esize must be 128).
bool encode_3d(CUtensorMap* m, const void* base, int esize, long long d0, long long d1, long long d2, int b0,
               int b1);

// ---------------------------------------------------------------------------- shared memory opt-in
constexpr int kSmemLimit = 227 * 1024;

// Raises a kernel's dynamic shared memory limit once per CUDA context (the attribute belongs to
// the function in one context; setting it on every call costs tens of microseconds of host time).
struct AttrCache {
    std::atomic<unsigned long long> ctx[8] = {};
};

template <typename K>
int allow_smem(K kern, AttrCache& cache) {
    const unsigned long long id = current_context_id();
    if (id != 0)
        for (auto& c : cache.ctx)
            if (c.load(std::memory_order_acquire) == id) return MAMBA_OK;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    if (id != 0) cache.ctx[id % 8].store(id, std::memory_order_release);
    return MAMBA_OK;
}

// Reads (and with `clear`, resets) a unit's copy of the device status word; -1 if CUDA fails.
template <typename T>
int read_status(const T& symbol, bool clear) {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, symbol, sizeof v) != cudaSuccess) return -1;
    if (v != 0 && clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(symbol, &zero, sizeof zero) != cudaSuccess) return -1;
    }
    return v;
}

// ---------------------------------------------------------------------------- unit entry points
// Forward scan with the channel-per-lane kernel (dstate <= 16) or the four-lanes-per-channel
// kernel (any dstate).  `a` holds the tensors and sizes; the callee plans and launches.  Split
// sequences keep their carries in `scratch` (capacity `cap` bytes) when it is non-NULL, else in
// stream-ordered memory from cudaMallocAsync on `st`.
// Instantiated for TIn = float and uint16_t (bf16 bits), one unit each.
template <typename TIn>
int fwd_lane_run_t(const mamba_scan_shape* s, const FwdArgs& a, bool softplus, float2* scratch, size_t cap,
                   cudaStream_t st);
template <typename TIn>
int fwd_warp_run_t(const mamba_scan_shape* s, const FwdArgs& a, bool softplus, bool gate, float2* scratch,
                   size_t cap, cudaStream_t st);
// Segments of the time axis that the forward planner of each kernel picks for a shape (negative:
// an error code).  Host-only: no launch, no allocation.  In fwd_plan.cu.
template <typename TIn>
int fwd_lane_nseg_t(const mamba_scan_shape* s);
template <typename TIn>
int fwd_warp_nseg_t(const mamba_scan_shape* s);
template <typename TIn>
int fwd_lane_status_t(bool clear);
template <typename TIn>
int fwd_warp_status_t(bool clear);
// Decoding step (dtype MAMBA_F32 or MAMBA_BF16).
int step_run(const StepArgs& a, int in_dtype, cudaStream_t st);
// Backward pass launch (checkpoints already in a.ckpt).
int bwd_run(const BwdArgs& a, int in_dtype, bool zoh, bool vec, cudaStream_t st);
// Causal convolution: u from x (backward = false) or the gradients through it (backward = true).
int conv_run(const ConvArgs& a, int in_dtype, bool backward, cudaStream_t st);

}  // namespace mscan
