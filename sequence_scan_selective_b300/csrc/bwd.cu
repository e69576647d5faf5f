// Backward pass: launch of scan_bwd_kernel.
#include "host.cuh"
#include "scan_bwd.cuh"

namespace mscan {

template <typename TIn, bool ZOH>
static int bwd_launch(const BwdArgs& a, bool vec, cudaStream_t st) {
    static AttrCache attr_vec, attr_scalar;
    auto kern = vec ? scan_bwd_kernel<TIn, true, ZOH> : scan_bwd_kernel<TIn, false, ZOH>;
    int rc = allow_smem(kern, vec ? attr_vec : attr_scalar);
    if (rc) return rc;
    const dim3 grid((unsigned)((a.dim + bwd::kCh - 1) / bwd::kCh), (unsigned)a.batch);
    kern<<<grid, bwd::kThreads, bwd::Layout<TIn>::BYTES, st>>>(a);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "scan_bwd_kernel launch");
    return MAMBA_OK;
}

template <typename TIn>
static int finish_launch(const BwdArgs& a, cudaStream_t st) {
    const long long n = (long long)a.batch * a.dim * a.L;
    long long blocks = (n + 255) / 256;
    if (blocks > 148LL * 64) blocks = 148LL * 64;
    bwd_finish_kernel<TIn><<<(unsigned)blocks, 256, 0, st>>>(a, n);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "bwd_finish_kernel launch");
    return MAMBA_OK;
}

// One launch per block of 16 states, in order; with more than one block the per-(channel, step)
// gradients go through the fp32 accumulators in `a` and a final conversion.
int bwd_run(const BwdArgs& a_in, int in_dtype, bool zoh, bool vec, cudaStream_t st) {
    BwdArgs a = a_in;
    const bool bf = in_dtype == MAMBA_BF16;
    for (int nb = 0; nb < a.dstate; nb += bwd::kNS) {
        a.nb = nb;
        int rc = bf ? (zoh ? bwd_launch<uint16_t, true>(a, vec, st) : bwd_launch<uint16_t, false>(a, vec, st))
                    : (zoh ? bwd_launch<float, true>(a, vec, st) : bwd_launch<float, false>(a, vec, st));
        if (rc) return rc;
    }
    if (a.acc_du == nullptr) return MAMBA_OK;
    return bf ? finish_launch<uint16_t>(a, st) : finish_launch<float>(a, st);
}

}  // namespace mscan
