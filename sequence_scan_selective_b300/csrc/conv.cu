// Causal depthwise convolution kernels for the backward pass of the fused block: launches of
// conv_fwd_kernel (u for the recomputation) and conv_bwd_kernel (gradients through it).
#include "host.cuh"
#include "conv.cuh"

namespace mscan {

template <typename TIn>
static int conv_launch(const ConvArgs& a, bool backward, cudaStream_t st) {
    const long long rows = (long long)a.batch * a.dim;
    const long long grid = rows * a.ntile;
    if (grid > 0x7fffffffLL) return fail(MAMBA_ERR_ARG, "too many convolution tiles");
    if (backward)
        conv_bwd_kernel<TIn><<<(unsigned)grid, kConvThreads, 0, st>>>(a);
    else
        conv_fwd_kernel<TIn><<<(unsigned)grid, kConvThreads, 0, st>>>(a);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, backward ? "conv_bwd_kernel launch" : "conv_fwd_kernel launch");
    return MAMBA_OK;
}

int conv_run(const ConvArgs& a_in, int in_dtype, bool backward, cudaStream_t st) {
    ConvArgs a = a_in;
    a.ntile = (a.L + kConvTile - 1) / kConvTile;
    if (a.L == 0) return MAMBA_OK;
    return in_dtype == MAMBA_BF16 ? conv_launch<uint16_t>(a, backward, st) : conv_launch<float>(a, backward, st);
}

}  // namespace mscan
