// Decoding step: launch of state_step_kernel.
#include "host.cuh"
#include "state_step.cuh"

namespace mscan {

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
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "state_step_kernel launch");
    return MAMBA_OK;
}

int step_run(const StepArgs& a, int in_dtype, cudaStream_t st) {
    const bool bf = in_dtype == MAMBA_BF16;
    if (a.dstate <= 4) return bf ? step_dispatch<uint16_t, 4>(a, st) : step_dispatch<float, 4>(a, st);
    if (a.dstate <= 16) return bf ? step_dispatch<uint16_t, 16>(a, st) : step_dispatch<float, 16>(a, st);
    if (a.dstate <= 32) return bf ? step_dispatch<uint16_t, 32>(a, st) : step_dispatch<float, 32>(a, st);
    return bf ? step_dispatch<uint16_t, 64>(a, st) : step_dispatch<float, 64>(a, st);
}

}  // namespace mscan
