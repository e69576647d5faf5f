// Backward pass: launches of scan_bwd_kernel (per block of 16 states; with a split time axis, the
// carry, full and correction launches) and of the final conversion of the fp32 accumulators.
#include "host.cuh"
#include "scan_bwd.cuh"

namespace mscan {

// Register budget of the launch: 3 CTAs per SM (the reverse walk keeps each step's Abar) when
// the grid fits in one wave of 3 per SM and the simplified discretisation is used, else 4.
// MAMBA_SCAN_BWD_MINB=3 or =4 forces one (tests).
static int bwd_minb(long long ctas) {
    const int force = env_int("MAMBA_SCAN_BWD_MINB", 0);
    if (force == 3 || force == 4) return force;
    return ctas <= 3LL * sm_count() ? 3 : 4;
}

template <typename TIn, bool ZOH, int MODE>
static int bwd_launch(const BwdArgs& a, bool vec, unsigned nz, cudaStream_t st) {
    static AttrCache attr[2][2];
    const dim3 grid((unsigned)((a.dim + bwd::kCh - 1) / bwd::kCh), (unsigned)a.batch, nz);
    auto kern = vec ? scan_bwd_kernel<TIn, true, ZOH, MODE, 4> : scan_bwd_kernel<TIn, false, ZOH, MODE, 4>;
    bool three = false;
    if constexpr (!ZOH && MODE != bwd::kCarry) {
        three = bwd_minb((long long)grid.x * grid.y * grid.z) == 3;
        if (three) kern = vec ? scan_bwd_kernel<TIn, true, ZOH, MODE, 3> : scan_bwd_kernel<TIn, false, ZOH, MODE, 3>;
    }
    int rc = allow_smem(kern, attr[vec ? 1 : 0][three ? 1 : 0]);
    if (rc) return rc;
    kern<<<grid, bwd::kThreads, bwd::Layout<TIn>::BYTES, st>>>(a);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "scan_bwd_kernel launch");
    return MAMBA_OK;
}

template <typename TIn, bool ZOH>
static int bwd_block(const BwdArgs& a, bool vec, cudaStream_t st) {
    const unsigned S = (unsigned)a.nseg;
    int rc = MAMBA_OK;
    if (S > 1) rc = bwd_launch<TIn, ZOH, bwd::kCarry>(a, vec, S, st);
    if (rc == MAMBA_OK) rc = bwd_launch<TIn, ZOH, bwd::kFull>(a, vec, S, st);
    if (rc == MAMBA_OK && S > 1) rc = bwd_launch<TIn, ZOH, bwd::kCorr>(a, vec, S - 1, st);
    return rc;
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

// One pass per block of 16 states, in order.  With more than one block or a split time axis the
// per-(channel, step) gradients are summed in fp32 accumulators (for fp32 storage the outputs
// themselves) and, for bf16 storage, converted at the end.
int bwd_run(const BwdArgs& a_in, int in_dtype, bool zoh, bool vec, cudaStream_t st) {
    BwdArgs a = a_in;
    const bool bf = in_dtype == MAMBA_BF16;
    for (int nb = 0; nb < a.dstate; nb += bwd::kNS) {
        a.nb = nb;
        int rc = bf ? (zoh ? bwd_block<uint16_t, true>(a, vec, st) : bwd_block<uint16_t, false>(a, vec, st))
                    : (zoh ? bwd_block<float, true>(a, vec, st) : bwd_block<float, false>(a, vec, st));
        if (rc) return rc;
    }
    if (a.acc_du == nullptr || !bf) return MAMBA_OK;
    return finish_launch<uint16_t>(a, st);
}

}  // namespace mscan
