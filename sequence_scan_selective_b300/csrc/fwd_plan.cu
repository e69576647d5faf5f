// Host-side queries of the forward planners (no launch, no allocation): the number of segments
// of the time axis each forward kernel's planner picks for a shape.  mamba_scan.cu uses them to
// tell beforehand whether the training forward pass keeps checkpoints (it does only unsplit).
#include "fwd_lane.cuh"
#include "fwd_warp.cuh"

namespace mscan {

template <typename TIn>
int fwd_lane_nseg_t(const mamba_scan_shape* s) {
    if (s->dstate > 16) return fail(MAMBA_ERR_ARG, "the channel-per-lane kernel takes N <= 16");
    FwdPlan p;
    const int rc = s->dstate <= 8 ? plan_cl<TIn, 8>(s, sm_count(), p) : plan_cl<TIn, 16>(s, sm_count(), p);
    return rc ? rc : p.nseg;
}

template <typename TIn>
int fwd_warp_nseg_t(const mamba_scan_shape* s) {
    FwdPlan p;
    const int nsm = sm_count();
    const int rc = s->dstate <= 16 ? plan_warp<TIn, 16>(s, nsm, p)
                   : s->dstate <= 32 ? plan_warp<TIn, 32>(s, nsm, p) : plan_warp<TIn, 64>(s, nsm, p);
    return rc ? rc : p.nseg;
}

template int fwd_lane_nseg_t<float>(const mamba_scan_shape*);
template int fwd_lane_nseg_t<uint16_t>(const mamba_scan_shape*);
template int fwd_warp_nseg_t<float>(const mamba_scan_shape*);
template int fwd_warp_nseg_t<uint16_t>(const mamba_scan_shape*);

}  // namespace mscan
