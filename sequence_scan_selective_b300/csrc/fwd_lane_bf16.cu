// Channel-per-lane forward scan for bf16 inputs (one device module per input type).
#include "fwd_lane.cuh"

namespace mscan {
template int fwd_lane_run_t<uint16_t>(const mamba_scan_shape*, const FwdArgs&, bool, float2*, size_t, cudaStream_t);
template int fwd_lane_status_t<uint16_t>(bool);
}  // namespace mscan
