// Four-lanes-per-channel forward scan for fp32 inputs (one device module per input type).
#include "fwd_warp.cuh"

namespace mscan {
template int fwd_warp_run_t<float>(const mamba_scan_shape*, const FwdArgs&, bool, bool, float2*, size_t, cudaStream_t);
template int fwd_warp_status_t<float>(bool);
}  // namespace mscan
