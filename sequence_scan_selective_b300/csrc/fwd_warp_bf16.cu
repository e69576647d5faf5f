// Four-lanes-per-channel forward scan for bf16 inputs (one device module per input type).
#include "fwd_warp.cuh"

namespace mscan {
template int fwd_warp_run_t<uint16_t>(const mamba_scan_shape*, const FwdArgs&, bool, bool, float2*, size_t, cudaStream_t);
template int fwd_warp_status_t<uint16_t>(bool);
}  // namespace mscan
