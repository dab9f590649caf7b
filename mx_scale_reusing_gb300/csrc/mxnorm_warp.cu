// mxnorm_warp.cu -- dispatch of the warp-row MXNorm kernel by format
// family (kernel templates in mx_warp.cuh).
#include "mx_warp.cuh"

namespace mxnorm {

cudaError_t launch_mxnorm_warp_row(const WarpRowArgs& a, cudaStream_t s) {
  switch (a.fmt) {
    case kFmtE4M3:
    case kFmtE4M3H16:
    case kFmtE4M3H32: return launch_warp_row_fp8(a, s, true);
    case kFmtE2M1:
    case kFmtE2M1H16:
    case kFmtE2M1H32: return launch_warp_row_fp4(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_mx_cast_warp_row(const WarpRowArgs& a, cudaStream_t s) {
  return launch_warp_row_fp8(a, s, false);
}

}  // namespace mxnorm
