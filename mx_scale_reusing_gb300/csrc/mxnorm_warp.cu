// mxnorm_warp.cu -- dispatch of the warp-row MXNorm kernel by format
// (kernel templates in mx_warp.cuh).
#include "mx_warp.cuh"

namespace mxnorm {

cudaError_t launch_mxnorm_warp_row(const WarpRowArgs& a, cudaStream_t s) {
  switch (a.fmt) {
    case kFmtE4M3: return launch_warp_row_e4m3(a, s);
    case kFmtE4M3H16: return launch_warp_row_e4m3_h16(a, s);
    case kFmtE4M3H32: return launch_warp_row_e4m3_h32(a, s);
    case kFmtE2M1: return launch_warp_row_e2m1(a, s);
    case kFmtE2M1H16: return launch_warp_row_e2m1_h16(a, s);
    case kFmtE2M1H32: return launch_warp_row_e2m1_h32(a, s);
    default: return cudaErrorInvalidValue;
  }
}

// The cast alone (E4M3 only: kernel 2 of the two-pass baseline).
cudaError_t launch_mx_cast_warp_row(const WarpRowArgs& a, cudaStream_t s) {
  if (a.fmt != kFmtE4M3) return cudaErrorInvalidValue;
  return launch_warp_row_e4m3_cast(a, s);
}

}  // namespace mxnorm
