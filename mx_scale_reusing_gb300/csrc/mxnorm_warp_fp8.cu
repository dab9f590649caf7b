// mxnorm_warp_fp8.cu -- warp-row kernels for the FP8 E4M3 formats (plain,
// H16, H32), and the cast-only E4M3 form used by the two-pass baseline.
#include "mx_warp.cuh"

namespace mxnorm {

cudaError_t launch_warp_row_fp8(const WarpRowArgs& a, cudaStream_t s, bool estimate) {
  using namespace warp_row;
  if (!estimate) {
    if (a.fmt != kFmtE4M3) return cudaErrorInvalidValue;
    return launch_fmt<kFmtE4M3, false>(a, s);
  }
  switch (a.fmt) {
    case kFmtE4M3: return launch_fmt<kFmtE4M3, true>(a, s);
    case kFmtE4M3H16: return launch_fmt<kFmtE4M3H16, true>(a, s);
    case kFmtE4M3H32: return launch_fmt<kFmtE4M3H32, true>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mxnorm
