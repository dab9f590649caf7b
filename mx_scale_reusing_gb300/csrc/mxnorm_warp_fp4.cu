// mxnorm_warp_fp4.cu -- warp-row kernels for the FP4 E2M1 formats (plain,
// H16, H32).
#include "mx_warp.cuh"

namespace mxnorm {

cudaError_t launch_warp_row_fp4(const WarpRowArgs& a, cudaStream_t s) {
  using namespace warp_row;
  switch (a.fmt) {
    case kFmtE2M1: return launch_fmt<kFmtE2M1, true>(a, s);
    case kFmtE2M1H16: return launch_fmt<kFmtE2M1H16, true>(a, s);
    case kFmtE2M1H32: return launch_fmt<kFmtE2M1H32, true>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mxnorm
