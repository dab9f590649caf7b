// mxnorm_warp_fp8_h16.cu -- warp-row kernels for the MXNorm pass for FP8
// E4M3 codes after the 16-point Hadamard rotation.  One format per
// translation unit, so the formats compile in parallel.
#include "mx_warp.cuh"

namespace mxnorm {

cudaError_t launch_warp_row_e4m3_h16(const WarpRowArgs& a, cudaStream_t s) {
  return warp_row::launch_fmt<kFmtE4M3H16, true>(a, s);
}

}  // namespace mxnorm
