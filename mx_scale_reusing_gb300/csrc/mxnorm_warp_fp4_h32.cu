// mxnorm_warp_fp4_h32.cu -- warp-row kernels for the MXNorm pass for FP4
// E2M1 codes after the 32-point Hadamard rotation.  One format per
// translation unit, so the formats compile in parallel.
#include "mx_warp.cuh"

namespace mxnorm {

cudaError_t launch_warp_row_e2m1_h32(const WarpRowArgs& a, cudaStream_t s) {
  return warp_row::launch_fmt<kFmtE2M1H32, true>(a, s);
}

}  // namespace mxnorm
