// rmsnorm_static_ws.cu -- the two-pass RMSNorm-then-MXFP8 baseline for
// callers that must not allocate device memory.
//
// rmsnorm_mxfp8_ref_fwd needs a bf16 [T, H] workspace between its two
// kernels and takes it from the caller.  Some callers cannot provide one:
// code living inside a host framework that owns every device allocation
// through its own pool and forbids side allocations, code on a
// latency-critical path where cudaMalloc's implicit device synchronisation
// is not acceptable, or code that must run under a device-memory budget
// fixed up front.  For them this entry point keeps the workspace in a
// file-scope device array compiled into the library, so the call itself
// allocates nothing.
//
// Cost and limits: the array is MXNORM_STATIC_WS_BYTES (32 MiB, i.e.
// T * H <= 16,777,216 bf16 elements) and every GPU that loads this part of
// the library holds it until the process exits.  All calls on a device
// share the one array, so calls whose work overlaps on the GPU (different
// streams, or several host threads) race on it; callers must serialise
// them.  Every element the second kernel reads is written by the first
// kernel of the same call, so nothing has to start at zero.
//
// Device address: in host code `g_static_ws` names a host-side shadow, not
// device memory.  Every call looks up the array's address in the current
// device's context with cudaGetSymbolAddress (a host-side lookup; no device
// work), so the address stays right after cudaDeviceReset or under another
// context on the same device.  The first call on a device may load the
// module into that context: make it before any stream capture.
#include "launch.h"
#include "mx_device.cuh"
#include "mxnorm.h"

namespace mxnorm {
namespace {

constexpr size_t kStaticWsBytes = MXNORM_STATIC_WS_BYTES;

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

int static_fail(int status, const char* msg) {
  set_last_error(msg);
  return status;
}

}  // namespace
}  // namespace mxnorm

using namespace mxnorm;

extern "C" int rmsnorm_mxfp8_ref_fwd_static_ws(const void* x, int64_t T, int64_t H, float eps,
                                               uint8_t* codes, uint8_t* scales, float* inv_rms,
                                               void* stream) {
  set_last_error("");
  if (!(eps >= 0.0f)) return static_fail(MXNORM_ERR_INVALID_ARG, "eps must be >= 0");
  const int st = check_common(x, T, H, codes, scales, inv_rms);
  if (st != MXNORM_OK) return st;
  if (T > (int64_t)(kStaticWsBytes / 2) / H)
    return static_fail(MXNORM_ERR_UNSUPPORTED,
                       "T * H exceeds the static workspace (MXNORM_STATIC_WS_BYTES / 2 bf16 elements)");
  if (T == 0) return MXNORM_OK;
  void* ws = nullptr;
  cudaError_t err = cudaGetSymbolAddress(&ws, g_static_ws);
  if (err != cudaSuccess) return static_fail(MXNORM_ERR_CUDA, cudaGetErrorString(err));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  err = launch_rmsnorm_bf16(RmsNormArgs{x, T, H, eps, ws, inv_rms}, s);
  if (err != cudaSuccess) return static_fail(MXNORM_ERR_CUDA, cudaGetErrorString(err));
  err = launch_mx_cast_warp_row(WarpRowArgs{ws, T, H, 2, MXNORM_FMT_MXFP8_E4M3, codes, scales, nullptr}, s);
  if (err != cudaSuccess) return static_fail(MXNORM_ERR_CUDA, cudaGetErrorString(err));
  return MXNORM_OK;
}
