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
// device memory.  The first call on each device (with that device current)
// resolves the array's device address once with cudaGetSymbolAddress and
// caches it; that first call should come before any stream capture.
#include <mutex>

#include "launch.h"
#include "mx_device.cuh"
#include "mxnorm.h"

namespace mxnorm {
namespace {

constexpr size_t kStaticWsBytes = MXNORM_STATIC_WS_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_ws_mu;
void* g_ws_ptr[kMaxDevices] = {};

int static_fail(int status, const char* msg) {
  set_last_error(msg);
  return status;
}

// Device address of the workspace on the current device (resolved once).
cudaError_t workspace_on_current_device(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (g_ws_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_static_ws);
    if (err != cudaSuccess) return err;
    g_ws_ptr[dev] = p;
  }
  *out = g_ws_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace mxnorm

using namespace mxnorm;

extern "C" int rmsnorm_mxfp8_ref_fwd_static_ws(const void* x, int64_t T, int64_t H, float eps,
                                               uint8_t* codes, uint8_t* scales, float* inv_rms,
                                               void* stream) {
  set_last_error("");
  if (T < 0 || H <= 0 || H % kBlock != 0)
    return static_fail(MXNORM_ERR_INVALID_ARG, "T must be >= 0 and H a positive multiple of 32");
  if (!(eps >= 0.0f)) return static_fail(MXNORM_ERR_INVALID_ARG, "eps must be >= 0");
  if (H > MXNORM_MAX_H || T > (int64_t)(kStaticWsBytes / 2) / H)
    return static_fail(MXNORM_ERR_UNSUPPORTED,
                       "T * H exceeds the static workspace (MXNORM_STATIC_WS_BYTES / 2 bf16 elements)");
  if (T == 0) return MXNORM_OK;
  if (!x || !codes || !scales || !inv_rms) return static_fail(MXNORM_ERR_INVALID_ARG, "NULL pointer argument");
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(codes) & 15) ||
      (reinterpret_cast<uintptr_t>(inv_rms) & 3))
    return static_fail(MXNORM_ERR_MISALIGNED, "x and codes need 16-byte, inv_rms 4-byte alignment");
  void* ws = nullptr;
  cudaError_t err = workspace_on_current_device(&ws);
  if (err != cudaSuccess) return static_fail(MXNORM_ERR_CUDA, cudaGetErrorString(err));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  err = launch_rmsnorm_bf16(RmsNormArgs{x, T, H, eps, ws, inv_rms}, s);
  if (err != cudaSuccess) return static_fail(MXNORM_ERR_CUDA, cudaGetErrorString(err));
  err = launch_mx_cast_warp_row(WarpRowArgs{ws, T, H, 2, MXNORM_FMT_MXFP8_E4M3, codes, scales, nullptr}, s);
  if (err != cudaSuccess) return static_fail(MXNORM_ERR_CUDA, cudaGetErrorString(err));
  return MXNORM_OK;
}
