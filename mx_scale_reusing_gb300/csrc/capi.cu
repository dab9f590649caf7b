// capi.cu -- the extern "C" boundary of libmxnorm: argument validation,
// variant selection and launches.  Declarations and the full contract are
// in include/mxnorm.h.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "launch.h"
#include "mx_device.cuh"
#include "mxnorm.h"

namespace mxnorm {

namespace {

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return status;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

std::mutex g_grid_mu;
std::map<std::tuple<int, const void*, int, size_t>, int> g_grid_cache;  // -> CTAs per device fill

int cuda_fail(cudaError_t err, const char* what) {
  return fail(MXNORM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

}  // namespace

int check_common(const void* x, int64_t T, int64_t H, const void* codes, const void* scales,
                 const void* inv_rms) {
  if (T < 0) return fail(MXNORM_ERR_INVALID_ARG, "T = %lld < 0", (long long)T);
  if (H <= 0 || H % kBlock != 0)
    return fail(MXNORM_ERR_INVALID_ARG, "H = %lld is not a positive multiple of 32", (long long)H);
  if (H > MXNORM_MAX_H)
    return fail(MXNORM_ERR_UNSUPPORTED, "H = %lld exceeds MXNORM_MAX_H = %d", (long long)H, MXNORM_MAX_H);
  if (T == 0) return MXNORM_OK;
  if (!x || !codes || !scales || !inv_rms) return fail(MXNORM_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(x, 16)) return fail(MXNORM_ERR_MISALIGNED, "x is not 16-byte aligned");
  if (!aligned(codes, 16)) return fail(MXNORM_ERR_MISALIGNED, "codes is not 16-byte aligned");
  if (!aligned(inv_rms, 4)) return fail(MXNORM_ERR_MISALIGNED, "inv_rms is not 4-byte aligned");
  return MXNORM_OK;
}

void set_last_error(const char* msg) { g_last_error = msg; }

bool is_device_memory(const void* p) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    (void)cudaGetLastError();  // leave no sticky error behind for the launch check
    return false;
  }
  return attr.type == cudaMemoryTypeDevice;
}

int persistent_grid(const void* kernel, int threads, int64_t work_ctas, size_t dyn_smem) {
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, kernel, threads, dyn_smem);
  int fill = 0;
  {
    std::lock_guard<std::mutex> lk(g_grid_mu);
    auto it = g_grid_cache.find(key);
    if (it != g_grid_cache.end()) fill = it->second;
  }
  if (fill == 0) {
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, dyn_smem);
    fill = (sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
    std::lock_guard<std::mutex> lk(g_grid_mu);
    g_grid_cache[key] = fill;
  }
  int64_t g = work_ctas < fill ? work_ctas : fill;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace mxnorm

using namespace mxnorm;

extern "C" {

int mxnorm_quant_fwd_ex(const void* x, int64_t T, int64_t H, int p, int fmt, void* codes,
                        uint8_t* scales, float* inv_rms, int variant, void* stream) {
  g_last_error.clear();
  if (p != 1 && p != 2) return fail(MXNORM_ERR_INVALID_ARG, "p = %d is not 1 or 2", p);
  if (fmt < 0 || fmt >= kNumFmts) return fail(MXNORM_ERR_INVALID_ARG, "unknown fmt %d", fmt);
  if (variant < MXNORM_VARIANT_AUTO || variant > MXNORM_VARIANT_TILED_TMA)
    return fail(MXNORM_ERR_INVALID_ARG, "unknown variant %d", variant);
  int st = check_common(x, T, H, codes, scales, inv_rms);
  if (st != MXNORM_OK || T == 0) return st;
  if (variant == MXNORM_VARIANT_TILED_TMA && !tiled_supported(H, fmt))
    return fail(MXNORM_ERR_UNSUPPORTED, "tiled variant does not support H = %lld", (long long)H);

  WarpRowArgs a{x, T, H, p, fmt, codes, scales, inv_rms};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool use_tiled = variant == MXNORM_VARIANT_TILED_TMA;
  cudaError_t err = use_tiled ? launch_mxnorm_tiled(TiledArgs{a}, s) : launch_mxnorm_warp_row(a, s);
  if (err != cudaSuccess) return cuda_fail(err, "mxnorm_quant_fwd launch");
  return MXNORM_OK;
}

int mxnorm_tiled_wait_drill(const void* x, int64_t T, int64_t H, void* codes, uint8_t* scales, float* inv_rms,
                            int64_t withheld_tile, int64_t wait_limit_ns, void* stream) {
  g_last_error.clear();
  int st = check_common(x, T, H, codes, scales, inv_rms);
  if (st != MXNORM_OK) return st;
  if (T == 0) return fail(MXNORM_ERR_INVALID_ARG, "the drill needs at least one row");
  if (!tiled_supported(H, MXNORM_FMT_MXFP8_E4M3))
    return fail(MXNORM_ERR_UNSUPPORTED, "tiled variant does not support H = %lld", (long long)H);
  const int64_t ntiles = (T + 7) / 8;
  if (withheld_tile < 0 || withheld_tile >= ntiles)
    return fail(MXNORM_ERR_INVALID_ARG, "withheld_tile = %lld is not in [0, %lld)", (long long)withheld_tile,
                (long long)ntiles);
  if (wait_limit_ns < 100000 || wait_limit_ns > 1000000000)
    return fail(MXNORM_ERR_INVALID_ARG, "wait_limit_ns = %lld is not in [1e5, 1e9]", (long long)wait_limit_ns);
  TiledArgs t{WarpRowArgs{x, T, H, 2, MXNORM_FMT_MXFP8_E4M3, codes, scales, inv_rms}};
  t.wait_limit_ns = (unsigned long long)wait_limit_ns;
  t.withheld_tile = withheld_tile;
  cudaError_t err = launch_mxnorm_tiled(t, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "mxnorm_tiled_wait_drill launch");
  return MXNORM_OK;
}

int64_t mxnorm_mma_scale_bytes(int64_t rows, int64_t H) {
  if (rows < 0 || H <= 0 || H % 128 != 0) return -1;
  return ((rows + 127) / 128) * (H / 128) * 512;
}

int mxnorm_quant_fwd_layout(const void* x, int64_t T, int64_t H, int p, int fmt, void* codes, uint8_t* scales,
                            float* inv_rms, int scale_layout, void* stream) {
  if (scale_layout == MXNORM_SCALE_ROW_MAJOR)
    return mxnorm_quant_fwd_ex(x, T, H, p, fmt, codes, scales, inv_rms, MXNORM_VARIANT_AUTO, stream);
  g_last_error.clear();
  if (scale_layout != MXNORM_SCALE_MMA) return fail(MXNORM_ERR_INVALID_ARG, "unknown scale_layout %d", scale_layout);
  if (p != 1 && p != 2) return fail(MXNORM_ERR_INVALID_ARG, "p = %d is not 1 or 2", p);
  if (fmt < 0 || fmt >= kNumFmts) return fail(MXNORM_ERR_INVALID_ARG, "unknown fmt %d", fmt);
  int st = check_common(x, T, H, codes, scales, inv_rms);
  if (st != MXNORM_OK || T == 0) return st;
  if (H % 128 != 0) return fail(MXNORM_ERR_INVALID_ARG, "the MMA scale layout needs H %% 128 == 0 (H = %lld)", (long long)H);
  WarpRowArgs a{x, T, H, p, fmt, codes, scales, inv_rms};
  a.scale_tiled = 1;
  cudaError_t err = launch_mxnorm_warp_row(a, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "mxnorm_quant_fwd_layout launch");
  return MXNORM_OK;
}

int mx_cast_fwd(const void* x, int64_t T, int64_t H, int fmt, void* codes, uint8_t* scales, int scale_layout,
                void* stream) {
  g_last_error.clear();
  if (fmt != MXNORM_FMT_MXFP8_E4M3) return fail(MXNORM_ERR_UNSUPPORTED, "mx_cast_fwd supports MXFP8 E4M3 only");
  if (scale_layout != MXNORM_SCALE_ROW_MAJOR && scale_layout != MXNORM_SCALE_MMA)
    return fail(MXNORM_ERR_INVALID_ARG, "unknown scale_layout %d", scale_layout);
  if (T < 0) return fail(MXNORM_ERR_INVALID_ARG, "T = %lld < 0", (long long)T);
  if (H <= 0 || H % kBlock != 0)
    return fail(MXNORM_ERR_INVALID_ARG, "H = %lld is not a positive multiple of 32", (long long)H);
  if (H > MXNORM_MAX_H)
    return fail(MXNORM_ERR_UNSUPPORTED, "H = %lld exceeds MXNORM_MAX_H = %d", (long long)H, MXNORM_MAX_H);
  if (scale_layout == MXNORM_SCALE_MMA && H % 128 != 0)
    return fail(MXNORM_ERR_INVALID_ARG, "the MMA scale layout needs H %% 128 == 0 (H = %lld)", (long long)H);
  if (T == 0) return MXNORM_OK;
  if (!x || !codes || !scales) return fail(MXNORM_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(x, 16) || !aligned(codes, 16)) return fail(MXNORM_ERR_MISALIGNED, "x and codes need 16-byte alignment");
  WarpRowArgs a{x, T, H, 2, fmt, codes, scales, nullptr};
  a.scale_tiled = scale_layout == MXNORM_SCALE_MMA;
  cudaError_t err = launch_mx_cast_warp_row(a, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "mx_cast_fwd launch");
  return MXNORM_OK;
}

int mx_cast_gain_fwd(const void* w, int64_t N, int64_t K, const float* gamma, float c, void* codes,
                     uint8_t* scales, int scale_layout, void* stream) {
  g_last_error.clear();
  if (scale_layout != MXNORM_SCALE_ROW_MAJOR && scale_layout != MXNORM_SCALE_MMA)
    return fail(MXNORM_ERR_INVALID_ARG, "unknown scale_layout %d", scale_layout);
  if (N < 0) return fail(MXNORM_ERR_INVALID_ARG, "N = %lld < 0", (long long)N);
  if (K <= 0 || K % kBlock != 0)
    return fail(MXNORM_ERR_INVALID_ARG, "K = %lld is not a positive multiple of 32", (long long)K);
  if (K > MXNORM_MAX_H)
    return fail(MXNORM_ERR_UNSUPPORTED, "K = %lld exceeds MXNORM_MAX_H = %d", (long long)K, MXNORM_MAX_H);
  if (scale_layout == MXNORM_SCALE_MMA && K % 128 != 0)
    return fail(MXNORM_ERR_INVALID_ARG, "the MMA scale layout needs K %% 128 == 0 (K = %lld)", (long long)K);
  if (!std::isfinite(c)) return fail(MXNORM_ERR_INVALID_ARG, "c is not finite");
  if (N == 0) return MXNORM_OK;
  if (!w || !gamma || !codes || !scales) return fail(MXNORM_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(w, 16) || !aligned(gamma, 16) || !aligned(codes, 16))
    return fail(MXNORM_ERR_MISALIGNED, "w, gamma and codes need 16-byte alignment");
  GainCastArgs a{w, N, K, gamma, c, codes, scales, scale_layout == MXNORM_SCALE_MMA};
  cudaError_t err = launch_mx_cast_gain(a, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "mx_cast_gain_fwd launch");
  return MXNORM_OK;
}

int mxnorm_linear_fwd(const void* x_codes, const uint8_t* x_scales, const float* inv_rms, const void* w_codes,
                      const uint8_t* w_scales, int64_t T, int64_t K, int64_t N, void* out, void* stream) {
  g_last_error.clear();
  if (T < 0) return fail(MXNORM_ERR_INVALID_ARG, "T = %lld < 0", (long long)T);
  if (K <= 0 || K % 128 != 0) return fail(MXNORM_ERR_INVALID_ARG, "K = %lld is not a positive multiple of 128", (long long)K);
  if (N <= 0 || N % 256 != 0) return fail(MXNORM_ERR_INVALID_ARG, "N = %lld is not a positive multiple of 256", (long long)N);
  if (K > MXNORM_MAX_H || N > (1 << 24)) return fail(MXNORM_ERR_UNSUPPORTED, "K or N too large");
  // TMA tile coordinates are 32-bit: the rows of x and of the scale maps
  // (4 per 512-byte atom, K/128 atoms per 128 rows) must stay below 2^31.
  const int64_t kLimit = int64_t(1) << 31;
  if (T >= kLimit || ((T + 127) / 128) * (K / 32) >= kLimit || ((N + 127) / 128) * (K / 32) >= kLimit)
    return fail(MXNORM_ERR_UNSUPPORTED, "T = %lld, N = %lld, K = %lld exceed the 32-bit tile coordinates",
                (long long)T, (long long)N, (long long)K);
  if (T == 0) return MXNORM_OK;
  if (!x_codes || !x_scales || !inv_rms || !w_codes || !w_scales || !out)
    return fail(MXNORM_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(x_codes, 16) || !aligned(w_codes, 16) || !aligned(x_scales, 16) || !aligned(w_scales, 16) ||
      !aligned(out, 16) || !aligned(inv_rms, 4))
    return fail(MXNORM_ERR_MISALIGNED, "codes, scales and out need 16-byte alignment, inv_rms 4-byte");
  cudaError_t err = launch_mxfp8_linear(LinearArgs{x_codes, x_scales, inv_rms, w_codes, w_scales, T, K, N, out},
                                        static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "mxnorm_linear_fwd launch (tensor maps or launch)");
  return MXNORM_OK;
}

int mxnorm_quant_fwd(const void* x, int64_t T, int64_t H, int p, int fmt, void* codes,
                     uint8_t* scales, float* inv_rms, void* stream) {
  return mxnorm_quant_fwd_ex(x, T, H, p, fmt, codes, scales, inv_rms, MXNORM_VARIANT_AUTO, stream);
}

int rmsnorm_mxfp8_ref_fwd(const void* x, int64_t T, int64_t H, float eps, void* y_workspace,
                          uint8_t* codes, uint8_t* scales, float* inv_rms, void* stream) {
  g_last_error.clear();
  if (!(eps >= 0.0f)) return fail(MXNORM_ERR_INVALID_ARG, "eps must be >= 0");
  int st = check_common(x, T, H, codes, scales, inv_rms);
  if (st != MXNORM_OK || T == 0) return st;
  if (!y_workspace) return fail(MXNORM_ERR_INVALID_ARG, "NULL y_workspace");
  if (!aligned(y_workspace, 16)) return fail(MXNORM_ERR_MISALIGNED, "y_workspace is not 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = launch_rmsnorm_bf16(RmsNormArgs{x, T, H, eps, y_workspace, inv_rms}, s);
  if (err != cudaSuccess) return cuda_fail(err, "rmsnorm kernel launch");
  err = launch_mx_cast_warp_row(WarpRowArgs{y_workspace, T, H, 2, MXNORM_FMT_MXFP8_E4M3, codes, scales, nullptr}, s);
  if (err != cudaSuccess) return cuda_fail(err, "mxfp8 cast kernel launch");
  return MXNORM_OK;
}

int mxnorm_bwd_ste(const void* x, const void* dy, const float* inv_rms, int64_t T, int64_t H, void* dx,
                   void* stream) {
  g_last_error.clear();
  if (T < 0) return fail(MXNORM_ERR_INVALID_ARG, "T = %lld < 0", (long long)T);
  if (H <= 0 || H % kBlock != 0)
    return fail(MXNORM_ERR_INVALID_ARG, "H = %lld is not a positive multiple of 32", (long long)H);
  if (H > MXNORM_MAX_H)
    return fail(MXNORM_ERR_UNSUPPORTED, "H = %lld exceeds MXNORM_MAX_H = %d", (long long)H, MXNORM_MAX_H);
  if (T == 0) return MXNORM_OK;
  if (!x || !dy || !inv_rms || !dx) return fail(MXNORM_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(x, 16) || !aligned(dy, 16) || !aligned(dx, 16))
    return fail(MXNORM_ERR_MISALIGNED, "x, dy and dx must be 16-byte aligned");
  if (!aligned(inv_rms, 4)) return fail(MXNORM_ERR_MISALIGNED, "inv_rms is not 4-byte aligned");
  cudaError_t err = launch_mxnorm_bwd_ste(BwdArgs{x, dy, inv_rms, T, H, dx}, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "mxnorm_bwd_ste launch");
  return MXNORM_OK;
}

int mxnorm_quant_fwd_nvfp4(const void* x, int64_t T, int64_t H, int p, float tensor_scale, void* codes,
                           uint8_t* scales, float* inv_rms, void* stream) {
  g_last_error.clear();
  if (p != 1 && p != 2) return fail(MXNORM_ERR_INVALID_ARG, "p = %d is not 1 or 2", p);
  if (!(tensor_scale > 0.0f) || !(tensor_scale < 3.4028235e38f))
    return fail(MXNORM_ERR_INVALID_ARG, "tensor_scale must be a finite positive float");
  if (T < 0) return fail(MXNORM_ERR_INVALID_ARG, "T = %lld < 0", (long long)T);
  if (H <= 0 || H % 16 != 0)
    return fail(MXNORM_ERR_INVALID_ARG, "H = %lld is not a positive multiple of 16", (long long)H);
  if (H > MXNORM_MAX_H)
    return fail(MXNORM_ERR_UNSUPPORTED, "H = %lld exceeds MXNORM_MAX_H = %d", (long long)H, MXNORM_MAX_H);
  if (T == 0) return MXNORM_OK;
  if (!x || !codes || !scales || !inv_rms) return fail(MXNORM_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(x, 16) || !aligned(codes, 16)) return fail(MXNORM_ERR_MISALIGNED, "x and codes need 16-byte alignment");
  if (!aligned(inv_rms, 4)) return fail(MXNORM_ERR_MISALIGNED, "inv_rms is not 4-byte aligned");
  cudaError_t err = launch_nvfp4(Nvfp4Args{x, T, H, p, tensor_scale, codes, scales, inv_rms},
                                 static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "mxnorm_quant_fwd_nvfp4 launch");
  return MXNORM_OK;
}

int mxnorm_quant_fwd_nvfp4_dev(const void* x, int64_t T, int64_t H, int p, const float* tensor_scale,
                               void* codes, uint8_t* scales, float* inv_rms, void* stream) {
  g_last_error.clear();
  if (p != 1 && p != 2) return fail(MXNORM_ERR_INVALID_ARG, "p = %d is not 1 or 2", p);
  if (T < 0) return fail(MXNORM_ERR_INVALID_ARG, "T = %lld < 0", (long long)T);
  if (H <= 0 || H % 16 != 0)
    return fail(MXNORM_ERR_INVALID_ARG, "H = %lld is not a positive multiple of 16", (long long)H);
  if (H > MXNORM_MAX_H)
    return fail(MXNORM_ERR_UNSUPPORTED, "H = %lld exceeds MXNORM_MAX_H = %d", (long long)H, MXNORM_MAX_H);
  if (T == 0) return MXNORM_OK;
  if (!x || !tensor_scale || !codes || !scales || !inv_rms)
    return fail(MXNORM_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(x, 16) || !aligned(codes, 16)) return fail(MXNORM_ERR_MISALIGNED, "x and codes need 16-byte alignment");
  if (!aligned(inv_rms, 4) || !aligned(tensor_scale, 4))
    return fail(MXNORM_ERR_MISALIGNED, "inv_rms and tensor_scale need 4-byte alignment");
  Nvfp4Args a{x, T, H, p, 1.0f, codes, scales, inv_rms};
  a.g_dev = tensor_scale;
  cudaError_t err = launch_nvfp4(a, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "mxnorm_quant_fwd_nvfp4_dev launch");
  return MXNORM_OK;
}

int mxnorm_nvfp4_tensor_scale(const void* x, int64_t n, float* tensor_scale, void* stream) {
  g_last_error.clear();
  if (n < 0) return fail(MXNORM_ERR_INVALID_ARG, "n < 0");
  if (!tensor_scale || (n > 0 && !x)) return fail(MXNORM_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(tensor_scale, 4) || !aligned(x, 2))
    return fail(MXNORM_ERR_MISALIGNED, "tensor_scale needs 4-byte, x 2-byte alignment");
  cudaError_t err = launch_nvfp4_tensor_scale(x, n, tensor_scale, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "mxnorm_nvfp4_tensor_scale launch");
  return MXNORM_OK;
}

int mxnorm_absmax_bf16(const void* x, int64_t n, float* amax, void* stream) {
  g_last_error.clear();
  if (n < 0) return fail(MXNORM_ERR_INVALID_ARG, "n < 0");
  if (!amax || (n > 0 && !x)) return fail(MXNORM_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(amax, 4) || !aligned(x, 2)) return fail(MXNORM_ERR_MISALIGNED, "amax needs 4-byte, x 2-byte alignment");
  cudaError_t err = launch_absmax_bf16(x, n, amax, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "mxnorm_absmax_bf16 launch");
  return MXNORM_OK;
}

const char* mxnorm_status_string(int status) {
  switch (status) {
    case MXNORM_OK: return "MXNORM_OK";
    case MXNORM_ERR_INVALID_ARG: return "MXNORM_ERR_INVALID_ARG";
    case MXNORM_ERR_UNSUPPORTED: return "MXNORM_ERR_UNSUPPORTED";
    case MXNORM_ERR_MISALIGNED: return "MXNORM_ERR_MISALIGNED";
    case MXNORM_ERR_CUDA: return "MXNORM_ERR_CUDA";
    default: return "MXNORM_ERR_UNKNOWN";
  }
}

const char* mxnorm_last_error(void) { return g_last_error.c_str(); }

int mxnorm_abi_version(void) { return MXNORM_ABI_VERSION; }

int mxnorm_device_errors(uint32_t* flags, int clear) {
  if (!flags) return fail(MXNORM_ERR_INVALID_ARG, "NULL flags");
  uint32_t tiled = 0, linear = 0, nvfp4 = 0;
  cudaError_t err = read_device_error_word(&tiled, clear != 0);
  if (err == cudaSuccess) err = read_linear_error_word(&linear, clear != 0);
  if (err == cudaSuccess) err = read_nvfp4_error_word(&nvfp4, clear != 0);
  if (err != cudaSuccess) return cuda_fail(err, "reading the device error words");
  *flags = (tiled & 1u) | ((linear & 1u) << 1) | ((nvfp4 & 1u) << 2);
  return MXNORM_OK;
}

}  // extern "C"
