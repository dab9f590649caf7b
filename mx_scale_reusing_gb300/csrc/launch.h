// launch.h -- internal launcher interface between the C ABI (capi.cu) and
// the kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mxnorm {

struct WarpRowArgs {
  const void* x;      // bf16 [T, H]
  int64_t T;
  int64_t H;
  int p;              // 1 or 2 (ignored by the cast-only form)
  int fmt;            // Fmt
  void* codes;        // u8 [T, H] (E4M3) or [T, H/2] (E2M1)
  uint8_t* scales;    // u8 [T, H/32]
  float* inv_rms;     // f32 [T] (unused by the cast-only form)
  int scale_tiled = 0;  // 1: scales in the MMA atom layout (see scale_ptr in mx_row.cuh)
};

// True when p points into device memory (not mapped host or managed memory):
// the streaming kernels prefetch their first rows into L2 only then.
bool is_device_memory(const void* p);

struct RmsNormArgs {
  const void* x;      // bf16 [T, H]
  int64_t T;
  int64_t H;
  float eps;
  void* y;            // bf16 [T, H]
  float* inv_rms;     // f32 [T]
};

struct BwdArgs {
  const void* x;       // bf16 [T, H], the forward's input
  const void* dy;      // bf16 [T, H], gradient w.r.t. the normalised output
  const float* inv_rms;  // f32 [T], the forward's estimate
  int64_t T;
  int64_t H;
  void* dx;            // bf16 [T, H]
};

struct Nvfp4Args {
  const void* x;       // bf16 [T, H], H % 16 == 0
  int64_t T;
  int64_t H;
  int p;
  float g;             // fp32 tensor scale (> 0, finite), used when g_dev is null
  void* codes;         // u8 [T, H/2]
  uint8_t* scales;     // UE4M3 [T, H/16]
  float* inv_rms;      // f32 [T]
  const float* g_dev = nullptr;  // device word holding the tensor scale, or null
};

struct LinearArgs {
  const void* x_codes;       // E4M3 [T, K]
  const uint8_t* x_scales;   // E8M0, MMA atom layout, ceil(T/128) x K/128 atoms
  const float* inv_rms;      // f32 [T]
  const void* w_codes;       // E4M3 [N, K]
  const uint8_t* w_scales;   // E8M0, MMA atom layout, N/128 x K/128 atoms
  int64_t T;
  int64_t K;
  int64_t N;
  void* out;                 // bf16 [T, N]
};

struct GainCastArgs {
  const void* w;        // bf16 [N, K], one row per output feature
  int64_t N;
  int64_t K;            // % 32 == 0 (% 128 for the MMA layout)
  const float* gamma;   // f32 [K], 16-byte aligned
  float c;              // estimator constant, folded with gamma
  void* codes;          // E4M3 [N, K]
  uint8_t* scales;      // E8M0, row-major [N, K/32] or MMA atoms
  int scale_tiled;      // 1: MMA atom layout
};

struct TiledArgs {
  WarpRowArgs base;
  unsigned long long wait_limit_ns = 1000000000ull;  // limit of the pipeline waits
  int64_t withheld_tile = -1;  // failure-detection drill: a tile whose copy is never issued
};

// Launch a kernel with programmatic stream serialisation: it may be
// scheduled while the previous kernel on the stream finishes, and waits in
// pdl_enter() (mx_device.cuh) for that kernel's completion before touching
// memory.  Grids launched this way fit in one wave (persistent_grid), so the
// early launch never takes slots a running grid still needs.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Grid size for a grid-stride kernel: enough CTAs to fill every SM at the
// kernel's occupancy, never more than `work_ctas`.  Cached per device.
int persistent_grid(const void* kernel, int threads_per_cta, int64_t work_ctas,
                    size_t dyn_smem = 0);

cudaError_t launch_mxnorm_warp_row(const WarpRowArgs& a, cudaStream_t s);
cudaError_t launch_mx_cast_warp_row(const WarpRowArgs& a, cudaStream_t s);
cudaError_t launch_rmsnorm_bf16(const RmsNormArgs& a, cudaStream_t s);
cudaError_t launch_mxnorm_tiled(const TiledArgs& a, cudaStream_t s);
bool tiled_supported(int64_t H, int fmt);
cudaError_t launch_mxnorm_bwd_ste(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_nvfp4(const Nvfp4Args& a, cudaStream_t s);
cudaError_t launch_mxfp8_linear(const LinearArgs& a, cudaStream_t s);
cudaError_t launch_mx_cast_gain(const GainCastArgs& a, cudaStream_t s);
cudaError_t read_linear_error_word(uint32_t* out, bool clear);
cudaError_t launch_absmax_bf16(const void* x, int64_t n, float* amax, cudaStream_t s);
cudaError_t launch_nvfp4_tensor_scale(const void* x, int64_t n, float* g, cudaStream_t s);
cudaError_t read_nvfp4_error_word(uint32_t* out, bool clear);

// Replace the calling thread's message returned by mxnorm_last_error().
void set_last_error(const char* msg);

// Checks shared by the entry points that take (x, T, H, codes, scales,
// inv_rms): sizes, NULL pointers (T > 0) and alignment; returns an
// mxnorm_status and sets the thread's message on failure.
int check_common(const void* x, int64_t T, int64_t H, const void* codes, const void* scales,
                 const void* inv_rms);

// Copy (and optionally zero) the device error word that bounded waits set.
cudaError_t read_device_error_word(uint32_t* out, bool clear);

}  // namespace mxnorm
