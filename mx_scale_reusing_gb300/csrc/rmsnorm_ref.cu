// rmsnorm_ref.cu -- first kernel of the two-pass RMSNorm-then-MXFP8
// baseline: y = bf16(x * inv), inv = 1 / sqrt(mean(x^2) + eps), written to a
// bf16 workspace that the second kernel (the cast-only warp-row kernel)
// reads back.  This is the unfused pipeline the MXNorm pages compare
// against ("MXNorm: Reusing MXFP block scales ...", Resumen tecnico,
// section 1: RMSNorm and the MX cast run as separate operations, each
// gathering its own statistics, with a high-precision intermediate written
// and re-read; section 3, item 2).
//
// One warp per row, the same lane layout as the MXNorm warp-row kernel.
// The sum of squares is fp32: a VEC-wide pairwise sum per chunk, a serial
// sum over chunks and a 5-level warp tree, so its relative error is at most
// (log2 VEC + chunks + 5) * 2^-24; the mean, + eps and the correctly
// rounded reciprocal square root are fp32 (three more roundings).
#include "launch.h"
#include "mx_device.cuh"

namespace mxnorm {
namespace {

constexpr int kWarps = 8;

template <int VEC>
__device__ __forceinline__ void load_words(const uint16_t* src, uint32_t (&w)[VEC / 2]) {
  if constexpr (VEC == 8) {
    const uint4 v = ldg_stream16(src);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    const uint4 a = ldg_stream16(src);
    const uint4 b = ldg_stream16(src + 8);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
}

template <int VEC>
__device__ __forceinline__ float lane_sumsq(const uint32_t (&w)[VEC / 2]) {
  float s[VEC];
#pragma unroll
  for (int i = 0; i < VEC / 2; ++i) {
    const float a = bf16lo(w[i]), b = bf16hi(w[i]);
    s[2 * i] = __fmul_rn(a, a);
    s[2 * i + 1] = __fmul_rn(b, b);
  }
#pragma unroll
  for (int width = VEC / 2; width >= 1; width >>= 1)
#pragma unroll
    for (int i = 0; i < width; ++i) s[i] = __fadd_rn(s[i], s[i + width]);
  return s[0];
}

template <int VEC>
__device__ __forceinline__ void store_y(uint16_t* dst, const uint32_t (&w)[VEC / 2], float inv) {
  uint32_t o[VEC / 2];
#pragma unroll
  for (int i = 0; i < VEC / 2; ++i) {
    const __nv_bfloat16 lo = __float2bfloat16_rn(__fmul_rn(bf16lo(w[i]), inv));
    const __nv_bfloat16 hi = __float2bfloat16_rn(__fmul_rn(bf16hi(w[i]), inv));
    o[i] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
  }
  if constexpr (VEC == 8) {
    stg16(dst, o[0], o[1], o[2], o[3]);
  } else {
    stg16(dst, o[0], o[1], o[2], o[3]);
    stg16(dst + 8, o[4], o[5], o[6], o[7]);
  }
}

__device__ __forceinline__ float finish_inv(float ss, int H, float eps) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, off));
  return __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), eps));
}

// NCHUNK > 0: the row stays in registers between the two phases.
// NCHUNK == 0: any H; the second phase re-reads the row (L1/L2 hits).
// Two CTAs per SM (128 registers) time best for the register-resident row.
template <int VEC, int NCHUNK>
__global__ void __launch_bounds__(kWarps * 32, 2)
    rmsnorm_bf16_kernel(const uint16_t* __restrict__ x, int64_t T, int H, float eps,
                        uint16_t* __restrict__ y, float* __restrict__ inv_rms) {
  constexpr int CE = 32 * VEC;
  const int lane = threadIdx.x & 31;
  pdl_enter();
  const int64_t w0 = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int64_t nw = (int64_t)gridDim.x * kWarps;
  for (int64_t row = w0; row < T; row += nw) {
    const uint16_t* xr = x + row * (int64_t)H;
    uint16_t* yr = y + row * (int64_t)H;
    if constexpr (NCHUNK > 0) {
      uint32_t w[NCHUNK][VEC / 2];
#pragma unroll
      for (int c = 0; c < NCHUNK; ++c) {
        const int e0 = c * CE + lane * VEC;
        if (e0 < H) load_words<VEC>(xr + e0, w[c]);
        else
#pragma unroll
          for (int i = 0; i < VEC / 2; ++i) w[c][i] = 0u;
      }
      float ss = 0.0f;
#pragma unroll
      for (int c = 0; c < NCHUNK; ++c) ss = __fadd_rn(ss, lane_sumsq<VEC>(w[c]));
      const float inv = finish_inv(ss, H, eps);
#pragma unroll
      for (int c = 0; c < NCHUNK; ++c) {
        const int e0 = c * CE + lane * VEC;
        if (e0 < H) store_y<VEC>(yr + e0, w[c], inv);
      }
      if (lane == 0) inv_rms[row] = inv;
    } else {
      float ss = 0.0f;
      for (int e0 = lane * VEC; e0 < H; e0 += CE) {
        uint32_t w[VEC / 2];
        load_words<VEC>(xr + e0, w);
        ss = __fadd_rn(ss, lane_sumsq<VEC>(w));
      }
      const float inv = finish_inv(ss, H, eps);
      for (int e0 = lane * VEC; e0 < H; e0 += CE) {
        uint32_t w[VEC / 2];
        load_words<VEC>(xr + e0, w);
        store_y<VEC>(yr + e0, w, inv);
      }
      if (lane == 0) inv_rms[row] = inv;
    }
  }
}

template <int VEC, int NCHUNK>
cudaError_t launch_one(const RmsNormArgs& a, cudaStream_t s) {
  auto kern = rmsnorm_bf16_kernel<VEC, NCHUNK>;
  const int grid = persistent_grid(reinterpret_cast<const void*>(kern), kWarps * 32,
                                   (a.T + kWarps - 1) / kWarps);
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kWarps * 32), 0, s, static_cast<const uint16_t*>(a.x), a.T,
                    (int)a.H, a.eps, static_cast<uint16_t*>(a.y), a.inv_rms);
}

}  // namespace

cudaError_t launch_rmsnorm_bf16(const RmsNormArgs& a, cudaStream_t s) {
  if (a.H % 512 == 0) {
    switch (a.H / 512) {
      case 1: return launch_one<16, 1>(a, s);
      case 2: return launch_one<16, 2>(a, s);
      case 4: return launch_one<16, 4>(a, s);
      case 8: return launch_one<16, 8>(a, s);
      case 16: return launch_one<16, 16>(a, s);
      default: return launch_one<16, 0>(a, s);
    }
  }
  switch ((a.H + 255) / 256) {
    case 1: return launch_one<8, 1>(a, s);
    case 3: return launch_one<8, 3>(a, s);
    default: return launch_one<8, 0>(a, s);
  }
}

}  // namespace mxnorm
