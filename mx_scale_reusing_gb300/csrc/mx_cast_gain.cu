// mx_cast_gain.cu -- MXFP8 cast of MXNormLinear's gain-folded weight.
//
// MXNorm leaves the norm's gain out of the activation pass: gamma (and the
// estimator constant c) multiply the next linear layer's weight instead
// ("MXNorm: Reusing MXFP block scales for efficient tensor normalisation",
// Resumen tecnico, 2. Metodologia, Implementacion).  This kernel forms
// W'[n, k] = w[n, k] * g_k, g_k = RN_fp32(c * gamma_k), each product one
// fp32 multiplication, and casts every 32-element block of a row of W' to
// MXFP8 E4M3 (E8M0 scale, saturating round-to-nearest-even codes), in one
// read of w.
//
// Work split: a warp owns a 512-column strip (16 columns per lane, half an
// MX block) and walks rows of that strip, so each lane computes its 16
// gains once and keeps them in registers for every row it visits.  Grid:
// x = row groups (8 warps per CTA), y = strips; the rows of a strip are
// loaded kRowsAhead at a time to keep enough bytes in flight (a rolling
// prefetch across the groups measured no faster: it needs two CTAs per SM
// for registers).
#include "launch.h"
#include "mx_row.cuh"

namespace mxnorm {
namespace {

constexpr int kGainVec = 16;              // columns per lane
constexpr int kStrip = 32 * kGainVec;     // columns per warp
constexpr int kGainWarps = 8;             // warps per CTA
constexpr int kRowsAhead = 4;             // rows whose loads are issued together

template <bool LOAD32>
__global__ void __launch_bounds__(32 * kGainWarps, 3)
mx_cast_gain_kernel(const uint16_t* __restrict__ w, int64_t N, int K, const float* __restrict__ gamma, float c,
                    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int tiled, int l2_prefetch) {
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();
  {
    // lanes 0..kRowsAhead-1 prefetch the warp's strip of its first rows into
    // L2 while the previous launch ends (device memory only)
    const int64_t r = (int64_t)blockIdx.x * kGainWarps + (threadIdx.x >> 5) + (int64_t)lane * gridDim.x * kGainWarps;
    const int c0 = blockIdx.y * kStrip;
    if (l2_prefetch && lane < kRowsAhead && r < N)
      prefetch_l2(w + r * (int64_t)K + c0, (uint32_t)(2 * min(kStrip, K - c0)));
  }
  pdl_wait();
  const int col = blockIdx.y * kStrip + lane * kGainVec;
  const bool valid = col < K;  // K % 32 == 0: the two lanes of a block agree
  const int KB = K / kBlock;
  const int kb = col / kBlock;
  const bool lead = (lane & 1) == 0;

  float g[kGainVec];
  if (valid) {
    const float4* gp = reinterpret_cast<const float4*>(gamma + col);
#pragma unroll
    for (int q = 0; q < kGainVec / 4; ++q) {
      const float4 t = __ldg(gp + q);
      g[4 * q] = __fmul_rn(c, t.x);
      g[4 * q + 1] = __fmul_rn(c, t.y);
      g[4 * q + 2] = __fmul_rn(c, t.z);
      g[4 * q + 3] = __fmul_rn(c, t.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < kGainVec; ++i) g[i] = 0.0f;
  }

  const int64_t wstride = (int64_t)gridDim.x * kGainWarps;
  // row is the same for every lane of the warp, so the loop and the
  // shuffles below stay warp-uniform; stores are predicated per row.
  for (int64_t row = (int64_t)blockIdx.x * kGainWarps + (threadIdx.x >> 5); row < N;
       row += kRowsAhead * wstride) {
    uint32_t buf[kRowsAhead][kGainVec / 2];
#pragma unroll
    for (int u = 0; u < kRowsAhead; ++u) {
      const int64_t r = row + u * wstride;
      if (valid && r < N) {
        load_lane<kGainVec, LOAD32>(w + r * (int64_t)K + col, buf[u]);
      } else {
#pragma unroll
        for (int i = 0; i < kGainVec / 2; ++i) buf[u][i] = 0u;
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsAhead; ++u) {
      const int64_t r = row + u * wstride;
      float v[kGainVec];
#pragma unroll
      for (int i = 0; i < kGainVec / 2; ++i) {
        f2_unpack(f2_mul(f2_pack(bf16lo(buf[u][i]), bf16hi(buf[u][i])), f2_pack(g[2 * i], g[2 * i + 1])),
                  v[2 * i], v[2 * i + 1]);
      }
      float a = absmax_tree(v);
      a = max2_nan(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
      const uint32_t ab = __float_as_uint(a) & 0x7FFFFFFFu;
      const bool nonfinite = ab >= 0x7F800000u;
      int e = shared_exponent<8>((int)(ab >> 23));
      if (nonfinite) e = 0;  // keeps the multiply harmless; codes are replaced below
      scale_pairs(v, exp2_neg(e));
      uint32_t q[kGainVec / 4];
#pragma unroll
      for (int i = 0; i < kGainVec / 4; ++i) {
        q[i] = cvt_e4m3x4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        if (nonfinite) q[i] = 0x7F7F7F7Fu;
      }
      if (valid && r < N) {
        stg16(codes + r * (int64_t)K + col, q[0], q[1], q[2], q[3]);
        if (lead) *scale_ptr(scales, r, kb, KB, tiled) = nonfinite ? (uint8_t)0xFF : (uint8_t)(e + 127);
      }
    }
  }
}

}  // namespace

cudaError_t launch_mx_cast_gain(const GainCastArgs& a, cudaStream_t s) {
  if (a.N == 0) return cudaSuccess;
  const bool load32 = (reinterpret_cast<uintptr_t>(a.w) & 31u) == 0;
  const void* kern = load32 ? reinterpret_cast<const void*>(&mx_cast_gain_kernel<true>)
                            : reinterpret_cast<const void*>(&mx_cast_gain_kernel<false>);
  const int64_t strips = (a.K + kStrip - 1) / kStrip;
  const int64_t row_groups = (a.N + kGainWarps - 1) / kGainWarps;
  const int fill = persistent_grid(kern, 32 * kGainWarps, row_groups * strips);
  int64_t gx = fill / strips;
  if (gx < 1) gx = 1;
  if (gx > row_groups) gx = row_groups;
  const dim3 grid((unsigned)gx, (unsigned)strips);
  const int K = (int)a.K;
  return launch_pdl(load32 ? mx_cast_gain_kernel<true> : mx_cast_gain_kernel<false>, grid, dim3(32 * kGainWarps), 0,
                    s, static_cast<const uint16_t*>(a.w), a.N, K, a.gamma, a.c, static_cast<uint8_t*>(a.codes),
                    a.scales, a.scale_tiled, is_device_memory(a.w) ? 1 : 0);
}

}  // namespace mxnorm
