// mx_row.cuh -- per-lane MX cast of one chunk of a row and the row loop,
// shared by the warp-row kernel (global loads) and the tiled kernel
// (shared-memory loads).  Lane layout: lane l of chunk c holds elements
// [c*32*VEC + l*VEC, +VEC) of the row; an MX block spans 32/VEC lanes.
#pragma once

#include "mx_device.cuh"

namespace mxnorm {

// Lane's VEC bf16 values as VEC/2 bf16x2 words.
template <int VEC, bool LOAD32>
__device__ __forceinline__ void load_lane(const uint16_t* src, uint32_t (&w)[VEC / 2]) {
  if constexpr (VEC == 8) {
    const uint4 v = ldg_stream16(src);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (LOAD32) {
    ldg_stream32(src, w);
  } else {
    const uint4 a = ldg_stream16(src);
    const uint4 b = ldg_stream16(src + 8);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
}

// Cast one lane's VEC values of a chunk; returns through `e_out` the block's
// shared exponent (or kExpNone for a non-finite block).
template <int FMT, int VEC>
__device__ __forceinline__ void cast_lane(const uint32_t (&w)[VEC / 2], bool valid,
                                          uint8_t* code_dst, uint8_t* scale_dst, bool lead,
                                          int& e_out) {
  using Tr = FmtTraits<FMT>;
  constexpr int LPB = kBlock / VEC;  // lanes per block
  float v[VEC];
  bool nonfinite;
  int e;
  if constexpr (Tr::h16) {
    static_assert(VEC == 16, "H16 needs a whole 16-element group per lane");
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) {
      v[2 * i] = bf16lo(w[i]);
      v[2 * i + 1] = bf16hi(w[i]);
    }
    h16_inplace(v);
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < VEC; ++i) a = absmax_nan(a, v[i]);
#pragma unroll
    for (int off = 1; off < LPB; off <<= 1) {
      const float o = __shfl_xor_sync(0xFFFFFFFFu, a, off);
      asm("max.NaN.f32 %0, %0, %1;" : "+f"(a) : "f"(o));
    }
    const uint32_t ab = __float_as_uint(a) & 0x7FFFFFFFu;
    nonfinite = ab >= 0x7F800000u;
    e = shared_exponent<Tr::emax>((int)(ab >> 23));
  } else {
    uint32_t a = 0;
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) a = absmax_bf16x2(a, w[i]);
    a = max(a & 0xFFFFu, a >> 16);
#pragma unroll
    for (int off = 1; off < LPB; off <<= 1) a = max(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
    nonfinite = a >= 0x7F80u;
    e = shared_exponent<Tr::emax>((int)(a >> 7));
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) {
      v[2 * i] = bf16lo(w[i]);
      v[2 * i + 1] = bf16hi(w[i]);
    }
  }
  if (nonfinite) e = 0;  // keep the multiply harmless; codes are replaced below
  const float mul = exp2_neg(e);
#pragma unroll
  for (int i = 0; i < VEC; ++i) v[i] = __fmul_rn(v[i], mul);

  if (valid) {
    if constexpr (!Tr::fp4) {
      uint32_t q[VEC / 4];
#pragma unroll
      for (int i = 0; i < VEC / 4; ++i) {
        q[i] = cvt_e4m3x4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        if (nonfinite) q[i] = 0x7F7F7F7Fu;
      }
      if constexpr (VEC == 16) stg16(code_dst, q[0], q[1], q[2], q[3]);
      else stg8(code_dst, q[0], q[1]);
    } else {
      uint32_t q[VEC / 8];
#pragma unroll
      for (int i = 0; i < VEC / 8; ++i) {
        q[i] = cvt_e2m1x8(v[8 * i], v[8 * i + 1], v[8 * i + 2], v[8 * i + 3], v[8 * i + 4],
                          v[8 * i + 5], v[8 * i + 6], v[8 * i + 7]);
        if (nonfinite) q[i] = 0u;
      }
      if constexpr (VEC == 16) stg8(code_dst, q[0], q[1]);
      else stg4(code_dst, q[0]);
    }
    if (lead) *scale_dst = nonfinite ? (uint8_t)0xFF : (uint8_t)(e + 127);
  }
  e_out = nonfinite ? kExpNone : e;
}


// One row: loads through `load(e0, w)` (e0 = the lane's first element), MX
// cast of every chunk, stores of codes/scales and, when ESTIMATE, the row's
// inv_rms from the power mean of its block scales.  NCHUNK > 0 issues all
// of the row's loads before any arithmetic; NCHUNK == 0 handles any H in
// batches of four chunks.  Every lane of the warp must call it.
template <int FMT, int VEC, int NCHUNK, bool ESTIMATE, class Load>
__device__ __forceinline__ void mx_row(Load load, int H, int p, uint8_t* cr, uint8_t* sr,
                                       float* inv_dst) {
  using Tr = FmtTraits<FMT>;
  constexpr int LPB = kBlock / VEC;
  constexpr int CE = 32 * VEC;
  const int lane = threadIdx.x & 31;
  const bool lead = (lane % LPB) == 0;
  PowerMeanAcc acc{kExpNone, 0ull};
  bool row_nonfinite = false;

  auto do_chunk = [&](int c, const uint32_t (&w)[VEC / 2]) {
    const int e0 = c * CE + lane * VEC;
    const bool valid = e0 < H;
    int e;
    cast_lane<FMT, VEC>(w, valid, cr + (Tr::fp4 ? e0 / 2 : e0), sr + e0 / kBlock, lead, e);
    if constexpr (ESTIMATE) {
      if (valid && lead) {
        if (e == kExpNone) row_nonfinite = true;
        else pm_add(acc, e, p);
      }
    }
  };

  if constexpr (NCHUNK > 0) {
    uint32_t w[NCHUNK][VEC / 2];
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) {
      const int e0 = c * CE + lane * VEC;
      if (e0 < H) {
        load(e0, w[c]);
      } else {
#pragma unroll
        for (int i = 0; i < VEC / 2; ++i) w[c][i] = 0u;
      }
    }
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) do_chunk(c, w[c]);
  } else {
    constexpr int BATCH = 4;
    const int nchunk = (H + CE - 1) / CE;
    for (int c0 = 0; c0 < nchunk; c0 += BATCH) {
      uint32_t w[BATCH][VEC / 2];
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        const int e0 = (c0 + b) * CE + lane * VEC;
        if (e0 < H) {
          load(e0, w[b]);
        } else {
#pragma unroll
          for (int i = 0; i < VEC / 2; ++i) w[b][i] = 0u;
        }
      }
#pragma unroll
      for (int b = 0; b < BATCH; ++b)
        if (c0 + b < nchunk) do_chunk(c0 + b, w[b]);
    }
  }

  if constexpr (ESTIMATE) {
    const int K = H / kBlock;
    acc = pm_warp_reduce(acc, p);
    row_nonfinite = __any_sync(0xFFFFFFFFu, row_nonfinite);
    if (lane == 0) *inv_dst = row_nonfinite ? __uint_as_float(0x7FC00000u) : pm_inv_rms(acc, K, p);
  }
}

}  // namespace mxnorm
