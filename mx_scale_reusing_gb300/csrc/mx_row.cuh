// mx_row.cuh -- per-lane MX cast of one chunk of a row, the power-mean
// finish of a row, and the two row loops built on them: the streaming loop
// of the warp-row kernel (global loads, rolling prefetch across rows) and
// the single-row loop of the tiled kernel (shared-memory loads).
//
// Lane layout: lane l of chunk c holds elements [c*32*VEC + l*VEC, +VEC) of
// the row; an MX block spans 32/VEC lanes, whose first lane ("lead") writes
// the block's E8M0 byte and carries its exponent into the power mean.
#pragma once

#include "mx_device.cuh"

namespace mxnorm {

// Lane's VEC bf16 values (as VEC/2 bf16x2 words) from global memory.
template <int VEC, bool LOAD32>
__device__ __forceinline__ void load_lane(const uint16_t* src, uint32_t (&w)[VEC / 2]) {
  if constexpr (VEC == 8) {
    const uint4 v = ldg_stream16(src);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (VEC == 32) {
    uint32_t (&lo)[8] = *reinterpret_cast<uint32_t(*)[8]>(&w[0]);
    uint32_t (&hi)[8] = *reinterpret_cast<uint32_t(*)[8]>(&w[8]);
    if constexpr (LOAD32) {
      ldg_stream32(src, lo);
      ldg_stream32(src + 16, hi);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 a = ldg_stream16(src + 8 * q);
        w[4 * q] = a.x; w[4 * q + 1] = a.y; w[4 * q + 2] = a.z; w[4 * q + 3] = a.w;
      }
    }
  } else if constexpr (LOAD32) {
    ldg_stream32(src, w);
  } else {
    const uint4 a = ldg_stream16(src);
    const uint4 b = ldg_stream16(src + 8);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
}

// max(|a|, |b|, |c|) propagating NaN (sm_100+ three-input max).
__device__ __forceinline__ float absmax3(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)), "f"(fabsf(c)));
  return r;
}

// max(a, b, c) of non-negative values, propagating NaN.
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float max2_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// max_i |v_i| as a tree of three-input maxima (NaN wins over everything,
// Inf over every finite value).
__device__ __forceinline__ float absmax_tree(const float (&v)[16]) {
  const float a = absmax3(v[0], v[1], v[2]);
  const float b = absmax3(v[3], v[4], v[5]);
  const float c = absmax3(v[6], v[7], v[8]);
  const float d = absmax3(v[9], v[10], v[11]);
  const float e = absmax3(v[12], v[13], v[14]);
  return max2_nan(max3_nan(a, b, c), max3_nan(d, e, fabsf(v[15])));
}
__device__ __forceinline__ float absmax_tree(const float (&v)[32]) {
  const float (&lo)[16] = *reinterpret_cast<const float(*)[16]>(&v[0]);
  const float (&hi)[16] = *reinterpret_cast<const float(*)[16]>(&v[16]);
  return max2_nan(absmax_tree(lo), absmax_tree(hi));
}
__device__ __forceinline__ float absmax_tree(const float (&v)[8]) {
  const float a = absmax3(v[0], v[1], v[2]);
  const float b = absmax3(v[3], v[4], v[5]);
  return max3_nan(a, b, max2_nan(fabsf(v[6]), fabsf(v[7])));
}

// Cast one lane's VEC values of a chunk: block absmax (NaN/Inf-aware),
// shared exponent, scaled saturating RNE codes, stores of codes and (lead
// lane) of the scale byte.  Returns the block's exponent, or kExpNone for a
// block holding Inf/NaN.  Every lane of the warp must call it (shuffles).
template <int FMT, int VEC>
__device__ __forceinline__ int cast_lane(const uint32_t (&w)[VEC / 2], bool valid, uint8_t* code_dst,
                                         uint8_t* scale_dst, bool lead) {
  using Tr = FmtTraits<FMT>;
  constexpr int LPB = kBlock / VEC;  // lanes per block
  float v[VEC];
#pragma unroll
  for (int i = 0; i < VEC / 2; ++i) {
    v[2 * i] = bf16lo(w[i]);
    v[2 * i + 1] = bf16hi(w[i]);
  }
  if constexpr (Tr::rot == 16) {
    static_assert(VEC % 16 == 0, "H16 needs whole 16-element groups per lane");
#pragma unroll
    for (int g = 0; g < VEC; g += 16) h16_inplace(*reinterpret_cast<float(*)[16]>(&v[g]));
  } else if constexpr (Tr::rot == 32) {
    static_assert(VEC == 32, "H32 needs a whole 32-element block per lane");
    h32_inplace(*reinterpret_cast<float(*)[32]>(&v[0]));
  }
  float a = absmax_tree(v);
#pragma unroll
  for (int off = 1; off < LPB; off <<= 1) {
    a = max2_nan(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
  }
  const uint32_t ab = __float_as_uint(a) & 0x7FFFFFFFu;
  const bool nonfinite = ab >= 0x7F800000u;
  int e = shared_exponent<Tr::emax>((int)(ab >> 23));
  if (nonfinite) e = 0;  // keeps the multiply harmless; codes are replaced below
  scale_pairs(v, exp2_neg(e));

  if (valid) {
    if constexpr (!Tr::fp4) {
      uint32_t q[VEC / 4];
#pragma unroll
      for (int i = 0; i < VEC / 4; ++i) {
        q[i] = cvt_e4m3x4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        if (nonfinite) q[i] = 0x7F7F7F7Fu;
      }
      if constexpr (VEC == 32) {
        stg16(code_dst, q[0], q[1], q[2], q[3]);
        stg16(code_dst + 16, q[4], q[5], q[6], q[7]);
      } else if constexpr (VEC == 16) {
        stg16(code_dst, q[0], q[1], q[2], q[3]);
      } else {
        stg8(code_dst, q[0], q[1]);
      }
    } else {
      uint32_t q[VEC / 8];
#pragma unroll
      for (int i = 0; i < VEC / 8; ++i) {
        q[i] = cvt_e2m1x8(v[8 * i], v[8 * i + 1], v[8 * i + 2], v[8 * i + 3], v[8 * i + 4],
                          v[8 * i + 5], v[8 * i + 6], v[8 * i + 7]);
        if (nonfinite) q[i] = 0u;
      }
      if constexpr (VEC == 32) stg16(code_dst, q[0], q[1], q[2], q[3]);
      else if constexpr (VEC == 16) stg8(code_dst, q[0], q[1]);
      else stg4(code_dst, q[0]);
    }
    if (lead) *scale_dst = nonfinite ? (uint8_t)0xFF : (uint8_t)(e + 127);
  }
  return nonfinite ? kExpNone : e;
}

// Address of the E8M0 byte of (row, block kb) for a row of K blocks.
// Row-major: scales[row * K + kb].  MMA-tiled (tiled != 0, K % 4 == 0): the
// 512-byte atoms the block-scaled tensor-core MMA reads, one per 128 rows x
// 4 blocks, atoms ordered row-tile-major; inside an atom the byte of
// (r, k) sits at (r % 32) * 16 + (r / 32 % 4) * 4 + k % 4, so one
// tcgen05.cp of 32 lanes x 16 bytes lands row r's 4 scales in TMEM lane
// r % 32, column r / 32.
__device__ __forceinline__ uint8_t* scale_ptr(uint8_t* scales, int64_t row, int kb, int K, int tiled) {
  if (!tiled) return scales + row * (int64_t)K + kb;
  const int64_t atom = (row >> 7) * (int64_t)(K >> 2) + (kb >> 2);
  return scales + atom * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (kb & 3);
}

// The same address split for the streaming loop: scale_row(row) +
// (kb >> 2) * scale_quad_stride + (kb & 3), with a quad stride of 4 bytes
// (row-major) or 512 (one atom per 4 blocks), so the per-chunk address is
// one multiply-add and no branch.
__device__ __forceinline__ uint8_t* scale_row(uint8_t* scales, int64_t row, int K, int tiled) {
  if (!tiled) return scales + row * (int64_t)K;
  return scales + (row >> 7) * (int64_t)(K >> 2) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4;
}

// Power mean of a row from the exponents each lane collected (ev[c] for its
// chunks, meaningful where own[c]): m = the row's largest exponent (warp
// max), then the fixed-point sum sum_k 2^(F + p (e_k - m)) (terms below 2^0
// dropped: relative error < K 2^-F), then inv_rms in fp32 (pm_inv_rms).
// A block marked kExpNone (Inf/NaN) makes the row's inv_rms NaN.
template <int NCHUNK>
__device__ __forceinline__ float finish_row(const int (&ev)[NCHUNK], const bool (&own)[NCHUNK], int K, int p) {
  int mloc = kExpNone;
  bool bad = false;
#pragma unroll
  for (int c = 0; c < NCHUNK; ++c) {
    if (own[c]) {
      if (ev[c] == kExpNone) bad = true;
      else mloc = max(mloc, ev[c]);
    }
  }
  int m = mloc;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  unsigned long long s = 0ull;
#pragma unroll
  for (int c = 0; c < NCHUNK; ++c) {
    const int t = kFixedBits + p * (ev[c] - m);
    if (own[c] && ev[c] != kExpNone && t >= 0) s += 1ull << t;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
  bad = __any_sync(0xFFFFFFFFu, bad);
  if (bad) return __uint_as_float(0x7FC00000u);
  return pm_inv_rms(PowerMeanAcc{m, s}, K, p);
}

// Streaming row loop of the warp-row kernel: rows row0, row0 + rstride, ...
// of x, each NCHUNK chunks of 32*VEC elements.  A ring of AHEAD chunk
// buffers per lane keeps AHEAD loads in flight: the refill of a buffer is
// issued (for this row's chunk c + AHEAD, or the next row's first chunks)
// before the chunk it held is cast.  EXACT: H == NCHUNK * 32 * VEC.
template <int FMT, int VEC, int NCHUNK, int AHEAD, bool EXACT, bool LOAD32, bool ESTIMATE>
__device__ __forceinline__ void mx_rows_stream(const uint16_t* __restrict__ x, int64_t T, int H,
                                               uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                               float* __restrict__ inv_rms, int p, int64_t row,
                                               int64_t rstride, int scale_tiled) {
  static_assert(NCHUNK % AHEAD == 0, "the ring must tile the row");
  using Tr = FmtTraits<FMT>;
  constexpr int LPB = kBlock / VEC;
  constexpr int CE = 32 * VEC;
  const int Hc = EXACT ? NCHUNK * CE : H;
  const int lane = threadIdx.x & 31;
  const bool lead = (lane % LPB) == 0;
  const int K = Hc / kBlock;
  const int64_t code_row = Tr::fp4 ? (int64_t)(Hc / 2) : (int64_t)Hc;
  if (row >= T) return;

  // scale address of chunk c for this lane: scale_row(row) + loff + c * (VEC / 4) * qstride
  const int qstride = scale_tiled ? 512 : 4;
  const int kl = lane * VEC / kBlock;
  const int loff = (kl >> 2) * qstride + (kl & 3);
  uint32_t buf[AHEAD][VEC / 2];
  auto issue = [&](int64_t r, int c, uint32_t (&dst)[VEC / 2]) {
    const int e0 = c * CE + lane * VEC;
    if (EXACT || e0 < Hc) {
      load_lane<VEC, LOAD32>(x + r * (int64_t)Hc + e0, dst);
    } else {
#pragma unroll
      for (int i = 0; i < VEC / 2; ++i) dst[i] = 0u;
    }
  };
#pragma unroll
  for (int a = 0; a < AHEAD; ++a) issue(row, a, buf[a]);

  for (; row < T; row += rstride) {
    const int64_t next = row + rstride;
    uint8_t* cr = codes + row * code_row;
    uint8_t* sr = scale_row(scales, row, K, scale_tiled) + loff;
    int ev[NCHUNK];
    bool own[NCHUNK];
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) {
      uint32_t w[VEC / 2];
#pragma unroll
      for (int i = 0; i < VEC / 2; ++i) w[i] = buf[c % AHEAD][i];
      const int cc = c + AHEAD;
      if (cc < NCHUNK) issue(row, cc, buf[c % AHEAD]);
      else if (next < T) issue(next, cc - NCHUNK, buf[c % AHEAD]);
      const int e0 = c * CE + lane * VEC;
      const bool valid = EXACT || e0 < Hc;
      static_assert(VEC % 4 == 0, "a chunk spans whole quads of blocks");
      ev[c] = cast_lane<FMT, VEC>(w, valid, cr + (Tr::fp4 ? e0 / 2 : e0), sr + c * (VEC / 4) * qstride, lead);
      own[c] = valid && lead;
    }
    if constexpr (ESTIMATE) {
      const float inv = finish_row<NCHUNK>(ev, own, K, p);
      if (lane == 0) inv_rms[row] = inv;
    }
  }
}

// finish_row over a half warp (16 lanes, one row): the same reductions with
// shuffle offsets below 16, so the two halves of the warp finish their own
// rows side by side.  Returns the row's inv_rms in every lane of the half.
template <int NCHUNK>
__device__ __forceinline__ float finish_row_half(const int (&ev)[NCHUNK], const bool (&own)[NCHUNK], int K, int p) {
  int mloc = kExpNone;
  bool bad = false;
#pragma unroll
  for (int c = 0; c < NCHUNK; ++c) {
    if (own[c]) {
      if (ev[c] == kExpNone) bad = true;
      else mloc = max(mloc, ev[c]);
    }
  }
  int m = mloc;
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  unsigned long long s = 0ull;
#pragma unroll
  for (int c = 0; c < NCHUNK; ++c) {
    const int t = kFixedBits + p * (ev[c] - m);
    if (own[c] && ev[c] != kExpNone && t >= 0) s += 1ull << t;
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
  const unsigned half_bad = __ballot_sync(0xFFFFFFFFu, bad) >> (threadIdx.x & 16);
  if (half_bad & 0xFFFFu) return __uint_as_float(0x7FC00000u);
  return pm_inv_rms(PowerMeanAcc{m, s}, K, p);
}

// Streaming loop with two rows per warp, for rows of NCHUNK chunks of
// 16 * VEC elements (H = NCHUNK * 16 * VEC exactly): lanes 0-15 walk rows
// row0, row0 + rstride, ... and lanes 16-31 the row after each.  Short rows
// (H = 256 x odd) then keep 32-byte lanes and whole chunks, and the row
// tail (power-mean reductions, root and reciprocal) serves two rows per
// instruction.  A half whose row is past T still takes part in the
// shuffles but stores nothing.
template <int FMT, int VEC, int NCHUNK, int AHEAD, bool LOAD32, bool ESTIMATE>
__device__ __forceinline__ void mx_rows_stream_half(const uint16_t* __restrict__ x, int64_t T, int H,
                                                    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                    float* __restrict__ inv_rms, int p, int64_t pair_row,
                                                    int64_t rstride, int scale_tiled) {
  static_assert(NCHUNK % AHEAD == 0, "the ring must tile the row");
  static_assert(VEC % 8 == 0 && kBlock / VEC <= 16, "whole quads of blocks per chunk, blocks inside a half warp");
  using Tr = FmtTraits<FMT>;
  constexpr int LPB = kBlock / VEC;
  constexpr int CE = 16 * VEC;
  constexpr int Hc = NCHUNK * CE;
  constexpr int K = Hc / kBlock;
  const int lane = threadIdx.x & 31;
  const int hl = lane & 15;
  const int64_t half = lane >> 4;
  const bool lead = (hl % LPB) == 0;
  const int64_t code_row = Tr::fp4 ? (int64_t)(Hc / 2) : (int64_t)Hc;
  const int qstride = scale_tiled ? 512 : 4;
  const int kl = hl * VEC / kBlock;
  const int loff = (kl >> 2) * qstride + (kl & 3);
  (void)H;
  int64_t row = 2 * pair_row + half;
  if (2 * pair_row >= T) return;

  uint32_t buf[AHEAD][VEC / 2];
  auto issue = [&](int64_t r, int c, uint32_t (&dst)[VEC / 2]) {
    if (r < T) {
      load_lane<VEC, LOAD32>(x + r * (int64_t)Hc + c * CE + hl * VEC, dst);
    } else {
#pragma unroll
      for (int i = 0; i < VEC / 2; ++i) dst[i] = 0u;
    }
  };
#pragma unroll
  for (int a = 0; a < AHEAD; ++a) issue(row, a, buf[a]);

  for (; row - half < T; row += 2 * rstride) {
    const int64_t next = row + 2 * rstride;
    const bool live = row < T;
    uint8_t* cr = codes + row * code_row;
    uint8_t* sr = scale_row(scales, live ? row : 0, K, scale_tiled) + loff;
    int ev[NCHUNK];
    bool own[NCHUNK];
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) {
      uint32_t w[VEC / 2];
#pragma unroll
      for (int i = 0; i < VEC / 2; ++i) w[i] = buf[c % AHEAD][i];
      const int cc = c + AHEAD;
      if (cc < NCHUNK) issue(row, cc, buf[c % AHEAD]);
      else issue(next, cc - NCHUNK, buf[c % AHEAD]);
      const int e0 = c * CE + hl * VEC;
      // a chunk spans 16 * VEC elements = VEC / 2 blocks = VEC / 8 quads of blocks
      ev[c] = cast_lane<FMT, VEC>(w, live, cr + (Tr::fp4 ? e0 / 2 : e0), sr + c * (VEC / 8) * qstride, lead);
      own[c] = lead;
    }
    if constexpr (ESTIMATE) {
      const float inv = finish_row_half<NCHUNK>(ev, own, K, p);
      if (hl == 0 && live) inv_rms[row] = inv;
    }
  }
}

// One row through a loader `load(e0, w)` (e0 = the lane's first element):
// NCHUNK > 0 issues all of the row's loads before any arithmetic; NCHUNK ==
// 0 handles any H in batches of four chunks with the running-maximum
// power-mean accumulator.  Every lane of the warp must call it.
template <int FMT, int VEC, int NCHUNK, bool ESTIMATE, class Load>
__device__ __forceinline__ void mx_row(Load load, int H, int p, uint8_t* cr, uint8_t* scales, int64_t row,
                                       int scale_tiled, float* inv_dst) {
  using Tr = FmtTraits<FMT>;
  constexpr int LPB = kBlock / VEC;
  constexpr int CE = 32 * VEC;
  const int lane = threadIdx.x & 31;
  const bool lead = (lane % LPB) == 0;
  const int K = H / kBlock;

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
    int ev[NCHUNK];
    bool own[NCHUNK];
#pragma unroll
    for (int c = 0; c < NCHUNK; ++c) {
      const int e0 = c * CE + lane * VEC;
      const bool valid = e0 < H;
      ev[c] = cast_lane<FMT, VEC>(w[c], valid, cr + (Tr::fp4 ? e0 / 2 : e0),
                                  scale_ptr(scales, row, e0 / kBlock, K, scale_tiled), lead);
      own[c] = valid && lead;
    }
    if constexpr (ESTIMATE) {
      const float inv = finish_row<NCHUNK>(ev, own, K, p);
      if (lane == 0) *inv_dst = inv;
    }
  } else {
    PowerMeanAcc acc{kExpNone, 0ull};
    bool row_nonfinite = false;
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
      for (int b = 0; b < BATCH; ++b) {
        if (c0 + b < nchunk) {
          const int e0 = (c0 + b) * CE + lane * VEC;
          const bool valid = e0 < H;
          const int e = cast_lane<FMT, VEC>(w[b], valid, cr + (Tr::fp4 ? e0 / 2 : e0),
                                            scale_ptr(scales, row, e0 / kBlock, K, scale_tiled), lead);
          if (ESTIMATE && valid && lead) {
            if (e == kExpNone) row_nonfinite = true;
            else pm_add(acc, e, p);
          }
        }
      }
    }
    if constexpr (ESTIMATE) {
      acc = pm_warp_reduce(acc, p);
      row_nonfinite = __any_sync(0xFFFFFFFFu, row_nonfinite);
      if (lane == 0) *inv_dst = row_nonfinite ? __uint_as_float(0x7FC00000u) : pm_inv_rms(acc, K, p);
    }
  }
}

}  // namespace mxnorm
