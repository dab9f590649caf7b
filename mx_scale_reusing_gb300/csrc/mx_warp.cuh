// mx_warp.cuh -- the one-row-per-warp MXNorm kernel templates and their
// launch-shape selection, instantiated one format per translation unit
// (mxnorm_warp_fp8*.cu, mxnorm_warp_fp4*.cu) so the formats compile in
// parallel.
//
// Work split: each warp owns whole rows (grid-stride over T) and walks them
// as one stream of chunks of 32 * VEC elements (row loop: mx_rows_stream in
// mx_row.cuh).  Launched with programmatic stream serialisation, so
// back-to-back launches overlap one launch's start with the previous one's
// end: each kernel first lets the next grid be scheduled, prefetches its
// warps' first rows into L2 (device memory only; all of them when the whole
// input fits in a quarter of L2), then waits for the previous grid before
// any load.  Lane l of chunk c holds elements [c*32*VEC + l*VEC, +VEC):
// one 16-, 32- or 64-byte coalesced load.
//
// Method: "MXNorm: Reusing MXFP block scales for efficient tensor
// normalisation", Resumen tecnico, 2. Metodologia: "Fundamentos Teoricos"
// (rho~ = c(p,B) ((1/K) sum_k m~_k^p)^(-1/p), read with m~_k = s_k, c = 1)
// and "Implementacion" (the block maxima of the cast feed the estimate in
// one pass); OCP MX v1.0 6.3 for the cast.
#pragma once

#include "launch.h"
#include "mx_row.cuh"

namespace mxnorm {
namespace warp_row {


constexpr int kWarpsPerCta = 8;

// L2 prefetch before the dependent-launch wait: 0 none (x in host memory),
// 1 each warp's first row (or pair of rows), 2 up to 32 of each warp's rows,
// taken when the whole input fits in kWholeInputPrefetchBytes (a quarter of
// L2).  Mode 2 measured 5 % faster at 16384 x 768 (25 MB in) and 3 % slower
// at 32768 x 2048 (128 MiB in), where it would cover a quarter of the rows.
constexpr int64_t kWholeInputPrefetchBytes = (int64_t)32 << 20;

__device__ __forceinline__ int prefetch_lanes(int mode) { return mode == 2 ? 32 : mode; }

inline int prefetch_mode(const WarpRowArgs& a) {
  if (!is_device_memory(a.x)) return 0;
  return a.T * a.H * 2 <= kWholeInputPrefetchBytes ? 2 : 1;
}

// MINB: CTAs per SM the register allocation must allow (occupancy floor).
// TILED: the scale layout (0 row-major, 1 MMA atoms) as a compile-time
// constant; taken at run time it cost up to a fifth of the bandwidth on
// short rows (per-row address work).
template <int FMT, int VEC, int NCHUNK, int AHEAD, bool EXACT, bool LOAD32, bool ESTIMATE, int MINB, int TILED>
__global__ void __launch_bounds__(kWarpsPerCta * 32, MINB)
    mx_warp_row_kernel(const uint16_t* __restrict__ x, int64_t T, int H, uint8_t* __restrict__ codes,
                       uint8_t* __restrict__ scales, float* __restrict__ inv_rms, int p, int /*scale_tiled*/,
                       int l2_prefetch) {
  const int64_t warp0 = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
  pdl_launch_dependents();
  {
    // lane l prefetches the warp's l-th row: lane 0 alone in mode 1, up to 32 rows in mode 2
    const int64_t r = warp0 + (int64_t)(threadIdx.x & 31) * nwarps;
    if ((threadIdx.x & 31) < prefetch_lanes(l2_prefetch) && r < T) prefetch_l2(x + r * (int64_t)H, (uint32_t)(2 * H));
  }
  pdl_wait();
  mx_rows_stream<FMT, VEC, NCHUNK, AHEAD, EXACT, LOAD32, ESTIMATE>(x, T, H, codes, scales, inv_rms, p,
                                                                   warp0, nwarps, TILED);
}

// Two rows per warp (mx_rows_stream_half) for H = NCHUNK * 16 * VEC.
template <int FMT, int VEC, int NCHUNK, int AHEAD, bool ESTIMATE, int MINB, int TILED>
__global__ void __launch_bounds__(kWarpsPerCta * 32, MINB)
    mx_warp_2row_kernel(const uint16_t* __restrict__ x, int64_t T, int H, uint8_t* __restrict__ codes,
                        uint8_t* __restrict__ scales, float* __restrict__ inv_rms, int p, int /*scale_tiled*/,
                        int l2_prefetch) {
  const int64_t warp0 = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
  pdl_launch_dependents();
  {
    // lane l prefetches the warp's l-th pair of rows (lane 0 alone in mode 1)
    const int64_t pr = warp0 + (int64_t)(threadIdx.x & 31) * nwarps;
    if ((threadIdx.x & 31) < prefetch_lanes(l2_prefetch) && 2 * pr < T)
      prefetch_l2(x + 2 * pr * (int64_t)H, (uint32_t)(2 * H * (2 * pr + 1 < T ? 2 : 1)));
  }
  pdl_wait();
  mx_rows_stream_half<FMT, VEC, NCHUNK, AHEAD, true, ESTIMATE>(x, T, H, codes, scales, inv_rms, p, warp0, nwarps,
                                                               TILED);
}

// Any H (a multiple of 32): batches of four chunks per row.
template <int FMT, int VEC, bool LOAD32, bool ESTIMATE>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    mx_warp_row_generic_kernel(const uint16_t* __restrict__ x, int64_t T, int H,
                               uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                               float* __restrict__ inv_rms, int p, int scale_tiled, int l2_prefetch) {
  using Tr = FmtTraits<FMT>;
  const int64_t w0 = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  pdl_launch_dependents();
  if (l2_prefetch && (threadIdx.x & 31) == 0 && w0 < T)  // up to 64 KiB of the warp's first row
    prefetch_l2(x + w0 * (int64_t)H, (uint32_t)min(2 * H, 65536));
  pdl_wait();
  const int64_t code_row = Tr::fp4 ? (int64_t)(H / 2) : (int64_t)H;
  const int64_t warp0 = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
  for (int64_t row = warp0; row < T; row += nwarps) {
    const uint16_t* xr = x + row * (int64_t)H;
    auto load = [xr](int e0, uint32_t (&w)[VEC / 2]) { load_lane<VEC, LOAD32>(xr + e0, w); };
    mx_row<FMT, VEC, 0, ESTIMATE>(load, H, p, codes + row * code_row, scales, row, scale_tiled, inv_rms + row);
  }
}

template <class Kern>
cudaError_t launch_kernel(Kern kern, const WarpRowArgs& a, cudaStream_t stream, int rows_per_warp = 1) {
  const int64_t rows_per_cta = (int64_t)kWarpsPerCta * rows_per_warp;
  const int grid = persistent_grid(reinterpret_cast<const void*>(kern), kWarpsPerCta * 32,
                                   (a.T + rows_per_cta - 1) / rows_per_cta);
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kWarpsPerCta * 32), 0, stream, static_cast<const uint16_t*>(a.x),
                    a.T, (int)a.H, static_cast<uint8_t*>(a.codes), a.scales, a.inv_rms, a.p, a.scale_tiled,
                    prefetch_mode(a));
}

// Ring depth (chunks in flight per warp) and occupancy floor (CTAs of 8
// warps per SM the register budget must allow), per (format, lane width,
// chunks per row).  Chosen by interleaved timing of every candidate on
// 512 MiB inputs on GB300: FP8 rows with 32-byte lanes run best at depth 1
// with 3 CTAs/SM (80 registers; 64 registers lose ILP), FP4 rows (the H16
// rotation makes them ALU-heavier) at depth 2 with 4 CTAs/SM, and short rows
// of 16-byte lanes with the whole row in flight.  64-byte lanes (whole
// block per lane, used by the H32 rotation) hold 16 words per chunk.
template <int FMT, int VEC, int NCHUNK>
struct StreamTuning {
  static constexpr bool fp4 = FmtTraits<FMT>::fp4;
  // Unrotated FP8 rows of 16-byte lanes: 8192- and 2048-element rows keep 4
  // chunks in flight at 2 CTAs/SM; 1024-element rows the whole row at 3.
  static constexpr bool plain_fp8 = !fp4 && FmtTraits<FMT>::rot == 0;
  static constexpr bool fp8_deep = plain_fp8 && VEC == 16 && (NCHUNK == 16 || NCHUNK == 4);
  static constexpr bool fp8_two = plain_fp8 && VEC == 16 && NCHUNK == 2;
  static constexpr int ahead = (VEC == 8) ? NCHUNK
                               : (VEC == 32) ? ((!FmtTraits<FMT>::fp4 && NCHUNK % 2 == 0) ? 2 : 1)
                               : fp8_deep ? 4
                               : (fp4 && NCHUNK % 2 == 0) ? 2 : (NCHUNK == 2 ? 2 : 1);
  // 64-byte lanes: FP8 at 2 CTAs/SM, FP4 (H16 and H32) at 3 (80 registers;
  // measured 7 % and 3 % faster than 2)
  static constexpr int minb = (VEC == 32) ? (fp4 ? 3 : 2)
                              : fp8_deep ? 2
                              : fp8_two ? 3
                              : (VEC == 8 && NCHUNK == 1) ? 8 : (!fp4 && NCHUNK >= 8) ? 3 : 4;
};

template <int FMT, int VEC, int NCHUNK, bool LOAD32, bool ESTIMATE, int TILED>
cudaError_t launch_stream_layout(const WarpRowArgs& a, cudaStream_t s) {
  using Tu = StreamTuning<FMT, VEC, NCHUNK>;
  if (a.H == (int64_t)NCHUNK * 32 * VEC)
    return launch_kernel(mx_warp_row_kernel<FMT, VEC, NCHUNK, Tu::ahead, true, LOAD32, ESTIMATE, Tu::minb, TILED>, a,
                         s);
  return launch_kernel(mx_warp_row_kernel<FMT, VEC, NCHUNK, Tu::ahead, false, LOAD32, ESTIMATE, Tu::minb, TILED>, a,
                       s);
}

template <int FMT, int VEC, int NCHUNK, bool LOAD32, bool ESTIMATE>
cudaError_t launch_stream(const WarpRowArgs& a, cudaStream_t s) {
  if (a.scale_tiled) return launch_stream_layout<FMT, VEC, NCHUNK, LOAD32, ESTIMATE, 1>(a, s);
  return launch_stream_layout<FMT, VEC, NCHUNK, LOAD32, ESTIMATE, 0>(a, s);
}

// Two rows per warp, 32-byte lanes (interleaved sweeps, MXFP8 p = 2):
//   1 chunk  (H = 256): depth 1, 4 CTAs/SM (96 % of the HBM copy peak
//            against 68 % for one row per warp);
//   2 chunks (H = 512): the whole row in flight, 3 CTAs/SM (3 % faster than
//            one row per warp);
//   3 chunks (H = 768): the whole row, 2 CTAs/SM (100 % against 88 % for
//            one row per warp with 16-byte lanes);
//   4 chunks (H = 1024): depth 2, 3 CTAs/SM (3 % faster);
//   5 chunks (H = 1280): the whole row, 2 CTAs/SM.
template <int FMT, int NCHUNK, bool ESTIMATE>
cudaError_t launch_2row(const WarpRowArgs& a, cudaStream_t s) {
  constexpr int AHEAD = NCHUNK == 4 ? 2 : NCHUNK;
  constexpr int MINB = NCHUNK == 1 ? 4 : (NCHUNK == 2 || NCHUNK == 4) ? 3 : 2;
  if (a.scale_tiled)
    return launch_kernel(mx_warp_2row_kernel<FMT, 16, NCHUNK, AHEAD, ESTIMATE, MINB, 1>, a, s, 2);
  return launch_kernel(mx_warp_2row_kernel<FMT, 16, NCHUNK, AHEAD, ESTIMATE, MINB, 0>, a, s, 2);
}

template <int FMT, int VEC, bool LOAD32, bool ESTIMATE>
cudaError_t launch_by_h(const WarpRowArgs& a, cudaStream_t s) {
  const int64_t CE = 32 * VEC;
  switch ((a.H + CE - 1) / CE) {
    case 1: return launch_stream<FMT, VEC, 1, LOAD32, ESTIMATE>(a, s);
    case 2: return launch_stream<FMT, VEC, 2, LOAD32, ESTIMATE>(a, s);
    case 3: return launch_stream<FMT, VEC, 3, LOAD32, ESTIMATE>(a, s);
    case 4: return launch_stream<FMT, VEC, 4, LOAD32, ESTIMATE>(a, s);
    case 8: return launch_stream<FMT, VEC, 8, LOAD32, ESTIMATE>(a, s);
    case 16: return launch_stream<FMT, VEC, 16, LOAD32, ESTIMATE>(a, s);
    default: return launch_kernel(mx_warp_row_generic_kernel<FMT, VEC, LOAD32, ESTIMATE>, a, s);
  }
}

// Lane width: a whole 32-element block per lane for the H32 rotation and
// for H16 when 1024-element chunks tile the row (two rotation groups per
// lane, no shuffle for the block maximum: measured 6.7 % faster than
// 16-element lanes for MXFP4+H16 at H = 4096, 3.2 % for MXFP8+H16), 16
// elements for H16 otherwise or when 512-element chunks tile the row,
// else 8.
template <int FMT, bool ESTIMATE>
cudaError_t launch_fmt(const WarpRowArgs& a, cudaStream_t s) {
  constexpr int rot = FmtTraits<FMT>::rot;
  const bool x32 = (reinterpret_cast<uintptr_t>(a.x) & 31) == 0;
  if constexpr (rot != 32) {
    // H = 256 x {1, 3, 5}: two rows per warp (rows of 512 x odd bytes keep
    // 32-byte lanes aligned when x is)
    if (x32 && a.H % 512 == 256) {
      switch (a.H / 256) {
        case 1: return launch_2row<FMT, 1, ESTIMATE>(a, s);
        case 3: return launch_2row<FMT, 3, ESTIMATE>(a, s);
        case 5: return launch_2row<FMT, 5, ESTIMATE>(a, s);
        default: break;
      }
    }
    // unrotated FP8 rows of 512 and 1024 elements too (measured faster than
    // one row per warp; the other formats keep their lanes)
    if constexpr (rot == 0 && !FmtTraits<FMT>::fp4) {
      if (x32 && a.H == 512) return launch_2row<FMT, 2, ESTIMATE>(a, s);
      if (x32 && a.H == 1024) return launch_2row<FMT, 4, ESTIMATE>(a, s);
    }
  }
  if constexpr (rot == 32) {
    if (x32) return launch_by_h<FMT, 32, true, ESTIMATE>(a, s);
    return launch_by_h<FMT, 32, false, ESTIMATE>(a, s);
  } else {
    if constexpr (rot == 16) {
      if (a.H % 1024 == 0) {
        if (x32) return launch_by_h<FMT, 32, true, ESTIMATE>(a, s);
        return launch_by_h<FMT, 32, false, ESTIMATE>(a, s);
      }
    }
    if (rot == 16 || a.H % 512 == 0) {
      if (x32) return launch_by_h<FMT, 16, true, ESTIMATE>(a, s);
      return launch_by_h<FMT, 16, false, ESTIMATE>(a, s);
    }
    if constexpr (rot == 0) return launch_by_h<FMT, 8, false, ESTIMATE>(a, s);
    return cudaErrorInvalidValue;
  }
}

}  // namespace warp_row

// Per-format entry points, one translation unit each (mxnorm_warp_fp8*.cu,
// mxnorm_warp_fp4*.cu); _cast is the E4M3 cast without the estimate.
cudaError_t launch_warp_row_e4m3(const WarpRowArgs& a, cudaStream_t s);
cudaError_t launch_warp_row_e4m3_cast(const WarpRowArgs& a, cudaStream_t s);
cudaError_t launch_warp_row_e4m3_h16(const WarpRowArgs& a, cudaStream_t s);
cudaError_t launch_warp_row_e4m3_h32(const WarpRowArgs& a, cudaStream_t s);
cudaError_t launch_warp_row_e2m1(const WarpRowArgs& a, cudaStream_t s);
cudaError_t launch_warp_row_e2m1_h16(const WarpRowArgs& a, cudaStream_t s);
cudaError_t launch_warp_row_e2m1_h32(const WarpRowArgs& a, cudaStream_t s);

}  // namespace mxnorm
