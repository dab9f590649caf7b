// mxnorm_nvfp4.cu -- MXNorm over the NVFP4 cast: 16-element blocks of FP4
// E2M1 values, a UE4M3 scale per block and an fp32 tensor scale g.
//
// The MXNorm pages quote a Llama 3 8B layer speedup with NVFP4 ("MXNorm:
// Reusing MXFP block scales ...", Resumen tecnico, section 4, Rendimiento)
// without describing the format; the recipe used here, per block in fp32:
//   sb   = RN(amax / RN(6 g))          (IEEE division)
//   s    = sat_RNE_E4M3(sb)            (block scale code, positive)
//   d    = RN(s g),  enc = RN(1/d)     (0 when s = 0)
//   code = sat_RNE_E2M1(RN(x * enc))   (element 2i in the low nibble)
// The estimator takes the decode scales s_k g as m~_k:
//   inv_rms = ((1/K) sum_k (s_k g)^p)^(-1/p),  K = H/16.
// An E4M3 value is M 2^e with integer M <= 15 and e = max(E,1) - 10, so
// sum_k s_k^p = 2^(-9p) sum_k M_k^p 2^(p (max(E_k,1) - 1)) is an exact
// integer sum (below 2^52 for K <= 2^16); only the final mean, root and the
// division by g round (fp32, IEEE).
//
// One warp per row (grid-stride), lane l of chunk c owning block
// 32 c + l: a 32-byte load, no block shuffles.  Rows stream through a ring
// of AHEAD chunk buffers as in the MXNorm warp-row kernel.
//
// The tensor scale comes from the caller, as an fp32 argument or as a
// device word (read by every thread at kernel start, so that a scale
// derived on the device needs no host round trip).  The library derives it
// from a tensor as g = RN(a / 2688), a the largest finite |x| (448 * 6:
// the tensor's largest block then gets the largest E4M3 scale), or 1 when
// no finite element is nonzero; a device word that is not a finite
// positive float sets bit 0 of g_nvfp4_error_word.
#include "launch.h"
#include "mx_row.cuh"

namespace mxnorm {

__device__ unsigned int g_nvfp4_error_word = 0u;

namespace {

constexpr int kWarps = 8;

// E4M3 code (positive) -> fp32 value.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t E = (c >> 3) & 0xFu, m = c & 7u;
  return E ? __uint_as_float(((E + 120u) << 23) | (m << 20)) : __fmul_rn((float)m, 0x1p-9f);
}

// One lane's block: stores its 8 code bytes and scale byte; returns the
// fixed-point term M^p 2^(p (max(E,1) - 1)) of s^p (or ~0ull for Inf/NaN).
__device__ __forceinline__ unsigned long long nvfp4_block(const uint32_t (&w)[8], bool valid, float sixg,
                                                          float g, int p, uint8_t* code_dst,
                                                          uint8_t* scale_dst) {
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16lo(w[i]);
    v[2 * i + 1] = bf16hi(w[i]);
  }
  const float amax = absmax_tree(v);
  const bool nonfinite = (__float_as_uint(amax) & 0x7FFFFFFFu) >= 0x7F800000u;
  const float sb = __fdiv_rn(nonfinite ? 0.0f : amax, sixg);
  const uint32_t sc = cvt_e4m3x2(sb, 0.0f) & 0xFFu;
  const float sval = e4m3_value(sc);
  const float enc = (sval == 0.0f) ? 0.0f : __frcp_rn(__fmul_rn(sval, g));
  scale_pairs(v, enc);
  if (valid) {
    uint32_t q0 = cvt_e2m1x8(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
    uint32_t q1 = cvt_e2m1x8(v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]);
    if (nonfinite) q0 = q1 = 0u;
    stg8(code_dst, q0, q1);
    *scale_dst = nonfinite ? (uint8_t)0x7F : (uint8_t)sc;
  }
  if (nonfinite) return ~0ull;
  const uint32_t E = (sc >> 3) & 0xFu, M = (E ? 8u : 0u) + (sc & 7u);
  const int sh = p * ((int)max(E, 1u) - 1);
  const unsigned long long mp = (p == 1) ? M : M * M;
  return mp << sh;
}

// inv_rms from the exact integer sum S = 2^(9p) sum_k s_k^p: +Inf for an
// all-zero row, NaN if a block held Inf/NaN.
__device__ __forceinline__ float nvfp4_inv(unsigned long long s, bool bad, int K, int p, float g) {
  if (bad) return __uint_as_float(0x7FC00000u);
  if (s == 0ull) return __uint_as_float(0x7F800000u);
  const float kscaled = (float)K * (p == 1 ? 512.0f : 262144.0f);  // K 2^(9p), exact
  float q = __fdiv_rn(kscaled, __ull2float_rn(s));
  if (p == 2) q = __fsqrt_rn(q);
  return __fdiv_rn(q, g);
}

template <int NCHUNK, int AHEAD, bool EXACT, bool LOAD32, int MINB>
__global__ void __launch_bounds__(kWarps * 32, MINB)
    nvfp4_row_kernel(const uint16_t* __restrict__ x, int64_t T, int H, int p, float g_arg,
                     const float* __restrict__ g_dev, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                     float* __restrict__ inv_rms, int l2_prefetch) {
  static_assert(NCHUNK == 0 || NCHUNK % AHEAD == 0, "the ring must tile the row");
  constexpr int CE = 512;
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();
  {
    const int64_t r0 = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);  // the warp's first row
    if (l2_prefetch && lane == 0 && r0 < T) prefetch_l2(x + r0 * (int64_t)H, (uint32_t)min(2 * H, 65536));
  }
  pdl_wait();
  float g = g_arg;
  if (g_dev != nullptr) {
    g = *g_dev;
    if (!(g > 0.0f && g <= 3.4028235e38f) && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&g_nvfp4_error_word, 1u);
  }
  const int Hc = (EXACT && NCHUNK > 0) ? NCHUNK * CE : H;
  const int K = Hc / 16;
  const float sixg = __fmul_rn(6.0f, g);
  int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int64_t rstride = (int64_t)gridDim.x * kWarps;
  if (row >= T) return;
  auto issue = [&](int64_t r, int c, uint32_t (&dst)[8]) {
    const int e0 = c * CE + lane * 16;
    if ((EXACT && NCHUNK > 0) || e0 < Hc) {
      load_lane<16, LOAD32>(x + r * (int64_t)Hc + e0, dst);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i] = 0u;
    }
  };
  if constexpr (NCHUNK > 0) {
    uint32_t buf[AHEAD][8];
#pragma unroll
    for (int a = 0; a < AHEAD; ++a) issue(row, a, buf[a]);
    for (; row < T; row += rstride) {
      const int64_t next = row + rstride;
      unsigned long long s = 0ull;
      bool bad = false;
#pragma unroll
      for (int c = 0; c < NCHUNK; ++c) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = buf[c % AHEAD][i];
        const int cc = c + AHEAD;
        if (cc < NCHUNK) issue(row, cc, buf[c % AHEAD]);
        else if (next < T) issue(next, cc - NCHUNK, buf[c % AHEAD]);
        const int e0 = c * CE + lane * 16;
        const bool valid = (EXACT && NCHUNK > 0) || e0 < Hc;
        const unsigned long long t = nvfp4_block(w, valid, sixg, g, p, codes + row * (int64_t)(Hc / 2) + e0 / 2,
                                                 scales + row * (int64_t)K + e0 / 16);
        if (valid) {
          if (t == ~0ull) bad = true;
          else s += t;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
      bad = __any_sync(0xFFFFFFFFu, bad);
      if (lane == 0) inv_rms[row] = nvfp4_inv(s, bad, K, p, g);
    }
  } else {
    const int nchunk = (H + CE - 1) / CE;
    for (; row < T; row += rstride) {
      unsigned long long s = 0ull;
      bool bad = false;
      for (int c = 0; c < nchunk; ++c) {
        uint32_t w[8];
        issue(row, c, w);
        const int e0 = c * CE + lane * 16;
        const bool valid = e0 < H;
        const unsigned long long t = nvfp4_block(w, valid, sixg, g, p, codes + row * (int64_t)(H / 2) + e0 / 2,
                                                 scales + row * (int64_t)K + e0 / 16);
        if (valid) {
          if (t == ~0ull) bad = true;
          else s += t;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
      bad = __any_sync(0xFFFFFFFFu, bad);
      if (lane == 0) inv_rms[row] = nvfp4_inv(s, bad, K, p, g);
    }
  }
}

template <int NCHUNK, int AHEAD, bool LOAD32, int MINB>
cudaError_t launch_one(const Nvfp4Args& a, cudaStream_t s) {
  const bool exact = NCHUNK > 0 && a.H == (int64_t)NCHUNK * 512;
  auto kern = exact ? nvfp4_row_kernel<NCHUNK, AHEAD, true, LOAD32, MINB>
                    : nvfp4_row_kernel<NCHUNK, AHEAD, false, LOAD32, MINB>;
  const int grid = persistent_grid(reinterpret_cast<const void*>(kern), kWarps * 32, (a.T + kWarps - 1) / kWarps);
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kWarps * 32), 0, s, static_cast<const uint16_t*>(a.x), a.T,
                    (int)a.H, a.p, a.g, a.g_dev, static_cast<uint8_t*>(a.codes), a.scales, a.inv_rms,
                    is_device_memory(a.x) ? 1 : 0);
}

// Four chunks in flight at 2 CTAs/SM time best on GB300 at H = 4096
// (98.8 % of the measured copy bandwidth; one chunk at 4 CTAs/SM 98.3 %,
// two at 4 CTAs/SM 94.5 %).
template <bool LOAD32>
cudaError_t launch_h(const Nvfp4Args& a, cudaStream_t s) {
  switch ((a.H + 511) / 512) {
    case 1: return launch_one<1, 1, LOAD32, 4>(a, s);
    case 2: return launch_one<2, 2, LOAD32, 4>(a, s);
    case 4: return launch_one<4, 4, LOAD32, 2>(a, s);
    case 8: return launch_one<8, 4, LOAD32, 2>(a, s);
    case 16: return launch_one<16, 4, LOAD32, 2>(a, s);
    default: return launch_one<0, 1, LOAD32, 4>(a, s);
  }
}

// max |x| over n bf16 values into *out (non-negative floats order like
// their bits, NaN above Inf; FINITE skips Inf and NaN): per-CTA tree, then
// one atomicMax per CTA.
template <bool FINITE>
__global__ void __launch_bounds__(256) absmax_bf16_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                          unsigned int* __restrict__ out) {
  unsigned int m = 0u;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t b = ((uint32_t)x[i] << 16) & 0x7FFFFFFFu;
    if (!FINITE || b < 0x7F800000u) m = max(m, b);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  __shared__ unsigned int red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i) m = max(m, red[i]);
    atomicMax(out, m);
  }
}

// In place: the largest finite magnitude's bits at *g become the tensor
// scale RN(a / 2688), or 1 when a = 0.
__global__ void nvfp4_scale_from_amax_kernel(float* g) {
  const float a = __uint_as_float(*reinterpret_cast<const unsigned int*>(g));
  *g = a > 0.0f ? __fdiv_rn(a, 2688.0f) : 1.0f;
}

template <bool FINITE>
cudaError_t launch_absmax(const void* x, int64_t n, float* amax, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(amax, 0, sizeof(float), s);
  if (err != cudaSuccess || n == 0) return err;
  auto kern = absmax_bf16_kernel<FINITE>;
  const int grid = persistent_grid(reinterpret_cast<const void*>(kern), 256, (n + 255) / 256);
  kern<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(x), n, reinterpret_cast<unsigned int*>(amax));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_nvfp4(const Nvfp4Args& a, cudaStream_t s) {
  const bool x32 = (reinterpret_cast<uintptr_t>(a.x) & 31) == 0;
  return x32 ? launch_h<true>(a, s) : launch_h<false>(a, s);
}

cudaError_t launch_absmax_bf16(const void* x, int64_t n, float* amax, cudaStream_t s) {
  return launch_absmax<false>(x, n, amax, s);
}

cudaError_t launch_nvfp4_tensor_scale(const void* x, int64_t n, float* g, cudaStream_t s) {
  cudaError_t err = launch_absmax<true>(x, n, g, s);
  if (err != cudaSuccess) return err;
  nvfp4_scale_from_amax_kernel<<<1, 1, 0, s>>>(g);
  return cudaGetLastError();
}

cudaError_t read_nvfp4_error_word(uint32_t* out, bool clear) {
  unsigned int v = 0;
  cudaError_t err = cudaMemcpyFromSymbol(&v, g_nvfp4_error_word, sizeof v);
  if (err != cudaSuccess) return err;
  *out = v;
  if (clear) {
    const unsigned int zero = 0;
    err = cudaMemcpyToSymbol(g_nvfp4_error_word, &zero, sizeof zero);
  }
  return err;
}

}  // namespace mxnorm
