// mx_device.cuh -- device-side building blocks shared by the libmxnorm kernels.
//
// Formats (OCP Microscaling Formats v1.0, sections 5 and 6.3):
//   * MX block: 32 consecutive elements along H sharing one E8M0 scale.
//   * E8M0 scale code = e + 127, value 2^e, e in [-127, 127]; 0xFF = NaN.
//   * shared exponent e = floor(log2 amax) - emax_elem, emax_elem = 8 for FP8
//     E4M3 (max 448) and 2 for FP4 E2M1 (max 6); an all-zero block gets -127.
//   * element codes: saturating round-to-nearest-even of v * 2^-e; the
//     hardware cvt.rn.satfinite conversions implement exactly that map (the
//     exhaustive cast tests hold them to it).
// Estimator ("MXNorm: Reusing MXFP block scales for efficient tensor
// normalisation", Resumen tecnico, 2. Metodologia, Fundamentos Teoricos):
//   inv_rms = c(p,B) * ((1/K) sum_k s_k^p)^(-1/p) with s_k = 2^e_k, c = 1.
// The power mean runs on the integer exponents, as a fixed-point sum of
// 2^(F + p (e_k - m)) relative to the running maximum m (PowerMeanAcc).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace mxnorm {

constexpr int kBlock = 32;               // MX block size
constexpr int kFixedBits = 48;           // F: fixed-point fraction bits of the power-mean sum
constexpr int kMaxH = 1 << 20;           // K <= 2^15 keeps K * 2^F below 2^64
constexpr int kExpNone = -1000;          // "no block seen yet" for the running maximum

enum Fmt : int {
  kFmtE4M3 = 0,      // MXFP8 E4M3
  kFmtE2M1 = 1,      // MXFP4 E2M1
  kFmtE2M1H16 = 2,   // (1/4) H16 rotation, then MXFP4
  kFmtE4M3H16 = 3,   // (1/4) H16 rotation, then MXFP8
  kFmtE2M1H32 = 4,   // H32 / sqrt(32) rotation, then MXFP4
  kFmtE4M3H32 = 5,   // H32 / sqrt(32) rotation, then MXFP8
};
constexpr int kNumFmts = 6;

template <int FMT>
struct FmtTraits {
  static constexpr bool fp4 = FMT == kFmtE2M1 || FMT == kFmtE2M1H16 || FMT == kFmtE2M1H32;
  static constexpr int emax = fp4 ? 2 : 8;  // largest element exponent: 6 = 1.5*2^2, 448 = 1.75*2^8
  static constexpr int rot = (FMT == kFmtE2M1H16 || FMT == kFmtE4M3H16) ? 16
                             : (FMT == kFmtE2M1H32 || FMT == kFmtE4M3H32) ? 32 : 0;
};

// ------------------------------------------------------ dependent launch
// Programmatic dependent launch (the streaming kernels are launched with
// programmatic stream serialisation, launch_pdl in launch.h): first let
// the next grid on the stream be scheduled as this one's CTAs finish, then
// wait until the previous grid on the stream has completed and its writes
// are visible.  Called before any global memory access, so stream order is
// kept; what overlaps is one launch's start with the previous one's end.
// Without a programmatic predecessor the wait returns at once.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_launch_dependents();
  pdl_wait();
}

// Bring `bytes` (a multiple of 16, p 16-byte aligned) at p into L2 without
// waiting (the TMA engine's bulk prefetch).  A hint with no effect on memory
// semantics: L2 is the GPU's point of coherence, so a line prefetched
// before a predecessor kernel writes it is updated in place.  The streaming
// kernels issue it for their first rows between pdl_launch_dependents and
// pdl_wait, so the first DRAM round trip overlaps the previous kernel's end.
// Device memory only (the launcher checks): never at mapped host memory.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ loads
// Streaming 16-byte load: read once, keep it out of L1.
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Streaming 32-byte load (sm_100+ 256-bit global load); p must be 32-byte aligned.
__device__ __forceinline__ void ldg_stream32(const void* p, uint32_t (&w)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}

__device__ __forceinline__ void stg16(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void stg8(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void stg4(void* p, uint32_t a) {
  asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}

// bf16x2 word -> two fp32 values (exact: bf16 is the top half of a binary32).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ------------------------------------------------------ packed fp32 pairs
// sm_100+ executes add/sub/mul on two fp32 lanes of a 64-bit register pair
// per instruction; each half is rounded exactly like the scalar op (.rn,
// no flush to zero).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// v[i] *= s for every element, two per instruction.
template <int N>
__device__ __forceinline__ void scale_pairs(float (&v)[N], float s) {
  const unsigned long long ss = f2_pack(s, s);
#pragma unroll
  for (int i = 0; i < N; i += 2) f2_unpack(f2_mul(f2_pack(v[i], v[i + 1]), ss), v[i], v[i + 1]);
}

// ------------------------------------------------------------ exponents
// Shared exponent from the biased exponent field of the block absmax:
// floor(log2 amax) = field - 127 for normal amax; zero and subnormal amax
// give an exponent below -127 + emax and clamp to -127 (bf16 and fp32 alike).
template <int EMAX>
__device__ __forceinline__ int shared_exponent(int exp_field) {
  return max(exp_field - 127 - EMAX, -127);
}

// 2^-e as an fp32 for e in [-127, 125] (biased field 127 - e in [2, 254]).
__device__ __forceinline__ float exp2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// ----------------------------------------------------------------- casts
// Two fp32 -> packed E4M3x2 (lo element in the low byte), saturating RNE.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Four fp32 -> four E4M3 bytes in one word (element 0 in the low byte).
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d) {
  return cvt_e4m3x2(a, b) | (cvt_e4m3x2(c, d) << 16);
}
// Eight fp32 -> eight E2M1 nibbles in one word (element 0 in the low nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                               float v5, float v6, float v7) {
  uint32_t r;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return r;
}

// ------------------------------------------------------------------- H16
// y = (1/4) H16 v in place for 16 fp32 values: Sylvester Hadamard in natural
// order, butterfly stages h = 1, 2, 4, 8, each add/sub rounded to fp32, then
// the 1/4 scale ("Entrenamiento Previo ... con MXFP4", Metodologia, item 3:
// deterministic 16x16 Hadamard rotation before the MXFP4 cast).
// The stages are evaluated on the pairs q_j = (v_j, v_{j+8}), j = 0..7: for
// h = 1, 2, 4 a packed add/sub of q_i and q_{i+h} is exactly the scalar
// butterfly on (v_i, v_{i+h}) and on (v_{i+8}, v_{i+h+8}); stage 8 combines
// the two halves of each pair.  Every element sees the same fp32 operations
// in the same stage order as the scalar definition, so results are
// bit-identical to it.
__device__ __forceinline__ void h16_inplace(float (&v)[16]) {
  unsigned long long q[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) q[j] = f2_pack(v[j], v[j + 8]);
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if ((i & h) == 0) {
        const unsigned long long a = q[i], b = q[i + h];
        q[i] = f2_add(a, b);
        q[i + h] = f2_sub(a, b);
      }
    }
  }
  const unsigned long long quarter = f2_pack(0.25f, 0.25f);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float lo, hi;
    f2_unpack(q[j], lo, hi);
    const unsigned long long y = f2_pack(__fadd_rn(lo, hi), __fsub_rn(lo, hi));
    f2_unpack(f2_mul(y, quarter), v[j], v[j + 8]);
  }
}

// y = H32 v / sqrt(32) in place for 32 fp32 values: butterfly stages
// h = 1, 2, 4, 8, 16 in fp32, then each value times RN_fp32(1/sqrt(32)).
// Same pairing idea as h16_inplace with q_j = (v_j, v_{j+16}): stages 1..8
// packed, stage 16 across the halves; bit-identical to the scalar order.
__device__ __forceinline__ void h32_inplace(float (&v)[32]) {
  unsigned long long q[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) q[j] = f2_pack(v[j], v[j + 16]);
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const unsigned long long a = q[i], b = q[i + h];
        q[i] = f2_add(a, b);
        q[i + h] = f2_sub(a, b);
      }
    }
  }
  const float c32 = 0.17677669f;  // RN_fp32(1/sqrt(32)) = 0x3E3504F3
  const unsigned long long cc = f2_pack(c32, c32);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float lo, hi;
    f2_unpack(q[j], lo, hi);
    const unsigned long long y = f2_pack(__fadd_rn(lo, hi), __fsub_rn(lo, hi));
    f2_unpack(f2_mul(y, cc), v[j], v[j + 16]);
  }
}

// ------------------------------------------------------------ power mean
// Running fixed-point sum S = sum_k 2^(F + p (e_k - m)) with m the largest
// exponent seen; terms below 2^0 are dropped and right shifts truncate, so
// the relative error is below K * 2^-F.  Merging two partial sums rescales
// both to the larger maximum.
struct PowerMeanAcc {
  int m;
  unsigned long long s;
};

__device__ __forceinline__ unsigned long long shr64(unsigned long long v, int sh) {
  return sh >= 64 ? 0ull : (v >> sh);
}

__device__ __forceinline__ void pm_add(PowerMeanAcc& a, int e, int p) {
  if (e > a.m) {
    a.s = shr64(a.s, p * (e - a.m));
    a.m = e;
  }
  const int t = kFixedBits + p * (e - a.m);
  if (t >= 0) a.s += 1ull << t;
}

__device__ __forceinline__ PowerMeanAcc pm_merge(PowerMeanAcc a, PowerMeanAcc b, int p) {
  PowerMeanAcc r;
  r.m = max(a.m, b.m);
  r.s = shr64(a.s, p * (r.m - a.m)) + shr64(b.s, p * (r.m - b.m));
  return r;
}

__device__ __forceinline__ PowerMeanAcc pm_warp_reduce(PowerMeanAcc a, int p) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    PowerMeanAcc o;
    o.m = __shfl_xor_sync(0xFFFFFFFFu, a.m, off);
    o.s = __shfl_xor_sync(0xFFFFFFFFu, a.s, off);
    a = pm_merge(a, o, p);
  }
  return a;
}

// inv_rms = 2^-m * (K / S_real)^(1/p) with S_real = S * 2^-F, i.e.
// 1 / M_p with M_p = ((1/K) sum_k 2^(p e_k))^(1/p).  fp32 throughout: S
// rounds once to fp32, K * 2^F / S is one IEEE division, the square root
// (p = 2) is IEEE, and 2^-m scales exactly (m <= 125 for bf16 or rotated
// fp32 input, so 2^-m and the result stay normal).  Relative error below
// 2^-22 (two roundings of 2^-24 plus the fixed-point truncation).
__device__ __forceinline__ float pm_inv_rms(PowerMeanAcc a, int K, int p) {
  const float s = __ull2float_rn(a.s);
  const float kf = __uint_as_float((uint32_t)(127 + kFixedBits) << 23) * (float)K;  // K * 2^F, exact
  float q = __fdiv_rn(kf, s);
  if (p == 2) q = __fsqrt_rn(q);
  return __fmul_rn(q, exp2_neg(a.m));
}

}  // namespace mxnorm
