// mxnorm_linear.cu -- consumer side of MXNormLinear on the 5th-generation
// tensor cores: an MXFP8 block-scaled GEMM whose epilogue applies MXNorm's
// per-row inverse RMS.
//
// "MXNorm: Reusing MXFP block scales for efficient tensor normalisation",
// Resumen tecnico, 2. Metodologia, "Implementacion": MXNormLinear folds the
// norm's gain into the next linear layer's weight, so the layer computes
//     out[t, n] = rho~[t] * sum_k x^[t, k] w'^[n, k]
// with x^ the MXFP8 codes and E8M0 block scales of the row (mxnorm_quant_fwd
// with the MMA scale layout), rho~ = inv_rms, and w'^ the MXFP8 cast of
// W' = diag(c gamma) W, i.e. one row per output feature, quantised along K
// (mx_cast_gain_fwd folds c gamma in and casts in one pass; mx_cast_fwd casts
// a weight that already holds them).  The row scale commutes with the
// matmul, so it is applied once per output element in the epilogue.
//
// Tiling: 256 x 256 output tiles, each computed by a pair of CTAs on the two
// SMs of a TPC (a cluster of 2): tcgen05.mma with cta_group::2, M = 256
// (128 rows per CTA), N = 256, kind::mxf8f6f4 with 1X E8M0 block scales, one
// instruction per 32-element K step.  Each CTA stages its own 128 x rows and
// one half (128 rows) of the tile's 256 w rows, K 128 bytes at a time
// through a 6-deep shared-memory ring; the pair's tensor cores read both w
// halves, so every w byte crosses L2 -> SM once per pair rather than once per
// CTA.  Persistent pairs, warp-specialised (11 warps, 352 threads per CTA):
//   warp 0 lane 0  TMA producer (both CTAs): 2-D tiled loads of the CTA's x
//                  rows and w half (128-byte swizzle) per stage and, every
//                  g stages, of the 512-byte scale atoms of those g stages
//                  (its own x atoms, the atoms of both w halves; one copy
//                  per operand, since consecutive stages' atoms are
//                  contiguous), all completing on the leader's stage "full"
//                  mbarrier (cta_group::2 form), which expects both CTAs'
//                  bytes;
//   warp 1 lane 0  leader CTA: MMA issuer.  At every even stage it waits
//                  for "sf_full" (which covers that stage and the next),
//                  per stage it issues four tcgen05.mma and commits to the
//                  "empty" mbarriers of both CTAs (multicast); after a tile's
//                  last stage it commits to both CTAs' "acc_full";
//   warp 2 lane 0  leader CTA: scale-factor copier.  Per pair of stages
//                  (2i, 2i + 1; the last alone when the count is odd) it
//                  waits for each stage's "full", copies its atoms into both
//                  CTAs' TMEM (tcgen05.cp, cta_group::2: each CTA's shared
//                  memory into its own TMEM), then commits once to the even
//                  stage's "sf_full".  Copies issued by the MMA thread itself
//                  would wait between its stages; from a thread of their own
//                  they overlap the MMAs in flight, and one hand-off per two
//                  stages halves the issuer's waits;
//   warps 3-10     epilogue (both CTAs), two per TMEM lane quadrant (32 rows)
//                  with 128 columns each: tcgen05.ld of all 128 fp32
//                  accumulators at once (one wait), then, before any other
//                  work, an arrival on the leader's "acc_empty" (16 per
//                  tile) frees TMEM for the next tile's MMAs; the values are
//                  multiplied by rho~[row],
//                  rounded to packed bf16 in registers, and each lane stores
//                  its row's 128 outputs straight to global memory (32-byte
//                  stores when out is 32-byte aligned, else 16-byte ones).
// Each CTA's tensor core reads the B scales of all 256 columns from its own
// TMEM, so both CTAs load both w atoms.  TMEM (512 columns, allocated for the
// pair): accumulators in columns 0-255, the scale factors of ring stage s in
// columns 256 + 16 s (A: 4 columns, B: 8).  Every mbarrier wait is bounded
// (2 s by %globaltimer); on expiry the waiter sets bit 0 of the linear error
// word and the pair winds down, waiting (bounded) for its own bulk copies and
// MMAs before it frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "launch.h"
#include "mx_device.cuh"

namespace mxnorm {

__device__ unsigned int g_linear_error_word = 0u;

namespace {

constexpr int BM = 128, BN = 256, BK = 128;     // BM rows per CTA (256 per pair); BK bytes = E4M3 elements
constexpr int kStages = 6;
// The copy warp signals once per pair of stages (2i, 2i + 1) on the even
// stage's barrier, so each barrier's uses stay kStages stages apart.
static_assert(kStages % 2 == 0, "pairs of stages map onto the ring");
constexpr int kStageA = BM * BK;                 // 16 KiB
constexpr int kStageB = (BN / 2) * BK;           // 16 KiB: this CTA's half of the tile's w rows
// Scale atoms (512 bytes: 128 rows x 4 blocks) of consecutive K stages are
// contiguous in the MMA layout, so the producer loads those of a group of
// g = 4, 2 or 1 stages (whichever divides the tile's K stages) with one
// copy per operand, into a ring of group buffers: the x atoms, then the
// atoms of both w halves.  The producer refills a buffer only after the
// stage kStages before the refilling one has completed (its MMAs, so also
// the scale copies before them), so the last stage of the group the buffer
// held must lie at least kStages back: (groups - 1) g + 1 >= kStages, a
// ring of ceil((kStages - 1) / g) + 1 groups: 3, 4 or 6.
constexpr int kSfRing = 3 * 4 * 3 * 512;          // 18 KiB: the largest ring (3 groups of 4 stages)
constexpr int kEpiWarps = 8;                     // two per TMEM lane quadrant, 128 columns each
constexpr int kThreads = 32 * (3 + kEpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTxBytes = kStageA + kStageB;  // one CTA's operand bytes per stage
constexpr unsigned long long kWaitNs = 2000000000ull;
constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + (size_t)kStages * (kStageA + kStageB) + kSfRing + 256;

__host__ __device__ constexpr int sf_ring_groups(int g) { return (kStages - 1 + g - 1) / g + 1; }
static_assert(sf_ring_groups(4) * 3 * 4 * 512 <= kSfRing && sf_ring_groups(2) * 3 * 2 * 512 <= kSfRing &&
                  sf_ring_groups(1) * 3 * 512 <= kSfRing,
              "every scale-group ring fits its shared memory");


__device__ __forceinline__ uint32_t saddr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A waiting thread sleeps in try_wait until the phase completes or this
// hint runs out, instead of spinning: the eight epilogue warps wait through
// every tile's main loop, and spinning cost issue slots and power (8.7 %
// slower at the power cap, about 3 % in short runs).  The single-thread
// roles sleep too: letting them spin measured 11 % slower.
constexpr uint32_t kSuspendHintNs = 1000000u;

__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0u;
}

// Bounded wait; false (and bit 0 of the error word set) on timeout.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  if (try_wait(bar, parity)) return true;
  const unsigned long long t0 = gtimer();
  while (!try_wait(bar, parity)) {
    if (gtimer() - t0 > kWaitNs) {
      atomicOr(&g_linear_error_word, 1u);
      return false;
    }
  }
  return true;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive on an mbarrier of either CTA.  The default (CTA-scope) release:
// what the waiter needs ordered is the tcgen05 work fenced around the
// barrier, and a cluster-scope release here costs microseconds per arrival.
__device__ __forceinline__ void arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// All threads of both CTAs (per-thread form: callers may arrive diverged).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// K-major operand tile with 128-byte swizzle: 8-row atoms of 1024 bytes,
// leading offset unused, stride 1024 bytes, descriptor version 1.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// A 512-byte scale atom as a plain 32-row x 16-byte matrix (8-row groups
// 128 bytes apart) for tcgen05.cp.
__device__ __forceinline__ uint64_t desc_atom(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: E4M3 x E4M3,
// both K-major, E8M0 scales, M = 256 (the pair), N = 256, scale byte `sf` of
// each 32-bit TMEM scale word for A and B (the 32-element K step within the
// 128-element stage).
__device__ __forceinline__ uint32_t idesc_mxf8(int sf) {
  return ((uint32_t)sf << 4) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) | ((uint32_t)((2 * BM) >> 4) << 24) |
         ((uint32_t)sf << 29);
}

// 2-D tiled TMA load into this CTA's shared memory, completing on an
// mbarrier of either CTA of the pair (bar: a shared::cluster address), so
// the peer's loads count towards the leader's stage barrier directly.
__device__ __forceinline__ void tma_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Persistent tile order: groups of kGroupM 256-row tiles walk the column
// tiles together (row tile fastest inside a group), so the pairs running at
// one time share both their x and w tiles in L2.
constexpr int kGroupM = 16;
__device__ __forceinline__ void tile_coords(int64_t tile, int64_t num_m, int num_n, int64_t& mt, int& nt) {
  const int64_t per_group = (int64_t)kGroupM * num_n;
  const int64_t g = tile / per_group;
  const int64_t in = tile - g * per_group;
  const int64_t rows_here = min((int64_t)kGroupM, num_m - g * kGroupM);
  mt = g * kGroupM + in % rows_here;
  nt = (int)(in / rows_here);
}


// One lane's 128 consecutive bf16 outputs (64 packed words) to global
// memory: 32-byte stores (whole sectors) when the row start allows, else
// 16-byte ones.
template <bool kV8>
__device__ __forceinline__ void store_row128(uint16_t* dst, const uint32_t (&o)[64]) {
#pragma unroll
  for (int q = 0; q < 64; q += 8) {
    if constexpr (kV8) {
      asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + 2 * q), "r"(o[q]), "r"(o[q + 1]),
                   "r"(o[q + 2]), "r"(o[q + 3]), "r"(o[q + 4]), "r"(o[q + 5]), "r"(o[q + 6]), "r"(o[q + 7])
                   : "memory");
    } else {
      asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(dst + 2 * q), "r"(o[q]), "r"(o[q + 1]), "r"(o[q + 2]),
                   "r"(o[q + 3])
                   : "memory");
      asm volatile("st.global.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(dst + 2 * q + 8), "r"(o[q + 4]), "r"(o[q + 5]),
                   "r"(o[q + 6]), "r"(o[q + 7])
                   : "memory");
    }
  }
}

// 64 TMEM columns of this warp's 32 lanes (two 32-column loads, completed
// by the caller's tcgen05.wait::ld).
__device__ __forceinline__ void tmem_load64(uint32_t taddr, uint32_t (&v)[64]) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t* w = v + 32 * q;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]), "=r"(w[8]),
          "=r"(w[9]), "=r"(w[10]), "=r"(w[11]), "=r"(w[12]), "=r"(w[13]), "=r"(w[14]), "=r"(w[15]), "=r"(w[16]),
          "=r"(w[17]), "=r"(w[18]), "=r"(w[19]), "=r"(w[20]), "=r"(w[21]), "=r"(w[22]), "=r"(w[23]), "=r"(w[24]),
          "=r"(w[25]), "=r"(w[26]), "=r"(w[27]), "=r"(w[28]), "=r"(w[29]), "=r"(w[30]), "=r"(w[31])
        : "r"(taddr + (uint32_t)(32 * q)));
  }
}

// v * r in fp32 (IEEE products), rounded to bf16 and packed in pairs.
__device__ __forceinline__ void scale_pack64(const uint32_t (&v)[64], float r, uint32_t* o) {
  const unsigned long long rr = f2_pack(r, r);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float lo, hi;
    f2_unpack(f2_mul(f2_pack(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), rr), lo, hi);
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    o[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

template <bool kV8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mxfp8_linear_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_sfx, const __grid_constant__ CUtensorMap tm_sfw,
                        const float* __restrict__ inv_rms, uint16_t* __restrict__ out, int64_t T, int K, int N,
                        int sf_group) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + kStages * kStageA;
  uint8_t* sSF = sB + kStages * kStageB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sSF + kSfRing);
  // bars: full[kStages], empty[kStages], sf_full[kStages], acc_full, acc_empty, drain, drain_sf;
  // then the TMEM base word.  The leader's full[s] counts both CTAs' bytes; the peer uses only
  // empty[] and acc_full.
  const uint32_t full0 = saddr(bars), empty0 = saddr(bars + kStages), sf_full0 = saddr(bars + 2 * kStages);
  const uint32_t acc_full = saddr(bars + 3 * kStages), acc_empty = saddr(bars + 3 * kStages + 1);
  const uint32_t drain = saddr(bars + 3 * kStages + 2), drain_sf = saddr(bars + 3 * kStages + 3);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kStages + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int num_n = N / BN, num_kt = K / BK;
  const int sf_bufs = sf_ring_groups(sf_group), sf_bytes = 3 * sf_group * 512;
  const int64_t num_m = (T + 2 * BM - 1) / (2 * BM);  // 256-row tiles
  const int64_t row_atoms = (T + BM - 1) / BM;          // 128-row scale atoms of x
  const int64_t tiles = num_m * num_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(full0 + 8 * s));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(empty0 + 8 * s));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sf_full0 + 8 * s));
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(acc_full));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(acc_empty), "r"(2 * kEpiWarps));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(drain));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(drain_sf));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // one warp of each CTA allocates the pair's TMEM together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncwarp();
  cluster_sync();  // both CTAs' barriers are initialised before either arrives remotely
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int64_t it = 0;
      int sf_pos = 0, sf_buf = 0;  // stage within its scale group, the group's ring buffer
      bool ok = true;
      for (int64_t tile = pair; tile < tiles && ok; tile += npairs) {
        int64_t mt;
        int nt;
        tile_coords(tile, num_m, num_n, mt, nt);
        const int64_t xrow = (2 * mt + rank) * BM;
        // rows past T load as zeros (TMA); their scale atom is any valid one
        const int64_t xatom = min(2 * mt + (int64_t)rank, row_atoms - 1);
        for (int kt = 0; kt < num_kt; ++kt, ++it) {
          const int s = (int)(it % kStages);
          const uint32_t use = (uint32_t)(it / kStages);
          if (use > 0 && !(ok = wait_bounded(empty0 + 8 * s, (use - 1) & 1u))) break;
          const uint32_t fb = map_to_rank(full0 + 8 * s, 0);  // the leader's stage barrier
          const bool group_start = sf_pos == 0;  // groups tile the K stages of every tile
          if (rank == 0)
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full0 + 8 * s),
                         "r"(2 * (kTxBytes + (group_start ? (uint32_t)sf_bytes : 0u)))
                         : "memory");
          tma_2d_pair(saddr(sA + s * kStageA), &tm_x, kt * BK, (int)xrow, fb);
          tma_2d_pair(saddr(sB + s * kStageB), &tm_w, kt * BK, nt * BN + (int)rank * (BN / 2), fb);
          if (group_start) {
            // the group's scale atoms: 4 rows of the 128-byte-wide scale maps each
            const uint32_t sf = saddr(sSF + sf_buf * sf_bytes);
            tma_2d_pair(sf, &tm_sfx, 0, (int)(4 * (xatom * num_kt + kt)), fb);
            tma_2d_pair(sf + sf_group * 512, &tm_sfw, 0, (int)(4 * ((int64_t)(2 * nt) * num_kt + kt)), fb);
            tma_2d_pair(sf + 2 * sf_group * 512, &tm_sfw, 0, (int)(4 * ((int64_t)(2 * nt + 1) * num_kt + kt)), fb);
          }
          if (++sf_pos == sf_group) {
            sf_pos = 0;
            if (++sf_buf == sf_bufs) sf_buf = 0;
          }
        }
      }
      // every copy issued (both CTAs') must have landed before the pair may
      // exit: the leader waits for its barriers' last phases
      if (rank == 0)
        for (int64_t i = (it > kStages ? it - kStages : 0); i < it; ++i)
          (void)wait_bounded(full0 + 8 * (int)(i % kStages), (uint32_t)(i / kStages) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      int64_t it = 0, tcount = 0;
      bool ok = true;
      for (int64_t tile = pair; tile < tiles && ok; tile += npairs, ++tcount) {
        if (tcount > 0 && !(ok = wait_bounded(acc_empty, (uint32_t)((tcount - 1) & 1)))) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        for (int kt = 0; kt < num_kt; ++kt, ++it) {
          const int s = (int)(it % kStages);
          // the stage's operands have landed and its scale factors are in TMEM: the copy warp
          // signals once per pair of stages (2i, 2i + 1), on the even one's barrier
          if (!(it & 1) && !(ok = wait_bounded(sf_full0 + 8 * s, (uint32_t)(it / kStages) & 1u))) break;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t tsf = tmem + 256 + 16 * s;
          const uint32_t a0 = saddr(sA + s * kStageA), b0 = saddr(sB + s * kStageB);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t accum = (kt | j) ? 1u : 0u;
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %6, 0;\n\t"
                "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
                    tmem),
                "l"(desc_sw128(a0 + 32 * j)), "l"(desc_sw128(b0 + 32 * j)), "r"(idesc_mxf8(j)), "r"(tsf), "r"(tsf + 4),
                "r"(accum));
          }
          asm volatile(
              "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                  empty0 + 8 * s),
              "h"((uint16_t)3)
              : "memory");
        }
        if (!ok) break;
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                acc_full),
            "h"((uint16_t)3)
            : "memory");
      }
      // all MMAs and scale copies of this thread complete before TMEM is freed
      asm volatile(
          "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
              drain),
          "h"((uint16_t)1)
          : "memory");
      (void)wait_bounded(drain, 0);
    }
  } else if (warp == 2) {
    if (lane == 0 && rank == 0) {
      // Scale-factor copier: tcgen05.cp from a thread of its own, so the
      // copies overlap the MMAs in flight (issued from the MMA thread they
      // wait, in order, between its stages).  Slot s of TMEM is free again
      // once full[s] shows the next use of stage s: the producer refilled it
      // only after the MMAs that read the slot completed.
      const int64_t my_tiles = pair < tiles ? (tiles - 1 - pair) / npairs + 1 : 0;
      const int64_t total = my_tiles * num_kt;
      int sf_pos = 0, sf_buf = 0;  // the producer's scale-group walk, in step with it
      bool ok = true;
      for (int64_t it = 0; it < total && ok; it += 2) {
        // a pair of stages (the last one alone when the count is odd), one signal
        const int s0 = (int)(it % kStages);
        for (int64_t jt = it; jt < it + 2 && jt < total; ++jt) {
          const int s = (int)(jt % kStages);
          if (!(ok = wait_bounded(full0 + 8 * s, (uint32_t)(jt / kStages) & 1u))) break;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t tsf = tmem + 256 + 16 * s;
          const uint32_t sf = saddr(sSF + sf_buf * sf_bytes) + (uint32_t)(sf_pos * 512);
          if (++sf_pos == sf_group) {
            sf_pos = 0;
            if (++sf_buf == sf_bufs) sf_buf = 0;
          }
          asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(tsf), "l"(desc_atom(sf)));
          asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(tsf + 4),
                       "l"(desc_atom(sf + sf_group * 512)));
          asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(tsf + 8),
                       "l"(desc_atom(sf + 2 * sf_group * 512)));
        }
        if (!ok) break;
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                sf_full0 + 8 * s0),
            "h"((uint16_t)1)
            : "memory");
      }
      // its copies complete before TMEM is freed
      asm volatile(
          "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
              drain_sf),
          "h"((uint16_t)1)
          : "memory");
      (void)wait_bounded(drain_sf, 0);
    }
  } else {
    // Epilogue warps 3 .. 3 + kEpiWarps - 1: TMEM lane quadrant warp % 4
    // (the lanes a warp may access), columns 128 * half .. + 128.
    const int quad = warp & 3;
    const int half = (warp - 3) / 4;
    const uint32_t acc_empty_leader = map_to_rank(acc_empty, 0);
    int64_t tcount = 0;
    for (int64_t tile = pair; tile < tiles; tile += npairs, ++tcount) {
      if (!wait_bounded(acc_full, (uint32_t)(tcount & 1))) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // Read the warp's 32 x 128 share of the accumulators (all four loads
      // in flight, one wait) and hand TMEM back to the MMA issuer first; the
      // tile's coordinates and the row's inv_rms come after, off the MMAs'
      // path, and the next tile's MMAs overlap the conversion and stores.
      const uint32_t taddr = tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)(128 * half);
      uint32_t v[128];
      tmem_load64(taddr, *reinterpret_cast<uint32_t(*)[64]>(v));
      tmem_load64(taddr + 64, *reinterpret_cast<uint32_t(*)[64]>(v + 64));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) arrive_remote(acc_empty_leader);
      int64_t mt;
      int nt;
      tile_coords(tile, num_m, num_n, mt, nt);
      const int64_t row = (2 * mt + rank) * BM + 32 * quad + lane;
      const int c0 = nt * BN + 128 * half;
      const float r = row < T ? inv_rms[row] : 0.0f;
      uint32_t o[64];
      scale_pack64(*reinterpret_cast<uint32_t(*)[64]>(v), r, o);
      scale_pack64(*reinterpret_cast<uint32_t(*)[64]>(v + 64), r, o + 32);
      if (row < T) store_row128<kV8>(out + row * (int64_t)N + c0, o);
    }
  }

  // Neither CTA leaves (or frees TMEM) while the pair's MMAs may still read
  // its shared memory or the other CTA may still arrive on its barriers.
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncwarp();
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// rows x K uint8 codes, box of `box_rows` rows x 128 bytes, 128-byte swizzle
bool encode_codes(CUtensorMap* map, const void* base, int64_t rows, int64_t K, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// CTA pairs of the kernel that the current device runs at the same time
// (clusters stay inside one GPC, so this can be below SMs / 2), cached per
// device.
cudaError_t resident_pairs(const void* kern, int variant, int* out) {
  static std::mutex mu;
  static int cache[2][64] = {{0}};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && cache[variant][dev] > 0) {
    *out = cache[variant][dev];
    return cudaSuccess;
  }
  int sms = 0;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sms - sms % 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  int clusters = 0;
  if ((err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg)) != cudaSuccess) return err;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  if (dev >= 0 && dev < 64) cache[variant][dev] = clusters;
  *out = clusters;
  return cudaSuccess;
}

// MMA-layout scale bytes viewed as rows of 128 bytes (a 512-byte atom is 4
// rows), box of 4 g rows, no swizzle: one TMA load per group of g atoms.
bool encode_scales(CUtensorMap* map, const void* base, int64_t bytes, int g) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)(bytes / 128)};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, (cuuint32_t)(4 * g)};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_mxfp8_linear(const LinearArgs& a, cudaStream_t s) {
  CUtensorMap tm_x, tm_w, tm_sfx, tm_sfw;
  const int64_t num_kt = a.K / BK;
  const int g = num_kt % 4 == 0 ? 4 : num_kt % 2 == 0 ? 2 : 1;  // scale atoms loaded per copy
  const int64_t sfx_bytes = ((a.T + BM - 1) / BM) * num_kt * 512;
  const int64_t sfw_bytes = ((a.N + BM - 1) / BM) * num_kt * 512;
  if (!encode_codes(&tm_x, a.x_codes, a.T, a.K, BM) || !encode_codes(&tm_w, a.w_codes, a.N, a.K, BN / 2) ||
      !encode_scales(&tm_sfx, a.x_scales, sfx_bytes, g) ||
      !encode_scales(&tm_sfw, a.w_scales, sfw_bytes, g))
    return cudaErrorInvalidValue;
  // rows start 32-byte aligned when out is (N is a multiple of 256)
  const bool v8 = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;
  const void* kern = v8 ? reinterpret_cast<const void*>(mxfp8_linear_kernel<true>)
                        : reinterpret_cast<const void*>(mxfp8_linear_kernel<false>);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  int co_resident = 0;
  if ((err = resident_pairs(kern, v8 ? 0 : 1, &co_resident)) != cudaSuccess) return err;
  // persistent pairs: as many as can run at once (a pair that waited for a
  // second wave would start its share of tiles only after the first wave
  // finished), never more than tiles
  const int64_t tiles = ((a.T + 2 * BM - 1) / (2 * BM)) * (a.N / BN);
  const int64_t pairs = std::max<int64_t>(1, std::min<int64_t>(tiles, co_resident));
  const int grid = (int)(2 * pairs);
  if (v8)
    mxfp8_linear_kernel<true><<<grid, kThreads, kSmemBytes, s>>>(tm_x, tm_w, tm_sfx, tm_sfw, a.inv_rms,
                                                                 static_cast<uint16_t*>(a.out), a.T, (int)a.K,
                                                                 (int)a.N, g);
  else
    mxfp8_linear_kernel<false><<<grid, kThreads, kSmemBytes, s>>>(tm_x, tm_w, tm_sfx, tm_sfw, a.inv_rms,
                                                                  static_cast<uint16_t*>(a.out), a.T, (int)a.K,
                                                                  (int)a.N, g);
  return cudaGetLastError();
}

cudaError_t read_linear_error_word(uint32_t* out, bool clear) {
  unsigned int v = 0;
  cudaError_t err = cudaMemcpyFromSymbol(&v, g_linear_error_word, sizeof v);
  if (err != cudaSuccess) return err;
  *out = v;
  if (clear) {
    const unsigned int zero = 0;
    err = cudaMemcpyToSymbol(g_linear_error_word, &zero, sizeof zero);
  }
  return err;
}

}  // namespace mxnorm
