// mxnorm_tiled.cu -- row-tiled MXNorm kernel with bulk async copies (the TMA
// engine) staging row tiles of x into a shared-memory ring.
//
// Persistent CTAs (grid = SMs x resident CTAs).  Each CTA walks tiles of
// R = 8 consecutive rows (tile i of the CTA is tile blockIdx.x + i*gridDim.x).
// Rows of a tile are contiguous in x, so one cp.async.bulk moves a whole
// tile (R*H*2 bytes) into one stage of a STAGES-deep ring; its completion
// is tracked by the stage's "full" mbarrier (transaction bytes).  Warp 0's
// elected lane is the producer; warps 1..8 are consumers, one row of the
// tile each, running the same per-row code as the warp-row kernel on
// shared-memory loads, then arriving on the stage's "empty" mbarrier.
// The producer refills a stage after all eight consumers released it.
//
// Every wait is bounded by a wall-clock deadline (%globaltimer, one second
// unless the launch asks for less): on expiry the waiter sets bit 0 of the
// device error word (read with mxnorm_device_errors) and stops; before the
// CTA exits, the producer waits (bounded by one second) for every copy it
// issued, so no bulk copy can still be writing into shared memory of a
// retired CTA.  The failure-detection drill (mxnorm_tiled_wait_drill) runs
// the same kernel with a short limit and one tile whose copy the producer
// never issues: the consumers of that tile, and the producer waiting for
// them to release its stage, give up after the limit; the drain skips the
// withheld copy, since none is in flight.
//
// Method as in the warp-row kernel ("MXNorm: Reusing MXFP block scales ...",
// Resumen tecnico, 2. Metodologia, Fundamentos Teoricos / Implementacion).
#include "launch.h"
#include "mx_row.cuh"

namespace mxnorm {

__device__ unsigned int g_device_error_word = 0u;

namespace {

constexpr int kConsumers = 8;                 // consumer warps = rows per tile
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kSmemBudget = 200 * 1024;       // ring bytes per CTA
constexpr int kMaxStages = 8;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s: the normal limit, and the drain's

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// try_wait with a suspend-time hint: the waiting thread sleeps until the
// phase completes or hint_ns runs out, instead of spinning (1.2 % faster
// for this kernel).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0u;
}

// Bounded wait for the phase with the given parity; false after limit_ns
// (and the device error word then has bit 0 set).  Each try sleeps at most
// 1 ms and never longer than the limit itself.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  const uint32_t hint = (uint32_t)(limit_ns < 1000000ull ? limit_ns : 1000000ull);
  if (mbar_try_wait(bar, parity, hint)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity, hint)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(&g_device_error_word, 1u);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

template <int VEC>
__device__ __forceinline__ void lds_lane(uint32_t saddr, uint32_t (&w)[VEC / 2]) {
#pragma unroll
  for (int q = 0; q < VEC / 8; ++q) {
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[4 * q]), "=r"(w[4 * q + 1]), "=r"(w[4 * q + 2]), "=r"(w[4 * q + 3])
                 : "r"(saddr + 16u * q));
  }
}

template <int FMT, int VEC, int NCHUNK>
__global__ void __launch_bounds__(kThreads, 1)
    mx_tiled_kernel(const uint16_t* __restrict__ x, int64_t T, int H, uint8_t* __restrict__ codes,
                    uint8_t* __restrict__ scales, float* __restrict__ inv_rms, int p, int stages,
                    unsigned long long wait_ns, int64_t withheld_tile) {
  using Tr = FmtTraits<FMT>;
  extern __shared__ __align__(128) unsigned char smem[];
  // layout: [full mbarriers x kMaxStages][empty x kMaxStages] then the ring
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  unsigned char* ring = smem + 2 * kMaxStages * sizeof(uint64_t);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row_bytes = (int64_t)H * 2;
  const int64_t stage_bytes = row_bytes * kConsumers;
  const int64_t ntiles = (T + kConsumers - 1) / kConsumers;
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = smem_addr(bars + kMaxStages);
  const uint32_t ring0 = smem_addr(ring);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kConsumers);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = evict_first_policy();
      int64_t issued = 0, withheld_at = -1;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, ++issued) {
        const int s = (int)(issued % stages);
        const uint32_t use = (uint32_t)(issued / stages);
        if (use > 0) ok = mbar_wait_bounded(empty0 + 8 * s, (use - 1) & 1u, wait_ns);
        if (!ok) break;
        if (tile == withheld_tile) {  // drill: this stage's phase never completes
          withheld_at = issued;
          continue;
        }
        const int64_t r0 = tile * kConsumers;
        const int64_t nrows = min((int64_t)kConsumers, T - r0);
        const uint32_t bytes = (uint32_t)(nrows * row_bytes);
        mbar_arrive_expect_tx(full0 + 8 * s, bytes);
        bulk_g2s(ring0 + (uint32_t)(s * stage_bytes), x + r0 * H, bytes, full0 + 8 * s, pol);
      }
      // Drain: the last use of every stage must have landed before exit
      // (a withheld copy was never issued, so there is nothing to wait for).
      for (int64_t i = (issued > stages ? issued - stages : 0); i < issued; ++i) {
        if (i == withheld_at) continue;
        const int s = (int)(i % stages);
        (void)mbar_wait_bounded(full0 + 8 * s, (uint32_t)(i / stages) & 1u);
      }
    }
    return;
  }

  const int r = warp - 1;  // consumer's row within each tile
  int64_t i = 0;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
    const int s = (int)(i % stages);
    const uint32_t use = (uint32_t)(i / stages);
    if (!mbar_wait_bounded(full0 + 8 * s, use & 1u, wait_ns)) break;
    const int64_t row = tile * kConsumers + r;
    if (row < T) {
      const uint32_t srow = ring0 + (uint32_t)(s * stage_bytes + r * row_bytes);
      auto load = [srow](int e0, uint32_t (&w)[VEC / 2]) { lds_lane<VEC>(srow + 2u * (uint32_t)e0, w); };
      const int64_t code_row = Tr::fp4 ? (int64_t)(H / 2) : (int64_t)H;
      mx_row<FMT, VEC, NCHUNK, true>(load, H, p, codes + row * code_row, scales, row, 0, inv_rms + row);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
}

int stages_for(int64_t H) {
  const int64_t stage_bytes = H * 2 * kConsumers;
  int64_t s = kSmemBudget / stage_bytes;
  if (s > kMaxStages) s = kMaxStages;
  return (int)s;
}

size_t smem_for(int stages, int64_t H) {
  return 2 * kMaxStages * sizeof(uint64_t) + (size_t)stages * (size_t)(H * 2 * kConsumers);
}

template <int FMT, int VEC, int NCHUNK>
cudaError_t launch_one(const TiledArgs& t, cudaStream_t s) {
  const WarpRowArgs& a = t.base;
  auto kern = mx_tiled_kernel<FMT, VEC, NCHUNK>;
  const int stages = stages_for(a.H);
  const size_t smem = smem_for(stages, a.H);
  cudaError_t err = cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t ntiles = (a.T + kConsumers - 1) / kConsumers;
  const int grid = persistent_grid(reinterpret_cast<const void*>(kern), kThreads, ntiles, smem);
  kern<<<grid, kThreads, smem, s>>>(static_cast<const uint16_t*>(a.x), a.T, (int)a.H,
                                    static_cast<uint8_t*>(a.codes), a.scales, a.inv_rms, a.p, stages,
                                    t.wait_limit_ns, t.withheld_tile);
  return cudaGetLastError();
}

template <int FMT, int VEC>
cudaError_t launch_by_h(const TiledArgs& t, cudaStream_t s) {
  const int64_t CE = 32 * VEC;
  switch ((t.base.H + CE - 1) / CE) {
    case 1: return launch_one<FMT, VEC, 1>(t, s);
    case 2: return launch_one<FMT, VEC, 2>(t, s);
    case 3: return launch_one<FMT, VEC, 3>(t, s);
    case 4: return launch_one<FMT, VEC, 4>(t, s);
    case 8: return launch_one<FMT, VEC, 8>(t, s);
    default: return launch_one<FMT, VEC, 0>(t, s);
  }
}

template <int FMT>
cudaError_t launch_fmt(const TiledArgs& t, cudaStream_t s) {
  constexpr int rot = FmtTraits<FMT>::rot;
  if constexpr (rot == 32) {
    return launch_by_h<FMT, 32>(t, s);
  } else {
    if (rot == 16 || t.base.H % 512 == 0) return launch_by_h<FMT, 16>(t, s);
    if constexpr (rot == 0) return launch_by_h<FMT, 8>(t, s);
    return cudaErrorInvalidValue;
  }
}

}  // namespace

bool tiled_supported(int64_t H, int fmt) {
  (void)fmt;
  return H >= kBlock && H % kBlock == 0 && stages_for(H) >= 2;
}

cudaError_t read_device_error_word(uint32_t* out, bool clear) {
  unsigned int v = 0;
  cudaError_t err = cudaMemcpyFromSymbol(&v, g_device_error_word, sizeof v);
  if (err != cudaSuccess) return err;
  *out = v;
  if (clear) {
    const unsigned int zero = 0;
    err = cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof zero);
  }
  return err;
}

cudaError_t launch_mxnorm_tiled(const TiledArgs& t, cudaStream_t s) {
  switch (t.base.fmt) {
    case kFmtE4M3: return launch_fmt<kFmtE4M3>(t, s);
    case kFmtE2M1: return launch_fmt<kFmtE2M1>(t, s);
    case kFmtE2M1H16: return launch_fmt<kFmtE2M1H16>(t, s);
    case kFmtE4M3H16: return launch_fmt<kFmtE4M3H16>(t, s);
    case kFmtE2M1H32: return launch_fmt<kFmtE2M1H32>(t, s);
    case kFmtE4M3H32: return launch_fmt<kFmtE4M3H32>(t, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mxnorm
