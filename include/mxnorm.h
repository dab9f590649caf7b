/*
 * mxnorm.h -- C ABI of libmxnorm: MXNorm's fused MX-quantise + scale-reuse
 * inverse-RMS pass, and the two-pass RMSNorm-then-MXFP8 baseline, for
 * NVIDIA GB300 (sm_103a).
 *
 * Method.  "MXNorm: Reusing MXFP block scales for efficient tensor
 * normalisation" (gist.science summary), Resumen tecnico:
 *   - 2. Metodologia, "Fundamentos Teoricos": the inverse RMS is estimated
 *     as rho~ = c(p,B) * ((1/K) sum_{k=1..K} m~_k^p)^(-1/p) over the K = H/B
 *     blocks of a row, p = 1 (arithmetic) or 2 (quadratic power mean);
 *   - 2. Metodologia, "Implementacion": one fused pass computes the block
 *     maxima, the estimate and the MX codes; the gain gamma is folded into
 *     the next linear layer's weight (MXNormLinear), so no gamma here;
 *   - the paper's English abstract: the RMS comes from the block scales of
 *     the MXFP8 cast, a reduction 32x smaller than RMSNorm's.
 * Encodings and the shared-exponent rule: OCP Microscaling Formats (MX)
 * v1.0, sections 5 and 6.3.  MXFP4 with a deterministic 16x16 Hadamard
 * rotation: "Entrenamiento Previo de Modelos de Lenguaje Grandes con MXFP4"
 * (gist.science summary), Metodologia, item 3.
 *
 * What one call computes, per row of x (bf16, H elements, H % 32 == 0):
 *   v      = x, or for the *_H16 formats the rotation (1/4) H16 applied to
 *            each aligned group of 16 elements in fp32 (Sylvester order,
 *            butterfly stages 1, 2, 4, 8, each add rounded to fp32, then
 *            * 1/4), or for the *_H32 formats H32 / sqrt(32) on each block
 *            (stages 1 .. 16, then * RN_fp32(1/sqrt(32)) = 0x3E3504F3);
 *   a_k    = max |v_j| over block k (32 elements), k = 0..K-1;
 *   e_k    = max(floor(log2 a_k) - emax, -127), emax = 8 (E4M3) or 2 (E2M1),
 *            e_k = -127 when a_k = 0;  scales[k] = e_k + 127 (E8M0);
 *   codes  = saturating round-to-nearest-even of v_j * 2^-e_k in FP8 E4M3
 *            (one byte per element) or FP4 E2M1 (two elements per byte,
 *            element 2i in the LOW nibble); the sign of v_j is kept, so -0
 *            and negatives that round to zero encode as 0x80 (E4M3) / 0x8;
 *   inv_rms = ((1/K) sum_k 2^(p e_k))^(-1/p), fp32 (c(p,B) = 1: a caller
 *            that wants the corrected estimate multiplies by c, e.g. folded
 *            with gamma into the consumer weight).
 * A block holding Inf or NaN gets scale 0xFF (E8M0 NaN), codes 0x7F (E4M3)
 * or 0 (E2M1), and its row's inv_rms is NaN.
 *
 * Memory and ownership.  Every pointer is a device-accessible pointer owned
 * by the caller: device memory, or pinned host memory mapped into the
 * device's address space (the kernel then reads and writes it across the
 * host link).  Row-major, densely packed (row stride = row length):
 *   x        bf16   [T, H]          16-byte aligned
 *   codes    uint8  [T, H]  (E4M3 formats)  16-byte aligned
 *            uint8  [T, H/2] (E2M1 formats)
 *   scales   uint8  [T, H/32]       any alignment
 *   inv_rms  float  [T]             4-byte aligned
 * No call allocates device memory (the one buffer the library holds is the
 * static workspace of rmsnorm_mxfp8_ref_fwd_static_ws, below); the library
 * keeps no state between calls except a per-thread error string and a
 * per-device cache of launch shapes, and it never
 * synchronises: work is queued on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and the call returns.  Outputs are fully
 * written when the stream reaches the kernel's end; after an error return
 * they are unspecified.  Inputs and outputs must not overlap.
 * The streaming kernels (the fused pass, NVFP4, the backward, the RMSNorm
 * baseline's first kernel, the gain-folded cast) are launched with
 * programmatic stream serialisation: each may be scheduled while the
 * previous kernel on the stream finishes, waits for that kernel's
 * completion before any load or store, and lets the next kernel be
 * scheduled early.  Before the wait it may prefetch its first input rows
 * into L2 (device memory only): a hint with no effect on what any load
 * returns, since L2 is the GPU's point of coherence.  Stream order holds as usual; a kernel of the caller's
 * launched after one of them with the programmatic-serialisation attribute
 * must, as any programmatic dependent, wait (griddepcontrol.wait,
 * cudaGridDependencySynchronize) before reading its outputs.
 *
 * Errors.  Arguments are checked on the host before any launch:
 *   T < 0, H <= 0, H % 32 != 0, p not in {1, 2}, unknown fmt or variant,
 *   a NULL pointer                              -> MXNORM_ERR_INVALID_ARG
 *   H > MXNORM_MAX_H, or a variant that does not
 *   support the shape                           -> MXNORM_ERR_UNSUPPORTED
 *   a pointer below its alignment               -> MXNORM_ERR_MISALIGNED
 *   a CUDA launch error                         -> MXNORM_ERR_CUDA
 * T == 0 returns MXNORM_OK and launches nothing.  mxnorm_last_error() gives
 * the calling thread's last message.  There is no CPU fallback.
 */
#ifndef MXNORM_H_
#define MXNORM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MXNORM_BLOCK 32
#define MXNORM_MAX_H (1 << 20)
#define MXNORM_ABI_VERSION 1

typedef enum {
  MXNORM_FMT_MXFP8_E4M3 = 0,      /* FP8 E4M3 codes, one byte per element            */
  MXNORM_FMT_MXFP4_E2M1 = 1,      /* FP4 E2M1 codes, two per byte                    */
  MXNORM_FMT_MXFP4_E2M1_H16 = 2,  /* (1/4) H16 rotation, then FP4 E2M1 codes         */
  MXNORM_FMT_MXFP8_E4M3_H16 = 3,  /* (1/4) H16 rotation, then FP8 E4M3 codes         */
  MXNORM_FMT_MXFP4_E2M1_H32 = 4,  /* H32/sqrt(32) rotation, then FP4 E2M1 codes      */
  MXNORM_FMT_MXFP8_E4M3_H32 = 5   /* H32/sqrt(32) rotation, then FP8 E4M3 codes      */
} mxnorm_fmt;

typedef enum {
  MXNORM_OK = 0,
  MXNORM_ERR_INVALID_ARG = 1,
  MXNORM_ERR_UNSUPPORTED = 2,
  MXNORM_ERR_MISALIGNED = 3,
  MXNORM_ERR_CUDA = 4
} mxnorm_status;

typedef enum {
  MXNORM_VARIANT_AUTO = 0,       /* the library picks                        */
  MXNORM_VARIANT_WARP_ROW = 1,   /* one warp per row, vector loads            */
  MXNORM_VARIANT_TILED_TMA = 2   /* row tiles staged in shared memory by bulk
                                    async copies (TMA engine), persistent CTAs */
} mxnorm_variant;

/* Layouts of the E8M0 scales a call writes or reads. */
#define MXNORM_SCALE_ROW_MAJOR 0   /* scales[row * (H/32) + k]                          */
#define MXNORM_SCALE_MMA 1         /* the 512-byte atoms the block-scaled tensor-core MMA
                                    * reads (H % 128 == 0): one atom per 128 rows x 4
                                    * blocks, atoms ordered (row tile, block group) with
                                    * the block group fastest; inside an atom the byte of
                                    * (r, k) is at (r % 32) * 16 + ((r / 32) % 4) * 4 + k % 4.
                                    * Rows are padded to a multiple of 128: the buffer
                                    * holds mxnorm_mma_scale_bytes(T, H) bytes, and the
                                    * bytes of padding rows are unspecified. */

/* Bytes of an MXNORM_SCALE_MMA scale buffer for rows x H (-1 if H % 128 != 0). */
int64_t mxnorm_mma_scale_bytes(int64_t rows, int64_t H);

/* MXNorm forward: MX codes + E8M0 scales + fp32 inverse-RMS estimate of
 * every row of x, in one pass over x (the estimator of "Fundamentos
 * Teoricos" evaluated on the scales of the cast, see above).
 * p: 1 or 2.  fmt: an mxnorm_fmt.  stream: cudaStream_t or NULL. */
int mxnorm_quant_fwd(const void* x, int64_t T, int64_t H, int p, int fmt, void* codes,
                     uint8_t* scales, float* inv_rms, void* stream);

/* As mxnorm_quant_fwd, with an explicit kernel variant (mxnorm_variant).
 * Every variant writes bit-identical outputs. */
int mxnorm_quant_fwd_ex(const void* x, int64_t T, int64_t H, int p, int fmt, void* codes,
                        uint8_t* scales, float* inv_rms, int variant, void* stream);

/* As mxnorm_quant_fwd (variant AUTO) with the scales written in
 * scale_layout (MXNORM_SCALE_ROW_MAJOR or MXNORM_SCALE_MMA); the MMA layout
 * feeds mxnorm_linear_fwd without a conversion pass. */
int mxnorm_quant_fwd_layout(const void* x, int64_t T, int64_t H, int p, int fmt, void* codes, uint8_t* scales,
                            float* inv_rms, int scale_layout, void* stream);

/* The MX cast alone (no estimator) of T rows of H bf16 values: MXFP8 E4M3
 * codes [T, H] and E8M0 scales in scale_layout.  Used for the consumer
 * weight of MXNormLinear: pass the rows of W'^T (one per output feature,
 * W' = diag(c * gamma) W) to get the w_codes / w_scales of
 * mxnorm_linear_fwd.  fmt must be MXNORM_FMT_MXFP8_E4M3. */
int mx_cast_fwd(const void* x, int64_t T, int64_t H, int fmt, void* codes, uint8_t* scales, int scale_layout,
                void* stream);

/* MXFP8 cast of MXNormLinear's gain-folded weight in one pass ("MXNorm ...",
 * Resumen tecnico, 2. Metodologia, "Implementacion": the norm's gain, with
 * the estimator constant c, moves into the next linear layer's weight).
 * w: bf16 [N, K] device, row n = the weights of output feature n (W^T of
 * y = x W), 16-byte aligned.  gamma: fp32 [K] device, 16-byte aligned.
 * Element (n, k) of the cast input is w[n, k] * g_k with
 * g_k = RN_fp32(c * gamma_k), each product rounded to fp32 (IEEE
 * round-to-nearest-even, subnormals kept); then each 32-element block gets
 * its E8M0 scale and saturating RNE E4M3 codes exactly as mx_cast_fwd.  A
 * block holding Inf/NaN after the product gets scale 0xFF and codes 0x7F.
 * codes: E4M3 [N, K] device, 16-byte aligned; scales: scale_layout
 * (MXNORM_SCALE_MMA gives the w_scales of mxnorm_linear_fwd; needs
 * K % 128 == 0).  Preconditions: N >= 0, 0 < K <= MXNORM_MAX_H,
 * K % 32 == 0, c finite.  Errors: INVALID_ARG / MISALIGNED / UNSUPPORTED,
 * checked before any launch; N == 0 returns OK with no launch.  The call
 * owns no memory and is asynchronous on stream (cudaStream_t or NULL). */
int mx_cast_gain_fwd(const void* w, int64_t N, int64_t K, const float* gamma, float c, void* codes,
                     uint8_t* scales, int scale_layout, void* stream);

/* Consumer side of MXNormLinear ("MXNorm ...", Resumen tecnico, 2.
 * Metodologia, "Implementacion": the gain is folded into the next linear
 * layer's weight): an MXFP8 block-scaled GEMM on the tensor cores whose
 * epilogue applies the row's inverse RMS,
 *     out[t, n] = bf16( inv_rms[t] * sum_k x^[t, k] * w^[n, k] ),
 * x^ / w^ the values of the E4M3 codes times their E8M0 block scales (32
 * elements along K), accumulated in fp32, the product with inv_rms rounded
 * to fp32 and then to bf16.
 *   x_codes   E4M3 [T, K]                 16-byte aligned
 *   x_scales  E8M0, MXNORM_SCALE_MMA      mxnorm_mma_scale_bytes(T, K) bytes
 *   inv_rms   f32  [T]                    e.g. from mxnorm_quant_fwd_layout
 *   w_codes   E4M3 [N, K]                 16-byte aligned
 *   w_scales  E8M0, MXNORM_SCALE_MMA      mxnorm_mma_scale_bytes(N, K) bytes
 *   out       bf16 [T, N]                 16-byte aligned
 * K % 128 == 0, K <= MXNORM_MAX_H, N % 256 == 0, N <= 2^24, any T below
 * 2^31.  The tensor-memory copies address rows with 32-bit coordinates, so
 * ceil(T/128) * K/32 and ceil(N/128) * K/32 must also stay below 2^31;
 * larger problems return MXNORM_ERR_UNSUPPORTED before any launch.  Errors
 * and stream semantics as mxnorm_quant_fwd; bit 1 of mxnorm_device_errors
 * reports a timed-out pipeline wait of this kernel. */
int mxnorm_linear_fwd(const void* x_codes, const uint8_t* x_scales, const float* inv_rms, const void* w_codes,
                      const uint8_t* w_scales, int64_t T, int64_t K, int64_t N, void* out, void* stream);

/* Two-pass baseline: the unfused pipeline MXNorm replaces ("MXNorm ...",
 * Resumen tecnico, section 1: RMSNorm and the MXFP8 cast as separate
 * operations).  Kernel 1: inv = 1/sqrt(mean(x^2) + eps) in fp32 (the sum
 * of squares, the mean and + eps each rounded to fp32, then a correctly
 * rounded fp32 reciprocal square root), y = bf16(fp32(x * inv)) written to
 * y_workspace, inv to inv_rms.
 * Kernel 2: MXFP8 E4M3 cast of y (same rules as above) into codes/scales.
 * y_workspace: bf16 [T, H], 16-byte aligned, caller-owned; it holds y on
 * return.  No gain (gamma = 1). */
int rmsnorm_mxfp8_ref_fwd(const void* x, int64_t T, int64_t H, float eps, void* y_workspace,
                          uint8_t* codes, uint8_t* scales, float* inv_rms, void* stream);

/* MXNorm over the NVFP4 cast.  The pages quote its Llama 3 8B layer speedup
 * ("MXNorm ...", Resumen tecnico, section 4, Rendimiento) without the
 * format; the recipe here: 16-element blocks of FP4 E2M1 values, one UE4M3
 * scale per block, an fp32 tensor scale g > 0 given by the caller (e.g.
 * amax / (448 * 6) from mxnorm_absmax_bf16).  Per block, in fp32 with IEEE
 * rounding: sb = amax / (6 g); s = E4M3(sb) saturating RNE; d = s g;
 * enc = 1 / d (0 when s = 0); codes = E2M1(x * enc) saturating RNE, sign
 * kept, element 2i in the low nibble.  The estimator takes the decode scales
 * s_k g:  inv_rms = ((1/K) sum_k (s_k g)^p)^(-1/p), K = H/16; +Inf for an
 * all-zero row.  A block holding Inf/NaN gets scale 0x7F, codes 0, and its
 * row's inv_rms is NaN.
 *   x        bf16  [T, H], H % 16 == 0   16-byte aligned
 *   codes    uint8 [T, H/2]              16-byte aligned
 *   scales   uint8 [T, H/16] (UE4M3)
 *   inv_rms  f32   [T]                   4-byte aligned
 * Errors as mxnorm_quant_fwd (a non-finite or non-positive tensor_scale is
 * MXNORM_ERR_INVALID_ARG). */
int mxnorm_quant_fwd_nvfp4(const void* x, int64_t T, int64_t H, int p, float tensor_scale, void* codes,
                           uint8_t* scales, float* inv_rms, void* stream);

/* As mxnorm_quant_fwd_nvfp4, with the tensor scale read from device memory
 * at the start of the kernel (tensor_scale: one fp32, 4-byte aligned), so a
 * scale derived on the device -- mxnorm_nvfp4_tensor_scale on the same
 * stream -- reaches the cast without a host round trip.  The value must be
 * finite and > 0: otherwise the outputs are unspecified and bit 2 of
 * mxnorm_device_errors is set.  Other errors and stream semantics as
 * mxnorm_quant_fwd_nvfp4. */
int mxnorm_quant_fwd_nvfp4_dev(const void* x, int64_t T, int64_t H, int p, const float* tensor_scale,
                               void* codes, uint8_t* scales, float* inv_rms, void* stream);

/* The NVFP4 tensor scale of n bf16 values, on the device: with a the
 * largest finite |x| (Inf and NaN elements are skipped; the cast marks
 * their blocks anyway), *tensor_scale = RN_fp32(a / 2688) -- 2688 = 448 * 6,
 * so the tensor's largest block gets the largest E4M3 block scale -- or 1
 * when no finite element is nonzero.  Always a finite positive fp32.
 * tensor_scale: device pointer to one fp32 (4-byte aligned), written on
 * `stream` (zeroed, reduced into, then converted: the call queues three
 * operations and returns). */
int mxnorm_nvfp4_tensor_scale(const void* x, int64_t n, float* tensor_scale, void* stream);

/* max |x| over n bf16 values, written as an fp32 to the device pointer amax
 * (NaN if any x is NaN).  Zeroes *amax first on the same stream. */
int mxnorm_absmax_bf16(const void* x, int64_t n, float* amax, void* stream);

/* Straight-through backward of MXNorm ("MXNorm ...", Resumen tecnico,
 * 2. Metodologia, "Gradientes": RMSNorm's gradient logic reused through a
 * straight-through estimator, nothing kept but what RMSNorm keeps).  The MX
 * cast counts as the identity and RMSNorm's backward runs with the forward's
 * estimate rho~ = inv_rms in place of 1/RMS:
 *     dx = rho~ * dy - rho~^3 * x * (1/H) * sum_j dy_j * x_j
 * (fp32 arithmetic, dx rounded to bf16).  Works as plain RMSNorm's backward
 * when inv_rms holds the exact 1/RMS.
 *   x        bf16 [T, H]  the forward's input            16-byte aligned
 *   dy       bf16 [T, H]  gradient w.r.t. x * rho~        16-byte aligned
 *   inv_rms  f32  [T]     the forward's estimate           4-byte aligned
 *   dx       bf16 [T, H]  output                           16-byte aligned
 * Errors and stream semantics as mxnorm_quant_fwd. */
int mxnorm_bwd_ste(const void* x, const void* dy, const float* inv_rms, int64_t T, int64_t H, void* dx,
                   void* stream);

/* Allocation-free form of rmsnorm_mxfp8_ref_fwd.  The paper has no
 * counterpart: this exists for callers that cannot allocate device memory
 * (a host framework that owns every allocation through its own pool, a
 * latency-critical path that cannot afford cudaMalloc's implicit
 * synchronisation, a device-memory budget fixed up front).  The bf16
 * workspace between the two kernels lives in a file-scope device array of
 * MXNORM_STATIC_WS_BYTES compiled into the library, held by every GPU that
 * loads it until the process exits; the call itself allocates nothing.
 *   - T * H must not exceed MXNORM_STATIC_WS_BYTES / 2 (16,777,216 bf16
 *     elements); larger problems return MXNORM_ERR_UNSUPPORTED.
 *   - All calls on a device share the array: calls whose work overlaps on
 *     the GPU (other streams, other host threads) race on it and must be
 *     serialised by the caller.  The array keeps the last call's y; nothing
 *     in it needs to start at zero.
 *   - Every call looks up the array's address in the current device's
 *     context (cudaGetSymbolAddress, host-side, no device work), so it
 *     stays valid after cudaDeviceReset or under another context; the first
 *     call on a device may load the library's module into that context:
 *     make it before any stream capture.
 * Arguments, outputs and other errors as rmsnorm_mxfp8_ref_fwd without
 * y_workspace. */
#define MXNORM_STATIC_WS_BYTES (32u << 20)
int rmsnorm_mxfp8_ref_fwd_static_ws(const void* x, int64_t T, int64_t H, float eps, uint8_t* codes,
                                    uint8_t* scales, float* inv_rms, void* stream);

/* Static text for a status code. */
const char* mxnorm_status_string(int status);

/* The calling thread's last error message ("" if none). */
const char* mxnorm_last_error(void);

/* MXNORM_ABI_VERSION of the loaded library. */
int mxnorm_abi_version(void);

/* Failure-detection drill for the tiled variant's bounded waits: the
 * MXFP8, p = 2 pass of mxnorm_quant_fwd_ex with MXNORM_VARIANT_TILED_TMA,
 * except that the producer never issues the copy of one 8-row tile
 * (withheld_tile, in [0, ceil(T/8))) and every pipeline wait gives up after
 * wait_limit_ns (in [1e5, 1e9] ns) instead of one second.  The consumers of
 * that tile, and the producer waiting for them to release its stage, give
 * up after the limit; the kernel ends, bit 0 of mxnorm_device_errors is
 * set, and the call's outputs are invalid (the withheld tile's rows, and
 * later rows of the CTA that owned it, are never written).  No copy is left
 * in flight and nothing faults: a caller can check its failure handling end
 * to end, then clear the word and carry on with the same context.
 * Arguments and other errors as mxnorm_quant_fwd_ex (T == 0 is
 * MXNORM_ERR_INVALID_ARG here). */
int mxnorm_tiled_wait_drill(const void* x, int64_t T, int64_t H, void* codes, uint8_t* scales, float* inv_rms,
                            int64_t withheld_tile, int64_t wait_limit_ns, void* stream);

/* Device-side error word of the current device, or'ed by kernels whose
 * bounded waits gave up (bit 0: a shared-memory pipeline wait of the tiled
 * variant timed out; bit 1: one of mxnorm_linear_fwd; bit 2: the device
 * tensor scale given to mxnorm_quant_fwd_nvfp4_dev was not a finite
 * positive float; the outputs of the affected call are then invalid).
 * Synchronous: copies the word to *flags (and zeroes it when clear != 0).
 * Call after the work in question has completed. */
int mxnorm_device_errors(uint32_t* flags, int clear);

#ifdef __cplusplus
}
#endif

#endif /* MXNORM_H_ */
