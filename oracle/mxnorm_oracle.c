/*
 * mxnorm_oracle.c -- plain, slow, scalar CPU oracle for MXNorm.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library: every definition below is written out again from the format
 * and method definitions it cites.
 *
 * Sources (cited by title and section):
 *   [MXN]  "MXNorm: Reusing MXFP block scales for efficient tensor
 *          normalisation" (gist.science summary), "Resumen tecnico",
 *          section 2 "Metodologia: MXNorm", subsections "Fundamentos
 *          Teoricos" (the estimator formula for rho~ with c(p,B) and the
 *          power mean of K block maxima) and "Implementacion" (fusion of
 *          the norm with the MX cast).
 *   [ABS]  the same paper's English abstract (gptget.net page, section
 *          "Original abstract"): the RMS is estimated from the block scales
 *          computed by the MXFP8 cast, a 32x smaller reduction.
 *   [MXFP4] "Entrenamiento Previo de Modelos de Lenguaje Grandes con MXFP4"
 *          (gist.science summary), "Metodologia", item 3: deterministic
 *          16x16 Hadamard rotation (H16) before the MXFP4 cast.
 *   [OCP]  OCP Microscaling Formats (MX) v1.0: section 5 (E8M0 scale, FP8
 *          E4M3 and FP4 E2M1 element encodings) and section 6.3 (shared
 *          exponent = floor(log2(amax)) - emax_elem).
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *   - m~_k in the estimator is the E8M0 block scale value s_k = 2^e_k.
 *   - c(p,B) = 1 (the pages call it pre-computed but print no value).
 *   - e_k = clamp(floor(log2 a_k) - emax_elem, -127, 127); a_k = 0 -> -127.
 *   - element codes are the nearest finite grid value to v/s_k, ties to the
 *     code with an even last mantissa bit, magnitudes above the largest
 *     finite value saturate, and the sign bit is the sign of v (so -0 and
 *     negatives that round to zero keep the sign).
 *   - a block holding a NaN or an Inf gets scale code 0xFF (E8M0 NaN), E4M3
 *     codes 0x7F (E4M3 NaN) or E2M1 codes 0x0, and its row's inv_rms is NaN.
 *   - H16: fp32 butterfly, stages h = 1, 2, 4, 8 in that order, each pair
 *     (v_i, v_{i+h}) -> (v_i + v_{i+h}, v_i - v_{i+h}) rounded to fp32, then
 *     every value times 0.25 in fp32; no bf16 re-rounding.
 *   - H32: the same fp32 butterfly with stages h = 1, 2, 4, 8, 16, then every
 *     value times c32 = RN_fp32(1/sqrt(32)) in fp32 (the orthonormal
 *     H32/sqrt(32)); the page names H32 but not its normalisation.
 *   - E2M1 packing: element 2i in the low nibble of byte i.
 *   - RMSNorm baseline: inv = RN_fp32(1/sqrt(mean(x^2) + eps)),
 *     y = RN_bf16(RN_fp32(x * inv)), then the MXFP8 cast of y.
 *   - NVFP4 variant (the pages quote its layer speedup but not the format):
 *     16-element blocks, E2M1 elements, a UE4M3 block scale and a caller-
 *     given fp32 tensor scale g > 0.  Per block, in fp32: sixg = RN(6 g),
 *     sb = RN(amax / sixg), s = sat_RNE_E4M3(sb) (positive), d = RN(s g),
 *     enc = RN(1 / d) (0 when s = 0), r_j = RN(x_j * enc), codes =
 *     sat_RNE_E2M1(r_j).  The estimator's m~_k is the block's decode scale
 *     s_k * g; inv_rms = ((1/K) sum_k (s_k g)^p)^(-1/p), K = H/16, +Inf when
 *     every s_k is 0.  A block with Inf/NaN: scale code 0x7F, codes 0, row
 *     inv_rms NaN.  The tensor scale the library derives from a tensor is
 *     g = RN_fp32(a / 2688) with a the largest finite |x| (2688 = 448 * 6,
 *     so the tensor's largest block gets the largest E4M3 scale), and
 *     g = 1 when no finite element is nonzero.
 *   - Backward (straight-through estimator, [MXN] section 2, "Gradientes":
 *     RMSNorm's gradient logic reused, nothing saved but the normaliser):
 *     the cast is treated as the identity and RMSNorm's backward runs with
 *     the saved estimate rho~ in place of 1/RMS,
 *       dx = rho~ * dy - rho~^3 * x * (1/H) * sum_j dy_j x_j,
 *     evaluated in fp64 and rounded once to bf16.
 *
 * Arithmetic: fp64 throughout (every intermediate value of the cast is exact
 * in fp64; the power-mean sum carries a relative error below K * 2^-53).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define OR_FMT_MXFP8_E4M3 0
#define OR_FMT_MXFP4_E2M1 1
#define OR_FMT_MXFP4_E2M1_H16 2
#define OR_FMT_MXFP8_E4M3_H16 3
#define OR_FMT_MXFP4_E2M1_H32 4
#define OR_FMT_MXFP8_E4M3_H32 5

#define OR_BLOCK 32            /* MX block size B, [ABS]: "32x decrease" */
#define OR_SCALE_NAN 0xFF      /* E8M0 NaN code, [OCP] section 5.4 */

/* ---------------------------------------------------------------- values */

/* A bf16 is the upper 16 bits of an IEEE binary32; the value is exact in
 * both float and double. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Magnitude of a non-negative bf16 pattern, with the pattern above bf16 max
 * (0x7F80) read as 2^128: the value round-to-nearest compares against
 * before it overflows to Inf (IEEE 754-2019, 4.3.1 and 7.4). */
static double bf16_magnitude_unbounded(uint16_t b)
{
    return (b & 0x7FFFu) == 0x7F80u ? ldexp(1.0, 128) : fabs((double)bf16_bits_to_float(b));
}

/* Round a float to the nearest bf16, ties to an even last bit, by comparing
 * the two bf16 neighbours of f exactly (in double); beyond bf16 max + half
 * an ulp it overflows to Inf. */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x40);   /* quiet NaN */
    uint16_t lo = (uint16_t)(u >> 16);                   /* truncation: |lo| <= |f| */
    if ((u & 0xFFFFu) == 0) return lo;
    uint16_t hi = (uint16_t)(lo + 1);                     /* next magnitude up */
    double dlo = fabs((double)bf16_bits_to_float(lo));
    double dhi = bf16_magnitude_unbounded(hi);
    double a = fabs((double)f);
    double dist_lo = a - dlo, dist_hi = dhi - a;
    if (dist_lo < dist_hi) return lo;
    if (dist_hi < dist_lo) return hi;
    return (lo & 1u) ? hi : lo;
}

/* Round a double to the nearest bf16 (ties to an even last bit), IEEE 754
 * style: a magnitude from bf16 max + half an ulp (2^128 - 2^119, a tie that
 * goes to the even neighbour 2^128) upwards overflows to Inf.  The two bf16
 * neighbours are found from the float nearest below in magnitude and
 * compared exactly. */
static uint16_t double_to_bf16_rne(double d)
{
    if (isnan(d)) return 0x7FC0;
    if (isinf(d)) return (uint16_t)(signbit(d) ? 0xFF80u : 0x7F80u);
    double a = fabs(d);
    /* largest bf16 magnitude <= a: truncate the float of a toward zero */
    float f = (float)a;
    if ((double)f > a) f = nextafterf(f, 0.0f);
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t lo = (uint16_t)(u >> 16);
    if ((double)bf16_bits_to_float(lo) > a) lo = (uint16_t)(lo - 1);
    uint16_t hi = (uint16_t)(lo + 1);
    double dlo = a - (double)bf16_bits_to_float(lo);
    double dhi = bf16_magnitude_unbounded(hi) - a;
    uint16_t m = (dlo < dhi) ? lo : (dhi < dlo) ? hi : ((lo & 1u) ? hi : lo);
    if (dlo == 0.0) m = lo;
    return (uint16_t)(m | (signbit(d) ? 0x8000u : 0u));
}

/* ------------------------------------------------------- element grids */

/* FP8 E4M3 magnitude of code c in [0, 126]: bias 7, 3 mantissa bits,
 * E = 0 subnormal; code 127 (S.1111.111) is NaN and has no value. [OCP] 5.3 */
static double e4m3_value(int c)
{
    int E = c >> 3, M = c & 7;
    if (E == 0) return ldexp((double)M / 8.0, -6);
    return ldexp(1.0 + (double)M / 8.0, E - 7);
}

/* FP4 E2M1 magnitude of code c in [0, 7]: bias 1, 1 mantissa bit,
 * E = 0 subnormal.  Values 0, 0.5, 1, 1.5, 2, 3, 4, 6.  [OCP] 5.3 */
static double e2m1_value(int c)
{
    int E = c >> 1, M = c & 1;
    if (E == 0) return (double)M * 0.5;
    return ldexp(1.0 + (double)M / 2.0, E - 1);
}

/* Index of the grid value nearest to mag >= 0 among grid[0..n-1] (ascending),
 * ties to the even index (= even last mantissa bit, since the magnitude code
 * IS the index), anything at or above grid[n-1] saturating to n-1.  The
 * grid is scanned in full; the midpoint of two grid values is exact in
 * double, so the comparison is exact. */
static int nearest_grid_index(double mag, const double *grid, int n)
{
    if (mag >= grid[n - 1]) return n - 1;
    int lo = 0;
    for (int i = 0; i < n; ++i)
        if (grid[i] <= mag) lo = i;
    if (grid[lo] == mag) return lo;
    int hi = lo + 1;
    double mid = 0.5 * (grid[lo] + grid[hi]);
    if (mag < mid) return lo;
    if (mag > mid) return hi;
    return (lo % 2 == 0) ? lo : hi;
}

static double g_e4m3_grid[127];
static double g_e2m1_grid[8];
static int g_grids_ready = 0;

static void init_grids(void)
{
    if (g_grids_ready) return;
    for (int c = 0; c < 127; ++c) g_e4m3_grid[c] = e4m3_value(c);
    for (int c = 0; c < 8; ++c) g_e2m1_grid[c] = e2m1_value(c);
    g_grids_ready = 1;
}

/* Saturating round-to-nearest-even FP8 E4M3 code of a finite real r. */
uint8_t oracle_cast_e4m3(double r)
{
    init_grids();
    int mag = nearest_grid_index(fabs(r), g_e4m3_grid, 127);
    return (uint8_t)((signbit(r) ? 0x80 : 0x00) | mag);
}

/* Saturating round-to-nearest-even FP4 E2M1 nibble of a finite real r. */
uint8_t oracle_cast_e2m1(double r)
{
    init_grids();
    int mag = nearest_grid_index(fabs(r), g_e2m1_grid, 8);
    return (uint8_t)((signbit(r) ? 0x8 : 0x0) | mag);
}

/* Value of an E4M3 code (NaN for 0x7F / 0xFF). */
double oracle_decode_e4m3(uint8_t code)
{
    int mag = code & 0x7F;
    if (mag == 0x7F) return NAN;
    double v = e4m3_value(mag);
    return (code & 0x80) ? -v : v;
}

/* Value of an E2M1 nibble. */
double oracle_decode_e2m1(uint8_t nibble)
{
    double v = e2m1_value(nibble & 0x7);
    return (nibble & 0x8) ? -v : v;
}

/* ----------------------------------------------------------- E8M0 scale */

/* Shared exponent of a block with absmax amax >= 0: floor(log2 amax) minus
 * the element format's largest exponent, clamped to E8M0's [-127, 127];
 * amax = 0 gives -127.  [OCP] 6.3.  floor(log2) comes from frexp, which is
 * exact for every double including subnormal inputs. */
int oracle_e8m0_exponent(double amax, int emax_elem)
{
    if (amax == 0.0) return -127;
    int ex;
    (void)frexp(amax, &ex);            /* amax = f * 2^ex, f in [0.5, 1) */
    int e = (ex - 1) - emax_elem;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* ------------------------------------------------------------------ H16 */

/* Unnormalised Sylvester-Hadamard butterfly on n = 16 or 32 fp32 values in
 * place: stages h = 1, 2, 4, ... n/2, each pair (v_i, v_{i+h}) with
 * (i & h) == 0 replaced by (v_i + v_{i+h}, v_i - v_{i+h}) rounded to fp32.
 * The result is H_n v with H_n[i][j] = (-1)^popcount(i & j). */
static void hadamard_butterfly(float *v, int n)
{
    for (int h = 1; h < n; h <<= 1) {
        for (int i = 0; i < n; ++i) {
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                float s = a + b;
                float d = a - b;
                v[i] = s;
                v[i + h] = d;
            }
        }
    }
}

/* y = (1/4) * H16 * v for one group of 16 fp32 values, H16 the Sylvester
 * Hadamard matrix in natural order, H16[i][j] = (-1)^popcount(i & j).
 * Butterfly stages h = 1, 2, 4, 8; each add/sub rounded to fp32, then the
 * 1/4 scale in fp32.  [MXFP4] Metodologia, item 3. */
void oracle_h16_group(const float *in, float *out)
{
    float v[16];
    for (int i = 0; i < 16; ++i) v[i] = in[i];
    hadamard_butterfly(v, 16);
    for (int i = 0; i < 16; ++i) {
        float q = v[i] * 0.25f;
        out[i] = q;
    }
}

/* y = H32 * v / sqrt(32) for one group of 32 fp32 values: butterfly stages
 * h = 1 .. 16 in fp32, then each value times RN_fp32(1/sqrt(32)) in fp32.
 * [MXFP4] Metodologia, item 3 (H32). */
void oracle_h32_group(const float *in, float *out)
{
    const float c32 = (float)(1.0 / sqrt(32.0));
    float v[32];
    for (int i = 0; i < 32; ++i) v[i] = in[i];
    hadamard_butterfly(v, 32);
    for (int i = 0; i < 32; ++i) {
        float q = v[i] * c32;
        out[i] = q;
    }
}

/* -------------------------------------------------------------- helpers */

static int is_fp8(int fmt)
{
    return fmt == OR_FMT_MXFP8_E4M3 || fmt == OR_FMT_MXFP8_E4M3_H16 || fmt == OR_FMT_MXFP8_E4M3_H32;
}

/* rotation size applied before the cast: 0 (none), 16 or 32 */
static int rotation_of(int fmt)
{
    if (fmt == OR_FMT_MXFP4_E2M1_H16 || fmt == OR_FMT_MXFP8_E4M3_H16) return 16;
    if (fmt == OR_FMT_MXFP4_E2M1_H32 || fmt == OR_FMT_MXFP8_E4M3_H32) return 32;
    return 0;
}

static int emax_of(int fmt) { return is_fp8(fmt) ? 8 : 2; }

static int check_args(int64_t T, int64_t H, int fmt)
{
    if (T < 0 || H <= 0 || H % OR_BLOCK != 0) return 1;
    if (fmt < OR_FMT_MXFP8_E4M3 || fmt > OR_FMT_MXFP8_E4M3_H32) return 1;
    return 0;
}

/* Element values of block k of a row, as exact doubles (after H16 when the
 * format asks for it). */
static void block_values(const uint16_t *row, int64_t k, int fmt, double *v)
{
    const uint16_t *b = row + k * OR_BLOCK;
    const int rot = rotation_of(fmt);
    if (rot == 16) {
        for (int g = 0; g < OR_BLOCK; g += 16) {
            float in[16], out[16];
            for (int i = 0; i < 16; ++i) in[i] = bf16_bits_to_float(b[g + i]);
            oracle_h16_group(in, out);
            for (int i = 0; i < 16; ++i) v[g + i] = (double)out[i];
        }
    } else if (rot == 32) {
        float in[32], out[32];
        for (int i = 0; i < 32; ++i) in[i] = bf16_bits_to_float(b[i]);
        oracle_h32_group(in, out);
        for (int i = 0; i < 32; ++i) v[i] = (double)out[i];
    } else {
        for (int j = 0; j < OR_BLOCK; ++j) v[j] = (double)bf16_bits_to_float(b[j]);
    }
}

/* MX cast of one block: writes the scale code and the element codes;
 * returns the shared exponent e (or 128 for a non-finite block). */
static int cast_block(const double *v, int fmt, uint8_t *scale_out,
                      uint8_t *codes_row, int64_t k)
{
    int finite = 1;
    double amax = 0.0;
    for (int j = 0; j < OR_BLOCK; ++j) {
        if (!isfinite(v[j])) finite = 0;
        else if (fabs(v[j]) > amax) amax = fabs(v[j]);
    }
    if (!finite) {
        *scale_out = OR_SCALE_NAN;
        if (is_fp8(fmt))
            for (int j = 0; j < OR_BLOCK; ++j) codes_row[k * OR_BLOCK + j] = 0x7F;
        else
            for (int j = 0; j < OR_BLOCK / 2; ++j) codes_row[k * (OR_BLOCK / 2) + j] = 0x00;
        return 128;
    }
    int e = oracle_e8m0_exponent(amax, emax_of(fmt));
    *scale_out = (uint8_t)(e + 127);
    if (is_fp8(fmt)) {
        for (int j = 0; j < OR_BLOCK; ++j)
            codes_row[k * OR_BLOCK + j] = oracle_cast_e4m3(ldexp(v[j], -e));
    } else {
        for (int j = 0; j < OR_BLOCK; j += 2) {
            uint8_t lo = oracle_cast_e2m1(ldexp(v[j], -e));
            uint8_t hi = oracle_cast_e2m1(ldexp(v[j + 1], -e));
            codes_row[k * (OR_BLOCK / 2) + j / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
    return e;
}

/* ------------------------------------------------------------- MX cast */

/* MX cast only (no estimator) of T rows of H bf16 values.
 * codes: [T, H] (E4M3) or [T, H/2] (E2M1); scales: [T, H/32]. */
int oracle_mx_cast_rows(const uint16_t *x, int64_t T, int64_t H, int fmt,
                        uint8_t *codes, uint8_t *scales)
{
    if (check_args(T, H, fmt)) return 1;
    const int64_t K = H / OR_BLOCK;
    const int64_t code_bytes = is_fp8(fmt) ? H : H / 2;
    double v[OR_BLOCK];
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *row = x + t * H;
        for (int64_t k = 0; k < K; ++k) {
            block_values(row, k, fmt, v);
            (void)cast_block(v, fmt, scales + t * K + k, codes + t * code_bytes, k);
        }
    }
    return 0;
}

/* MX cast (MXFP8 E4M3) of the gain-folded weight of MXNormLinear ("MXNorm
 * ...", Resumen tecnico, 2. Metodologia, "Implementacion": the norm's gain
 * gamma, and with it the constant c, is folded into the next linear layer's
 * weight).  Row n of W' holds w[n, j] * g_j with g_j = RN_fp32(c * gamma_j):
 * each product is one fp32 multiplication (round to nearest even; this file
 * is compiled without contraction), then the MX cast of those fp32 values
 * as in oracle_mx_cast_rows.  w: bf16 bits [N, K]; gamma: fp32 [K]. */
int oracle_mx_cast_gain_rows(const uint16_t *w, int64_t N, int64_t K, const float *gamma, float c,
                             uint8_t *codes, uint8_t *scales)
{
    if (check_args(N, K, OR_FMT_MXFP8_E4M3)) return 1;
    const int64_t KB = K / OR_BLOCK;
    double v[OR_BLOCK];
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            for (int j = 0; j < OR_BLOCK; ++j) {
                const int64_t idx = kb * OR_BLOCK + j;
                const float g = c * gamma[idx];
                const float y = bf16_bits_to_float(w[n * K + idx]) * g;
                v[j] = (double)y;
            }
            (void)cast_block(v, OR_FMT_MXFP8_E4M3, scales + n * KB + kb, codes + n * K, kb);
        }
    }
    return 0;
}

/* --------------------------------------------------------------- MXNorm */

/* MXNorm forward of T rows: the MX cast of each row plus
 *   inv_rms = c(p,B) * ((1/K) sum_k s_k^p)^(-1/p),   c(p,B) = 1,
 * with s_k = 2^e_k the block scales ([MXN] Fundamentos Teoricos, formula;
 * [ABS]).  The sum runs over k in index order in fp64 (s_k^p lies in
 * [2^-254, 2^254], inside fp64's range); 1/mean or 1/sqrt(mean) is taken in
 * fp64 and rounded once to fp32. */
int oracle_mxnorm_rows(const uint16_t *x, int64_t T, int64_t H, int p, int fmt,
                       uint8_t *codes, uint8_t *scales, float *inv_rms)
{
    if (check_args(T, H, fmt)) return 1;
    if (p != 1 && p != 2) return 1;
    const int64_t K = H / OR_BLOCK;
    const int64_t code_bytes = is_fp8(fmt) ? H : H / 2;
    double v[OR_BLOCK];
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *row = x + t * H;
        double sum = 0.0;
        int row_finite = 1;
        for (int64_t k = 0; k < K; ++k) {
            block_values(row, k, fmt, v);
            int e = cast_block(v, fmt, scales + t * K + k, codes + t * code_bytes, k);
            if (e == 128) { row_finite = 0; continue; }
            sum += ldexp(1.0, p * e);                       /* s_k^p */
        }
        if (!row_finite) { inv_rms[t] = NAN; continue; }
        double mean = sum / (double)K;
        double m_p = (p == 1) ? mean : sqrt(mean);        /* power mean M_p */
        inv_rms[t] = (float)(1.0 / m_p);
    }
    return 0;
}

/* ------------------------------------------------- RMSNorm + MXFP8 cast */

/* The two-pass baseline: exact-definition RMSNorm, then the MXFP8 cast of
 * its bf16 output.  RMS = sqrt((1/D) sum x^2) ([MXN] Fundamentos Teoricos,
 * the RMSNorm formula the estimator replaces); eps is added under the root.
 * x^2 is exact in fp64 and the sum runs in index order.  y: [T, H] bf16. */
int oracle_rmsnorm_mxfp8_rows(const uint16_t *x, int64_t T, int64_t H, float eps,
                              uint16_t *y, uint8_t *codes, uint8_t *scales,
                              float *inv_rms)
{
    if (check_args(T, H, OR_FMT_MXFP8_E4M3)) return 1;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *row = x + t * H;
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            double xj = (double)bf16_bits_to_float(row[j]);
            ss += xj * xj;
        }
        float inv = (float)(1.0 / sqrt(ss / (double)H + (double)eps));
        inv_rms[t] = inv;
        for (int64_t j = 0; j < H; ++j) {
            /* x (8 significant bits) * inv (24 bits) is exact in fp64, so the
             * cast to float is the single fp32 rounding of the product. */
            float prod = (float)((double)bf16_bits_to_float(row[j]) * (double)inv);
            y[t * H + j] = float_to_bf16_rne(prod);
        }
    }
    return oracle_mx_cast_rows(y, T, H, OR_FMT_MXFP8_E4M3, codes, scales);
}

/* --------------------------------------------------------------- NVFP4 */

/* Value of a non-negative E4M3 code (its magnitude bits). */
static double e4m3_code_value(uint8_t c)
{
    return e4m3_value(c & 0x7F);
}

/* NVFP4 tensor scale of n bf16 values (see the header comment): the
 * largest finite magnitude a, then a / 2688 rounded once to fp32.  The
 * quotient is formed in double and rounded to float: for one division of
 * two floats that equals the correctly rounded float quotient (double
 * carries more than 2 * 24 + 2 bits). */
float oracle_nvfp4_tensor_scale(const uint16_t *x, int64_t n)
{
    double a = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double v = fabs((double)bf16_bits_to_float(x[i]));
        if (isfinite(v) && v > a) a = v;
    }
    return a > 0.0 ? (float)(a / 2688.0) : 1.0f;
}

/* NVFP4 forward of T rows (see the header comment): codes [T, H/2] (element
 * 2i in the low nibble), scales [T, H/16] (UE4M3 codes), inv_rms [T]. */
int oracle_nvfp4_rows(const uint16_t *x, int64_t T, int64_t H, int p, float g,
                      uint8_t *codes, uint8_t *scales, float *inv_rms)
{
    if (T < 0 || H <= 0 || H % 16 != 0 || (p != 1 && p != 2) || !(g > 0.0f) || !isfinite(g)) return 1;
    const int64_t K = H / 16;
    const float sixg = 6.0f * g;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *row = x + t * H;
        double sum = 0.0;
        int row_finite = 1;
        for (int64_t k = 0; k < K; ++k) {
            double amax = 0.0;
            int finite = 1;
            for (int j = 0; j < 16; ++j) {
                double v = (double)bf16_bits_to_float(row[k * 16 + j]);
                if (!isfinite(v)) finite = 0;
                else if (fabs(v) > amax) amax = fabs(v);
            }
            uint8_t *crow = codes + t * (H / 2) + k * 8;
            if (!finite) {
                scales[t * K + k] = 0x7F;
                for (int j = 0; j < 8; ++j) crow[j] = 0;
                row_finite = 0;
                continue;
            }
            const float sb = (float)amax / sixg;
            const uint8_t sc = oracle_cast_e4m3((double)sb);
            scales[t * K + k] = sc;
            const float sval = (float)e4m3_code_value(sc);
            const float d = sval * g;
            const float enc = (sval == 0.0f) ? 0.0f : 1.0f / d;
            for (int j = 0; j < 16; j += 2) {
                const float r0 = bf16_bits_to_float(row[k * 16 + j]) * enc;
                const float r1 = bf16_bits_to_float(row[k * 16 + j + 1]) * enc;
                crow[j / 2] = (uint8_t)(oracle_cast_e2m1((double)r0) | (oracle_cast_e2m1((double)r1) << 4));
            }
            const double m = (double)sval * (double)g;      /* m~_k = s_k g */
            sum += (p == 1) ? m : m * m;
        }
        if (!row_finite) { inv_rms[t] = NAN; continue; }
        if (sum == 0.0) { inv_rms[t] = INFINITY; continue; }
        const double mean = sum / (double)K;
        const double m_p = (p == 1) ? mean : sqrt(mean);
        inv_rms[t] = (float)(1.0 / m_p);
    }
    return 0;
}

/* ------------------------------------------------------- MXNormLinear */

/* Consumer side of MXNormLinear ([MXN] section 2, Implementacion: the gain
 * is folded into the next layer's weight, the row scale commutes with the
 * matmul): out[t][n] = inv_rms[t] * sum_k xv[t][k] * wv[n][k], where xv / wv
 * are E4M3 code values times their E8M0 block scales (32 elements along K,
 * row-major scale arrays [rows][K/32]).  fp64, every product exact. */
int oracle_mxfp8_linear(const uint8_t *xc, const uint8_t *xs, const float *inv_rms, const uint8_t *wc,
                        const uint8_t *ws, int64_t T, int64_t K, int64_t N, double *out)
{
    if (T < 0 || K <= 0 || K % OR_BLOCK != 0 || N <= 0) return 1;
    const int64_t KB = K / OR_BLOCK;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double xv = ldexp(oracle_decode_e4m3(xc[t * K + k]), (int)xs[t * KB + k / OR_BLOCK] - 127);
                const double wv = ldexp(oracle_decode_e4m3(wc[n * K + k]), (int)ws[n * KB + k / OR_BLOCK] - 127);
                acc += xv * wv;
            }
            out[t * N + n] = (double)inv_rms[t] * acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------ backward */

/* Straight-through backward of T rows: x, dy bf16 [T, H], inv_rms [T] (the
 * forward's rho~), dx bf16 [T, H] (and, if dx64 is not NULL, the unrounded
 * fp64 values).  fp64 throughout, one bf16 rounding. */
int oracle_mxnorm_bwd_ste_rows(const uint16_t *x, const uint16_t *dy, const float *inv_rms,
                               int64_t T, int64_t H, uint16_t *dx, double *dx64)
{
    if (T < 0 || H <= 0) return 1;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t *xr = x + t * H, *gr = dy + t * H;
        double dot = 0.0;
        for (int64_t j = 0; j < H; ++j)
            dot += (double)bf16_bits_to_float(gr[j]) * (double)bf16_bits_to_float(xr[j]);
        const double r = (double)inv_rms[t];
        const double k = r * r * r * dot / (double)H;
        for (int64_t j = 0; j < H; ++j) {
            const double g = r * (double)bf16_bits_to_float(gr[j]) - k * (double)bf16_bits_to_float(xr[j]);
            dx[t * H + j] = double_to_bf16_rne(g);
            if (dx64) dx64[t * H + j] = g;
        }
    }
    return 0;
}

/* ------------------------------------------------- array entry points */

void oracle_cast_e4m3_array(const double *r, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_cast_e4m3(r[i]);
}

void oracle_cast_e2m1_array(const double *r, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_cast_e2m1(r[i]);
}

void oracle_e8m0_exponent_array(const double *amax, int64_t n, int emax_elem, int32_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e8m0_exponent(amax[i], emax_elem);
}

void oracle_h16_groups(const float *in, int64_t n_groups, float *out)
{
    for (int64_t g = 0; g < n_groups; ++g) oracle_h16_group(in + 16 * g, out + 16 * g);
}

void oracle_h32_groups(const float *in, int64_t n_groups, float *out)
{
    for (int64_t g = 0; g < n_groups; ++g) oracle_h32_group(in + 32 * g, out + 32 * g);
}

void oracle_float_to_bf16_array(const float *in, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = float_to_bf16_rne(in[i]);
}
