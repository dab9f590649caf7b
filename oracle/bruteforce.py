"""Exact-rational brute force of MXNorm for tiny inputs -- TEST INFRASTRUCTURE ONLY.

A second implementation, independent of ``mxnorm_oracle.c``: every value is
a ``fractions.Fraction`` decoded from its bit fields, every element code is
chosen by scanning all finite codes of the format for the nearest value, and
the final fp32 rounding of inv_rms is decided exactly (squares compared with
rationals), not through floating point.  Slow: meant for rows of a few
hundred elements.  It shares no code with the C oracle or the CUDA library.

Sources: "MXNorm: Reusing MXFP block scales for efficient tensor
normalisation", Resumen tecnico, 2. Metodologia, "Fundamentos Teoricos"
(estimator formula); the MXFP4 page's Metodologia item 3 (H16); OCP
Microscaling Formats v1.0 sections 5 (encodings) and 6.3 (shared exponent).
Readings as in the C oracle: m~_k = s_k, c(p,B) = 1, sign kept on zero codes,
saturation to the largest finite value, ties to an even mantissa.
"""
from __future__ import annotations

from fractions import Fraction
from math import floor, isqrt

BLOCK = 32


# ---------------------------------------------------------------- decoding
def bf16_value(bits: int) -> Fraction | None:
    """Exact value of a bf16 bit pattern (1 sign, 8 exponent, 7 mantissa
    bits, bias 127); None for Inf/NaN."""
    s, e, m = bits >> 15, (bits >> 7) & 0xFF, bits & 0x7F
    if e == 0xFF:
        return None
    v = Fraction(m, 128) * Fraction(2) ** -126 if e == 0 else (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)
    return -v if s else v


def fp32_value(bits: int) -> Fraction | None:
    s, e, m = bits >> 31, (bits >> 23) & 0xFF, bits & 0x7FFFFF
    if e == 0xFF:
        return None
    v = Fraction(m, 1 << 23) * Fraction(2) ** -126 if e == 0 else (1 + Fraction(m, 1 << 23)) * Fraction(2) ** (e - 127)
    return -v if s else v


def e4m3_values():
    """{code: value} for every finite E4M3 code (bias 7, 3 mantissa bits)."""
    out = {}
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 0xF, c & 7
        if e == 0xF and m == 7:
            continue  # NaN
        v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        out[c] = -v if s else v
    return out


def e2m1_values():
    """{nibble: value} for every E2M1 code (bias 1, 1 mantissa bit)."""
    out = {}
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        v = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
        out[c] = -v if s else v
    return out


_E4M3 = e4m3_values()
_E2M1 = e2m1_values()


# ------------------------------------------------------------ fp32 rounding
def round_to_fp32(q: Fraction) -> Fraction:
    """Nearest binary32 value to q (ties to an even significand); finite q
    within range only."""
    if q == 0:
        return Fraction(0)
    a = abs(q)
    e = floor_log2(a)
    e = max(e, -126)                       # subnormal spacing below 2^-126
    ulp = Fraction(2) ** (e - 23)
    n = a / ulp
    k = floor(n)
    rem = n - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    r = k * ulp
    return -r if q < 0 else r


def floor_log2(a: Fraction) -> int:
    """floor(log2 a) for a > 0, exactly."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


# -------------------------------------------------------------------- H16
def h16_fp32(group):
    """(1/4) H16 v with fp32 rounding after every butterfly add/sub and after
    the 1/4 scale; stages h = 1, 2, 4, 8.  group: 16 Fractions (fp32 values)."""
    v = list(group)
    h = 1
    while h < 16:
        for i in range(16):
            if i & h == 0:
                a, b = v[i], v[i + h]
                v[i], v[i + h] = round_to_fp32(a + b), round_to_fp32(a - b)
        h *= 2
    return [round_to_fp32(x / 4) for x in v]


def h32_fp32(group):
    """H32 v / sqrt(32): fp32 butterfly stages h = 1 .. 16, then each value
    times RN_fp32(1/sqrt(32)) rounded to fp32.  group: 32 Fractions."""
    v = list(group)
    h = 1
    while h < 32:
        for i in range(32):
            if i & h == 0:
                a, b = v[i], v[i + h]
                v[i], v[i + h] = round_to_fp32(a + b), round_to_fp32(a - b)
        h *= 2
    c32 = _round_inv_power_mean(Fraction(32), 2)      # RN_fp32(32^(-1/2)), decided exactly
    return [round_to_fp32(x * c32) for x in v]


def _is_fp8(fmt: str) -> bool:
    return fmt.startswith("mxfp8")


def _rotation(fmt: str) -> int:
    return 16 if fmt.endswith("_h16") else 32 if fmt.endswith("_h32") else 0


# ------------------------------------------------------------------- cast
def nearest_code(r: Fraction, table: dict, sign_bit: int) -> int:
    """Code whose value is nearest to r among all finite codes of the format
    that carry r's sign bit; ties to an even mantissa (code LSB 0)."""
    sign_mask = 0x80 if len(table) > 16 else 0x8
    best = None
    for c, v in table.items():
        if bool(c & sign_mask) != bool(sign_bit):
            continue
        d = abs(r - v)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0 and (best[1] & 1) == 1):
            best = (d, c)
    return best[1]


def mx_block(values, signs, fmt: str):
    """Scale exponent and codes of one 32-element block of exact values
    (with their sign bits, which decide the sign of zero codes)."""
    emax = 8 if _is_fp8(fmt) else 2
    amax = max(abs(v) for v in values)
    e = -127 if amax == 0 else max(-127, min(127, floor_log2(amax) - emax))
    s = Fraction(2) ** e
    table = _E4M3 if _is_fp8(fmt) else _E2M1
    return e, [nearest_code(v / s, table, sb) for v, sb in zip(values, signs)]


def mx_cast_gain_row(bits_row, gamma_bits, c_bits):
    """Gain-folded MXFP8 cast of one bf16 weight row: v_j =
    RN_fp32(x_j * RN_fp32(c * gamma_j)) in exact arithmetic, then the MX
    cast; gamma_bits and c_bits are fp32 bit patterns of finite values.
    Returns (code bytes, scale codes)."""
    c = fp32_value(c_bits)
    codes, scales = [], []
    for k in range(0, len(bits_row), BLOCK):
        vals, signs = [], []
        for x_b, g_b in zip(bits_row[k:k + BLOCK], gamma_bits[k:k + BLOCK]):
            g = round_to_fp32(c * fp32_value(g_b))
            x = bf16_value(x_b)
            v = round_to_fp32(x * g)
            # IEEE sign of a product, zero included: the xor of the signs
            g_neg = (g < 0) or (g == 0 and ((c_bits >> 31) ^ (g_b >> 31)))
            vals.append(v)
            signs.append(int((x_b >> 15) & 1) ^ int(bool(g_neg)))
        e, cs = mx_block(vals, signs, "mxfp8")
        scales.append(e + 127)
        codes.extend(cs)
    return codes, scales


def mxnorm_row(bits_row, p: int, fmt: str):
    """MXNorm of one finite bf16 row (list of ints): (code bytes, scale
    codes, inv_rms as an exact fp32 value).

    For the rotated formats (*_h16, *_h32) a rotated value that is exactly
    zero raises ValueError: the sign IEEE arithmetic gives such a zero is not
    modelled here, so callers use inputs whose rotations have no exact zeros."""
    H = len(bits_row)
    assert H % BLOCK == 0
    K = H // BLOCK
    vals, signs = [], []
    rot_n = _rotation(fmt)
    if rot_n:
        rotate = h16_fp32 if rot_n == 16 else h32_fp32
        for g in range(0, H, rot_n):
            rot = rotate([bf16_value(b) for b in bits_row[g:g + rot_n]])
            if any(v == 0 for v in rot):
                raise ValueError("rotated value is exactly zero")
            vals.extend(rot)
            signs.extend(1 if v < 0 else 0 for v in rot)
    else:
        vals = [bf16_value(b) for b in bits_row]
        signs = [b >> 15 for b in bits_row]
    codes, scales, s_pow_sum = [], [], Fraction(0)
    for k in range(K):
        sl = slice(k * BLOCK, (k + 1) * BLOCK)
        e, c = mx_block(vals[sl], signs[sl], fmt)
        scales.append(e + 127)
        s_pow_sum += Fraction(2) ** (p * e)          # s_k^p
        if _is_fp8(fmt):
            codes.extend(c)
        else:
            codes.extend(c[j] | (c[j + 1] << 4) for j in range(0, BLOCK, 2))
    inv = _round_inv_power_mean(s_pow_sum / K, p)
    return codes, scales, inv


def _round_inv_power_mean(mean: Fraction, p: int) -> Fraction:
    """RN_fp32(mean^(-1/p)) decided exactly."""
    if p == 1:
        return round_to_fp32(1 / mean)
    # p = 2: y = 1/sqrt(mean).  Start from an integer square root estimate,
    # then pick the fp32 value f whose rounding interval holds y, comparing
    # squares exactly: y in (lo, hi) <=> lo^2 < 1/mean < hi^2.
    target = 1 / mean
    scale = 1 << 200
    approx = Fraction(isqrt(int(target * scale * scale)), scale)
    f = round_to_fp32(approx)
    for _ in range(4):
        e = max(floor_log2(f), -126)
        ulp = Fraction(2) ** (e - 23)
        lo_mid = f - ulp / 2 if f != Fraction(2) ** e or e == -126 else f - ulp / 4
        hi_mid = f + ulp / 2
        if lo_mid * lo_mid < target < hi_mid * hi_mid:
            return f
        if target == hi_mid * hi_mid or target == lo_mid * lo_mid:
            raise ArithmeticError("exact tie in sqrt rounding cannot happen for these inputs")
        f = round_to_fp32(f + ulp) if target >= hi_mid * hi_mid else round_to_fp32(f - ulp)
    raise ArithmeticError("fp32 rounding of 1/sqrt did not settle")


# ------------------------------------------------------------------ NVFP4
def nvfp4_row(bits_row, p: int, g_bits: int):
    """NVFP4 of one finite bf16 row with tensor scale g (fp32 bit pattern):
    (code bytes, UE4M3 scale codes, inv_rms as an exact fp32 value or None
    for +Inf).  Every fp32 operation is an exact rational rounded by
    round_to_fp32; the block-scale cast scans all E4M3 codes."""
    g = fp32_value(g_bits)
    H = len(bits_row)
    assert H % 16 == 0
    K = H // 16
    sixg = round_to_fp32(6 * g)
    codes, scales, ssum = [], [], Fraction(0)
    for k in range(K):
        vals = [bf16_value(b) for b in bits_row[16 * k:16 * k + 16]]
        signs = [b >> 15 for b in bits_row[16 * k:16 * k + 16]]
        amax = max(abs(v) for v in vals)
        sb = round_to_fp32(amax / sixg)
        sc = nearest_code(sb, _E4M3, 0)
        scales.append(sc)
        sval = _E4M3[sc]
        enc = Fraction(0) if sval == 0 else round_to_fp32(1 / round_to_fp32(sval * g))
        nib = [nearest_code(round_to_fp32(v * enc), _E2M1, sgn) for v, sgn in zip(vals, signs)]
        codes.extend(nib[j] | (nib[j + 1] << 4) for j in range(0, 16, 2))
        ssum += (sval * g) ** p
    if ssum == 0:
        return codes, scales, None
    return codes, scales, _round_inv_power_mean(ssum / K, p)
