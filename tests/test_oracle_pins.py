"""Pins of the CPU oracle against facts fixed outside it.

Every test here checks the oracle (oracle/) against something it does not
compute itself: the bit-field definitions of bf16/E4M3/E2M1/E8M0 (OCP
Microscaling Formats v1.0, sections 5 and 6.3), library conversions (torch's
float8_e4m3fn cast, ml_dtypes' float4_e2m1fn cast), scipy's Sylvester
Hadamard matrix, closed forms of the estimator of "MXNorm: Reusing MXFP
block scales for efficient tensor normalisation" (Resumen tecnico, 2.
Metodologia, Fundamentos Teoricos) on constant and two-level rows, the
growth bounds of its section 4 ("Analisis de Picos": O(K) for p = 1 against
RMSNorm's O(sqrt(D))), and an exact-rational brute force on tiny rows.
No GPU is used.
"""
from fractions import Fraction
import math
import os

import numpy as np
import pytest
import torch

from mx_scale_reusing_gb300 import synth

ALL_BF16 = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)


def bf16_values(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def finite_bf16_bits():
    b = ALL_BF16
    return b[((b >> 7) & 0xFF) != 0xFF]


# ----------------------------------------------------------------- E8M0
@pytest.mark.parametrize("emax", [8, 2])
def test_e8m0_exponent_exhaustive_vs_bit_fields(oracle_mod, emax):
    """All 32640 finite non-negative bf16 amax values: the oracle's
    floor(log2) via frexp must equal the exponent read off the bf16 bit
    fields (normal: E - 127; subnormal: bit_length(M) - 1 - 133)."""
    bits = finite_bf16_bits()
    bits = bits[bits < 0x8000]
    got = oracle_mod.e8m0_exponent(bf16_values(bits), emax)
    E = (bits.astype(np.int64) >> 7) & 0xFF
    M = bits.astype(np.int64) & 0x7F
    fl = np.where(E > 0, E - 127, np.array([int(m).bit_length() - 1 - 133 if m else 0 for m in M]))
    want = np.clip(fl - emax, -127, 127)
    want[bits == 0] = -127
    np.testing.assert_array_equal(got, want)


def test_e8m0_exponent_fp32_range(oracle_mod):
    a = np.array([2.0 ** -149, 2.0 ** -126, 1.0, 1.9999, 2.0, 448.0, 3.0e38])
    np.testing.assert_array_equal(oracle_mod.e8m0_exponent(a, 8), [-127, -127, -8, -8, -7, 0, 119])


# ------------------------------------------------------ spec fixtures
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "ocp_mx_v1_encodings.txt")


def golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].split()
        if line:
            rows.append(line)
    return rows


def spec_value(tok: str) -> float:
    if tok == "nan":
        return math.nan
    if tok == "-0":
        return -0.0
    return float.fromhex(tok) if "p" in tok else float(tok)


def test_golden_ocp_encodings(oracle_mod):
    """The oracle's E4M3 / E2M1 decodes, E8M0 scale values and shared
    exponent against the OCP MX v1.0 tables (tests/golden)."""
    rows = golden_rows()
    assert len(rows) >= 30
    for kind, a, b, *rest in rows:
        if kind in ("e4m3", "e2m1"):
            code, want = int(a, 16), spec_value(b)
            got = oracle_mod.decode_e4m3(code) if kind == "e4m3" else oracle_mod.decode_e2m1(code)
            if math.isnan(want):
                assert math.isnan(got), (kind, a)
            else:
                assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), (kind, a, got)
                if kind == "e4m3":  # and the cast maps the value back to its code
                    assert oracle_mod.cast_e4m3([want])[0] == code, (kind, a)
                else:
                    assert oracle_mod.cast_e2m1([want])[0] == code, (kind, a)
        elif kind == "e8m0":
            code, want = int(a, 16), spec_value(b)
            if math.isnan(want):
                assert code == 0xFF
            else:  # the scale a code stands for: 2^(code - 127)
                assert math.ldexp(1.0, code - 127) == want
                e = oracle_mod.e8m0_exponent([want * 256.0], 8)[0]  # amax = scale * 2^emax
                assert e + 127 == code or code == 0x00, (a, e)
        elif kind == "shared":
            emax, amax, want = int(a), spec_value(b), int(rest[0])
            assert oracle_mod.e8m0_exponent([amax], emax)[0] == want, (emax, b)
        else:
            raise AssertionError(f"unknown fixture kind {kind}")


# ----------------------------------------------------------------- E4M3
def test_e4m3_decode_table(oracle_mod):
    """Spot values of the E4M3 encoding (bias 7, 3 mantissa bits, no Inf)."""
    assert oracle_mod.decode_e4m3(0x7E) == 448.0
    assert oracle_mod.decode_e4m3(0x38) == 1.0
    assert oracle_mod.decode_e4m3(0x08) == 2.0 ** -6
    assert oracle_mod.decode_e4m3(0x01) == 2.0 ** -9
    assert oracle_mod.decode_e4m3(0x07) == 7 * 2.0 ** -9
    assert oracle_mod.decode_e4m3(0xC0) == -2.0
    assert math.isnan(oracle_mod.decode_e4m3(0x7F)) and math.isnan(oracle_mod.decode_e4m3(0xFF))
    mags = [oracle_mod.decode_e4m3(c) for c in range(127)]
    assert all(a < b for a, b in zip(mags, mags[1:]))


def test_e4m3_cast_exhaustive_bf16_vs_torch(oracle_mod):
    """Every finite bf16 value r (the values r = x / 2^e a bf16 x can give):
    where |r| <= 464 torch's float8_e4m3fn conversion (RNE, ties to even) is
    the same map; above 464 torch goes to NaN while the MX cast saturates
    to +-448 (0x7E)."""
    bits = finite_bf16_bits()
    r = bf16_values(bits)
    got = oracle_mod.cast_e4m3(r)
    lib = torch.from_numpy(r.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    small = np.abs(r) <= 464
    np.testing.assert_array_equal(got[small], lib[small])
    big = ~small
    np.testing.assert_array_equal(got[big], np.where(r[big] < 0, 0xFE, 0x7E))
    # sign kept on zeros and on negatives that round to zero
    assert oracle_mod.cast_e4m3([-0.0])[0] == 0x80
    assert oracle_mod.cast_e4m3([-(2.0 ** -11)])[0] == 0x80


def test_e4m3_cast_random_fp32_vs_torch(oracle_mod):
    rng = np.random.default_rng(11)
    r = (rng.standard_normal(200_000) * np.exp2(rng.integers(-14, 9, 200_000))).astype(np.float32)
    r = r[np.abs(r) <= 464].astype(np.float64)
    lib = torch.from_numpy(r.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle_mod.cast_e4m3(r), lib)


def test_e4m3_cast_ties_by_hand(oracle_mod):
    """Midpoints between neighbouring E4M3 values go to the even mantissa."""
    cases = {
        1.0625: 0x38,           # between 1.0 (M=0) and 1.125 (M=1) -> 1.0
        1.1875: 0x3A,           # between 1.125 (M=1) and 1.25 (M=2) -> 1.25
        2.0 ** -10: 0x00,       # half the smallest subnormal -> 0
        3 * 2.0 ** -10: 0x02,   # between 1 and 2 subnormal steps -> 2
        464.0: 0x7E,            # between 448 and 480 (not finite) -> 448
        15 * 2.0 ** -10: 0x08,  # between 7/8*2^-6 (0x07) and 2^-6 (0x08) -> 0x08
    }
    got = oracle_mod.cast_e4m3(list(cases))
    assert got.tolist() == list(cases.values())


# ----------------------------------------------------------------- E2M1
def test_e2m1_decode_table(oracle_mod):
    assert [oracle_mod.decode_e2m1(c) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert [oracle_mod.decode_e2m1(c) for c in range(8, 16)] == [-0.0, -0.5, -1, -1.5, -2, -3, -4, -6]


def test_e2m1_cast_exhaustive_vs_ml_dtypes(oracle_mod):
    """Every finite bf16 value and fp32 values one ulp around every tie point:
    ml_dtypes' float4_e2m1fn conversion is a saturating RNE cast that keeps
    the sign of zero, the same map."""
    ml_dtypes = pytest.importorskip("ml_dtypes")
    r = bf16_values(finite_bf16_bits())
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0], np.float32)
    near = np.concatenate([ties, np.nextafter(ties, np.float32(0)), np.nextafter(ties, np.float32(100))])
    r = np.concatenate([r, near, -near]).astype(np.float32)
    lib = r.astype(ml_dtypes.float4_e2m1fn).view(np.uint8) & 0xF
    np.testing.assert_array_equal(oracle_mod.cast_e2m1(r.astype(np.float64)), lib)


def test_e2m1_cast_by_hand(oracle_mod):
    cases = {0.25: 0x0, 0.2500001: 0x1, 0.75: 0x2, 1.25: 0x2, 1.75: 0x4, 2.5: 0x4,
             3.5: 0x6, 5.0: 0x6, 5.0001: 0x7, 100.0: 0x7, -0.1: 0x8, -6.5: 0xF}
    assert oracle_mod.cast_e2m1(list(cases)).tolist() == list(cases.values())


# ------------------------------------------------------------------ H16
def test_h16_matches_sylvester_matrix_on_small_integers(oracle_mod):
    """On small integers fp32 is exact, so the butterfly must equal the
    explicit product (1/4) * H16 @ v with scipy's Sylvester Hadamard."""
    from scipy.linalg import hadamard
    Hm = hadamard(16).astype(np.float64)
    rng = np.random.default_rng(3)
    v = rng.integers(-1000, 1000, size=(64, 16)).astype(np.float32)
    got = oracle_mod.h16(v).reshape(64, 16).astype(np.float64)
    np.testing.assert_array_equal(got, (v.astype(np.float64) @ Hm.T) / 4.0)


def test_h16_closed_forms(oracle_mod):
    e0 = np.zeros(16, np.float32)
    e0[0] = 1
    np.testing.assert_array_equal(oracle_mod.h16(e0), np.full(16, 0.25, np.float32))
    c = np.full(16, 3.0, np.float32)
    want = np.zeros(16, np.float32)
    want[0] = 12.0
    np.testing.assert_array_equal(oracle_mod.h16(c), want)
    # involution: ((1/4) H16)^2 = I, exact on small integers
    v = np.arange(-8, 8, dtype=np.float32) * 4
    np.testing.assert_array_equal(oracle_mod.h16(oracle_mod.h16(v)), v)


def test_h32_butterfly_matches_sylvester_matrix(oracle_mod):
    """On small integers the fp32 butterfly is exact, so the oracle's H32 /
    sqrt(32) equals the exact product with scipy's Sylvester hadamard(32)
    followed by one fp32 multiply with RN_fp32(1/sqrt(32))."""
    from scipy.linalg import hadamard
    Hm = hadamard(32).astype(np.float64)
    rng = np.random.default_rng(7)
    v = rng.integers(-500, 500, size=(64, 32)).astype(np.float32)
    exact = (v.astype(np.float64) @ Hm.T)                   # integers, exact in fp32
    c32 = np.float32(1.0 / np.sqrt(32.0))
    assert c32 == np.float32(0.17677669)
    want = (exact.astype(np.float32) * c32).astype(np.float32)
    np.testing.assert_array_equal(oracle_mod.h32(v).reshape(64, 32), want)


def test_h32_closed_forms(oracle_mod):
    e0 = np.zeros(32, np.float32)
    e0[0] = 1
    np.testing.assert_array_equal(oracle_mod.h32(e0), np.full(32, np.float32(1 / np.sqrt(32)), np.float32))
    c = np.full(32, 2.0, np.float32)
    out = oracle_mod.h32(c)
    assert out[0] == np.float32(np.float32(64.0) * np.float32(1 / np.sqrt(32))) and (out[1:] == 0).all()
    rng = np.random.default_rng(8)
    v = rng.standard_normal((500, 32)).astype(np.float32)
    y = oracle_mod.h32(v).reshape(500, 32).astype(np.float64)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(v.astype(np.float64), axis=1), rtol=2e-6)
    # (H32/sqrt 32)^2 = I up to the fp32 roundings of the two passes
    np.testing.assert_allclose(oracle_mod.h32(oracle_mod.h32(v)).reshape(500, 32), v, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("fmt,rot", [("mxfp8_h16", 16), ("mxfp4_h32", 32), ("mxfp8_h32", 32)])
def test_rotated_formats_cast_the_rotated_values(oracle_mod, fmt, rot):
    """A rotated format equals the plain MX cast applied to the rotation's
    output (the rotation runs first, per aligned group), checked through the
    independent per-element casts."""
    x = synth.make_random_rows(4, 256, seed=9, scale=2.0)
    codes, scales, inv = oracle_mod.mxnorm_quant(x, 2, fmt)
    v = synth.bf16_bits_to_f32(x)
    y = (oracle_mod.h16 if rot == 16 else oracle_mod.h32)(v).reshape(v.shape).astype(np.float64)
    amax = np.abs(y).reshape(4, 8, 32).max(-1)
    emax = 8 if fmt.startswith("mxfp8") else 2
    e = oracle_mod.e8m0_exponent(amax, emax)
    np.testing.assert_array_equal(scales, e + 127)
    r = y / np.repeat(np.exp2(e.astype(np.float64)), 32, axis=1)
    if fmt.startswith("mxfp8"):
        np.testing.assert_array_equal(codes, oracle_mod.cast_e4m3(r))
    else:
        nib = oracle_mod.cast_e2m1(r)
        np.testing.assert_array_equal(codes, nib[:, 0::2] | (nib[:, 1::2] << 4))


def test_h16_preserves_norm(oracle_mod):
    rng = np.random.default_rng(4)
    v = rng.standard_normal((1000, 16)).astype(np.float32)
    y = oracle_mod.h16(v).reshape(1000, 16)
    np.testing.assert_allclose(np.linalg.norm(y.astype(np.float64), axis=1),
                               np.linalg.norm(v.astype(np.float64), axis=1), rtol=1e-6)


# --------------------------------------------------- estimator closed forms
def const_row(value_bits, H):
    return np.full((1, H), value_bits, np.uint16)


@pytest.mark.parametrize("p", [1, 2])
@pytest.mark.parametrize("bits", [0x3F80, 0x4040, 0xC2C8, 0x0001, 0x0080, 0x7F7F, 0x3C00])
def test_constant_row_estimate_is_the_block_scale(oracle_mod, p, bits):
    """A constant row has s_k = s for every block, so the power mean is s and
    inv_rms = 1/s exactly for both p (the estimator formula with c = 1)."""
    H = 256
    codes, scales, inv = oracle_mod.mxnorm_quant(const_row(bits, H), p, "mxfp8")
    amax = abs(float(synth.bf16_bits_to_f32(np.array([bits]))[0]))
    e = max(-127, math.floor(math.log2(amax)) - 8)
    assert (scales == e + 127).all()
    assert inv[0] == np.float32(2.0 ** -e)


@pytest.mark.parametrize("a,b", [(0, 0), (0, 3), (-5, 7), (-100, 90), (2, -60)])
def test_two_level_row_closed_form(oracle_mod, a, b):
    """Half the blocks with scale 2^a, half with 2^b:
    M_1 = (2^a + 2^b)/2, M_2 = sqrt((4^a + 4^b)/2); inv_rms = RN_fp32(1/M_p)."""
    H, K = 512, 16
    x = np.zeros((1, H), np.float32)
    x[0, : H // 2] = 2.0 ** (a + 8)     # amax 2^(a+8) -> e = a for E4M3
    x[0, H // 2:] = 2.0 ** (b + 8)
    xb = synth.f32_to_bf16_bits(x)
    _, scales, inv1 = oracle_mod.mxnorm_quant(xb, 1, "mxfp8")
    _, _, inv2 = oracle_mod.mxnorm_quant(xb, 2, "mxfp8")
    assert scales[0, : K // 2].tolist() == [a + 127] * (K // 2)
    assert scales[0, K // 2:].tolist() == [b + 127] * (K // 2)
    m1 = (Fraction(2) ** a + Fraction(2) ** b) / 2
    m2sq = (Fraction(4) ** a + Fraction(4) ** b) / 2
    assert inv1[0] == np.float32(float(1 / m1))
    want2 = 1.0 / math.sqrt(float(m2sq))
    assert abs(float(inv2[0]) - want2) <= 0.5 * float(np.spacing(np.float32(want2)))


@pytest.mark.parametrize("p", [1, 2])
def test_single_nonzero_block(oracle_mod, p):
    """One block at scale s, K-1 zero blocks at 2^-127:
    M_p = ((s^p + (K-1) 2^(-127p)) / K)^(1/p) ~= K^(-1/p) s."""
    H, K = 1024, 32
    x = np.zeros((1, H), np.float32)
    x[0, 40:72] = 3.0     # block 1 (elements 32..63) partly, block 2 partly
    x[0, 32:64] = 3.0     # block 1 fully: amax 3 -> e = 1 - 8 = -7
    x[0, 64:72] = 0.0
    xb = synth.f32_to_bf16_bits(x)
    _, scales, inv = oracle_mod.mxnorm_quant(xb, p, "mxfp8")
    assert scales[0, 1] == 120 and (np.delete(scales[0], 1) == 0).all()
    mp = ((Fraction(2) ** (-7 * p) + (K - 1) * Fraction(2) ** (-127 * p)) / K)
    want = 1.0 / (float(mp) if p == 1 else math.sqrt(float(mp)))
    assert abs(float(inv[0]) - want) <= 0.5 * float(np.spacing(np.float32(want)))
    approx = K ** (1.0 / p) * 2.0 ** 7
    assert abs(float(inv[0]) / approx - 1) < 1e-6


def test_zero_row(oracle_mod):
    x = np.zeros((2, 64), np.uint16)
    x[1] = 0x8000  # -0
    codes, scales, inv = oracle_mod.mxnorm_quant(x, 2, "mxfp8")
    assert (scales == 0).all()
    assert (codes[0] == 0).all() and (codes[1] == 0x80).all()
    assert (inv == np.float32(2.0 ** 127)).all()


def test_nonfinite_block_reading(oracle_mod):
    x = synth.make_random_rows(2, 96, 1)
    x[0, 40] = 0x7F80          # +Inf in block 1
    x[1, 70] = 0x7FC0          # NaN in block 2
    codes, scales, inv = oracle_mod.mxnorm_quant(x, 2, "mxfp8")
    assert scales[0, 1] == 0xFF and (codes[0, 32:64] == 0x7F).all()
    assert scales[1, 2] == 0xFF and (codes[1, 64:96] == 0x7F).all()
    assert scales[0, 0] != 0xFF and scales[0, 2] != 0xFF
    assert np.isnan(inv).all()
    c4, s4, i4 = oracle_mod.mxnorm_quant(x, 2, "mxfp4")
    assert s4[0, 1] == 0xFF and (c4[0, 16:32] == 0).all() and np.isnan(i4).all()


# ----------------------------------------------------------- invariants
@pytest.mark.parametrize("fmt,emax,qmax", [("mxfp8", 8, 448.0), ("mxfp4", 2, 6.0), ("mxfp4_h16", 2, 6.0),
                                           ("mxfp8_h16", 8, 448.0), ("mxfp4_h32", 2, 6.0), ("mxfp8_h32", 8, 448.0)])
@pytest.mark.parametrize("p", [1, 2])
def test_cast_and_growth_invariants(oracle_mod, fmt, emax, qmax, p):
    """|dec(q)| <= qmax; |dec(q) - x/s| <= half a grid step unless saturated;
    saturation only when |x|/s > qmax; and the growth bound of the estimator,
    |v_j| * inv_rms < K^(1/p) * 2^(emax+1) (section 4, Analisis de Picos:
    O(K) growth for p = 1, tighter for p = 2)."""
    w = synth.WORKLOADS["llama3_8b_65536x4096"]
    x = synth.make_activations(w, rows=8)
    codes, scales, inv = oracle_mod.mxnorm_quant(x, p, fmt)
    K = w.K
    v = synth.bf16_bits_to_f32(x).astype(np.float64)
    if fmt.endswith("_h16"):
        v = oracle_mod.h16(v.astype(np.float32)).reshape(v.shape).astype(np.float64)
    elif fmt.endswith("_h32"):
        v = oracle_mod.h32(v.astype(np.float32)).reshape(v.shape).astype(np.float64)
    s = np.exp2(scales.astype(np.float64) - 127)
    r = v / np.repeat(s, 32, axis=1)
    if fmt.startswith("mxfp8"):
        dec = np.vectorize(oracle_mod.decode_e4m3)(codes)
        grid = np.array([oracle_mod.decode_e4m3(c) for c in range(127)])
    else:
        nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(codes.shape[0], -1)
        dec = np.vectorize(oracle_mod.decode_e2m1)(nib)
        grid = np.array([oracle_mod.decode_e2m1(c) for c in range(8)])
    assert (np.abs(dec) <= qmax).all()
    sat = np.abs(r) > qmax
    assert (np.abs(dec[sat]) == qmax).all()
    step = np.diff(grid)
    idx = np.clip(np.searchsorted(grid, np.abs(r[~sat]), side="right") - 1, 0, len(step) - 1)
    assert (np.abs(np.abs(dec[~sat]) - np.abs(r[~sat])) <= step[idx] / 2).all()
    # amax/s lies in [2^emax, 2^(emax+1)) for non-zero blocks
    amax = np.abs(v).reshape(v.shape[0], K, 32).max(-1)
    assert ((amax / s >= 2.0 ** emax) & (amax / s < 2.0 ** (emax + 1))).all()
    bound = K ** (1.0 / p) * 2.0 ** (emax + 1)
    assert (np.abs(v) * inv[:, None].astype(np.float64) < bound).all()


def test_growth_bound_is_tight_for_p1_with_one_outlier(oracle_mod):
    """One huge element against tiny blocks: p = 1 lets |x| * inv approach
    K * 2^(emax+1) while p = 2 stays below sqrt(K) * 2^(emax+1)."""
    H, K = 4096, 128
    x = np.full((1, H), 2.0 ** -100, np.float32)
    x[0, 0] = 2.0 ** 20 * 1.99
    xb = synth.f32_to_bf16_bits(x)
    v = abs(float(synth.bf16_bits_to_f32(xb)[0, 0]))
    _, _, inv1 = oracle_mod.mxnorm_quant(xb, 1, "mxfp8")
    _, _, inv2 = oracle_mod.mxnorm_quant(xb, 2, "mxfp8")
    assert v * float(inv1[0]) > 0.95 * K * 2.0 ** 9
    assert v * float(inv2[0]) > 0.95 * math.sqrt(K) * 2.0 ** 9
    assert v * float(inv2[0]) < math.sqrt(K) * 2.0 ** 9


# ------------------------------------------------------ brute force rows
def _check_rows_vs_bruteforce(oracle_mod, x, p, fmt):
    from oracle import bruteforce as bf
    codes, scales, inv = oracle_mod.mxnorm_quant(x, p, fmt)
    for t in range(x.shape[0]):
        bc, bs, bi = bf.mxnorm_row([int(b) for b in x[t]], p, fmt)
        assert codes[t].tolist() == bc, (t, fmt, p)
        assert scales[t].tolist() == bs, (t, fmt, p)
        assert Fraction(float(inv[t])) == bi, (t, fmt, p, float(inv[t]), float(bi))


def test_tiny_workload_vs_bruteforce(oracle_mod):
    """The tiny oracle case (64 x 256, seed 0, N(0,1), channels 17 and 200
    x50, MXFP8, p = 2) row by row against the exact-rational brute force."""
    w = synth.WORKLOADS["tiny_64x256"]
    _check_rows_vs_bruteforce(oracle_mod, synth.make_activations(w), 2, "mxfp8")


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "mxfp4_h16", "mxfp8_h16", "mxfp4_h32", "mxfp8_h32"])
@pytest.mark.parametrize("p", [1, 2])
@pytest.mark.parametrize("H", [32, 64, 96, 256])
def test_random_tiny_rows_vs_bruteforce(oracle_mod, fmt, p, H):
    rng = np.random.default_rng(H * 10 + p)
    x = rng.standard_normal((3, H)).astype(np.float32) * np.exp2(rng.integers(-20, 20, (3, 1))).astype(np.float32)
    x[:, rng.integers(0, H)] *= 40
    _check_rows_vs_bruteforce(oracle_mod, synth.f32_to_bf16_bits(x), p, fmt)


def test_subnormal_and_extreme_rows_vs_bruteforce(oracle_mod):
    x = np.zeros((3, 64), np.uint16)
    x[0] = np.arange(1, 65, dtype=np.uint16)            # bf16 subnormals
    x[1] = 0x7F7F - np.arange(64, dtype=np.uint16)      # near the bf16 maximum
    x[2, ::2] = 0x0001
    x[2, 1::2] = 0x8003                                 # mixed-sign subnormals
    for p in (1, 2):
        _check_rows_vs_bruteforce(oracle_mod, x, p, "mxfp8")
        _check_rows_vs_bruteforce(oracle_mod, x, p, "mxfp4")


# --------------------------------------------------- RMSNorm baseline
def test_rmsnorm_baseline_constant_rows(oracle_mod):
    """Constant row c: RMS = |c|, inv = RN_fp32(1/sqrt(c^2 + eps))."""
    for c in [1.0, -3.0, 0.5, 100.0]:
        x = synth.f32_to_bf16_bits(np.full((1, 128), c, np.float32))
        y, codes, scales, inv = oracle_mod.rmsnorm_mxfp8(x, 1e-5)
        want = np.float32(1.0 / math.sqrt(c * c + 1e-5))
        assert inv[0] == want
        ref, _ = oracle_mod.mx_cast(y, "mxfp8")
        assert (codes == ref).all()


def test_rmsnorm_baseline_vs_torch_rms_norm(oracle_mod):
    """y against torch.nn.functional.rms_norm in fp64 (library routine):
    within one bf16 ulp (the oracle rounds x*inv to fp32 then to bf16)."""
    x = synth.make_activations(synth.WORKLOADS["llama3_1b_32768x2048"], rows=4)
    y, codes, scales, inv = oracle_mod.rmsnorm_mxfp8(x, 1e-5)
    xt = torch.from_numpy(synth.bf16_bits_to_f32(x).astype(np.float64))
    ref = torch.nn.functional.rms_norm(xt, (x.shape[1],), eps=1e-5).numpy()
    yv = synth.bf16_bits_to_f32(y).astype(np.float64)
    assert (np.abs(yv - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30).all()
    rms = np.sqrt((synth.bf16_bits_to_f32(x).astype(np.float64) ** 2).mean(1) + 1e-5)
    np.testing.assert_allclose(inv.astype(np.float64), 1 / rms, rtol=2 ** -24)
    c2, s2 = oracle_mod.mx_cast(y, "mxfp8")
    assert (c2 == codes).all() and (s2 == scales).all()


def test_h16_rotation_preserves_row_rms(oracle_mod):
    """H16/4 is orthonormal, so rotating a row keeps its RMS (the reason the
    rotated path may feed the same estimator)."""
    x = synth.make_activations(synth.WORKLOADS["llama3_8b_mxfp4_h16_65536x4096"], rows=4)
    v = synth.bf16_bits_to_f32(x).astype(np.float32)
    y = oracle_mod.h16(v).reshape(v.shape).astype(np.float64)
    np.testing.assert_allclose(np.sqrt((y ** 2).mean(1)), np.sqrt((v.astype(np.float64) ** 2).mean(1)), rtol=1e-6)


# ------------------------------------------------------- backward (STE)
def _rms_inv(xv):
    return 1.0 / np.sqrt((xv.astype(np.float64) ** 2).mean(-1))


def test_bwd_matches_finite_differences_of_rmsnorm(oracle_mod):
    """With the exact 1/RMS as the saved normaliser, the straight-through
    backward is RMSNorm's exact gradient: compare with central differences of
    L(x) = sum_j w_j x_j / RMS(x) in fp64 ("MXNorm ...", Gradientes)."""
    rng = np.random.default_rng(12)
    T, H = 3, 64
    xb = synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wb = synth.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    xv = synth.bf16_bits_to_f32(xb).astype(np.float64)
    wv = synth.bf16_bits_to_f32(wb).astype(np.float64)
    inv = _rms_inv(xv).astype(np.float32)
    dx = synth.bf16_bits_to_f32(oracle_mod.mxnorm_bwd_ste(xb, wb, inv)).astype(np.float64)

    def L(row, t):
        return float((wv[t] * row).sum() / np.sqrt((row ** 2).mean()))

    for t in range(T):
        fd = np.empty(H)
        for i in range(H):
            h = 1e-6 * max(1.0, abs(xv[t, i]))
            e = np.zeros(H)
            e[i] = h
            fd[i] = (L(xv[t] + e, t) - L(xv[t] - e, t)) / (2 * h)
        scale = np.abs(fd).max()
        assert np.abs(dx[t] - fd).max() <= 2.0 ** -7 * scale, t


def test_bwd_is_orthogonal_to_x_for_the_exact_normaliser(oracle_mod):
    """RMSNorm is scale invariant, so its gradient is orthogonal to x:
    sum_j dx_j x_j = 0 (up to the bf16 rounding of dx)."""
    x = synth.make_activations(synth.WORKLOADS["llama3_1b_32768x2048"], rows=4)
    dyb = synth.make_random_rows(4, 2048, seed=13)
    xv = synth.bf16_bits_to_f32(x).astype(np.float64)
    dx = synth.bf16_bits_to_f32(oracle_mod.mxnorm_bwd_ste(x, dyb, _rms_inv(xv).astype(np.float32))).astype(np.float64)
    dot = (dx * xv).sum(1)
    assert (np.abs(dot) <= 2.0 ** -7 * (np.abs(dx) * np.abs(xv)).sum(1)).all()


def test_bwd_closed_forms(oracle_mod):
    """dy orthogonal to x: dx = rho dy exactly (then bf16); dy = y = rho x with
    rho = 1/RMS: dx = 0."""
    H = 32
    x = np.zeros((2, H), np.float32)
    x[:, 0] = 2.0
    dy = np.zeros((2, H), np.float32)
    dy[0, 1:] = np.linspace(-1, 1, H - 1)
    inv = np.array([0.75, 1.0 / np.sqrt(4.0 / H)], np.float32)
    dy[1] = x[1] * inv[1]
    dx = synth.bf16_bits_to_f32(oracle_mod.mxnorm_bwd_ste(synth.f32_to_bf16_bits(x), synth.f32_to_bf16_bits(dy), inv))
    want0 = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits((0.75 * synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(dy[0]))).astype(np.float32)))
    np.testing.assert_array_equal(dx[0], want0)
    assert np.abs(dx[1]).max() <= 1e-6


@pytest.mark.parametrize("a", [-100, -60, -40, 50, 60])
def test_bwd_scale_equivariance_at_extreme_row_scales(oracle_mod, a):
    """dx(2^a x, dy, 2^-a r) = 2^-a dx(x, dy, r) exactly: every term of
    r dy - r^3 x mean(dy x) scales by 2^-a, so the unrounded result must too
    (fp64 keeps the products of such rows far from its own range limits).
    Pins the oracle on rows whose amax is near 2^-100 .. 2^60 against its
    values on ordinary rows."""
    T, H = 4, 256
    x = synth.make_random_rows(T, H, seed=31, scale=2.0)
    dy = synth.make_random_rows(T, H, seed=32)
    inv = np.array([0.5, 0.75, 1.25, 3.0], np.float32)
    xs = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(x) * np.float32(2.0 ** a))
    assert np.array_equal(synth.bf16_bits_to_f32(xs), synth.bf16_bits_to_f32(x) * np.float32(2.0 ** a))
    _, ref = oracle_mod.mxnorm_bwd_ste(x, dy, inv, with_f64=True)
    _, got = oracle_mod.mxnorm_bwd_ste(xs, dy, (inv * np.float32(2.0 ** -a)).astype(np.float32), with_f64=True)
    assert np.array_equal(got, ref * 2.0 ** -a)


def test_bwd_zero_and_subnormal_rows_exact(oracle_mod):
    """The two rows whose forward estimate is the largest, 2^127: an all-zero
    row gives dx = 2^127 dy exactly (bf16 Inf where that exceeds the bf16
    range), and a row of bf16 subnormals matches the definition evaluated in
    exact rationals (fp64's rounding stays below 2^-50 of the largest term)."""
    from oracle import bruteforce as bf
    H = 64
    r = np.float32(2.0 ** 127)
    dyb = synth.make_random_rows(2, H, seed=33)
    dyb[0, :4] = [0x3FFF, 0x4000, 0xC000, 0x4010]   # 1.9921875 (2^127 of it is bf16 max), 2, -2, 2.25
    xb = np.zeros((2, H), np.uint16)
    xb[1] = (np.arange(H, dtype=np.uint16) * 37) % 0x7F + 1
    xb[1, ::3] |= np.uint16(0x8000)
    dx, dx64 = oracle_mod.mxnorm_bwd_ste(xb, dyb, np.array([r, r], np.float32), with_f64=True)
    dyv = synth.bf16_bits_to_f32(dyb[0]).astype(np.float64)
    assert np.array_equal(dx64[0], dyv * 2.0 ** 127)
    big = np.abs(dyv) * 2.0 ** 127 >= (2 - 2.0 ** -8) * 2.0 ** 127
    assert big.sum() >= 3 and ((dx[0] & 0x7FFF) == 0x7F80)[big].all()
    assert np.array_equal(dx[0][~big], dyb[0][~big] + np.uint16(127 << 7))
    rq = Fraction(2) ** 127
    xs = [bf.bf16_value(int(b)) for b in xb[1]]
    gs = [bf.bf16_value(int(b)) for b in dyb[1]]
    dot = sum(g * v for g, v in zip(gs, xs))
    exact = [rq * g - rq ** 3 * v * dot / H for g, v in zip(gs, xs)]
    scale = max(abs(rq * g) for g in gs) + max(abs(rq ** 3 * v * dot / H) for v in xs)
    for j in range(H):
        assert abs(Fraction(float(dx64[1, j])) - exact[j]) <= scale * Fraction(1, 2 ** 50), j


# ------------------------------------------------------------------ NVFP4
def _f32_bits(v):
    import struct
    return struct.unpack("<I", struct.pack("<f", float(np.float32(v))))[0]


@pytest.mark.parametrize("g", [1.0, 0.0123, 3.7e-3, 2.5e-5])
@pytest.mark.parametrize("p", [1, 2])
def test_nvfp4_vs_bruteforce(oracle_mod, g, p):
    from oracle import bruteforce as bf
    rng = np.random.default_rng(int(g * 1e6) + p)
    x = rng.standard_normal((4, 64)).astype(np.float32) * np.float32(3.0)
    x[1, 5] *= 200
    x[2, :16] *= 1e-6       # a block whose scale underflows for large g
    xb = synth.f32_to_bf16_bits(x)
    gf = float(np.float32(g))
    c, s, i = oracle_mod.nvfp4_quant(xb, p, gf)
    for t in range(4):
        bc, bs, bi = bf.nvfp4_row([int(v) for v in xb[t]], p, _f32_bits(gf))
        assert list(c[t]) == bc and list(s[t]) == bs
        assert (bi is None and np.isinf(i[t])) or Fraction(float(i[t])) == bi


def test_nvfp4_closed_forms(oracle_mod):
    """Constant row 6.0 with g = 1: block scale 6/6 = 1.0 (E4M3 0x38), codes
    6.0 (0x7 | 0x7 << 4), inv_rms = 1/(1 * 1) = 1.  A zero row: scales 0,
    codes 0, inv_rms +Inf.  A block beyond 448 * 6 * g saturates its scale
    at 448 (0x7E) and its codes at 6."""
    x = synth.f32_to_bf16_bits(np.full((1, 32), 6.0, np.float32))
    c, s, i = oracle_mod.nvfp4_quant(x, 2, 1.0)
    assert (s == 0x38).all() and (c == 0x77).all() and i[0] == 1.0
    c, s, i = oracle_mod.nvfp4_quant(np.zeros((1, 32), np.uint16), 2, 1.0)
    assert (s == 0).all() and (c == 0).all() and np.isinf(i[0])
    x = synth.f32_to_bf16_bits(np.full((1, 16), 5000.0, np.float32))
    c, s, i = oracle_mod.nvfp4_quant(x, 1, 1.0)
    assert (s == 0x7E).all() and (c == 0x77).all()
    assert i[0] == np.float32(1.0 / 448.0)


def test_nvfp4_invariants(oracle_mod):
    """Decoded values never exceed 6 * s * g, the block scale is the E4M3
    rounding of amax / (6 g), and the p = 2 estimate is the quadratic mean of
    the decode scales."""
    w = synth.WORKLOADS["llama3_8b_65536x4096"]
    x = synth.make_activations(w, rows=4)
    xv = synth.bf16_bits_to_f32(x).astype(np.float64)
    g = float(np.float32(np.abs(xv).max() / (448 * 6)))
    c, s, i = oracle_mod.nvfp4_quant(x, 2, g)
    sval = np.vectorize(oracle_mod.decode_e4m3)(s)
    amax = np.abs(xv).reshape(4, -1, 16).max(-1)
    np.testing.assert_array_equal(s, oracle_mod.cast_e4m3((amax.astype(np.float32) / np.float32(6 * np.float32(g))).astype(np.float64)))
    nib = np.stack([c & 0xF, c >> 4], -1).reshape(4, -1)
    dec = np.vectorize(oracle_mod.decode_e2m1)(nib).reshape(4, -1, 16)
    assert (np.abs(dec) <= 6).all()
    want = 1.0 / np.sqrt(((sval * g) ** 2).mean(1))
    np.testing.assert_allclose(i, want, rtol=1e-6)


# ---------------------------------------------------------- MXNormLinear
def _e4m3_values(codes):
    from oracle import bruteforce as bf
    table = np.full(256, np.nan)
    for c, v in bf.e4m3_values().items():
        table[c] = float(v)
    return table[codes]


def test_linear_matches_matmul_of_dequantized(oracle_mod):
    """The consumer GEMM equals diag(inv) @ (Xv @ Wv^T) with numpy's matmul on
    the dequantised operands (E4M3 values from the brute-force code table
    times 2^(scale - 127))."""
    x = synth.make_activations(synth.WORKLOADS["llama3_125m_16384x768"], rows=8)
    xc, xs, inv = oracle_mod.mxnorm_quant(x, 2, "mxfp8")
    w = synth.make_random_rows(24, 768, seed=3, scale=0.05)
    wc, ws = oracle_mod.mx_cast(w, "mxfp8")
    xv = _e4m3_values(xc) * np.repeat(np.exp2(xs.astype(np.float64) - 127), 32, axis=1)
    wv = _e4m3_values(wc) * np.repeat(np.exp2(ws.astype(np.float64) - 127), 32, axis=1)
    want = inv.astype(np.float64)[:, None] * (xv @ wv.T)
    got = oracle_mod.mxfp8_linear(xc, xs, inv, wc, ws)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-300)


def test_linear_identity_weight(oracle_mod):
    """W^ = identity (code 1.0, scale 2^0): out = inv * x^."""
    K = 64
    xc = np.array([[0x38 + (k % 7) for k in range(K)], [0xB0 + (k % 5) for k in range(K)]], np.uint8)
    xs = np.array([[120, 130], [127, 100]], np.uint8)
    inv = np.array([0.5, 3.0], np.float32)
    wc = np.zeros((K, K), np.uint8)
    wc[np.arange(K), np.arange(K)] = 0x38
    ws = np.full((K, K // 32), 127, np.uint8)
    got = oracle_mod.mxfp8_linear(xc, xs, inv, wc, ws)
    xv = _e4m3_values(xc) * np.repeat(np.exp2(xs.astype(np.float64) - 127), 32, axis=1)
    np.testing.assert_array_equal(got, inv.astype(np.float64)[:, None] * xv)


# ------------------------------------------------ gain-folded weight cast
def test_gain_cast_unit_gain_is_the_plain_cast(oracle_mod):
    from mx_scale_reusing_gb300 import synth
    w = synth.make_random_rows(16, 512, seed=21, scale=3.0)
    c1, s1 = oracle_mod.mx_cast_gain(w, np.ones(512, np.float32), 1.0)
    c0, s0 = oracle_mod.mx_cast(w, "mxfp8")
    np.testing.assert_array_equal(c1, c0)
    np.testing.assert_array_equal(s1, s0)


def test_gain_cast_power_of_two_shifts_the_scales(oracle_mod):
    """gamma = 2^j everywhere (c = 1): every product is exact, so the codes
    are the plain cast's and each scale code moves by j (normal-range
    blocks, away from the E8M0 clamps)."""
    from mx_scale_reusing_gb300 import synth
    w = synth.make_random_rows(16, 256, seed=22, scale=1.0)
    for j in (-5, 3):
        c1, s1 = oracle_mod.mx_cast_gain(w, np.full(256, 2.0 ** j, np.float32), 1.0)
        c0, s0 = oracle_mod.mx_cast(w, "mxfp8")
        np.testing.assert_array_equal(c1, c0)
        np.testing.assert_array_equal(s1.astype(int), s0.astype(int) + j)


def test_gain_cast_vs_bruteforce(oracle_mod):
    """Random fp32 gains (incl. +-0 and negatives) and c = 1.37: the C
    oracle equals the exact-fraction implementation."""
    from oracle import bruteforce as bf
    from mx_scale_reusing_gb300 import synth
    rng = np.random.default_rng(23)
    K = 96
    w = synth.make_random_rows(4, K, seed=24, scale=2.0)
    gamma = (np.exp(rng.normal(0, 0.7, K)) * rng.choice([-1.0, 1.0], K)).astype(np.float32)
    gamma[[3, 40]] = [0.0, -0.0]
    gamma[7] = np.float32(3.0e-39)  # subnormal gain
    c = np.float32(1.37)
    oc, os_ = oracle_mod.mx_cast_gain(w, gamma, float(c))
    gb = gamma.view(np.uint32).tolist()
    cb = int(np.array([c], np.float32).view(np.uint32)[0])
    for n in range(w.shape[0]):
        codes, scales = bf.mx_cast_gain_row([int(b) for b in w[n]], gb, cb)
        assert oc[n].tolist() == codes, n
        assert os_[n].tolist() == scales, n


# ------------------------------------------- Theorem 1 diagnostic (bounds)
@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4", "mxfp4_h16", "mxfp8_h16", "mxfp8_h32"])
@pytest.mark.parametrize("p", [1, 2])
def test_theorem1_ratio_within_e8m0_bounds(oracle_mod, fmt, p):
    """RMS_exact * inv_rms lies in the interval the E8M0 rule forces (derived
    in oracle/theorem1.py from 2^emax s <= amax < 2^(emax+1) s and the
    block's sum of squares in [amax^2, 32 amax^2]); rotated formats get
    1e-6 relative slack for the fp32 rounding of the rotation."""
    from oracle import theorem1
    from mx_scale_reusing_gb300 import synth
    for name, rows in (("tiny_64x256", None), ("llama3_125m_16384x768", 1024)):
        w = synth.WORKLOADS[name]
        x = synth.make_activations(w, rows=rows)
        r = theorem1.ratio(x, p, fmt)
        lo, hi = theorem1.bounds(p, fmt, w.H)
        slack = 1e-6 if "_h" in fmt else 0.0
        assert (r >= lo * (1 - slack)).all() and (r < hi * (1 + slack)).all(), (name, r.min(), r.max(), lo, hi)


@pytest.mark.parametrize("fmt,emax", [("mxfp8", 8), ("mxfp4", 2)])
def test_theorem1_ratio_constant_rows(oracle_mod, fmt, emax):
    """A constant row v gives |v| / 2^(floor(log2 |v|) - emax) for both p,
    which reaches both ends of the p = 2 bound's top octave."""
    from oracle import theorem1
    from mx_scale_reusing_gb300 import synth
    vals = np.array([1.0, -1.5, 3.0, 0.75, 1.9921875, 2.0 ** -20, 300.0], np.float32)
    x = synth.f32_to_bf16_bits(np.repeat(vals[:, None], 256, axis=1))
    v = synth.bf16_bits_to_f32(x[:, 0]).astype(np.float64)
    want = np.abs(v) / np.exp2(np.floor(np.log2(np.abs(v))) - emax)
    for p in (1, 2):
        np.testing.assert_allclose(theorem1.ratio(x, p, fmt), want, rtol=1e-7)
    assert (want >= 2.0 ** emax).all() and (want < 2.0 ** (emax + 1)).all()


# ------------------------------ gain-folded cast: where each rounding falls
def _fp32_grid_above(v):
    """Smallest float32 strictly above the positive rational v (normal range)."""
    from fractions import Fraction as F
    import math
    e = math.floor(math.log2(v))
    if F(2) ** e > v:
        e -= 1
    if F(2) ** (e + 1) <= v:
        e += 1
    step = F(2) ** (e - 23)
    k = math.floor(v / step) + 1
    return k * step


def _f32_bits(v) -> int:
    return int(np.array([float(v)], np.float32).view(np.uint32)[0])


def _gain_row(x_bits0, g0, anchor_bits=0x4396):
    """A 32-element row: element 0 = (x_bits0, gain g0), element 1 = the
    anchor (300 in bf16 by default) with gain 1, the rest 0 with gain 1.
    With c * anchor = 300 the block amax is 300 and its scale 2^0."""
    w = np.zeros((1, 32), np.uint16)
    w[0, 0] = x_bits0
    w[0, 1] = anchor_bits
    g = np.ones(32, np.float32)
    g[0] = np.float32(float(g0))
    return w, g


def test_gain_cast_each_product_rounds_to_fp32(oracle_mod):
    """x * g is exactly above the E4M3 tie 17/16 (between 1.0 and 1.125) by
    less than half an fp32 ulp, so RN_fp32(x * g) = 17/16 and the tie goes to
    the even code 1.0 (0x38); a product kept exact (or in fp64) would give
    1.125 (0x39).  The case is found by exact search over bf16 x = 1 + m/128."""
    from fractions import Fraction as F
    tie, half_ulp = F(17, 16), F(1, 2 ** 24)
    for m in range(9, 128):
        x = F(128 + m, 128)
        g = _fp32_grid_above(tie / x)
        if tie < x * g < tie + half_ulp:
            break
    else:
        pytest.fail("no case found")
    x_bits = 0x3F80 | m  # bf16 of 1 + m/128
    w, gam = _gain_row(x_bits, g)
    assert F(float(np.float32(float(g)))) == g
    codes, scales = oracle_mod.mx_cast_gain(w, gam, 1.0)
    assert scales[0, 0] == 127 and codes[0, 0] == 0x38


def test_gain_cast_gain_rounds_before_the_product(oracle_mod):
    """g = RN_fp32(c * gamma) is formed first: c = 3 and a gamma whose exact
    product with c is not an fp32 value, chosen so that x * RN(c * gamma)
    lands within half an fp32 ulp above the tie 17/16 (RN -> the tie -> 1.0,
    code 0x38) while the exact x * c * gamma lies above that window and
    rounds to 1.125 (0x39)."""
    from fractions import Fraction as F
    tie, half_ulp = F(17, 16), F(1, 2 ** 24)
    c = F(3)
    found = None
    for m in range(9, 128):
        x = F(128 + m, 128)
        # fp32 gains g just above tie / x; gamma = g / 3 rounded to fp32 so
        # that RN(3 * gamma) = g while 3 * gamma != g
        g = _fp32_grid_above(tie / x)
        if not (tie < x * g < tie + half_ulp):
            continue
        for gam in (_fp32_grid_above(g / c), _fp32_grid_above(g / c) - F(2) ** -25):
            cg = c * gam
            rn = F(float(np.float32(float(cg))))
            if rn == g and cg != g and x * cg >= tie + half_ulp:
                found = (m, gam)
                break
        if found:
            break
    if not found:
        pytest.skip("no discriminating case in the searched range")
    m, gam = found
    w, gvec = _gain_row(0x3F80 | m, gam, anchor_bits=0x42C8)  # 100 * c = 300
    assert F(float(gvec[0])) == gam
    codes, scales = oracle_mod.mx_cast_gain(w, gvec, 3.0)
    assert scales[0, 0] == 127 and codes[0, 0] == 0x38


@pytest.mark.parametrize("x,g,tie,code_x", [
    # RN(3 * RN(1/g)) = 3.5 exactly, the E2M1 tie between 3 and 4 -> even 4 (0x6);
    # RN(3 / g) = 3.4999998 would give 3 (0x5)
    (3.0, 0.8571429252624512, 3.5, 0x6),
    # RN(3.25 * RN(1/g)) = 0.74999994 -> 0.5 (0x1); RN(3.25 / g) = 0.75, the
    # tie between 0.5 and 1 -> even 1 (0x2)
    (3.25, 4.333333492279053, 0.75, 0x1),
])
def test_nvfp4_elements_scale_by_the_rounded_reciprocal(oracle_mod, x, g, tie, code_x):
    """The recipe's element step is r = RN(x * enc) with enc = RN(1 / d), not
    RN(x / d).  Two hand-derived cases where the two readings fall on either
    side of an E2M1 tie decide it.  The block scale is 1 (the block maximum a
    = 6g rounded to bf16 gives RN(a / RN(6g)) within an E4M3 half-step of 1),
    so d = RN(1 * g) = g."""
    from fractions import Fraction as F
    from oracle import bruteforce as bf
    gq = F(float(np.float32(g)))
    assert gq == F(g)  # g is an fp32 value
    enc = bf.round_to_fp32(1 / gq)
    assert (bf.round_to_fp32(F(x) * enc) == tie) != (bf.round_to_fp32(F(x) / gq) == tie)
    amax = float(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.array([6.0 * g], np.float32)))[0])
    row = np.zeros((1, 16), np.float32)
    row[0, 0], row[0, 1] = x, amax
    xb = synth.f32_to_bf16_bits(row)
    c, s, _ = oracle_mod.nvfp4_quant(xb, 2, float(np.float32(g)))
    assert s[0, 0] == 0x38                   # block scale 1.0
    assert c[0, 0] & 0xF == code_x           # element 0: the product reading's code
    assert c[0, 0] >> 4 == 0x7               # the block maximum: 6


@pytest.mark.parametrize("n", [16, 32])
def test_rotation_fp32_values_match_bruteforce(oracle_mod, n):
    """The rotated fp32 values themselves (not only the codes cast from
    them) equal the exact-fraction butterfly with the stated stage order and
    one fp32 rounding per add/sub and per final scale: on general fp32
    inputs a different stage order or a skipped rounding changes them."""
    from oracle import bruteforce as bf
    rng = np.random.default_rng(40 + n)
    v = (rng.standard_normal((24, n)) * np.exp(rng.normal(0, 3, (24, 1)))).astype(np.float32)
    v[0] = np.float32(1.0) + np.arange(n, dtype=np.float32) * np.float32(2.0 ** -20)  # rounding in every stage
    v[1] = (rng.standard_normal(n) * 2.0 ** -124).astype(np.float32)  # products of the 1/4 scale reach subnormals
    got = (oracle_mod.h16 if n == 16 else oracle_mod.h32)(v.reshape(-1)).reshape(v.shape)
    rot = bf.h16_fp32 if n == 16 else bf.h32_fp32
    for r in range(v.shape[0]):
        want = rot([Fraction(float(a)) for a in v[r]])
        assert [Fraction(float(a)) for a in got[r]] == want, r


def test_nvfp4_block_scale_divides_by_rounded_6g(oracle_mod):
    """sb = RN(amax / RN(6g)): with amax = 1 and g = 0.10666666 (fp32), RN(6g)
    makes sb the E4M3 tie 1.5625 exactly, which goes to the even scale 1.5
    (0x3C); dividing by the exact 6g would give 1.625 (0x3D)."""
    from fractions import Fraction as F
    from oracle import bruteforce as bf
    g = 0.10666666179895401
    gq = F(g)
    assert F(float(np.float32(g))) == gq
    assert bf.round_to_fp32(1 / bf.round_to_fp32(6 * gq)) == F(25, 16)
    assert bf.nearest_code(bf.round_to_fp32(1 / (6 * gq)), bf._E4M3, 0) == 0x3D
    row = np.zeros((1, 16), np.float32)
    row[0, 3] = 1.0
    _, s, _ = oracle_mod.nvfp4_quant(synth.f32_to_bf16_bits(row), 2, g)
    assert s[0, 0] == 0x3C


def test_nvfp4_reciprocal_of_the_rounded_decode_scale(oracle_mod):
    """enc = RN(1 / RN(s g)): block scale s = 1.125 (amax 2.4375), g =
    0.36111107 (fp32), element x = 0.5078125.  With d = RN(s g) the product
    RN(x * enc) is the E2M1 tie 1.25, which goes to the even 1.0 (0x2); with
    the exact s g it would give 1.5 (0x3)."""
    from fractions import Fraction as F
    from oracle import bruteforce as bf
    g, x, amax = 0.3611110746860504, 0.5078125, 2.4375
    gq, s = F(g), F(9, 8)
    assert F(float(np.float32(g))) == gq
    rt = bf.round_to_fp32
    assert bf.nearest_code(rt(F(amax) / rt(6 * gq)), bf._E4M3, 0) == 0x39   # s = 1.125
    assert rt(F(x) * rt(1 / rt(s * gq))) == F(5, 4)
    assert bf.nearest_code(rt(F(x) * rt(1 / (s * gq))), bf._E2M1, 0) == 0x3
    row = np.zeros((1, 16), np.float32)
    row[0, 0], row[0, 1] = x, amax
    c, sc, _ = oracle_mod.nvfp4_quant(synth.f32_to_bf16_bits(row), 2, g)
    assert sc[0, 0] == 0x39 and c[0, 0] & 0xF == 0x2 and c[0, 0] >> 4 == 0x7


def test_bf16_rounding_overflows_to_inf_like_torch(oracle_mod):
    """The oracle's fp32 -> bf16 rounding against torch's bfloat16
    conversion (round to nearest even, IEEE overflow to Inf): every fp32
    pattern in the top binade, around the overflow threshold bf16 max + half
    an ulp = 2^128 - 2^119 (a tie that goes to the even neighbour, Inf), and
    random patterns over the whole range."""
    rng = np.random.default_rng(44)
    top = np.arange(0x7F000000, 0x7F800001, 97, dtype=np.uint32)
    edge = np.arange(0x7F7F7F00, 0x7F7F8100, dtype=np.uint32)
    rand = rng.integers(0, 0x7F800000, 200000, dtype=np.uint32)
    u = np.concatenate([top, edge, rand, np.array([0x7F7F7FFF, 0x7F7F8000, 0x7F7FFFFF, 0x7F800000], np.uint32)])
    u = np.concatenate([u, u | np.uint32(0x80000000)])
    f = u.view(np.float32)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod.float_to_bf16(f)
    assert np.array_equal(got, want)
    assert got[np.where(u == 0x7F7F8000)[0][0]] == 0x7F80 and got[np.where(u == 0x7F7F7FFF)[0][0]] == 0x7F7F


def test_nvfp4_tensor_scale(oracle_mod):
    """g = RN_fp32(a / 2688), a the largest finite |x|: exact powers of two
    where a = 2688 * 2^j, numpy's IEEE fp32 division elsewhere, Inf and NaN
    ignored, 1.0 for a tensor with no finite nonzero element."""
    for j in (-20, -3, 0, 5, 60):
        x = np.zeros(64, np.float32)
        x[7] = -2688.0 * 2.0 ** j
        assert oracle_mod.nvfp4_tensor_scale(synth.f32_to_bf16_bits(x)) == 2.0 ** j
    rng = np.random.default_rng(45)
    for _ in range(200):
        xb = synth.make_random_rows(1, 300, seed=int(rng.integers(1 << 30)), scale=float(np.exp(rng.normal(0, 8))))[0]
        a = np.abs(synth.bf16_bits_to_f32(xb)).max()
        assert oracle_mod.nvfp4_tensor_scale(xb) == float(np.float32(a) / np.float32(2688.0))
    xb = synth.f32_to_bf16_bits(np.array([3.0, -5.0, 0.5], np.float32))
    xb = np.concatenate([xb, np.array([0x7F80, 0xFFC1, 0xFF80], np.uint16)])
    assert oracle_mod.nvfp4_tensor_scale(xb) == float(np.float32(5.0) / np.float32(2688.0))
    assert oracle_mod.nvfp4_tensor_scale(np.array([0, 0x8000, 0x7FC0], np.uint16)) == 1.0
    assert oracle_mod.nvfp4_tensor_scale(np.array([0x0001], np.uint16)) == float(np.float32(2.0 ** -133) / np.float32(2688.0))
