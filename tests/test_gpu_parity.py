"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Codes and E8M0 scales must be bit-exact; inv_rms must lie within 1e-6
relative of the oracle's.  The kernel's fixed-point power-mean sum is within
2^-33 of the exact sum; it then rounds the sum to fp32, divides and (p = 2)
takes the square root, each IEEE-rounded, for at most 2 * 2^-24 relative;
the oracle is exact in fp64 up to its final fp32 rounding (2^-24), so the two
differ by at most 3 * 2^-24 = 1.8e-7.  The two-pass baseline's inv is an
fp32 sum of squares: its bound is derived beside that test.
"""
import numpy as np
import pytest
import torch

import oracle
import mx_scale_reusing_gb300 as mx
from mx_scale_reusing_gb300 import synth

pytestmark = pytest.mark.gpu

INV_RTOL = 1e-6
FMTS = ["mxfp8", "mxfp4", "mxfp4_h16", "mxfp8_h16", "mxfp4_h32", "mxfp8_h32"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mx_scale_reusing_gb300 import _build
    _build.build()
    oracle.build()
    mx.lib()


def dev(xb: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).view(torch.bfloat16).cuda()


def run(xb, p, fmt, variant="auto"):
    x = dev(xb)
    c, s, i = mx.quant_fwd(x, p=p, fmt=fmt, variant=variant)
    torch.cuda.synchronize()
    return c.cpu().numpy(), s.cpu().numpy(), i.cpu().numpy()


def assert_inv_close(got, want, rtol=INV_RTOL):
    got = got.astype(np.float64)
    want = want.astype(np.float64)
    nan = np.isnan(want)
    assert (np.isnan(got) == nan).all(), "NaN pattern of inv_rms differs"
    rel = np.abs(got[~nan] / want[~nan] - 1.0)
    assert rel.size == 0 or rel.max() <= rtol, f"inv_rms rel err {rel.max():.3e}"


def assert_parity(xb, p, fmt, variant="auto", rows=None):
    c, s, i = run(xb, p, fmt, variant)
    ref_rows = np.arange(xb.shape[0]) if rows is None else np.asarray(rows)
    oc, os_, oi = oracle.mxnorm_quant(xb[ref_rows], p, fmt)
    bad = np.nonzero((c[ref_rows] != oc).any(1))[0]
    assert bad.size == 0, f"codes differ in {bad.size} rows, first row {ref_rows[bad[0]]}"
    assert np.array_equal(s[ref_rows], os_), "scales differ"
    assert_inv_close(i[ref_rows], oi)
    return c, s, i


def variants_for(H):
    v = ["warp_row"]
    if H * 2 * 8 * 2 <= 200 * 1024:
        v.append("tiled_tma")
    return v


# ------------------------------------------------------- exhaustive casts
def cast_sweep_rows(values_bits: np.ndarray, anchor_bits: int, H: int = 4096) -> np.ndarray:
    """Blocks of [anchor, 31 test values]: the anchor fixes the block's
    exponent at e = 0, so the cast sees each test value unscaled."""
    per = 31
    nblk = -(-values_bits.size // per)
    padded = np.zeros(nblk * per, np.uint16)
    padded[: values_bits.size] = values_bits
    blocks = np.concatenate([np.full((nblk, 1), anchor_bits, np.uint16), padded.reshape(nblk, per)], 1)
    K = H // 32
    nrow = -(-nblk // K)
    rows = np.zeros((nrow * K, 32), np.uint16)
    rows[:nblk] = blocks
    rows[nblk:, 0] = anchor_bits
    return rows.reshape(nrow, H)


@pytest.mark.parametrize("variant", ["warp_row", "tiled_tma"])
def test_e4m3_cast_every_bf16_below_512(variant):
    """Every bf16 magnitude below 512 (incl. subnormals, +-0, ties and the
    saturating range (448, 512)) through the hardware E4M3 cast."""
    mags = np.arange(0, 0x4400, dtype=np.uint16)
    vals = np.concatenate([mags, mags | np.uint16(0x8000)])
    xb = cast_sweep_rows(vals, 0x4380)  # anchor 256.0
    c, s, _ = assert_parity(xb, 2, "mxfp8", variant)
    assert (s == 127).all()


@pytest.mark.parametrize("variant", ["warp_row", "tiled_tma"])
def test_e2m1_cast_every_bf16_below_8(variant):
    mags = np.arange(0, 0x4100, dtype=np.uint16)
    vals = np.concatenate([mags, mags | np.uint16(0x8000)])
    xb = cast_sweep_rows(vals, 0x4080)  # anchor 4.0
    c, s, _ = assert_parity(xb, 2, "mxfp4", variant)
    assert (s == 127).all()


def test_scale_exponent_every_bf16_amax():
    """One block per finite bf16 magnitude as the block's absmax."""
    mags = np.arange(0, 0x7F80, dtype=np.uint16)
    K = 128
    nrow = -(-mags.size // K)
    blocks = np.zeros((nrow * K, 32), np.uint16)
    blocks[: mags.size, 5] = mags
    blocks[: mags.size, 9] = mags | np.uint16(0x8000)
    xb = blocks.reshape(nrow, K * 32)
    for fmt in ("mxfp8", "mxfp4"):
        assert_parity(xb, 1, fmt)


# ---------------------------------------------------------- workloads
_cache = {}


def workload_input(name, rows=None):
    key = (name, rows)
    if key not in _cache:
        _cache.clear()
        _cache[key] = synth.make_activations(synth.WORKLOADS[name], rows=rows)
    return _cache[key]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("p", [1, 2])
@pytest.mark.parametrize("variant", ["warp_row", "tiled_tma"])
def test_tiny_workload_all_elements(fmt, p, variant):
    assert_parity(workload_input("tiny_64x256"), p, fmt, variant)


@pytest.mark.parametrize("p", [1, 2])
@pytest.mark.parametrize("variant", ["warp_row", "tiled_tma"])
def test_llama3_125m_all_elements(p, variant):
    """16384 x 768: every element against the oracle (ragged chunking: 768 is
    three 256-element chunks per warp, 8-row tiles for the tiled kernel)."""
    assert_parity(workload_input("llama3_125m_16384x768"), p, "mxfp8", variant)


def oracle_all_rows(xb, p, fmt):
    """The oracle over every row, rows split across the host cores."""
    return oracle.rows_in_threads(lambda a: oracle.mxnorm_quant(a, p, fmt), xb)


@pytest.mark.parametrize("name,fmt,ps", [
    ("llama3_1b_32768x2048", "mxfp8", (2,)),
    ("llama3_8b_65536x4096", "mxfp8", (1, 2)),
    ("llama3_8b_65536x4096", "mxfp4", (2,)),
    ("llama3_8b_mxfp4_h16_65536x4096", "mxfp4_h16", (2,)),
    ("llama3_8b_mxfp4_h16_65536x4096", "mxfp4_h32", (2,)),
    ("llama3_8b_mxfp4_h16_65536x4096", "mxfp8_h16", (2,)),
    ("llama3_8b_mxfp4_h16_65536x4096", "mxfp8_h32", (2,)),
])
def test_full_size_workloads_every_row(name, fmt, ps):
    """Full-size inputs in the launch configuration the benchmark times,
    compared with the oracle element by element on every row: codes and
    E8M0 scales bit-exact, inv_rms within 1e-6 relative -- the estimator of
    "MXNorm ...", 2. Metodologia, Fundamentos Teoricos, on the block scales
    of the cast.  The auto variant is checked against the oracle; the
    explicit warp-row and tiled variants must equal it bit for bit."""
    xb = workload_input(name)
    T, H = xb.shape
    for p in ps:
        c, s, i = run(xb, p, fmt, "auto")
        oc, os_, oi = oracle_all_rows(xb, p, fmt)
        bad = np.nonzero((c != oc).any(1))[0]
        assert bad.size == 0, f"codes differ in {bad.size} of {T} rows, first row {bad[:1]}"
        bad = np.nonzero((s != os_).any(1))[0]
        assert bad.size == 0, f"scales differ in {bad.size} of {T} rows, first row {bad[:1]}"
        assert_inv_close(i, oi)
        del oc, os_, oi
        for v in variants_for(H):
            c2, s2, i2 = run(xb, p, fmt, v)
            assert np.array_equal(c2, c) and np.array_equal(s2, s) and np.array_equal(i2, i), v


# --------------------------------------------------------- edge cases
SHAPES = [(1, 32), (3, 96), (13, 800), (7, 8224), (33, 256), (11, 512), (9, 768), (41, 1024), (17, 2048), (100, 4096),
          (5, 4128), (6, 8192), (7, 1280), (2, 256), (1, 768)]


@pytest.mark.parametrize("T,H", SHAPES)
@pytest.mark.parametrize("fmt", FMTS)
def test_ragged_shapes(T, H, fmt):
    xb = synth.make_random_rows(T, H, seed=T * 7 + H, scale=3.0)
    for v in ["auto"] + variants_for(H):
        for p in (1, 2):
            assert_parity(xb, p, fmt, v)


def special_rows(H):
    rows = []
    rows.append(np.zeros(H, np.uint16))                          # +0 row
    rows.append(np.full(H, 0x8000, np.uint16))                   # -0 row
    rows.append(np.arange(H, dtype=np.uint16) % 0x7F + 1)        # subnormals
    rows.append(np.full(H, 0x3F80, np.uint16))                   # constant 1.0
    rows.append(np.full(H, 0xC2C8, np.uint16))                   # constant -100
    rows.append(0x7F7F - (np.arange(H, dtype=np.uint16) % 64))   # near bf16 max
    r = synth.make_random_rows(1, H, 3)[0]
    r[: H // 2] = 0                                              # half zero blocks
    rows.append(r)
    r = np.full(H, 0x0001, np.uint16)
    r[7] = 0x7F00                                                # one huge outlier
    rows.append(r)
    r = synth.make_random_rows(1, H, 4)[0]
    r[H - 3] = 0x7F80                                            # +Inf
    rows.append(r)
    r = synth.make_random_rows(1, H, 5)[0]
    r[1] = 0xFFC1                                                # NaN
    rows.append(r)
    return np.stack(rows)


@pytest.mark.parametrize("H", [32, 256, 4096])
@pytest.mark.parametrize("fmt", FMTS)
def test_special_rows(H, fmt):
    xb = special_rows(H)
    for v in ["auto"] + variants_for(H):
        for p in (1, 2):
            c, s, i = assert_parity(xb, p, fmt, v)
    assert (s[0] == 0).all() and i[0] == np.float32(2.0 ** 127)


def tiny_block_rows(H, seed):
    """Rows whose 32-element blocks sit at bf16 exponent fields from 60 down
    to 0 (2^-67 .. subnormal), one level per block, with random mantissas
    and signs; the last rows mix a normal value into tiny blocks.  The
    rotations' fp32 sums and their final scale (1/4 or 1/sqrt(32)) then
    produce subnormal fp32 values, which must round exactly as the oracle's
    butterfly does (no flush to zero), and blocks whose amax is subnormal
    get the clamped scale exponent -127."""
    rng = np.random.default_rng(seed)
    K = H // 32
    fields = np.linspace(60, 0, K).round().astype(np.int64)
    rows = []
    for r in range(6):
        f = np.repeat(np.clip(fields - 2 * r, 0, 254), 32)
        mant = rng.integers(0, 128, H)
        sign = rng.integers(0, 2, H) << 15
        row = (sign | (f << 7) | mant).astype(np.uint16)
        if r >= 4:
            row[rng.integers(0, H, 4)] = 0x3F80  # 1.0 inside some tiny blocks
        rows.append(row)
    return np.stack(rows)


@pytest.mark.parametrize("fmt", FMTS)
def test_tiny_blocks(fmt):
    xb = tiny_block_rows(1024, 3)
    for p in (1, 2):
        assert_parity(xb, p, fmt)


def test_variants_agree_at_full_size_repeatedly():
    """The benchmark's full 65536 x 4096 workload, eight launches of each
    variant back to back: the tiled (bulk-copy ring) and warp-row kernels
    agree bit for bit on every launch and no bounded pipeline wait gives up
    (a property that holds at any size; the oracle checks sampled rows)."""
    xb = workload_input("llama3_8b_65536x4096")
    x = dev(xb)
    mx.device_errors(clear=True)
    ref = mx.quant_fwd(x, 2, "mxfp8", "warp_row")
    torch.cuda.synchronize()
    for i in range(8):
        v = "tiled_tma" if i % 2 == 0 else "warp_row"
        c, s, inv = mx.quant_fwd(x, 2, "mxfp8", v)
        torch.cuda.synchronize()
        assert torch.equal(c, ref[0]) and torch.equal(s, ref[1]) and torch.equal(inv, ref[2]), f"launch {i} ({v})"
    assert mx.device_errors() == 0
    rows = np.array([0, 1, 4095, 32768, 65535])
    oc, os_, oi = oracle.mxnorm_quant(xb[rows], 2, "mxfp8")
    assert np.array_equal(ref[0][rows].cpu().numpy(), oc) and np.array_equal(ref[1][rows].cpu().numpy(), os_)


def test_empty_input_is_a_noop():
    x = torch.empty((0, 4096), dtype=torch.bfloat16, device="cuda")
    c, s, i = mx.quant_fwd(x)
    assert c.shape == (0, 4096) and s.shape == (0, 128) and i.shape == (0,)


def test_outputs_stay_in_bounds():
    """Guard bytes around every output buffer survive the call."""
    T, H = 37, 768
    xb = synth.make_random_rows(T, H, 9)
    x = dev(xb)
    for fmt in FMTS:
        cb = mx.code_bytes(H, fmt)
        for v in ["warp_row", "tiled_tma"]:
            g = 4096
            codes = torch.full((T * cb + 2 * g,), 0xA5, dtype=torch.uint8, device="cuda")
            scales = torch.full((T * H // 32 + 2 * g,), 0x5A, dtype=torch.uint8, device="cuda")
            inv = torch.full((T + 2 * g,), 7.0, dtype=torch.float32, device="cuda")
            out = (codes[g:g + T * cb].view(T, cb), scales[g:g + T * H // 32].view(T, H // 32), inv[g:g + T])
            mx.quant_fwd(x, 2, fmt, v, out=out)
            torch.cuda.synchronize()
            assert (codes[:g] == 0xA5).all() and (codes[-g:] == 0xA5).all()
            assert (scales[:g] == 0x5A).all() and (scales[-g:] == 0x5A).all()
            assert (inv[:g] == 7.0).all() and (inv[-g:] == 7.0).all()
            oc, os_, oi = oracle.mxnorm_quant(xb, 2, fmt)
            assert np.array_equal(out[0].cpu().numpy(), oc) and np.array_equal(out[1].cpu().numpy(), os_)


def test_runs_on_caller_stream():
    xb = workload_input("llama3_125m_16384x768")
    x = dev(xb)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        c, sc, i = mx.quant_fwd(x, 2, "mxfp8")
    s.synchronize()
    oc, os_, oi = oracle.mxnorm_quant(xb[:512], 2, "mxfp8")
    assert np.array_equal(c[:512].cpu().numpy(), oc)
    assert mx.device_errors() == 0


# --------------------------------------------------- two-pass baseline
def baseline_inv_rtol(H):
    """fp32 sum of squares: pairwise over a lane's 8 or 16 values, serial over
    the row's chunks, then a 5-level warp tree -- at most L = log2(VEC) +
    chunks + 5 roundings on a sum of non-negative terms, relative error
    <= L * 2^-24; the mean and + eps add two roundings, the correctly
    rounded reciprocal square root halves the input error and adds 2^-24,
    and the oracle's own final rounding adds 2^-24."""
    vec = 16 if H % 512 == 0 else 8
    chunks = -(-H // (32 * vec))
    L = int(np.log2(vec)) + chunks + 5
    return (L + 2) * 2.0 ** -25 + 2 * 2.0 ** -24


@pytest.mark.parametrize("name", ["tiny_64x256", "llama3_1b_32768x2048", "llama3_8b_65536x4096"])
def test_rmsnorm_mxfp8_baseline(name):
    """The two-pass baseline on every row of the workload."""
    xb = workload_input(name)
    T, H = xb.shape
    y, c, s, i = mx.rmsnorm_mxfp8_ref_fwd(dev(xb), eps=1e-5)
    torch.cuda.synchronize()
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16)
    c, s, i = c.cpu().numpy(), s.cpu().numpy(), i.cpu().numpy()
    oy, oc, os_, oi = oracle.rows_in_threads(lambda a: oracle.rmsnorm_mxfp8(a, 1e-5), xb)
    assert_inv_close(i, oi, rtol=baseline_inv_rtol(H))
    # y is x * inv in fp32 rounded to bf16, with the GPU's own inv
    want_y = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(xb) * i[:, None])
    assert np.array_equal(yb, want_y)
    # within one bf16 ulp of the oracle's y
    a, b = synth.bf16_bits_to_f32(yb), synth.bf16_bits_to_f32(oy)  # differences of bf16 values: exact in fp32
    assert (np.abs(a - b) <= np.abs(b) * 2.0 ** -7 + 1e-38).all()
    # stage 2 is the MXFP8 cast of the GPU's y, bit-exact
    rc, rs = oracle.rows_in_threads(lambda a: oracle.mx_cast(a, "mxfp8"), yb)
    assert np.array_equal(c, rc) and np.array_equal(s, rs)


@pytest.mark.parametrize("T,H", [(5, 32), (9, 768), (3, 800), (4, 8224)])
def test_rmsnorm_baseline_ragged(T, H):
    xb = synth.make_random_rows(T, H, seed=H)
    y, c, s, i = mx.rmsnorm_mxfp8_ref_fwd(dev(xb))
    torch.cuda.synchronize()
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16)
    _, _, _, oi = oracle.rmsnorm_mxfp8(xb, 1e-5)
    assert_inv_close(i.cpu().numpy(), oi, rtol=baseline_inv_rtol(H))
    rc, rs = oracle.mx_cast(yb, "mxfp8")
    assert np.array_equal(c.cpu().numpy(), rc) and np.array_equal(s.cpu().numpy(), rs)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode,chunks", [("staged", 1), ("staged", 3), ("staged", 8), ("zero_copy", 1)])
def test_host_buffer_path(fmt, mode, chunks):
    """quant_fwd_host (pinned host in, pinned host out; staged over three
    streams, or zero-copy with the kernel on the pinned buffers) gives the
    same bytes as the oracle."""
    xb = synth.make_random_rows(1000, 768, seed=21, scale=2.0)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory()
    c, s, i = mx.quant_fwd_host(x, p=2, fmt=fmt, chunks=chunks, mode=mode)
    torch.cuda.synchronize()
    oc, os_, oi = oracle.mxnorm_quant(xb, 2, fmt)
    assert np.array_equal(c.numpy(), oc) and np.array_equal(s.numpy(), os_)
    assert_inv_close(i.numpy(), oi)
