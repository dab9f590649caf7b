"""Parity of the straight-through backward kernel (mxnorm_bwd_ste, through
the C ABI) with the CPU oracle.

The oracle evaluates dx = r dy - r^3 x (1/H) sum(dy x) in fp64 (exact for
these inputs up to fp64 rounding); the kernel evaluates the same expression
grouped as xh = RN(r x), m = RN(RN(sum RN(dy xh)) / H), dx = RN(r RN(dy - xh m))
in fp32.  With exact X = r x, M = sum(dy X)/H, S = sum|dy X|, u = 2^-24 and
L the fp32 summation depth (log2 VEC + chunks + 5):
  |sum_gpu - H M| <= (L + 3) u S        (two roundings per product, L adds)
  |m - M|         <= (L + 3) u S / H + u |M|
  |dx_f32 - dx*|  <= r |X_j| (L + 3) u S / H + r u (3 |X_j| |M| + 2 |dy_j|) + 2 u |dx*_j|
plus, where an intermediate is an fp32 subnormal, absolute terms of half the
subnormal spacing eta = 2^-149 carried through the same products:
  r eta (|X_j| (mean|dy| + 1) + |M| + 1) + eta.
With the final bf16 rounding (2^-8 relative):
  |dx_gpu - dx*| <= 2^-8 |dx*| + (1 + 2^-8) E_j.
Where the oracle's bf16 dx is Inf or NaN the kernel's must be the same
pattern.
"""
import numpy as np
import pytest
import torch

import oracle
import mx_scale_reusing_gb300 as mx
from mx_scale_reusing_gb300 import synth

pytestmark = pytest.mark.gpu
U = 2.0 ** -24
ETA = 2.0 ** -149


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mx_scale_reusing_gb300 import _build
    _build.build()
    oracle.build()
    mx.lib()


def dev_bf16(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()


def bwd_bound(xv, gv, r, exact, H):
    """E_j above (per element) for rows xv, dy gv (fp64) and inv r [T, 1]."""
    X = r * xv
    M = (gv * X).sum(1, keepdims=True) / H
    S = np.abs(gv * X).sum(1, keepdims=True)
    vec = 16 if H % 512 == 0 else 8
    L = int(np.log2(vec)) + -(-H // (32 * vec)) + 5
    E = r * np.abs(X) * (L + 3) * U * S / H + r * U * (3 * np.abs(X) * np.abs(M) + 2 * np.abs(gv)) \
        + 2 * U * np.abs(exact)
    E += r * ETA * (np.abs(X) * (np.abs(gv).mean(1, keepdims=True) + 1) + np.abs(M) + 1) + ETA
    return E * (1 + 2.0 ** -16)


def compare_bwd(got_b, xb, gb, inv, min_equal=0.99):
    """The kernel's dx bits for rows xb, dy gb, inv against the oracle."""
    H = xb.shape[1]
    ob, exact = oracle.rows_in_threads(lambda a, b, c: oracle.mxnorm_bwd_ste(a, b, c, with_f64=True), xb, gb, inv)
    nonfin = (ob & 0x7F80) == 0x7F80
    assert np.array_equal(nonfin, (got_b & 0x7F80) == 0x7F80), "Inf/NaN pattern of dx differs"
    inf = nonfin & ((ob & 0x7F) == 0)
    assert np.array_equal(inf, nonfin & ((got_b & 0x7F) == 0)), "Inf against NaN"
    assert np.array_equal(got_b[inf], ob[inf]), "sign of an Inf differs"
    got = synth.bf16_bits_to_f32(got_b).astype(np.float64)
    xv = synth.bf16_bits_to_f32(xb).astype(np.float64)
    gv = synth.bf16_bits_to_f32(gb).astype(np.float64)
    r = inv.astype(np.float64)[:, None]
    fin = ~nonfin
    E = bwd_bound(xv, gv, r, exact, H)
    err = np.abs(got - exact)
    bound = 2.0 ** -8 * np.abs(exact) + (1 + 2.0 ** -8) * E + 1e-38
    assert (err[fin] <= bound[fin]).all(), f"max excess {(err - bound)[fin].max():.3e}"
    same = (got_b == ob).mean()
    assert same >= min_equal, f"only {same:.4f} of dx bit-equal to the oracle's rounding"


def check_bwd(xb, gb, inv, min_equal=0.99):
    dx = mx.bwd_ste(dev_bf16(xb), dev_bf16(gb), torch.from_numpy(inv).cuda())
    torch.cuda.synchronize()
    dxb = dx.view(torch.int16).cpu().numpy().view(np.uint16)
    compare_bwd(dxb, xb, gb, inv, min_equal)
    return dxb


@pytest.mark.parametrize("T,H", [(64, 256), (13, 800), (5, 4128), (100, 4096), (7, 8192), (9, 768), (3, 32)])
def test_bwd_ragged_shapes(T, H):
    xb = synth.make_random_rows(T, H, seed=T + H, scale=2.0)
    gb = synth.make_random_rows(T, H, seed=T * H + 1)
    _, _, inv = oracle.mxnorm_quant(xb, 2, "mxfp8")
    check_bwd(xb, gb, inv)


@pytest.mark.parametrize("name,rows", [("llama3_1b_32768x2048", 2048), ("llama3_8b_65536x4096", 1024)])
def test_bwd_workloads(name, rows):
    w = synth.WORKLOADS[name]
    xb = synth.make_activations(w, rows=rows)
    gb = synth.make_random_rows(rows, w.H, seed=w.seed + 100)
    for p in (1, 2):
        _, _, inv = oracle.mxnorm_quant(xb, p, "mxfp8")
        check_bwd(xb, gb, inv)


def test_bwd_full_size_every_row():
    """65536 x 4096 (the benchmark's launch) with the forward's estimates,
    every row against the oracle, checked in slices of 8192 rows."""
    w = synth.WORKLOADS["llama3_8b_65536x4096"]
    xb = synth.make_activations(w)
    gb = synth.make_random_rows(w.T, w.H, seed=77)
    _, _, inv = oracle.rows_in_threads(lambda a: oracle.mxnorm_quant(a, 2, "mxfp8"), xb)
    dx = mx.bwd_ste(dev_bf16(xb), dev_bf16(gb), torch.from_numpy(inv).cuda())
    torch.cuda.synchronize()
    dxb = dx.view(torch.int16).cpu().numpy().view(np.uint16)
    del dx
    for r0 in range(0, w.T, 8192):
        sl = slice(r0, r0 + 8192)
        compare_bwd(dxb[sl], xb[sl], gb[sl], inv[sl])


def test_bwd_with_exact_rms_is_orthogonal_to_x():
    """With the exact 1/RMS the kernel's dx is orthogonal to x (RMSNorm is
    scale invariant), to within its rounding."""
    xb = synth.make_random_rows(32, 2048, seed=3)
    gb = synth.make_random_rows(32, 2048, seed=4)
    xv = synth.bf16_bits_to_f32(xb).astype(np.float64)
    inv = (1.0 / np.sqrt((xv ** 2).mean(1))).astype(np.float32)
    dx = mx.bwd_ste(dev_bf16(xb), dev_bf16(gb), torch.from_numpy(inv).cuda())
    torch.cuda.synchronize()
    d = synth.bf16_bits_to_f32(dx.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    assert (np.abs((d * xv).sum(1)) <= 2.0 ** -7 * (np.abs(d) * np.abs(xv)).sum(1)).all()


def test_bwd_empty():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    dx = mx.bwd_ste(x, x.clone(), torch.empty((0,), dtype=torch.float32, device="cuda"))
    assert dx.shape == (0, 256)


def extreme_rows(H, seed):
    """Rows at the ends of the forward's range, with their estimates far
    from 1: ordinary rows scaled by 2^-100, 2^-60, 2^-40, 2^50 and 2^60, an
    all-zero row (inv_rms = 2^127), a row of bf16 subnormals (also 2^127)
    and a row of tiny normals beside one subnormal element."""
    base = synth.make_random_rows(5, H, seed=seed, scale=1.5)
    v = synth.bf16_bits_to_f32(base) * np.array([2.0 ** -100, 2.0 ** -60, 2.0 ** -40, 2.0 ** 50, 2.0 ** 60],
                                                np.float32)[:, None]
    rows = list(synth.f32_to_bf16_bits(v.astype(np.float32)))
    rows.append(np.zeros(H, np.uint16))
    sub = (np.arange(H, dtype=np.uint16) * 37) % 0x7F + 1
    sub[::3] |= np.uint16(0x8000)
    rows.append(sub)
    tiny = synth.f32_to_bf16_bits((synth.bf16_bits_to_f32(base[0]) * np.float32(2.0 ** -120)).astype(np.float32))
    tiny[5] = 0x0003
    rows.append(tiny)
    return np.stack(rows)


@pytest.mark.parametrize("H", [256, 800, 4096])
@pytest.mark.parametrize("p", [1, 2])
@pytest.mark.parametrize("dy_scale", [1.0, 2.0 ** -60, 2.0 ** 60])
def test_bwd_extreme_rows(H, p, dy_scale):
    """The forward's estimate at the ends of its range (inv_rms up to 2^127
    for zero and subnormal rows, down to 2^-60): rho~^3 alone leaves fp32
    there, the kernel's grouping keeps every intermediate in range, and dx
    matches the oracle within the bound, Inf where 2^127 dy overflows bf16."""
    xb = extreme_rows(H, seed=H + p)
    T = xb.shape[0]
    g = synth.bf16_bits_to_f32(synth.make_random_rows(T, H, seed=H * 3 + p)) * np.float32(dy_scale)
    gb = synth.f32_to_bf16_bits(g.astype(np.float32))
    _, _, inv = oracle.mxnorm_quant(xb, p, "mxfp8")
    assert inv[5] == np.float32(2.0 ** 127) and inv[6] == np.float32(2.0 ** 127)
    assert inv[4] < 2.0 ** -50 and inv[0] > 2.0 ** 90
    # the all-zero row scales dy by 2^127 exactly: Inf in bf16 beyond 2 |dy|
    check_bwd(xb, gb, inv, min_equal=0.98)


def test_bwd_outputs_stay_in_bounds():
    """Guard elements around dx survive the call, on ragged shapes (the
    generic-H path, one partial chunk, the 4096 fast path)."""
    g = 4096
    for T, H in ((13, 800), (3, 32), (9, 4096)):
        xb = synth.make_random_rows(T, H, seed=T + H, scale=2.0)
        gb = synth.make_random_rows(T, H, seed=T * H)
        _, _, inv = oracle.mxnorm_quant(xb, 2, "mxfp8")
        buf = torch.full((T * H + 2 * g,), 3.0, dtype=torch.bfloat16, device="cuda")
        dx = mx.bwd_ste(dev_bf16(xb), dev_bf16(gb), torch.from_numpy(inv).cuda(), out=buf[g:g + T * H])
        torch.cuda.synchronize()
        assert (buf[:g] == 3.0).all() and (buf[-g:] == 3.0).all(), (T, H)
        compare_bwd(dx.view(torch.int16).cpu().numpy().view(np.uint16).reshape(T, H), xb, gb, inv)
