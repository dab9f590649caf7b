"""Parity of the straight-through backward kernel (mxnorm_bwd_ste, through
the C ABI) with the CPU oracle.

The oracle evaluates dx = r dy - r^3 x (1/H) sum(dy x) exactly in fp64; the
kernel in fp32.  Bound per element (u = 2^-24, L = fp32 summation depth of
the dot product: log2 VEC + chunks + 5): the dot's error is at most
L u sum|dy x|, which reaches dx_j through (r^3 / H)|x_j|; r^3 and k take
four more roundings (5 u |k x_j| with the fma's), r dy_j one, the fma one
more (2 u r|dy_j|).  With the final bf16 rounding:
  |dx_gpu - dx_exact| <= 2^-8 |dx_exact| + (1 + 2^-8) E_j.
"""
import numpy as np
import pytest
import torch

import oracle
import mx_scale_reusing_gb300 as mx
from mx_scale_reusing_gb300 import synth

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


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


def check_bwd(xb, gb, inv, rows=None):
    T, H = xb.shape
    dx = mx.bwd_ste(dev_bf16(xb), dev_bf16(gb), torch.from_numpy(inv).cuda())
    torch.cuda.synchronize()
    got = synth.bf16_bits_to_f32(dx.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    rows = np.arange(T) if rows is None else np.asarray(rows)
    ob, exact = oracle.mxnorm_bwd_ste(xb[rows], gb[rows], inv[rows], with_f64=True)
    xv = synth.bf16_bits_to_f32(xb[rows]).astype(np.float64)
    gv = synth.bf16_bits_to_f32(gb[rows]).astype(np.float64)
    r = inv[rows].astype(np.float64)[:, None]
    dot = (xv * gv).sum(1, keepdims=True)
    S = np.abs(xv * gv).sum(1, keepdims=True)
    k = r ** 3 * dot / H
    vec = 16 if H % 512 == 0 else 8
    L = int(np.log2(vec)) + -(-H // (32 * vec)) + 5
    E = U * (2 * r * np.abs(gv) + 5 * np.abs(k * xv)) + (r ** 3 / H) * np.abs(xv) * L * U * S
    err = np.abs(got[rows] - exact)
    bound = 2.0 ** -8 * np.abs(exact) + (1 + 2.0 ** -8) * E + 1e-38
    assert (err <= bound).all(), f"max excess {(err - bound).max():.3e}"
    same = (dx.view(torch.int16).cpu().numpy().view(np.uint16)[rows] == ob).mean()
    assert same > 0.99, f"only {same:.4f} of dx bit-equal to the oracle's rounding"


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


def test_bwd_full_size_sampled():
    """65536 x 4096 (the benchmark's launch), oracle on sampled rows."""
    w = synth.WORKLOADS["llama3_8b_65536x4096"]
    xb = synth.make_activations(w)
    gb = synth.make_random_rows(w.T, w.H, seed=77)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([np.arange(16), np.arange(w.T - 16, w.T), rng.integers(0, w.T, 96)]))
    inv = np.zeros(w.T, np.float32)
    _, _, inv_rows = oracle.mxnorm_quant(xb[rows], 2, "mxfp8")
    inv[rows] = inv_rows
    inv[inv == 0] = 1.0
    check_bwd(xb, gb, inv, rows)


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
