"""The consumer side of MXNormLinear on the GPU (through the C ABI): the
MMA scale-atom layout written by the quantisers, the weight cast, and the
block-scaled tensor-core GEMM with the inv_rms epilogue against the fp64
oracle.

GEMM bound: the tensor cores accumulate in fp32; with S = sum_k |x^_k w^_k|
the accumulator is within (K/32 + 32) u S of the exact sum (u = 2^-24: one
rounding per 32-element MMA step into the accumulator, and at most 32 more
inside a step), the product with inv_rms adds u, and the bf16 output
rounding 2^-8 relative:
  |out - exact| <= 2^-8 |exact| + (1 + 2^-8) (inv (K/32 + 32) u S + u |exact|).
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


def dev(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()


def to_mma_layout(scales_rm):
    """Row-major [rows, K/32] scales -> the flat MMA atom layout (rows padded
    to 128 with zeros): atom (row tile, block group) of 512 bytes, byte of
    (r, k) at (r % 32) * 16 + ((r / 32) % 4) * 4 + k % 4."""
    rows, kb = scales_rm.shape
    rp = -(-rows // 128) * 128
    s = np.zeros((rp, kb), np.uint8)
    s[:rows] = scales_rm
    s = s.reshape(rp // 128, 4, 32, kb // 4, 4).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(s).reshape(-1)


def mma_mask(rows, kb):
    """True where a byte of the MMA layout belongs to a real row."""
    return to_mma_layout(np.ones((rows, kb), np.uint8)) == 1


@pytest.mark.parametrize("T,H", [(128, 128), (300, 768), (1000, 4096), (77, 2048)])
@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4_h16"])
def test_quant_mma_scale_layout(T, H, fmt):
    xb = synth.make_random_rows(T, H, seed=T + H, scale=2.0)
    x = dev(xb)
    c_rm, s_rm, i_rm = mx.quant_fwd(x, 2, fmt)
    c_t, s_t, i_t = mx.quant_fwd_mma(x, 2, fmt)
    torch.cuda.synchronize()
    assert torch.equal(c_rm, c_t) and torch.equal(i_rm, i_t)
    assert s_t.numel() == mx.mma_scale_bytes(T, H)
    mask = mma_mask(T, H // 32)
    got = s_t.cpu().numpy()
    np.testing.assert_array_equal(got[mask], to_mma_layout(s_rm.cpu().numpy())[mask])
    oc, os_, oi = oracle.mxnorm_quant(xb, 2, fmt)
    np.testing.assert_array_equal(got[mask], to_mma_layout(os_)[mask])


@pytest.mark.parametrize("layout", ["row_major", "mma"])
def test_weight_cast(layout):
    wb = synth.make_random_rows(512, 768, seed=5, scale=0.02)
    c, s = mx.mx_cast(dev(wb), layout)
    torch.cuda.synchronize()
    oc, os_ = oracle.mx_cast(wb, "mxfp8")
    np.testing.assert_array_equal(c.cpu().numpy(), oc)
    if layout == "row_major":
        np.testing.assert_array_equal(s.cpu().numpy(), os_)
    else:
        np.testing.assert_array_equal(s.cpu().numpy(), to_mma_layout(os_))


def linear_case(T, K, N, seed, rows=None, out_offset=0):
    if K <= 4096:
        x = synth.make_activations(synth.WORKLOADS["llama3_8b_65536x4096"], rows=T)[:, :K]
    else:
        x = synth.make_random_rows(T, K, seed=seed + 1, scale=2.0)
    xb = np.ascontiguousarray(x)
    xc, xs, inv = oracle.mxnorm_quant(xb, 2, "mxfp8")
    wb = synth.make_random_rows(N, K, seed=seed, scale=0.03)
    wc, ws = oracle.mx_cast(wb, "mxfp8")
    out = None
    if out_offset:  # an output that starts out_offset elements into its allocation
        out = torch.empty(T * N + out_offset, dtype=torch.bfloat16, device="cuda")[out_offset:].view(T, N)
    out = mx.linear_fwd(torch.from_numpy(xc).cuda(), torch.from_numpy(to_mma_layout(xs)).cuda(),
                        torch.from_numpy(inv).cuda(), torch.from_numpy(wc).cuda(),
                        torch.from_numpy(to_mma_layout(ws)).cuda(), out=out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    rows = np.arange(T) if rows is None else np.asarray(rows)
    want = oracle.mxfp8_linear(xc[rows], xs[rows], inv[rows], wc, ws)
    # S = sum_k |x^ w^| per output, for the accumulation bound
    from oracle import bruteforce as bf
    table = np.full(256, np.nan)
    for code, v in bf.e4m3_values().items():
        table[code] = float(v)
    xv = np.abs(table[xc[rows]]) * np.repeat(np.exp2(xs[rows].astype(np.float64) - 127), 32, axis=1)
    wv = np.abs(table[wc]) * np.repeat(np.exp2(ws.astype(np.float64) - 127), 32, axis=1)
    S = xv @ wv.T
    r = inv[rows].astype(np.float64)[:, None]
    bound = 2.0 ** -8 * np.abs(want) + (1 + 2.0 ** -8) * (r * (K / 32 + 32) * U * S + U * np.abs(want)) + 1e-30
    err = np.abs(got[rows] - want)
    assert (err <= bound).all(), f"max excess {(err - bound).max():.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}"
    return got, want


@pytest.mark.parametrize("T,K,N", [(128, 128, 256), (200, 256, 512), (1000, 768, 768), (131, 4096, 256)])
def test_linear_small(T, K, N):
    linear_case(T, K, N, seed=T + K + N)


def test_linear_llama3_8b_layer_sampled():
    """A Llama-3-8B projection shape (K = 4096, N = 4096) on 2048 tokens, the
    oracle on sampled rows including both ends and a ragged tail tile."""
    T = 2048 + 77
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(8), np.arange(T - 8, T), rng.integers(0, T, 24)]))
    linear_case(T, 4096, 4096, seed=9, rows=rows)


def test_linear_many_tiles_per_pair_sampled():
    """Several 256 x 256 tiles per persistent CTA pair (33 row tiles x 16
    column tiles), so the accumulator hand-off between the pair's epilogue
    and its MMA issuer runs through many phases; sampled rows of every row
    tile, the ragged last one included."""
    T = 8192 + 77
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([np.arange(0, T, 251), np.arange(T - 4, T), rng.integers(0, T, 8)]))
    linear_case(T, 1024, 4096, seed=11, rows=rows)


def test_linear_long_k():
    """K = 8192: 64 K stages per tile, so the 6-deep stage ring and its
    TMEM scale slots wrap many times inside one accumulation."""
    linear_case(300, 8192, 512, seed=13)


def test_linear_out_16_byte_aligned():
    """An output only 16-byte aligned (the API's minimum) takes the 16-byte
    store form of the epilogue."""
    linear_case(384, 256, 512, seed=5, out_offset=8)


def test_linear_no_device_error_flag():
    linear_case(256, 512, 256, seed=1)
    assert mx.device_errors() == 0
