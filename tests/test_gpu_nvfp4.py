"""Parity of the NVFP4 MXNorm kernel (mxnorm_quant_fwd_nvfp4, through the C
ABI) with the CPU oracle: codes and UE4M3 scales bit-exact, inv_rms within
1e-6 relative (the kernel's sum of s_k^p is exact; its fp32 mean, root and
division by g add at most 4 roundings of 2^-24, the oracle's one more)."""
import numpy as np
import pytest
import torch

import oracle
import mx_scale_reusing_gb300 as mx
from mx_scale_reusing_gb300 import synth

pytestmark = pytest.mark.gpu


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


def check(xb, p, g, rows=None):
    c, s, i = mx.quant_fwd_nvfp4(dev(xb), p, g)
    torch.cuda.synchronize()
    c, s, i = c.cpu().numpy(), s.cpu().numpy(), i.cpu().numpy()
    rows = np.arange(xb.shape[0]) if rows is None else np.asarray(rows)
    oc, os_, oi = oracle.nvfp4_quant(xb[rows], p, g)
    assert np.array_equal(c[rows], oc), "codes differ"
    assert np.array_equal(s[rows], os_), "scales differ"
    gi, wi = i[rows].astype(np.float64), oi.astype(np.float64)
    assert (np.isnan(gi) == np.isnan(wi)).all() and (np.isinf(gi) == np.isinf(wi)).all()
    fin = np.isfinite(wi)
    assert (np.abs(gi[fin] / wi[fin] - 1) <= 1e-6).all()
    return c, s, i


@pytest.mark.parametrize("T,H", [(64, 256), (3, 16), (5, 48), (13, 800), (9, 768), (7, 4112), (100, 4096), (4, 8192)])
@pytest.mark.parametrize("g", [1.0, 3.1e-3, 7.7e-6])
@pytest.mark.parametrize("p", [1, 2])
def test_nvfp4_shapes(T, H, g, p):
    xb = synth.make_random_rows(T, H, seed=T * H + 3, scale=2.0)
    check(xb, p, float(np.float32(g)))


def test_nvfp4_special_rows():
    H = 256
    rows = [np.zeros(H, np.uint16), np.full(H, 0x8000, np.uint16),
            synth.f32_to_bf16_bits(np.full(H, 6.0, np.float32)),
            synth.f32_to_bf16_bits(np.full(H, 5000.0, np.float32)),        # saturating scale
            synth.f32_to_bf16_bits(np.full(H, -1e-30, np.float32)),        # scale underflows to 0
            np.arange(H, dtype=np.uint16) % 0x7F + 1]                      # subnormals
    r = synth.make_random_rows(1, H, 5)[0]
    r[40] = 0x7F80
    rows.append(r)
    r = synth.make_random_rows(1, H, 6)[0]
    r[3] = 0xFFC1
    rows.append(r)
    xb = np.stack(rows)
    for p in (1, 2):
        c, s, i = check(xb, p, 1.0)
    assert np.isinf(i[0]) and np.isnan(i[-1]) and np.isnan(i[-2])


@pytest.mark.parametrize("p", [1, 2])
def test_nvfp4_full_size_sampled(p):
    w = synth.WORKLOADS["llama3_8b_65536x4096"]
    xb = synth.make_activations(w)
    x = dev(xb)
    amax = float(mx.absmax(x).item())
    assert amax == float(np.abs(synth.bf16_bits_to_f32(xb)).max())
    g = mx.nvfp4_tensor_scale(x)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([np.arange(16), np.arange(w.T - 16, w.T), rng.integers(0, w.T, 128)]))
    check(xb, p, g, rows)


def test_absmax_helper():
    xb = synth.make_random_rows(33, 1000, seed=1)
    xb[7, 999] = 0xC700        # -32768
    got = float(mx.absmax(dev(xb)).item())
    assert got == float(np.abs(synth.bf16_bits_to_f32(xb)).max()) == 32768.0
    xb[3, 3] = 0x7FC0
    assert np.isnan(float(mx.absmax(dev(xb)).item()))
