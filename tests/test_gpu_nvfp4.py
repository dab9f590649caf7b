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
    oc, os_, oi = oracle.rows_in_threads(lambda a: oracle.nvfp4_quant(a, p, g), np.ascontiguousarray(xb[rows]))
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
def test_nvfp4_full_size_every_row(p):
    """65536 x 4096, the launch the benchmark times: every row against the
    oracle, with the tensor scale the library derives on the device."""
    w = synth.WORKLOADS["llama3_8b_65536x4096"]
    xb = synth.make_activations(w)
    x = dev(xb)
    amax = float(mx.absmax(x).item())
    assert amax == float(np.abs(synth.bf16_bits_to_f32(xb)).max())
    g = mx.nvfp4_tensor_scale(x)
    assert g.item() == oracle.nvfp4_tensor_scale(xb)
    c, s, i = mx.quant_fwd_nvfp4(x, p)   # the scale derived and read on the device
    torch.cuda.synchronize()
    c2, s2, i2 = check(xb, p, g.item())  # the same scale by value, every row against the oracle
    assert np.array_equal(c.cpu().numpy(), c2) and np.array_equal(s.cpu().numpy(), s2)
    assert np.array_equal(i.cpu().numpy(), i2)


def tie_case_rows(H):
    """The hand-derived cases that fix the recipe's rounding steps (each a
    16-element block, repeated along rows of H): (x, g, expected byte 0 of
    the codes, expected scale code).
      * RN(x * RN(1/g)) against RN(x / g) on either side of an E2M1 tie:
        x = 3 with g = 0.85714293 gives the tie 3.5 -> 4 (low nibble 0x6);
        x = 3.25 with g = 4.3333335 gives 0.74999994 -> 0.5 (0x1);
      * sb = RN(amax / RN(6 g)) with amax 1, g = 0.10666666: the E4M3 tie
        1.5625 -> scale 1.5 (0x3C) (the exact 6 g would give 0x3D);
      * enc = RN(1 / RN(s g)), s = 1.125 (amax 2.4375), g = 0.36111107,
        x = 0.5078125: the E2M1 tie 1.25 -> 1.0 (0x2) (exact s g: 0x3).
    The block maximum 6 g (rounded to bf16) puts the first two cases' scale
    at 1.0 (0x38) and encodes as 6 (high nibble 0x7)."""
    cases = []
    for x, g, lo in ((3.0, 0.8571429252624512, 0x6), (3.25, 4.333333492279053, 0x1)):
        amax = float(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.array([6.0 * g], np.float32)))[0])
        blk = np.zeros(16, np.float32)
        blk[0], blk[1] = x, amax
        cases.append((blk, g, 0x70 | lo, 0x38))
    blk = np.zeros(16, np.float32)
    blk[3] = 1.0
    cases.append((blk, 0.10666666179895401, None, 0x3C))
    blk = np.zeros(16, np.float32)
    blk[0], blk[1] = 0.5078125, 2.4375
    cases.append((blk, 0.3611110746860504, 0x72, 0x39))
    return [(synth.f32_to_bf16_bits(np.tile(b, (3, H // 16))), g, c0, sc) for b, g, c0, sc in cases]


@pytest.mark.parametrize("H", [16, 4096, 800])
@pytest.mark.parametrize("p", [1, 2])
def test_nvfp4_tie_cases_on_the_gpu(H, p):
    """The four hand-derived tie cases of the recipe's rounding steps through
    the kernel: bit-exact against the oracle and against the codes derived
    by hand (rows of one block, of the 4096-element fast path, and of a
    ragged 800-element row)."""
    for xb, g, code0, scale in tie_case_rows(H):
        c, s, _ = check(xb, p, float(np.float32(g)))
        assert (s == scale).all()
        if code0 is not None:
            assert (c[:, ::8] == code0).all()


def test_nvfp4_device_tensor_scale_closed_forms():
    """The library's device-side tensor scale against the oracle's and the
    closed forms: a = 2688 * 2^j gives 2^j exactly, Inf/NaN are skipped, an
    all-zero tensor gives 1."""
    for j in (-30, 0, 7):
        xb = synth.make_random_rows(5, 96, seed=j + 40)
        xb[2, 17] = synth.f32_to_bf16_bits(np.array([-2688.0 * 2.0 ** j], np.float32))[0]
        xb[:, :] = np.where(np.abs(synth.bf16_bits_to_f32(xb)) > 2688.0 * 2.0 ** j,
                            np.uint16(0), xb)
        assert mx.nvfp4_tensor_scale(dev(xb)).item() == 2.0 ** j == oracle.nvfp4_tensor_scale(xb)
    xb = synth.make_random_rows(7, 160, seed=9, scale=50.0)
    xb[3, 3], xb[4, 4], xb[5, 5] = 0x7F80, 0xFFC1, 0xFF80
    assert mx.nvfp4_tensor_scale(dev(xb)).item() == oracle.nvfp4_tensor_scale(xb)
    assert mx.nvfp4_tensor_scale(dev(np.zeros((2, 64), np.uint16))).item() == 1.0
    assert mx.device_errors() == 0


def test_nvfp4_bad_device_tensor_scale_sets_the_error_bit():
    """A device tensor scale that is not a finite positive float: the call
    returns, bit 2 of the device error word is set, and clearing it leaves
    the next call clean."""
    xb = synth.make_random_rows(8, 256, seed=5)
    mx.device_errors(clear=True)
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        mx.quant_fwd_nvfp4(dev(xb), 2, torch.tensor([bad], dtype=torch.float32, device="cuda"))
        torch.cuda.synchronize()
        assert mx.device_errors(clear=True) == 4, bad
    check(xb, 2, 1.0)
    assert mx.device_errors() == 0


def test_absmax_helper():
    xb = synth.make_random_rows(33, 1000, seed=1)
    xb[7, 999] = 0xC700        # -32768
    got = float(mx.absmax(dev(xb)).item())
    assert got == float(np.abs(synth.bf16_bits_to_f32(xb)).max()) == 32768.0
    xb[3, 3] = 0x7FC0
    assert np.isnan(float(mx.absmax(dev(xb)).item()))


def test_nvfp4_outputs_stay_in_bounds():
    """Guard bytes around the codes, scales and inv_rms buffers survive the
    call, on ragged shapes (one partial chunk, a generic row length)."""
    g = 4096
    for T, H in ((37, 800), (5, 16), (9, 4096)):
        xb = synth.make_random_rows(T, H, seed=T + H, scale=3.0)
        codes = torch.full((T * H // 2 + 2 * g,), 0xA5, dtype=torch.uint8, device="cuda")
        scales = torch.full((T * H // 16 + 2 * g,), 0x5A, dtype=torch.uint8, device="cuda")
        inv = torch.full((T + 2 * g,), 7.0, dtype=torch.float32, device="cuda")
        out = (codes[g:g + T * H // 2], scales[g:g + T * H // 16], inv[g:g + T])
        mx.quant_fwd_nvfp4(dev(xb), 2, 0.01, out=out)
        torch.cuda.synchronize()
        for buf, fill in ((codes, 0xA5), (scales, 0x5A), (inv, 7.0)):
            assert (buf[:g] == fill).all() and (buf[-g:] == fill).all(), (T, H)
        oc, os_, oi = oracle.nvfp4_quant(xb, 2, float(np.float32(0.01)))
        assert np.array_equal(out[0].cpu().numpy().reshape(T, -1), oc)
        assert np.array_equal(out[1].cpu().numpy().reshape(T, -1), os_)
