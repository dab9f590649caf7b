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


@pytest.mark.parametrize("T,K,N", [(128, 128, 256), (200, 256, 512), (1000, 768, 768), (131, 4096, 256),
                                   (77, 384, 256), (260, 1152, 512), (129, 640, 256)])
def test_linear_small(T, K, N):
    """K stage counts of 1 to 32, odd and even: the producer loads the scale
    atoms of 1, 2 or 4 stages per copy, whichever divides the count."""
    linear_case(T, K, N, seed=T + K + N)


@pytest.mark.parametrize("K", [768, 1152])
def test_linear_many_tiles_scale_groups_of_2_and_1(K):
    """Many tiles per CTA pair with scale atoms loaded 2 (K = 768) or 1
    (K = 1152) stages per copy, so the scale-group ring wraps across tile
    boundaries many times; sampled rows of every row tile."""
    T = 8192 + 77
    rows = np.unique(np.concatenate([np.arange(0, T, 257), np.arange(T - 4, T)]))
    linear_case(T, K, 2048, seed=K, rows=rows)


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


# ------------------------------------------------ gain-folded weight cast
def gains(K, seed):
    """Norm gains around 1 with both signs, exact zeros of both signs and a
    subnormal, as float32."""
    rng = np.random.default_rng(seed)
    g = (np.exp(rng.normal(0.0, 0.6, K)) * rng.choice([-1.0, 1.0], K, p=[0.1, 0.9])).astype(np.float32)
    g[[0, K // 2]] = [0.0, -0.0]
    g[K - 1] = np.float32(2.0e-39)
    return g


def check_gain_cast(wb, g, c, layout, w_dev=None, rows=None):
    w = dev(wb) if w_dev is None else w_dev
    codes, scales = mx.mx_cast_gain(w, torch.from_numpy(g).cuda(), c, layout)
    torch.cuda.synchronize()
    N, K = wb.shape
    rows = np.arange(N) if rows is None else np.asarray(rows)
    oc, os_ = oracle.rows_in_threads(lambda a: oracle.mx_cast_gain(a, g, c), np.ascontiguousarray(wb[rows]))
    got_c = codes.cpu().numpy()
    np.testing.assert_array_equal(got_c[rows], oc)
    got_s = scales.cpu().numpy()
    if layout == "row_major":
        np.testing.assert_array_equal(got_s[rows], os_)
    else:
        full = np.zeros((N, K // 32), np.uint8)
        full[rows] = os_
        mask = to_mma_layout(np.isin(np.arange(N), rows)[:, None].repeat(K // 32, 1).astype(np.uint8)) == 1
        np.testing.assert_array_equal(got_s[mask], to_mma_layout(full)[mask])


@pytest.mark.parametrize("layout", ["row_major", "mma"])
@pytest.mark.parametrize("N,K", [(512, 768), (77, 4096), (300, 1152), (1, 128), (1029, 2560)])
def test_gain_cast_parity(N, K, layout):
    """Strips of 512 columns with a ragged last strip (768, 1152, 2560),
    row counts off the 8-warp and 128-row tiles, c != 1."""
    wb = synth.make_random_rows(N, K, seed=N + K, scale=0.03)
    check_gain_cast(wb, gains(K, N), 1.7, layout)


def test_gain_cast_short_rows_row_major():
    """K = 32 and 96: one strip, most lanes idle."""
    for K in (32, 96):
        wb = synth.make_random_rows(40, K, seed=K, scale=1.0)
        check_gain_cast(wb, gains(K, K), 0.75, "row_major")


def test_gain_cast_special_values():
    """Inf/NaN weights, gains whose product with c overflows (Inf, and NaN
    where the weight is 0), subnormal products, blocks of zeros."""
    N, K = 64, 512
    wb = synth.make_random_rows(N, K, seed=3, scale=1.0)
    wb[1, 5] = 0x7F80          # +Inf
    wb[2, 40] = 0x7FC1         # NaN
    wb[3, :32] = 0             # zero block
    wb[4, 64:96] = 0x0001      # bf16 subnormals
    wb[5, 300] = 0             # zero times an infinite gain -> NaN
    g = gains(K, 4)
    g[300] = np.float32(3.0e38)  # c * g overflows to Inf
    g[100:132] = np.float32(1.0e-30)  # products far below the fp32 normal range
    check_gain_cast(wb, g, 1.7, "row_major")
    check_gain_cast(wb, g, 1.7, "mma")


def test_gain_cast_16_byte_aligned_weight():
    """A weight only 16-byte aligned takes the 16-byte load form."""
    N, K = 96, 1024
    wb = synth.make_random_rows(N, K, seed=8, scale=0.05)
    buf = torch.empty(N * K + 8, dtype=torch.bfloat16, device="cuda")
    w = buf[8:].view(N, K)
    w.copy_(dev(wb))
    assert w.data_ptr() % 32 == 16
    check_gain_cast(wb, gains(K, 8), 1.0, "mma", w_dev=w)


@pytest.mark.parametrize("layout", ["mma", "row_major"])
def test_gain_cast_llama3_8b_gate_up_every_row(layout):
    """The Llama-3-8B fused gate/up weight (28672 x 4096), the launch the
    benchmark times: every row against the oracle, codes and scales
    bit-exact ("MXNorm ...", 2. Metodologia, Implementacion: the norm's gain
    folded into the next layer's weight)."""
    N, K = 28672, 4096
    wb = synth.make_random_rows(N, K, seed=12, scale=0.02)
    check_gain_cast(wb, gains(K, 12), 1.0, layout)


def test_linear_with_gain_folded_weight():
    """MXNormLinear end to end: activations through the fused pass (MMA
    scales), the weight through the gain-folded cast, the GEMM; against the
    oracle's chain (gain cast, then the fp64 GEMM)."""
    T, K, N = 300, 1024, 512
    xb = synth.make_random_rows(T, K, seed=21, scale=2.0)
    wb = synth.make_random_rows(N, K, seed=22, scale=0.03)
    g = gains(K, 23)
    xc, xs, inv = mx.quant_fwd_mma(dev(xb))
    wc, ws = mx.mx_cast_gain(dev(wb), torch.from_numpy(g).cuda(), 1.3, "mma")
    out = mx.linear_fwd(xc, xs, inv, wc, ws)
    torch.cuda.synchronize()
    oxc, oxs, oxi = oracle.mxnorm_quant(xb, 2, "mxfp8")
    owc, ows = oracle.mx_cast_gain(wb, g, 1.3)
    np.testing.assert_array_equal(wc.cpu().numpy(), owc)
    want = oracle.mxfp8_linear(oxc, oxs, oxi, owc, ows)
    got = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - want)
    assert (err <= 2.0 ** -7 * np.abs(want) + 2.0 ** -12 * np.abs(want).max()).all()


def test_linear_matches_cublaslt_mxfp8():
    """A check that does not go through the oracle: with inv_rms = 1 the
    kernel is a plain MXFP8 block-scaled GEMM with a bf16 output, which
    cuBLASLt also computes (torch._scaled_mm with E8M0 scales, read in the
    same tensor-core scale layout).  Both accumulate in fp32 on the tensor
    cores, so they agree to the bf16 rounding of the output (bit-equal when
    the library keeps the same K order); a misread scale layout would be
    off by powers of two."""
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("this torch has no E8M0 dtype")
    T, K, N = 2048, 2048, 1024
    xb = synth.make_random_rows(T, K, seed=31, scale=2.0)
    wb = synth.make_random_rows(N, K, seed=32, scale=0.03)
    xc, xs, _ = mx.quant_fwd_mma(dev(xb))
    wc, ws = mx.mx_cast(dev(wb), "mma")
    ones = torch.ones((T,), dtype=torch.float32, device="cuda")
    ours = mx.linear_fwd(xc, xs, ones, wc, ws)
    try:
        ref = torch._scaled_mm(xc.view(torch.float8_e4m3fn), wc.view(torch.float8_e4m3fn).t(),
                               scale_a=xs.view(torch.float8_e8m0fnu), scale_b=ws.view(torch.float8_e8m0fnu),
                               out_dtype=torch.bfloat16)
    except (RuntimeError, TypeError, NotImplementedError) as e:
        pytest.skip(f"cuBLASLt MXFP8 GEMM unavailable: {e}")
    torch.cuda.synchronize()
    a, b = ours.double(), ref.double()
    assert ((a - b).abs() <= 2.0 ** -7 * b.abs() + 2.0 ** -12 * b.abs().max()).all()
    print(f"bit-equal fraction vs cuBLASLt: {(ours.view(torch.int16) == ref.view(torch.int16)).double().mean().item():.6f}")


def test_weight_cast_and_quant_layout_outputs_stay_in_bounds():
    """Guard bytes around the gain-folded cast's codes and scales (both
    layouts) and around the fused pass's MMA-layout scales survive, on
    ragged row counts (not multiples of 8 or 128)."""
    gd = 4096
    for N, K in ((77, 4096), (301, 1152), (1, 128)):
        wb = synth.make_random_rows(N, K, seed=N + K, scale=0.05)
        gam = gains(K, N)
        for layout, lid in (("row_major", 0), ("mma", 1)):
            nsc = N * K // 32 if lid == 0 else mx.mma_scale_bytes(N, K)
            codes = torch.full((N * K + 2 * gd,), 0xA5, dtype=torch.uint8, device="cuda")
            scales = torch.full((nsc + 2 * gd,), 0x5A, dtype=torch.uint8, device="cuda")
            gt, wt = torch.from_numpy(gam).cuda(), dev(wb)
            st = mx.lib().mx_cast_gain_fwd(wt.data_ptr(), N, K, gt.data_ptr(), 1.3,
                                           codes[gd:].data_ptr(), scales[gd:].data_ptr(), lid, None)
            torch.cuda.synchronize()
            assert st == 0
            assert (codes[:gd] == 0xA5).all() and (codes[gd + N * K:] == 0xA5).all(), (N, K, layout)
            assert (scales[:gd] == 0x5A).all() and (scales[gd + nsc:] == 0x5A).all(), (N, K, layout)
            oc, os_ = oracle.mx_cast_gain(wb, gam, 1.3)
            assert np.array_equal(codes[gd:gd + N * K].cpu().numpy().reshape(N, K), oc)
    for T, H in ((300, 768), (5, 4096)):
        xb = synth.make_random_rows(T, H, seed=T, scale=2.0)
        nsc = mx.mma_scale_bytes(T, H)
        codes = torch.full((T * H + 2 * gd,), 0xA5, dtype=torch.uint8, device="cuda")
        scales = torch.full((nsc + 2 * gd,), 0x5A, dtype=torch.uint8, device="cuda")
        inv = torch.full((T + 2 * gd,), 7.0, dtype=torch.float32, device="cuda")
        xt = dev(xb)
        st = mx.lib().mxnorm_quant_fwd_layout(xt.data_ptr(), T, H, 2, 0, codes[gd:].data_ptr(),
                                              scales[gd:].data_ptr(), inv[gd:].data_ptr(), 1, None)
        torch.cuda.synchronize()
        assert st == 0
        assert (codes[:gd] == 0xA5).all() and (codes[gd + T * H:] == 0xA5).all()
        assert (scales[:gd] == 0x5A).all() and (scales[gd + nsc:] == 0x5A).all()
        assert (inv[:gd] == 7.0).all() and (inv[gd + T:] == 7.0).all()
        oc, os_, oi = oracle.mxnorm_quant(xb, 2, "mxfp8")
        got = scales[gd:gd + nsc].cpu().numpy()
        mask = mma_mask(T, H // 32)
        assert np.array_equal(got[mask], to_mma_layout(os_)[mask])


def test_linear_out_stays_in_bounds():
    """Guard elements around the GEMM's output survive, with T off the
    128-row tile (a ragged last tile) and several 256-column tiles."""
    gd = 4096
    T, K, N = 300, 512, 768
    xb = synth.make_random_rows(T, K, seed=31, scale=2.0)
    wb = synth.make_random_rows(N, K, seed=32, scale=0.05)
    xc, xs, inv = mx.quant_fwd_mma(dev(xb))
    wc, ws = mx.mx_cast(dev(wb), "mma")
    buf = torch.full((T * N + 2 * gd,), 5.0, dtype=torch.bfloat16, device="cuda")
    out = mx.linear_fwd(xc, xs, inv, wc, ws, out=buf[gd:gd + T * N])
    torch.cuda.synchronize()
    assert (buf[:gd] == 5.0).all() and (buf[-gd:] == 5.0).all()
    assert mx.device_errors() == 0
    ref = mx.linear_fwd(xc, xs, inv, wc, ws)
    torch.cuda.synchronize()
    assert torch.equal(out.view(T, N), ref)
