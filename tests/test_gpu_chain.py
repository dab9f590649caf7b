"""Kernels launched back to back on one stream, each reading what the one
before it wrote.  The streaming kernels are launched so that the next one
may be scheduled while its predecessor finishes; each waits for the
predecessor's completion before it touches memory.  A chain whose buffers
are poisoned (NaN) before every pass must give exactly the outputs of the
same chain with a synchronisation between kernels -- launched directly and
replayed as a CUDA graph."""
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


def chain(x, dy, bufs, stream, sync_each=False):
    """quant_fwd writes inv_rms -> bwd_ste reads it and writes dx ->
    quant_fwd of dx (MXFP8+H16) -> the two-pass baseline on dx (its second
    kernel reads the first one's y)."""
    inv, codes, scales, dx, c2, s2, i2, y3, c3, s3, i3 = bufs
    for t in (inv, i2, i3):
        t.fill_(float("nan"))
    dx.fill_(float("nan"))
    y3.fill_(float("nan"))
    steps = [
        lambda: mx.quant_fwd(x, 2, "mxfp8", out=(codes, scales, inv), stream=stream),
        lambda: mx.bwd_ste(x, dy, inv, out=dx, stream=stream),
        lambda: mx.quant_fwd(dx, 1, "mxfp8_h16", out=(c2, s2, i2), stream=stream),
        lambda: mx.rmsnorm_mxfp8_ref_fwd(dx, 1e-5, out=(y3, c3, s3, i3), stream=stream),
    ]
    for f in steps:
        f()
        if sync_each:
            torch.cuda.synchronize()


@pytest.mark.parametrize("T,H", [(8192, 4096), (16384, 768), (4096, 2048)])
def test_dependent_launches_back_to_back(T, H):
    xb = synth.make_random_rows(T, H, seed=T + H, scale=2.0)
    gb = synth.make_random_rows(T, H, seed=T * 3 + H)
    x, dy = dev(xb), dev(gb)

    def alloc():
        return (torch.empty((T,), dtype=torch.float32, device="cuda"),
                torch.empty((T, H), dtype=torch.uint8, device="cuda"),
                torch.empty((T, H // 32), dtype=torch.uint8, device="cuda"),
                torch.empty((T, H), dtype=torch.bfloat16, device="cuda"),
                torch.empty((T, H), dtype=torch.uint8, device="cuda"),
                torch.empty((T, H // 32), dtype=torch.uint8, device="cuda"),
                torch.empty((T,), dtype=torch.float32, device="cuda"),
                torch.empty((T, H), dtype=torch.bfloat16, device="cuda"),
                torch.empty((T, H), dtype=torch.uint8, device="cuda"),
                torch.empty((T, H // 32), dtype=torch.uint8, device="cuda"),
                torch.empty((T,), dtype=torch.float32, device="cuda"))

    ref = alloc()
    chain(x, dy, ref, torch.cuda.current_stream(), sync_each=True)
    torch.cuda.synchronize()
    assert not torch.isnan(ref[3].float()).any()
    # the first link against the oracle (the rest follow from it bit for bit)
    oc, os_, oi = oracle.rows_in_threads(lambda a: oracle.mxnorm_quant(a, 2, "mxfp8"), xb)
    assert np.array_equal(ref[1].cpu().numpy(), oc) and np.array_equal(ref[2].cpu().numpy(), os_)

    s = torch.cuda.Stream()
    got = alloc()
    with torch.cuda.stream(s):
        for _ in range(4):
            chain(x, dy, got, s)
    torch.cuda.synchronize()
    for a, b in zip(ref, got):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))

    g_bufs = alloc()
    with torch.cuda.stream(s):
        chain(x, dy, g_bufs, s)  # warm the launch-shape caches before capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        chain(x, dy, g_bufs, s)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, g_bufs):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert mx.device_errors() == 0
