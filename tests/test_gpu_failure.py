"""Failure detection on the GPU without a fault: the tiled kernel's bounded
pipeline waits are made to run out, through the drill entry point
(mxnorm_tiled_wait_drill), which withholds one tile's bulk copy and shortens
the wait limit.  The call must return within a bound, report the expiry in
bit 0 of the device error word, leave every row it could process correct,
and leave the context usable: the next normal launch is exact and clean."""
import time

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


def inv_close(got, want):
    """inv_rms within the estimator's 1e-6 relative tolerance."""
    return bool((np.abs(got.astype(np.float64) / want.astype(np.float64) - 1.0) <= 1e-6).all())


@pytest.mark.parametrize("T,H,withheld", [(4096, 4096, 0), (4096, 4096, 311), (1000, 768, 124)])
def test_tiled_wait_expires_and_is_reported(T, H, withheld):
    xb = synth.make_activations(synth.WORKLOADS["llama3_8b_65536x4096"], rows=T)[:, :H].copy()
    x = dev(xb)
    oc, os_, oi = oracle.rows_in_threads(lambda a: oracle.mxnorm_quant(a, 2, "mxfp8"), xb)
    mx.device_errors(clear=True)
    assert mx.device_errors() == 0
    out = (torch.full((T, H), 0xA5, dtype=torch.uint8, device="cuda"),
           torch.full((T, H // 32), 0xA5, dtype=torch.uint8, device="cuda"),
           torch.full((T,), -7.0, dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    c, s, i = mx.tiled_wait_drill(x, withheld_tile=withheld, wait_limit_ns=2_000_000, out=out)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 0.5, f"the drill took {elapsed:.3f} s"
    assert mx.device_errors(clear=False) & 1 == 1
    c, s, i = c.cpu().numpy(), s.cpu().numpy(), i.cpu().numpy()
    untouched = (i == -7.0) & (c == 0xA5).all(1)
    tile_rows = np.arange(withheld * 8, min(T, withheld * 8 + 8))
    assert untouched[tile_rows].all(), "rows of the withheld tile were written"
    done = ~untouched
    assert np.array_equal(c[done], oc[done]) and np.array_equal(s[done], os_[done])
    assert inv_close(i[done], oi[done])
    # the word clears, and the context is usable: a normal tiled launch is exact and clean
    mx.device_errors(clear=True)
    assert mx.device_errors() == 0
    c2, s2, i2 = mx.quant_fwd(x, 2, "mxfp8", "tiled_tma")
    torch.cuda.synchronize()
    assert np.array_equal(c2.cpu().numpy(), oc) and np.array_equal(s2.cpu().numpy(), os_)
    assert inv_close(i2.cpu().numpy(), oi)
    assert mx.device_errors() == 0


def test_drill_rejects_bad_arguments():
    x = dev(synth.make_random_rows(16, 256, seed=1))
    for tile, ns in ((-1, 2_000_000), (2, 2_000_000), (0, 10), (0, 2_000_000_000)):
        with pytest.raises(mx.MXNormError) as e:
            mx.tiled_wait_drill(x, withheld_tile=tile, wait_limit_ns=ns)
        assert e.value.status == 1
    assert mx.device_errors() == 0
