"""The allocation-free baseline entry point, rmsnorm_mxfp8_ref_fwd_static_ws.

It serves callers that cannot allocate device memory themselves (a host
framework owning all allocations, a latency-critical path that cannot take
cudaMalloc's synchronisation, a fixed memory budget): its workspace is a
device array built into the library.  This test calls it through the C ABI
twice in a row and checks each result against rmsnorm_mxfp8_ref_fwd with a
caller-provided workspace (same kernels, so the outputs must be identical:
codes and scales bit-exact, inv_rms equal), and that a call takes no
device memory.  Its argument checks, which need no GPU, are in the CPU
suite (test_abi.py).  Kept in a file of its own, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import mx_scale_reusing_gb300 as mx
from mx_scale_reusing_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mx_scale_reusing_gb300 import _build
    _build.build()
    lib = mx.lib()
    lib.rmsnorm_mxfp8_ref_fwd_static_ws.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                                    ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                                    ctypes.c_void_p, ctypes.c_void_p]
    lib.rmsnorm_mxfp8_ref_fwd_static_ws.restype = ctypes.c_int
    return lib


def _static_call(L, x, T, H, stream):
    codes = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    scales = torch.empty((T, H // 32), dtype=torch.uint8, device="cuda")
    inv = torch.empty((T,), dtype=torch.float32, device="cuda")
    rc = L.rmsnorm_mxfp8_ref_fwd_static_ws(x.data_ptr(), T, H, ctypes.c_float(1e-5), codes.data_ptr(),
                                           scales.data_ptr(), inv.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, L.mxnorm_last_error()
    return codes, scales, inv


def test_static_workspace_matches_caller_workspace_twice(L):
    stream = torch.cuda.current_stream()
    inputs = [synth.make_activations(synth.WORKLOADS["llama3_8b_65536x4096"], rows=2048),
              synth.make_random_rows(777, 768, seed=5, scale=4.0)]
    for xb in inputs:                       # two calls in a row, different shapes
        T, H = xb.shape
        x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        c, s, i = _static_call(L, x, T, H, stream)
        _, rc, rs, ri = mx.rmsnorm_mxfp8_ref_fwd(x, eps=1e-5)
        torch.cuda.synchronize()
        assert torch.equal(c, rc) and torch.equal(s, rs)
        assert torch.equal(i, ri)


def test_static_workspace_call_takes_no_device_memory(L):
    """After a first call (which may load the module), further calls leave
    the device's free memory unchanged: the outputs are allocated before the
    first reading, and the call itself allocates nothing."""
    stream = torch.cuda.current_stream()
    xb = synth.make_random_rows(2048, 4096, seed=6, scale=2.0)
    T, H = xb.shape
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    codes = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    scales = torch.empty((T, H // 32), dtype=torch.uint8, device="cuda")
    inv = torch.empty((T,), dtype=torch.float32, device="cuda")

    def call():
        rc = L.rmsnorm_mxfp8_ref_fwd_static_ws(x.data_ptr(), T, H, ctypes.c_float(1e-5), codes.data_ptr(),
                                               scales.data_ptr(), inv.data_ptr(),
                                               ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, L.mxnorm_last_error()

    call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
