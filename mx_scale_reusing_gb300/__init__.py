"""libmxnorm Python binding: argument marshalling over the C ABI.

Every step of the computation runs in the CUDA library (libmxnorm.so, built
in-tree by ``mx_scale_reusing_gb300._build``); this module only checks
tensors, allocates outputs with torch and passes raw device pointers plus the
current CUDA stream.  There is no CPU fallback: without the built library
every call raises ``MXNormLibraryMissing``.

Method: "MXNorm: Reusing MXFP block scales for efficient tensor
normalisation", Resumen tecnico, 2. Metodologia ("Fundamentos Teoricos":
inverse RMS from the power mean of the MX block scales; "Implementacion":
one fused pass).  The function names follow the C ABI in include/mxnorm.h.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "FMT", "VARIANT", "MXNormError", "MXNormLibraryMissing", "lib", "library_path",
    "mxnorm_quant_fwd", "quant_fwd", "quant_fwd_host", "rmsnorm_mxfp8_ref_fwd", "device_errors",
    "code_bytes", "bwd_ste", "quant_fwd_nvfp4", "absmax", "nvfp4_tensor_scale", "quant_fwd_mma", "mx_cast",
    "linear_fwd", "mma_scale_bytes", "tiled_wait_drill",
]

FMT = {"mxfp8": 0, "mxfp4": 1, "mxfp4_h16": 2, "mxfp8_h16": 3, "mxfp4_h32": 4, "mxfp8_h32": 5}
VARIANT = {"auto": 0, "warp_row": 1, "tiled_tma": 2}
STATUS = {0: "MXNORM_OK", 1: "MXNORM_ERR_INVALID_ARG", 2: "MXNORM_ERR_UNSUPPORTED",
          3: "MXNORM_ERR_MISALIGNED", 4: "MXNORM_ERR_CUDA"}

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libmxnorm.so")
_lib = None


class MXNormLibraryMissing(RuntimeError):
    """libmxnorm.so is not built: every call raises this (there is no CPU
    fallback)."""


class MXNormError(RuntimeError):
    """A C-ABI call returned a non-zero mxnorm_status; `status` holds it and
    the message is the library's mxnorm_last_error() text."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded C library (raises MXNormLibraryMissing if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise MXNormLibraryMissing(
            f"{library_path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(library_path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.mxnorm_quant_fwd.argtypes = [vp, i64, i64, i32, i32, vp, vp, vp, vp]
    L.mxnorm_quant_fwd.restype = i32
    L.mxnorm_quant_fwd_ex.argtypes = [vp, i64, i64, i32, i32, vp, vp, vp, i32, vp]
    L.mxnorm_quant_fwd_ex.restype = i32
    L.rmsnorm_mxfp8_ref_fwd.argtypes = [vp, i64, i64, ctypes.c_float, vp, vp, vp, vp, vp]
    L.rmsnorm_mxfp8_ref_fwd.restype = i32
    L.mxnorm_status_string.argtypes = [i32]
    L.mxnorm_status_string.restype = ctypes.c_char_p
    L.mxnorm_last_error.argtypes = []
    L.mxnorm_last_error.restype = ctypes.c_char_p
    L.mxnorm_abi_version.restype = i32
    L.mxnorm_quant_fwd_nvfp4.argtypes = [vp, i64, i64, i32, ctypes.c_float, vp, vp, vp, vp]
    L.mxnorm_quant_fwd_nvfp4.restype = i32
    L.mxnorm_absmax_bf16.argtypes = [vp, i64, vp, vp]
    L.mxnorm_absmax_bf16.restype = i32
    L.mxnorm_quant_fwd_nvfp4_dev.argtypes = [vp, i64, i64, i32, vp, vp, vp, vp, vp]
    L.mxnorm_quant_fwd_nvfp4_dev.restype = i32
    L.mxnorm_nvfp4_tensor_scale.argtypes = [vp, i64, vp, vp]
    L.mxnorm_nvfp4_tensor_scale.restype = i32
    L.mxnorm_bwd_ste.argtypes = [vp, vp, vp, i64, i64, vp, vp]
    L.mxnorm_mma_scale_bytes.argtypes = [i64, i64]
    L.mxnorm_mma_scale_bytes.restype = i64
    L.mxnorm_quant_fwd_layout.argtypes = [vp, i64, i64, i32, i32, vp, vp, vp, i32, vp]
    L.mxnorm_quant_fwd_layout.restype = i32
    L.mx_cast_fwd.argtypes = [vp, i64, i64, i32, vp, vp, i32, vp]
    L.mx_cast_fwd.restype = i32
    L.mx_cast_gain_fwd.argtypes = [vp, i64, i64, vp, ctypes.c_float, vp, vp, i32, vp]
    L.mx_cast_gain_fwd.restype = i32
    L.mxnorm_linear_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, vp, vp]
    L.mxnorm_linear_fwd.restype = i32
    L.mxnorm_bwd_ste.restype = i32
    L.mxnorm_tiled_wait_drill.argtypes = [vp, i64, i64, vp, vp, vp, i64, i64, vp]
    L.mxnorm_tiled_wait_drill.restype = i32
    L.mxnorm_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
    L.mxnorm_device_errors.restype = i32
    _lib = L
    return L


def _check(status: int):
    if status != 0:
        raise MXNormError(status, lib().mxnorm_last_error().decode())


def code_bytes(H: int, fmt: str) -> int:
    """Bytes of codes per row of H elements: one per E4M3 code, one per two
    E2M1 codes."""
    return H if fmt.startswith("mxfp8") else H // 2


def _stream_ptr(device, stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _require(t, name: str, device, dtype=None, min_numel: int = 0, byte_elems: bool = False):
    """Raise ValueError unless t is a contiguous CUDA tensor on `device` with
    dtype `dtype` (or 1-byte elements when byte_elems) and at least
    min_numel elements: the C ABI takes bare pointers and cannot check how
    large a buffer is."""
    if not (getattr(t, "is_cuda", False) and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if byte_elems and t.element_size() != 1:
        raise ValueError(f"{name} must have 1-byte elements (uint8 or an 8-bit float)")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, not {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call's tensors are on {device}")
    if t.numel() < min_numel:
        raise ValueError(f"{name} holds {t.numel()} elements, the call writes or reads {min_numel}")


def mxnorm_quant_fwd(x_ptr: int, T: int, H: int, p: int, fmt: int, codes_ptr: int, scales_ptr: int,
                     inv_rms_ptr: int, stream_ptr: int = 0, variant: int = 0) -> None:
    """Raw C-ABI call on device pointers (ints); raises MXNormError."""
    _check(lib().mxnorm_quant_fwd_ex(x_ptr, T, H, p, fmt, codes_ptr, scales_ptr, inv_rms_ptr,
                                     variant, stream_ptr))


def quant_fwd(x, p: int = 2, fmt: str = "mxfp8", variant: str = "auto", out=None, stream=None):
    """MXNorm forward of a contiguous bf16 CUDA tensor x [..., H].

    Returns (codes uint8 [..., H or H/2], scales uint8 [..., H/32],
    inv_rms float32 [...]).  `out` may pass preallocated tensors in that
    order.  Runs on `stream` (default: the current stream); asynchronous.
    """
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()):
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor")
    H = x.shape[-1]
    T = x.numel() // H if H else 0
    lead = tuple(x.shape[:-1])
    if out is None:
        codes = torch.empty(lead + (code_bytes(H, fmt),), dtype=torch.uint8, device=x.device)
        scales = torch.empty(lead + (H // 32,), dtype=torch.uint8, device=x.device)
        inv = torch.empty(lead, dtype=torch.float32, device=x.device)
    else:
        codes, scales, inv = out
        _require(codes, "codes", x.device, min_numel=T * code_bytes(H, fmt), byte_elems=True)
        _require(scales, "scales", x.device, min_numel=T * (H // 32), byte_elems=True)
        _require(inv, "inv_rms", x.device, torch.float32, T)
    with torch.cuda.device(x.device):
        _check(lib().mxnorm_quant_fwd_ex(x.data_ptr(), T, H, int(p), FMT[fmt], codes.data_ptr(),
                                         scales.data_ptr(), inv.data_ptr(), VARIANT[variant],
                                         _stream_ptr(x.device, stream)))
    return codes, scales, inv


def rmsnorm_mxfp8_ref_fwd(x, eps: float = 1e-5, out=None, stream=None):
    """Two-pass RMSNorm-then-MXFP8 baseline.  Returns (y bf16 workspace,
    codes uint8, scales uint8, inv_rms float32)."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()):
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor")
    H = x.shape[-1]
    T = x.numel() // H if H else 0
    lead = tuple(x.shape[:-1])
    if out is None:
        y = torch.empty_like(x)
        codes = torch.empty(lead + (H,), dtype=torch.uint8, device=x.device)
        scales = torch.empty(lead + (H // 32,), dtype=torch.uint8, device=x.device)
        inv = torch.empty(lead, dtype=torch.float32, device=x.device)
    else:
        y, codes, scales, inv = out
        _require(y, "y", x.device, torch.bfloat16, T * H)
        _require(codes, "codes", x.device, min_numel=T * H, byte_elems=True)
        _require(scales, "scales", x.device, min_numel=T * (H // 32), byte_elems=True)
        _require(inv, "inv_rms", x.device, torch.float32, T)
    with torch.cuda.device(x.device):
        _check(lib().rmsnorm_mxfp8_ref_fwd(x.data_ptr(), T, H, float(eps), y.data_ptr(), codes.data_ptr(),
                                           scales.data_ptr(), inv.data_ptr(), _stream_ptr(x.device, stream)))
    return y, codes, scales, inv


def absmax(x, stream=None):
    """max |x| of a contiguous bf16 CUDA tensor, as a 1-element float32 CUDA
    tensor (asynchronous)."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()):
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor")
    out = torch.empty((1,), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        _check(lib().mxnorm_absmax_bf16(x.data_ptr(), x.numel(), out.data_ptr(), _stream_ptr(x.device, stream)))
    return out


def nvfp4_tensor_scale(x, stream=None):
    """The NVFP4 tensor scale of a contiguous bf16 CUDA tensor, derived by
    the library on the device (mxnorm_nvfp4_tensor_scale: the largest finite
    |x| / (448 * 6), rounded to fp32; 1 when there is none but zero).
    Returns a 1-element float32 CUDA tensor; asynchronous."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()):
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor")
    out = torch.empty((1,), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        _check(lib().mxnorm_nvfp4_tensor_scale(x.data_ptr(), x.numel(), out.data_ptr(),
                                               _stream_ptr(x.device, stream)))
    return out


def quant_fwd_nvfp4(x, p: int = 2, tensor_scale=None, out=None, stream=None):
    """MXNorm over the NVFP4 cast of a contiguous bf16 CUDA tensor [..., H]
    (H % 16 == 0).  Returns (codes uint8 [..., H/2], scales uint8 [..., H/16]
    UE4M3, inv_rms float32 [...]).  tensor_scale: a float (passed by value),
    a 1-element float32 CUDA tensor (read by the kernel on the device), or
    None for nvfp4_tensor_scale(x) derived on the device (no host round
    trip either way but the float)."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()):
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor")
    H = x.shape[-1]
    T = x.numel() // H if H else 0
    lead = tuple(x.shape[:-1])
    if tensor_scale is None:
        tensor_scale = nvfp4_tensor_scale(x, stream)
    if out is None:
        out = (torch.empty(lead + (H // 2,), dtype=torch.uint8, device=x.device),
               torch.empty(lead + (H // 16,), dtype=torch.uint8, device=x.device),
               torch.empty(lead, dtype=torch.float32, device=x.device))
    codes, scales, inv = out
    _require(codes, "codes", x.device, min_numel=T * (H // 2), byte_elems=True)
    _require(scales, "scales", x.device, min_numel=T * (H // 16), byte_elems=True)
    _require(inv, "inv_rms", x.device, torch.float32, T)
    with torch.cuda.device(x.device):
        if isinstance(tensor_scale, torch.Tensor):
            _require(tensor_scale, "tensor_scale", x.device, torch.float32, 1)
            _check(lib().mxnorm_quant_fwd_nvfp4_dev(x.data_ptr(), T, H, int(p), tensor_scale.data_ptr(),
                                                    codes.data_ptr(), scales.data_ptr(), inv.data_ptr(),
                                                    _stream_ptr(x.device, stream)))
        else:
            _check(lib().mxnorm_quant_fwd_nvfp4(x.data_ptr(), T, H, int(p), float(tensor_scale), codes.data_ptr(),
                                                scales.data_ptr(), inv.data_ptr(), _stream_ptr(x.device, stream)))
    return codes, scales, inv


SCALE_LAYOUT = {"row_major": 0, "mma": 1}


def mma_scale_bytes(rows: int, H: int) -> int:
    """Bytes of an MMA-layout scale buffer for rows x H (H % 128 == 0)."""
    n = lib().mxnorm_mma_scale_bytes(rows, H)
    if n < 0:
        raise ValueError("the MMA scale layout needs H % 128 == 0")
    return n


def _scale_buffer(rows, H, layout, device):
    import torch
    if layout == "mma":
        return torch.empty((mma_scale_bytes(rows, H),), dtype=torch.uint8, device=device)
    return torch.empty((rows, H // 32), dtype=torch.uint8, device=device)


def quant_fwd_mma(x, p: int = 2, fmt: str = "mxfp8", stream=None):
    """mxnorm_quant_fwd with the scales in the tensor-core MMA atom layout
    (for mxnorm_linear_fwd).  Returns (codes, scales (flat uint8), inv_rms)."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()):
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor")
    H = x.shape[-1]
    T = x.numel() // H if H else 0
    codes = torch.empty(tuple(x.shape[:-1]) + (code_bytes(H, fmt),), dtype=torch.uint8, device=x.device)
    scales = _scale_buffer(T, H, "mma", x.device)
    inv = torch.empty(tuple(x.shape[:-1]), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        _check(lib().mxnorm_quant_fwd_layout(x.data_ptr(), T, H, int(p), FMT[fmt], codes.data_ptr(),
                                             scales.data_ptr(), inv.data_ptr(), 1, _stream_ptr(x.device, stream)))
    return codes, scales, inv


def mx_cast(x, layout: str = "row_major", stream=None):
    """MXFP8 E4M3 cast alone (no estimator) of bf16 rows: (codes, scales)."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()):
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor")
    H = x.shape[-1]
    T = x.numel() // H if H else 0
    codes = torch.empty(tuple(x.shape), dtype=torch.uint8, device=x.device)
    scales = _scale_buffer(T, H, layout, x.device)
    with torch.cuda.device(x.device):
        _check(lib().mx_cast_fwd(x.data_ptr(), T, H, 0, codes.data_ptr(), scales.data_ptr(), SCALE_LAYOUT[layout],
                                 _stream_ptr(x.device, stream)))
    return codes, scales


def mx_cast_gain(w, gamma, c: float = 1.0, layout: str = "mma", stream=None):
    """MXFP8 cast of MXNormLinear's gain-folded weight: rows of
    w[n, k] * RN_fp32(c * gamma[k]), each product rounded to fp32.
    w: contiguous bf16 CUDA tensor [N, K] (one row per output feature);
    gamma: contiguous float32 CUDA tensor [K].  Returns (codes, scales)."""
    import torch
    if not (w.is_cuda and w.dtype == torch.bfloat16 and w.is_contiguous() and w.dim() == 2):
        raise ValueError("w must be a contiguous 2-D bfloat16 CUDA tensor")
    N, K = w.shape
    _require(gamma, "gamma", w.device, torch.float32)
    if tuple(gamma.shape) != (K,):
        raise ValueError("gamma must hold K entries")
    codes = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    scales = _scale_buffer(N, K, layout, w.device)
    with torch.cuda.device(w.device):
        _check(lib().mx_cast_gain_fwd(w.data_ptr(), N, K, gamma.data_ptr(), float(c), codes.data_ptr(),
                                      scales.data_ptr(), SCALE_LAYOUT[layout], _stream_ptr(w.device, stream)))
    return codes, scales


def linear_fwd(x_codes, x_scales, inv_rms, w_codes, w_scales, out=None, stream=None):
    """MXNormLinear's consumer GEMM on the tensor cores: out = bf16(inv_rms[t]
    * sum_k x^[t,k] w^[n,k]); scales in the MMA layout.  Returns out [T, N]."""
    import torch
    if getattr(x_codes, "dim", lambda: 0)() != 2 or getattr(w_codes, "dim", lambda: 0)() != 2:
        raise ValueError("x_codes and w_codes must be 2-D [rows, K]")
    T, K = x_codes.shape
    N = w_codes.shape[0]
    if w_codes.shape[1] != K:
        raise ValueError(f"w_codes has K = {w_codes.shape[1]}, x_codes has K = {K}")
    dev = x_codes.device
    _require(x_codes, "x_codes", dev, byte_elems=True)
    _require(w_codes, "w_codes", dev, byte_elems=True)
    if K % 128 == 0:  # else the C ABI reports the shape error
        _require(x_scales, "x_scales", dev, min_numel=mma_scale_bytes(T, K), byte_elems=True)
        _require(w_scales, "w_scales", dev, min_numel=mma_scale_bytes(N, K), byte_elems=True)
    _require(inv_rms, "inv_rms", dev, torch.float32, T)
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    _require(out, "out", dev, torch.bfloat16, T * N)
    with torch.cuda.device(dev):
        _check(lib().mxnorm_linear_fwd(x_codes.data_ptr(), x_scales.data_ptr(), inv_rms.data_ptr(),
                                       w_codes.data_ptr(), w_scales.data_ptr(), T, K, N, out.data_ptr(),
                                       _stream_ptr(dev, stream)))
    return out


def bwd_ste(x, dy, inv_rms, out=None, stream=None):
    """Straight-through backward of MXNorm: dx = r dy - r^3 x mean(dy x)
    with r = inv_rms from the forward.  x, dy: contiguous bf16 CUDA tensors
    [..., H]; inv_rms: float32 [...].  Returns dx (bf16, like x)."""
    import torch
    for t in (x, dy):
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
            raise ValueError("x and dy must be contiguous bfloat16 CUDA tensors")
    if dy.shape != x.shape or inv_rms.dtype != torch.float32 or not inv_rms.is_contiguous():
        raise ValueError("dy must match x, inv_rms must be contiguous float32")
    H = x.shape[-1]
    T = x.numel() // H if H else 0
    if inv_rms.numel() != T:
        raise ValueError("inv_rms needs one value per row")
    _require(dy, "dy", x.device)
    _require(inv_rms, "inv_rms", x.device, torch.float32, T)
    dx = torch.empty_like(x) if out is None else out
    _require(dx, "out", x.device, torch.bfloat16, T * H)
    with torch.cuda.device(x.device):
        _check(lib().mxnorm_bwd_ste(x.data_ptr(), dy.data_ptr(), inv_rms.data_ptr(), T, H, dx.data_ptr(),
                                    _stream_ptr(x.device, stream)))
    return dx


def tiled_wait_drill(x, withheld_tile: int = 0, wait_limit_ns: int = 2_000_000, out=None, stream=None):
    """Failure-detection drill (mxnorm_tiled_wait_drill): the tiled MXFP8
    pass with one tile's copy withheld, so that its bounded waits expire
    after wait_limit_ns and bit 0 of device_errors() gets set.  Returns the
    (invalid) outputs (codes, scales, inv_rms)."""
    import torch
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()):
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor")
    H = x.shape[-1]
    T = x.numel() // H if H else 0
    if out is None:
        out = (torch.empty((T, H), dtype=torch.uint8, device=x.device),
               torch.empty((T, H // 32), dtype=torch.uint8, device=x.device),
               torch.empty((T,), dtype=torch.float32, device=x.device))
    codes, scales, inv = out
    _require(codes, "codes", x.device, min_numel=T * H, byte_elems=True)
    _require(scales, "scales", x.device, min_numel=T * (H // 32), byte_elems=True)
    _require(inv, "inv_rms", x.device, torch.float32, T)
    with torch.cuda.device(x.device):
        _check(lib().mxnorm_tiled_wait_drill(x.data_ptr(), T, H, codes.data_ptr(), scales.data_ptr(),
                                             inv.data_ptr(), int(withheld_tile), int(wait_limit_ns),
                                             _stream_ptr(x.device, stream)))
    return codes, scales, inv


def device_errors(clear: bool = True) -> int:
    """The device error flags: bit 0, a bounded wait of the tiled kernel
    timed out; bit 1, a pipeline wait of the GEMM timed out; bit 2, a device
    NVFP4 tensor scale was not a finite positive float."""
    v = ctypes.c_uint32(0)
    _check(lib().mxnorm_device_errors(ctypes.byref(v), int(clear)))
    return v.value


_host_ws = {}


def quant_fwd_host(x, p: int = 2, fmt: str = "mxfp8", out=None, device=None, chunks: int = 8,
                   variant: str = "auto", mode: str = "auto"):
    """MXNorm forward of a bf16 CPU tensor; returns (codes, scales, inv_rms)
    CPU tensors, valid once the current stream of `device` has synchronised.

    mode "zero_copy": x and the outputs are pinned host memory, which is
    mapped into the GPU's address space; the kernel reads x and writes its
    outputs across the host link directly (no staging buffers, no copy
    engine).  On Grace-Blackwell this runs at the host link's speed.
    mode "staged": the rows are split into `chunks` pieces over three CUDA
    streams: per piece a host->device copy of x, the C-ABI call, and
    device->host copies of codes, scales and inv_rms, so copies in both
    directions overlap with each other and with the kernels; device
    staging buffers are cached per (device, shape, fmt).
    mode "auto": zero_copy when x and every output are pinned, else staged.
    """
    import torch
    if x.is_cuda or x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bfloat16 CPU tensor")
    device = torch.device(device if device is not None else "cuda")
    if device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    H = x.shape[-1]
    T = x.numel() // H if H else 0
    cb = code_bytes(H, fmt)
    if out is None:
        out = (torch.empty((T, cb), dtype=torch.uint8).pin_memory(),
               torch.empty((T, H // 32), dtype=torch.uint8).pin_memory(),
               torch.empty((T,), dtype=torch.float32).pin_memory())
    pinned = x.is_pinned() and all(t.is_pinned() and t.is_contiguous() for t in out)
    if mode == "auto":
        mode = "zero_copy" if pinned else "staged"
    if mode == "zero_copy":
        if not pinned:
            raise ValueError("zero_copy needs x and every output in pinned (page-locked) host memory")
        with torch.cuda.device(device):
            _check(lib().mxnorm_quant_fwd_ex(x.data_ptr(), T, H, int(p), FMT[fmt], out[0].data_ptr(),
                                             out[1].data_ptr(), out[2].data_ptr(), VARIANT[variant],
                                             _stream_ptr(device, None)))
        return out
    if mode != "staged":
        raise ValueError(f"unknown mode {mode!r}")
    oc, os_, oi = (t.view(-1) for t in out)
    key = (device.index, T, H, fmt)
    ws = _host_ws.get(key)
    if ws is None:
        ws = {"x": torch.empty((T, H), dtype=torch.bfloat16, device=device),
              "c": torch.empty((T, cb), dtype=torch.uint8, device=device),
              "s": torch.empty((T, H // 32), dtype=torch.uint8, device=device),
              "i": torch.empty((T,), dtype=torch.float32, device=device),
              "streams": [torch.cuda.Stream(device=device) for _ in range(3)]}
        _host_ws[key] = ws
    xv = x.view(T, H)
    cur = torch.cuda.current_stream(device)
    streams = ws["streams"]
    for s in streams:
        s.wait_stream(cur)
    rc = max(1, -(-T // max(1, chunks)))
    L = lib()
    for j, r0 in enumerate(range(0, T, rc)):
        r1 = min(T, r0 + rc)
        s = streams[j % len(streams)]
        with torch.cuda.stream(s):
            xd = ws["x"][r0:r1]
            xd.copy_(xv[r0:r1], non_blocking=True)
            cd, sd, idd = ws["c"][r0:r1], ws["s"][r0:r1], ws["i"][r0:r1]
            _check(L.mxnorm_quant_fwd_ex(xd.data_ptr(), r1 - r0, H, int(p), FMT[fmt], cd.data_ptr(),
                                         sd.data_ptr(), idd.data_ptr(), VARIANT[variant],
                                         ctypes.c_void_p(s.cuda_stream)))
            oc[r0 * cb:r1 * cb].copy_(cd.reshape(-1), non_blocking=True)
            os_[r0 * (H // 32):r1 * (H // 32)].copy_(sd.reshape(-1), non_blocking=True)
            oi[r0:r1].copy_(idd, non_blocking=True)
    for s in streams:
        cur.wait_stream(s)
    return out
