"""CPU oracle for MXNorm -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or runs anything here, and this package
never imports the product.  The arithmetic lives in ``mxnorm_oracle.c``
(plain scalar C, fp64); this module only compiles it with gcc and marshals
numpy arrays.  ``bruteforce.py`` is a second, pure-Python implementation in
exact rational arithmetic for tiny inputs.

Method sources (by page title and section):
  * "MXNorm: Reusing MXFP block scales for efficient tensor normalisation",
    Resumen tecnico, 2. Metodologia, "Fundamentos Teoricos" (formula) and
    "Implementacion" (fusion of the norm and the MX cast);
  * the same paper's English abstract (scales reused from the MXFP8 cast);
  * "Entrenamiento Previo ... con MXFP4", Metodologia, item 3 (deterministic
    H16 Hadamard rotation);
  * OCP Microscaling Formats v1.0, sections 5 and 6.3 (encodings, shared
    exponent rule).

Parity status of each function is stated in its docstring; all are pinned by
the ``-m "not gpu"`` tests except the statistical behaviour of the estimator
(the pages' Theorem 1), which the pages give no constant for: parity
unpinned there.  ``theorem1.py`` reports that behaviour as a diagnostic (the
empirical constant per workload); only the bounds the E8M0 rule forces on it
are pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

FMT_MXFP8_E4M3 = 0
FMT_MXFP4_E2M1 = 1
FMT_MXFP4_E2M1_H16 = 2
FMT_MXFP8_E4M3_H16 = 3
FMT_MXFP4_E2M1_H32 = 4
FMT_MXFP8_E4M3_H32 = 5
FMT_NAMES = {"mxfp8": FMT_MXFP8_E4M3, "mxfp4": FMT_MXFP4_E2M1, "mxfp4_h16": FMT_MXFP4_E2M1_H16,
             "mxfp8_h16": FMT_MXFP8_E4M3_H16, "mxfp4_h32": FMT_MXFP4_E2M1_H32, "mxfp8_h32": FMT_MXFP8_E4M3_H32}
FP8_FMTS = (FMT_MXFP8_E4M3, FMT_MXFP8_E4M3_H16, FMT_MXFP8_E4M3_H32)
BLOCK = 32

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxnorm_oracle.c")
_LIB = os.path.join(_HERE, "libmxnorm_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (-O2, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
    p = ctypes.c_void_p
    lib.oracle_mxnorm_rows.argtypes = [p, i64, i64, i32, i32, p, p, p]
    lib.oracle_mxnorm_rows.restype = i32
    lib.oracle_mx_cast_rows.argtypes = [p, i64, i64, i32, p, p]
    lib.oracle_mx_cast_rows.restype = i32
    lib.oracle_mx_cast_gain_rows.argtypes = [p, i64, i64, p, f32, p, p]
    lib.oracle_mx_cast_gain_rows.restype = i32
    lib.oracle_rmsnorm_mxfp8_rows.argtypes = [p, i64, i64, f32, p, p, p, p]
    lib.oracle_rmsnorm_mxfp8_rows.restype = i32
    lib.oracle_cast_e4m3_array.argtypes = [p, i64, p]
    lib.oracle_cast_e2m1_array.argtypes = [p, i64, p]
    lib.oracle_e8m0_exponent_array.argtypes = [p, i64, i32, p]
    lib.oracle_h16_groups.argtypes = [p, i64, p]
    lib.oracle_h32_groups.argtypes = [p, i64, p]
    lib.oracle_float_to_bf16_array.argtypes = [p, i64, p]
    lib.oracle_mxnorm_bwd_ste_rows.argtypes = [p, p, p, i64, i64, p, p]
    lib.oracle_nvfp4_rows.argtypes = [p, i64, i64, i32, f32, p, p, p]
    lib.oracle_mxfp8_linear.argtypes = [p, p, p, p, p, i64, i64, i64, p]
    lib.oracle_mxfp8_linear.restype = i32
    lib.oracle_nvfp4_rows.restype = i32
    lib.oracle_nvfp4_tensor_scale.argtypes = [p, i64]
    lib.oracle_nvfp4_tensor_scale.restype = f32
    lib.oracle_mxnorm_bwd_ste_rows.restype = i32
    lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_decode_e4m3.restype = ctypes.c_double
    lib.oracle_decode_e2m1.argtypes = [ctypes.c_uint8]
    lib.oracle_decode_e2m1.restype = ctypes.c_double
    _lib = lib
    return lib


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def rows_in_threads(fn, *row_arrays, threads: int | None = None):
    """fn(*slices) over slices of the row arrays (split along axis 0), one
    slice per host thread, results concatenated along rows (each output
    array of a tuple separately).  The oracle's C calls release the GIL, so
    the slices run on separate cores; every row is still computed exactly
    as one call over all rows would compute it (rows are independent)."""
    from concurrent.futures import ThreadPoolExecutor
    n = row_arrays[0].shape[0]
    k = max(1, min(threads or host_threads(), n))
    bounds = np.linspace(0, n, k + 1).astype(np.int64)
    parts = [tuple(np.ascontiguousarray(a[lo:hi]) for a in row_arrays) for lo, hi in zip(bounds[:-1], bounds[1:])]
    with ThreadPoolExecutor(max_workers=k) as ex:
        outs = list(ex.map(lambda args: fn(*args), parts))
    if isinstance(outs[0], tuple):
        return tuple(np.concatenate([o[i] for o in outs]) for i in range(len(outs[0])))
    return np.concatenate(outs)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _fmt_id(fmt) -> int:
    return FMT_NAMES[fmt] if isinstance(fmt, str) else int(fmt)


def _as_bf16_bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
    return x


def code_bytes_per_row(H: int, fmt) -> int:
    """Code bytes of one row: H for the FP8 formats, H/2 for FP4."""
    return H if _fmt_id(fmt) in FP8_FMTS else H // 2


def mxnorm_quant(x_bits: np.ndarray, p: int = 2, fmt="mxfp8"):
    """MXNorm forward of bf16 rows [T, H]: (codes u8, scales u8 [T, H/32], inv_rms f32 [T]).

    Follows the estimator of "MXNorm ...", Fundamentos Teoricos, with
    m~_k = s_k (the E8M0 scale) and c(p,B) = 1.  Pinned by the closed-form,
    exhaustive and brute-force tests under tests/.
    """
    lib = _load()
    x = _as_bf16_bits(x_bits)
    T, H = x.shape
    f = _fmt_id(fmt)
    codes = np.empty((T, code_bytes_per_row(H, f)), np.uint8)
    scales = np.empty((T, H // BLOCK), np.uint8)
    inv = np.empty((T,), np.float32)
    rc = lib.oracle_mxnorm_rows(_ptr(x), T, H, int(p), f, _ptr(codes), _ptr(scales), _ptr(inv))
    if rc != 0:
        raise ValueError(f"oracle rejected arguments T={T} H={H} p={p} fmt={fmt}")
    return codes, scales, inv


def mx_cast(x_bits: np.ndarray, fmt="mxfp8"):
    """MX cast only (codes, scales) of bf16 rows [T, H]; OCP MX v1.0 6.3."""
    lib = _load()
    x = _as_bf16_bits(x_bits)
    T, H = x.shape
    f = _fmt_id(fmt)
    codes = np.empty((T, code_bytes_per_row(H, f)), np.uint8)
    scales = np.empty((T, H // BLOCK), np.uint8)
    if lib.oracle_mx_cast_rows(_ptr(x), T, H, f, _ptr(codes), _ptr(scales)) != 0:
        raise ValueError("oracle rejected arguments")
    return codes, scales


def rmsnorm_mxfp8(x_bits: np.ndarray, eps: float = 1e-5):
    """Two-pass baseline: RMSNorm (no gain) then MXFP8 cast of its bf16 output.

    Returns (y bf16 bits [T, H], codes, scales, inv_rms)."""
    lib = _load()
    x = _as_bf16_bits(x_bits)
    T, H = x.shape
    y = np.empty((T, H), np.uint16)
    codes = np.empty((T, H), np.uint8)
    scales = np.empty((T, H // BLOCK), np.uint8)
    inv = np.empty((T,), np.float32)
    if lib.oracle_rmsnorm_mxfp8_rows(_ptr(x), T, H, float(eps), _ptr(y), _ptr(codes), _ptr(scales), _ptr(inv)) != 0:
        raise ValueError("oracle rejected arguments")
    return y, codes, scales, inv


def mx_cast_gain(w_bits: np.ndarray, gamma, c: float = 1.0):
    """MXFP8 cast (codes, row-major scales) of the gain-folded weight rows
    w[n, j] * RN_fp32(c * gamma_j), each product rounded to fp32 ("MXNorm
    ...", 2. Metodologia, Implementacion: gamma folded into the next layer's
    weight)."""
    lib = _load()
    w = _as_bf16_bits(w_bits)
    N, K = w.shape
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    if g.shape != (K,):
        raise ValueError("gamma must have K entries")
    codes = np.empty((N, K), np.uint8)
    scales = np.empty((N, K // BLOCK), np.uint8)
    if lib.oracle_mx_cast_gain_rows(_ptr(w), N, K, _ptr(g), float(np.float32(c)), _ptr(codes), _ptr(scales)) != 0:
        raise ValueError("oracle rejected arguments")
    return codes, scales


def mxfp8_linear(x_codes, x_scales, inv_rms, w_codes, w_scales) -> np.ndarray:
    """out[t, n] = inv_rms[t] * sum_k xv[t, k] wv[n, k] in fp64 (MXNormLinear's
    consumer GEMM with the gain folded into w); scales row-major [rows, K/32]."""
    lib = _load()
    xc = np.ascontiguousarray(x_codes, np.uint8)
    wc = np.ascontiguousarray(w_codes, np.uint8)
    xs = np.ascontiguousarray(x_scales, np.uint8)
    ws = np.ascontiguousarray(w_scales, np.uint8)
    inv = np.ascontiguousarray(inv_rms, np.float32)
    T, K = xc.shape
    N = wc.shape[0]
    if wc.shape[1] != K or xs.shape != (T, K // BLOCK) or ws.shape != (N, K // BLOCK) or inv.shape != (T,):
        raise ValueError("shape mismatch")
    out = np.empty((T, N), np.float64)
    if lib.oracle_mxfp8_linear(_ptr(xc), _ptr(xs), _ptr(inv), _ptr(wc), _ptr(ws), T, K, N, _ptr(out)) != 0:
        raise ValueError("oracle rejected arguments")
    return out


def nvfp4_quant(x_bits: np.ndarray, p: int, tensor_scale: float):
    """NVFP4 forward (16-element blocks, UE4M3 block scales over a tensor
    scale g): (codes u8 [T, H/2], scales u8 [T, H/16], inv_rms f32 [T])."""
    lib = _load()
    x = _as_bf16_bits(x_bits)
    T, H = x.shape
    codes = np.empty((T, H // 2), np.uint8)
    scales = np.empty((T, H // 16), np.uint8)
    inv = np.empty((T,), np.float32)
    if lib.oracle_nvfp4_rows(_ptr(x), T, H, int(p), float(tensor_scale), _ptr(codes), _ptr(scales), _ptr(inv)) != 0:
        raise ValueError("oracle rejected arguments")
    return codes, scales, inv


def nvfp4_tensor_scale(x_bits: np.ndarray) -> float:
    """The NVFP4 tensor scale of a bf16 tensor: RN_fp32(a / (448 * 6)) with
    a the largest finite |x|, 1.0 when there is none but zero."""
    x = _as_bf16_bits(x_bits)
    return float(_load().oracle_nvfp4_tensor_scale(_ptr(x), x.size))


def mxnorm_bwd_ste(x_bits: np.ndarray, dy_bits: np.ndarray, inv_rms: np.ndarray, with_f64: bool = False):
    """Straight-through backward: dx = r dy - r^3 x mean(dy x) with r the
    forward's inv_rms ("MXNorm ...", 2. Metodologia, Gradientes: RMSNorm's
    gradient logic reused).  Returns dx as bf16 bits [T, H] (and the
    unrounded fp64 values when with_f64)."""
    lib = _load()
    x = _as_bf16_bits(x_bits)
    dy = _as_bf16_bits(dy_bits)
    inv = np.ascontiguousarray(inv_rms, dtype=np.float32)
    T, H = x.shape
    if dy.shape != x.shape or inv.shape != (T,):
        raise ValueError("shape mismatch")
    dx = np.empty((T, H), np.uint16)
    dx64 = np.empty((T, H), np.float64) if with_f64 else None
    if lib.oracle_mxnorm_bwd_ste_rows(_ptr(x), _ptr(dy), _ptr(inv), T, H, _ptr(dx),
                                      _ptr(dx64) if with_f64 else None) != 0:
        raise ValueError("oracle rejected arguments")
    return (dx, dx64) if with_f64 else dx


def cast_e4m3(r) -> np.ndarray:
    """Saturating RNE E4M3 codes of finite reals r (any shape)."""
    lib = _load()
    r = np.ascontiguousarray(r, dtype=np.float64)
    out = np.empty(r.shape, np.uint8)
    lib.oracle_cast_e4m3_array(_ptr(r), r.size, _ptr(out))
    return out


def cast_e2m1(r) -> np.ndarray:
    """Saturating RNE E2M1 nibbles (0..15) of finite reals r (any shape)."""
    lib = _load()
    r = np.ascontiguousarray(r, dtype=np.float64)
    out = np.empty(r.shape, np.uint8)
    lib.oracle_cast_e2m1_array(_ptr(r), r.size, _ptr(out))
    return out


def e8m0_exponent(amax, emax_elem: int) -> np.ndarray:
    """Shared exponent clamp(floor(log2 amax) - emax_elem, -127, 127), 0 -> -127."""
    lib = _load()
    a = np.ascontiguousarray(amax, dtype=np.float64)
    out = np.empty(a.shape, np.int32)
    lib.oracle_e8m0_exponent_array(_ptr(a), a.size, int(emax_elem), _ptr(out))
    return out


def h16(v) -> np.ndarray:
    """(1/4) * H16 applied to each consecutive group of 16 fp32 values."""
    lib = _load()
    a = np.ascontiguousarray(v, dtype=np.float32)
    if a.size % 16:
        raise ValueError("h16 needs a multiple of 16 values")
    out = np.empty_like(a)
    lib.oracle_h16_groups(_ptr(a), a.size // 16, _ptr(out))
    return out


def h32(v) -> np.ndarray:
    """H32 / sqrt(32) applied to each consecutive group of 32 fp32 values."""
    lib = _load()
    a = np.ascontiguousarray(v, dtype=np.float32)
    if a.size % 32:
        raise ValueError("h32 needs a multiple of 32 values")
    out = np.empty_like(a)
    lib.oracle_h32_groups(_ptr(a), a.size // 32, _ptr(out))
    return out


def float_to_bf16(v) -> np.ndarray:
    """Round fp32 values to bf16 bit patterns, nearest, ties to even."""
    lib = _load()
    a = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    lib.oracle_float_to_bf16_array(_ptr(a), a.size, _ptr(out))
    return out


def decode_e4m3(code: int) -> float:
    """Value of an E4M3 code byte (OCP MX v1.0, section 5.3)."""
    return _load().oracle_decode_e4m3(int(code))


def decode_e2m1(nibble: int) -> float:
    """Value of an E2M1 code nibble (OCP MX v1.0, section 5.3)."""
    return _load().oracle_decode_e2m1(int(nibble))
