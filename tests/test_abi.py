"""Host-side checks of the C ABI: the library loads, exports every function
include/mxnorm.h declares, and rejects bad arguments with the documented
status before touching the GPU (these calls never reach a CUDA API)."""
import ctypes
import os
import re

import pytest

import mx_scale_reusing_gb300 as mx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from mx_scale_reusing_gb300 import _build
    _build.build()
    return mx.lib()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"mxnorm_quant_fwd", "mxnorm_quant_fwd_ex", "rmsnorm_mxfp8_ref_fwd"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_abi_version_and_strings(L):
    assert L.mxnorm_abi_version() == 1
    assert L.mxnorm_status_string(0) == b"MXNORM_OK"
    assert L.mxnorm_status_string(3) == b"MXNORM_ERR_MISALIGNED"
    assert L.mxnorm_status_string(99) == b"MXNORM_ERR_UNKNOWN"


FAKE = 1 << 40  # never dereferenced: validation fails or T == 0 first


@pytest.mark.parametrize("T,H,p,fmt,variant,status", [
    (0, 4096, 2, 0, 0, 0),            # empty input: no-op
    (-1, 4096, 2, 0, 0, 1),
    (8, 0, 2, 0, 0, 1),
    (8, 33, 2, 0, 0, 1),
    (8, 4096, 3, 0, 0, 1),
    (8, 4096, 0, 0, 0, 1),
    (8, 4096, 2, 7, 0, 1),
    (8, 4096, 2, 0, 9, 1),
    (8, (1 << 20) + 32, 2, 0, 0, 2),   # above MXNORM_MAX_H
    (8, 8192, 2, 0, 2, 2),            # tiled variant does not take H = 8192
])
def test_quant_fwd_validation(L, T, H, p, fmt, variant, status):
    rc = L.mxnorm_quant_fwd_ex(FAKE, T, H, p, fmt, FAKE, FAKE, FAKE, variant, None)
    assert rc == status, L.mxnorm_last_error()
    if status:
        assert L.mxnorm_last_error()


def test_null_and_misaligned_pointers(L):
    assert L.mxnorm_quant_fwd(None, 8, 64, 2, 0, FAKE, FAKE, FAKE, None) == 1
    assert L.mxnorm_quant_fwd(FAKE + 8, 8, 64, 2, 0, FAKE, FAKE, FAKE, None) == 3
    assert L.mxnorm_quant_fwd(FAKE, 8, 64, 2, 0, FAKE + 4, FAKE, FAKE, None) == 3
    assert L.mxnorm_quant_fwd(FAKE, 8, 64, 2, 0, FAKE, FAKE, FAKE + 2, None) == 3
    assert L.rmsnorm_mxfp8_ref_fwd(FAKE, 8, 64, 1e-5, None, FAKE, FAKE, FAKE, None) == 1
    assert L.rmsnorm_mxfp8_ref_fwd(FAKE, 8, 64, 1e-5, FAKE + 8, FAKE, FAKE, FAKE, None) == 3
    assert L.rmsnorm_mxfp8_ref_fwd(FAKE, 8, 64, -1.0, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert L.rmsnorm_mxfp8_ref_fwd(FAKE, 0, 64, 1e-5, FAKE, FAKE, FAKE, FAKE, None) == 0


def test_bwd_validation(L):
    assert L.mxnorm_bwd_ste(FAKE, FAKE, FAKE, 0, 4096, FAKE, None) == 0
    assert L.mxnorm_bwd_ste(FAKE, FAKE, FAKE, -1, 4096, FAKE, None) == 1
    assert L.mxnorm_bwd_ste(FAKE, FAKE, FAKE, 8, 100, FAKE, None) == 1
    assert L.mxnorm_bwd_ste(FAKE, None, FAKE, 8, 128, FAKE, None) == 1
    assert L.mxnorm_bwd_ste(FAKE, FAKE + 8, FAKE, 8, 128, FAKE, None) == 3
    assert L.mxnorm_bwd_ste(FAKE, FAKE, FAKE + 1, 8, 128, FAKE, None) == 3
    assert L.mxnorm_bwd_ste(FAKE, FAKE, FAKE, 8, (1 << 20) + 32, FAKE, None) == 2


def test_nvfp4_validation(L):
    q = L.mxnorm_quant_fwd_nvfp4
    assert q(FAKE, 0, 4096, 2, 1.0, FAKE, FAKE, FAKE, None) == 0
    assert q(FAKE, 8, 4096, 3, 1.0, FAKE, FAKE, FAKE, None) == 1
    assert q(FAKE, 8, 4096, 2, 0.0, FAKE, FAKE, FAKE, None) == 1
    assert q(FAKE, 8, 4096, 2, float("inf"), FAKE, FAKE, FAKE, None) == 1
    assert q(FAKE, 8, 4096, 2, float("nan"), FAKE, FAKE, FAKE, None) == 1
    assert q(FAKE, 8, 24, 2, 1.0, FAKE, FAKE, FAKE, None) == 1
    assert q(FAKE, 8, 48, 2, 1.0, FAKE + 8, FAKE, FAKE, None) == 3
    assert L.mxnorm_absmax_bf16(FAKE, -1, FAKE, None) == 1
    assert L.mxnorm_absmax_bf16(FAKE, 8, None, None) == 1
    d = L.mxnorm_quant_fwd_nvfp4_dev
    assert d(FAKE, 0, 4096, 2, FAKE, FAKE, FAKE, FAKE, None) == 0
    assert d(FAKE, 8, 4096, 3, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert d(FAKE, 8, 4096, 2, None, FAKE, FAKE, FAKE, None) == 1
    assert d(FAKE, 8, 24, 2, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert d(FAKE, 8, 48, 2, FAKE + 2, FAKE, FAKE, FAKE, None) == 3
    assert d(FAKE, 8, 48, 2, FAKE, FAKE + 8, FAKE, FAKE, None) == 3
    assert d(FAKE, 8, (1 << 20) + 16, 2, FAKE, FAKE, FAKE, FAKE, None) == 2
    ts = L.mxnorm_nvfp4_tensor_scale
    assert ts(FAKE, -1, FAKE, None) == 1
    assert ts(FAKE, 8, None, None) == 1
    assert ts(None, 8, FAKE, None) == 1
    assert ts(FAKE, 8, FAKE + 2, None) == 3


def test_static_workspace_validation(L):
    """The allocation-free baseline entry checks its arguments as
    rmsnorm_mxfp8_ref_fwd does (same checks, same statuses), then the size
    of its built-in workspace: T * H above MXNORM_STATIC_WS_BYTES / 2."""
    f = L.rmsnorm_mxfp8_ref_fwd_static_ws
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    H = 4096
    limit_rows = (32 << 20) // 2 // H
    assert f(FAKE, limit_rows + 1, H, 1e-5, FAKE, FAKE, FAKE, None) == 2
    assert b"static workspace" in L.mxnorm_last_error()
    assert f(FAKE, 0, H, 1e-5, FAKE, FAKE, FAKE, None) == 0
    assert f(FAKE, -1, H, 1e-5, FAKE, FAKE, FAKE, None) == 1
    assert f(FAKE, 8, 100, 1e-5, FAKE, FAKE, FAKE, None) == 1
    assert f(FAKE, 8, (1 << 20) + 32, 1e-5, FAKE, FAKE, FAKE, None) == 2
    assert b"MXNORM_MAX_H" in L.mxnorm_last_error()
    assert f(FAKE, 8, H, -1.0, FAKE, FAKE, FAKE, None) == 1
    assert f(FAKE, 8, H, float("nan"), FAKE, FAKE, FAKE, None) == 1
    assert f(None, 8, H, 1e-5, FAKE, FAKE, FAKE, None) == 1
    assert f(FAKE, 8, H, 1e-5, FAKE, None, FAKE, None) == 1
    assert f(FAKE + 8, 8, H, 1e-5, FAKE, FAKE, FAKE, None) == 3
    assert f(FAKE, 8, H, 1e-5, FAKE + 4, FAKE, FAKE, None) == 3
    assert f(FAKE, 8, H, 1e-5, FAKE, FAKE, FAKE + 2, None) == 3


def test_wait_drill_validation(L):
    """The drill entry point refuses what it cannot run before any launch:
    an empty input, a tile outside the input, a wait limit outside
    [1e5, 1e9] ns, and the usual shape, pointer and alignment errors."""
    w = L.mxnorm_tiled_wait_drill
    assert w(FAKE, 0, 4096, FAKE, FAKE, FAKE, 0, 2000000, None) == 1
    assert w(FAKE, 16, 4096, FAKE, FAKE, FAKE, 2, 2000000, None) == 1
    assert w(FAKE, 16, 4096, FAKE, FAKE, FAKE, -1, 2000000, None) == 1
    assert w(FAKE, 16, 4096, FAKE, FAKE, FAKE, 0, 99999, None) == 1
    assert w(FAKE, 16, 4096, FAKE, FAKE, FAKE, 0, 1000000001, None) == 1
    assert w(FAKE, 16, 100, FAKE, FAKE, FAKE, 0, 2000000, None) == 1
    assert w(FAKE, 16, 8192, FAKE, FAKE, FAKE, 0, 2000000, None) == 2   # the tiled ring holds H <= 6400
    assert w(None, 16, 4096, FAKE, FAKE, FAKE, 0, 2000000, None) == 1
    assert w(FAKE + 8, 16, 4096, FAKE, FAKE, FAKE, 0, 2000000, None) == 3


def test_linear_and_layout_validation(L):
    assert L.mxnorm_mma_scale_bytes(300, 768) == 3 * 6 * 512
    assert L.mxnorm_mma_scale_bytes(300, 96) == -1
    lin = L.mxnorm_linear_fwd
    assert lin(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 128, 256, FAKE, None) == 0
    assert lin(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 96, 256, FAKE, None) == 1
    assert lin(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 128, 128, FAKE, None) == 1
    assert lin(FAKE, FAKE, FAKE, None, FAKE, 8, 128, 256, FAKE, None) == 1
    assert lin(FAKE, FAKE + 8, FAKE, FAKE, FAKE, 8, 128, 256, FAKE, None) == 3
    # 32-bit tile coordinates: too many rows, or too many scale-map rows
    assert lin(FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 31, 128, 256, FAKE, None) == 2
    assert lin(FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 28, 1 << 15, 256, FAKE, None) == 2  # 2^21 tiles x 2^10
    assert lin(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 1 << 20, 1 << 24, FAKE, None) == 2
    assert lin(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1 << 15, 1 << 12, FAKE, None) == 0
    q = L.mxnorm_quant_fwd_layout
    assert q(FAKE, 8, 96, 2, 0, FAKE, FAKE, FAKE, 1, None) == 1
    assert q(FAKE, 8, 128, 2, 0, FAKE, FAKE, FAKE, 7, None) == 1
    assert L.mx_cast_fwd(FAKE, 8, 128, 1, FAKE, FAKE, 0, None) == 2
    assert L.mx_cast_fwd(FAKE, 8, 96, 0, FAKE, FAKE, 1, None) == 1


def test_gain_cast_validation(L):
    g = L.mx_cast_gain_fwd
    assert g(FAKE, 0, 128, FAKE, 1.0, FAKE, FAKE, 1, None) == 0      # no rows: no launch
    assert g(FAKE, -1, 128, FAKE, 1.0, FAKE, FAKE, 0, None) == 1
    assert g(FAKE, 8, 48, FAKE, 1.0, FAKE, FAKE, 0, None) == 1       # K % 32
    assert g(FAKE, 8, 96, FAKE, 1.0, FAKE, FAKE, 1, None) == 1       # MMA layout needs K % 128
    assert g(FAKE, 8, 128, FAKE, 1.0, FAKE, FAKE, 5, None) == 1      # unknown layout
    assert g(FAKE, 8, 128, FAKE, float("inf"), FAKE, FAKE, 0, None) == 1
    assert g(FAKE, 8, 128, None, 1.0, FAKE, FAKE, 0, None) == 1
    assert g(FAKE, 8, 128, FAKE + 4, 1.0, FAKE, FAKE, 0, None) == 3  # gamma alignment
    assert g(FAKE, 8, 128, FAKE, 1.0, FAKE + 8, FAKE, 0, None) == 3  # codes alignment
    assert g(FAKE, 8, (1 << 20) + 32, FAKE, 1.0, FAKE, FAKE, 0, None) == 2


def test_python_binding_raises_on_status(L):
    with pytest.raises(mx.MXNormError) as ei:
        mx.mxnorm_quant_fwd(FAKE, 8, 48, 2, 0, FAKE, FAKE, FAKE)
    assert ei.value.status == 1 and "multiple of 32" in str(ei.value)


def test_product_path_does_not_import_oracle():
    """The package (binding, generator, build script) never imports the
    oracle, and the oracle never imports the package."""
    pkg = os.path.join(ROOT, "mx_scale_reusing_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            assert not re.search(r"^\s*(import|from)\s+oracle", open(os.path.join(pkg, f)).read(), re.M), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            assert "mx_scale_reusing_gb300" not in open(os.path.join(ROOT, "oracle", f)).read(), f


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(mx, "_lib", None)
    monkeypatch.setattr(mx, "library_path", str(tmp_path / "absent.so"))
    with pytest.raises(mx.MXNormLibraryMissing):
        mx.lib()


class _FakeCuda:
    """Stands in for a CUDA tensor in the binding's argument checks (no GPU
    here): the attributes _require reads."""

    def __init__(self, numel, dtype, device="cuda:0", contiguous=True, esize=None):
        import torch
        self._n, self.dtype, self.device = numel, dtype, torch.device(device)
        self.is_cuda, self._c = True, contiguous
        self._es = esize if esize is not None else torch.empty((), dtype=dtype).element_size()

    def is_contiguous(self):
        return self._c

    def numel(self):
        return self._n

    def element_size(self):
        return self._es


def test_binding_buffer_checks():
    """Buffers handed to the C ABI are checked for device, dtype, layout and
    size before any call: the ABI takes bare pointers."""
    import torch
    d0 = torch.device("cuda:0")
    ok = _FakeCuda(100, torch.float32)
    mx._require(ok, "inv_rms", d0, torch.float32, 100)
    with pytest.raises(ValueError, match="holds 99"):
        mx._require(_FakeCuda(99, torch.float32), "inv_rms", d0, torch.float32, 100)
    with pytest.raises(ValueError, match="must be torch.float32"):
        mx._require(_FakeCuda(100, torch.float16), "inv_rms", d0, torch.float32, 100)
    with pytest.raises(ValueError, match="is on cuda:1"):
        mx._require(_FakeCuda(100, torch.float32, "cuda:1"), "inv_rms", d0, torch.float32, 100)
    with pytest.raises(ValueError, match="contiguous"):
        mx._require(_FakeCuda(100, torch.float32, contiguous=False), "inv_rms", d0, torch.float32)
    with pytest.raises(ValueError, match="1-byte"):
        mx._require(_FakeCuda(100, torch.int16), "codes", d0, byte_elems=True)
    mx._require(_FakeCuda(100, torch.uint8), "codes", d0, byte_elems=True, min_numel=100)
    with pytest.raises(ValueError, match="contiguous CUDA"):
        mx._require(torch.zeros(4), "x", d0)


def test_binding_rejects_host_tensors():
    import torch
    x = torch.zeros((4, 32), dtype=torch.bfloat16)
    for fn in (lambda: mx.quant_fwd(x), lambda: mx.mx_cast(x), lambda: mx.quant_fwd_mma(x),
               lambda: mx.mx_cast_gain(x, torch.ones(32)), lambda: mx.bwd_ste(x, x, torch.ones(4))):
        with pytest.raises(ValueError):
            fn()


def test_header_is_plain_c_and_links(L):
    """include/mxnorm.h compiles as strict C11 with nothing but the C
    library, and a C program that takes every declared entry point links
    against libmxnorm.so and runs its host-only calls."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    work = os.path.join(ROOT, "_build", "c_abi_check")
    os.makedirs(work, exist_ok=True)
    src = os.path.join(work, "use_mxnorm.c")
    with open(src, "w") as f:
        f.write('#include "mxnorm.h"\n#include <stdio.h>\n#include <string.h>\n'
                "typedef void (*fn_t)(void);\n"
                "static const fn_t entry_points[] = {\n"
                + "".join(f"    (fn_t){n},\n" for n in names)
                + "};\n"
                "int main(void) {\n"
                '    printf("%d %d %s|%s\\n", mxnorm_abi_version(), (int)(sizeof entry_points / sizeof entry_points[0]),\n'
                "           mxnorm_status_string(MXNORM_ERR_INVALID_ARG), mxnorm_last_error());\n"
                "    return 0;\n}\n")
    libdir = os.path.dirname(mx.library_path)
    exe = os.path.join(work, "use_mxnorm")
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        src, "-L", libdir, "-l:" + os.path.basename(mx.library_path), "-Wl,-rpath," + libdir,
                        "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    version, count, rest = r.stdout.split(" ", 2)
    assert int(version) == L.mxnorm_abi_version() and int(count) == len(names)
    assert rest.startswith(L.mxnorm_status_string(1).decode())
