"""Host-side checks of the C ABI library that need no GPU: it builds for
sm_103a, loads, exports every function the header declares, computes sizes,
and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import build as mxbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxfp8_cast.h")


@pytest.fixture(scope="module")
def lib():
    mxbuild.build()
    return mx.library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(mx_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_expected_entry_points():
    fns = header_functions()
    assert set(fns) == set(mx.ABI_SYMBOLS), fns


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_size_helpers(lib):
    assert mx.mx_blocked_bytes(1, 1) == 512
    assert mx.mx_blocked_bytes(128, 4) == 512
    assert mx.mx_blocked_bytes(129, 5) == 256 * 8
    assert mx.mx_blocked_bytes(16384, 512) == 16384 * 512
    assert mx.mx_blocked_bytes(-1, 4) == -1
    # grouped bounds: rows + groups * 128 (dim0), columns ceil(M/32) + 4 G (dim1)
    assert mx.mx_grouped_m_scale_bytes(16640, 5120, 4, 0) == (16640 + 512) * 160
    assert mx.mx_grouped_m_scale_bytes(16640, 5120, 4, 1) == 5120 * (520 + 16)
    assert mx.mx_grouped_m_scale_bytes(16640, 5120, 0, 0) == -1
    assert mx.mx_3d_scale_bytes(16, 8192, 5120) == 16 * 5120 * 256
    assert mx.mx_3d_scale_bytes(2, 96, 160) == 2 * 256 * 4


def test_strerror(lib):
    texts = [lib.mx_strerror(code) for code in (0, -1, -2, -3, -4, -5, -6)]
    assert all(texts) and len(set(texts)) == len(texts)
    assert lib.mx_strerror(-99) == b"unknown error"


def test_error_codes_match_header():
    text = open(HEADER).read()
    codes = dict((k, int(v)) for k, v in re.findall(r"\b(MX_(?:OK|ERR_\w+))\s*=\s*(-?\d+)", text))
    assert codes == {name: getattr(mx, name) for name in codes}
    assert set(codes) == {n for n in dir(mx) if re.fullmatch(r"MX_(OK|ERR_\w+)", n)}


class _OnDevice:
    """Stands in for a CUDA tensor on device `index` (no GPU here)."""

    def __init__(self, index):
        self.index = index

    def get_device(self):
        return self.index


def test_binding_refuses_tensors_on_several_devices():
    assert mx._device(_OnDevice(1), None, _OnDevice(1)) == 1
    with pytest.raises(ValueError, match="one CUDA device"):
        mx._device(_OnDevice(0), _OnDevice(1))


# Fake, never-dereferenced device addresses: argument checks run before any
# CUDA call, so these return without touching a device.
A = 1 << 20          # 16-byte aligned
B = (1 << 20) + 8    # misaligned


def test_cast_rejects_null(lib):
    assert lib.mx_cast_dim0_dim1(None, 64, 64, A, A, A, A, None) == mx.MX_ERR_NULL
    assert lib.mx_cast_dim0_dim1(A, 64, 64, A, None, A, A, None) == mx.MX_ERR_NULL
    assert lib.mx_cast_dim1(A, 64, 64, None, A, None) == mx.MX_ERR_NULL
    assert lib.mx_scales_to_blocked(None, 4, 4, A, None) == mx.MX_ERR_NULL
    assert lib.mx_cast_3d_dim1(A, 2, 64, 64, A, None, None) == mx.MX_ERR_NULL
    assert lib.mx_cast_grouped_m(A, 64, 64, A, 2, A, A, A, A, A, A, None, None) == mx.MX_ERR_NULL


@pytest.mark.parametrize("M,K", [(0, 64), (64, 0), (33, 64), (64, 48), (-32, 64), (1 << 31, 32)])
def test_cast_rejects_shapes(lib, M, K):
    assert lib.mx_cast_dim0_dim1(A, M, K, A, A, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_dim1(A, M, K, A, A, None) == mx.MX_ERR_SHAPE


def test_other_shape_rules(lib):
    assert lib.mx_scales_to_blocked(A, 0, 4, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_3d_dim1(A, 2, 48, 64, A, A, None) == mx.MX_ERR_SHAPE   # N % 32
    assert lib.mx_cast_3d_dim1(A, 0, 64, 64, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_grouped_m(A, 64, 40, A, 2, A, A, A, A, A, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_grouped_m(A, 0, 64, A, 2, A, A, A, A, A, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_grouped_m(A, 64, 64, A, 0, A, A, A, A, A, A, A, None) == mx.MX_ERR_GROUPS


def test_cast_rejects_misalignment(lib):
    assert lib.mx_cast_dim0_dim1(B, 64, 64, A, A, A, A, None) == mx.MX_ERR_ALIGN
    assert lib.mx_cast_dim0_dim1(A, 64, 64, A, A, B, A, None) == mx.MX_ERR_ALIGN
    assert lib.mx_cast_dim1(A, 64, 64, A, B, None) == mx.MX_ERR_ALIGN
    assert lib.mx_scales_to_blocked(A, 4, 4, B, None) == mx.MX_ERR_ALIGN
    assert lib.mx_cast_3d_dim1(A, 2, 64, 64, B, A, None) == mx.MX_ERR_ALIGN
    assert lib.mx_cast_grouped_m(A, 64, 64, A + 2, 2, A, A, A, A, A, A, A, None) == mx.MX_ERR_ALIGN


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(mx, "_LIB", None)
    monkeypatch.setattr(mx, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        mx.library()


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "mxfp8_block_scaled_dim0_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\b(import|from)\s+oracle\b|mx_oracle|oracle_\w+\(", text), f


def test_selftest_watchdog_rejects_bad_limits(lib):
    assert lib.mx_selftest_watchdog(0, None) == mx.MX_ERR_SHAPE
    assert lib.mx_selftest_watchdog(10**11, None) == mx.MX_ERR_SHAPE


def test_new_entry_points_reject_bad_arguments(lib):
    assert mx.mx_3d_dim0_scale_bytes(16, 8192, 5120) == 16 * 8192 * 160
    assert mx.mx_3d_dim0_scale_bytes(2, 50, 96) == 2 * 128 * 4
    assert lib.mx_cast_dim0(None, 64, 64, A, A, None) == mx.MX_ERR_NULL
    assert lib.mx_cast_dim0(A, 0, 64, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_dim0(A, 64, 48, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_dim0(A, 64, 64, B, A, None) == mx.MX_ERR_ALIGN
    assert lib.mx_cast_3d_dim0(A, 2, 64, 64, None, A, None) == mx.MX_ERR_NULL
    assert lib.mx_cast_3d_dim0(A, 2, 0, 64, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_3d_dim0(A, 2, 64, 40, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_3d_dim0(A, 2, 64, 64, A, B, None) == mx.MX_ERR_ALIGN
    assert lib.mx_cast_3d_dim0_dim1(A, 2, 64, 64, A, A, None, A, None) == mx.MX_ERR_NULL
    assert lib.mx_cast_3d_dim0_dim1(A, 2, 50, 64, A, A, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_3d_dim0_dim1(A, 2, 64, 64, A, A, B, A, None) == mx.MX_ERR_ALIGN
    assert lib.mx_dequant_blocked(A, 64, 64, None, A, None) == mx.MX_ERR_NULL
    assert lib.mx_dequant_blocked(A, 0, 64, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_dequant_blocked(A, 64, 48, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_dequant_blocked(A, 64, 64, A, B, None) == mx.MX_ERR_ALIGN


def test_scaled_fp8_entry_points_reject_bad_arguments(lib):
    import ctypes as C
    F = C.c_void_p(A)
    assert lib.mx_cast_tensorwise(None, 64, A, F, F, None) == mx.MX_ERR_NULL
    assert lib.mx_cast_tensorwise(A, 0, A, F, F, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_tensorwise(B, 64, A, F, F, None) == mx.MX_ERR_ALIGN
    assert lib.mx_cast_tensorwise(A, 64, A, C.c_void_p(A + 2), F, None) == mx.MX_ERR_ALIGN
    assert lib.mx_cast_rowwise(A, 64, 64, None, A, None) == mx.MX_ERR_NULL
    assert lib.mx_cast_rowwise(A, 64, 12, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_rowwise(A, 0, 64, A, A, None) == mx.MX_ERR_SHAPE
    assert lib.mx_cast_rowwise(A, 64, 64, B, A, None) == mx.MX_ERR_ALIGN


def test_bounds_entry_points_in_release_build(lib):
    """The release library has no checks compiled in: both report -1 without
    touching a device."""
    assert lib.mx_bounds_check(0) == -1
    assert lib.mx_selftest_bounds(None, None) == mx.MX_ERR_NULL
    assert lib.mx_selftest_bounds(A, None) == -1


def test_stall_hook_only_in_the_checked_build(lib):
    """Arming the diagnostic stall is host-only.  The release build has no
    stall hook and says so (-1); the checked build arms it."""
    assert lib.mx_selftest_arm_stall(0, 1_000_000) == -1
    assert lib.mx_selftest_arm_stall(-1, 1_000_000) == mx.MX_ERR_SHAPE
    blib = ctypes.CDLL(mxbuild.build(bounds=True))
    blib.mx_selftest_arm_stall.argtypes = [ctypes.c_int64, ctypes.c_int64]
    assert blib.mx_selftest_arm_stall(0, 1_000_000) == mx.MX_OK
    assert blib.mx_selftest_arm_stall(0, 10) == mx.MX_ERR_SHAPE


def test_bounds_checked_library_exports_every_symbol():
    path = mxbuild.build(bounds=True)
    blib = ctypes.CDLL(path)
    for name in header_functions():
        assert hasattr(blib, name), name


def test_c_program_compiles_links_and_calls_host_helpers(lib, tmp_path):
    """The header is usable from plain C: a C99 program includes it, links
    against the library and calls the host-only helpers (no GPU needed)."""
    import subprocess
    src = tmp_path / "use_abi.c"
    src.write_text(
        '#include <stdio.h>\n#include "mxfp8_cast.h"\n'
        "int main(void) {\n"
        '  printf("%lld %lld %s\\n", (long long)mx_blocked_bytes(129, 5),\n'
        "         (long long)mx_grouped_m_scale_bytes(16640, 5120, 4, 0),\n"
        "         mx_strerror(MX_ERR_DEVICE));\n"
        "  return mx_cast_dim0_dim1(0, 64, 64, 0, 0, 0, 0, 0) == MX_ERR_NULL ? 0 : 1;\n"
        "}\n")
    exe = tmp_path / "use_abi"
    libdir = os.path.dirname(mx.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lmxfp8_cast",
                    "-Wl,-rpath," + libdir], check=True, capture_output=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split()[:2] == [str(256 * 8), str((16640 + 512) * 160)]
    assert "current" in r.stdout


# ---- the binding's dtype and rank checks ---------------------------------------
#
# The C ABI takes untyped pointers, so a float16 tensor handed over as bf16
# input, or float offsets as int32 group ends, would be read as the wrong bits.
# The binding refuses them; these checks run before any CUDA call, so CPU
# tensors reach them here.

def _bf16(*shape):
    import torch
    return torch.zeros(shape, dtype=torch.bfloat16)


def _u8(n):
    import torch
    return torch.zeros(n, dtype=torch.uint8)


def test_binding_refuses_float16_input(lib):
    import torch
    x = torch.zeros((64, 64), dtype=torch.float16)
    for fn, args in ((mx.mx_cast_dim0_dim1, (_u8(4096), _u8(4096), _u8(4096), _u8(4096))),
                     (mx.mx_cast_dim0, (_u8(4096), _u8(4096))),
                     (mx.mx_cast_dim1, (_u8(4096), _u8(4096))),
                     (mx.mx_cast_rowwise, (_u8(4096), _bf16(64))),
                     (mx.mx_cast_tensorwise, (_u8(4096), torch.zeros(1), torch.zeros(1)))):
        with pytest.raises(TypeError, match="bfloat16"):
            fn(x, *args)
    with pytest.raises(TypeError, match="bfloat16"):
        mx.mx_cast_3d_dim1(torch.zeros((2, 32, 32), dtype=torch.int16), _u8(2048), _u8(4096))


def test_binding_refuses_wrong_offset_and_status_dtypes(lib):
    import torch
    M, K, G = 256, 64, 2
    x = _bf16(M, K)
    n0, n1 = mx.mx_grouped_m_scale_bytes(M, K, G, 0), mx.mx_grouped_m_scale_bytes(M, K, G, 1)
    good = dict(offs=torch.tensor([100, 256], dtype=torch.int32), q0=_u8(M * K), s0=_u8(n0),
                r0=torch.zeros(G + 1, dtype=torch.int64), q1=_u8(M * K), s1=_u8(n1),
                c1=torch.zeros(G + 1, dtype=torch.int64), st=torch.zeros(1, dtype=torch.int32))

    def call(**over):
        a = dict(good, **over)
        mx.mx_cast_grouped_m(x, a["offs"], a["q0"], a["s0"], a["r0"], a["q1"], a["s1"],
                             a["c1"], a["st"])

    with pytest.raises(TypeError, match="int32"):
        call(offs=torch.tensor([100.0, 256.0], dtype=torch.float32))
    with pytest.raises(TypeError, match="int32"):
        call(offs=torch.tensor([100, 256], dtype=torch.int64))
    with pytest.raises(TypeError, match="int64"):
        call(r0=torch.zeros(G + 1, dtype=torch.int32).repeat(2))
    with pytest.raises(TypeError, match="int32"):
        call(st=torch.zeros(1, dtype=torch.float32))
    with pytest.raises(TypeError, match="uint8"):
        call(q0=torch.zeros(M * K, dtype=torch.int8))
    # correct dtypes on the CPU: refused for not being CUDA tensors
    with pytest.raises(ValueError, match="CUDA"):
        call()


def test_binding_refuses_wrong_ranks_and_output_dtypes(lib):
    import torch
    with pytest.raises(ValueError, match="2 dimensions"):
        mx.mx_cast_dim0_dim1(_bf16(2, 64, 64), _u8(1), _u8(1), _u8(1), _u8(1))
    with pytest.raises(ValueError, match="3 dimensions"):
        mx.mx_cast_3d_dim0(_bf16(64, 64), _u8(1), _u8(1))
    with pytest.raises(TypeError, match="float32"):
        mx.mx_cast_tensorwise(_bf16(64), _u8(64), torch.zeros(1, dtype=torch.float64),
                              torch.zeros(1))
    with pytest.raises(TypeError, match="bfloat16"):
        mx.mx_cast_rowwise(_bf16(64, 64), _u8(4096), torch.zeros(64, dtype=torch.float16))
    with pytest.raises(TypeError, match="bfloat16"):
        mx.mx_dequant_blocked(_u8(64 * 64).view(64, 64), _u8(512),
                              torch.zeros((64, 64), dtype=torch.float16))
    # fp8 and e8m0 views of the byte buffers are accepted by the checks
    if hasattr(torch, "float8_e4m3fn"):
        q = torch.zeros((64, 64), dtype=torch.float8_e4m3fn)
        with pytest.raises(ValueError, match="CUDA"):
            mx.mx_dequant_blocked(q, _u8(512), _bf16(64, 64))
