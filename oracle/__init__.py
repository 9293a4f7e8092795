"""CPU oracle for MX-FP8 casting (ctypes binding over ``mx_oracle.c``).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
and its Python binding never import it; the two share no code.

Every function takes and returns numpy arrays on the host:
  * bf16 inputs are ``uint16`` arrays of raw bit patterns;
  * fp8 e4m3 data and e8m0 scales are ``uint8`` arrays of raw bytes.

The rule (per 32-element block, OCP MX v1.0 conversion with E4M3 elements and
an E8M0 scale): shared exponent floor(log2(amax)) - 8 clamped to [-127, 127]
and biased by 127, zero block -> 0, elements x * 2^-e rounded to the nearest
e4m3 value (ties to even) and saturated to +-448.  Directions and tiling
follow pytorch/ao PR #1869 "triton kernel to cast to mx across dim0 and dim1"
(summary); grouped and 3D variants follow pytorch/ao PR #2990
"[mxfp8 moe training] add compile support" (padding bound, 3D via reshape).
"""
import ctypes

import numpy as np

from . import build as _build

_lib = None


def _configure(lib):
    """Declare the argument and result types of every oracle entry point."""
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_e4m3_rne_sat.argtypes = [ctypes.c_double]
    lib.oracle_e4m3_rne_sat.restype = ctypes.c_uint8
    lib.oracle_e4m3_rne_sat_array.argtypes = [P, I64, P]
    lib.oracle_e4m3_rne_sat_array.restype = None
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_block_scale.argtypes = [P, ctypes.c_int]
    lib.oracle_block_scale.restype = ctypes.c_uint8
    lib.oracle_cast_dim0.argtypes = [P, I64, I64, P, P]
    lib.oracle_cast_dim0.restype = None
    lib.oracle_cast_dim1.argtypes = [P, I64, I64, P, P]
    lib.oracle_cast_dim1.restype = None
    lib.oracle_blocked_bytes.argtypes = [I64, I64]
    lib.oracle_blocked_bytes.restype = I64
    lib.oracle_to_blocked.argtypes = [P, I64, I64, P]
    lib.oracle_to_blocked.restype = None
    lib.oracle_from_blocked.argtypes = [P, I64, I64, P]
    lib.oracle_from_blocked.restype = None
    lib.oracle_cast_dim0_dim1_blocked.argtypes = [P, I64, I64, P, P, P, P]
    lib.oracle_cast_dim0_dim1_blocked.restype = ctypes.c_int
    lib.oracle_cast_grouped_m.argtypes = [P, I64, I64, P, ctypes.c_int,
                                          P, P, P, P, P, P]
    lib.oracle_cast_grouped_m.restype = ctypes.c_int
    lib.oracle_cast_3d_dim1.argtypes = [P, I64, I64, I64, P, P]
    lib.oracle_cast_3d_dim1.restype = ctypes.c_int
    lib.oracle_cast_3d_dim0.argtypes = [P, I64, I64, I64, P, P]
    lib.oracle_cast_3d_dim0.restype = ctypes.c_int
    lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
    lib.oracle_double_to_bf16.restype = ctypes.c_uint16
    lib.oracle_dequant_blocked.argtypes = [P, I64, I64, P, P]
    lib.oracle_dequant_blocked.restype = ctypes.c_int
    lib.oracle_cast_tensorwise.argtypes = [P, I64, P, P, P]
    lib.oracle_cast_tensorwise.restype = None
    lib.oracle_cast_rowwise.argtypes = [P, I64, I64, P, P]
    lib.oracle_cast_rowwise.restype = None
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_threads.restype = None
    lib.oracle_threads.argtypes = []
    lib.oracle_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(_build.build()))
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _bits(x):
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("bf16 input must be a uint16 array of bit patterns")
    return x


def _cdiv(a, b):
    return -(-a // b)


# ---- host threads ---------------------------------------------------------------

def set_threads(n: int) -> int:
    """Spread the dim0 / dim1 casts (and every call built on them) over n
    host threads; returns the count in effect (1 if the library was built
    without OpenMP).  The result does not depend on it."""
    lib = _load()
    lib.oracle_set_threads(int(n))
    return int(lib.oracle_threads())


def threads() -> int:
    return int(_load().oracle_threads())


# ---- scalar encodings -------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def e4m3_rne_sat(v: float) -> int:
    """e4m3fn byte of v: nearest, ties to even, saturated to +-448."""
    return int(_load().oracle_e4m3_rne_sat(float(v)))


def e4m3_rne_sat_array(v):
    """Element-wise e4m3_rne_sat of a float64 array (uint8 result)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_rne_sat_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_to_double(b: int) -> float:
    return _load().oracle_e4m3_to_double(int(b))


def block_scale(values) -> int:
    """e8m0 byte of one block given as real values (float64)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    return int(_load().oracle_block_scale(_ptr(v), v.size))


# ---- whole-matrix casts ------------------------------------------------------

def cast_dim0(x):
    """(M, K) bf16 bits -> q0 (M, K) e4m3 bytes, plain scales (M, K/32)."""
    x = _bits(x)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((M, K // 32), np.uint8)
    _load().oracle_cast_dim0(_ptr(x), M, K, _ptr(q), _ptr(s))
    return q, s


def cast_dim1(x):
    """(M, K) bf16 bits -> q1 (K, M) e4m3 bytes, plain scales (K, M/32)."""
    x = _bits(x)
    M, K = x.shape
    q = np.empty((K, M), np.uint8)
    s = np.empty((K, M // 32), np.uint8)
    _load().oracle_cast_dim1(_ptr(x), M, K, _ptr(q), _ptr(s))
    return q, s


def blocked_bytes(R: int, C: int) -> int:
    return int(_load().oracle_blocked_bytes(R, C))


def to_blocked(s):
    """Plain scales (R, C) -> 1-D blocked layout of blk(R, C) bytes."""
    s = np.ascontiguousarray(s, dtype=np.uint8)
    R, C = s.shape
    out = np.empty(blocked_bytes(R, C), np.uint8)
    _load().oracle_to_blocked(_ptr(s), R, C, _ptr(out))
    return out


def from_blocked(blk, R: int, C: int):
    blk = np.ascontiguousarray(blk, dtype=np.uint8)
    if blk.size < blocked_bytes(R, C):
        raise ValueError("blocked buffer too small")
    s = np.empty((R, C), np.uint8)
    _load().oracle_from_blocked(_ptr(blk), R, C, _ptr(s))
    return s


def cast_dim0_dim1_blocked(x, dim0=True, dim1=True):
    """Fused cast: returns (q0, s0_blk, q1, s1_blk); skipped parts are None."""
    x = _bits(x)
    M, K = x.shape
    q0 = np.empty((M, K), np.uint8) if dim0 else None
    s0 = np.empty(blocked_bytes(M, K // 32), np.uint8) if dim0 else None
    q1 = np.empty((K, M), np.uint8) if dim1 else None
    s1 = np.empty(blocked_bytes(K, M // 32), np.uint8) if dim1 else None
    null = ctypes.c_void_p(0)
    rc = _load().oracle_cast_dim0_dim1_blocked(
        _ptr(x), M, K,
        _ptr(q0) if dim0 else null, _ptr(s0) if dim0 else null,
        _ptr(q1) if dim1 else null, _ptr(s1) if dim1 else null)
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return q0, s0, q1, s1


def grouped_m_scale_bytes(M: int, K: int, G: int, dim: int) -> int:
    if dim == 0:
        return (M + 128 * G) * _cdiv(K // 32, 4) * 4
    return _cdiv(K, 128) * 128 * (_cdiv(M, 32) + 4 * G)


def cast_grouped_m(x, offs):
    """Groups along M.  offs: int32 cumulative group ends (last == M).
    Returns q0, s0_blk, s0_row_offs, q1, s1_blk, s1_col_offs."""
    x = _bits(x)
    M, K = x.shape
    offs = np.ascontiguousarray(offs, dtype=np.int32)
    G = offs.size
    q0 = np.empty((M, K), np.uint8)
    q1 = np.empty((K, M), np.uint8)
    s0 = np.empty(grouped_m_scale_bytes(M, K, G, 0), np.uint8)
    s1 = np.empty(grouped_m_scale_bytes(M, K, G, 1), np.uint8)
    r0 = np.empty(G + 1, np.int64)
    c1 = np.empty(G + 1, np.int64)
    rc = _load().oracle_cast_grouped_m(_ptr(x), M, K, _ptr(offs), G,
                                       _ptr(q0), _ptr(s0), _ptr(r0),
                                       _ptr(q1), _ptr(s1), _ptr(c1))
    if rc == -5:
        raise ValueError("invalid group offsets")
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return q0, s0, r0, q1, s1, c1


def cast_3d_dim1(w):
    """(E, N, K) bf16 bits -> q1 (K, E*N) bytes and E per-expert blocked
    scale tiles concatenated (E * blk(K, N/32) bytes)."""
    w = _bits(w)
    E, N, K = w.shape
    q1 = np.empty((K, E * N), np.uint8)
    s1 = np.empty(E * blocked_bytes(K, N // 32), np.uint8)
    rc = _load().oracle_cast_3d_dim1(_ptr(w), E, N, K, _ptr(q1), _ptr(s1))
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return q1, s1


def cast_3d_dim0(w):
    """(E, N, K) bf16 bits -> q0 (E, N, K) bytes and E per-expert blocked
    scale tiles concatenated (E * blk(N, K/32) bytes)."""
    w = _bits(w)
    E, N, K = w.shape
    q0 = np.empty((E, N, K), np.uint8)
    s0 = np.empty(E * blocked_bytes(N, K // 32), np.uint8)
    rc = _load().oracle_cast_3d_dim0(_ptr(w), E, N, K, _ptr(q0), _ptr(s0))
    if rc != 0:
        raise MemoryError("oracle scratch allocation failed")
    return q0, s0


def cast_3d_dim0_dim1(w):
    """Both directions of a 3D weight: (q0, s0_blk) of cast_3d_dim0 and
    (q1, s1_blk) of cast_3d_dim1."""
    return cast_3d_dim0(w) + cast_3d_dim1(w)


# ---- dequantisation ---------------------------------------------------------

def double_to_bf16(v: float) -> int:
    return int(_load().oracle_double_to_bf16(float(v)))


def dequant_blocked(q, s_blk):
    """q (R, C) e4m3 bytes with blocked scales blk(R, C/32) -> (R, C) bf16
    bits: element value times 2^(scale - 127), rounded once to bf16."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    R, C = q.shape
    s_blk = np.ascontiguousarray(s_blk, dtype=np.uint8).reshape(-1)
    if C % 32 or s_blk.size < blocked_bytes(R, C // 32):
        raise ValueError("C must be a multiple of 32 and s_blk hold blk(R, C/32) bytes")
    out = np.empty((R, C), np.uint16)
    if _load().oracle_dequant_blocked(_ptr(q), R, C, _ptr(s_blk), _ptr(out)) != 0:
        raise MemoryError("oracle scratch allocation failed")
    return out


# ---- tensorwise and rowwise fp8 ---------------------------------------------

def cast_tensorwise(x):
    """bf16 bits (any shape) -> (q uint8 of the same shape, scale float32,
    amax float32): one scale 448 / amax for the whole tensor."""
    x = _bits(x)
    q = np.empty(x.shape, np.uint8)
    scale = np.zeros(1, np.float32)
    amax = np.zeros(1, np.float32)
    _load().oracle_cast_tensorwise(_ptr(x), x.size, _ptr(q), _ptr(scale), _ptr(amax))
    return q, scale[0], amax[0]


def cast_rowwise(x):
    """(M, K) bf16 bits -> (q (M, K) uint8, scale (M,) bf16 bits): one scale
    amax / 448 per row, rounded to bf16."""
    x = _bits(x)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    scale = np.empty(M, np.uint16)
    _load().oracle_cast_rowwise(_ptr(x), M, K, _ptr(q), _ptr(scale))
    return q, scale


def library_path() -> str:
    return _build.build()


__all__ = [
    "bf16_to_double", "e4m3_rne_sat", "e4m3_rne_sat_array", "e4m3_to_double", "block_scale",
    "cast_dim0", "cast_dim1", "blocked_bytes", "to_blocked", "from_blocked",
    "cast_dim0_dim1_blocked", "grouped_m_scale_bytes", "cast_grouped_m",
    "cast_3d_dim1", "cast_3d_dim0", "cast_3d_dim0_dim1", "double_to_bf16",
    "dequant_blocked", "cast_tensorwise", "cast_rowwise", "library_path",
]
