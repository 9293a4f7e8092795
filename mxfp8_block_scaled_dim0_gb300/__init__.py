"""MX-FP8 casts of bf16 matrices on sm_103a (GB300): Python binding.

Thin ctypes layer over the C ABI of ``libmxfp8_cast.so`` (declared in
``include/mxfp8_cast.h``).  Functions named like the C entry points take torch
tensors, check their shapes and that they share one CUDA device, make that
device current for the call, and pass raw device pointers plus its current
CUDA stream; every step of the cast runs in the library's CUDA kernels.  There
is no CPU fallback: if the library has not been built, importing the binding
raises.

Convenience wrappers (``cast_dim0_dim1``, ``cast_dim0``, ``cast_dim1``,
``cast_grouped_m``, ``cast_3d_dim1``, ``cast_3d_dim0``, ``cast_3d_dim0_dim1``,
``scales_to_blocked``, ``dequant_blocked``, ``cast_tensorwise``,
``cast_rowwise``) allocate outputs with torch and call the same entry points.
"""
import ctypes
import functools
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmxfp8_cast.so")

MX_OK = 0
MX_ERR_NULL = -1
MX_ERR_SHAPE = -2
MX_ERR_ALIGN = -3
MX_ERR_CUDA = -4
MX_ERR_GROUPS = -5
MX_ERR_DEVICE = -6

# Every function the header declares, for load checks.
ABI_SYMBOLS = (
    "mx_cast_dim0_dim1", "mx_cast_dim0", "mx_cast_dim1", "mx_scales_to_blocked",
    "mx_cast_grouped_m", "mx_cast_3d_dim1", "mx_cast_3d_dim0", "mx_cast_3d_dim0_dim1",
    "mx_dequant_blocked", "mx_blocked_bytes", "mx_grouped_m_scale_bytes", "mx_3d_scale_bytes",
    "mx_3d_dim0_scale_bytes", "mx_cast_tensorwise", "mx_cast_rowwise", "mx_bounds_check",
    "mx_selftest_bounds",
    "mx_strerror", "mx_last_cuda_error", "mx_watchdog",
    "mx_selftest_watchdog", "mx_selftest_arm_stall", "mx_cast_dim0_dim1_noalloc",
)


class MXError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        msg = "%s failed: %s (%d)" % (where, _lib().mx_strerror(code).decode(), code)
        if code == MX_ERR_CUDA:
            msg += " [cudaError %d]" % _lib().mx_last_cuda_error()
        super().__init__(msg)


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                "libmxfp8_cast.so is not built (expected at %s); build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` or "
                "`python -m mxfp8_block_scaled_dim0_gb300.build`" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        sig = {
            "mx_cast_dim0_dim1": ([P, I64, I64, P, P, P, P, P], ctypes.c_int),
            "mx_cast_dim0": ([P, I64, I64, P, P, P], ctypes.c_int),
            "mx_cast_dim1": ([P, I64, I64, P, P, P], ctypes.c_int),
            "mx_scales_to_blocked": ([P, I64, I64, P, P], ctypes.c_int),
            "mx_cast_grouped_m": ([P, I64, I64, P, I32, P, P, P, P, P, P, P, P], ctypes.c_int),
            "mx_cast_3d_dim1": ([P, I64, I64, I64, P, P, P], ctypes.c_int),
            "mx_cast_3d_dim0": ([P, I64, I64, I64, P, P, P], ctypes.c_int),
            "mx_cast_3d_dim0_dim1": ([P, I64, I64, I64, P, P, P, P, P], ctypes.c_int),
            "mx_dequant_blocked": ([P, I64, I64, P, P, P], ctypes.c_int),
            "mx_cast_tensorwise": ([P, I64, P, P, P, P], ctypes.c_int),
            "mx_cast_rowwise": ([P, I64, I64, P, P, P], ctypes.c_int),
            "mx_blocked_bytes": ([I64, I64], I64),
            "mx_grouped_m_scale_bytes": ([I64, I64, I32, I32], I64),
            "mx_3d_scale_bytes": ([I64, I64, I64], I64),
            "mx_3d_dim0_scale_bytes": ([I64, I64, I64], I64),
            "mx_strerror": ([ctypes.c_int], ctypes.c_char_p),
            "mx_last_cuda_error": ([], ctypes.c_int),
            "mx_watchdog": ([ctypes.c_int], ctypes.c_int),
            "mx_bounds_check": ([ctypes.c_int], ctypes.c_int),
            "mx_selftest_bounds": ([P, P], ctypes.c_int),
            "mx_selftest_watchdog": ([I64, P], ctypes.c_int),
            "mx_selftest_arm_stall": ([I64, I64], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = lib
    return _LIB


def library():
    """The loaded ctypes library (raises ImportError if it is not built)."""
    return _lib()


# ---- marshalling helpers ----------------------------------------------------

def _ptr(t):
    # ctypes converts a plain int (or None) for a c_void_p parameter.
    return t.data_ptr() if t is not None else None


# cudaStream_t (as an int) of a device's current stream; cheaper than
# building a torch.cuda.Stream object per call.  Builds of torch without the
# raw accessor take the public route.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None) or (
    lambda dev: torch.cuda.current_stream(dev).cuda_stream)


def _stream(stream, dev=None):
    """The call's cudaStream_t: `stream` (a torch.cuda.Stream or a raw
    handle), else the current stream of device index `dev` (default: the
    current device)."""
    if stream is None:
        return _raw_stream(torch.cuda.current_device() if dev is None else dev)
    if isinstance(stream, torch.cuda.Stream):
        if dev is not None and stream.device_index != dev:
            raise ValueError("stream is on cuda:%d, the tensors on cuda:%d"
                             % (stream.device_index, dev))
        return stream.cuda_stream
    return int(stream)


def _device(*tensors):
    """Index of the one CUDA device that all the call's tensors live on."""
    devs = {t.get_device() for t in tensors if t is not None}
    if any(d < 0 for d in devs):
        raise ValueError("every tensor of a call must be a CUDA tensor, got %s"
                         % ", ".join(sorted({str(t.device) for t in tensors if t is not None})))
    if len(devs) != 1:
        raise ValueError("all tensors of a call must be on one CUDA device, got %s"
                         % ", ".join("cuda:%d" % d for d in sorted(devs)))
    return devs.pop()


def _call(name, dev, stream, *args):
    """Call entry point `name` with device index `dev` current (the library
    launches on the current device) and the stream appended: by default the
    current stream of that device."""
    fn = getattr(_lib(), name)
    if torch.cuda.current_device() == dev:
        rc = fn(*args, _stream(stream, dev))
    else:
        with torch.cuda.device(dev):
            rc = fn(*args, _stream(stream, dev))
    _check(rc, name)


# dtypes each kind of argument may have.  The C ABI sees only pointers, so
# this is the one place where a float16 tensor passed as bf16 input, or float
# offsets passed as int32 group ends, can be refused.
BF16 = (torch.bfloat16,)
BYTES = tuple(d for d in (torch.uint8, getattr(torch, "float8_e4m3fn", None),
                          getattr(torch, "float8_e8m0fnu", None)) if d is not None)
I32 = (torch.int32,)
I64 = (torch.int64,)
F32 = (torch.float32,)


def _dev_tensor(t, name, nbytes=None, dtypes=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError("%s must have dtype %s, got %s"
                        % (name, " or ".join(str(d) for d in dtypes), t.dtype))
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dimensions, got shape %s" % (name, ndim, tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if nbytes is not None and t.nbytes < nbytes:
        raise ValueError("%s holds %d bytes, needs %d" % (name, t.nbytes, nbytes))
    return t


def _check(rc, where):
    if rc != MX_OK:
        raise MXError(rc, where)


# ---- sizes ------------------------------------------------------------------

# The size helpers are pure functions of their arguments; shapes repeat from
# call to call, so their results are cached on the Python side.
@functools.lru_cache(maxsize=4096)
def mx_blocked_bytes(R, C):
    return int(_lib().mx_blocked_bytes(R, C))


@functools.lru_cache(maxsize=4096)
def mx_grouped_m_scale_bytes(M, K, G, dim):
    return int(_lib().mx_grouped_m_scale_bytes(M, K, G, dim))


@functools.lru_cache(maxsize=4096)
def mx_3d_scale_bytes(E, N, K):
    return int(_lib().mx_3d_scale_bytes(E, N, K))


@functools.lru_cache(maxsize=4096)
def mx_3d_dim0_scale_bytes(E, N, K):
    return int(_lib().mx_3d_dim0_scale_bytes(E, N, K))


# ---- entry points (same names as the C ABI) ----------------------------------

def mx_cast_dim0_dim1(x, q0, s0_blk, q1, s1_blk, stream=None):
    """Fused dim0 + dim1 cast of bf16 x (M x K) into caller buffers."""
    _dev_tensor(x, "x", dtypes=BF16, ndim=2)
    M, K = x.shape
    _dev_tensor(q0, "q0", M * K, BYTES)
    _dev_tensor(q1, "q1", M * K, BYTES)
    _dev_tensor(s0_blk, "s0_blk", mx_blocked_bytes(M, K // 32), BYTES)
    _dev_tensor(s1_blk, "s1_blk", mx_blocked_bytes(K, M // 32), BYTES)
    dev = _device(x, q0, s0_blk, q1, s1_blk)
    _call("mx_cast_dim0_dim1", dev, stream, _ptr(x), M, K, _ptr(q0), _ptr(s0_blk), _ptr(q1),
          _ptr(s1_blk))


def mx_cast_dim0(x, q0, s0_blk, stream=None):
    _dev_tensor(x, "x", dtypes=BF16, ndim=2)
    M, K = x.shape
    _dev_tensor(q0, "q0", M * K, BYTES)
    _dev_tensor(s0_blk, "s0_blk", mx_blocked_bytes(M, K // 32), BYTES)
    _call("mx_cast_dim0", _device(x, q0, s0_blk), stream, _ptr(x), M, K, _ptr(q0), _ptr(s0_blk))


def mx_cast_dim1(x, q1, s1_blk, stream=None):
    _dev_tensor(x, "x", dtypes=BF16, ndim=2)
    M, K = x.shape
    _dev_tensor(q1, "q1", M * K, BYTES)
    _dev_tensor(s1_blk, "s1_blk", mx_blocked_bytes(K, M // 32), BYTES)
    _call("mx_cast_dim1", _device(x, q1, s1_blk), stream, _ptr(x), M, K, _ptr(q1), _ptr(s1_blk))


def mx_scales_to_blocked(s, out, stream=None):
    _dev_tensor(s, "s", dtypes=BYTES, ndim=2)
    R, C = s.shape
    _dev_tensor(out, "out", mx_blocked_bytes(R, C), BYTES)
    _call("mx_scales_to_blocked", _device(s, out), stream, _ptr(s), R, C, _ptr(out))


def mx_cast_grouped_m(x, offs, q0, s0_blk, s0_row_offs, q1, s1_blk, s1_col_offs, status,
                      stream=None):
    _dev_tensor(x, "x", dtypes=BF16, ndim=2)
    M, K = x.shape
    _dev_tensor(offs, "offs", dtypes=I32, ndim=1)
    G = offs.numel()
    _dev_tensor(q0, "q0", M * K, BYTES)
    _dev_tensor(q1, "q1", M * K, BYTES)
    if G >= 1:
        _dev_tensor(s0_blk, "s0_blk", mx_grouped_m_scale_bytes(M, K, G, 0), BYTES)
        _dev_tensor(s1_blk, "s1_blk", mx_grouped_m_scale_bytes(M, K, G, 1), BYTES)
    _dev_tensor(s0_row_offs, "s0_row_offs", 8 * (G + 1), I64)
    _dev_tensor(s1_col_offs, "s1_col_offs", 8 * (G + 1), I64)
    _dev_tensor(status, "status", 4, I32)
    dev = _device(x, offs, q0, s0_blk, s0_row_offs, q1, s1_blk, s1_col_offs, status)
    _call("mx_cast_grouped_m", dev, stream, _ptr(x), M, K, _ptr(offs), G, _ptr(q0), _ptr(s0_blk),
          _ptr(s0_row_offs), _ptr(q1), _ptr(s1_blk), _ptr(s1_col_offs), _ptr(status))


def mx_cast_3d_dim1(w, q1, s1_blk, stream=None):
    _dev_tensor(w, "w", dtypes=BF16, ndim=3)
    E, N, K = w.shape
    _dev_tensor(q1, "q1", E * N * K, BYTES)
    _dev_tensor(s1_blk, "s1_blk", mx_3d_scale_bytes(E, N, K), BYTES)
    dev = _device(w, q1, s1_blk)
    _call("mx_cast_3d_dim1", dev, stream, _ptr(w), E, N, K, _ptr(q1), _ptr(s1_blk))


def mx_cast_3d_dim0(w, q0, s0_blk, stream=None):
    _dev_tensor(w, "w", dtypes=BF16, ndim=3)
    E, N, K = w.shape
    _dev_tensor(q0, "q0", E * N * K, BYTES)
    _dev_tensor(s0_blk, "s0_blk", mx_3d_dim0_scale_bytes(E, N, K), BYTES)
    dev = _device(w, q0, s0_blk)
    _call("mx_cast_3d_dim0", dev, stream, _ptr(w), E, N, K, _ptr(q0), _ptr(s0_blk))


def mx_cast_3d_dim0_dim1(w, q0, s0_blk, q1, s1_blk, stream=None):
    _dev_tensor(w, "w", dtypes=BF16, ndim=3)
    E, N, K = w.shape
    _dev_tensor(q0, "q0", E * N * K, BYTES)
    _dev_tensor(q1, "q1", E * N * K, BYTES)
    _dev_tensor(s0_blk, "s0_blk", mx_3d_dim0_scale_bytes(E, N, K), BYTES)
    _dev_tensor(s1_blk, "s1_blk", mx_3d_scale_bytes(E, N, K), BYTES)
    dev = _device(w, q0, s0_blk, q1, s1_blk)
    _call("mx_cast_3d_dim0_dim1", dev, stream, _ptr(w), E, N, K, _ptr(q0), _ptr(s0_blk), _ptr(q1),
          _ptr(s1_blk))


def mx_dequant_blocked(q, s_blk, out, stream=None):
    """bf16 out (R x C) = e4m3 q (R x C) times 2^(scale - 127), scales in
    blocked layout."""
    _dev_tensor(q, "q", dtypes=BYTES, ndim=2)
    R, C = q.shape
    _dev_tensor(s_blk, "s_blk", mx_blocked_bytes(R, C // 32), BYTES)
    _dev_tensor(out, "out", 2 * R * C, BF16)
    dev = _device(q, s_blk, out)
    _call("mx_dequant_blocked", dev, stream, _ptr(q), R, C, _ptr(s_blk), _ptr(out))


def mx_cast_tensorwise(x, q, scale, amax, stream=None):
    """Tensorwise fp8 of bf16 x (any shape): q (x.numel() bytes), scale and
    amax (one float32 each)."""
    _dev_tensor(x, "x", dtypes=BF16)
    n = x.numel()
    _dev_tensor(q, "q", n, BYTES)
    _dev_tensor(scale, "scale", 4, F32)
    _dev_tensor(amax, "amax", 4, F32)
    dev = _device(x, q, scale, amax)
    _call("mx_cast_tensorwise", dev, stream, _ptr(x), n, _ptr(q), _ptr(scale), _ptr(amax))


def mx_cast_rowwise(x, q, scale, stream=None):
    """Rowwise fp8 of bf16 x (M x K): q (M x K bytes), scale (M bf16)."""
    _dev_tensor(x, "x", dtypes=BF16, ndim=2)
    M, K = x.shape
    _dev_tensor(q, "q", M * K, BYTES)
    _dev_tensor(scale, "scale", 2 * M, BF16)
    _call("mx_cast_rowwise", _device(x, q, scale), stream, _ptr(x), M, K, _ptr(q), _ptr(scale))


def mx_selftest_watchdog(wait_ns=50_000_000, stream=None):
    """Run the bounded-wait failure path on the device (no fault): a warp
    waits on a barrier that never completes and gives up after wait_ns."""
    _check(_lib().mx_selftest_watchdog(int(wait_ns), _stream(stream)), "mx_selftest_watchdog")


def mx_selftest_arm_stall(at, wait_ns=20_000_000):
    """Checked builds: arm a stall for this thread's next cast, tiled
    dequantisation or bulk-staged rowwise launch.  CTA 0 gives up waiting at
    its `at`-th tile and takes the abort path, without any fault (see
    include/mxfp8_cast.h).  A release build has no stall hook."""
    rc = _lib().mx_selftest_arm_stall(int(at), int(wait_ns))
    if rc == -1:
        raise RuntimeError("mx_selftest_arm_stall: release build, no stall hook compiled in")
    _check(rc, "mx_selftest_arm_stall")


def mx_bounds_check(clear=True):
    """Stores refused by a bounds-checked build of the library (-1: release
    build, no checks)."""
    rc = _lib().mx_bounds_check(1 if clear else 0)
    if rc < -1:
        raise MXError(rc, "mx_bounds_check")
    return rc


def mx_selftest_bounds(buf16, stream=None):
    """Bounds-checked builds: one refused store just past an 8-byte span over
    buf16 (a 16-byte CUDA tensor); returns 0, or -1 in a release build."""
    _dev_tensor(buf16, "buf16", 16)
    dev = _device(buf16)
    with torch.cuda.device(dev):
        rc = _lib().mx_selftest_bounds(_ptr(buf16), _stream(stream, dev))
    if rc < -1:
        raise MXError(rc, "mx_selftest_bounds")
    return rc


def mx_watchdog(clear=True):
    rc = _lib().mx_watchdog(1 if clear else 0)
    if rc < 0:
        raise MXError(rc, "mx_watchdog")
    return rc


# ---- allocating wrappers ------------------------------------------------------

def _u8(n, device):
    return torch.empty(n, dtype=torch.uint8, device=device)


def cast_dim0_dim1(x, stream=None):
    """Returns (q0 (M,K), s0_blk, q1 (K,M), s1_blk) as uint8 tensors."""
    M, K = x.shape
    q0 = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    q1 = torch.empty((K, M), dtype=torch.uint8, device=x.device)
    s0 = _u8(mx_blocked_bytes(M, K // 32), x.device)
    s1 = _u8(mx_blocked_bytes(K, M // 32), x.device)
    mx_cast_dim0_dim1(x, q0, s0, q1, s1, stream)
    return q0, s0, q1, s1


def cast_dim0(x, stream=None):
    M, K = x.shape
    q0 = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s0 = _u8(mx_blocked_bytes(M, K // 32), x.device)
    mx_cast_dim0(x, q0, s0, stream)
    return q0, s0


def cast_dim1(x, stream=None):
    M, K = x.shape
    q1 = torch.empty((K, M), dtype=torch.uint8, device=x.device)
    s1 = _u8(mx_blocked_bytes(K, M // 32), x.device)
    mx_cast_dim1(x, q1, s1, stream)
    return q1, s1


def scales_to_blocked(s, stream=None):
    R, C = s.shape
    out = _u8(mx_blocked_bytes(R, C), s.device)
    mx_scales_to_blocked(s, out, stream)
    return out


def cast_grouped_m(x, offs, stream=None):
    """offs: int32 CUDA tensor of cumulative group ends.  Returns
    (q0, s0_blk, s0_row_offs, q1, s1_blk, s1_col_offs, status)."""
    M, K = x.shape
    G = offs.numel()
    dev = x.device
    q0 = torch.empty((M, K), dtype=torch.uint8, device=dev)
    q1 = torch.empty((K, M), dtype=torch.uint8, device=dev)
    s0 = _u8(mx_grouped_m_scale_bytes(M, K, G, 0), dev)
    s1 = _u8(mx_grouped_m_scale_bytes(M, K, G, 1), dev)
    r0 = torch.empty(G + 1, dtype=torch.int64, device=dev)
    c1 = torch.empty(G + 1, dtype=torch.int64, device=dev)
    st = torch.empty(1, dtype=torch.int32, device=dev)
    mx_cast_grouped_m(x, offs, q0, s0, r0, q1, s1, c1, st, stream)
    return q0, s0, r0, q1, s1, c1, st


def cast_3d_dim1(w, stream=None):
    E, N, K = w.shape
    q1 = torch.empty((K, E * N), dtype=torch.uint8, device=w.device)
    s1 = _u8(mx_3d_scale_bytes(E, N, K), w.device)
    mx_cast_3d_dim1(w, q1, s1, stream)
    return q1, s1


def cast_3d_dim0(w, stream=None):
    """Returns (q0 (E, N, K), s0_blk) as uint8 tensors."""
    E, N, K = w.shape
    q0 = torch.empty((E, N, K), dtype=torch.uint8, device=w.device)
    s0 = _u8(mx_3d_dim0_scale_bytes(E, N, K), w.device)
    mx_cast_3d_dim0(w, q0, s0, stream)
    return q0, s0


def cast_3d_dim0_dim1(w, stream=None):
    """Returns (q0 (E, N, K), s0_blk, q1 (K, E*N), s1_blk)."""
    E, N, K = w.shape
    q0 = torch.empty((E, N, K), dtype=torch.uint8, device=w.device)
    q1 = torch.empty((K, E * N), dtype=torch.uint8, device=w.device)
    s0 = _u8(mx_3d_dim0_scale_bytes(E, N, K), w.device)
    s1 = _u8(mx_3d_scale_bytes(E, N, K), w.device)
    mx_cast_3d_dim0_dim1(w, q0, s0, q1, s1, stream)
    return q0, s0, q1, s1


def dequant_blocked(q, s_blk, stream=None):
    """bf16 tensor of the same shape as the 2D uint8 tensor q."""
    R, C = q.shape
    out = torch.empty((R, C), dtype=torch.bfloat16, device=q.device)
    mx_dequant_blocked(q, s_blk, out, stream)
    return out


def cast_tensorwise(x, stream=None):
    """Returns (q uint8 shaped like x, scale float32 (1,), amax float32 (1,))."""
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scale = torch.empty(1, dtype=torch.float32, device=x.device)
    amax = torch.empty(1, dtype=torch.float32, device=x.device)
    mx_cast_tensorwise(x, q, scale, amax, stream)
    return q, scale, amax


def cast_rowwise(x, stream=None):
    """Returns (q (M, K) uint8, scale (M,) bfloat16)."""
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    scale = torch.empty(M, dtype=torch.bfloat16, device=x.device)
    mx_cast_rowwise(x, q, scale, stream)
    return q, scale
