"""mx_cast_dim0_dim1_noalloc: the fused cast for callers that must not
allocate device memory, checked against mx_cast_dim0_dim1.

Such callers are, for instance, processes whose GPU memory a framework's
caching allocator reserved up front (an allocation from outside its pool can
fail or fragment it), or code that must not risk the device-wide
synchronisation an allocation can bring.  This entry point keeps its one
piece of scratch, the tile-claim counter of long launches, in device memory
that the library reserves when it is loaded.

Each test makes two calls in a row on one stream, through the C ABI, and
requires exactly the bytes that mx_cast_dim0_dim1 gives for the same input:
the second call finds the scratch as the first left it and must still start
from a cleared counter.  The outputs are filled with other bytes before each
call.  This file is collected last, so that a run that stops at its first
failure has run every other test before it.
"""
import ctypes

import pytest
import torch

import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()
    yield
    torch.cuda.synchronize()
    assert mx.mx_watchdog(clear=True) == 0


def _entry():
    fn = mx.library().mx_cast_dim0_dim1_noalloc
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    fn.argtypes = [P, I64, I64, P, P, P, P, P]
    fn.restype = ctypes.c_int
    return fn


def _buffers(M, K, fill):
    dev = "cuda"
    return (torch.full((M, K), fill, dtype=torch.uint8, device=dev),
            torch.full((mx.mx_blocked_bytes(M, K // 32),), fill, dtype=torch.uint8, device=dev),
            torch.full((K, M), fill, dtype=torch.uint8, device=dev),
            torch.full((mx.mx_blocked_bytes(K, M // 32),), fill, dtype=torch.uint8, device=dev))


# 8192 x 10240: 5120 tiles, 33 rounds on 152 SMs, so the call claims its last
# tiles through the scratch counter; 1024 x 2048: too short to claim, no
# scratch used.
@pytest.mark.parametrize("M, K", [(8192, 10240), (1024, 2048)])
def test_two_calls_in_a_row_match_mx_cast_dim0_dim1(M, K):
    fn = _entry()
    st = torch.cuda.current_stream()
    for i in range(2):
        x = W.normal((M, K), 4100 + 10 * i + M // 1024, device="cuda")
        want = _buffers(M, K, 0)
        mx.mx_cast_dim0_dim1(x, *want, stream=st)
        got = _buffers(M, K, 0x5A)
        rc = fn(x.data_ptr(), M, K, *(t.data_ptr() for t in got), st.cuda_stream)
        assert rc == 0, "call %d returned %d" % (i, rc)
        torch.cuda.synchronize()
        for name, g, w in zip(("q0", "s0_blk", "q1", "s1_blk"), got, want):
            assert torch.equal(g, w), "call %d: %s differs from mx_cast_dim0_dim1" % (i, name)
