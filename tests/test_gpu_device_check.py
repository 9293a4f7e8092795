"""Pointers that are not device memory of the current device are refused on
the host with MX_ERR_DEVICE before anything is enqueued, leaving the outputs
untouched and no CUDA error behind.  The refused pointer here is always an
output that the kernel writes with plain stores, in pinned host memory (which
is mapped into the device's address space).  The library also accepts memory
from the caching allocator's expandable segments (virtual memory mappings).
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def cuda_only():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _x(M, K, seed):
    bits = W.bf16_bits(W.normal((M, K), seed, std=0.02))
    return bits, torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def test_host_output_refused_then_next_call_is_fine():
    M, K = 128, 256
    bits, x = _x(M, K, 61)
    lib = mx.library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    q0_host = torch.full((M, K), 0xA5, dtype=torch.uint8).pin_memory()
    s0 = torch.full((mx.mx_blocked_bytes(M, K // 32),), 0x5A, dtype=torch.uint8, device="cuda")
    rc = lib.mx_cast_dim0(_p(x), M, K, _p(q0_host), _p(s0), stream)
    assert rc == mx.MX_ERR_DEVICE
    torch.cuda.synchronize()
    assert bool((q0_host == 0xA5).all())
    assert bool((s0 == 0x5A).all())
    # The binding refuses the host tensor before reaching the library.
    with pytest.raises(ValueError, match="CUDA tensor"):
        mx.mx_cast_dim0(x, q0_host, s0)
    # No error is left behind: the same call on device buffers succeeds.
    q0 = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    assert lib.mx_cast_dim0(_p(x), M, K, _p(q0), _p(s0), stream) == mx.MX_OK
    torch.cuda.synchronize()
    oq0, os0 = oracle.cast_dim0(bits)
    assert np.array_equal(q0.cpu().numpy(), oq0)
    assert np.array_equal(oracle.from_blocked(s0.cpu().numpy(), M, K // 32), os0)


def test_host_dequant_output_refused():
    R, C = 128, 128
    lib = mx.library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    q = torch.zeros((R, C), dtype=torch.uint8, device="cuda")
    s = torch.full((mx.mx_blocked_bytes(R, C // 32),), 127, dtype=torch.uint8, device="cuda")
    out_host = torch.full((R, C), 7, dtype=torch.int16).pin_memory()
    assert lib.mx_dequant_blocked(_p(q), R, C, _p(s), _p(out_host), stream) == mx.MX_ERR_DEVICE
    torch.cuda.synchronize()
    assert bool((out_host == 7).all())


_EXPANDABLE = r"""
import numpy as np, torch
import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import workloads as W
M, K = 256, 384
bits = W.bf16_bits(W.normal((M, K), 62, std=0.02))
x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
q0, s0, q1, s1 = mx.cast_dim0_dim1(x)
torch.cuda.synchronize()
oq0, os0, oq1, os1 = oracle.cast_dim0_dim1_blocked(bits)
assert np.array_equal(q0.cpu().numpy(), oq0) and np.array_equal(q1.cpu().numpy(), oq1)
assert np.array_equal(s0.cpu().numpy(), os0) and np.array_equal(s1.cpu().numpy(), os1)
print("expandable ok")
"""


def test_expandable_segments_allocator():
    env = dict(os.environ, PYTORCH_CUDA_ALLOC_CONF="expandable_segments:True")
    r = subprocess.run([sys.executable, "-c", _EXPANDABLE], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "expandable ok" in r.stdout, r.stdout + r.stderr
