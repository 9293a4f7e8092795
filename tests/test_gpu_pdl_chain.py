"""Kernels launched back to back on one stream, each reading what the one
before it wrote.

Every cast and dequantisation kernel starts as a programmatic dependent of
the previous launch on its stream and, before it waits for that launch to
finish, asks L2 for the first tiles it will read.  In these chains the
previous launch is the writer of exactly those tiles, into buffers that held
other data before, with no host synchronisation in between; the end of each
chain is compared with the oracle on every byte.  A read that saw a buffer's
old contents would show as wrong bytes.  The buffers are about the size of L2
(128 MiB of bf16), so that lines are both prefetched and evicted.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_and_threads():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()
    assert mx.mx_watchdog(clear=True) == 0
    oracle.set_threads(os.cpu_count() or 1)
    yield
    oracle.set_threads(1)
    torch.cuda.synchronize()
    assert mx.mx_watchdog(clear=True) == 0


def u8(n):
    return torch.empty(n, dtype=torch.uint8, device="cuda")


def same(got, want, what):
    g = got.detach().cpu().contiguous().view(torch.uint8).numpy().ravel()
    w = np.ascontiguousarray(want).view(np.uint8).ravel()
    assert g.shape == w.shape, (what, g.shape, w.shape)
    bad = np.flatnonzero(g != w)
    assert bad.size == 0, "%s: %d of %d bytes differ, first at %d" % (what, bad.size, g.size, bad[0])


def test_dequant_then_fused_cast():
    """dequant writes x; the fused cast reads x right behind it."""
    M, K = 4096, 16384
    q_a, s_a = mx.cast_dim0(W.normal((M, K), 2101, device="cuda"))
    x = W.normal((M, K), 2102, device="cuda", std=3.0)          # old contents
    q0, s0 = u8(M * K), u8(mx.mx_blocked_bytes(M, K // 32))
    q1, s1 = u8(M * K), u8(mx.mx_blocked_bytes(K, M // 32))
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    mx.mx_dequant_blocked(q_a, s_a, x, stream=st)
    mx.mx_cast_dim0_dim1(x, q0, s0, q1, s1, stream=st)
    torch.cuda.synchronize()
    xd = oracle.dequant_blocked(q_a.cpu().numpy(), s_a.cpu().numpy())
    same(x, xd, "dequantised x")
    for name, g, w in zip(("q0", "s0", "q1", "s1"), (q0, s0, q1, s1),
                          oracle.cast_dim0_dim1_blocked(xd)):
        same(g, w, "cast of the dequantised x: " + name)


def test_cast_then_dequant():
    """The dim0 cast writes q and its scales over other bytes; dequantisation
    reads them right behind it."""
    M, K = 4096, 16384
    a = W.normal((M, K), 2103, device="cuda")
    q = torch.full((M, K), 0x7E, dtype=torch.uint8, device="cuda")   # old contents
    s = torch.full((mx.mx_blocked_bytes(M, K // 32),), 0x90, dtype=torch.uint8, device="cuda")
    out = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    mx.mx_cast_dim0(a, q, s, stream=st)
    mx.mx_dequant_blocked(q, s, out, stream=st)
    torch.cuda.synchronize()
    oq, os_ = oracle.cast_dim0(W.bf16_bits(a))
    os_blk = oracle.to_blocked(os_)
    same(q, oq, "q")
    same(s, os_blk, "blocked scales")
    same(out, oracle.dequant_blocked(oq, os_blk), "dequantised")


def test_dequant_then_grouped_cast():
    """dequant writes x; the grouped cast (misaligned group starts) reads it
    right behind it, three times in a row with different contents."""
    M, K = 8000, 2048
    offs = torch.tensor([1000, 1003, 4444, 8000], dtype=torch.int32, device="cuda")
    x = W.normal((M, K), 2104, device="cuda", std=5.0)          # old contents
    st = torch.cuda.current_stream()
    for i in range(3):
        q_a, s_a = mx.cast_dim0(W.normal((M, K), 2110 + i, device="cuda"))
        torch.cuda.synchronize()
        mx.mx_dequant_blocked(q_a, s_a, x, stream=st)
        got = mx.cast_grouped_m(x, offs, stream=st)
        torch.cuda.synchronize()
        assert int(got[6].item()) == 0
        xd = oracle.dequant_blocked(q_a.cpu().numpy(), s_a.cpu().numpy())
        want = oracle.cast_grouped_m(xd, offs.cpu().numpy())
        for name, g, w in zip(("q0", "s0", "s0_row_offs", "q1", "s1", "s1_col_offs"), got, want):
            same(g, w, "step %d %s" % (i, name))
