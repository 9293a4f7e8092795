"""The abort paths of the production kernels, driven without any fault.

A stall armed from the host (mx_selftest_arm_stall) makes CTA 0 of the next
launch wait, where it would issue a tile's loads, on a barrier that nothing
completes, with a short limit.  The wait runs out; the CTA stops every role,
lets the copies it has in flight land (TMA loads into its input ring, bulk
stores out of its staging), sets the watchdog word and the kernel returns.
The next call on the same context must be byte-exact.

The stall hook is compiled into the checked build of the library only
(-DMX_DEBUG_BOUNDS, which also checks every thread-issued global store); the
release build's kernels carry no hook (a never-taken check measured up to 4%
on one kernel).  The abort code itself (the roles' wind-down and the drain)
is the same in both builds.  These tests load the checked build and also
require that no store was refused on the way.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import build as mxbuild
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def checked_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    saved = (mx.LIB_PATH, mx._LIB)
    mx.LIB_PATH, mx._LIB = mxbuild.build(bounds=True), None
    try:
        torch.cuda.synchronize()
        assert mx.mx_watchdog(clear=True) == 0
        assert mx.mx_bounds_check(clear=True) == 0
        yield
        torch.cuda.synchronize()
        assert mx.mx_bounds_check(clear=True) == 0
    finally:
        mx.LIB_PATH, mx._LIB = saved


def _fresh():
    torch.cuda.synchronize()
    assert mx.mx_watchdog(clear=True) == 0


def _after_abort():
    t0 = time.time()
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert mx.mx_watchdog(clear=True) == 1       # CTA 0 gave up and said so
    assert mx.mx_watchdog(clear=True) == 0


@pytest.mark.parametrize("at", [0, 27])
def test_claimed_cast_abort_path_then_exact(at):
    """A launch long enough for the claim schedule (8192 x 10240: 33 rounds,
    the last six claimed): CTA 0 gives up before its first tile (at = 0) or
    at its first claimed tile (at = 27; its first claim, made with every other
    CTA's first, always finds a tile).  It never makes its last claim, so the
    launch's counter is not reset by the kernel; clearing the watchdog resets
    it, and the next launch on the stream is byte-exact."""
    _fresh()
    x = W.normal((8192, 10240), 12)
    xb = x.cuda()
    mx.mx_selftest_arm_stall(at, 20_000_000)
    mx.cast_dim0_dim1(xb)
    _after_abort()
    q0, s0, q1, s1 = mx.cast_dim0_dim1(xb)
    torch.cuda.synchronize()
    want = oracle.cast_dim0_dim1_blocked(W.bf16_bits(x))
    for got, ref in zip((q0, s0, q1, s1), want):
        assert np.array_equal(got.cpu().numpy().ravel(), np.asarray(ref).ravel())
    assert mx.mx_watchdog(clear=True) == 0


@pytest.mark.parametrize("at", [0, 2])
def test_fused_cast_abort_path_then_exact(at):
    _fresh()
    # 4096 x 1024: 256 tiles, so CTA 0 runs two (at = 0: before its first
    # tile, with the ring full of loads; at = 2: past its last one, no stall)
    x = W.spiky(4096, 1024, 11, scale_frac=0.05, zero_frac=0.05)
    xb = x.cuda()
    mx.mx_selftest_arm_stall(at, 20_000_000)
    mx.cast_dim0_dim1(xb)
    if at == 0:
        _after_abort()
    else:
        torch.cuda.synchronize()
        assert mx.mx_watchdog(clear=True) == 0   # the armed tile never came: no stall
    q0, s0, q1, s1 = mx.cast_dim0_dim1(xb)
    torch.cuda.synchronize()
    want = oracle.cast_dim0_dim1_blocked(W.bf16_bits(x))
    for got, ref in zip((q0, s0, q1, s1), want):
        assert np.array_equal(got.cpu().numpy().ravel(), np.asarray(ref).ravel())
    assert mx.mx_watchdog(clear=True) == 0


def test_grouped_cast_abort_path_then_exact():
    _fresh()
    # 66 tile-rows x 5 tile-columns = 330 tiles over 152 CTAs in contiguous
    # runs, so CTA 0 owns tiles 0 and 1: it stalls at its second tile, after
    # one tile has gone through all roles; the tail zeroing still runs.
    x = W.wide(8000, 640, 12, zero_frac=0.02)
    offs = torch.tensor([130, 130, 700, 7999, 8000], dtype=torch.int32, device="cuda")
    mx.mx_selftest_arm_stall(1, 20_000_000)
    mx.cast_grouped_m(x.cuda(), offs)
    _after_abort()
    got = mx.cast_grouped_m(x.cuda(), offs)
    torch.cuda.synchronize()
    want = oracle.cast_grouped_m(W.bf16_bits(x), offs.cpu().numpy())
    for i in range(6):
        assert np.array_equal(got[i].cpu().numpy().ravel(), np.asarray(want[i]).ravel()), i
    assert int(got[6].item()) == 0
    assert mx.mx_watchdog(clear=True) == 0


def test_rowwise_abort_path_then_exact():
    _fresh()
    # CTA 0 stalls before its first step, with its ring of bulk copies issued
    x = W.normal((4096, 2048), 13)
    xb = x.cuda()
    mx.mx_selftest_arm_stall(0, 20_000_000)
    mx.cast_rowwise(xb)
    _after_abort()
    q, scale = mx.cast_rowwise(xb)
    torch.cuda.synchronize()
    oq, oscale = oracle.cast_rowwise(W.bf16_bits(x))
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(scale.view(torch.int16).cpu().numpy().view(np.uint16), oscale)
    assert mx.mx_watchdog(clear=True) == 0


def test_dequant_abort_path_then_exact():
    _fresh()
    # 4096 x 1024: 256 tiles of 128 x 128, so CTA 0 runs two; it stalls
    # before its first, with its loads in flight
    x = W.wide(4096, 1024, 14, zero_frac=0.02)
    q0, s0 = mx.cast_dim0(x.cuda())
    mx.mx_selftest_arm_stall(0, 20_000_000)
    mx.dequant_blocked(q0, s0)
    _after_abort()
    d = mx.dequant_blocked(q0, s0)
    torch.cuda.synchronize()
    oq0, os0 = oracle.cast_dim0(W.bf16_bits(x))
    want = oracle.dequant_blocked(oq0, oracle.to_blocked(os0))
    assert np.array_equal(d.view(torch.int16).cpu().numpy().view(np.uint16), want)
    assert mx.mx_watchdog(clear=True) == 0


def test_arm_stall_rejects_bad_arguments():
    lib = mx.library()
    assert lib.mx_selftest_arm_stall(-1, 1_000_000) == mx.MX_ERR_SHAPE
    assert lib.mx_selftest_arm_stall(0, 10) == mx.MX_ERR_SHAPE
