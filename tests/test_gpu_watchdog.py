"""Failure detection without a GPU fault: a bounded wait that runs out sets
the device watchdog word, the kernel returns normally, and the context keeps
working (the next cast is still byte-exact)."""
import time

import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()
    assert mx.mx_watchdog(clear=True) == 0
    t0 = time.time()
    mx.mx_selftest_watchdog(50_000_000)          # 50 ms limit
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert mx.mx_watchdog(clear=True) == 1      # the wait gave up and said so
    assert mx.mx_watchdog(clear=True) == 0      # cleared
    x = W.spiky(256, 256, 3)
    q0, s0, q1, s1 = mx.cast_dim0_dim1(x.cuda())
    torch.cuda.synchronize()
    r0, rs0, r1, rs1 = oracle.cast_dim0_dim1_blocked(W.bf16_bits(x))
    assert np.array_equal(q0.cpu().numpy(), r0) and np.array_equal(s1.cpu().numpy(), rs1)
    assert mx.mx_watchdog(clear=True) == 0


# ---- the abort path of the production kernels -----------------------------------
#
# A stall armed from the host makes CTA 0 of the next launch wait, at a chosen
# tile, on a barrier that nothing completes, with a short limit.  The wait
# runs out; the CTA stops every role, lets the TMA loads already issued into
# its input ring (and its bulk stores) land, sets the watchdog word and the
# kernel returns.  The next call on the same context must be byte-exact.

def _fresh():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()
    torch.cuda.synchronize()
    assert mx.mx_watchdog(clear=True) == 0


def _after_abort():
    t0 = time.time()
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert mx.mx_watchdog(clear=True) == 1       # CTA 0 gave up and said so
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
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = mx.library()
    assert lib.mx_selftest_arm_stall(-1, 1_000_000) == mx.MX_ERR_SHAPE
    assert lib.mx_selftest_arm_stall(0, 10) == mx.MX_ERR_SHAPE
