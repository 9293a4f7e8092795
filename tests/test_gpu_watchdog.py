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
