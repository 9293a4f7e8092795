"""The oracle's multi-threaded casts equal its sequential ones, byte for byte.

The dim0 cast spreads rows and the dim1 cast spreads columns over host
threads (OpenMP); each row or column is computed by the same scalar code
either way, so every output of every entry point built on them must be
identical at 1 thread and at many.  The sequential path is the one the pins
in test_oracle_pins.py check.
"""
import os

import numpy as np
import pytest

import oracle
from mxfp8_block_scaled_dim0_gb300 import workloads as W


@pytest.fixture
def many_threads():
    n = max(2, min(8, os.cpu_count() or 2))
    yield n
    oracle.set_threads(1)


def _both(fn, n):
    oracle.set_threads(1)
    a = fn()
    got = oracle.set_threads(n)
    b = fn()
    oracle.set_threads(1)
    return a, b, got


def _equal(a, b):
    a = a if isinstance(a, tuple) else (a,)
    b = b if isinstance(b, tuple) else (b,)
    assert len(a) == len(b)
    for u, v in zip(a, b):
        assert np.array_equal(np.asarray(u), np.asarray(v))


def test_threads_setting_round_trips(many_threads):
    got = oracle.set_threads(many_threads)
    assert got in (1, many_threads)   # 1: built without OpenMP
    assert oracle.threads() == got
    assert oracle.set_threads(0) == 1  # clamped
    oracle.set_threads(1)


def test_fused_cast_independent_of_threads(many_threads):
    # 1,000 rows do not split evenly over the threads; K spans several tiles.
    x = W.bf16_bits(W.spiky(992, 416, 321, scale_frac=0.05, zero_frac=0.05))
    a, b, _ = _both(lambda: oracle.cast_dim0_dim1_blocked(x), many_threads)
    _equal(a, b)
    a, b, _ = _both(lambda: oracle.cast_dim0(x), many_threads)
    _equal(a, b)
    a, b, _ = _both(lambda: oracle.cast_dim1(x), many_threads)
    _equal(a, b)


def test_grouped_and_3d_independent_of_threads(many_threads):
    x = W.bf16_bits(W.wide(700, 160, 322, zero_frac=0.02))
    offs = np.array([3, 3, 250, 699, 700], np.int32)
    a, b, _ = _both(lambda: oracle.cast_grouped_m(x, offs), many_threads)
    _equal(a, b)
    w = W.bf16_bits(W.experts(3, 96, 160, 323))
    a, b, _ = _both(lambda: oracle.cast_3d_dim0_dim1(w), many_threads)
    _equal(a, b)
