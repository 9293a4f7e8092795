"""Parity cases through the bounds-checked build of the library
(-DMX_DEBUG_BOUNDS): every global store the kernels issue is checked against
its output buffer, and a store that would leave it is refused and counted.
Every case must match the oracle and the count must stay zero; a self-test
shows that a store past its buffer is refused and counted.  The device-side
stand-in for a memory checker, which this machine pool does not offer.
"""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import build as mxbuild
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def bounds_library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    saved = (mx.LIB_PATH, mx._LIB)
    mx.LIB_PATH, mx._LIB = mxbuild.build(bounds=True), None
    try:
        assert mx.mx_bounds_check(clear=True) == 0
        yield
        torch.cuda.synchronize()
    finally:
        mx.LIB_PATH, mx._LIB = saved


def eq(got, want, what):
    g = got.detach().cpu().contiguous().view(torch.uint8).numpy().ravel()
    w = np.ascontiguousarray(want).view(np.uint8).ravel()
    assert np.array_equal(g, w), what


def no_refused_stores():
    torch.cuda.synchronize()
    assert mx.mx_bounds_check(clear=True) == 0


@pytest.mark.parametrize("M,K", [(32, 32), (160, 96), (544, 1056), (96, 4128)])
def test_fused_dim0_dim1_in_bounds(M, K):
    x = W.spiky(M, K, M + K, scale_frac=0.05, zero_frac=0.05)
    got = mx.cast_dim0_dim1(x.cuda())
    want = oracle.cast_dim0_dim1_blocked(W.bf16_bits(x))
    for name, g, w in zip(("q0", "s0", "q1", "s1"), got, want):
        eq(g, w, name)
    q0, s0, _, _ = got
    eq(mx.dequant_blocked(q0, s0), oracle.dequant_blocked(want[0], want[1]), "dequant")
    eq(mx.cast_dim1(x.cuda())[0], want[2], "dim1 only")
    no_refused_stores()


def test_dim0_only_and_blocking_in_bounds():
    x = W.wide(77, 96, 5)
    q0, s0 = mx.cast_dim0(x.cuda())
    oq, os_ = oracle.cast_dim0(W.bf16_bits(x))
    eq(q0, oq, "q0")
    eq(s0, oracle.to_blocked(os_), "s0")
    s = torch.randint(0, 256, (300, 17), dtype=torch.uint8)
    eq(mx.scales_to_blocked(s.cuda()), oracle.to_blocked(s.numpy()), "blocked")
    no_refused_stores()


@pytest.mark.parametrize("M,K,offs", [
    (300, 160, [1, 45, 45, 190, 300]),
    (4224, 640, [0, 1000, 1000, 2999, 4224, 4224]),
    (4097, 2048, None),                          # odd M: every q1 row piecewise
    (3000, 256, "many"),                         # more than 1024 groups: offsets kernel
])
def test_grouped_in_bounds(M, K, offs):
    if offs is None:
        offs = W.group_ends(M, 3, 33, min_size=0).tolist()
    elif offs == "many":
        offs = sorted(np.random.default_rng(7).integers(0, M, 1499).tolist()) + [M]
    x = W.wide(M, K, M + 3 * K, zero_frac=0.01)
    got = mx.cast_grouped_m(x.cuda(), torch.tensor(offs, dtype=torch.int32, device="cuda"))
    want = oracle.cast_grouped_m(W.bf16_bits(x), np.array(offs, np.int32))
    for i, name in enumerate(("q0", "s0", "r0", "q1", "s1", "c1")):
        eq(got[i], want[i], name)
    assert int(got[6].item()) == 0
    no_refused_stores()


def test_grouped_banded_in_bounds():
    """A shape whose CTA runs reach 64 tiles takes the banded grouped kernel:
    40960 x 4096 with a 30000-row group (banded) and a 10960-row group (one
    band)."""
    import os
    M, K = 40960, 4096
    offs = [30000, 40960]
    x = W.normal((M, K), 41, device="cuda")
    got = mx.cast_grouped_m(x, torch.tensor(offs, dtype=torch.int32, device="cuda"))
    oracle.set_threads(os.cpu_count() or 1)
    try:
        want = oracle.cast_grouped_m(W.bf16_bits(x), np.array(offs, np.int32))
    finally:
        oracle.set_threads(1)
    for i, name in enumerate(("q0", "s0", "r0", "q1", "s1", "c1")):
        eq(got[i], want[i], name)
    assert int(got[6].item()) == 0
    no_refused_stores()


@pytest.mark.parametrize("E,N,K", [(2, 96, 160), (3, 256, 160), (3, 50, 96)])
def test_3d_in_bounds(E, N, K):
    w = W.experts(E, N, K, E * N + K)
    bits = W.bf16_bits(w)
    q0, s0 = mx.cast_3d_dim0(w.cuda())
    oq0, os0 = oracle.cast_3d_dim0(bits)
    eq(q0, oq0, "q0")
    eq(s0, os0, "s0")
    if N % 32 == 0:
        got = mx.cast_3d_dim0_dim1(w.cuda())
        for name, g, want in zip(("q0", "s0", "q1", "s1"), got, oracle.cast_3d_dim0_dim1(bits)):
            eq(g, want, name)
        q1, s1 = mx.cast_3d_dim1(w.cuda())
        oq1, os1 = oracle.cast_3d_dim1(bits)
        eq(q1, oq1, "q1")
        eq(s1, os1, "s1")
    no_refused_stores()


# Rowwise launch shapes: 8 rows per step (8 and 6 stages), 2 rows per step,
# three 32 KB stages with a one-row last step, and the re-reading kernel.
@pytest.mark.parametrize("M,K", [(1, 8), (77, 96), (1000, 512), (37, 8200), (39001, 2048),
                                 (3, 24584)])
def test_scaled_fp8_in_bounds(M, K):
    x = W.wide(M, K, 7 * M + K, zero_frac=0.02)
    bits = W.bf16_bits(x)
    q, scale = mx.cast_rowwise(x.cuda())
    oq, oscale = oracle.cast_rowwise(bits)
    eq(q, oq, "rowwise q")
    eq(scale, oscale, "rowwise scale")
    tq, tscale, tamax = mx.cast_tensorwise(x.cuda())
    oq, oscale, oamax = oracle.cast_tensorwise(bits)
    eq(tq, oq, "tensorwise q")
    assert np.float32(tscale.item()) == oscale and np.float32(tamax.item()) == oamax
    no_refused_stores()


def test_out_of_bounds_store_is_refused_and_counted():
    no_refused_stores()
    buf = torch.full((16,), 0xA5, dtype=torch.uint8, device="cuda")
    assert mx.mx_selftest_bounds(buf) == 0
    torch.cuda.synchronize()
    assert mx.mx_bounds_check(clear=True) == 1
    assert torch.all(buf == 0xA5)
    no_refused_stores()
