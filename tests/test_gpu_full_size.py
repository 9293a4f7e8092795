"""Full-size parity: the two largest workloads against the oracle, every byte.

  square16384_weight   (16384, 16384) bf16, the benchmark's workload and launch
                       (mx_cast_dim0_dim1): q0, q1 and both padded blocked
                       scale buffers
  experts16x8192x5120  (16, 8192, 5120) bf16 expert weights: the per-expert
                       dim1 cast (mx_cast_3d_dim1), and the dim0 and fused
                       dim0 + dim1 casts of the same weights
  grouped, tall group  (65536, 5120) MoE activations in 3 groups, one of them
                       tall enough for the grouped kernel's banded tile order;
                       and (400000, 512) in 1101 groups (banded order with the
                       group table in global memory)

The inputs are generated on the GPU (the same recipe as on the CPU, drawn by
the CUDA generator), copied to the host once, and cast by the oracle spread
over every host core (its result does not depend on the thread count; see
test_oracle_threads.py).  The transpose property dim1(X) == dim0(X^T) is
checked on top, between two full-size GPU launches.  Shapes from pytorch/ao
PR #1869 "triton kernel to cast to mx across dim0 and dim1" (summary: MKN up
to 16384) and PR #2990 "[mxfp8 moe training] add compile support"
(microbenchmark table and perf analysis: B = (E, 8192, 5120)).
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


def assert_bytes_equal(got, want, what):
    got = np.asarray(got).ravel()
    want = np.asarray(want).ravel()
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if np.array_equal(got, want):
        return
    bad = np.flatnonzero(got != want)
    i = bad[0]
    raise AssertionError("%s: %d of %d bytes differ; first at %d: got %#x want %#x"
                         % (what, bad.size, got.size, i, got[i], want[i]))


def to_np(t):
    return t.detach().cpu().numpy()


def test_square16384_weight_every_byte_and_transpose_property():
    x = W.make("square16384_weight", device="cuda")["x"]
    M, K = x.shape
    q0, s0, q1, s1 = mx.cast_dim0_dim1(x)
    torch.cuda.synchronize()
    oq0, os0, oq1, os1 = oracle.cast_dim0_dim1_blocked(W.bf16_bits(x))
    assert_bytes_equal(to_np(q0), oq0, "q0")
    assert_bytes_equal(to_np(s0), os0, "s0 blocked")
    assert_bytes_equal(to_np(q1), oq1, "q1")
    assert_bytes_equal(to_np(s1), os1, "s1 blocked")
    del oq0, os0, oq1, os1
    # the dim1 outputs equal the dim0 outputs of X^T, at full size on the GPU
    xt = x.t().contiguous()
    del q0, s0
    t0, ts0, _, _ = mx.cast_dim0_dim1(xt)
    assert torch.equal(t0, q1)
    assert torch.equal(ts0, s1)


@pytest.fixture(scope="module")
def experts_case():
    """The expert weights on the GPU and the oracle's casts of them (both
    directions, per-expert blocked scales), computed once for the module."""
    w = W.make("experts16x8192x5120", device="cuda")["x"]
    want = oracle.cast_3d_dim0_dim1(W.bf16_bits(w))
    return w, want


def test_experts_dim1_every_byte(experts_case):
    w, (_, _, oq1, os1) = experts_case
    q1, s1 = mx.cast_3d_dim1(w)
    torch.cuda.synchronize()
    assert_bytes_equal(to_np(q1), oq1, "q1")
    assert_bytes_equal(to_np(s1), os1, "s1 per expert")


def test_experts_dim0_and_fused_every_byte(experts_case):
    w, (oq0, os0, oq1, os1) = experts_case
    q0, s0 = mx.cast_3d_dim0(w)
    torch.cuda.synchronize()
    assert_bytes_equal(to_np(q0), oq0, "dim0 q0")
    assert_bytes_equal(to_np(s0), os0, "dim0 s0 per expert")
    del q0, s0
    q0, s0, q1, s1 = mx.cast_3d_dim0_dim1(w)
    torch.cuda.synchronize()
    assert_bytes_equal(to_np(q0), oq0, "fused q0")
    assert_bytes_equal(to_np(s0), os0, "fused s0 per expert")
    assert_bytes_equal(to_np(q1), oq1, "fused q1")
    assert_bytes_equal(to_np(s1), os1, "fused s1 per expert")


def test_grouped_tall_group_every_byte():
    """Grouped-M cast with a group far taller than a CTA's run of tiles
    (65536 x 5120; groups of 40000, 1 and 25535 rows): the tall group's tiles
    are walked in bands of tile-rows, the others as whole column strips; every
    output byte against the oracle."""
    M, K = 65536, 5120
    x = W.normal((M, K), 1006, device="cuda")
    offs = [40000, 40001, 65536]
    got = mx.cast_grouped_m(x, torch.tensor(offs, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(got[6].item()) == 0
    want = oracle.cast_grouped_m(W.bf16_bits(x), np.array(offs, np.int32))
    for name, g, w in zip(("q0", "s0", "s0_row_offs", "q1", "s1", "s1_col_offs"), got, want):
        assert_bytes_equal(to_np(g), w, name)


def test_grouped_banded_with_many_groups_every_byte():
    """More than 1024 groups take the separate offsets kernel and a group
    table in global memory.  400000 x 512 in 1101 groups (300000 rows, 1099
    groups of 45 rows, then 50545 rows) makes the runs 101 tiles long, so the
    two tall groups are walked in bands: both paths together, every byte
    against the oracle."""
    M, K = 400000, 512
    sizes = [300000] + [45] * 1099
    sizes.append(M - sum(sizes))
    offs = np.cumsum(sizes).astype(np.int32)
    assert len(offs) == 1101 and offs[-1] == M and sizes[-1] == 50545
    x = W.normal((M, K), 1007, device="cuda")
    got = mx.cast_grouped_m(x, torch.from_numpy(offs).cuda())
    torch.cuda.synchronize()
    assert int(got[6].item()) == 0
    want = oracle.cast_grouped_m(W.bf16_bits(x), offs)
    for name, g, w in zip(("q0", "s0", "s0_row_offs", "q1", "s1", "s1_col_offs"), got, want):
        assert_bytes_equal(to_np(g), w, name)
