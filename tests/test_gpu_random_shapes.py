"""Seeded random shapes through every entry point, each against the oracle.

The fixed parity cases in the other files cover the hand-picked edges; this
sweep draws sizes at random (ragged rows and columns, odd M, K not a multiple
of 128, random group offsets with empty groups, experts whose N is not a
multiple of 128, rows on both sides of the tiled dequantisation kernel's
threshold) and compares every output byte with the oracle.  The draws are
seeded, so a failure names a reproducible case.
"""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu

N_CASES = 32


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()
    assert mx.mx_watchdog(clear=True) == 0
    yield
    torch.cuda.synchronize()
    assert mx.mx_watchdog(clear=True) == 0


def same(got, want, what):
    g = got.detach().cpu().contiguous().view(torch.uint8).numpy().ravel()
    w = np.ascontiguousarray(want).view(np.uint8).ravel()
    assert g.shape == w.shape, (what, g.shape, w.shape)
    bad = np.flatnonzero(g != w)
    assert bad.size == 0, "%s: %d of %d bytes differ, first at %d" % (what, bad.size, g.size, bad[0])


def rng_for(i, salt):
    return np.random.default_rng(1000 * salt + i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_fused_dim0_dim1(i):
    r = rng_for(i, 1)
    M, K = 32 * int(r.integers(1, 60)), 32 * int(r.integers(1, 60))
    x = W.spiky(M, K, 5000 + i, scale_frac=0.05, zero_frac=0.03)
    want = oracle.cast_dim0_dim1_blocked(W.bf16_bits(x))
    got = mx.cast_dim0_dim1(x.cuda())
    for name, g, w in zip(("q0", "s0", "q1", "s1"), got, want):
        same(g, w, "fused %dx%d %s" % (M, K, name))
    q1, s1 = mx.cast_dim1(x.cuda())
    same(q1, want[2], "dim1 %dx%d q1" % (M, K))
    same(s1, want[3], "dim1 %dx%d s1" % (M, K))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_dim0_any_rows(i):
    r = rng_for(i, 2)
    M, K = int(r.integers(1, 1500)), 32 * int(r.integers(1, 80))
    x = W.wide(M, K, 6000 + i, zero_frac=0.02)
    q, s = oracle.cast_dim0(W.bf16_bits(x))
    gq, gs = mx.cast_dim0(x.cuda())
    same(gq, q, "dim0 %dx%d q0" % (M, K))
    same(gs, oracle.to_blocked(s), "dim0 %dx%d s0" % (M, K))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_grouped(i):
    r = rng_for(i, 3)
    M = int(r.integers(1, 3000))
    K = 32 * int(r.integers(1, 40))
    G = int(r.integers(1, 20))
    ends = np.sort(r.integers(0, M + 1, G - 1)) if G > 1 else np.zeros(0, np.int64)
    offs = np.concatenate([ends, [M]]).astype(np.int32)
    x = W.wide(M, K, 7000 + i, zero_frac=0.01)
    want = oracle.cast_grouped_m(W.bf16_bits(x), offs)
    got = mx.cast_grouped_m(x.cuda(), torch.from_numpy(offs).cuda())
    assert int(got[6].item()) == 0
    for name, g, w in zip(("q0", "s0", "s0_row_offs", "q1", "s1", "s1_col_offs"), got, want):
        same(g, w, "grouped M=%d K=%d offs=%s %s" % (M, K, offs.tolist(), name))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_3d(i):
    r = rng_for(i, 4)
    E, K = int(r.integers(1, 6)), 32 * int(r.integers(1, 30))
    N = 32 * int(r.integers(1, 12))
    w = W.experts(E, N, K, 8000 + i)
    want = oracle.cast_3d_dim0_dim1(W.bf16_bits(w))
    got = mx.cast_3d_dim0_dim1(w.cuda())
    for name, g, ww in zip(("q0", "s0", "q1", "s1"), got, want):
        same(g, ww, "3d %dx%dx%d %s" % (E, N, K, name))
    n_any = int(r.integers(1, 300))                      # dim0 alone: any N
    w2 = W.experts(E, n_any, K, 8500 + i)
    want0 = oracle.cast_3d_dim0(W.bf16_bits(w2))
    got0 = mx.cast_3d_dim0(w2.cuda())
    same(got0[0], want0[0], "3d dim0 N=%d q0" % n_any)
    same(got0[1], want0[1], "3d dim0 N=%d s0" % n_any)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_dequant(i):
    r = rng_for(i, 5)
    R = int(r.integers(1, 700))
    C = 32 * int(r.integers(1, 80))                      # both sides of 1024 values
    q = r.integers(0, 256, size=(R, C), dtype=np.uint8)
    s = r.integers(90, 170, size=(R, C // 32), dtype=np.uint8)
    s_blk = oracle.to_blocked(s)
    want = oracle.dequant_blocked(q, s_blk)
    got = mx.dequant_blocked(torch.from_numpy(q).cuda(), torch.from_numpy(s_blk).cuda())
    torch.cuda.synchronize()
    g = got.view(torch.int16).cpu().numpy().view(np.uint16)
    nan = ((want & 0x7F80) == 0x7F80) & ((want & 0x7F) != 0)
    assert np.all(((g[nan] & 0x7F80) == 0x7F80) & ((g[nan] & 0x7F) != 0)), "dequant NaN %dx%d" % (R, C)
    bad = np.flatnonzero(g[~nan] != want[~nan])
    assert bad.size == 0, "dequant %dx%d: %d values differ" % (R, C, bad.size)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_scaled_fp8(i):
    r = rng_for(i, 6)
    M, K = int(r.integers(1, 600)), 8 * int(r.integers(1, 700))
    x = W.wide(M, K, 9000 + i, zero_frac=0.02)
    bits = W.bf16_bits(x)
    oq, oscale = oracle.cast_rowwise(bits)
    gq, gscale = mx.cast_rowwise(x.cuda())
    same(gq, oq, "rowwise %dx%d q" % (M, K))
    same(gscale, oscale, "rowwise %dx%d scale" % (M, K))
    tq, tscale, tamax = oracle.cast_tensorwise(bits)
    gq, gs, ga = mx.cast_tensorwise(x.cuda())
    same(gq, tq, "tensorwise %dx%d q" % (M, K))
    same(gs, np.array([tscale], np.float32), "tensorwise scale")
    same(ga, np.array([tamax], np.float32), "tensorwise amax")


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_scales_to_blocked(i):
    r = rng_for(i, 7)
    R, C = int(r.integers(1, 3000)), int(r.integers(1, 300))
    s = r.integers(0, 256, size=(R, C), dtype=np.uint8)
    same(mx.scales_to_blocked(torch.from_numpy(s).cuda()), oracle.to_blocked(s),
         "blocked %dx%d" % (R, C))
