"""GPU parity of the dim0-only casts (2D and 3D expert weights), the fused 3D
dim0 + dim1 cast and MX dequantisation, through the C ABI, against the CPU
oracle on the same seeded inputs: byte for byte for fp8 data, e8m0 scales and
padded blocked buffers; bit for bit for dequantised bf16 (any NaN pattern
where the oracle gives NaN).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096
CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.library()
    assert mx.mx_watchdog(clear=True) == 0
    yield
    torch.cuda.synchronize()
    assert mx.mx_watchdog(clear=True) == 0


def guarded(nbytes):
    buf = torch.full((nbytes + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    return buf, buf[:nbytes]


def check_guard(buf, nbytes, what):
    assert np.all(buf[nbytes:].cpu().numpy() == CANARY), "%s: write past its end" % what


def assert_bytes_equal(got, want, what):
    got = np.asarray(got).ravel()
    want = np.asarray(want).ravel()
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.flatnonzero(got != want)
    if bad.size:
        i = bad[0]
        raise AssertionError("%s: %d of %d differ; first at %d: got %#x want %#x"
                             % (what, bad.size, got.size, i, got[i], want[i]))


def assert_bf16_equal(got, want, what):
    """Bit-exact bf16, except that where the oracle gives NaN any NaN passes."""
    got = np.asarray(got, np.uint16).ravel()
    want = np.asarray(want, np.uint16).ravel()
    nan_w = ((want & 0x7F80) == 0x7F80) & ((want & 0x7F) != 0)
    nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    assert np.array_equal(nan_g, nan_w), "%s: NaN positions differ" % what
    assert_bytes_equal(got[~nan_w], want[~nan_w], what)


def to_np(t):
    return t.detach().cpu().numpy()


def bf16_np(t):
    return to_np(t.view(torch.int16)).view(np.uint16)


# ---- 2D dim0 only ------------------------------------------------------------------

@pytest.mark.parametrize("M,K", [(1, 32), (32, 32), (77, 96), (160, 96), (333, 4128),
                                 (1024, 160), (544, 1056)])
def test_dim0_only_matches_oracle(M, K):
    x = W.spiky(M, K, 5 * M + K, scale_frac=0.05, zero_frac=0.05)
    n0 = mx.mx_blocked_bytes(M, K // 32)
    bq, q0 = guarded(M * K)
    bs, s0 = guarded(n0)
    mx.mx_cast_dim0(x.cuda(), q0, s0)
    torch.cuda.synchronize()
    check_guard(bq, M * K, "q0")
    check_guard(bs, n0, "s0")
    oq, os_ = oracle.cast_dim0(W.bf16_bits(x))
    assert_bytes_equal(to_np(q0), oq, "q0")
    assert_bytes_equal(to_np(s0), oracle.to_blocked(os_), "s0 blocked")


def test_dim0_only_equals_fused_dim0_full_size():
    """At 16384^2 the dim0-only launch writes the same q0 / s0 bytes as the
    fused launch, which test_gpu_full_size.py compares with the oracle byte
    for byte; sampled rows are also checked against the oracle here."""
    x = W.make("square16384_weight", device="cuda")["x"]
    M, K = x.shape
    q0, s0 = mx.cast_dim0(x)
    f0, fs0, _, _ = mx.cast_dim0_dim1(x)
    torch.cuda.synchronize()
    assert torch.equal(q0, f0) and torch.equal(s0, fs0)
    rows = torch.randperm(M, generator=torch.Generator().manual_seed(8))[:48].sort().values
    oq, os_ = oracle.cast_dim0(W.bf16_bits(x[rows.cuda()]))
    assert_bytes_equal(to_np(q0[rows.cuda()]), oq, "q0 rows")
    plain = oracle.from_blocked(to_np(s0), M, K // 32)
    assert_bytes_equal(plain[rows.numpy()], os_, "s0 rows")


# ---- 3D expert weights: dim0 and fused --------------------------------------------

CASES_3D_DIM0 = [(1, 128, 128), (3, 256, 160), (2, 96, 160), (3, 50, 96), (5, 1, 32),
                 (4, 160, 4128), (2, 200, 64)]
CASES_3D_FUSED = [(1, 128, 128), (3, 256, 160), (2, 96, 160), (5, 32, 64), (4, 160, 4128)]


@pytest.mark.parametrize("E,N,K", CASES_3D_DIM0)
def test_3d_dim0_matches_oracle(E, N, K):
    w = W.experts(E, N, K, 3 * E * N + K)
    nq, ns = E * N * K, mx.mx_3d_dim0_scale_bytes(E, N, K)
    bq, q0 = guarded(nq)
    bs, s0 = guarded(ns)
    mx.mx_cast_3d_dim0(w.cuda(), q0, s0)
    torch.cuda.synchronize()
    check_guard(bq, nq, "q0")
    check_guard(bs, ns, "s0")
    oq, os_ = oracle.cast_3d_dim0(W.bf16_bits(w))
    assert_bytes_equal(to_np(q0), oq, "q0")
    assert_bytes_equal(to_np(s0), os_, "s0 per expert")


@pytest.mark.parametrize("E,N,K", CASES_3D_FUSED)
def test_3d_fused_matches_oracle(E, N, K):
    w = W.experts(E, N, K, 5 * E * N + K)
    nq = E * N * K
    n0, n1 = mx.mx_3d_dim0_scale_bytes(E, N, K), mx.mx_3d_scale_bytes(E, N, K)
    bq0, q0 = guarded(nq)
    bs0, s0 = guarded(n0)
    bq1, q1 = guarded(nq)
    bs1, s1 = guarded(n1)
    mx.mx_cast_3d_dim0_dim1(w.cuda(), q0, s0, q1, s1)
    torch.cuda.synchronize()
    for b, n, name in ((bq0, nq, "q0"), (bs0, n0, "s0"), (bq1, nq, "q1"), (bs1, n1, "s1")):
        check_guard(b, n, name)
    oq0, os0, oq1, os1 = oracle.cast_3d_dim0_dim1(W.bf16_bits(w))
    assert_bytes_equal(to_np(q0), oq0, "q0")
    assert_bytes_equal(to_np(s0), os0, "s0 per expert")
    assert_bytes_equal(to_np(q1), oq1, "q1")
    assert_bytes_equal(to_np(s1), os1, "s1 per expert")


# ---- dequantisation ---------------------------------------------------------------

def _golden_dequant():
    path = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_dequant.txt")
    cases = []
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            name, q, s, out = [t.strip() for t in line.split("|")]
            cases.append((name, int(q, 16), int(s, 16), out))
    return cases


def _pairs(qs, ss):
    """Element bytes qs with scale bytes ss: row i holds 32 copies of qs[i]."""
    q = np.repeat(np.asarray(qs, np.uint8)[:, None], 32, axis=1)
    s_blk = oracle.to_blocked(np.asarray(ss, np.uint8).reshape(-1, 1))
    return q, s_blk


def _gpu_dequant(q, s_blk):
    R, C = q.shape
    bo = torch.full((R * C + GUARD // 2,), 0x5A5A, dtype=torch.int16, device="cuda")
    out = bo[:R * C].view(torch.bfloat16).view(R, C)
    mx.mx_dequant_blocked(torch.from_numpy(q).cuda(), torch.from_numpy(s_blk).cuda(), out)
    torch.cuda.synchronize()
    assert torch.all(bo[R * C:] == 0x5A5A), "dequant wrote past its output"
    return bf16_np(out)


def test_dequant_hand_worked():
    cases = _golden_dequant()
    q, s_blk = _pairs([c[1] for c in cases], [c[2] for c in cases])
    got = _gpu_dequant(q, s_blk)
    assert np.all(got == got[:, :1])
    for (name, _, _, want), g in zip(cases, got[:, 0]):
        if want == "nan":
            assert (g & 0x7F80) == 0x7F80 and (g & 0x7F), name
        else:
            assert g == int(want, 16), (name, hex(g), want)


def test_dequant_every_element_every_scale():
    qs = np.tile(np.arange(256, dtype=np.uint8), 256)
    ss = np.repeat(np.arange(256, dtype=np.uint8), 256)
    q, s_blk = _pairs(qs, ss)
    assert_bf16_equal(_gpu_dequant(q, s_blk), oracle.dequant_blocked(q, s_blk), "all pairs")


def test_dequant_every_element_every_scale_tiled():
    """The same 65,536 (element, scale) pairs laid out in rows of 1024 values,
    the tiled kernel's path: block b (row b // 32, scale column b % 32) has
    scale byte b % 256 and elements (32 (b // 256) + i) % 256, so every scale
    byte meets every element byte four times."""
    R, C = 256, 1024
    b = np.arange(R * C // 32)
    s = (b % 256).astype(np.uint8).reshape(R, C // 32)
    q = ((32 * (b[:, None] // 256) + np.arange(32)[None, :]) % 256).astype(np.uint8)
    q = q.reshape(R, C)
    s_blk = oracle.to_blocked(s)
    assert_bf16_equal(_gpu_dequant(q, s_blk), oracle.dequant_blocked(q, s_blk), "all pairs tiled")


@pytest.mark.parametrize("M,K", [(32, 32), (160, 96), (544, 1056), (96, 4128), (256, 2048),
                                 (1024, 160)])
def test_dequant_of_cast_matches_oracle(M, K):
    """Cast on the GPU, dequantise both copies on the GPU, against the oracle
    dequantising the oracle's cast (the two casts are byte-identical)."""
    x = W.wide(M, K, 11 * M + K, zero_frac=0.02)
    q0, s0, q1, s1 = mx.cast_dim0_dim1(x.cuda())
    d0 = mx.dequant_blocked(q0, s0)
    d1 = mx.dequant_blocked(q1, s1)
    torch.cuda.synchronize()
    oq0, os0, oq1, os1 = oracle.cast_dim0_dim1_blocked(W.bf16_bits(x))
    assert_bf16_equal(bf16_np(d0), oracle.dequant_blocked(oq0, os0), "dequant dim0")
    assert_bf16_equal(bf16_np(d1), oracle.dequant_blocked(oq1, os1), "dequant dim1")


# Rows shorter than 1024 values take the thread-store kernel, longer ones the
# tiled kernel, whose last tile column may hold only 32 .. 96 columns (C % 128
# != 0) and whose last tile row may be partial.
@pytest.mark.parametrize("R,C", [(1, 32), (77, 96), (1, 128), (77, 160), (300, 224), (3, 8192),
                                 (1, 1024), (129, 4128), (130, 1056), (77, 1120), (5, 1056)])
def test_dequant_ragged_shapes(R, C):
    rng = np.random.default_rng(R * 7 + C)
    q = rng.integers(0, 256, size=(R, C), dtype=np.uint8)
    s = rng.integers(100, 160, size=(R, C // 32), dtype=np.uint8)
    s_blk = oracle.to_blocked(s)
    assert_bf16_equal(_gpu_dequant(q, s_blk), oracle.dequant_blocked(q, s_blk), "random")


def test_dequant_full_size_sampled():
    """Dequantise the 16384^2 weight's dim0 copy (the benchmark's launch) and
    check sampled rows against the oracle."""
    x = W.make("square16384_weight", device="cuda")["x"]
    M, K = x.shape
    q0, s0 = mx.cast_dim0(x)
    d = mx.dequant_blocked(q0, s0)
    torch.cuda.synchronize()
    rows = torch.randperm(M, generator=torch.Generator().manual_seed(9))[:32].sort().values
    plain = oracle.from_blocked(to_np(s0), M, K // 32)[rows.numpy()]
    want = oracle.dequant_blocked(to_np(q0[rows.cuda()]), oracle.to_blocked(plain))
    assert_bf16_equal(bf16_np(d[rows.cuda()]), want, "dequant rows")


def test_cuda_graph_capture_of_the_other_entry_points():
    """dim0, 3D, dequantisation, tensorwise (memset + two kernels) and rowwise
    calls captured in one CUDA graph replay to the bytes of direct calls."""
    x = W.wide(384, 256, 91).cuda()
    w = W.experts(2, 96, 160, 92).cuda()
    calls = [
        (lambda: mx.cast_dim0(x), lambda o: mx.mx_cast_dim0(x, *o)),
        (lambda: mx.cast_3d_dim0_dim1(w), lambda o: mx.mx_cast_3d_dim0_dim1(w, *o)),
        (lambda: mx.cast_3d_dim0(w), lambda o: mx.mx_cast_3d_dim0(w, *o)),
        (lambda: mx.cast_tensorwise(x), lambda o: mx.mx_cast_tensorwise(x, *o)),
        (lambda: mx.cast_rowwise(x), lambda o: mx.mx_cast_rowwise(x, *o)),
    ]
    refs = [make() for make, _ in calls]
    q0, s0 = refs[0]
    dq_ref = mx.dequant_blocked(q0, s0)
    outs = [tuple(torch.empty_like(t) for t in r) for r in refs]
    dq_out = torch.empty_like(dq_ref)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for (_, call), o in zip(calls, outs):
            call(o)
        mx.mx_dequant_blocked(q0, s0, dq_out)
    for o in outs:
        for t in o:
            t.zero_()
    dq_out.zero_()
    g.replay()
    torch.cuda.synchronize()
    for r, o in zip(refs, outs):
        for a, b in zip(r, o):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert torch.equal(dq_ref.view(torch.int16), dq_out.view(torch.int16))
