"""GPU parity of the tensorwise and rowwise fp8 casts through the C ABI
against the CPU oracle on the same seeded inputs: e4m3 bytes exactly, the
scales bit for bit (any NaN pattern where the oracle gives NaN, either e4m3
NaN byte for NaN elements).
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


def to_np(t):
    return t.detach().cpu().numpy()


def assert_q_equal(got, want, what):
    got = np.asarray(got, np.uint8).ravel()
    want = np.asarray(want, np.uint8).ravel()
    nan_w = (want & 0x7F) == 0x7F
    assert np.array_equal((got & 0x7F) == 0x7F, nan_w), "%s: NaN positions differ" % what
    bad = np.flatnonzero(got[~nan_w] != want[~nan_w])
    if bad.size:
        i = bad[0]
        raise AssertionError("%s: %d of %d bytes differ; first at %d: got %#x want %#x"
                             % (what, bad.size, want.size, i, got[~nan_w][i], want[~nan_w][i]))


def f32_bits(v):
    return int(np.float32(v).view(np.uint32))


def same_f32(a, b):
    a, b = np.float32(a), np.float32(b)
    return (np.isnan(a) and np.isnan(b)) or f32_bits(a) == f32_bits(b)


def run_tensorwise(bits):
    """bf16 bit patterns (numpy uint16, any shape) through the ABI with a
    guarded q buffer."""
    n = bits.size
    x = torch.from_numpy(bits.astype(np.int16).reshape(-1)).cuda().view(torch.bfloat16)
    buf = torch.full((n + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    scale = torch.full((1,), 7.0, dtype=torch.float32, device="cuda")
    amax = torch.full((1,), 7.0, dtype=torch.float32, device="cuda")
    mx.mx_cast_tensorwise(x, buf[:n], scale, amax)
    torch.cuda.synchronize()
    assert np.all(to_np(buf[n:]) == CANARY), "q written past its end"
    return to_np(buf[:n]), to_np(scale)[0], to_np(amax)[0]


def run_rowwise(bits):
    M, K = bits.shape
    x = torch.from_numpy(bits.astype(np.int16)).cuda().view(torch.bfloat16)
    buf = torch.full((M * K + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    sbuf = torch.full((M + GUARD,), 0x5A5A, dtype=torch.int16, device="cuda")
    mx.mx_cast_rowwise(x, buf[:M * K], sbuf[:M].view(torch.bfloat16))
    torch.cuda.synchronize()
    assert np.all(to_np(buf[M * K:]) == CANARY), "q written past its end"
    assert np.all(to_np(sbuf[M:]) == 0x5A5A), "scale written past its end"
    return to_np(buf[:M * K]).reshape(M, K), to_np(sbuf[:M]).view(np.uint16)


def compare_tensorwise(bits, what):
    q, scale, amax = run_tensorwise(bits)
    oq, oscale, oamax = oracle.cast_tensorwise(bits)
    assert same_f32(amax, oamax), (what, amax, oamax)
    assert same_f32(scale, oscale), (what, scale, oscale)
    assert_q_equal(q, oq, what)


def compare_rowwise(bits, what):
    q, scale = run_rowwise(bits)
    oq, oscale = oracle.cast_rowwise(bits)
    nan_s = ((oscale & 0x7F80) == 0x7F80) & ((oscale & 0x7F) != 0)
    assert np.array_equal(((scale & 0x7F80) == 0x7F80) & ((scale & 0x7F) != 0), nan_s), what
    assert np.array_equal(scale[~nan_s], oscale[~nan_s]), what
    assert_q_equal(q, oq, what)


def _golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_scaled_fp8.txt")
    out = []
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            kind, xs, sc, qs = [t.strip() for t in line.split("|")]
            out.append((kind, [int(v, 16) for v in xs.split()], int(sc, 16),
                        [int(v, 16) for v in qs.split()]))
    return out


def test_hand_worked_cases():
    for kind, xs, sc, qs in _golden():
        if kind == "tensorwise":
            for reps in (1, 8):                      # tail-only and vector paths
                q, scale, _ = run_tensorwise(np.array(xs * reps, np.uint16))
                assert f32_bits(scale) == sc, (xs, hex(f32_bits(scale)))
                assert list(q) == qs * reps, (xs, [hex(v) for v in q])
        else:
            row = np.array([xs + [0] * 4], np.uint16)  # K = 8: zeros keep the amax
            q, scale = run_rowwise(row)
            assert scale[0] == sc, (xs, hex(scale[0]))
            assert list(q[0]) == qs + [0] * 4, (xs, [hex(v) for v in q[0]])


@pytest.mark.parametrize("shape", [(1,), (7,), (8,), (1000,), (12293,), (256, 384), (1024, 4128)])
@pytest.mark.parametrize("kind", ["spiky", "wide"])
def test_tensorwise_matches_oracle(shape, kind):
    n = int(np.prod(shape))
    seed = n + (1 if kind == "wide" else 0)
    t = W.spiky(1, n, seed, scale_frac=0.05, zero_frac=0.02) if kind == "spiky" else \
        W.wide(1, n, seed, zero_frac=0.02)
    compare_tensorwise(W.bf16_bits(t).reshape(shape), "%s %s" % (kind, shape))


def test_tensorwise_edge_tensors():
    compare_tensorwise(np.zeros(100, np.uint16), "all zero")
    compare_tensorwise(np.array([0x0001, 0x8001] * 20, np.uint16), "smallest subnormals")
    base = W.bf16_bits(W.wide(1, 64, 5)).ravel()
    for name, val in (("nan", 0x7FC0), ("inf", 0x7F80), ("-inf", 0xFF80)):
        b = base.copy()
        b[17] = val
        compare_tensorwise(b, name)


def test_tensorwise_full_size_sampled():
    """16384^2 weight: amax against numpy over the whole tensor; sampled rows
    against the oracle run on those rows plus the row holding the global
    amax (so the oracle's amax, hence its scale, is the global one)."""
    x = W.make("square16384_weight", device="cuda")["x"]
    M, K = x.shape
    q, scale, amax = mx.cast_tensorwise(x)
    torch.cuda.synchronize()
    bits = W.bf16_bits(x)
    mag = bits & 0x7FFF
    top = int(np.argmax(mag))
    rows = np.sort(np.random.default_rng(2).choice(M, 40, replace=False))
    rows = np.unique(np.append(rows, top // K))
    oq, oscale, oamax = oracle.cast_tensorwise(bits[rows])
    assert same_f32(to_np(amax)[0], oamax) and same_f32(to_np(scale)[0], oscale)
    assert np.float32(oamax) == np.float32(
        (mag.reshape(-1)[top].astype(np.uint32) << 16).view(np.float32))
    assert_q_equal(to_np(q)[rows], oq, "sampled rows")


# Launch shapes covered: 8, 4, 2 and 1 rows per bulk-staged step (32 to 256
# threads per row), rings of 2, 3, 6 and 8 stages (39001 x 2048: three 32 KB
# stages and a one-row last step), and the re-reading kernel for rows over
# 24576 values.
@pytest.mark.parametrize("M,K", [(1, 8), (3, 24), (77, 96), (256, 384), (64, 4128), (1000, 512),
                                 (37, 8200), (5, 16392), (3, 24584), (2, 40000), (39001, 2048)])
def test_rowwise_matches_oracle(M, K):
    t = W.wide(M, K, 3 * M + K, zero_frac=0.02)
    compare_rowwise(W.bf16_bits(t), "%dx%d" % (M, K))


def test_rowwise_edge_rows():
    rows = W.bf16_bits(W.spiky(8, 64, 9, scale_frac=0.1, zero_frac=0.05)).copy()
    rows[0] = 0                                  # zero row -> scale 0, zeros
    rows[1, :] = 0x8000                          # negative zeros
    rows[2, :] = 0x0001                          # scale underflows to 0
    rows[3, 5] = 0x7FC0                          # NaN
    rows[4, 9] = 0x7F80                          # +Inf
    rows[5, :] = 0x0300                          # amax 2^-121: tiny but representable scale
    compare_rowwise(rows, "edge rows")


def test_rowwise_full_size_sampled():
    x = W.make("square16384_weight", device="cuda")["x"]
    M, K = x.shape
    q, scale = mx.cast_rowwise(x)
    torch.cuda.synchronize()
    rows = torch.randperm(M, generator=torch.Generator().manual_seed(12))[:48].sort().values
    oq, oscale = oracle.cast_rowwise(W.bf16_bits(x[rows.cuda()]))
    assert np.array_equal(to_np(scale.view(torch.int16))[rows.numpy()].view(np.uint16), oscale)
    assert_q_equal(to_np(q[rows.cuda()]), oq, "sampled rows")


def test_rowwise_every_mantissa_pair():
    """Rows whose largest element A runs over all 128 mantissas at three
    exponents (so the row scale bf16(A / 448) takes every mantissa the
    formula can give), each row holding every bf16 value of both signs in the
    12 binades below A plus those of A's binade up to A: every pairing of an
    element significand with a scale significand that lands on the e4m3 grid,
    against the oracle's division in double."""
    rows = []
    for e in (10, 127, 200):
        for m in range(128):
            a = (e << 7) | m
            vals = [a]
            for ee in range(max(e - 12, 0), e):
                vals += [(ee << 7) | mm for mm in range(128)]
            vals += [(e << 7) | mm for mm in range(m + 1)]
            vals += [v | 0x8000 for v in vals]
            rows.append(vals)
    K = -(-max(len(r) for r in rows) // 8) * 8
    bits = np.zeros((len(rows), K), np.uint16)
    for i, r in enumerate(rows):
        bits[i, :len(r)] = r
    compare_rowwise(bits, "every mantissa pair")
