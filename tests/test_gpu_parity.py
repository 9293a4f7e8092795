"""GPU parity: the CUDA path through the C ABI against the CPU oracle, byte
for byte (fp8 data, e8m0 scales, padded blocked buffers, group offsets).

Sizes span several 128x128 tiles with ragged tails, up to the grouped MoE
workload (16640 x 5120, 4 groups) compared in full; the two largest workloads
are compared byte for byte in test_gpu_full_size.py.  Every expected value
comes from the oracle run on the same seeded input in the same test.
"""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096          # canary bytes after every output buffer
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


def guarded(nbytes, fill=CANARY):
    """uint8 CUDA buffer of nbytes plus GUARD canary bytes; returns (buf, view)."""
    buf = torch.full((nbytes + GUARD,), fill, dtype=torch.uint8, device="cuda")
    return buf, buf[:nbytes]


def check_guard(buf, nbytes, what):
    tail = buf[nbytes:].cpu().numpy()
    assert np.all(tail == CANARY), "%s: write past the end of its buffer" % what


def assert_bytes_equal(got, want, what):
    got = np.asarray(got).ravel()
    want = np.asarray(want).ravel()
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.flatnonzero(got != want)
    if bad.size:
        i = bad[0]
        raise AssertionError("%s: %d of %d bytes differ; first at %d: got %#x want %#x"
                             % (what, bad.size, got.size, i, got[i], want[i]))


def to_np(t):
    return t.detach().cpu().numpy()


def run_fused(xb, dim0=True):
    """Run the fused (or dim1-only) cast through the ABI with guarded buffers."""
    M, K = xb.shape
    n0 = mx.mx_blocked_bytes(M, K // 32)
    n1 = mx.mx_blocked_bytes(K, M // 32)
    bq1, q1 = guarded(M * K)
    bs1, s1 = guarded(n1)
    if dim0:
        bq0, q0 = guarded(M * K)
        bs0, s0 = guarded(n0)
        mx.mx_cast_dim0_dim1(xb, q0, s0, q1, s1)
    else:
        mx.mx_cast_dim1(xb, q1, s1)
    torch.cuda.synchronize()
    check_guard(bq1, M * K, "q1")
    check_guard(bs1, n1, "s1")
    out = {"q1": to_np(q1).reshape(K, M), "s1": to_np(s1)}
    if dim0:
        check_guard(bq0, M * K, "q0")
        check_guard(bs0, n0, "s0")
        out["q0"] = to_np(q0).reshape(M, K)
        out["s0"] = to_np(s0)
    return out


def compare_fused(x_cpu, dim0=True):
    xb = x_cpu.cuda()
    got = run_fused(xb, dim0)
    bits = W.bf16_bits(x_cpu)
    q0, s0, q1, s1 = oracle.cast_dim0_dim1_blocked(bits, dim0=dim0, dim1=True)
    if dim0:
        assert_bytes_equal(got["q0"], q0, "q0")
        assert_bytes_equal(got["s0"], s0, "s0 blocked")
    assert_bytes_equal(got["q1"], q1, "q1")
    assert_bytes_equal(got["s1"], s1, "s1 blocked")


# ---- fused dim0 + dim1 and dim1-only ------------------------------------------

SHAPES = [(32, 32), (32, 96), (96, 32), (128, 128), (160, 96), (256, 384), (416, 288),
          (544, 1056), (1024, 160), (96, 4128)]


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("kind", ["spiky", "wide"])
def test_fused_matches_oracle(M, K, kind):
    seed = 7 * M + K
    if kind == "spiky":
        x = W.spiky(M, K, seed, scale_frac=0.05, zero_frac=0.05)
    else:
        x = W.wide(M, K, seed, zero_frac=0.02)
    compare_fused(x, dim0=True)


@pytest.mark.parametrize("M,K", [(32, 32), (160, 96), (544, 1056), (96, 4128)])
def test_dim1_only_matches_oracle(M, K):
    compare_fused(W.wide(M, K, M + 3 * K), dim0=False)


def test_named_small_workloads_exact():
    """The 1024^2 spiky and 4096^2 wide-range workloads, every byte."""
    compare_fused(W.make("square1024_spiky")["x"])
    compare_fused(W.make("square4096_wide")["x"])


def test_edge_values(golden_blocks):
    """Hand-worked blocks (all 448, powers of two, subnormals, ties, bf16 max)
    tiled over a matrix as row blocks (top half) and column blocks (bottom
    half), plus an all-subnormal block, against the oracle."""
    cases = [c for c in golden_blocks if not c[1]]
    n = len(cases)
    M, K = 256, 32 * n
    X = np.zeros((M, K), np.uint16)
    for i in range(128):
        for j in range(n):
            X[i, 32 * j:32 * j + 32] = cases[(i + j) % n][3]
    for i in range(4):
        for j in range(K):
            X[128 + 32 * i:160 + 32 * i, j] = cases[(i + j) % n][3]
    X[224:256, 64:96] = 0x0001
    x = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16)
    compare_fused(x)


def test_nan_inf_blocks_reading():
    """Not pinned by the pages (no workload holds NaN/Inf): a block with NaN,
    -NaN, Inf or -Inf gets scale byte 0xFF and every element the e4m3 NaN
    0x7F; all other blocks are unaffected.  Every byte equals the oracle's,
    in both directions and through the grouped kernel."""
    M, K = 64, 64
    bits = W.bf16_bits(W.normal((M, K), 5)).copy()
    bits[3, 40] = 0x7FC0          # NaN
    bits[40, 5] = 0x7F80          # +Inf
    bits[50, 60] = 0xFF80         # -Inf
    bits[20, 10] = 0xFFC1         # a NaN with the sign bit set and a payload
    xn = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    got = run_fused(xn.cuda())
    bits = W.bf16_bits(xn)
    q0, s0, q1, s1 = oracle.cast_dim0_dim1_blocked(bits)
    assert_bytes_equal(got["s0"], s0, "s0")
    assert_bytes_equal(got["s1"], s1, "s1")
    assert np.count_nonzero(oracle.from_blocked(s0, M, K // 32) == 0xFF) == 4
    assert_bytes_equal(got["q0"], q0, "q0")
    assert_bytes_equal(got["q1"], q1, "q1")
    assert np.count_nonzero(q0 == 0x7F) == 4 * 32   # four NaN blocks per direction
    compare_grouped(xn, [17, 64])


def test_repeat_calls_identical_and_stream_ordered():
    x = W.wide(256, 256, 99).cuda()
    a = mx.cast_dim0_dim1(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = mx.cast_dim0_dim1(x, stream=s)
    s.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)


# ---- standalone blocked layout ---------------------------------------------------

@pytest.mark.parametrize("R,C", [(1, 1), (128, 4), (130, 5), (300, 17), (16640, 160),
                                 (5120, 4096), (257, 64), (1000, 3)])
def test_scales_to_blocked_matches_oracle(R, C):
    g = torch.Generator().manual_seed(R * 31 + C)
    s = torch.randint(0, 256, (R, C), dtype=torch.uint8, generator=g)
    n = mx.mx_blocked_bytes(R, C)
    buf, out = guarded(n)
    mx.mx_scales_to_blocked(s.cuda(), out)
    torch.cuda.synchronize()
    check_guard(buf, n, "blocked")
    assert_bytes_equal(to_np(out), oracle.to_blocked(s.numpy()), "blocked")


def test_scales_to_blocked_unaligned_source():
    s = torch.randint(0, 256, (300, 41), dtype=torch.uint8)
    big = torch.zeros(300 * 41 + 3, dtype=torch.uint8)
    big[3:] = s.ravel()
    src = big.cuda()[3:].view(300, 41)
    out = mx.scales_to_blocked(src)
    torch.cuda.synchronize()
    assert_bytes_equal(to_np(out), oracle.to_blocked(s.numpy()), "blocked")


def test_fused_scales_equal_standalone_blocking_of_plain_scales():
    """The blocked scales written by the fused kernel equal the standalone
    blocking kernel applied to the oracle's plain scales."""
    x = W.wide(384, 640, 12)
    got = run_fused(x.cuda())
    _, p0 = oracle.cast_dim0(W.bf16_bits(x))
    b0 = mx.scales_to_blocked(torch.from_numpy(p0).cuda())
    torch.cuda.synchronize()
    assert_bytes_equal(got["s0"], to_np(b0), "s0")


# ---- grouped along M -----------------------------------------------------------

def run_grouped(x_cpu, offs_list, fill=CANARY):
    M, K = x_cpu.shape
    G = len(offs_list)
    xb = x_cpu.cuda()
    offs = torch.tensor(offs_list, dtype=torch.int32, device="cuda")
    n0 = mx.mx_grouped_m_scale_bytes(M, K, G, 0)
    n1 = mx.mx_grouped_m_scale_bytes(M, K, G, 1)
    bq0, q0 = guarded(M * K, fill)
    bq1, q1 = guarded(M * K, fill)
    bs0, s0 = guarded(n0, fill)
    bs1, s1 = guarded(n1, fill)
    r0 = torch.full((G + 1,), -7, dtype=torch.int64, device="cuda")
    c1 = torch.full((G + 1,), -7, dtype=torch.int64, device="cuda")
    st = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    mx.mx_cast_grouped_m(xb, offs, q0, s0, r0, q1, s1, c1, st)
    torch.cuda.synchronize()
    for b, n, w in ((bq0, M * K, "q0"), (bq1, M * K, "q1"), (bs0, n0, "s0"), (bs1, n1, "s1")):
        check_guard(b, n, w)
    return dict(q0=to_np(q0).reshape(M, K), s0=to_np(s0), r0=to_np(r0), q1=to_np(q1).reshape(K, M),
                s1=to_np(s1), c1=to_np(c1), status=int(st.item()))


def compare_grouped(x_cpu, offs_list):
    got = run_grouped(x_cpu, offs_list)
    assert got["status"] == 0
    q0, s0, r0, q1, s1, c1 = oracle.cast_grouped_m(W.bf16_bits(x_cpu), np.array(offs_list, np.int32))
    assert_bytes_equal(got["r0"], r0, "s0_row_offs")
    assert_bytes_equal(got["c1"], c1, "s1_col_offs")
    assert_bytes_equal(got["q0"], q0, "q0")
    assert_bytes_equal(got["s0"], s0, "s0 grouped blocked")
    assert_bytes_equal(got["q1"], q1, "q1")
    assert_bytes_equal(got["s1"], s1, "s1 grouped blocked")


GROUP_CASES = [
    (128, 64, [128]),
    (300, 160, [1, 45, 45, 190, 300]),         # ragged, with an empty group
    (257, 96, [257]),                          # single ragged group
    (512, 256, [128, 384, 384, 512]),          # multiples of 128
    (1000, 384, [0, 0, 333, 334, 999, 1000]),  # empty leading groups, size-1 groups
    (2080, 544, [17, 400, 1111, 2080]),
    (4224, 640, [0, 1000, 1000, 2999, 4224, 4224]),   # empty first, middle and last groups
]


@pytest.mark.parametrize("M,K,offs", GROUP_CASES)
def test_grouped_matches_oracle(M, K, offs):
    compare_grouped(W.wide(M, K, M + K, zero_frac=0.01), offs)


def test_grouped_random_sizes_many_groups():
    M, K = 3000, 256
    offs = W.group_ends(M, 37, 77, min_size=0).tolist()
    compare_grouped(W.spiky(M, K, 8, scale_frac=0.03, zero_frac=0.03), offs)


@pytest.mark.parametrize("M,K,G,seed", [(9999, 1024, 5, 31), (16000, 512, 9, 32), (4097, 2048, 3, 33)])
def test_grouped_multi_tile_runs(M, K, G, seed):
    """Enough tiles that every CTA walks several tiles down a column strip, so
    partial 16-byte chunks of q1 are carried from tile to tile; odd M makes
    the misalignment differ from one q1 row to the next; some groups empty."""
    offs = W.group_ends(M, G, seed, min_size=0).tolist()
    compare_grouped(W.wide(M, K, seed, zero_frac=0.005), offs)


@pytest.mark.parametrize("offs", [
    [4112, 8208, 12304, 16384],     # unshifted starts at odd multiples of 16
    [4122, 8250, 12390, 16384],     # shifted starts, boxes at 16 and 0 mod 32
    [4164, 8282, 12462, 16384],     # the MoE workload's starts
])
def test_grouped_box_alignment_paths(offs):
    """16384 x 2048, 13-14 tiles per CTA, group starts whose q1 boxes begin
    at odd and even multiples of 16 bytes, with and without a shift: the
    boxes from carried chunks, the run-start boxes one chunk later, the
    narrow run-end tails and the piecewise partial tiles, every byte against
    the oracle."""
    compare_grouped(W.wide(16384, 2048, offs[0], zero_frac=0.005), offs)


def test_grouped_many_groups_two_kernel_path():
    """More groups than the cast kernel tabulates itself (1024): the padded
    offsets come from the separate offsets kernel, launched before it."""
    M, K = 3000, 64
    offs = W.group_ends(M, 1500, 91, min_size=0).tolist()
    compare_grouped(W.wide(M, K, 92, zero_frac=0.01), offs)


def test_grouped_many_groups_invalid_offsets():
    M, K = 3000, 64
    offs = W.group_ends(M, 1500, 93, min_size=0).tolist()
    offs[700], offs[701] = offs[701] + 1, offs[700]      # decreasing
    got = run_grouped(W.normal((M, K), 4), offs, fill=CANARY)
    assert got["status"] == mx.MX_ERR_GROUPS
    for k in ("q0", "q1", "s0", "s1"):
        assert np.all(got[k] == CANARY), k


def test_grouped_moe_workload_full():
    """The 16640 x 5120, 4-group MoE workload, every byte."""
    w = W.make("moe16640x5120_g4")
    compare_grouped(w["x"], w["offs"].tolist())


@pytest.mark.parametrize("offs", [[100, 50, 200], [50, 300], [-5, 200], [100, 150]])
def test_grouped_invalid_offsets_write_nothing(offs):
    M, K = 200, 64
    got = run_grouped(W.normal((M, K), 3), offs, fill=CANARY)
    assert got["status"] == mx.MX_ERR_GROUPS
    for k in ("q0", "q1", "s0", "s1"):
        assert np.all(got[k] == CANARY), k


# ---- 3D expert weights -------------------------------------------------------------

@pytest.mark.parametrize("E,N,K", [(1, 128, 128), (3, 256, 160), (2, 96, 160), (5, 32, 64),
                                   (4, 160, 4128)])
def test_3d_matches_oracle(E, N, K):
    w = W.experts(E, N, K, E * N + K)
    wb = w.cuda()
    nq, ns = E * N * K, mx.mx_3d_scale_bytes(E, N, K)
    bq, q1 = guarded(nq)
    bs, s1 = guarded(ns)
    mx.mx_cast_3d_dim1(wb, q1, s1)
    torch.cuda.synchronize()
    check_guard(bq, nq, "q1")
    check_guard(bs, ns, "s1")
    oq1, os1 = oracle.cast_3d_dim1(W.bf16_bits(w))
    assert_bytes_equal(to_np(q1).reshape(K, E * N), oq1, "q1")
    assert_bytes_equal(to_np(s1), os1, "s1 per expert")


def test_cuda_graph_capture_replays_identically():
    """The C-ABI calls can be captured into a CUDA graph (tensor maps are
    encoded on the host at capture time) and replay to the same bytes."""
    x = W.wide(512, 384, 77).cuda()
    ref = mx.cast_dim0_dim1(x)
    outs = tuple(torch.empty_like(t) for t in ref)
    offs = torch.tensor([100, 300, 512], dtype=torch.int32, device="cuda")
    gref = mx.cast_grouped_m(x, offs)
    gouts = tuple(torch.empty_like(t) for t in gref)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mx.mx_cast_dim0_dim1(x, *outs)
        mx.mx_cast_grouped_m(x, offs, *gouts)
    for t in outs + gouts:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref + gref, outs + gouts):
        assert torch.equal(a, b)


def test_concurrent_host_threads_and_streams():
    """Four host threads, each with its own stream (and so its own descriptor
    cache), cast different inputs twenty times over; every result equals the
    oracle."""
    import threading
    xs = [W.wide(512, 384 + 32 * i, 100 + i).cuda() for i in range(4)]
    results = [None] * 4
    errors = []

    def work(i):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(20):
                    out = mx.cast_dim0_dim1(xs[i], stream=st)
                st.synchronize()
            results[i] = tuple(to_np(t) for t in out)
        except Exception as e:                       # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(4):
        want = oracle.cast_dim0_dim1_blocked(W.bf16_bits(xs[i].cpu()))
        for name, g, w in zip(("q0", "s0", "q1", "s1"), results[i], want):
            assert_bytes_equal(g, w, "thread %d %s" % (i, name))
