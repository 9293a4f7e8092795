"""The claim schedule of the 2D / 3D casts, every byte against the oracle.

Launches of 32 rounds of tiles or more (tiles per CTA) deal out all but the
last six rounds in advance and let the CTAs claim the rest from a counter
kept per stream, which the launch's last claimer resets.  These tests run
such launches (8192 x 10240: 5120 tiles, 33 rounds on 152 SMs):

- fused, dim0-only, dim1-only and 3D casts, against the oracle;
- five launches in a row on one stream with different inputs (each must find
  the counter reset by the previous one);
- two streams casting at the same time (each stream has its own counter);
- a cast captured in a CUDA graph (captured launches take the static
  schedule) and replayed twice.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu

M, K = 8192, 10240


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


def same(got, want, what):
    g = got.detach().cpu().contiguous().view(torch.uint8).numpy().ravel()
    w = np.ascontiguousarray(want).view(np.uint8).ravel()
    assert g.shape == w.shape, (what, g.shape, w.shape)
    bad = np.flatnonzero(g != w)
    assert bad.size == 0, "%s: %d of %d bytes differ, first at %d" % (what, bad.size, g.size, bad[0])


def test_claimed_launch_is_long_enough():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert (M // 128) * (K // 128) // min(sms, (M // 128) * (K // 128)) >= 32


def test_fused_dim0_dim1_with_claims():
    x = W.spiky(M, K, 3101, scale_frac=0.05, zero_frac=0.02)
    want = oracle.cast_dim0_dim1_blocked(W.bf16_bits(x))
    xc = x.cuda()
    got = mx.cast_dim0_dim1(xc)
    for name, g, w in zip(("q0", "s0", "q1", "s1"), got, want):
        same(g, w, "fused " + name)
    q0, s0 = mx.cast_dim0(xc)
    same(q0, want[0], "dim0 q0")
    same(s0, want[1], "dim0 s0")
    q1, s1 = mx.cast_dim1(xc)
    same(q1, want[2], "dim1 q1")
    same(s1, want[3], "dim1 s1")


def test_3d_with_claims():
    w = W.experts(4, 2048, K, 3102)                       # (E * N, K) = (8192, 10240)
    want = oracle.cast_3d_dim0_dim1(W.bf16_bits(w))
    got = mx.cast_3d_dim0_dim1(w.cuda())
    for name, g, ww in zip(("q0", "s0", "q1", "s1"), got, want):
        same(g, ww, "3d " + name)


def test_five_launches_in_a_row_on_one_stream():
    xs = [W.normal((M, K), 3110 + i) for i in range(5)]
    dev = [x.cuda() for x in xs]
    outs = []
    torch.cuda.synchronize()
    for x in dev:                                         # back to back, no host sync
        outs.append(mx.cast_dim0_dim1(x))
    torch.cuda.synchronize()
    for i, (x, got) in enumerate(zip(xs, outs)):
        want = oracle.cast_dim0_dim1_blocked(W.bf16_bits(x))
        for name, g, w in zip(("q0", "s0", "q1", "s1"), got, want):
            same(g, w, "launch %d %s" % (i, name))


def test_two_streams_at_once():
    xs = [W.normal((M, K), 3120 + i) for i in range(4)]
    dev = [x.cuda() for x in xs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [None] * 4
    torch.cuda.synchronize()
    for i, x in enumerate(dev):                           # alternate the streams
        with torch.cuda.stream(streams[i % 2]):
            outs[i] = mx.cast_dim0_dim1(x)
    torch.cuda.synchronize()
    for i, (x, got) in enumerate(zip(xs, outs)):
        want = oracle.cast_dim0_dim1_blocked(W.bf16_bits(x))
        for name, g, w in zip(("q0", "s0", "q1", "s1"), got, want):
            same(g, w, "stream %d launch %d %s" % (i % 2, i, name))


def test_graph_capture_takes_the_static_schedule():
    x = W.normal((M, K), 3130)
    xc = x.cuda()
    q0 = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    q1 = torch.empty((K, M), dtype=torch.uint8, device="cuda")
    s0 = torch.empty(mx.mx_blocked_bytes(M, K // 32), dtype=torch.uint8, device="cuda")
    s1 = torch.empty(mx.mx_blocked_bytes(K, M // 32), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side), torch.cuda.graph(graph, stream=side):
        mx.mx_cast_dim0_dim1(xc, q0, s0, q1, s1)
    want = oracle.cast_dim0_dim1_blocked(W.bf16_bits(x))
    for rep in range(2):
        for t in (q0, s0, q1, s1):
            t.fill_(0x5A)
        graph.replay()
        torch.cuda.synchronize()
        for name, g, w in zip(("q0", "s0", "q1", "s1"), (q0, s0, q1, s1), want):
            same(g, w, "replay %d %s" % (rep, name))
    # and an ordinary launch on the same stream afterwards still claims correctly
    got = mx.cast_dim0_dim1(xc)
    torch.cuda.synchronize()
    for name, g, w in zip(("q0", "s0", "q1", "s1"), got, want):
        same(g, w, "after the graph " + name)
