"""GPU parity past 32-bit element offsets: a 65536 x 65536 bf16 matrix (2^32
elements, 8 GiB) through the fused cast, dequantisation and the tensorwise
cast, checked on sampled rows and columns against the CPU oracle.  Offsets
into X, q0, q1 and the dequantised output pass 2^31 and 2^32 here.
"""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu

N = 65536


@pytest.fixture(scope="module")
def big():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 40 * 2 ** 30:
        pytest.skip("needs about 40 GiB of free device memory")
    g = torch.Generator(device="cuda")
    g.manual_seed(2024)
    x = torch.randn((N, N), generator=g, device="cuda", dtype=torch.bfloat16)
    x.mul_(0.02)
    yield x
    del x
    torch.cuda.empty_cache()


def _rows(n, seed):
    rng = np.random.default_rng(seed)
    picks = rng.choice(N, n, replace=False)
    return np.sort(np.concatenate([picks, [0, N - 1]]))


def test_fused_and_dequant_beyond_32bit_offsets(big):
    x = big
    q0, s0, q1, s1 = mx.cast_dim0_dim1(x)
    torch.cuda.synchronize()
    rows = _rows(14, 1)
    idx = torch.from_numpy(rows).cuda()
    oq0, os0 = oracle.cast_dim0(W.bf16_bits(x[idx]))
    assert np.array_equal(q0[idx].cpu().numpy(), oq0)
    plain0 = oracle.from_blocked(s0.cpu().numpy(), N, N // 32)
    assert np.array_equal(plain0[rows], os0)
    cols = _rows(14, 2)
    cidx = torch.from_numpy(cols).cuda()
    oq1, os1 = oracle.cast_dim1(W.bf16_bits(x[:, cidx]))
    assert np.array_equal(q1[cidx].cpu().numpy(), oq1)
    plain1 = oracle.from_blocked(s1.cpu().numpy(), N, N // 32)
    assert np.array_equal(plain1[cols], os1)
    del q1, s1
    d = mx.dequant_blocked(q0, s0)
    torch.cuda.synchronize()
    want = oracle.dequant_blocked(oq0, oracle.to_blocked(os0))
    got = d[idx].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_tensorwise_beyond_32bit_offsets(big):
    x = big
    q, scale, amax = mx.cast_tensorwise(x)
    torch.cuda.synchronize()
    bits_rows = _rows(10, 3)
    mag = (x.view(torch.int16) & 0x7FFF).amax().item()        # largest magnitude bits
    top_row = int(((x.view(torch.int16) & 0x7FFF) == mag).any(dim=1).nonzero()[0])
    rows = np.unique(np.append(bits_rows, top_row))
    idx = torch.from_numpy(rows).cuda()
    oq, oscale, oamax = oracle.cast_tensorwise(W.bf16_bits(x[idx]))
    assert np.float32(amax.item()) == oamax and np.float32(scale.item()) == oscale
    assert np.array_equal(q[idx].cpu().numpy(), oq)
