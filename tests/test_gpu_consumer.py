"""The blocked scale layout as a real consumer reads it: a block-scaled
MX-FP8 GEMM (torch._scaled_mm with e8m0 scales, cuBLAS) on the cast outputs
must equal the GEMM of the dequantised values.  A wrong tile order, storage
row or padding would scramble the scales and the products.  Both directions
are checked: dim0 copies contract over K, dim1 copies over M.  Skipped when
this torch build has no MX-FP8 _scaled_mm."""
import numpy as np
import pytest
import torch

import oracle
import mxfp8_block_scaled_dim0_gb300 as mx
from mxfp8_block_scaled_dim0_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def dequant(q, s_plain):
    """float64 values of e4m3 bytes q (R x C) with plain e8m0 scales (R x C/32)."""
    e4 = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    scale = np.exp2(np.repeat(s_plain.astype(np.float64), 32, axis=1) - 127.0)
    return e4 * scale


def scaled_mm(a_q, b_q_t, a_s, b_s):
    return torch._scaled_mm(a_q.view(torch.float8_e4m3fn), b_q_t.view(torch.float8_e4m3fn),
                            a_s.view(torch.float8_e8m0fnu), b_s.view(torch.float8_e8m0fnu),
                            out_dtype=torch.float32)


def check(got, want):
    got = got.double().cpu().numpy()
    err = np.abs(got - want) / (np.abs(want).max() + 1e-30)
    assert err.max() < 1e-5, err.max()


def test_blocked_scales_feed_block_scaled_gemm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, N, K = 256, 384, 512
    x = W.wide(M, K, 61, zero_frac=0.0).cuda()
    y = W.wide(N, K, 62, zero_frac=0.0).cuda()
    qx0, sx0, qx1, sx1 = mx.cast_dim0_dim1(x)
    qy0, sy0, qy1, sy1 = mx.cast_dim0_dim1(y)
    torch.cuda.synchronize()
    try:
        c = scaled_mm(qx0, qy0.t(), sx0, sy0)          # (M, K) @ (K, N), blocks along K
    except (RuntimeError, TypeError, ValueError) as e:
        pytest.skip("no MX-FP8 torch._scaled_mm here: %s" % str(e).splitlines()[0][:120])
    torch.cuda.synchronize()
    ax = dequant(qx0.cpu().numpy(), oracle.from_blocked(sx0.cpu().numpy(), M, K // 32))
    ay = dequant(qy0.cpu().numpy(), oracle.from_blocked(sy0.cpu().numpy(), N, K // 32))
    check(c, ax @ ay.T)
    # dim1 copies: (K, M) @ (M, N') with blocks along M, the contraction
    z = W.wide(M, 128, 63, zero_frac=0.0).cuda()
    qz0, sz0, qz1, sz1 = mx.cast_dim0_dim1(z)
    torch.cuda.synchronize()
    c1 = scaled_mm(qx1, qz1.t(), sx1, sz1)              # (K, M) @ (M, 128)
    torch.cuda.synchronize()
    bx = dequant(qx1.cpu().numpy(), oracle.from_blocked(sx1.cpu().numpy(), K, M // 32))
    bz = dequant(qz1.cpu().numpy(), oracle.from_blocked(sz1.cpu().numpy(), 128, M // 32))
    check(c1, bx @ bz.T)
