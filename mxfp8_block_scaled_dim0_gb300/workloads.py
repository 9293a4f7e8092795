"""Seeded synthetic inputs for the MX-FP8 casts.

This module only draws random numbers and shapes; it holds none of the MX
arithmetic, so the CPU oracle and the CUDA path can both take their inputs
from it.  All tensors are bf16 (rounded to nearest even from float32 by
``Tensor.to``) and are drawn from ``torch.Generator`` seeded per workload.

Workloads (shapes and value mixes follow the pages' experiments: MKN
1024..16384 in pytorch/ao PR #1869 "triton kernel to cast to mx across dim0
and dim1", summary; A = (16640, 5120) with 4 groups and B = (E, 8192, 5120)
in pytorch/ao PR #2990 "[mxfp8 moe training] add compile support",
microbenchmark table and perf analysis):

  square1024_spiky    1024 x 1024, N(0,1); 1% of 32-blocks scaled by 2^k,
                      k uniform in [-20, 20]; 0.5% of 32-blocks zeroed
  square4096_wide     4096 x 4096, N(0,1) * row lognormal(0,2) * column
                      lognormal(0,1); 0.1% of 32-blocks zeroed
  square16384_weight  16384 x 16384, N(0,1) * 0.02
  moe16640x5120_g4    16640 x 5120, N(0,1); 4 groups along M, sizes
                      1 + multinomial(16636, uniform over 4)
  experts16x8192x5120 (16, 8192, 5120), N(0,1) * 0.02 * per-expert
                      lognormal(0,1)

"32-blocks" selected for scaling or zeroing are split evenly between row
blocks (1 x 32 along a row) and column blocks (32 x 1 along a column), so both
cast directions see them.
"""
from dataclasses import dataclass
from typing import Optional

import torch

SEED_BASE = 1000


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "2d", "grouped_m" or "3d"
    shape: tuple         # (M, K) or (E, N, K)
    seed: int
    groups: int = 0


WORKLOADS = {
    w.name: w for w in [
        Workload("square1024_spiky", "2d", (1024, 1024), SEED_BASE + 1),
        Workload("square4096_wide", "2d", (4096, 4096), SEED_BASE + 2),
        Workload("square16384_weight", "2d", (16384, 16384), SEED_BASE + 3),
        Workload("moe16640x5120_g4", "grouped_m", (16640, 5120), SEED_BASE + 4, 4),
        Workload("experts16x8192x5120", "3d", (16, 8192, 5120), SEED_BASE + 5),
    ]
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _pick_blocks(x: torch.Tensor, frac: float, g_cpu: torch.Generator):
    """Choose frac of the 32-blocks of a 2D tensor, half along rows and half
    along columns.  Returns (row_blocks, col_blocks) as (r, c0) index pairs:
    row block = x[r, c0:c0+32], column block = x[r0:r0+32, c].  Row blocks
    are drawn from the M * (K // 32) whole blocks along rows; column blocks
    from ceil(M / 32) * K, the last one cut short when M % 32 != 0.  (For M
    and K multiples of 32 both counts are M * K / 32.)"""
    M, K = x.shape
    nb = (M * K) // 32
    n = int(round(frac * nb))
    n_row = n // 2
    n_col = n - n_row
    rb = torch.randperm(M * (K // 32), generator=g_cpu)[:n_row]
    cb = torch.randperm(((M + 31) // 32) * K, generator=g_cpu)[:n_col]
    row_blocks = [(int(i) // (K // 32), (int(i) % (K // 32)) * 32) for i in rb]
    col_blocks = [((int(i) // K) * 32, int(i) % K) for i in cb]
    return row_blocks, col_blocks


def spiky(M: int, K: int, seed: int, device="cpu", scale_frac=0.01,
          zero_frac=0.005, kmin=-20, kmax=20) -> torch.Tensor:
    """N(0,1) with a fraction of 32-blocks scaled by 2^k and some zeroed."""
    g = _gen(seed, device)
    g_cpu = _gen(seed + 7919, "cpu")
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    rows, cols = _pick_blocks(x, scale_frac, g_cpu)
    ks = torch.randint(kmin, kmax + 1, (len(rows) + len(cols),), generator=g_cpu)
    i = 0
    for r, c0 in rows:
        x[r, c0:c0 + 32] *= 2.0 ** int(ks[i]); i += 1
    for r0, c in cols:
        x[r0:r0 + 32, c] *= 2.0 ** int(ks[i]); i += 1
    rows, cols = _pick_blocks(x, zero_frac, g_cpu)
    for r, c0 in rows:
        x[r, c0:c0 + 32] = 0.0
    for r0, c in cols:
        x[r0:r0 + 32, c] = 0.0
    return x.to(torch.bfloat16)


def wide(M: int, K: int, seed: int, device="cpu", zero_frac=0.001) -> torch.Tensor:
    """N(0,1) times per-row lognormal(0,2) and per-column lognormal(0,1)."""
    g = _gen(seed, device)
    g_cpu = _gen(seed + 7919, "cpu")
    z = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    r = torch.exp(2.0 * torch.randn((M, 1), generator=g, device=device))
    c = torch.exp(torch.randn((1, K), generator=g, device=device))
    x = z * r * c
    rows, cols = _pick_blocks(x, zero_frac, g_cpu)
    for rr, c0 in rows:
        x[rr, c0:c0 + 32] = 0.0
    for r0, cc in cols:
        x[r0:r0 + 32, cc] = 0.0
    return x.to(torch.bfloat16)


def normal(shape, seed: int, device="cpu", std=1.0) -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def experts(E: int, N: int, K: int, seed: int, device="cpu", std=0.02) -> torch.Tensor:
    """(E, N, K) weights: N(0,1) * std * per-expert lognormal(0,1)."""
    g = _gen(seed, device)
    x = torch.randn((E, N, K), generator=g, device=device, dtype=torch.float32)
    m = torch.exp(torch.randn((E, 1, 1), generator=g, device=device))
    x.mul_(m * std)
    return x.to(torch.bfloat16)


def group_ends(M: int, G: int, seed: int, min_size: int = 1) -> torch.Tensor:
    """Cumulative group ends (int32, CPU): sizes = min_size + multinomial of
    the remaining rows over G equally likely groups."""
    g = _gen(seed + 104729, "cpu")
    rest = M - min_size * G
    if rest < 0:
        raise ValueError("too many groups for M")
    picks = torch.multinomial(torch.full((G,), 1.0 / G), rest, replacement=True,
                              generator=g) if rest > 0 else torch.zeros(0, dtype=torch.long)
    sizes = torch.bincount(picks, minlength=G) + min_size
    return torch.cumsum(sizes, 0).to(torch.int32)


def make(name: str, device="cpu", rows: Optional[int] = None):
    """Build a named workload.  ``rows`` optionally keeps only the first rows
    of a 2D workload (M) or the first experts of a 3D one (E), for bounded
    samples.  Returns a dict with "x" and, for grouped workloads, "offs"."""
    w = WORKLOADS[name]
    if w.kind == "2d":
        M, K = w.shape
        if rows is not None:
            M = min(M, rows)
        if name.endswith("spiky"):
            x = spiky(M, K, w.seed, device)
        elif name.endswith("wide"):
            x = wide(M, K, w.seed, device)
        else:
            x = normal((M, K), w.seed, device, std=0.02)
        return {"x": x}
    if w.kind == "grouped_m":
        M, K = w.shape
        if rows is not None:
            M = min(M, rows)
        x = normal((M, K), w.seed, device)
        offs = group_ends(M, w.groups, w.seed)
        return {"x": x, "offs": offs}
    E, N, K = w.shape
    if rows is not None:
        E = max(1, min(E, rows))
    return {"x": experts(E, N, K, w.seed, device)}


def bf16_bits(t: torch.Tensor):
    """Raw bf16 bit patterns of a tensor as a numpy uint16 array (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
