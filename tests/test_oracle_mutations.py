"""The oracle pins catch planted mistakes.

Each case copies the oracle's C source, plants one plausible mistake (a wrong
exponent offset, a wrong layout formula, a reversed dim1 index, round half up,
a dropped saturation, wrong group column offsets, flushed bf16 subnormals, a
scale not rounded to fp32, unpadded 3D expert scales, a dequantisation
exponent off by one, a wrong rowwise divisor), builds it into a
temporary library, swaps it in for the real oracle and runs the pins that
should notice.  At least one of them must fail; the unmutated oracle passes
them all (the ordinary pin run).  Everything runs on the CPU.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from oracle import build as obuild
import test_oracle_pins as pins
from conftest import ROOT, parse_golden_blocks

GOLDEN = os.path.join(ROOT, "tests", "golden", "hand_worked_blocks.txt")


def _golden():
    return parse_golden_blocks(GOLDEN)


# (name, source text to replace, replacement, pins that must notice)
MUTATIONS = [
    ("exponent offset -7 instead of -8",
     "int e = (p - 1) - E4M3_EMAX;", "int e = (p - 1) - E4M3_EMAX + 1;",
     [lambda: pins.test_hand_worked_blocks_dim0_and_dim1(_golden()),
      pins.test_scale_closed_form_all_magnitudes]),
    ("blocked layout with row group and column swapped",
     "out[tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + cc] = s[r * C + c];",
     "out[tile * 512 + (rr % 32) * 16 + (rr / 32) + cc * 4] = s[r * C + c];",
     [pins.test_blocked_single_tile_positions, pins.test_blocked_hand_examples]),
    ("dim1 bytes reversed inside a block",
     "q[k * M + j * MX_BLOCK + i] = qb[i];",
     "q[k * M + j * MX_BLOCK + (MX_BLOCK - 1 - i)] = qb[i];",
     [lambda: pins.test_dim1_equals_dim0_of_transpose("wide"),
      lambda: pins.test_hand_worked_blocks_dim0_and_dim1(_golden())]),
    ("e4m3 rounding half up instead of half to even",
     "double r = nearbyint(a / spacing) * spacing;   /* ties to even */",
     "double r = floor(a / spacing + 0.5) * spacing;   /* ties to even */",
     [lambda: pins.test_hand_worked_blocks_dim0_and_dim1(_golden()),
      pins.test_element_cast_exhaustive_vs_libraries]),
    ("no saturation at 448",
     "    if (r > E4M3_MAXNORM)\n        r = E4M3_MAXNORM;",
     "    if (0)\n        r = E4M3_MAXNORM;",
     [lambda: pins.test_hand_worked_blocks_dim0_and_dim1(_golden()),
      pins.test_element_cast_exhaustive_vs_libraries]),
    ("group dim1 column offsets by 32-row blocks",
     "s1_col_offs[g + 1] = s1_col_offs[g] + ceil_div(mg, 128) * 4;",
     "s1_col_offs[g + 1] = s1_col_offs[g] + ceil_div(mg, 32);",
     [pins.test_grouped_ragged_groups_match_standalone_casts]),
    ("bf16 rounding flushes subnormals",
     "    if (e < -126)\n        e = -126;", "    if (0)\n        e = -126;",
     [pins.test_dequant_hand_worked, pins.test_dequant_every_element_every_scale]),
    ("tensorwise scale not rounded to fp32",
     "s = to_f32(E4M3_MAXNORM / amax);", "s = E4M3_MAXNORM / amax;",
     [lambda: pins.test_tensorwise_against_float32_arithmetic("wide"),
      pins.test_scaled_fp8_hand_worked,
      lambda: pins.test_tensorwise_every_element_under_inexact_scales(13.0)]),
    ("3D dim0 expert scales packed without per-expert padding",
     "oracle_to_blocked(s0 + e * N * Kb, N, Kb, s0_blk + e * per);",
     "oracle_to_blocked(s0 + e * N * Kb, N, Kb, s0_blk + e * N * Kb);",
     [pins.test_3d_dim0_reductions]),
    ("dequantisation scale exponent off by one",
     "oracle_double_to_bf16(ldexp(v, (int)sc - E8M0_BIAS))",
     "oracle_double_to_bf16(ldexp(v, (int)sc - E8M0_BIAS + 1))",
     [pins.test_dequant_hand_worked, pins.test_dequant_round_trip_exact_blocks]),
    ("rowwise scale from a 480 divisor",
     "uint16_t sb = oracle_double_to_bf16(amax / E4M3_MAXNORM);",
     "uint16_t sb = oracle_double_to_bf16(amax / 480.0);",
     [pins.test_scaled_fp8_hand_worked,
      lambda: pins.test_rowwise_against_float32_arithmetic("wide")]),
]


def _build_mutant(tmp_path, old, new):
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, "mutation anchor not found exactly once: %r" % old
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fno-fast-math", "-fPIC", "-shared", "-o",
                    str(lib), str(path), "-lm"], check=True, capture_output=True)
    return str(lib)


@pytest.mark.parametrize("name,old,new,checks", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, name, old, new, checks):
    lib = oracle._configure(ctypes.CDLL(_build_mutant(tmp_path, old, new)))
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = 0
    for check in checks:
        try:
            check()
        except AssertionError:
            caught += 1
    assert caught >= 1, "no pin noticed: %s" % name
