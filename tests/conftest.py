import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def parse_golden_blocks(path):
    """Parse tests/golden/hand_worked_blocks.txt into a list of
    (name, is_reading, scale_byte, inputs_u16[32], outputs_u8[32])."""
    def expand(field):
        out = []
        for tok in field.split():
            if "*" in tok:
                n, v = tok.split("*")
                out += [int(v, 16)] * int(n)
            else:
                out.append(int(tok, 16))
        return out

    cases = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            reading = line.startswith("reading:")
            if reading:
                line = line[len("reading:"):].strip()
            name, scale, xs, qs = [p.strip() for p in line.split("|")]
            xs, qs = expand(xs), expand(qs)
            assert len(xs) == 32 and len(qs) == 32, name
            cases.append((name, reading, int(scale, 16), xs, qs))
    return cases


@pytest.fixture(scope="session")
def golden_blocks():
    return parse_golden_blocks(os.path.join(ROOT, "tests", "golden", "hand_worked_blocks.txt"))
