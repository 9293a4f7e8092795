"""Host logic of bench.py on CPU: byte accounting, the whole-job value, the
max-over-ranks timing with two gloo ranks, the clock-record parser, and the
traffic file guard."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def test_algorithmic_bytes_match_the_buffers():
    # 16384^2: 2 B read + 2 B written per element + two 8 MiB blocked buffers
    assert bench.algorithmic_bytes(16384, 16384) == 4 * 16384 * 16384 + 2 * 16384 * 512
    # ragged: padded blocked scale buffers are part of what must be written
    assert bench.algorithmic_bytes(160, 96) == 4 * 160 * 96 + 256 * 4 + 128 * 8


def test_whole_job_value():
    assert bench.whole_job_value(1e9, 10, 2, 4.0) == pytest.approx(5.0)


def test_roofline_launch_time_is_bounded_by_the_step_time():
    # One launch per step: the launch's time is the step's time, and the
    # fraction follows from the bytes over it.
    nbytes, steps, elapsed = 1_090_519_040, 20, 20 * 171.9e-6
    r = bench.roofline(nbytes, 1, steps, elapsed, 6791.4, "measured", "k", None, "stream launches")
    ms_per_step = 1e3 * elapsed / steps
    assert r["avg_launch_us"] <= 1000 * ms_per_step / r["launches_per_step"] + 1e-9
    assert r["achieved"] == pytest.approx(nbytes / (elapsed / steps) / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6791.4)
    assert r["frac"] == pytest.approx(bench.whole_job_value(nbytes, steps, 1, elapsed) / 6791.4)
    # Two launches per step (tensorwise): each averages half of the step.
    r2 = bench.roofline(nbytes, 2, steps, elapsed, 6791.4, "measured", "k", None, "x")
    assert r2["avg_launch_us"] == pytest.approx(1000 * ms_per_step / 2)
    assert r2["achieved"] == pytest.approx(r["achieved"])
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r


def test_cpu_baseline_record():
    cb = bench.cpu_baseline(0.3)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0
    assert cb["nproc"] == bench.host_cores() >= 1
    assert 1 <= cb["cores"] <= cb["nproc"]
    assert cb["cores_1"]["value"] > 0 and cb["cores_1"]["unit"] == "GB/s"
    assert isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    import oracle
    assert oracle.threads() == 1   # timing leaves the oracle sequential


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, ws, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    w, r, _ = bench.dist_env()
    bench.barrier(w)
    elapsed = 1.0 + rank            # rank 1 is the slow one
    m = bench.max_over_ranks(elapsed, w)
    out[rank] = (w, r, m, bench.whole_job_value(1e9, 4, w, m))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        w, rr, m, v = out[r]
        assert (w, rr) == (2, r)
        assert m == 2.0                      # the slower rank's time, on every rank
        assert v == pytest.approx(1e9 * 4 * 2 / 2.0 / 1e9)


def test_clock_parser(tmp_path):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "c.csv")
    with open(s.path, "w") as f:
        f.write("0, 1965 MHz, 2070 MHz, 700.00 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 1980 MHz, 2070 MHz, 900.00 W, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 1995 MHz, 2070 MHz, 910.00 W, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n")

    class Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s.proc = Done()
    info = s.stop()
    assert info["sm_mhz"] == 1980.0 and info["sm_max_mhz"] == 2070.0
    assert info["reasons"] == ["sw_power_cap"] and info["samples"] == 3


def test_traffic_is_null_for_other_kernel_code(tmp_path, monkeypatch):
    f = tmp_path / "t.txt"
    f.write_text("kernel_source_sha256_16: 0000000000000000\ndram_bytes_per_full_launch: 123\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.measured_traffic() is None
    f.write_text("kernel_source_sha256_16: %s\ndram_bytes_per_full_launch: 123\n"
                 % bench.kernel_source_hash())
    assert bench.measured_traffic() == 123.0


def test_kernel_hash_ignores_comments_and_layout():
    import bench
    a = "int f(int x) {\n  return x + 1;  // one more\n}\n"
    b = "/* header */\nint f(int x) { return x + 1; }\n"
    c = "int f(int x) { return x + 2; }\n"
    assert bench._code_tokens(a) == bench._code_tokens(b)
    assert bench._code_tokens(a) != bench._code_tokens(c)


def test_reference_arm_prints_the_contract_line(capsys, monkeypatch):
    """The reference arm (the oracle on the host cores) runs without a GPU:
    one JSON line with every key the bench contract asks of it."""
    import argparse
    import json
    for var in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    args = argparse.Namespace(gpus=1, steps=2, warmup=1)
    assert bench.run_reference(args, budget_s=1.5) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["higher_is_better"] is True and line["vs_baseline"] is None
    assert line["steps"] == 2 and line["warmup"] == 1 and line["n_gpus"] == 1
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert cb["nproc"] >= cb["cores"] and cb["cores_1"]["value"] > 0 and cb["cpu_model"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "square16384_weight"
