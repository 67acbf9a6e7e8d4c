"""Host-side logic of bench.py, on the CPU: the max-over-ranks reduction
with two gloo ranks, the reference arm's rank handling and JSON line, the
byte formula, and the clock-sample summary."""
import io
import json
import os
import socket
from contextlib import redirect_stdout

import pytest

import bench
import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(values[rank], torch.device("cpu"))))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    values = [3.5, 7.25]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=5) for _ in range(2))
    assert got == {0: 7.25, 1: 7.25}


def test_max_over_ranks_without_group_is_identity():
    import torch
    assert bench.max_over_ranks(1.25, torch.device("cpu")) == 1.25


def test_reference_arm_other_ranks_do_nothing(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1"])
    assert rc == 0 and buf.getvalue() == ""


def test_reference_arm_json_line(monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "3", "--warmup", "1",
                         "--reference-seconds", "1.5", "--workload", "c1"])
    assert rc == 0
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GB/s" and line["value"] > 0 and line["steps"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_algorithmic_bytes_formula(name):
    for p in synth.workload(name):
        read = p.W * p.T * p.H * p.partial_bytes + p.T * p.H * 2 + p.H * 2
        if p.kind == "moe_combine":           # + int32 index and fp32 gate per slot
            read += p.T * p.W * 8
        write = (2 + p.norm_out) * p.T * p.H * 2 + (p.T * p.H + 4 * p.T) * p.fp8_out
        write += (p.T * p.H // 2 + p.T * p.H // 16) * p.nvfp4_out   # codes + block scales
        assert p.algorithmic_bytes() == read + write
        assert bench.call_bytes(p, p.T) == read + write


def test_clock_summary_filters_the_timed_region():
    c = bench.ClockSampler(None)
    c.samples = [(0.0, 1500.0, 2070.0, []), (1.0, 2070.0, 2070.0, []),
                 (1.5, 2060.0, 2070.0, ["sw_power_cap"]), (3.0, 900.0, 2070.0, [])]
    s = c.summary(0.9, 2.0)
    assert s["samples"] == 2 and s["sm_mhz"] == 2065.0 and s["reasons"] == ["sw_power_cap"]
    s = c.summary(2.1, 2.2)                 # nothing inside: nearest samples
    assert s["samples"] > 0 and "nearest" in s["note"]


def test_bars_and_config_summary():
    """The acceptance bars on the fraction of the HBM roofline (75 % for
    T >= 4096, 40 % for T <= 128, none in between) and the per-configuration
    summary bench.py adds to its JSON line."""
    assert bench.bar_for(4096) == 0.75 and bench.bar_for(32768) == 0.75
    assert bench.bar_for(128) == 0.40 and bench.bar_for(1) == 0.40
    assert bench.bar_for(129) is None and bench.bar_for(4095) is None
    probs = synth.workload("decode")[-2:]          # T = 64 and 128
    per_call = [dict(call=p.name, T=p.T, W=p.W, H=p.H, bytes=p.algorithmic_bytes(),
                     kernel_us=t, frac=f) for p, t, f in zip(probs, (2.5, 3.1), (0.37, 0.6))]
    s = bench.config_summary("decode", probs, K=10, ms=0.056, stats={}, calib_ms=0.0056,
                             per_call=per_call, n_sets=3, set_bytes=10 ** 8, l2=10 ** 8,
                             peak=6800.0, world=1, clocks=None)
    step_bytes = sum(p.algorithmic_bytes() for p in probs)
    assert s["bytes_per_step"] == step_bytes and s["rows_per_step"] == 192
    assert abs(s["gbs"] - step_bytes * 10 / 0.056e-3 / 1e9) < 1e-6
    assert abs(s["frac"] - s["gbs"] / 6800.0) < 1e-12
    assert s["bar"]["decode@T64"] == {"target_frac": 0.40, "frac": 0.37, "met": False}
    assert s["bar"]["decode@T128"]["met"] is True
