"""Host-side logic of bench.py: replica aggregation over ranks (gloo, world size 2), the
reference arm's rank handling, the clock-sample parser and the traffic bookkeeping."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _agg_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, units = bench.aggregate(10.0 + rank, 100.0 * (rank + 1), world)
        q.put((rank, ms, units))
    finally:
        dist.destroy_process_group()


def test_aggregate_max_time_sum_units_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_agg_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, units in got:
        assert ms == 11.0          # the slowest rank's time
        assert units == 300.0      # every rank's work


def test_aggregate_single_rank_is_identity():
    assert bench.aggregate(3.5, 7.0, 1) == (3.5, 7.0)


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--gpus", "2"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip())
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert "workload" in line["config"]


def test_warmup_below_three_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_clock_summary_parses_samples_and_reasons():
    c = bench.ClockSampler("GPU-1234-abcd")
    c.out = "\n".join([
        "GPU-1234-abcd, 1965, 2070, 900.1, Not Active, Not Active, Not Active, Not Active",
        "GPU-1234-abcd, 1980, 2070, 1100.0, Not Active, Not Active, Not Active, Active",
        "GPU-9999-ffff, 300, 2070, 100.0, Active, Not Active, Not Active, Not Active",
        "GPU-1234-abcd, 1995, 2070, 1200.0, Not Active, Not Active, Not Active, Active",
    ])
    s = c.summary()
    assert s["sm_mhz"] == 1980 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_without_samples_is_none():
    c = bench.ClockSampler(None)
    c.out = ""
    assert c.summary() is None


def test_traffic_is_null_when_sources_differ(monkeypatch):
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "0" * 16)
    assert bench.dram_traffic_per_launch() is None


def test_weight_bytes_of_the_step():
    # four matrices of 50,135,040 bytes (4.5 bits per weight)
    assert bench.weight_bytes_per_step() == 4 * 50135040


def test_launch_count_rule_matches_the_planner():
    """bench.py counts one kernel per one-token call whose row is quantized inside the engine;
    the row-length limit must be the planner's."""
    import re
    here = os.path.dirname(os.path.abspath(__file__))
    src = open(os.path.join(here, "..", "gguf_block_quantized_quant_gb300", "csrc", "qg_plan.h")).read()
    m = re.search(r"constexpr int ONE_FUSED_K_MAX = (\d+);", src)
    assert m is not None
    import bench
    assert bench.ONE_FUSED_K_MAX == int(m.group(1))
