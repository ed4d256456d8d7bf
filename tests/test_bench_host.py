"""Host-side logic of bench.py: multi-rank aggregation over gloo (world size 2,
CPU), clock-sample parsing, traffic lookup, and the reference arm's rank rule."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_aggregate_takes_the_slowest_rank():
    r = bench.aggregate([2.0, 4.0], flops_per_rank=8e12)
    assert r["ms_per_step"] == 4.0
    assert abs(r["value_tflops"] - 2 * 8e12 / 4e-3 / 1e12) < 1e-9
    r1 = bench.aggregate([2.0], flops_per_rank=8e12)
    assert abs(r1["value_tflops"] - 4000.0) < 1e-9


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    times = bench.gather_max(1.5 + rank, world)       # rank r measured 1.5 + r ms per step
    bench.barrier(world)
    agg = bench.aggregate(times, 1e12)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"times": times, "agg": agg}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for r in res:
        assert r["times"] == [1.5, 2.5]
        assert r["agg"]["ms_per_step"] == 2.5
        assert abs(r["agg"]["value_tflops"] - 2 * 1e12 / 2.5e-3 / 1e12) < 1e-9


def test_clock_sampler_parses_samples(tmp_path):
    p = tmp_path / "c.csv"
    p.write_text("0, 1980, 2070, 1200.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
                 "0, 1965, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
                 "0, 2070, 2070, 150.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n")
    cs = bench.ClockSampler(0)
    cs.proc, cs.path = object(), str(p)
    s = cs.summary()
    assert s["sm_mhz"] == pytest.approx(1972.5)        # median of the samples under load
    assert s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_sampler_nvml_samples():
    # NVML's reason bits: 0x4 software power cap, 0x8 hardware slowdown, 0x20 software
    # thermal, 0x40 hardware thermal (the NVML header's nvmlClocksEventReason* values).
    assert bench.nvml_reason_flags(0x0) == ["Not Active"] * 4
    assert bench.nvml_reason_flags(0x48) == ["Active", "Active", "Not Active", "Not Active"]
    assert bench.nvml_reason_flags(0x24) == ["Not Active", "Not Active", "Active", "Active"]
    cs = bench.ClockSampler(0)
    cs.rows = [(1980.0, 2070.0, 1200.5, bench.nvml_reason_flags(0x4)),
               (1965.0, 2070.0, 1350.0, bench.nvml_reason_flags(0x4)),
               (2070.0, 2070.0, 150.0, bench.nvml_reason_flags(0x1))]      # idle sample
    s = cs.summary()
    assert s["source"] == "nvml" and s["samples"] == 3 and s["samples_under_load"] == 2
    assert s["sm_mhz"] == pytest.approx(1972.5)
    assert s["reasons"] == ["sw_power_cap"]


def test_recorded_traffic_needs_current_sources():
    # Returns an int only for a workload listed with the current source digest, else None.
    v = bench.recorded_traffic("no_such_workload")
    assert v is None


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0
    assert out.stdout.strip() == ""


def test_reference_arm_stays_within_minutes():
    import bench
    for steps, warmup in [(3000, 50), (1, 0), (20, 3), (100000, 10)]:
        per = bench.reference_step_seconds(steps, warmup)
        total = per * (steps + warmup / 4)
        assert 0.01 <= per <= 10.0
        assert total <= 70.0 or per == 0.01, (steps, warmup, total)


def test_code_digest_ignores_comments_and_blank_lines():
    # the traffic record is keyed by this digest: documentation edits must not change it
    from grouped_gemm_persistent_gb300.build import _strip_comments, code_digest
    src = 'int a = 1; // note\n/* block\n comment */ const char* s = "a//b /* c */";\n\n  char q = \'"\'; int b; /* t */\n'
    assert _strip_comments(src) == 'int a = 1;\n const char* s = "a//b /* c */";\n  char q = \'"\'; int b;'
    assert _strip_comments("x = 1;  // one\n") == _strip_comments("x = 1;\n\n/* two */\n")
    assert _strip_comments("x = 1;") != _strip_comments("x = 2;")
    assert code_digest() == code_digest() and len(code_digest()) == 64
