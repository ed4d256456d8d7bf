#!/usr/bin/env python
"""Benchmark of the bf16 GEMM / grouped GEMM hot path (TFLOP/s, % of dense-bf16 peak).

One step = one pass of the whole hot path over one batch of synthetic input:
  * dense GEMM M=N=K=4096, A row-major, B column-major, U(-1,1), fused
    bias + GELU(tanh), bf16 out (seed 1),
  * dense GEMM M=N=K=8192, A and B row-major, N(0,1)/sqrt(K), fp32 out (seed 2), and
  * grouped MoE GEMM, 64 experts, K=4096, N=1536, 65536 tokens split by a
    Dirichlet(0.5) multinomial (seed 3), bf16 out,
each one launch of the persistent kernel through the C ABI (plus the small
counter reset before a dense stream-K launch).  Each part is timed with CUDA
events on the launching stream every step; value = FLOPs of the step / the sum
of the parts' median step times (mean, p10 and p90 are reported beside it).
L2 (129 MB) is flushed between timed steps by writing a 256 MiB buffer (and then
reading another, so the written lines go back to HBM before the next step) outside
the timed events.  `e2e` times the same steps through the public API with the
inputs copied from pinned host memory every step and C read back, pipelined
across two device buffer sets (step i's upload overlaps step i-1's kernels).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Under torchrun (N > 1) every rank runs the same per-GPU workload (independent
problems, weak scaling, no data-path collective); the time is the max over ranks
and value is the work of all ranks over that time.  `--impl reference` times
the CPU oracle (the plain fp64 definition) on bounded samples of the workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "dense4096_bias_gelu+dense8192_f32+grouped_moe"
WORKLOADS = {
    HEADLINE: ["dense_4096_bias_gelu", "dense_8192_f32", "grouped_moe"],
    "dense4096_bias_gelu+grouped_moe": ["dense_4096_bias_gelu", "grouped_moe"],
    "dense_4096_bias_gelu": ["dense_4096_bias_gelu"],
    "dense_8192_f32": ["dense_8192_f32"],
    "grouped_moe": ["grouped_moe"],
    "grouped_moe_devcounts": ["grouped_moe_devcounts"],
    "skinny_bcast": ["skinny_bcast"],
    "skinny_bcast_ikbo": ["skinny_bcast_ikbo"],
    "dense_256": ["dense_256"],
    "dense_4096_rmsnorm_bias_gelu": ["dense_4096_bias_gelu_rmsnorm"],
}
RMS_EPS = 1e-6
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
NOMINAL_BF16_TFLOPS = 2250.0   # GB300 dense bf16 (without 2:4 sparsity)
METRIC = "bf16 GEMM TFLOP/s and % of GB300 dense-BF16 peak (dense + grouped)"


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------------------------------
# distributed plumbing (host side; the data path has no collective)

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(step_ms_per_rank: list[float], flops_per_rank: float) -> dict:
    """Whole-job numbers from per-rank step times: the job is as slow as its slowest rank."""
    world = len(step_ms_per_rank)
    t = max(step_ms_per_rank)
    return {"ms_per_step": t, "value_tflops": world * flops_per_rank / (t * 1e-3) / 1e12}


def gather_max(x: float, world: int) -> list[float]:
    if world == 1:
        return [x]
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    out = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(out, t)
    return [float(v.item()) for v in out]


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------------------------
# peaks, clocks, traffic

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# NVML clock-event reason bits (nvmlClocksEventReason*) for the reasons the line reports.
NVML_REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                    "hw_thermal_slowdown": 0x40}
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def nvml_reason_flags(mask: int) -> list[str]:
    """NVML's clock-event reason bit mask -> "Active" / "Not Active" per REASON_NAMES."""
    return ["Active" if mask & NVML_REASON_BITS[n] else "Not Active" for n in REASON_NAMES]


class _Nvml:
    """Read-only NVML queries through the driver's own library (no Python package needed):
    SM clock, its maximum, board power and the clock-event reasons of one device."""

    def __init__(self, torch_index: int):
        import ctypes
        import torch
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        props = torch.cuda.get_device_properties(torch_index)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.h)) != 0:
            lib.nvmlShutdown()
            raise OSError("no NVML device for " + bus.decode())
        try:
            self.reasons_fn = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        ct, lib, h = self.ct, self.lib, self.h
        sm, mx, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if (lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(sm)) != 0 or lib.nvmlDeviceGetMaxClockInfo(h, 1, ct.byref(mx)) != 0
                or lib.nvmlDeviceGetPowerUsage(h, ct.byref(mw)) != 0 or self.reasons_fn(h, ct.byref(rs)) != 0):
            return None
        return (float(sm.value), float(mx.value), mw.value / 1000.0, nvml_reason_flags(rs.value))

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock, power and throttle reasons sampled while the timed region runs: every ~2 ms
    through NVML when the driver's library loads, else nvidia-smi every 100 ms (short timed
    regions then catch few samples)."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.002

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.nvml = None
        self.rows = None
        self.thread = None
        self.stop = None

    def _nvml_loop(self):
        while not self.stop.is_set():
            r = self.nvml.sample()
            if r is not None:
                self.rows.append(r)
            time.sleep(self.PERIOD_S)

    def __enter__(self):
        try:
            import threading
            self.nvml = _Nvml(self.gpu)
            self.rows, self.stop = [], threading.Event()
            self.thread = threading.Thread(target=self._nvml_loop, daemon=True)
            self.thread.start()
            return self
        except (OSError, AttributeError, ImportError):
            self.nvml = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=5)
            self.nvml.close()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.rows is not None:
            rows, source = self.rows, "nvml"
        elif self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        else:
            rows, source = [], "nvidia-smi"
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": source}
        reasons = sorted({REASON_NAMES[i] for _, _, _, flags in rows for i, f in enumerate(flags) if f.lower() == "active"})
        pmax = max(r[2] for r in rows)
        loaded = [r for r in rows if r[2] >= 0.5 * pmax] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded), "power_w_max": pmax,
                "source": source}


def recorded_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernel code
    (the digest ignores comments, so documentation edits keep the record valid)."""
    from grouped_gemm_persistent_gb300.build import code_digest
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    digest = code_digest()[:16]
    for line in open(path):
        parts = line.split()
        if len(parts) == 4 and parts[0] == "traffic" and parts[1] == kernel_key and parts[2] == digest:
            return int(parts[3])
    return None


# ------------------------------------------------------------------------------------------
# statistics of per-step times

def step_stats(ms: list[float]) -> dict:
    """Median, mean and the 10th / 90th percentiles of per-step times (ms)."""
    a = np.asarray(ms, dtype=np.float64)
    return {"median": float(np.median(a)), "mean": float(a.mean()), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90)), "min": float(a.min()), "max": float(a.max()), "n": int(a.size)}


# ------------------------------------------------------------------------------------------
# workload construction (inputs generated on the CPU from the seeded generators)

class Part:
    def __init__(self, name):
        from grouped_gemm_persistent_gb300 import workloads as wl
        self.name = name
        self.grouped = name in wl.GROUPED_WORKLOADS
        self.bcast = name.endswith("_ikbo")          # in-kernel broadcast form of a repeated-row workload
        self.devcounts = name.endswith("_devcounts")  # MoE with the token counts in device memory
        self.rmsnorm = name.endswith("_rmsnorm")      # RMS normalisation of A's rows fused into the GEMM
        base = name
        for suffix in ("_ikbo", "_devcounts", "_rmsnorm"):
            if base.endswith(suffix):
                base = base[: -len(suffix)]
        self.grouped = self.grouped or self.devcounts
        self.case = wl.grouped_case(base) if self.grouped else wl.dense_case(base)
        self.flops = self.case.flops
        self.bytes = self.case.bcast_bytes if self.bcast else self.case.algorithmic_bytes
        if self.rmsnorm:
            # the row-statistics pass reads A once more and writes/reads one fp32 factor per row
            self.bytes += self.case.M * self.case.K * 2 + 8 * self.case.M
        # the broadcast form stores far more than it computes: its roofline is the C write
        self.bound = "hbm" if (self.bcast or self.flops / self.bytes < 300) else "tensor"

    def describe(self):
        c = self.case
        if self.grouped:
            return {"name": self.name, "G": c.G, "K": c.K, "N": c.N, "tokens": int(c.counts.sum()),
                    "empty_groups": int((c.counts == 0).sum()), "out": c.c_dtype, "epilogue": c.epi,
                    "inputs": c.recipe}
        if self.bcast:
            return {"name": self.name, "M": c.M, "N": c.N, "K": c.K, "users": c.users.shape[0], "repeat": c.repeat,
                    "out": c.c_dtype, "epilogue": c.epi, "inputs": c.recipe,
                    "form": "in-kernel broadcast of the user rows (A not materialised)"}
        d = {"name": self.name, "M": c.M, "N": c.N, "K": c.K, "a": "col" if c.a_col_major else "row",
             "b": "col" if c.b_col_major else "row", "out": c.c_dtype, "epilogue": c.epi, "inputs": c.recipe}
        if self.rmsnorm:
            d["norm"] = f"RMS of A's rows (eps {RMS_EPS}): row-statistics pass + row scale in the GEMM epilogue"
        return d

    # -- device side
    def to_device(self, torch):
        c = self.case
        a_src = c.users if self.bcast else c.a
        self.host = {"a": a_src.contiguous().pin_memory(), "b": c.b.contiguous().pin_memory()}
        if c.bias is not None:
            self.host["bias"] = c.bias.contiguous().pin_memory()
        self.dev = {k: v.cuda() for k, v in self.host.items()}
        dt = torch.float32 if c.c_dtype == "f32" else torch.bfloat16
        rows = int(c.counts.sum()) if self.grouped else c.M
        self.dev["out"] = torch.empty((rows, c.N), dtype=dt, device="cuda")
        self.host["out"] = torch.empty((rows, c.N), dtype=dt).pin_memory()
        if self.devcounts:
            self.dev_counts = torch.tensor(c.counts, dtype=torch.int32, device="cuda")
        if self.rmsnorm:
            self.dev["row_scale"] = torch.empty(c.M, dtype=torch.float32, device="cuda")
        self.sets = [self.dev]
        self.tables = []
        if self.grouped:
            import grouped_gemm_persistent_gb300 as tg
            self.tables.append(tg.build_moe_table(self.dev["a"], self.dev["b"], c.counts, self.dev["out"],
                                                  bias=self.dev.get("bias"), epilogue=c.epi))
        self.h2d_bytes = sum(v.numel() * v.element_size() for k, v in self.host.items() if k != "out")
        self.d2h_bytes = self.host["out"].numel() * self.host["out"].element_size()

    def add_buffer_set(self, torch):
        """A second set of device inputs and outputs, so the end-to-end loop can copy one
        step's inputs while the previous step computes on the other set."""
        d = {k: torch.empty_like(v) for k, v in self.dev.items()}
        self.sets.append(d)
        if self.grouped:
            import grouped_gemm_persistent_gb300 as tg
            self.tables.append(tg.build_moe_table(d["a"], d["b"], self.case.counts, d["out"],
                                                  bias=d.get("bias"), epilogue=self.case.epi))

    def h2d(self, k):
        for name, v in self.host.items():
            if name not in ("out", "row_scale"):
                self.sets[k][name].copy_(v, non_blocking=True)

    def d2h(self, k):
        self.host["out"].copy_(self.sets[k]["out"], non_blocking=True)

    def launch(self, stream, k=0):
        import grouped_gemm_persistent_gb300 as tg
        c, d = self.case, self.sets[k]
        if self.devcounts:
            tg.moe_gemm_device(d["a"], d["b"], self.dev_counts, d["out"], bias=d.get("bias"), epilogue=c.epi,
                               stream=stream)
        elif self.grouped:
            tg.grouped_gemm_table(self.tables[k], stream)
        elif self.bcast:
            tg.gemm_bcast(d["a"], d["b"], c.repeat, d["out"], bias=d.get("bias"), epilogue=c.epi, stream=stream)
        elif self.rmsnorm:
            b = d["b"].t() if c.b_col_major else d["b"]
            tg.gemm_rmsnorm(d["a"], b, RMS_EPS, d["out"], row_scale=d["row_scale"], bias=d.get("bias"),
                            epilogue=c.epi, stream=stream)
        else:
            a = d["a"].t() if c.a_col_major else d["a"]
            b = d["b"].t() if c.b_col_major else d["b"]
            tg.gemm(a, b, d["out"], bias=d.get("bias"), epilogue=c.epi, stream=stream)


    # -- oracle side (CPU baseline): rows of this part, FLOPs done
    def prepare_oracle(self):
        """The oracle's inputs as bf16 bit patterns, converted once, outside any timing."""
        from grouped_gemm_persistent_gb300 import workloads as wl
        c = self.case
        if self.grouped:
            g = int(np.argmax(c.counts))
            r0, r1 = c.offsets[g], c.offsets[g + 1]
            self._obits = (g, wl.bf16_bits(c.a[r0:r1]), wl.bf16_bits(c.b[g]), None)
        else:
            bias = wl.bf16_bits(c.bias) if c.bias is not None else None
            self._obits = (0, wl.bf16_bits(c.a), wl.bf16_bits(c.b), bias)

    def oracle_rows(self, n_rows: int, seed: int):
        """The oracle on a random sample of C: n_rows rows of the part (the largest expert's,
        for a grouped part) times a random block of up to 256 columns, from the same
        inputs.  Returns (FLOPs, rows)."""
        import oracle
        c = self.case
        if not hasattr(self, "_obits"):
            self.prepare_oracle()
        g, a_bits, b_bits, bias = self._obits
        rng = np.random.default_rng(seed)
        m = a_bits.shape[0] if self.grouped else c.M
        rows = np.sort(rng.choice(m, size=min(n_rows, m), replace=False))
        nc = min(256, c.N)
        c0 = int(rng.integers(0, c.N - nc + 1))
        b_col = (not self.grouped) and c.b_col_major
        b_sub = b_bits[c0:c0 + nc] if b_col else np.ascontiguousarray(b_bits[:, c0:c0 + nc])
        if self.grouped:
            oracle.gemm(a_bits, b_sub, rows=rows)
        else:
            oracle.gemm(a_bits, b_sub, a_col_major=c.a_col_major, b_col_major=b_col,
                        bias=None if bias is None else bias[c0:c0 + nc], epi=c.epi, rows=rows,
                        row_norm_eps=RMS_EPS if self.rmsnorm else None)
        return 2 * len(rows) * nc * c.K, len(rows)


def oracle_sample(parts, target_s: float, seed: int = 0):
    """Time the oracle on growing row samples of every part until about target_s seconds of work."""
    import oracle
    flops, secs, rows_done = 0, 0.0, {}
    n = 8
    share = target_s / len(parts)
    for p in parts:
        spent, r_total = 0.0, 0
        n = 8
        while spent < share:
            t0 = time.perf_counter()
            f, done = p.oracle_rows(n, seed + r_total)
            dt = time.perf_counter() - t0
            flops += f
            spent += dt
            r_total += done
            if spent < share:
                n = int(min(max(n * 2, n * (share - spent) / max(dt, 1e-3)), 4096))
        secs += spent
        rows_done[p.name] = r_total
    return {"flops": flops, "seconds": secs, "rows": rows_done, "cores": oracle.num_threads()}


# ------------------------------------------------------------------------------------------
# arms

def reference_step_seconds(steps: int, warmup: int) -> float:
    """Oracle work per timed step of the reference arm: about 60 s for the whole run
    (warm-up steps count a quarter; the last call of a step overshoots its share, so the
    run takes about twice that), whatever --steps and --warmup are, between 0.01 s (at
    least one small sample) and 10 s per step."""
    return max(0.01, min(10.0, 60.0 / max(1.0, steps + warmup / 4)))


def run_reference(args, parts_names):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    parts = [Part(n) for n in parts_names]
    for p in parts:
        p.prepare_oracle()
    per_step_s = reference_step_seconds(args.steps, args.warmup)
    # Step i samples part i mod len(parts): one oracle call per step keeps the whole run
    # within minutes even at thousands of steps (a call re-widens the part's whole B).
    for i in range(args.warmup):
        oracle_sample([parts[i % len(parts)]], per_step_s / 4)
    times, flops = [], 0
    for i in range(args.steps):
        r = oracle_sample([parts[i % len(parts)]], per_step_s, seed=1000 + i)
        times.append(r["seconds"])
        flops += r["flops"]
    total = sum(times)
    value = flops / total / 1e12
    sample = (f"step i: oracle (fp64 CPU) on random output rows x a 256-column block of part i mod {len(parts)}, about "
              f"{per_step_s:.3f} s of work (at least one call); last step rows {r['rows']}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "parts": [p.describe() for p in parts]},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, parts_names):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    import grouped_gemm_persistent_gb300 as tg
    from grouped_gemm_persistent_gb300.build import build
    if rank == 0:
        build()
    barrier(world)
    tg.load()

    t0 = time.perf_counter()
    parts = [Part(n) for n in parts_names]
    for p in parts:
        p.to_device(torch)
    log(f"[bench] inputs ready in {time.perf_counter() - t0:.1f} s")
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    # read after the flush write: evicts the write's dirty lines, so their write-back to
    # HBM happens here and not inside the next timed step
    flush_read = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    step_flops = sum(p.flops for p in parts)

    for _ in range(args.warmup):
        for p in parts:
            p.launch(stream)
    tg.device_status(stream)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)] for _ in range(args.steps)]
    launches0 = tg.launch_count()
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        for i in range(args.steps):
            if not args.warm:
                flush.zero_()                 # L2 flush, outside the timed events
                flush_read.sum()
            ev[i][0].record(stream)
            for j, p in enumerate(parts):
                p.launch(stream)
                ev[i][j + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
    launches = tg.launch_count() - launches0      # kernels of this library enqueued in the timed region
    tg.device_status(stream)
    part_ms = [[ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps)] for j in range(len(parts))]
    part_stats = [step_stats(x) for x in part_ms]
    step_ms = sum(st["median"] for st in part_stats)
    agg = aggregate(gather_max(step_ms, world), step_flops)

    # End to end through the public API: every step copies its inputs from pinned host
    # memory, runs the step and reads C back.  The loop is pipelined the way a serving
    # or training loop runs: two device buffer sets; step i's inputs are copied (copy
    # stream) while step i - 1 computes, and its C is read back (second copy stream)
    # while step i + 1 computes.  Dependencies are CUDA events between the streams.
    e2e = None
    if not args.no_e2e:
        for p in parts:
            p.add_buffer_set(torch)
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        e2e_steps = max(1, min(args.steps, args.e2e_steps))

        def e2e_loop(n_steps):
            launches_n = tg.launch_count()
            for i in range(n_steps):
                k = i % 2
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(comp_done[k])        # step i - 2 has read set k
                    for p in parts:
                        p.h2d(k)
                    h2d_done[k].record(s_in)
                stream.wait_event(h2d_done[k])
                if i >= 2:
                    stream.wait_event(d2h_done[k])           # step i - 2's C has left set k
                for p in parts:
                    p.launch(stream, k)
                comp_done[k].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[k])
                    for p in parts:
                        p.d2h(k)
                    d2h_done[k].record(s_out)
            return tg.launch_count() - launches_n

        e2e_loop(2)                                          # warm-up
        torch.cuda.synchronize()
        barrier(world)
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(s_in)
        launches_e2e = e2e_loop(e2e_steps)
        s_out.wait_event(comp_done[(e2e_steps - 1) % 2])
        s1.record(s_out)
        torch.cuda.synchronize()
        tg.device_status(stream)
        e2e_ms = s0.elapsed_time(s1) / e2e_steps
        e2e_agg = aggregate(gather_max(e2e_ms, world), step_flops)
        e2e = {"value": e2e_agg["value_tflops"], "unit": "TFLOP/s",
               "h2d_bytes_per_step": sum(p.h2d_bytes for p in parts),
               "d2h_bytes_per_step": sum(p.d2h_bytes for p in parts),
               "ms_per_step": e2e_agg["ms_per_step"], "steps": e2e_steps, "gpu_launches": launches_e2e,
               "pipelined": "step i's host-to-device copy overlaps step i-1's kernels and step i-2's "
                            "device-to-host copy (two device buffer sets, two copy streams)"}

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peaks, peak_src = load_peaks()
    # A timed region of a second or more runs at the power cap: compare with the
    # sustained cuBLAS figure; shorter bursts with the burst figure.
    timed_s = sum(sum(x) for x in part_ms) * 1e-3
    sustained = timed_s >= 1.0 and "bf16_tflops_sustained" in peaks
    # dominant kernel: the part with the largest device time
    dom = max(range(len(parts)), key=lambda j: part_stats[j]["median"])
    dp = parts[dom]
    dom_ms = part_stats[dom]["median"]
    peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    peak_kind = "bf16_tflops_sustained (timed region %.1f s)" % timed_s if sustained else "bf16_tflops (burst)"
    traffic = recorded_traffic(dp.name)
    if dp.bound == "hbm":
        achieved = dp.bytes / (dom_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "kernel": f"gemm_kernel ({dp.name})",
                    "peak_source": f"{peak_src} hbm_gbs (copy)", "algorithmic_bytes": dp.bytes}
    else:
        achieved = dp.flops / (dom_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic, "kernel": ("row_rms_kernel + " if dp.rmsnorm else "") + f"gemm_kernel ({dp.name})",
                    "peak_source": f"{peak_src} {peak_kind}", "algorithmic_bytes": dp.bytes}

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        for p in parts:
            p.prepare_oracle()
        r = oracle_sample(parts, args.cpu_seconds)
        cpu = {"value": r["flops"] / r["seconds"] / 1e12, "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
               "sample": f"oracle (fp64 CPU) on random output rows {r['rows']} x 256-column blocks of the step's parts, "
                         f"{r['seconds']:.1f} s"}

    # The bf16 peak three ways: nominal dense, clock-derived (SMs x 8192 FLOP/clk x the median
    # SM clock sampled under load in the timed region; sparse in short runs, where the samples
    # fall between launches), and the measured cuBLAS figures the roofline uses.
    clk = clocks.summary()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    clock_peak = sms * 8192 * clk["sm_mhz"] * 1e6 / 1e12 if clk.get("sm_mhz") else None
    parts_out = []
    for j, p in enumerate(parts):
        st = part_stats[j]
        ms = st["median"]
        tf = p.flops / (ms * 1e-3) / 1e12
        parts_out.append({**p.describe(), "ms": ms, "ms_stats": st, "tflops": tf,
                          "gbs": p.bytes / (ms * 1e-3) / 1e9, "algorithmic_bytes": p.bytes,
                          "frac_of_peak": tf / peak, "frac_of_burst_peak": tf / peaks["bf16_tflops"],
                          "frac_of_nominal": tf / NOMINAL_BF16_TFLOPS,
                          "frac_of_clock_peak": tf / clock_peak if clock_peak else None,
                          "roofline_ms": 1e3 * max(p.flops / (peak * 1e12), p.bytes / (peaks["hbm_gbs"] * 1e9))})
    line = {
        "metric": METRIC, "value": agg["value_tflops"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": agg["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "parts": parts_out, "l2": "warm (not flushed between steps)" if args.warm else
                   "flushed between steps (256 MiB write, then a 256 MiB read that evicts its dirty lines), "
                   "outside the timed events",
                   "parallelism": f"independent replicas x{world}" if world > 1 else "single GPU",
                   "frac_of_peak": agg["value_tflops"] / (world * peak),
                   "bf16_peaks_tflops": {"nominal_dense": NOMINAL_BF16_TFLOPS, "clock_derived": clock_peak,
                                         "sms": sms, "measured_burst": peaks["bf16_tflops"],
                                         "measured_sustained": peaks.get("bf16_tflops_sustained")}},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                   "samples": clk["samples"], "samples_under_load": clk.get("samples_under_load"),
                   "source": clk.get("source")},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--e2e-steps", type=int, default=50, help="steps of the end-to-end loop (at most --steps)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--warm", action="store_true",
                    help="do not flush L2 between timed steps (reported as warm; the default is cold)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        log("[bench] warm-up below 3 steps is not a valid measurement; using 3")
        args.warmup = 3
    names = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, names)
    return run_ours(args, names)


if __name__ == "__main__":
    sys.exit(main())
