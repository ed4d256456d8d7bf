"""Per-pair timeline of one GEMM launch, from the library's trace hook (tg_debug_trace).

    python -m grouped_gemm_persistent_gb300.trace dense_4096_bias_gelu [dense_8192_f32 grouped_moe ...]

For each named workload (the seeded inputs of ``workloads``): five untraced
launches, then three traced ones, each after an L2 flush (256 MiB written, then
256 MiB read).  The trace records, per work unit (a whole tile, a column half
or a stream-K piece), the CTA that ran it, the time of its first k-block, of
its last MMA and of the end of its epilogue; per CTA, its entry, end of set-up,
start of teardown and exit (``%globaltimer``, ns).  One JSON line per traced
launch:

* ``span_us``: first CTA entry to the last epilogue end.
* ``ramp_us``: per pair, entry to its first k-block (min / median / max).
* ``final_epi_us``: per pair, the epilogue of its last unit, which no later
  main loop hides.
* ``idle_tail_us`` / ``idle_tail_share``: per pair, the time from its last
  epilogue end to the end of the launch, and its share of pairs x span: the
  load imbalance at the end that a dynamic tile scheduler could at best recover.
* ``busy_share``: the units' main-loop time (first k-block to last MMA) over
  pairs x span.
* ``unit_mma_us``, ``units_per_pair``, ``gap_between_units_us`` (one pair's next
  first k-block after its previous last MMA; negative when the next unit's
  loads were already in the ring).
* ``by_round``: per round r (each pair's r-th unit in time order), main-loop and
  epilogue times (min / median / max).
"""
from __future__ import annotations

import argparse
import json
import sys

import numpy as np
import torch

from . import _binding as tg
from . import workloads as wl

L2_FLUSH_BYTES = 256 << 20


def _q(x) -> list[float] | None:
    x = np.asarray(x, dtype=np.float64)
    if x.size == 0:
        return None
    return [round(float(np.min(x)), 2), round(float(np.median(x)), 2), round(float(np.max(x)), 2)]


def launcher(name: str):
    """A zero-argument function that launches the named workload on the current stream."""
    if name in wl.GROUPED_WORKLOADS:
        case = wl.grouped_case(name)
        a, b = case.a.cuda(), case.b.cuda()
        out = torch.empty((int(case.counts.sum()), case.N), dtype=torch.bfloat16, device="cuda")
        table = tg.build_moe_table(a, b, case.counts, out)
        return lambda: tg.grouped_gemm_table(table)
    case = wl.dense_case(name)
    a, b = case.a.cuda(), case.b.cuda()
    av = a.t() if case.a_col_major else a
    bv = b.t() if case.b_col_major else b
    bias = case.bias.cuda() if case.bias is not None else None
    out = torch.empty((case.M, case.N), dtype=torch.float32 if case.c_dtype == "f32" else torch.bfloat16,
                      device="cuda")
    return lambda: tg.gemm(av, bv, out, bias=bias, epilogue=case.epi)


def summarize(tiles: np.ndarray, ctas: np.ndarray) -> dict:
    """Statistics of one traced launch (arrays as read back from the trace buffers)."""
    T = tiles[tiles[:, 1] > 0]
    C = ctas[ctas[:, 0] > 0]
    t0 = int(C[:, 0].min())
    end = int(T[:, 3].max())
    span = end - t0
    pairs = sorted(set(int(x) for x in T[:, 0]))
    ramp, fin, tail, busy, gaps, nunits, rounds = [], [], [], [], [], [], {}
    for blk in pairs:
        R = T[T[:, 0] == blk]
        R = R[np.argsort(R[:, 1])]
        ramp.append(R[0, 1] - ctas[blk, 0])
        fin.append(R[-1, 3] - R[-1, 2])
        tail.append(end - R[-1, 3])
        busy.append(int(np.sum(R[:, 2] - R[:, 1])))
        gaps.extend((R[1:, 1] - R[:-1, 2]).tolist())
        nunits.append(len(R))
        for r, row in enumerate(R):
            rounds.setdefault(r, ([], []))
            rounds[r][0].append(row[2] - row[1])
            rounds[r][1].append(row[3] - row[2])
    P = len(pairs)
    us = lambda x: np.asarray(x, dtype=np.float64) / 1e3
    return {
        "span_us": round(span / 1e3, 2), "units": int(len(T)), "pairs": P,
        "ramp_us": _q(us(ramp)), "final_epi_us": _q(us(fin)),
        "idle_tail_us": _q(us(tail)), "idle_tail_share": round(float(np.sum(tail)) / (P * span), 4),
        "busy_share": round(float(np.sum(busy)) / (P * span), 4),
        "unit_mma_us": _q(us(T[:, 2] - T[:, 1])), "units_per_pair": [min(nunits), max(nunits)],
        "gap_between_units_us": _q(us(gaps)),
        "by_round": {str(r): {"n": len(v[0]), "mma_us": _q(us(v[0])), "epi_us": _q(us(v[1]))}
                     for r, v in sorted(rounds.items())},
    }


def trace(name: str, reps: int = 3, max_units: int = 8192, max_ctas: int = 512) -> list[dict]:
    run = launcher(name)
    s = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    flush_read = torch.zeros_like(flush)
    for _ in range(5):
        run()
    torch.cuda.synchronize()
    out = []
    for rep in range(reps):
        tiles = torch.zeros((max_units, 4), dtype=torch.int64, device="cuda")
        ctas = torch.zeros((max_ctas, 4), dtype=torch.int64, device="cuda")
        flush.zero_()
        flush_read.sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tg.debug_trace(tiles, ctas)
        e0.record(s)
        run()
        e1.record(s)
        tg.device_status()
        d = {"workload": name, "rep": rep, "event_ms": round(e0.elapsed_time(e1), 4)}
        d.update(summarize(tiles.cpu().numpy(), ctas.cpu().numpy()))
        out.append(d)
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("workloads", nargs="+", choices=sorted(wl.DENSE_WORKLOADS + wl.GROUPED_WORKLOADS))
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)
    for name in args.workloads:
        for d in trace(name, args.reps):
            print(json.dumps(d), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
