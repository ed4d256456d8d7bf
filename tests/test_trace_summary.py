"""The timeline summary of grouped_gemm_persistent_gb300.trace on a hand-made trace (no GPU)."""
import numpy as np

from grouped_gemm_persistent_gb300.trace import summarize


def test_summary_of_a_two_pair_trace():
    # CTA records: entry, set-up done, teardown start, exit (ns); blocks 0 and 2 lead pairs
    ctas = np.zeros((4, 4), dtype=np.int64)
    ctas[:, 0] = [1000, 1000, 1100, 1100]
    # units: block, first k-block, last MMA, epilogue end
    tiles = np.array([[0, 3000, 13000, 14000],
                      [0, 13100, 23000, 24000],
                      [2, 3100, 13100, 14100],
                      [0, 0, 0, 0]], dtype=np.int64)
    d = summarize(tiles, ctas)
    assert d["units"] == 3 and d["pairs"] == 2
    assert d["span_us"] == 23.0                       # 1000 -> 24000
    assert d["ramp_us"] == [2.0, 2.0, 2.0]
    assert d["final_epi_us"] == [1.0, 1.0, 1.0]
    assert d["idle_tail_us"] == [0.0, 4.95, 9.9]       # pair 2 ends at 14100
    assert abs(d["idle_tail_share"] - 9.9 / 46.0) < 1e-4
    assert abs(d["busy_share"] - (10.0 + 9.9 + 10.0) / 46.0) < 1e-4
    assert d["units_per_pair"] == [1, 2]
    assert d["gap_between_units_us"] == [0.1, 0.1, 0.1]
    assert d["by_round"]["0"]["n"] == 2 and d["by_round"]["1"]["mma_us"] == [9.9, 9.9, 9.9]
