"""The allocation-free grouped GEMM entry point, tg_grouped_gemm_noalloc.

Some callers cannot allocate device memory while they run: a serving loop that
reserved all of its memory at start-up so no request can stall or fail on an
allocation, or a program whose device memory is handed out by its own
allocator under a fixed budget.  For them the library offers a grouped GEMM
whose per-problem descriptors live in a fixed table inside the library instead
of a per-call workspace.  These tests call it through the C ABI and compare it
with tg_grouped_gemm, on two calls in a row with different problem sets (the
table keeps the previous call's contents, which must not matter).

The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import grouped_gemm_persistent_gb300 as tg
import oracle
from grouped_gemm_persistent_gb300 import _binding
from grouped_gemm_persistent_gb300 import workloads as wl
from grouped_gemm_persistent_gb300.build import build


def _problem_set(counts, N, K, seed, epi):
    case = wl.grouped_random(counts, N, K, seed, epi=epi)
    a, b = case.a.cuda(), case.b.cuda()
    bias = case.bias.cuda() if case.bias is not None else None
    rows = int(np.sum(counts))
    out_ref = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    out_na = torch.full((rows, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    t_ref = tg.build_moe_table(a, b, counts, out_ref, bias=bias, epilogue=epi)
    t_na = tg.build_moe_table(a, b, counts, out_na, bias=bias, epilogue=epi)
    return case, (a, b, bias), out_ref, out_na, t_ref, t_na


@pytest.mark.gpu
def test_noalloc_matches_grouped_gemm_on_two_calls():
    build()
    lib = tg.load()
    stream = torch.cuda.current_stream().cuda_stream
    sets = [([0, 300, 5, 0, 130, 257, 1, 0], 136, 200, 41, "bias_gelu"),   # empty first/middle/last groups
            ([64, 0, 513], 264, 128, 42, "none")]                        # fewer problems than the first call
    for counts, N, K, seed, epi in sets:
        case, keep, out_ref, out_na, t_ref, t_na = _problem_set(counts, N, K, seed, epi)
        assert lib.tg_grouped_gemm(t_ref, len(counts), stream) == tg.TG_OK, lib.tg_last_error_message()
        rc = lib.tg_grouped_gemm_noalloc(t_na, len(counts), stream)
        assert rc == tg.TG_OK, lib.tg_last_error_message()
        tg.device_status()
        ref = out_ref.float().cpu().double().numpy()
        got = out_na.float().cpu().double().numpy()
        assert not np.isnan(got).any(), "a row of a non-empty problem was not written"
        # the tolerance of the parity tests: |err| <= 1e-2 * (S + |bias|) + 1e-5, S from the oracle
        for g in range(case.G):
            r0, r1 = case.offsets[g], case.offsets[g + 1]
            if r1 == r0:
                continue
            bias = wl.bf16_bits(case.bias[g]) if case.bias is not None else None
            _, s = oracle.gemm(wl.bf16_bits(case.a[r0:r1]), wl.bf16_bits(case.b[g]), bias=bias, epi=epi)
            bias_abs = np.abs(case.bias[g].double().numpy()) if case.bias is not None else None
            r = oracle.compare(got[r0:r1], ref[r0:r1], s, bias_abs)
            assert r["ok"], f"problem {g}: {r}"


def test_noalloc_rejects_more_problems_than_its_table():
    # Host-side check, made before any device work (no GPU needed).
    build()
    lib = tg.load()
    P = _binding.GroupProblem
    n = 257
    arr = (P * n)(*[P(64, 64, 64, 0x10000, 64, 0, 0x20000, 64, 0, 0x30000, 64, 0, 0, None) for _ in range(n)])
    assert lib.tg_grouped_gemm_noalloc(arr, n, None) == tg.TG_ERR_UNSUPPORTED
    msg = lib.tg_last_error_message()
    assert b"256" in msg and b"tg_grouped_gemm" in msg
