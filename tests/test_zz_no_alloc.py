"""The allocation-free grouped GEMM entry point, tg_grouped_gemm_noalloc.

Some callers cannot allocate device memory while they run: a serving loop that
reserved all of its memory at start-up so no request can stall or fail on an
allocation, or a program whose device memory is handed out by its own
allocator under a fixed budget.  For them the library offers a grouped GEMM
whose per-problem descriptors live in a fixed table inside the library instead
of a per-call workspace.  These tests call it through the C ABI, on three calls
in a row with different problem sets (the table keeps the previous call's
contents, which must not matter), and require its output to be bitwise equal
to tg_grouped_gemm's on the same problems and, element by element, within the
parity bound of the oracle's values.  The third call mixes layout and output
classes (each class takes its own slice of the table and its own launch) and
comes after a call with more problems, so an entry left over from the earlier
call at a shifted offset would show up as a wrong result; the fourth has N a
multiple of 64, so its row-major B problems take the 64-column-chunk view.

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


def _problems(counts, N, K, seed, epi, classes):
    """Problems with the given row counts; classes[g] = (B column-major, output dtype) of problem g."""
    case = wl.grouped_random(counts, N, K, seed, epi=epi)
    keep, ref_tab, na_tab, outs = [], [], [], []
    for g, m in enumerate(counts):
        b_col, c_dtype = classes[g % len(classes)]
        r0, r1 = case.offsets[g], case.offsets[g + 1]
        a = case.a[r0:r1].cuda()
        b = case.b[g].t().contiguous().cuda().t() if b_col else case.b[g].cuda()   # same values, other layout
        bias = case.bias[g].cuda() if case.bias is not None else None
        o_ref = torch.full((m, N), float("nan"), dtype=c_dtype, device="cuda")
        o_na = torch.full((m, N), float("nan"), dtype=c_dtype, device="cuda")
        keep += [a, b, bias]
        ref_tab.append(tg.make_problem(a, b, o_ref, bias=bias, epilogue=epi))
        na_tab.append(tg.make_problem(a, b, o_na, bias=bias, epilogue=epi))
        outs.append((o_ref, o_na))
    P = _binding.GroupProblem
    return case, keep, (P * len(counts))(*ref_tab), (P * len(counts))(*na_tab), outs


@pytest.mark.gpu
def test_noalloc_matches_grouped_gemm_and_oracle_on_three_calls():
    build()
    lib = tg.load()
    stream = torch.cuda.current_stream().cuda_stream
    row_bf16 = [(False, torch.bfloat16)]
    mixed = [(False, torch.bfloat16), (True, torch.float32), (False, torch.float32), (True, torch.bfloat16)]
    sets = [([0, 300, 5, 0, 130, 257, 1, 0, 64, 17, 200], 136, 200, 41, "bias_gelu", row_bf16),  # empty first/middle/last
            ([64, 0, 513], 264, 128, 42, "none", row_bf16),                                 # fewer problems
            ([33, 0, 129, 256, 7, 90], 200, 136, 43, "bias", mixed),                       # four classes
            ([300, 0, 64, 129], 256, 128, 44, "bias_gelu", mixed)]                         # N-major B as 64-column chunks
    for counts, N, K, seed, epi, classes in sets:
        case, keep, t_ref, t_na, outs = _problems(counts, N, K, seed, epi, classes)
        assert lib.tg_grouped_gemm(t_ref, len(counts), stream) == tg.TG_OK, lib.tg_last_error_message()
        rc = lib.tg_grouped_gemm_noalloc(t_na, len(counts), stream)
        assert rc == tg.TG_OK, lib.tg_last_error_message()
        tg.device_status()
        for g, (o_ref, o_na) in enumerate(outs):
            if counts[g] == 0:
                continue
            assert not torch.isnan(o_na.float()).any(), f"problem {g}: a row was not written"
            # same kernel, same problem: bitwise equal to tg_grouped_gemm
            iv = torch.int32 if o_na.dtype == torch.float32 else torch.int16
            assert torch.equal(o_na.view(iv), o_ref.view(iv)), f"problem {g} differs from tg_grouped_gemm"
            # and within the parity bound of the oracle, element by element
            r0, r1 = case.offsets[g], case.offsets[g + 1]
            bias = wl.bf16_bits(case.bias[g]) if case.bias is not None else None
            y, s = oracle.gemm(wl.bf16_bits(case.a[r0:r1]), wl.bf16_bits(case.b[g]), bias=bias, epi=epi)
            bias_abs = np.abs(case.bias[g].double().numpy()) if case.bias is not None else None
            r = oracle.compare(o_na.float().cpu().double().numpy(), y, s, bias_abs)
            assert r["ok"], f"problem {g}: {r}"
        del keep


@pytest.mark.gpu
def test_noalloc_refuses_a_capturing_stream_and_consumes_an_armed_trace():
    build()
    lib = tg.load()
    case, keep, _, t_na, outs = _problems([70, 200], 128, 64, 44, "none", [(False, torch.bfloat16)])
    # The descriptor copy reads a per-thread host buffer that the next call overwrites,
    # so a captured call would replay with someone else's descriptors: refused up front.
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rc = lib.tg_grouped_gemm_noalloc(t_na, 2, torch.cuda.current_stream().cuda_stream)
    assert rc == tg.TG_ERR_UNSUPPORTED
    assert b"captured" in lib.tg_last_error_message()
    # an armed trace is consumed by the no-alloc launch, not left for the next call
    tiles = torch.zeros((64, 4), dtype=torch.int64, device="cuda")
    tg.debug_trace(tiles, None)
    assert lib.tg_grouped_gemm_noalloc(t_na, 2, torch.cuda.current_stream().cuda_stream) == tg.TG_OK
    tg.device_status()
    assert (tiles[:, 1] > 0).any(), "the no-alloc launch did not write the armed trace"
    tiles.zero_()
    a = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    tg.gemm(a, a.t())
    tg.device_status()
    assert not tiles.any(), "the trace stayed armed after the no-alloc launch"
    del keep


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
