"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the binding, run the oracle on the same bytes, and
compare element by element within the stated bound."""
from __future__ import annotations

import numpy as np
import torch

import grouped_gemm_persistent_gb300 as tg
import oracle
from grouped_gemm_persistent_gb300 import workloads as wl


def to_device(t: torch.Tensor) -> torch.Tensor:
    """Copy a (possibly row-padded) CPU view to the GPU keeping its strides."""
    if t.is_contiguous():
        return t.cuda()
    r, c = t.shape
    ld = t.stride(0)
    assert t.stride(1) == 1
    full = torch.empty((r, ld), dtype=t.dtype, device="cuda")
    full[:, :c].copy_(t)
    return full[:, :c]


def device_operands(case: wl.DenseCase):
    a = to_device(case.a)
    b = to_device(case.b)
    a_view = a.t() if case.a_col_major else a      # logical [M, K]
    b_view = b.t() if case.b_col_major else b      # logical [K, N]
    bias = case.bias.cuda() if case.bias is not None else None
    return a_view, b_view, bias


def run_dense(case: wl.DenseCase, out: torch.Tensor | None = None) -> torch.Tensor:
    a, b, bias = device_operands(case)
    dt = torch.float32 if case.c_dtype == "f32" else torch.bfloat16
    return tg.gemm(a, b, out, bias=bias, epilogue=case.epi, out_dtype=dt)


def oracle_dense(case: wl.DenseCase, rows=None):
    bias = wl.bf16_bits(case.bias) if case.bias is not None else None
    return oracle.gemm(wl.bf16_bits(case.a), wl.bf16_bits(case.b), a_col_major=case.a_col_major,
                       b_col_major=case.b_col_major, bias=bias, epi=case.epi, rows=rows)


def to_f64(c: torch.Tensor) -> np.ndarray:
    return c.float().cpu().double().numpy()


def check_dense(case: wl.DenseCase, c_gpu: torch.Tensor, rows=None) -> dict:
    y, s = oracle_dense(case, rows)
    c = to_f64(c_gpu if rows is None else c_gpu[torch.as_tensor(rows, device=c_gpu.device)])
    bias_abs = np.abs(case.bias.double().numpy()) if case.bias is not None else None
    r = oracle.compare(c, y, s, bias_abs)
    assert r["ok"], f"{case.name}: {r}"
    # tight diagnostic: fp32 accumulation plus one output rounding stays far below this
    assert r["max_tight"] < 4.0, f"{case.name}: suspicious error pattern {r}"
    return r


def sample_rows(M: int, tile: int, n_random: int, seed: int) -> np.ndarray:
    """Random rows plus the first row, the last row, and every row of the ragged tail tile."""
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(M, size=min(n_random, M), replace=False).tolist()) if M else set()
    rows |= {0, M - 1} if M else set()
    tail0 = (M // tile) * tile
    rows |= set(range(tail0, M))
    rows |= set(range(max(0, M - tile), min(M, max(0, M - tile) + 8)))
    return np.array(sorted(rows), dtype=np.int64)
