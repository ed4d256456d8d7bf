"""Seeded synthetic inputs for the dense and grouped GEMM workloads.

This module only draws numbers: it holds none of the GEMM's arithmetic, so
both the CUDA path and the CPU oracle can be fed the very same bytes from it.
Everything is drawn on the CPU with torch's CPU generator (and numpy's PCG64
for the MoE routing split), then rounded to bf16 with round-to-nearest-even.

Workloads (the pages' own workloads run on Meta-internal models and data; these
synthetic inputs of the stated shapes and distributions stand in for them):

* ``dense_256``: M=N=K=256, A and B row-major, N(0,1)/sqrt(K), seed 0, bf16
  out, no epilogue.
* ``dense_4096_bias_gelu``: M=N=K=4096, A row-major, B column-major, U(-1,1),
  seed 1, bias bf16[N] ~ N(0, 0.1), bias + GELU(tanh), bf16 out.
* ``dense_8192_f32``: M=N=K=8192, A and B row-major, N(0,1)/sqrt(K), seed 2,
  fp32 out, no epilogue.
* ``grouped_moe``: G=64 experts, K=4096, N=1536; per-expert token counts are
  a multinomial split of 65536 tokens under Dirichlet(0.5) expert
  probabilities (numpy default_rng(3)); A_g [M_g, K] row-major, stored back to
  back in expert order; B_g [K, N] row-major, stacked [G, K, N]; N(0,1)/sqrt(K)
  from torch seed 3; bf16 out, no epilogue.
* ``skinny_bcast``: M=131072, K=1024, N=128; A is 1024 distinct user rows
  ~ N(0,1), row i = user[i // 128] (each user's 128 candidates contiguous),
  materialised; B row-major N(0,1)/sqrt(K); bias ~ N(0, 0.1); seed 4; bias
  epilogue, bf16 out.

Draw order within a seed: A (or the user rows), then B, then bias.  A
column-major operand is drawn directly in its storage shape (i.i.d. draws, so
the distribution is the same).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = ["DenseCase", "GroupedCase", "dense_case", "grouped_case", "dense_random",
           "grouped_random", "bf16_bits", "DENSE_WORKLOADS", "GROUPED_WORKLOADS"]


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The uint16 bit patterns of a CPU bf16 tensor (a view, no copy)."""
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return t.view(torch.int16).numpy().view(np.uint16)


@dataclass
class DenseCase:
    name: str
    M: int
    N: int
    K: int
    a: torch.Tensor            # storage: [M, K] row-major, or [K, M] if a_col_major
    b: torch.Tensor            # storage: [K, N] row-major, or [N, K] if b_col_major
    bias: torch.Tensor | None  # bf16 [N]
    a_col_major: bool
    b_col_major: bool
    c_dtype: str               # "bf16" or "f32"
    epi: str                   # "none", "bias", "bias_gelu"
    seed: int
    recipe: str = ""
    users: torch.Tensor | None = None   # broadcast form: the distinct A rows (A[i] = users[i // repeat])
    repeat: int = 1

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def bcast_bytes(self) -> int:
        """Algorithmic bytes of the broadcast form: user rows, B, bias read once, C written once."""
        cb = 2 if self.c_dtype == "bf16" else 4
        nb = 2 * self.N if self.bias is not None else 0
        return 2 * self.users.shape[0] * self.K + 2 * self.K * self.N + cb * self.M * self.N + nb

    @property
    def algorithmic_bytes(self) -> int:
        """Each input read once, the output written once."""
        cb = 2 if self.c_dtype == "bf16" else 4
        nb = 2 * self.N if self.bias is not None else 0
        return 2 * self.M * self.K + 2 * self.K * self.N + cb * self.M * self.N + nb


@dataclass
class GroupedCase:
    name: str
    G: int
    N: int
    K: int
    counts: np.ndarray          # int64 [G], tokens per group (M_g)
    a: torch.Tensor             # bf16 [sum M_g, K], groups back to back
    b: torch.Tensor             # bf16 [G, K, N] (row-major B_g)
    bias: torch.Tensor | None   # bf16 [G, N] or None
    c_dtype: str
    epi: str
    seed: int
    recipe: str = ""
    offsets: np.ndarray = field(init=False)

    def __post_init__(self):
        self.offsets = np.concatenate([[0], np.cumsum(self.counts)]).astype(np.int64)

    @property
    def flops(self) -> int:
        return int(2 * self.counts.sum() * self.N * self.K)

    @property
    def algorithmic_bytes(self) -> int:
        """A once, each non-empty group's B once, C once (+ bias of non-empty groups)."""
        cb = 2 if self.c_dtype == "bf16" else 4
        live = int((self.counts > 0).sum())
        m = int(self.counts.sum())
        nb = 2 * self.N * live if self.bias is not None else 0
        return 2 * m * self.K + 2 * live * self.K * self.N + cb * m * self.N + nb


def _draw(gen: torch.Generator, shape, dist: str, scale: float = 1.0) -> torch.Tensor:
    if dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
    elif dist == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "int4":   # integers in [-4, 4]: exact in bf16
        x = torch.randint(-4, 5, shape, generator=gen).to(torch.float32)
    else:
        raise ValueError(dist)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def dense_random(M: int, N: int, K: int, seed: int, *, dist: str = "normal", scale_by_k: bool = True,
                 a_col_major: bool = False, b_col_major: bool = False, c_dtype: str = "bf16",
                 epi: str = "none", bias_std: float = 0.1, lda: int | None = None,
                 ldb: int | None = None, name: str = "") -> DenseCase:
    """A seeded dense problem.  ``lda``/``ldb`` pad the storage rows (padding is random too)."""
    gen = torch.Generator().manual_seed(seed)
    scale = 1.0 / math.sqrt(K) if (dist == "normal" and scale_by_k and K > 0) else 1.0
    a_shape = (K, M) if a_col_major else (M, K)
    b_shape = (N, K) if b_col_major else (K, N)
    a_full = (a_shape[0], lda if lda is not None else a_shape[1])
    b_full = (b_shape[0], ldb if ldb is not None else b_shape[1])
    a = _draw(gen, a_full, dist, scale)[:, : a_shape[1]]
    b = _draw(gen, b_full, dist, scale)[:, : b_shape[1]]
    bias = None
    if epi != "none":
        bias = (torch.randn((N,), generator=gen, dtype=torch.float32) * bias_std).to(torch.bfloat16)
    return DenseCase(name or f"dense_{M}x{N}x{K}_s{seed}", M, N, K, a, b, bias, a_col_major,
                     b_col_major, c_dtype, epi, seed,
                     recipe=f"{dist}{'/sqrt(K)' if scale != 1.0 else ''}, seed {seed}")


def dense_case(name: str) -> DenseCase:
    if name == "dense_256":
        return dense_random(256, 256, 256, 0, dist="normal", name=name)
    if name == "dense_4096_bias_gelu":
        return dense_random(4096, 4096, 4096, 1, dist="uniform", b_col_major=True,
                            epi="bias_gelu", name=name)
    if name == "dense_8192_f32":
        return dense_random(8192, 8192, 8192, 2, dist="normal", c_dtype="f32", name=name)
    if name == "skinny_bcast":
        return skinny_bcast()
    raise KeyError(name)


def skinny_bcast(M: int = 131072, K: int = 1024, N: int = 128, repeat: int = 128,
                 seed: int = 4) -> DenseCase:
    gen = torch.Generator().manual_seed(seed)
    users = torch.randn((M // repeat, K), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    a = users.repeat_interleave(repeat, dim=0)
    b = _draw(gen, (K, N), "normal", 1.0 / math.sqrt(K))
    bias = (torch.randn((N,), generator=gen, dtype=torch.float32) * 0.1).to(torch.bfloat16)
    return DenseCase("skinny_bcast", M, N, K, a, b, bias, False, False, "bf16", "bias", seed,
                     recipe=f"{M // repeat} user rows N(0,1) x{repeat}, B N(0,1)/sqrt(K), seed {seed}",
                     users=users, repeat=repeat)


def moe_counts(G: int, tokens: int, alpha: float, seed: int) -> np.ndarray:
    """Tokens per expert: multinomial(tokens, Dirichlet(alpha * 1_G)), numpy PCG64."""
    rng = np.random.default_rng(seed)
    p = rng.dirichlet([alpha] * G)
    return rng.multinomial(tokens, p).astype(np.int64)


def grouped_random(counts, N: int, K: int, seed: int, *, dist: str = "normal", c_dtype: str = "bf16",
                   epi: str = "none", name: str = "") -> GroupedCase:
    counts = np.asarray(counts, dtype=np.int64)
    G = counts.shape[0]
    gen = torch.Generator().manual_seed(seed)
    scale = 1.0 / math.sqrt(K) if (dist == "normal" and K > 0) else 1.0
    m = int(counts.sum())
    rows = 4096
    a = torch.empty((m, K), dtype=torch.bfloat16)
    for r0 in range(0, m, rows):
        r1 = min(m, r0 + rows)
        a[r0:r1] = _draw(gen, (r1 - r0, K), dist, scale)
    b = torch.empty((G, K, N), dtype=torch.bfloat16)
    for g in range(G):
        b[g] = _draw(gen, (K, N), dist, scale)
    bias = None
    if epi != "none":
        bias = (torch.randn((G, N), generator=gen, dtype=torch.float32) * 0.1).to(torch.bfloat16)
    return GroupedCase(name or f"grouped_G{G}_N{N}_K{K}_s{seed}", G, N, K, counts, a, b, bias,
                       c_dtype, epi, seed, recipe=f"{dist}{'/sqrt(K)' if scale != 1.0 else ''}, seed {seed}")


def grouped_case(name: str) -> GroupedCase:
    if name == "grouped_moe":
        counts = moe_counts(64, 65536, 0.5, 3)
        return grouped_random(counts, 1536, 4096, 3, name=name)
    raise KeyError(name)


DENSE_WORKLOADS = ("dense_256", "dense_4096_bias_gelu", "dense_8192_f32", "skinny_bcast")
GROUPED_WORKLOADS = ("grouped_moe",)
