"""The seeded input generators match the recipe the benchmark and the tests state.

CPU only.  The full-size workloads are large, so these checks use the cheap
parts of each recipe (counts, shapes, seeds, the repeat structure) and small
cases of the same generators.
"""
import hashlib

import numpy as np
import pytest
import torch

from grouped_gemm_persistent_gb300 import workloads as wl


def _digest(t: torch.Tensor) -> str:
    return hashlib.sha256(wl.bf16_bits(t).tobytes()).hexdigest()


def test_moe_counts_recipe():
    c = wl.moe_counts(64, 65536, 0.5, 3)
    assert c.shape == (64,) and c.dtype == np.int64
    assert int(c.sum()) == 65536 and (c >= 0).all()
    assert int((c == 0).sum()) == 1                      # seed 3 draws one empty expert
    assert np.array_equal(c, wl.moe_counts(64, 65536, 0.5, 3))
    assert not np.array_equal(c, wl.moe_counts(64, 65536, 0.5, 4))


def test_dense_generator_is_seeded_and_shaped():
    a = wl.dense_random(64, 40, 72, 1, dist="uniform", b_col_major=True, epi="bias_gelu")
    b = wl.dense_random(64, 40, 72, 1, dist="uniform", b_col_major=True, epi="bias_gelu")
    c = wl.dense_random(64, 40, 72, 2, dist="uniform", b_col_major=True, epi="bias_gelu")
    assert a.a.shape == (64, 72) and a.b.shape == (40, 72) and a.bias.shape == (40,)
    assert a.a.dtype == torch.bfloat16 and a.b.dtype == torch.bfloat16
    assert _digest(a.a) == _digest(b.a) and _digest(a.b) == _digest(b.b)
    assert _digest(a.a) != _digest(c.a)
    assert float(a.a.float().abs().max()) <= 1.0              # U(-1, 1)
    n = wl.dense_random(256, 256, 256, 0, dist="normal")
    # N(0,1)/sqrt(K): the sample standard deviation is close to 1/16
    assert abs(float(n.a.float().std()) - 1 / 16) < 0.005


def test_padded_leading_dimension_keeps_the_logical_matrix():
    p = wl.dense_random(10, 24, 20, 5, lda=24, ldb=32)
    assert p.a.shape == (10, 20) and p.a.stride() == (24, 1)
    assert p.b.shape == (20, 24) and p.b.stride() == (32, 1)


def test_grouped_generator_layout():
    g = wl.grouped_random([3, 0, 5], 16, 24, 7, epi="bias")
    assert g.a.shape == (8, 24) and g.b.shape == (3, 24, 16) and g.bias.shape == (3, 16)
    assert list(g.offsets) == [0, 3, 3, 8]
    h = wl.grouped_random([3, 0, 5], 16, 24, 7, epi="bias")
    assert _digest(g.a) == _digest(h.a) and _digest(g.b) == _digest(h.b)


def test_skinny_rows_repeat_their_user_row():
    s = wl.skinny_bcast(M=64 * 8, K=32, N=16, repeat=8)
    assert s.a.shape == (512, 32) and s.users.shape == (64, 32)
    for i in (0, 7, 8, 100, 511):
        assert torch.equal(s.a[i], s.users[i // 8])


@pytest.mark.parametrize("name", wl.DENSE_WORKLOADS)
def test_dense_workload_shapes(name):
    if name in ("dense_8192_f32", "skinny_bcast"):
        pytest.skip("large; its generator is covered above")
    c = wl.dense_case(name)
    assert c.a.shape == (c.M, c.K)
    assert (c.b.shape == (c.N, c.K)) if c.b_col_major else (c.b.shape == (c.K, c.N))


def test_bf16_bits_round_trip():
    x = torch.tensor([0.0, -0.0, 1.0, -2.5, 3.0e38, 1.0e-40], dtype=torch.float32).to(torch.bfloat16)
    bits = wl.bf16_bits(x)
    assert bits.dtype == np.uint16
    assert bits.tolist()[:4] == [0x0000, 0x8000, 0x3F80, 0xC020]     # 0, -0, 1, -2.5
    back = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    assert np.array_equal(wl.bf16_bits(back), bits)
