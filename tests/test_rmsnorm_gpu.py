"""GPU parity of the RMS normalisation fused into the GEMM (tg_row_rms, tg_gemm_rmsnorm).

C = epilogue(rmsnorm(A) . B) from the CUDA path against the oracle's
row-normalised product, element by element, within
|err| <= 1e-2 * sum_k |a'_ik b_kj| (+ 1e-2 |bias_j|) + 1e-5 where a' is the
normalised A (the row factor is exact to fp32, far inside that bound).
"""
import numpy as np
import pytest
import torch

import grouped_gemm_persistent_gb300 as tg
import oracle
from grouped_gemm_persistent_gb300 import workloads as wl

from parity import sample_rows, to_device, to_f64

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(autouse=True, scope="module")
def _built():
    from grouped_gemm_persistent_gb300.build import build
    build()
    tg.load()


def pad8(x: int) -> int:
    return -(-x // 8) * 8


def run_fused(case, eps, out=None, row_scale=None):
    a = to_device(case.a)
    b = to_device(case.b)
    b_view = b.t() if case.b_col_major else b
    bias = case.bias.cuda() if case.bias is not None else None
    dt = torch.float32 if case.c_dtype == "f32" else torch.bfloat16
    if row_scale is None:
        row_scale = torch.empty(case.M, dtype=torch.float32, device="cuda")
    c = tg.gemm_rmsnorm(a, b_view, eps, out, row_scale=row_scale, bias=bias, epilogue=case.epi, out_dtype=dt)
    return c, row_scale


def check_fused(case, c_gpu, eps, rows=None):
    bias = wl.bf16_bits(case.bias) if case.bias is not None else None
    y, s = oracle.gemm(wl.bf16_bits(case.a), wl.bf16_bits(case.b), b_col_major=case.b_col_major, bias=bias,
                       epi=case.epi, rows=rows, row_norm_eps=eps)
    c = to_f64(c_gpu if rows is None else c_gpu[torch.as_tensor(rows, device=c_gpu.device)])
    bias_abs = np.abs(case.bias.double().numpy()) if case.bias is not None else None
    r = oracle.compare(c, y, s, bias_abs)
    assert r["ok"], f"{case.name}: {r}"
    assert r["max_tight"] < 4.0, f"{case.name}: suspicious error pattern {r}"
    return r


def mean_square_factor(a_bits: np.ndarray, eps: float) -> np.ndarray:
    """1 / sqrt(mean_k a_ik^2 + eps) in float64 from the bf16 bit patterns (the definition)."""
    x = (a_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    K = x.shape[1]
    ms = (x * x).sum(axis=1) / K if K else np.zeros(x.shape[0])
    return 1.0 / np.sqrt(ms + eps)


@pytest.mark.parametrize("M,N,K", [(300, 264, 200), (129, 136, 64), (1, 8, 8), (700, 512, 1024), (64, 128, 72)])
@pytest.mark.parametrize("epi", ["none", "bias", "bias_gelu"])
@pytest.mark.parametrize("b_col", [False, True])
def test_fused_matches_oracle(M, N, K, epi, b_col):
    # uniform A with a per-row spread of magnitudes, so the factors differ from row to row
    case = wl.dense_random(M, N, K, 11, dist="uniform", b_col_major=b_col, epi=epi,
                           ldb=pad8(K if b_col else N))
    spread = torch.exp2(torch.arange(M, dtype=torch.float32) % 7 - 3).to(torch.bfloat16)[:, None]
    case.a = (case.a.float() * spread.float()).to(torch.bfloat16)     # powers of two: exact in bf16
    c, _ = run_fused(case, EPS)
    check_fused(case, c, EPS)


@pytest.mark.parametrize("c_dtype", ["bf16", "f32"])
def test_fused_output_dtypes_and_tiles(c_dtype, monkeypatch):
    case = wl.dense_random(520, 392, 320, 12, dist="normal", c_dtype=c_dtype, epi="bias_gelu")
    for tile in ("1x128", "1x256", "2x128", "2x256"):
        monkeypatch.setenv("TG_TILE", tile)
        c, _ = run_fused(case, EPS)
        check_fused(case, c, EPS)


@pytest.mark.parametrize("M,K,lda", [(1000, 1024, 1024), (37, 65, 72), (5, 7, 8), (3, 1, 8), (4099, 4096, 4104)])
def test_row_factor_matches_definition(M, K, lda):
    gen = torch.Generator().manual_seed(M + K)
    full = (torch.randn((M, lda), generator=gen) * 3.0).to(torch.bfloat16)
    a = full[:, :K]
    r = tg.row_rms(to_device(a), EPS)
    want = mean_square_factor(wl.bf16_bits(a), EPS)
    got = r.cpu().double().numpy()
    # fp32 sum of K squares, one division and one reciprocal square root
    np.testing.assert_allclose(got, want, rtol=4e-6 + 2 ** -24 * K, atol=0)


def test_row_factor_left_for_reuse_is_the_standalone_one():
    case = wl.dense_random(384, 256, 512, 13, dist="normal")
    _, rs = run_fused(case, 1e-5)
    r = tg.row_rms(to_device(case.a), 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(rs, r)


def test_zero_row_and_k_zero_give_the_epilogue_of_zero():
    case = wl.dense_random(200, 136, 128, 14, dist="normal", epi="bias_gelu")
    case.a[7].zero_()                                   # zero row, eps > 0: rmsnorm gives zeros
    c, rs = run_fused(case, EPS)
    check_fused(case, c, EPS)
    assert rs[7].item() == pytest.approx(1.0 / np.sqrt(EPS), rel=1e-6)
    k0 = wl.dense_random(130, 136, 0, 15, epi="bias_gelu")
    c0, rs0 = run_fused(k0, 0.0)                        # empty rows: product 0 even with eps = 0
    check_fused(k0, c0, 0.0)
    assert torch.isinf(rs0).all()


def test_deterministic_and_scale_invariant():
    case = wl.dense_random(256, 256, 384, 16, dist="normal", epi="bias")
    c1, _ = run_fused(case, 0.0)
    c2, _ = run_fused(case, 0.0)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)
    # rmsnorm(4 A) = rmsnorm(A) with eps = 0; scaling by a power of two is exact in bf16
    scaled = wl.dense_random(256, 256, 384, 16, dist="normal", epi="bias")
    scaled.a = (scaled.a.float() * 4.0).to(torch.bfloat16)
    c3, _ = run_fused(scaled, 0.0)
    check_fused(scaled, c3, 0.0)
    assert (c3.float() - c1.float()).abs().max().item() <= 2 ** -7 * c1.float().abs().max().item()


def test_workload_4096_bias_gelu_sampled():
    case = wl.dense_case("dense_4096_bias_gelu")
    c, _ = run_fused(case, EPS)
    rows = sample_rows(case.M, 128, 48, seed=17)
    check_fused(case, c, EPS, rows=rows)
