"""Pins for the CPU oracle: it is checked against things other than itself.

Each pin is chosen so that a plausible mistake in the oracle (a dropped K
term, a transposed operand, a wrong bias index or sign, a wrong GELU constant,
a broken magnitude sum S) fails at least one of them; ``test_mutants_are_caught``
plants such mistakes in copies of the oracle source and checks exactly that.

Pins used:
  * hand-worked products from tests/golden/hand_examples.txt;
  * identity and permutation matrices (C must equal B, or B's rows permuted,
    exactly);
  * a rank-1 outer product with a closed-form result;
  * integer-valued inputs against numpy's exact int64 matmul (values and S);
  * tiny random bf16 problems against exact rational arithmetic (fractions);
  * random problems against torch's float64 CPU matmul (a library routine);
  * GELU(tanh) against torch.nn.functional.gelu(approximate="tanh") in float64,
    and against the exact erf GELU within the known approximation gap.
"""
import math
import os
import subprocess
import sys
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from grouped_gemm_persistent_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.txt")


def bits(x) -> np.ndarray:
    """float array -> bf16 bit patterns (round to nearest even via torch)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def widen(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def load_golden():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0], "M": int(vals[1]), "N": int(vals[2]), "K": int(vals[3]), "epi": vals[4]}
            cases.append(cur)
        else:
            cur[key] = np.array([float(v) for v in vals])
    return cases


# ----------------------------------------------------------------------------------------
# Pin suite, parameterised by the oracle build so the mutant test can reuse it.

def pin_golden(orc):
    for c in load_golden():
        M, N, K = c["M"], c["N"], c["K"]
        a = bits(c["A"].reshape(M, K))
        b = bits(c["B"].reshape(K, N))
        bias = bits(c["bias"]) if "bias" in c else None
        y, s = orc.gemm(a, b, bias=bias, epi=c["epi"])
        assert np.array_equal(y, c["C"].reshape(M, N)), c["name"]


def pin_identity_permutation(orc):
    rng = np.random.default_rng(11)
    M, N = 40, 24
    b = bits(rng.standard_normal((M, N)))
    eye = bits(np.eye(M))
    y, _ = orc.gemm(eye, b)
    assert np.array_equal(y, widen(b)), "I . B != B"
    # B stored column-major: same logical matrix, transposed storage
    y, _ = orc.gemm(eye, np.ascontiguousarray(b.T), b_col_major=True)
    assert np.array_equal(y, widen(b)), "I . B (col-major B) != B"
    perm = rng.permutation(M)
    P = np.zeros((M, M))
    P[np.arange(M), perm] = 1.0
    y, _ = orc.gemm(bits(P), b)
    assert np.array_equal(y, widen(b)[perm]), "P . B != rows of B permuted"
    # A . I = A, A column-major
    a = bits(rng.standard_normal((M, N)))
    y, _ = orc.gemm(np.ascontiguousarray(a.T), bits(np.eye(N)), a_col_major=True)
    assert np.array_equal(y, widen(a)), "A . I (col-major A) != A"


def pin_rank1(orc):
    # a_ik = u_i s_k, b_kj = t_k v_j with s_k t_k = +-1: C_ij = u_i v_j sum_k s_k t_k
    rng = np.random.default_rng(5)
    M, N, K = 17, 13, 96
    u = rng.integers(-16, 17, M).astype(np.float64)
    v = rng.integers(-16, 17, N).astype(np.float64)
    s = rng.choice([0.5, 1.0, 2.0, 4.0], K) * rng.choice([-1.0, 1.0], K)
    sign = rng.choice([-1.0, 1.0], K)
    t = sign / s
    A = np.outer(u, s)
    B = np.outer(t, v)
    y, S = orc.gemm(bits(A), bits(B))
    assert np.array_equal(y, np.outer(u, v) * sign.sum())
    assert np.array_equal(S, np.abs(np.outer(u, v)) * K)


def pin_integer_exact(orc):
    rng = np.random.default_rng(7)
    M, N, K = 37, 29, 300
    A = rng.integers(-4, 5, (M, K))
    B = rng.integers(-4, 5, (K, N))
    bias = rng.integers(-8, 9, N)
    y, S = orc.gemm(bits(A), bits(B))
    assert np.array_equal(y, (A @ B).astype(np.float64))
    assert np.array_equal(S, (np.abs(A) @ np.abs(B)).astype(np.float64))
    y, S = orc.gemm(bits(A), bits(B), bias=bits(bias), epi="bias")
    assert np.array_equal(y, (A @ B + bias[None, :]).astype(np.float64))
    # column-major storage of both operands, and padded leading dimensions
    Ap = np.zeros((K, M + 5))
    Ap[:, :M] = A.T
    Bp = np.full((N, K + 3), 7.0)
    Bp[:, :K] = B.T
    y, _ = orc.gemm(bits(Ap)[:, :M], bits(Bp)[:, :K], a_col_major=True, b_col_major=True)
    assert np.array_equal(y, (A @ B).astype(np.float64))


def pin_fraction_bruteforce(orc):
    rng = np.random.default_rng(3)
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (8, 8, 8), (2, 7, 5)]:
        a = bits(rng.standard_normal((M, K)))
        b = bits(rng.standard_normal((K, N)))
        bias = bits(rng.standard_normal(N))
        fa, fb, fbias = widen(a), widen(b), widen(bias)
        for epi in ("none", "bias"):
            y, S = orc.gemm(a, b, bias=bias, epi=epi)
            for i in range(M):
                for j in range(N):
                    exact = sum(Fraction(fa[i, k]) * Fraction(fb[k, j]) for k in range(K))
                    sabs = sum(abs(Fraction(fa[i, k]) * Fraction(fb[k, j])) for k in range(K))
                    if epi == "bias":
                        exact += Fraction(fbias[j])
                    assert abs(Fraction(y[i, j]) - exact) <= Fraction(1, 10 ** 15) * (sabs + abs(Fraction(fbias[j])) + 1)
                    assert abs(Fraction(S[i, j]) - sabs) <= Fraction(1, 10 ** 15) * (sabs + 1)


def pin_torch_float64(orc):
    case = wl.dense_random(96, 80, 200, seed=21, dist="normal")
    a, b = wl.bf16_bits(case.a), wl.bf16_bits(case.b)
    y, S = orc.gemm(a, b)
    ref = case.a.double() @ case.b.double()
    assert np.all(np.abs(y - ref.numpy()) <= 1e-12 * S + 1e-300)
    Sref = case.a.double().abs() @ case.b.double().abs()
    assert np.allclose(S, Sref.numpy(), rtol=1e-12, atol=0)
    # column-major B, U(-1,1), bias + GELU against torch's tanh GELU in float64
    case = wl.dense_random(64, 48, 130, seed=22, dist="uniform", b_col_major=True, epi="bias_gelu")
    y, S = orc.gemm(wl.bf16_bits(case.a), wl.bf16_bits(case.b), b_col_major=True,
                    bias=wl.bf16_bits(case.bias), epi="bias_gelu")
    z = case.a.double() @ case.b.double().T + case.bias.double()[None, :]
    ref = torch.nn.functional.gelu(z, approximate="tanh")
    assert np.all(np.abs(y - ref.numpy()) <= 1e-12 * (S + 1.0))


def pin_gelu(orc):
    zs = np.concatenate([np.linspace(-12, 12, 481), [0.0, 1e-8, -1e-8, 30.0, -30.0]])
    ours = np.array([orc.gelu_tanh(float(z)) for z in zs])
    ref = torch.nn.functional.gelu(torch.tensor(zs, dtype=torch.float64), approximate="tanh").numpy()
    assert np.all(np.abs(ours - ref) <= 1e-15 * np.maximum(1.0, np.abs(zs)))
    # the tanh form stays within 1e-3 of the exact GELU z * Phi(z) everywhere
    erf_gelu = np.array([0.5 * z * (1.0 + math.erf(z / math.sqrt(2.0))) for z in zs])
    assert np.max(np.abs(ours - erf_gelu)) < 1e-3
    assert orc.gelu_tanh(0.0) == 0.0


def pin_rows_and_degenerate(orc):
    case = wl.dense_random(50, 33, 70, seed=4, dist="uniform", epi="bias_gelu")
    a, b, bias = wl.bf16_bits(case.a), wl.bf16_bits(case.b), wl.bf16_bits(case.bias)
    y, S = orc.gemm(a, b, bias=bias, epi="bias_gelu")
    rows = np.array([49, 0, 17, 17])
    yr, Sr = orc.gemm(a, b, bias=bias, epi="bias_gelu", rows=rows)
    assert np.array_equal(yr, y[rows]) and np.array_equal(Sr, S[rows])
    # K = 0: the sum is empty, so y = epi(0)
    a0 = np.zeros((5, 0), dtype=np.uint16)
    b0 = np.zeros((0, 33), dtype=np.uint16)
    y0, S0 = orc.gemm(a0, b0)
    assert np.array_equal(y0, np.zeros((5, 33))) and np.array_equal(S0, np.zeros((5, 33)))
    y0, _ = orc.gemm(a0, b0, bias=bias, epi="bias")
    assert np.array_equal(y0, np.broadcast_to(widen(bias), (5, 33)))
    # M = 0: no rows
    ye, _ = orc.gemm(np.zeros((0, 70), dtype=np.uint16), b)
    assert ye.shape == (0, 33)


def pin_f16_widening_exhaustive(orc):
    # every binary16 bit pattern against numpy's float16 -> float64 conversion
    allbits = np.arange(65536, dtype=np.uint16)
    ref = allbits.view(np.float16).astype(np.float64)
    ours = np.array([orc.lib.oracle_f16_to_double(int(h)) for h in allbits])
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all(), f"f16 widening differs at {np.flatnonzero(~same)[:8]}"
    assert np.array_equal(np.signbit(ours[~np.isnan(ours)]), np.signbit(ref[~np.isnan(ref)]))


def pin_f16_gemm(orc):
    # fp16 operands: integer-exact product against int64 matmul, and a random one against torch float64
    rng = np.random.default_rng(17)
    A = rng.integers(-8, 9, (23, 70))
    B = rng.integers(-8, 9, (70, 19))
    bias = rng.integers(-4, 5, 19)
    f16 = lambda x: np.asarray(x, dtype=np.float16).view(np.uint16)
    y, S = orc.gemm(f16(A), f16(B), bias=f16(bias), epi="bias", in_dtype="f16")
    assert np.array_equal(y, (A @ B + bias[None, :]).astype(np.float64))
    assert np.array_equal(S, (np.abs(A) @ np.abs(B)).astype(np.float64))
    a = rng.standard_normal((31, 45)).astype(np.float16)
    b = rng.standard_normal((45, 27)).astype(np.float16)
    y, S = orc.gemm(a.view(np.uint16), np.ascontiguousarray(b.T).view(np.uint16), b_col_major=True, in_dtype="f16")
    ref = a.astype(np.float64) @ b.astype(np.float64)
    assert np.all(np.abs(y - ref) <= 1e-12 * S)


def pin_row_norm(orc):
    # rmsnorm(A) . B against numpy float64 (mean, sqrt and matmul are library routines)
    rng = np.random.default_rng(23)
    M, N, K, eps = 37, 29, 200, 1e-5
    a = bits(rng.standard_normal((M, K)) * rng.uniform(0.1, 4.0, (M, 1)))
    b = bits(rng.standard_normal((K, N)) / 8)
    bias = bits(rng.standard_normal(N) / 10)
    fa, fb = widen(a), widen(b)
    an = fa / np.sqrt(np.mean(fa * fa, axis=1, keepdims=True) + eps)
    y, S = orc.gemm(a, b, bias=bias, epi="bias", row_norm_eps=eps)
    ref = an @ fb + widen(bias)[None, :]
    assert np.all(np.abs(y - ref) <= 1e-12 * (np.abs(an) @ np.abs(fb) + 1.0))
    assert np.allclose(S, np.abs(an) @ np.abs(fb), rtol=1e-12, atol=0)
    # scale invariance: rmsnorm(c A) = rmsnorm(A) for c = 2^k (exact in bf16), up to eps
    y2, _ = orc.gemm(bits(widen(a) * 4.0), b, bias=bias, epi="bias", row_norm_eps=0.0)
    y1, _ = orc.gemm(a, b, bias=bias, epi="bias", row_norm_eps=0.0)
    assert np.allclose(y1, y2, rtol=1e-12, atol=1e-12)
    # a row of ones: mean square 1, scale 1/sqrt(1 + eps)
    ones = bits(np.ones((1, K)))
    y, _ = orc.gemm(ones, b, row_norm_eps=0.25)
    assert np.allclose(y, fb.sum(axis=0, keepdims=True) / np.sqrt(1.25), rtol=1e-13, atol=0)


PINS = [pin_golden, pin_identity_permutation, pin_rank1, pin_integer_exact,
        pin_fraction_bruteforce, pin_torch_float64, pin_gelu, pin_rows_and_degenerate,
        pin_f16_widening_exhaustive, pin_f16_gemm, pin_row_norm]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.default())


def test_bf16_widening_exact():
    for v in [0.0, -0.0, 1.0, -2.5, 3.140625, 1e-3, 65504.0, 1e30]:
        b = bits([v])[0]
        assert oracle.bf16_to_double(int(b)) == float(torch.tensor(v).to(torch.bfloat16).double())


def test_compare_detects_errors():
    y = np.array([[1.0, 2.0]])
    s = np.array([[1.0, 2.0]])
    assert oracle.compare(y, y, s)["ok"]
    assert not oracle.compare(y + 0.05, y, s)["ok"]
    assert not oracle.compare(np.array([[np.nan, 2.0]]), y, s)["ok"]
    # an all-NaN result is reported as bad (worst element found), not an exception
    import warnings
    with warnings.catch_warnings():
        warnings.simplefilter("ignore", RuntimeWarning)
        r = oracle.compare(np.full((1, 2), np.nan), y, s)
    assert not r["ok"] and r["n_bad"] == 2 and r["worst"] is not None


# ----------------------------------------------------------------------------------------
# Planted mistakes: each mutant of oracle.c must fail at least one pin.

MUTANTS = {
    "dropped_last_k": ("for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 0; k + 1 < K; ++k) {"),
    "transposed_b": ("B[k * ldb + j], in_dtype);", "B[j * ldb + k], in_dtype);"),
    "bias_sign": ("y[j] + widen(bias[j], in_dtype)", "y[j] - widen(bias[j], in_dtype)"),
    "bias_index": ("widen(bias[j], in_dtype)", "widen(bias[0], in_dtype)"),
    "gelu_cubic": ("0.044715 * z * z * z", "0.044715 * z * z"),
    "gelu_scale": ("sqrt(2.0 / 3.14159265358979323846)", "sqrt(1.0 / 3.14159265358979323846)"),
    "s_not_abs": ("s[j] += fabs(p);", "s[j] += p;"),
    "a_k_reversed": ("A[i * lda + k], in_dtype);", "A[i * lda + (K - 1 - k)], in_dtype);"),
    "norm_sum_not_mean": ("scale = 1.0 / sqrt(ss / (double)K + eps);", "scale = 1.0 / sqrt(ss + eps);"),
    "norm_abs_not_square": ("ss += a * a;", "ss += fabs(a);"),
    "gelu_half_dropped": ("return 0.5 * z * (1.0 + tanh(", "return z * (1.0 + tanh("),
    "gelu_tanh_sign": ("(1.0 + tanh(c * (z + 0.044715 * z * z * z)))", "(1.0 - tanh(c * (z + 0.044715 * z * z * z)))"),
    "norm_eps_dropped": ("scale = 1.0 / sqrt(ss / (double)K + eps);", "scale = 1.0 / sqrt(ss / (double)K);"),
    "f16_exponent_bias": ("v = ldexp((double)(1024 + f), e - 25);", "v = ldexp((double)(1024 + f), e - 24);"),
    "f16_subnormal_scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
}


def _run_pins_against(lib_path: str) -> list:
    caught = []
    orc = oracle.Oracle(lib_path)
    for pin in PINS:
        try:
            pin(orc)
        except (AssertionError, RuntimeError, ValueError, IndexError):
            caught.append(pin.__name__)
    return caught


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutant_src = tmp_path / "oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutant_src), out=str(tmp_path / "liboracle_mutant.so"))
    # A mutant may index out of bounds; run it in a child so a crash cannot take
    # the test process down.  A crash counts as caught.
    code = ("import sys; sys.path.insert(0, %r); sys.path.insert(0, %r); "
            "import test_oracle as t; print('CAUGHT=' + ','.join(t._run_pins_against(%r)))"
            % (os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
               os.path.dirname(os.path.abspath(__file__)), lib))
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    if proc.returncode != 0:
        return  # crashed or raised outside a pin: the mutant did not survive
    line = [l for l in proc.stdout.splitlines() if l.startswith("CAUGHT=")][-1]
    assert line != "CAUGHT=", f"mutant {name} passed every pin"
