"""CPU oracle for C = epilogue(A . B) with bf16 inputs, in fp64.

TEST INFRASTRUCTURE ONLY.  The test suite, the package's ``smoke()`` check and
the benchmark's CPU-baseline leg are the only callers.  The product path (the
CUDA library and its binding) never imports this package, and this package
imports nothing from the product.  It shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain C, built with gcc on first use);
this module marshals numpy arrays into it and states the acceptance bound.

Definition followed ("How We Built TLX", section "Introducing TLX", the
standard Triton tiled-matmul listing: an fp32 accumulator summed over K, then
stored; the TileGym/cuTile tutorial page: multiply, add bias, apply GELU in
one pass): y_ij = epi(sum_k a_ik b_kj (+ bias_j)), in double, k ascending.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

EPI = {"none": 0, "bias": 1, "bias_gelu": 2}

_default = None
_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    stale = (not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src))
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-ffp-contract=off", src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


class Oracle:
    """One loaded build of oracle.c (the default one, or a test's mutant)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, dp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double)
        vp = ctypes.c_void_p
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm.argtypes = [vp, ctypes.c_int, i64, vp, ctypes.c_int, i64,
                                    vp, ctypes.c_int, ctypes.c_int, i64, i64, i64, vp, i64, dp, dp]
        lib.oracle_gemm_norm.restype = ctypes.c_int
        lib.oracle_gemm_norm.argtypes = [vp, ctypes.c_int, i64, vp, ctypes.c_int, i64, vp, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_double, i64, i64, i64, vp, i64, dp, dp]
        lib.oracle_f16_to_double.restype = ctypes.c_double
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_gelu_tanh.restype = ctypes.c_double
        lib.oracle_gelu_tanh.argtypes = [ctypes.c_double]
        lib.oracle_num_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def gemm(self, a, b, *, a_col_major=False, b_col_major=False, bias=None, epi="none", rows=None,
             in_dtype="bf16", row_norm_eps=None):
        return _gemm(self.lib, a, b, a_col_major, b_col_major, bias, epi, rows, in_dtype, row_norm_eps)

    def gelu_tanh(self, z: float) -> float:
        return self.lib.oracle_gelu_tanh(z)


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def num_threads() -> int:
    """OpenMP threads the oracle runs with (all cores the process may use)."""
    return default().lib.oracle_num_threads()


def bf16_to_double(bits: int) -> float:
    return default().lib.oracle_bf16_to_double(bits)


def f16_to_double(bits: int) -> float:
    return default().lib.oracle_f16_to_double(bits)


def gelu_tanh(z: float) -> float:
    return default().gelu_tanh(z)


def _storage(x: np.ndarray, name: str):
    """(pointer, leading dimension) of a 2-D uint16 array with unit inner stride."""
    if x.dtype != np.uint16 or x.ndim != 2:
        raise ValueError(f"{name}: want a 2-D uint16 (bf16 bits) array, got {x.dtype} {x.shape}")
    if x.size == 0:
        return x.ctypes.data, max(x.shape[1], 1)
    if (x.shape[1] > 1 and x.strides[1] != 2) or x.strides[0] % 2:
        raise ValueError(f"{name}: inner stride must be 1 element")
    return x.ctypes.data, max(x.strides[0] // 2, x.shape[1])


def gemm(a: np.ndarray, b: np.ndarray, *, a_col_major: bool = False, b_col_major: bool = False,
         bias: np.ndarray | None = None, epi: str = "none", rows=None, in_dtype: str = "bf16",
         row_norm_eps: float | None = None):
    """Reference y and s for C = epi(A . B).

    ``a`` is A's storage: [M, K] (row-major) or [K, M] (column-major, i.e.
    A^T stored row-major).  ``b`` is [K, N] (row-major) or [N, K]
    (column-major).  Both hold bf16 bit patterns as uint16; a row stride
    larger than the row (a padded leading dimension) is allowed.  ``bias`` is
    uint16 [N].  ``rows`` selects output rows (default: all).  ``in_dtype``
    ("bf16" or "f16") is the element type the bit patterns of a, b and bias hold.
    ``row_norm_eps`` (a float) first replaces A by rmsnorm(A) with that eps.
    Returns (y, s), float64 arrays [len(rows), N] (s on the normalised A).
    """
    return _gemm(default().lib, a, b, a_col_major, b_col_major, bias, epi, rows, in_dtype, row_norm_eps)


IN_DTYPES = {"bf16": 0, "f16": 1}


def _gemm(lib, a, b, a_col_major, b_col_major, bias, epi, rows, in_dtype="bf16", row_norm_eps=None):
    pa, lda = _storage(a, "a")
    pb, ldb = _storage(b, "b")
    M, K = (a.shape[1], a.shape[0]) if a_col_major else a.shape
    Kb, N = (b.shape[1], b.shape[0]) if b_col_major else b.shape
    if Kb != K:
        raise ValueError(f"K mismatch: A has {K}, B has {Kb}")
    e = EPI[epi]
    pbias = None
    if e:
        bias = np.ascontiguousarray(bias, dtype=np.uint16)
        if bias.shape != (N,):
            raise ValueError("bias must be uint16 [N]")
        pbias = bias.ctypes.data
    if rows is None:
        prow, nrow, keep = None, M, None
    else:
        keep = np.ascontiguousarray(rows, dtype=np.int64)
        prow, nrow = keep.ctypes.data, keep.shape[0]
    y = np.empty((nrow, N), dtype=np.float64)
    s = np.empty((nrow, N), dtype=np.float64)
    rc = lib.oracle_gemm_norm(pa, int(a_col_major), lda, pb, int(b_col_major), ldb, pbias, e, IN_DTYPES[in_dtype],
                              int(row_norm_eps is not None), float(row_norm_eps or 0.0), M, N, K, prow, nrow,
                         y.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                         s.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed with code {rc}")
    del keep
    return y, s


def grouped_gemm(problems, rows_per_group=None):
    """Reference for a grouped GEMM: one plain GEMM per group, groups independent.

    ``problems`` is a list of dicts with keys a, b, and optionally a_col_major,
    b_col_major, bias, epi.  A group with M_g = 0 yields an empty result (the
    MoE reading: an expert that received no tokens produces no rows).
    ``rows_per_group`` optionally gives, per group, the rows to evaluate.
    Returns a list of (y, s) per group.
    """
    out = []
    for g, p in enumerate(problems):
        rows = None if rows_per_group is None else rows_per_group[g]
        out.append(gemm(p["a"], p["b"], a_col_major=p.get("a_col_major", False),
                        b_col_major=p.get("b_col_major", False), bias=p.get("bias"),
                        epi=p.get("epi", "none"), rows=rows, in_dtype=p.get("in_dtype", "bf16")))
    return out


def bound(s: np.ndarray, bias_abs: np.ndarray | None = None) -> np.ndarray:
    """Per-element acceptance bound 1e-2 * S_ij + 1e-5.

    With a bias epilogue the bias magnitude joins the sum the bound scales with
    (1e-2 * (S_ij + |bias_j|) + 1e-5): the stated bound has no bias term, and
    this is its plain extension to y = x + bias.  GELU's slope is below 1.13
    in magnitude, so the same bound covers bias + GELU.
    """
    scale = s if bias_abs is None else s + bias_abs[None, :]
    return 1e-2 * scale + 1e-5


def compare(c: np.ndarray, y: np.ndarray, s: np.ndarray, bias_abs: np.ndarray | None = None):
    """Element-wise check of a computed C against the oracle.

    Returns a dict: ok, max_abs_err, max_ratio (err / bound), n_bad, worst
    index, and the tight diagnostic max err / (2^-8 |y| + 2^-11 (S + |bias|)) that flags
    dropped or repeated K-slices the loose bound can miss.
    """
    c = np.asarray(c, dtype=np.float64)
    err = np.abs(c - y)
    bnd = bound(s, bias_abs)
    bad = ~(err <= bnd)  # NaN counts as bad
    ratio = err / bnd
    scale = s if bias_abs is None else s + bias_abs[None, :]
    tight = err / (2.0 ** -8 * np.abs(y) + 2.0 ** -11 * scale + 1e-30)
    # NaN ranks as the worst element
    worst = np.unravel_index(np.argmax(np.where(np.isnan(ratio), np.inf, ratio)), ratio.shape) if ratio.size else None
    return {
        "ok": bool(not bad.any()),
        "n_bad": int(bad.sum()),
        "max_abs_err": float(np.nanmax(err)) if err.size else 0.0,
        "max_ratio": float(np.nanmax(ratio)) if ratio.size else 0.0,
        "max_tight": float(np.nanmax(tight)) if tight.size else 0.0,
        "worst": tuple(int(v) for v in worst) if worst is not None else None,
    }
