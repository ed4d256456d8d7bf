"""Host-side tests of the C ABI (no GPU needed, no compute call is made).

The library must load, export every function include/tg.h declares, and turn
bad arguments into error codes on the host before anything is enqueued.
"""
import ctypes
import subprocess
import sys

import pytest

import grouped_gemm_persistent_gb300 as tg
from grouped_gemm_persistent_gb300 import _binding
from grouped_gemm_persistent_gb300.build import build

NULL = None
ALIGNED = 0x10000          # fake, 16-byte aligned device addresses: never dereferenced on these paths
ALIGNED_B = 0x20000
ALIGNED_C = 0x30000


@pytest.fixture(scope="module")
def lib():
    build()
    return tg.load()


def gemm(lib, A=ALIGNED, la=0, lda=64, B=ALIGNED_B, lb=0, ldb=64, C=ALIGNED_C, cd=0, ldc=64,
         M=64, N=64, K=64, epi=0, bias=NULL):
    return lib.tg_gemm(A, la, lda, B, lb, ldb, C, cd, ldc, M, N, K, epi, bias, NULL)


def test_exports_every_declared_symbol(lib):
    declared = tg.header_functions()
    assert {"tg_gemm", "tg_grouped_gemm", "tg_status_string", "tg_device_status"} <= set(declared)
    for name in declared:
        assert hasattr(lib, name), f"libtg.so does not export {name}"
    out = subprocess.run(["nm", "-D", "--defined-only", _binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(declared) <= exported


def test_no_driver_link_dependency(lib):
    # The driver entry point is looked up at run time, so the library loads on
    # machines without libcuda (this one) and picks up the box's driver there.
    out = subprocess.run(["ldd", _binding.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def test_status_strings(lib):
    for code in range(6):
        s = lib.tg_status_string(code)
        assert s and isinstance(s, bytes)
    assert lib.tg_status_string(99) == b"unknown status"
    assert lib.tg_version() == (0 << 16) | 2
    assert lib.tg_launch_count() == 0     # no kernel was enqueued by this thread


def test_degenerate_sizes_are_noops(lib):
    # M == 0 or N == 0: nothing to do, returns before touching the device
    assert gemm(lib, M=0) == tg.TG_OK
    assert gemm(lib, N=0, C=NULL) == tg.TG_OK
    assert gemm(lib, M=0, A=NULL, B=NULL, C=NULL) == tg.TG_OK


@pytest.mark.parametrize("kwargs,code", [
    (dict(M=-1), tg.TG_ERR_INVALID_ARG),
    (dict(K=-5), tg.TG_ERR_INVALID_ARG),
    (dict(C=NULL), tg.TG_ERR_INVALID_ARG),
    (dict(A=NULL), tg.TG_ERR_INVALID_ARG),
    (dict(B=NULL), tg.TG_ERR_INVALID_ARG),
    (dict(la=7), tg.TG_ERR_INVALID_ARG),
    (dict(lb=-1), tg.TG_ERR_INVALID_ARG),
    (dict(cd=3), tg.TG_ERR_INVALID_ARG),
    (dict(epi=9), tg.TG_ERR_INVALID_ARG),
    (dict(epi=1, bias=NULL), tg.TG_ERR_INVALID_ARG),
    (dict(epi=2, bias=NULL), tg.TG_ERR_INVALID_ARG),
    (dict(lda=32), tg.TG_ERR_INVALID_ARG),                   # row-major A: lda < K
    (dict(la=1, lda=32, M=64), tg.TG_ERR_INVALID_ARG),       # column-major A: lda < M
    (dict(ldb=32), tg.TG_ERR_INVALID_ARG),                   # row-major B: ldb < N
    (dict(lb=1, ldb=32), tg.TG_ERR_INVALID_ARG),             # column-major B: ldb < K
    (dict(ldc=10), tg.TG_ERR_INVALID_ARG),                   # ldc < N
    (dict(A=ALIGNED + 8), tg.TG_ERR_UNSUPPORTED),            # TMA needs 16-byte aligned bases
    (dict(B=ALIGNED_B + 2), tg.TG_ERR_UNSUPPORTED),
    (dict(C=ALIGNED_C + 4), tg.TG_ERR_UNSUPPORTED),
    (dict(lda=66, K=64), tg.TG_ERR_UNSUPPORTED),             # row stride not a multiple of 16 bytes
    (dict(ldc=66), tg.TG_ERR_UNSUPPORTED),
    (dict(cd=1, ldc=66), tg.TG_ERR_UNSUPPORTED),             # fp32: ldc % 4
    (dict(M=1 << 31), tg.TG_ERR_UNSUPPORTED),
    (dict(epi=1, bias=ALIGNED + 1), tg.TG_ERR_INVALID_ARG),  # bias must be 2-byte aligned
])
def test_bad_arguments(lib, kwargs, code):
    assert gemm(lib, **kwargs) == code
    assert lib.tg_last_error_message()  # a description is always left behind


def _no_gpu():
    # Calls below pass the host checks with fake addresses; with a GPU present they
    # would launch on them, so they only run where there is none.
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("the call would reach a real device with fake addresses")
    except ImportError:
        pass


def test_k_zero_needs_no_operands(lib):
    # K == 0 passes the checks with NULL A/B and odd ld (then needs a device)
    _no_gpu()
    rc = gemm(lib, A=NULL, B=NULL, lda=0, ldb=0, K=0)
    assert rc != tg.TG_ERR_INVALID_ARG and rc != tg.TG_ERR_UNSUPPORTED


def test_grouped_table_checks(lib):
    P = _binding.GroupProblem
    assert lib.tg_grouped_gemm(None, 0, None) == tg.TG_OK
    assert lib.tg_grouped_gemm(None, 3, None) == tg.TG_ERR_INVALID_ARG
    assert lib.tg_grouped_gemm(None, -1, None) == tg.TG_ERR_INVALID_ARG
    empty = (P * 3)(P(0, 64, 64), P(0, 64, 64), P(5, 0, 64))
    assert lib.tg_grouped_gemm(empty, 3, None) == tg.TG_OK  # every group empty: nothing to launch
    good = P(64, 64, 64, ALIGNED, 64, 0, ALIGNED_B, 64, 0, ALIGNED_C, 64, 0, 0, None)
    bad = P(64, 64, 64, ALIGNED, 64, 0, ALIGNED_B, 64, 0, None, 64, 0, 0, None)
    arr = (P * 3)(good, P(0, 64, 64), bad)
    assert lib.tg_grouped_gemm(arr, 3, None) == tg.TG_ERR_INVALID_ARG
    assert b"problem 2" in lib.tg_last_error_message()


def test_struct_layout_matches_header():
    # natural layout of tg_group_problem on LP64: 14 fields, 112 bytes
    assert ctypes.sizeof(_binding.GroupProblem) == 112
    assert _binding.GroupProblem.bias.offset == 96
    assert _binding.GroupProblem.epi.offset == 92
    assert _binding.GroupProblem.ab_dtype.offset == 104


def test_gemm_ex_checks(lib):
    P = _binding.GroupProblem
    good = P(64, 64, 64, ALIGNED, 64, 0, ALIGNED_B, 64, 0, ALIGNED_C, 64, 2, 0, None, 2)   # fp16 in, fp16 out
    assert lib.tg_gemm_ex(None, None) == tg.TG_ERR_INVALID_ARG
    bad_ab = P(64, 64, 64, ALIGNED, 64, 0, ALIGNED_B, 64, 0, ALIGNED_C, 64, 0, 0, None, 1)  # fp32 operands
    assert lib.tg_gemm_ex(ctypes.byref(bad_ab), None) == tg.TG_ERR_INVALID_ARG
    assert b"ab_dtype" in lib.tg_last_error_message()
    bad_c = P(64, 64, 64, ALIGNED, 64, 0, ALIGNED_B, 64, 0, ALIGNED_C, 64, 3, 0, None, 0)
    assert lib.tg_gemm_ex(ctypes.byref(bad_c), None) == tg.TG_ERR_INVALID_ARG
    empty = P(0, 64, 64, None, 64, 0, None, 64, 0, None, 64, 2, 0, None, 2)
    assert lib.tg_gemm_ex(ctypes.byref(empty), None) == tg.TG_OK
    assert good.ab_dtype == 2


def test_hooks_validate(lib):
    assert lib.tg_set_wait_budget_ms(3600001) == tg.TG_ERR_INVALID_ARG
    assert lib.tg_set_wait_budget_ms(0) == tg.TG_OK
    assert lib.tg_debug_withhold_stage(-2) == tg.TG_ERR_INVALID_ARG
    assert lib.tg_debug_withhold_stage(-1) == tg.TG_OK


def test_valid_call_without_device_fails_loudly():
    # On a machine with no GPU a valid call must return an error, never TG_OK
    # (no silent CPU path).  Run in a child so no CUDA state leaks into this process.
    code = ("import grouped_gemm_persistent_gb300 as tg; l = tg.load(); "
            "print(l.tg_gemm(0x10000, 0, 64, 0x20000, 0, 64, 0x30000, 0, 64, 64, 64, 64, 0, None, None))")
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    rc = int(out.stdout.strip().splitlines()[-1])
    assert rc in (tg.TG_ERR_NO_DEVICE, tg.TG_ERR_CUDA)


def test_bcast_argument_checks(lib):
    def bc(U=64, repeat=4, A=ALIGNED, lda=64, C=ALIGNED_C, K=64, N=64):
        return lib.tg_gemm_bcast(A, 0, lda, U, repeat, ALIGNED_B, 0, 64, C, 0, 64, N, K, 0, None, None)
    assert bc(repeat=0) == tg.TG_ERR_INVALID_ARG
    assert bc(U=-1) == tg.TG_ERR_INVALID_ARG
    assert bc(U=1 << 20, repeat=1 << 12) == tg.TG_ERR_UNSUPPORTED      # U * repeat >= 2^31
    assert bc(C=None) == tg.TG_ERR_INVALID_ARG
    assert bc(lda=32) == tg.TG_ERR_INVALID_ARG
    assert bc(U=0) == tg.TG_OK


def test_moe_argument_checks(lib):
    def moe(T=256, K=64, G=4, N=64, counts=0x40000, A=ALIGNED, B=ALIGNED_B, C=ALIGNED_C, stride=64 * 64, lb=0):
        return lib.tg_moe_gemm(A, 64, T, K, B, lb, 64, stride, G, N, C, 0, 64, counts, 0, None, None)
    assert moe(T=0) == tg.TG_OK and moe(G=0) == tg.TG_OK            # nothing to do
    assert moe(G=191) == tg.TG_ERR_UNSUPPORTED                          # schedule table limit
    assert moe(counts=None) == tg.TG_ERR_INVALID_ARG
    assert moe(counts=0x40002) == tg.TG_ERR_INVALID_ARG                 # counts must be 4-byte aligned
    assert moe(stride=64 * 63) == tg.TG_ERR_INVALID_ARG                 # one expert does not fit its stride
    assert moe(T=-1) == tg.TG_ERR_INVALID_ARG
    _no_gpu()
    rc = moe(N=60)                                                      # any N: per-expert maps clip the columns
    assert rc not in (tg.TG_ERR_INVALID_ARG, tg.TG_ERR_UNSUPPORTED)


def test_rmsnorm_argument_checks(lib):
    f = ctypes.c_float
    def rms(A=ALIGNED, lda=64, M=64, K=64, eps=1e-6, r=0x40000):
        return lib.tg_row_rms(A, lda, M, K, f(eps), r, None)
    assert rms(M=0) == tg.TG_OK                                         # nothing to do
    assert rms(M=-1) == tg.TG_ERR_INVALID_ARG
    assert rms(r=None) == tg.TG_ERR_INVALID_ARG
    assert rms(r=0x40002) == tg.TG_ERR_INVALID_ARG                      # fp32 output, 4-byte aligned
    assert rms(eps=-1.0) == tg.TG_ERR_INVALID_ARG
    assert rms(eps=float("nan")) == tg.TG_ERR_INVALID_ARG
    assert rms(A=None) == tg.TG_ERR_INVALID_ARG
    assert rms(lda=32) == tg.TG_ERR_INVALID_ARG                         # lda < K
    assert rms(lda=68) == tg.TG_ERR_UNSUPPORTED                         # rows not 16-byte aligned
    assert rms(A=ALIGNED + 2) == tg.TG_ERR_UNSUPPORTED

    def fused(M=64, N=64, K=64, A=ALIGNED, rs=0x40000, ldb=64, epi=0, bias=NULL):
        return lib.tg_gemm_rmsnorm(A, 64, ALIGNED_B, 0, ldb, ALIGNED_C, 0, 64, M, N, K, f(1e-6), rs, epi, bias, None)
    assert fused(M=0) == tg.TG_OK and fused(N=0) == tg.TG_OK
    assert fused(rs=None) == tg.TG_ERR_INVALID_ARG
    assert fused(A=None) == tg.TG_ERR_INVALID_ARG
    assert fused(ldb=32) == tg.TG_ERR_INVALID_ARG
    assert fused(epi=1) == tg.TG_ERR_INVALID_ARG                        # bias epilogue without a bias


def _declared_arity():
    """Parameter count of every function prototype in include/tg.h."""
    import re
    text = open(_binding.HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    arity = {}
    for name, params in re.findall(r"\b(tg_[a-z_]+)\s*\(([^)]*)\)\s*;", text):
        params = params.strip()
        arity[name] = 0 if params in ("", "void") else params.count(",") + 1
    return arity


def test_binding_argtypes_match_header_arity(lib):
    # the ctypes prototypes must take as many arguments as the C declarations
    arity = _declared_arity()
    assert set(arity) == set(tg.header_functions())
    for name, n in arity.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name} has no argtypes in the binding"
        assert len(fn.argtypes) == n, f"{name}: header takes {n} arguments, binding {len(fn.argtypes)}"
