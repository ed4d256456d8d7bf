"""ctypes binding of libtg (include/tg.h).  Argument marshalling only.

Every compute step runs in the CUDA kernels of libtg.so.  There is no Python,
PyTorch or CPU fallback: if the library is not built, or the device is not a
GB300 (sm_103a), these functions raise.  PyTorch supplies device memory and
streams; tensors are passed as raw device pointers with their strides.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# TG_LIB_PATH selects another build of the library (e.g. to compare two builds on one GPU).
LIB_PATH = os.environ.get("TG_LIB_PATH") or os.path.join(_PKG, "libtg.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "tg.h")

TG_OK, TG_ERR_INVALID_ARG, TG_ERR_UNSUPPORTED, TG_ERR_CUDA, TG_ERR_TIMEOUT, TG_ERR_NO_DEVICE = range(6)
STATUS_NAMES = {0: "TG_OK", 1: "TG_ERR_INVALID_ARG", 2: "TG_ERR_UNSUPPORTED", 3: "TG_ERR_CUDA",
                4: "TG_ERR_TIMEOUT", 5: "TG_ERR_NO_DEVICE"}
EPILOGUES = {"none": 0, "bias": 1, "bias_gelu": 2}
ROW_MAJOR, COL_MAJOR = 0, 1
BF16, F32, F16 = 0, 1, 2
_DTYPE_CODE = {torch.bfloat16: BF16, torch.float32: F32, torch.float16: F16}

_lib = None
_lock = threading.Lock()


class TGError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


class GroupProblem(ctypes.Structure):
    """Mirror of tg_group_problem (field order and natural alignment as in tg.h)."""
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
        ("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("layout_a", ctypes.c_int),
        ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64), ("layout_b", ctypes.c_int),
        ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64), ("c_dtype", ctypes.c_int),
        ("epi", ctypes.c_int),
        ("bias", ctypes.c_void_p),
        ("ab_dtype", ctypes.c_int),
    ]


def header_functions() -> list[str]:
    """Names of the functions include/tg.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tg_[a-z_]+)\s*\(", text)))


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libtg.so (built by grouped_gemm_persistent_gb300.build); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libtg.so is not built ({p}); run `python -m grouped_gemm_persistent_gb300.build`")
        lib = ctypes.CDLL(p)
        i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.tg_gemm.restype = ci
        lib.tg_gemm.argtypes = [vp, ci, i64, vp, ci, i64, vp, ci, i64, i64, i64, i64, ci, vp, vp]
        lib.tg_gemm_ex.restype = ci
        lib.tg_gemm_ex.argtypes = [ctypes.POINTER(GroupProblem), vp]
        lib.tg_gemm_bcast.restype = ci
        lib.tg_gemm_bcast.argtypes = [vp, ci, i64, i64, i64, vp, ci, i64, vp, ci, i64, i64, i64, ci, vp, vp]
        lib.tg_moe_gemm.restype = ci
        lib.tg_moe_gemm.argtypes = [vp, i64, i64, i64, vp, ci, i64, i64, i64, i64, vp, ci, i64, vp, ci, vp, vp]
        lib.tg_row_rms.restype = ci
        lib.tg_row_rms.argtypes = [vp, i64, i64, i64, ctypes.c_float, vp, vp]
        lib.tg_gemm_rmsnorm.restype = ci
        lib.tg_gemm_rmsnorm.argtypes = [vp, i64, vp, ci, i64, vp, ci, i64, i64, i64, i64, ctypes.c_float, vp, ci,
                                        vp, vp]
        lib.tg_grouped_gemm.restype = ci
        lib.tg_grouped_gemm.argtypes = [ctypes.POINTER(GroupProblem), ci, vp]
        lib.tg_grouped_gemm_noalloc.restype = ci
        lib.tg_grouped_gemm_noalloc.argtypes = [ctypes.POINTER(GroupProblem), ci, vp]
        lib.tg_status_string.restype = ctypes.c_char_p
        lib.tg_status_string.argtypes = [ci]
        lib.tg_last_error_message.restype = ctypes.c_char_p
        lib.tg_last_error_message.argtypes = []
        lib.tg_device_status.restype = ci
        lib.tg_device_status.argtypes = [vp]
        lib.tg_set_wait_budget_ms.restype = ci
        lib.tg_set_wait_budget_ms.argtypes = [ctypes.c_uint32]
        lib.tg_debug_withhold_stage.restype = ci
        lib.tg_debug_withhold_stage.argtypes = [i64]
        lib.tg_debug_withhold_stage_in.restype = ci
        lib.tg_debug_withhold_stage_in.argtypes = [i64, ctypes.c_int32]
        lib.tg_debug_trace.restype = ci
        lib.tg_debug_trace.argtypes = [vp, i64, vp, i64]
        lib.tg_version.restype = ctypes.c_uint32
        lib.tg_version.argtypes = []
        lib.tg_launch_count.restype = ctypes.c_uint64
        lib.tg_launch_count.argtypes = []
        if path is None:
            _lib = lib
        return lib


def _check(status: int) -> None:
    if status != TG_OK:
        msg = load().tg_last_error_message().decode(errors="replace")
        raise TGError(status, msg)


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _matrix(t: torch.Tensor, name: str):
    """(layout, ld) of a 2-D tensor view: row-major if its rows are contiguous, else column-major.

    With a single row (or column) the leading dimension is never used to step;
    it is then reported as the extent rounded up to 8 elements, which keeps the
    TMA stride rule satisfied.
    """
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(t.shape)}")
    r, c = t.shape
    s0, s1 = t.stride()
    if s1 == 1 or c == 1:
        return ROW_MAJOR, (s0 if r > 1 else -(-max(c, 1) // 8) * 8)
    if s0 == 1 or r == 1:
        return COL_MAJOR, (s1 if c > 1 else -(-max(r, 1) // 8) * 8)
    raise ValueError(f"{name}: neither rows nor columns are contiguous (strides {t.stride()})")


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def gemm(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None, *, bias: torch.Tensor | None = None,
         epilogue: str = "none", out_dtype: torch.dtype = torch.bfloat16, stream=None) -> torch.Tensor:
    """out[M,N] = epilogue(a[M,K] @ b[K,N]) on the GPU (tg_gemm, or tg_gemm_ex for fp16 operands).

    ``a``/``b`` are bf16 or fp16 CUDA tensors of the same type (``bias`` too);
    each may be a row-major or column-major view (a transposed view of a
    row-major tensor is column-major).  ``out`` (bf16, fp16 or fp32, rows
    contiguous, row stride may exceed N) is allocated if not given.
    Asynchronous on ``stream`` (default: torch's current stream).
    """
    if a.dtype not in (torch.bfloat16, torch.float16) or b.dtype != a.dtype:
        raise TypeError("a and b must both be torch.bfloat16 or both torch.float16")
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    if out.dtype not in _DTYPE_CODE or tuple(out.shape) != (M, N):
        raise ValueError("out must be [M, N] bf16, fp16 or fp32")
    la, lda = _matrix(a, "a")
    lb, ldb = _matrix(b, "b")
    lc, ldc = _matrix(out, "out")
    if lc != ROW_MAJOR:
        raise ValueError("out must be row-major")
    epi = EPILOGUES[epilogue]
    if epi and (bias is None or bias.dtype != a.dtype or bias.numel() != N or not bias.is_contiguous()):
        raise ValueError("this epilogue needs a contiguous bias of length N with the operands' dtype")
    if a.dtype == torch.bfloat16:
        _check(load().tg_gemm(_ptr(a), la, lda, _ptr(b), lb, ldb, _ptr(out), _DTYPE_CODE[out.dtype], ldc, M, N, K,
                              epi, _ptr(bias) if epi else None, _stream_handle(stream)))
    else:
        prob = GroupProblem(M, N, K, _ptr(a), lda, la, _ptr(b), ldb, lb, _ptr(out), ldc, _DTYPE_CODE[out.dtype], epi,
                            _ptr(bias) if epi else None, F16)
        _check(load().tg_gemm_ex(ctypes.byref(prob), _stream_handle(stream)))
    return out


def gemm_bcast(a_user: torch.Tensor, b: torch.Tensor, repeat: int, out: torch.Tensor | None = None, *,
               bias: torch.Tensor | None = None, epilogue: str = "none", out_dtype: torch.dtype = torch.bfloat16,
               stream=None) -> torch.Tensor:
    """out[U*repeat, N] = epilogue(A @ b) with A's row i*repeat + j equal to a_user[i] (tg_gemm_bcast).

    The repeated rows are never materialised: the kernel reads ``a_user`` [U, K]
    once per replica and stores each result row ``repeat`` times.
    """
    if a_user.dtype != torch.bfloat16 or b.dtype != torch.bfloat16:
        raise TypeError("a_user and b must be torch.bfloat16")
    U, K = a_user.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        out = torch.empty((U * repeat, N), dtype=out_dtype, device=a_user.device)
    if tuple(out.shape) != (U * repeat, N):
        raise ValueError("out must be [U * repeat, N]")
    la, lda = _matrix(a_user, "a_user")
    lb, ldb = _matrix(b, "b")
    lc, ldc = _matrix(out, "out")
    if lc != ROW_MAJOR:
        raise ValueError("out must be row-major")
    epi = EPILOGUES[epilogue]
    if epi and (bias is None or bias.dtype != torch.bfloat16 or bias.numel() != N or not bias.is_contiguous()):
        raise ValueError("this epilogue needs a contiguous bf16 bias of length N")
    _check(load().tg_gemm_bcast(_ptr(a_user), la, lda, U, repeat, _ptr(b), lb, ldb, _ptr(out),
                                _DTYPE_CODE[out.dtype], ldc, N, K, epi,
                                _ptr(bias) if epi else None, _stream_handle(stream)))
    return out


def _row_major_bf16(a: torch.Tensor, name: str) -> int:
    if a.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be torch.bfloat16")
    la, lda = _matrix(a, name)
    if la != ROW_MAJOR:
        raise ValueError(f"{name} must be row-major")
    return lda


def row_rms(a: torch.Tensor, eps: float, out: torch.Tensor | None = None, *, stream=None) -> torch.Tensor:
    """out[i] = 1 / sqrt(mean_k a[i, k]^2 + eps), fp32 [M], for a row-major bf16 ``a`` (tg_row_rms)."""
    lda = _row_major_bf16(a, "a")
    M, K = a.shape
    if out is None:
        out = torch.empty(M, dtype=torch.float32, device=a.device)
    if out.dtype != torch.float32 or out.numel() != M or not out.is_contiguous():
        raise ValueError("out must be a contiguous fp32 tensor of length M")
    _check(load().tg_row_rms(_ptr(a), lda, M, K, float(eps), _ptr(out), _stream_handle(stream)))
    return out


def gemm_rmsnorm(a: torch.Tensor, b: torch.Tensor, eps: float, out: torch.Tensor | None = None, *,
                 row_scale: torch.Tensor | None = None, bias: torch.Tensor | None = None, epilogue: str = "none",
                 out_dtype: torch.dtype = torch.bfloat16, stream=None) -> torch.Tensor:
    """out = epilogue(rmsnorm(a) @ b) with the normalisation fused into the GEMM (tg_gemm_rmsnorm).

    ``a`` is row-major bf16 [M, K]; ``b`` bf16 [K, N] in either layout.  The row
    factors land in ``row_scale`` (fp32 [M], allocated if not given).
    """
    lda = _row_major_bf16(a, "a")
    if b.dtype != torch.bfloat16:
        raise TypeError("b must be torch.bfloat16")
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    if out.dtype not in _DTYPE_CODE or tuple(out.shape) != (M, N):
        raise ValueError("out must be [M, N] bf16, fp16 or fp32")
    if row_scale is None:
        row_scale = torch.empty(M, dtype=torch.float32, device=a.device)
    if row_scale.dtype != torch.float32 or row_scale.numel() != M or not row_scale.is_contiguous():
        raise ValueError("row_scale must be a contiguous fp32 tensor of length M")
    lb, ldb = _matrix(b, "b")
    lc, ldc = _matrix(out, "out")
    if lc != ROW_MAJOR:
        raise ValueError("out must be row-major")
    epi = EPILOGUES[epilogue]
    if epi and (bias is None or bias.dtype != torch.bfloat16 or bias.numel() != N or not bias.is_contiguous()):
        raise ValueError("this epilogue needs a contiguous bf16 bias of length N")
    _check(load().tg_gemm_rmsnorm(_ptr(a), lda, _ptr(b), lb, ldb, _ptr(out), _DTYPE_CODE[out.dtype], ldc, M, N, K,
                                  float(eps), _ptr(row_scale), epi, _ptr(bias) if epi else None,
                                  _stream_handle(stream)))
    return out


def moe_gemm_device(a: torch.Tensor, b: torch.Tensor, counts: torch.Tensor, out: torch.Tensor | None = None, *,
                    bias: torch.Tensor | None = None, epilogue: str = "none",
                    out_dtype: torch.dtype = torch.bfloat16, stream=None) -> torch.Tensor:
    """MoE expert GEMM with the token counts on the GPU (tg_moe_gemm): no host round trip.

    ``a`` [T, K] bf16 row-major, rows grouped by expert; ``b`` [G, K, N] bf16 with
    each expert row-major (``b[g]`` contiguous rows) or column-major (a view of
    a [G, N, K] tensor); ``counts`` int32 CUDA tensor [G]; ``out`` [T, N]; rows
    past sum(counts) are not written.  ``bias`` is [G, N] bf16.
    """
    if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16:
        raise TypeError("a and b must be torch.bfloat16")
    if counts.dtype != torch.int32 or not counts.is_cuda or counts.dim() != 1 or not counts.is_contiguous():
        raise TypeError("counts must be a contiguous int32 CUDA tensor [G]")
    T, K = a.shape
    G, K2, N = b.shape
    if K != K2 or counts.shape[0] != G:
        raise ValueError("shapes: a [T, K], b [G, K, N], counts [G]")
    la, lda = _matrix(a, "a")
    if la != ROW_MAJOR:
        raise ValueError("a must be row-major")
    if b.stride(2) == 1:
        lb, ldb = ROW_MAJOR, b.stride(1)
    elif b.stride(1) == 1:
        lb, ldb = COL_MAJOR, b.stride(2)
    else:
        raise ValueError("each expert of b must be row- or column-major")
    if out is None:
        out = torch.empty((T, N), dtype=out_dtype, device=a.device)
    lc, ldc = _matrix(out, "out")
    epi = EPILOGUES[epilogue]
    if epi and (bias is None or bias.dtype != torch.bfloat16 or tuple(bias.shape) != (G, N) or not bias.is_contiguous()):
        raise ValueError("this epilogue needs a contiguous bf16 bias [G, N]")
    _check(load().tg_moe_gemm(_ptr(a), lda, T, K, _ptr(b), lb, ldb, b.stride(0), G, N, _ptr(out),
                              _DTYPE_CODE[out.dtype], ldc, counts.data_ptr(), epi, _ptr(bias) if epi else None,
                              _stream_handle(stream)))
    return out


def make_problem(a, b, out, *, bias=None, epilogue="none") -> GroupProblem:
    """One tg_group_problem from tensors (a may have 0 rows: an empty group)."""
    M, K = a.shape
    _, N = b.shape
    la, lda = _matrix(a, "a") if a.numel() else (ROW_MAJOR, max(K, 1))
    lb, ldb = _matrix(b, "b")
    _, ldc = _matrix(out, "out") if out.numel() else (ROW_MAJOR, max(N, 1))
    epi = EPILOGUES[epilogue]
    return GroupProblem(M, N, K, _ptr(a) if a.numel() else None, lda, la, _ptr(b), ldb, lb,
                        _ptr(out) if out.numel() else None, ldc, _DTYPE_CODE[out.dtype], epi,
                        _ptr(bias) if epi else None, F16 if b.dtype == torch.float16 else BF16)


def grouped_gemm_table(table, stream=None) -> None:
    """Call tg_grouped_gemm on a sequence of GroupProblem (or a ctypes array of them)."""
    arr = table if isinstance(table, ctypes.Array) else (GroupProblem * len(table))(*table)
    _check(load().tg_grouped_gemm(arr, len(arr), _stream_handle(stream)))


def grouped_gemm_table_noalloc(table, stream=None) -> None:
    """tg_grouped_gemm_noalloc: the same grouped GEMM with its problem table in the
    library's fixed device array (no device allocation; at most 256 non-empty problems)."""
    arr = table if isinstance(table, ctypes.Array) else (GroupProblem * len(table))(*table)
    _check(load().tg_grouped_gemm_noalloc(arr, len(arr), _stream_handle(stream)))


def build_moe_table(a: torch.Tensor, b: torch.Tensor, counts, out: torch.Tensor, *, bias: torch.Tensor | None = None,
                    epilogue: str = "none") -> ctypes.Array:
    """The tg_group_problem table of an MoE expert GEMM (see moe_grouped_gemm), built once for reuse."""
    counts = [int(c) for c in counts]
    G = len(counts)
    if b.dim() != 3 or b.shape[0] != G:
        raise ValueError("b must be [G, K, N] with G = len(counts)")
    total = sum(counts)
    if a.shape[0] != total or out.shape[0] != total:
        raise ValueError(f"a and out need {total} rows (sum of counts)")
    table = []
    r = 0
    for g, m in enumerate(counts):
        table.append(make_problem(a[r:r + m], b[g], out[r:r + m], bias=None if bias is None else bias[g],
                                  epilogue=epilogue))
        r += m
    return (GroupProblem * G)(*table)


def moe_grouped_gemm(a: torch.Tensor, b: torch.Tensor, counts, out: torch.Tensor | None = None, *,
                     bias: torch.Tensor | None = None, epilogue: str = "none",
                     out_dtype: torch.dtype = torch.bfloat16, stream=None) -> torch.Tensor:
    """MoE expert GEMM: rows of ``a`` [sum M_g, K] grouped by expert (``counts`` on the host),
    expert g's rows times ``b[g]`` ([G, K, N], each a row- or column-major view) into ``out`` [sum M_g, N].
    ``bias`` is [G, N] bf16 when the epilogue uses one."""
    if out is None:
        out = torch.empty((a.shape[0], b.shape[2]), dtype=out_dtype, device=a.device)
    grouped_gemm_table(build_moe_table(a, b, counts, out, bias=bias, epilogue=epilogue), stream)
    return out


def device_status(stream=None) -> None:
    """Synchronise ``stream`` and raise TGError if a kernel reported a timeout or CUDA failed."""
    _check(load().tg_device_status(_stream_handle(stream)))


def set_wait_budget_ms(ms: int) -> None:
    _check(load().tg_set_wait_budget_ms(ms))


def debug_withhold_stage(k_block: int, block: int = 0) -> None:
    """Arm the failure-path test hook for this thread's next launch (tg_debug_withhold_stage_in)."""
    _check(load().tg_debug_withhold_stage_in(k_block, block))


def debug_trace(tile_records: torch.Tensor | None, cta_records: torch.Tensor | None = None) -> None:
    """Arm a timeline trace of this thread's next launch (see tg_debug_trace in include/tg.h).

    ``tile_records`` is an int64 CUDA tensor [T, 4] and ``cta_records`` [B, 4]; the
    capacities passed to the library are T and B records of four stamps each."""
    for name, t in (("tile_records", tile_records), ("cta_records", cta_records)):
        if t is not None and (t.dim() != 2 or t.shape[1] != 4 or t.dtype != torch.int64 or not t.is_contiguous()
                              or not t.is_cuda):
            raise ValueError(f"{name} must be a contiguous int64 CUDA tensor of shape [n, 4]")
    tp = 0 if tile_records is None else tile_records.data_ptr()
    tc = 0 if tile_records is None else tile_records.shape[0]
    cp = 0 if cta_records is None else cta_records.data_ptr()
    cc = 0 if cta_records is None else cta_records.shape[0]
    _check(load().tg_debug_trace(tp or None, tc, cp or None, cc))


def launch_count() -> int:
    """Kernels this thread has enqueued through libtg so far (tg_launch_count)."""
    return int(load().tg_launch_count())


def version() -> tuple[int, int]:
    v = load().tg_version()
    return v >> 16, v & 0xFFFF
