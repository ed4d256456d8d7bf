"""grouped_gemm_persistent_gb300: bf16 GEMM and grouped (MoE) GEMM for NVIDIA GB300.

The compute path is libtg.so (hand-written CUDA for sm_103a: TMA producer,
tcgen05 MMA into TMEM, fused bias/GELU epilogue, persistent tile scheduler)
behind the C ABI in include/tg.h.  This package holds the ctypes binding
(argument marshalling only), the in-tree build script, and the seeded input
generators (``workloads``) shared by the tests and the benchmark.
"""
from ._binding import (BF16, COL_MAJOR, EPILOGUES, F16, F32, ROW_MAJOR, TG_ERR_CUDA, TG_ERR_INVALID_ARG,
                       TG_ERR_NO_DEVICE, TG_ERR_TIMEOUT, TG_ERR_UNSUPPORTED, TG_OK, GroupProblem, TGError,
                       build_moe_table, debug_trace, debug_withhold_stage, device_status, gemm, gemm_bcast, gemm_rmsnorm,
                       grouped_gemm_table, header_functions, launch_count, load, row_rms,
                       grouped_gemm_table_noalloc, make_problem, moe_gemm_device, moe_grouped_gemm, set_wait_budget_ms, version)

__all__ = ["gemm", "gemm_bcast", "gemm_rmsnorm", "row_rms", "moe_gemm_device", "moe_grouped_gemm", "grouped_gemm_table", "grouped_gemm_table_noalloc", "build_moe_table", "make_problem", "device_status", "set_wait_budget_ms",
           "debug_withhold_stage", "debug_trace", "launch_count", "version", "load", "header_functions", "GroupProblem", "TGError", "EPILOGUES",
           "ROW_MAJOR", "COL_MAJOR", "BF16", "F32", "F16", "TG_OK", "TG_ERR_INVALID_ARG", "TG_ERR_UNSUPPORTED",
           "TG_ERR_CUDA", "TG_ERR_TIMEOUT", "TG_ERR_NO_DEVICE"]
