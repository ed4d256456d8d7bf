// tg_launch.cuh - launch interface between the host API and the kernel
// instantiations.  The kernel template is instantiated only in tg_inst.cu
// (compiled once per (grouped, output dtype) pair so the variants build in
// parallel); the host API sees these declarations only.
#pragma once

#include <cuda_runtime.h>

#include "tg_kernel.cuh"

namespace tg {

// Enqueue one persistent launch of gemm_kernel<Cfg> with `grid` CTAs.
template <class Cfg>
cudaError_t launch(const Params& p, int grid, cudaStream_t stream);

// How many work units (CTAs, or CTA pairs) of gemm_kernel<Cfg> can be resident
// at once on the current device.
template <class Cfg>
cudaError_t resident_units(int* units);

// tg_aux.cu.  r[i] = 1 / sqrt(mean_k A[i][k]^2 + eps) for a row-major bf16 A; the
// first block also zeroes counters[0, n_counters) (stream-K tiles of the GEMM that follows).
cudaError_t launch_row_rms(const void* A, int64_t lda, int64_t M, int64_t K, float eps, float* r, int sms,
                           cudaStream_t stream, uint32_t* counters = nullptr, int n_counters = 0);
// counters[0, n) = 0, as a kernel the GEMM can follow as a programmatic dependent.
cudaError_t launch_clear_counters(uint32_t* counters, int n, cudaStream_t stream);
// maps[2 g], maps[2 g + 1] = expert g's A and C maps (templates over all T rows narrowed
// to the expert's rows from the device counts), for the device-counts MoE GEMM.
cudaError_t launch_moe_maps(const CUtensorMap& tmpl_a, const CUtensorMap& tmpl_c, const int32_t* counts, int G,
                            const void* A, int64_t a_row_bytes, void* C, int64_t c_row_bytes, int64_t T,
                            CUtensorMap* maps, cudaStream_t stream);

}  // namespace tg

// Every (BN, CTA_GROUP, A_MN, B_MN) combination for one (C_F32, MODE) pair
// (MODE 0 dense, 1 grouped table; the argument named GROUPED is that MODE).
// Index within the list: (CTA_GROUP == 2) * 8 + (BN == 256) * 4 + A_MN * 2 + B_MN.
#define TG_FOR_EACH_TILE(X, C_F32, GROUPED)          \
    X(128, 1, false, false, C_F32, GROUPED)          \
    X(128, 1, false, true, C_F32, GROUPED)           \
    X(128, 1, true, false, C_F32, GROUPED)           \
    X(128, 1, true, true, C_F32, GROUPED)            \
    X(256, 1, false, false, C_F32, GROUPED)          \
    X(256, 1, false, true, C_F32, GROUPED)           \
    X(256, 1, true, false, C_F32, GROUPED)           \
    X(256, 1, true, true, C_F32, GROUPED)            \
    X(128, 2, false, false, C_F32, GROUPED)          \
    X(128, 2, false, true, C_F32, GROUPED)           \
    X(128, 2, true, false, C_F32, GROUPED)           \
    X(128, 2, true, true, C_F32, GROUPED)            \
    X(256, 2, false, false, C_F32, GROUPED)          \
    X(256, 2, false, true, C_F32, GROUPED)           \
    X(256, 2, true, false, C_F32, GROUPED)           \
    X(256, 2, true, true, C_F32, GROUPED)

// The device-counts MoE form (MODE 2): A is always row-major [T, K].
// Index within the list: (CTA_GROUP == 2) * 4 + (BN == 256) * 2 + B_MN.
#define TG_FOR_EACH_MOE_TILE(X, C_F32)   \
    X(128, 1, false, false, C_F32, 2)     \
    X(128, 1, false, true, C_F32, 2)      \
    X(256, 1, false, false, C_F32, 2)     \
    X(256, 1, false, true, C_F32, 2)      \
    X(128, 2, false, false, C_F32, 2)     \
    X(128, 2, false, true, C_F32, 2)      \
    X(256, 2, false, false, C_F32, 2)     \
    X(256, 2, false, true, C_F32, 2)
