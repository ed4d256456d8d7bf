// tg_aux.cu - the small kernels launched before a GEMM: row statistics for the RMS
// normalisation fused into the GEMM, and the reset of the arrival counters of
// split tiles.
//
// rmsnorm(A) . B = diag(r) (A . B) with r_i = 1 / sqrt(mean_k A_ik^2 + eps): the
// normalisation is a per-row scale that the GEMM epilogue applies to its fp32
// accumulator, so the normalised A is never written to or read back from
// memory.  This pass computes r: it reads A once (memory-bound), one warp per
// row, 16-byte coalesced loads, fp32 sums in a fixed order (lane-strided
// partial sums, then a butterfly), so results are deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tg_launch.cuh"

namespace tg {

constexpr int RMS_WARPS = 8;   // rows in flight per 256-thread block
constexpr int UNROLL = 4;      // 16-byte loads in flight per lane

// Counters of split tiles start at zero in every GEMM launch that uses them.
__device__ __forceinline__ void clear_counters(uint32_t* counters, int n) {
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < n; i += blockDim.x) counters[i] = 0u;
}

__global__ void __launch_bounds__(RMS_WARPS * 32) row_rms_kernel(const uint16_t* __restrict__ A, int64_t lda,
                                                                  int64_t M, int64_t K, float eps,
                                                                  float* __restrict__ r, uint32_t* counters,
                                                                  int n_counters) {
    // the fused GEMM launched after this kernel may start its set-up and main loop now;
    // it waits for this grid's completion only before reading r (and the counters)
    ptx::grid_launch_dependents();
    clear_counters(counters, n_counters);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * RMS_WARPS;
    const int64_t kvec = K / 8;                          // whole 16-byte vectors per row
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * RMS_WARPS + warp; row < M; row += stride) {
        const uint16_t* a = A + row * lda;
        const uint4* av = reinterpret_cast<const uint4*>(a);
        float ss = 0.0f;
        auto add = [&ss](const uint4& w) {
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float lo = __uint_as_float(ws[h] << 16);
                const float hi = __uint_as_float(ws[h] & 0xffff0000u);
                ss = fmaf(lo, lo, ss);
                ss = fmaf(hi, hi, ss);
            }
        };
        int64_t v = lane;
        // UNROLL independent 16-byte loads in flight per lane, then the remainder
        for (; v + 32 * (UNROLL - 1) < kvec; v += 32 * UNROLL) {
            uint4 w[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) w[u] = __ldg(av + v + 32 * u);
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) add(w[u]);
        }
        for (; v < kvec; v += 32) add(__ldg(av + v));
        for (int64_t k = kvec * 8 + lane; k < K; k += 32) {
            const float x = __uint_as_float(static_cast<uint32_t>(__ldg(a + k)) << 16);
            ss = fmaf(x, x, ss);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        // an empty row has mean square 0 (and its product row is 0 whatever r is)
        if (lane == 0) r[row] = rsqrtf((K > 0 ? ss / static_cast<float>(K) : 0.0f) + eps);
    }
}

__global__ void __launch_bounds__(256) clear_counters_kernel(uint32_t* counters, int n) {
    ptx::grid_launch_dependents();
    clear_counters(counters, n);
}

cudaError_t launch_clear_counters(uint32_t* counters, int n, cudaStream_t stream) {
    clear_counters_kernel<<<1, 256, 0, stream>>>(counters, n);
    return cudaGetLastError();
}

cudaError_t launch_row_rms(const void* A, int64_t lda, int64_t M, int64_t K, float eps, float* r, int sms,
                           cudaStream_t stream, uint32_t* counters, int n_counters) {
    int64_t blocks = (M + RMS_WARPS - 1) / RMS_WARPS;
    const int64_t cap = static_cast<int64_t>(sms) * 8;   // a few resident blocks per SM, grid-stride beyond
    if (blocks > cap) blocks = cap;
    row_rms_kernel<<<static_cast<unsigned>(blocks), RMS_WARPS * 32, 0, stream>>>(static_cast<const uint16_t*>(A), lda,
                                                                                  M, K, eps, r, counters,
                                                                                  n_counters);
    return cudaGetLastError();
}

}  // namespace tg
