// tg_aux.cu - the small kernels launched before a GEMM: row statistics for the RMS
// normalisation fused into the GEMM, the reset of the arrival counters of
// stream-K tiles, and the per-expert tensor maps of the MoE GEMM whose token
// counts are in device memory.
//
// rmsnorm(A) . B = diag(r) (A . B) with r_i = 1 / sqrt(mean_k A_ik^2 + eps): the
// normalisation is a per-row scale that the GEMM epilogue applies to its fp32
// accumulator, so the normalised A is never written to or read back from
// memory.  This pass computes r: it reads A once (memory-bound), one warp per
// row, 16-byte coalesced loads, fp32 sums in a fixed order (lane-strided
// partial sums, then a butterfly), so results are deterministic.  HBM latency
// times bandwidth is several MB, so each lane keeps a whole batch of UNROLL
// loads in flight (a 4096-wide row in two batches) and all rows' warps are
// resident at once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tg_launch.cuh"

namespace tg {

constexpr int RMS_WARPS = 8;   // rows in flight per 256-thread block
constexpr int UNROLL = 8;      // 16-byte loads in flight per lane

// Counters of stream-K tiles start at zero in every GEMM launch that uses them.
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
        // batches of UNROLL independent 16-byte loads per lane (vectors v, v + 32, ...),
        // added in that order; a load past the row's end reads zeros, which add nothing
        for (int64_t v = lane; v < kvec; v += 32 * UNROLL) {
            uint4 w[UNROLL];
            if (v + 32 * (UNROLL - 1) < kvec) {
#pragma unroll
                for (int u = 0; u < UNROLL; ++u) w[u] = __ldg(av + v + 32 * u);
            } else {
#pragma unroll
                for (int u = 0; u < UNROLL; ++u)
                    w[u] = v + 32 * u < kvec ? __ldg(av + v + 32 * u) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) add(w[u]);
        }
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

// Per-expert A and C tensor maps of the device-counts MoE GEMM: expert g owns rows
// [off_g, off_g + counts[g]) of A [T, K] and C [T, N], off_g the sum of the counts
// before it.  maps[2 g] is the A template (a map over all T rows) with its base moved
// to row off_g and its row extent cut to counts[g]; maps[2 g + 1] likewise for C.
// Loads of a tile that runs past the expert's rows then read zeros, and its stores
// stop at the expert's last row, as with a separate problem per expert.  One warp:
// prefix sums 32 experts at a time, each lane writing its expert's two maps.
// Experts with no rows, and all experts once the running total passes T (the GEMM
// reports such counts and computes nothing), get no map.
__global__ void __launch_bounds__(32) moe_maps_kernel(const __grid_constant__ CUtensorMap tmpl_a,
                                                      const __grid_constant__ CUtensorMap tmpl_c,
                                                      const int32_t* __restrict__ counts, int G,
                                                      const uint8_t* a_base, int64_t a_row_bytes, uint8_t* c_base,
                                                      int64_t c_row_bytes, int64_t T, CUtensorMap* maps) {
    ptx::grid_launch_dependents();      // the GEMM may start its set-up; it waits before using the maps
    const int lane = threadIdx.x;
    long long off = 0;
    bool bad = false;
    for (int g0 = 0; g0 < G; g0 += 32) {
        const int g = g0 + lane;
        long long c = g < G ? static_cast<long long>(counts[g]) : 0ll;
        bad |= c < 0;
        c = c < 0 ? 0 : c;
        long long incl = c;
        for (int d = 1; d < 32; d <<= 1) {
            const long long x = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += x;
        }
        bad = __any_sync(0xffffffffu, bad);
        const long long first = off + incl - c;
        if (g < G && c > 0 && !bad && first + c <= T) {
            CUtensorMap* ma = maps + 2 * g;
            CUtensorMap* mc = ma + 1;
            const uint4* ta = reinterpret_cast<const uint4*>(&tmpl_a);
            const uint4* tc = reinterpret_cast<const uint4*>(&tmpl_c);
            uint4* da = reinterpret_cast<uint4*>(ma);
            uint4* dc = reinterpret_cast<uint4*>(mc);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                da[i] = ta[i];
                dc[i] = tc[i];
            }
            ptx::tensormap_replace_address(ma, a_base + first * a_row_bytes);
            ptx::tensormap_replace_dim<1>(ma, static_cast<uint32_t>(c));
            ptx::tensormap_replace_address(mc, c_base + first * c_row_bytes);
            ptx::tensormap_replace_dim<1>(mc, static_cast<uint32_t>(c));
        }
        off += __shfl_sync(0xffffffffu, incl, 31);
    }
    ptx::fence_tensormap_release();
}

cudaError_t launch_moe_maps(const CUtensorMap& tmpl_a, const CUtensorMap& tmpl_c, const int32_t* counts, int G,
                            const void* A, int64_t a_row_bytes, void* C, int64_t c_row_bytes, int64_t T,
                            CUtensorMap* maps, cudaStream_t stream) {
    moe_maps_kernel<<<1, 32, 0, stream>>>(tmpl_a, tmpl_c, counts, G, static_cast<const uint8_t*>(A), a_row_bytes,
                                          static_cast<uint8_t*>(C), c_row_bytes, T, maps);
    return cudaGetLastError();
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
