// tg_api.cu - host side of libtg: the C ABI declared in include/tg.h.
//
// Responsibilities: argument checks (before anything is enqueued), TMA tensor
// map encoding (cuTensorMapEncodeTiled, reached through the runtime's driver
// entry-point query so the library does not link libcuda), choice of kernel
// variant and persistent grid size, the stream-K plan of a dense launch (its
// partial-sum workspace and the counter reset before the GEMM), the grouped
// problem table (prefix sums of tile counts, copied into a stream-ordered
// workspace), and the per-device error record written by the kernels' bounded
// waits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "tg.h"
#include "tg_launch.cuh"

// Per-device record of the first in-kernel wait that ran out (zero at module load).
__device__ tg::ErrorRecord g_tg_error;

// Problem table of tg_grouped_gemm_noalloc (see that entry point below).
static __device__ __align__(256) tg::Problem g_noalloc_table[TG_NOALLOC_MAX_PROBLEMS];
static_assert(sizeof(g_noalloc_table) == 128 * 1024, "the header states a 128 KiB table");

namespace {

using tg::Config;
using tg::Params;
using tg::Problem;

constexpr uint32_t kDefaultBudgetMs = 1000;
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

thread_local std::string t_message;
// Test hook armed by tg_debug_withhold_stage(_in): k-block (-1 = off) and block.
struct WithholdArm {
    int64_t kb = -1;
    int32_t block = 0;
};
thread_local WithholdArm t_withhold;
struct TraceArm {
    uint64_t* tiles = nullptr;
    int64_t tiles_cap = 0;
    uint64_t* ctas = nullptr;
    int64_t ctas_cap = 0;
};
thread_local TraceArm t_trace;
thread_local uint64_t t_launches = 0;   // kernels this thread has enqueued (tg_launch_count)

std::atomic<uint32_t> g_budget_ms{0};

tg_status fail(tg_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_message = buf;
    return s;
}

tg_status cuda_fail(cudaError_t e, const char* what) {
    return fail(e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ? TG_ERR_NO_DEVICE : TG_ERR_CUDA,
                "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

uint32_t budget_ms() {
    uint32_t b = g_budget_ms.load();
    if (b == 0) {
        const char* env = std::getenv("TG_WAIT_BUDGET_MS");
        long v = env ? std::strtol(env, nullptr, 10) : 0;
        b = (v > 0 && v < 3600000) ? static_cast<uint32_t>(v) : kDefaultBudgetMs;
    }
    return b;
}

// ----------------------------------------------------------------------------------------
// per-device state

struct DeviceState {
    bool ready = false;
    int dev = 0;
    int cc_major = 0, cc_minor = 0, sms = 0;
    tg::ErrorRecord* err = nullptr;
    cudaMemPool_t pool = nullptr;          // created by the first call that allocates a workspace
    tg::Problem* noalloc_table = nullptr;  // device address of g_noalloc_table, looked up by the first no-alloc call
    int units[128] = {};  // resident work units per kernel variant (0 = not yet queried)
    int moe_units[16] = {};
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Checks and addresses of the current device, once per device: compute
// capability, SM count, and the device address of the error record (in host
// code a __device__ variable's name is only a stand-in for the symbol).
// Allocates nothing.
tg_status device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(TG_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        d.dev = dev;
        if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (d.cc_major != 10 || d.cc_minor != 3)
            return fail(TG_ERR_UNSUPPORTED, "device %d is sm_%d%d; libtg is built for sm_103a (GB300) only", dev,
                        d.cc_major, d.cc_minor);
        void* sym = nullptr;
        if ((e = cudaGetSymbolAddress(&sym, g_tg_error)) != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
        d.err = static_cast<tg::ErrorRecord*>(sym);
        d.ready = true;
    }
    *out = &d;
    return TG_OK;
}

// The library's stream-ordered memory pool on d's device, created by the first
// call that needs a workspace (grouped problem tables, stream-K partial sums).
tg_status device_pool(DeviceState* d, cudaMemPool_t* out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!d->pool) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = d->dev;
        cudaMemPool_t pool = nullptr;
        cudaError_t e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
        uint64_t keep = UINT64_MAX;  // keep freed workspace cached in the pool
        if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)) != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return cuda_fail(e, "cudaMemPoolSetAttribute");
        }
        d->pool = pool;
    }
    *out = d->pool;
    return TG_OK;
}

// ----------------------------------------------------------------------------------------
// tensor maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

tg_status encoder() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    static cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSuccess;
    std::call_once(once, [] {
        void* fn = nullptr;
        err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (err != cudaSuccess) return cuda_fail(err, "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)");
    if (!g_encode) return fail(TG_ERR_CUDA, "driver does not provide cuTensorMapEncodeTiled (query result %d)", int(q));
    return TG_OK;
}

tg_status make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
                   uint64_t ld_bytes, uint32_t box_inner, uint32_t box_outer, const char* what, int g) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {ld_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TG_ERR_UNSUPPORTED, "problem %d: cuTensorMapEncodeTiled(%s) failed with CUresult %d", g, what,
                    int(r));
    return TG_OK;
}

// 3-D map [outer][mid][inner] with strides (in bytes) for the two outer dimensions.
tg_status make_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t mid,
                      uint64_t outer, uint64_t mid_stride, uint64_t outer_stride, uint32_t box_inner,
                      uint32_t box_mid, uint32_t box_outer, const char* what) {
    const cuuint64_t dims[3] = {inner, mid, outer};
    const cuuint64_t strides[2] = {mid_stride, outer_stride};
    const cuuint32_t box[3] = {box_inner, box_mid, box_outer};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TG_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what, int(r));
    return TG_OK;
}

// 4-D map [d3][d2][d1][inner] with strides (in bytes) for the three outer dimensions.
tg_status make_map_4d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, const uint64_t dims_in[4],
                      const uint64_t strides_in[3], const uint32_t box_in[4], const char* what) {
    const cuuint64_t dims[4] = {dims_in[0], dims_in[1], dims_in[2], dims_in[3]};
    const cuuint64_t strides[3] = {strides_in[0], strides_in[1], strides_in[2]};
    const cuuint32_t box[4] = {box_in[0], box_in[1], box_in[2], box_in[3]};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, dt, 4, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TG_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what, int(r));
    return TG_OK;
}

// N-major B whose columns split into whole 64-column chunks can be read through the
// wide view {64 columns, k, chunk}: the chunk stride is 128 bytes, so every element of
// the view lies inside a row's first N columns (a ragged last chunk would not).
bool wide_b_ok(tg_layout lb, int64_t N, int bn_cta) {
    return lb == TG_ROW_MAJOR && N % 64 == 0 && bn_cta >= 128;
}

// ----------------------------------------------------------------------------------------
// argument checks

struct Prob {
    const void* A; tg_layout la; int64_t lda;
    const void* B; tg_layout lb; int64_t ldb;
    void* C; tg_dtype cd; int64_t ldc;
    int64_t M, N, K;
    tg_epilogue epi;
    const void* bias;
    tg_dtype ab;          // element type of A, B and bias: TG_BF16 or TG_F16
    const float* row_scale = nullptr;   // optional per-row factor on the accumulator (RMS norm)
};

Prob prob_of(const tg_group_problem& t) {
    return Prob{t.A, t.layout_a, t.lda, t.B, t.layout_b, t.ldb, t.C, t.c_dtype, t.ldc, t.M, t.N, t.K, t.epi, t.bias,
                t.ab_dtype};
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tg_status check(const Prob& q, int g) {
    if (q.la != TG_ROW_MAJOR && q.la != TG_COL_MAJOR) return fail(TG_ERR_INVALID_ARG, "problem %d: bad layout_a %d", g, int(q.la));
    if (q.lb != TG_ROW_MAJOR && q.lb != TG_COL_MAJOR) return fail(TG_ERR_INVALID_ARG, "problem %d: bad layout_b %d", g, int(q.lb));
    if (q.cd != TG_BF16 && q.cd != TG_F32 && q.cd != TG_F16)
        return fail(TG_ERR_INVALID_ARG, "problem %d: bad c_dtype %d", g, int(q.cd));
    if (q.ab != TG_BF16 && q.ab != TG_F16)
        return fail(TG_ERR_INVALID_ARG, "problem %d: bad ab_dtype %d (A and B are bf16 or fp16)", g, int(q.ab));
    if (q.epi != TG_EPI_NONE && q.epi != TG_EPI_BIAS && q.epi != TG_EPI_BIAS_GELU)
        return fail(TG_ERR_INVALID_ARG, "problem %d: bad epilogue %d", g, int(q.epi));
    if (q.M < 0 || q.N < 0 || q.K < 0)
        return fail(TG_ERR_INVALID_ARG, "problem %d: negative size M=%lld N=%lld K=%lld", g, (long long)q.M,
                    (long long)q.N, (long long)q.K);
    if (q.M > kMaxDim || q.N > kMaxDim || q.K > kMaxDim)
        return fail(TG_ERR_UNSUPPORTED, "problem %d: sizes must be below 2^31", g);
    if (q.M == 0 || q.N == 0) return TG_OK;  // nothing to compute; pointers unused

    if (!q.C) return fail(TG_ERR_INVALID_ARG, "problem %d: C is NULL", g);
    if (q.ldc < q.N) return fail(TG_ERR_INVALID_ARG, "problem %d: ldc=%lld < N=%lld", g, (long long)q.ldc, (long long)q.N);
    if (q.epi != TG_EPI_NONE && !q.bias) return fail(TG_ERR_INVALID_ARG, "problem %d: epilogue needs a bias", g);
    if (q.K > 0) {
        if (!q.A) return fail(TG_ERR_INVALID_ARG, "problem %d: A is NULL", g);
        if (!q.B) return fail(TG_ERR_INVALID_ARG, "problem %d: B is NULL", g);
        const int64_t min_lda = q.la == TG_ROW_MAJOR ? q.K : q.M;
        const int64_t min_ldb = q.lb == TG_ROW_MAJOR ? q.N : q.K;
        if (q.lda < min_lda)
            return fail(TG_ERR_INVALID_ARG, "problem %d: lda=%lld < %lld", g, (long long)q.lda, (long long)min_lda);
        if (q.ldb < min_ldb)
            return fail(TG_ERR_INVALID_ARG, "problem %d: ldb=%lld < %lld", g, (long long)q.ldb, (long long)min_ldb);
        if (q.lda > kMaxDim || q.ldb > kMaxDim) return fail(TG_ERR_UNSUPPORTED, "problem %d: ld must be below 2^31", g);
        if (!aligned16(q.A) || !aligned16(q.B))
            return fail(TG_ERR_UNSUPPORTED, "problem %d: A and B must be 16-byte aligned (TMA)", g);
        if ((q.lda * 2) % 16 || (q.ldb * 2) % 16)
            return fail(TG_ERR_UNSUPPORTED, "problem %d: lda and ldb must be multiples of 8 elements (TMA)", g);
    }
    const int64_t esize = q.cd == TG_F32 ? 4 : 2;
    if (q.ldc > kMaxDim) return fail(TG_ERR_UNSUPPORTED, "problem %d: ldc must be below 2^31", g);
    if (!aligned16(q.C)) return fail(TG_ERR_UNSUPPORTED, "problem %d: C must be 16-byte aligned (TMA)", g);
    if ((q.ldc * esize) % 16) return fail(TG_ERR_UNSUPPORTED, "problem %d: ldc * element size must be a multiple of 16 bytes (TMA)", g);
    if (q.bias && (reinterpret_cast<uintptr_t>(q.bias) & 1u)) return fail(TG_ERR_INVALID_ARG, "problem %d: bias is not 2-byte aligned", g);
    return TG_OK;
}

// ----------------------------------------------------------------------------------------
// kernel variants

using LaunchFn = cudaError_t (*)(const Params&, int, cudaStream_t);
using UnitsFn = cudaError_t (*)(int*);
struct Variant {
    LaunchFn launch;
    UnitsFn units;
    int bn, cta_group, tile_m, cw, bn_cta;
};

template <int BN, int CG, bool AMN, bool BMN, bool F32, int MODE>
constexpr Variant variant() {
    using C = Config<BN, CG, AMN, BMN, F32, MODE>;
    static_assert(C::MOE == (MODE == 2) && C::GROUPED == (MODE == 1), "kernel mode");
    return Variant{&tg::launch<C>, &tg::resident_units<C>, C::BN, C::CTA_GROUP, C::TILE_M, C::CW, C::BN_CTA};
}

#define TG_VARIANT_ENTRY(BN, CG, AMN, BMN, F32, GR) variant<BN, CG, AMN, BMN, F32, GR>(),

const Variant kVariants[] = {
    TG_FOR_EACH_TILE(TG_VARIANT_ENTRY, false, false)
    TG_FOR_EACH_TILE(TG_VARIANT_ENTRY, true, false)
    TG_FOR_EACH_TILE(TG_VARIANT_ENTRY, false, true)
    TG_FOR_EACH_TILE(TG_VARIANT_ENTRY, true, true)
};
constexpr int kTilesPerGroup = 16;
constexpr int kNumVariants = 4 * kTilesPerGroup;
static_assert(sizeof(kVariants) / sizeof(kVariants[0]) == kNumVariants, "variant table");

const Variant kMoeVariants[] = {
    TG_FOR_EACH_MOE_TILE(TG_VARIANT_ENTRY, false)
    TG_FOR_EACH_MOE_TILE(TG_VARIANT_ENTRY, true)
};
static_assert(sizeof(kMoeVariants) / sizeof(kMoeVariants[0]) == 16, "MoE variant table");
static_assert(TG_MOE_MAX_EXPERTS == tg::MOE_MAX_G, "header and kernel agree on the expert limit");

int moe_variant_index(bool f32, int cta_group, int bn, bool bmn) {
    return (f32 ? 8 : 0) + (cta_group == 2 ? 4 : 0) + (bn == 256 ? 2 : 0) + (bmn ? 1 : 0);
}

int variant_index(bool grouped, bool f32, int cta_group, int bn, bool amn, bool bmn) {
    const int tile = (cta_group == 2 ? 8 : 0) + (bn == 256 ? 4 : 0) + (amn ? 2 : 0) + (bmn ? 1 : 0);
    return ((grouped ? 2 : 0) + (f32 ? 1 : 0)) * kTilesPerGroup + tile;
}

tg_status resident(DeviceState* d, int vi, int* units) {
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (d->units[vi] > 0) { *units = d->units[vi]; return TG_OK; }
    }
    int u = 0;
    cudaError_t e = kVariants[vi].units(&u);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (u <= 0) return fail(TG_ERR_UNSUPPORTED, "kernel variant %d cannot be resident on this device", vi);
    std::lock_guard<std::mutex> lock(g_mu);
    d->units[vi] = u;
    *units = u;
    return TG_OK;
}

struct TileChoice {
    int cta_group;
    int bn;
};

// Tile shape of a launch.  BN = 256 unless every problem is at most 128 wide;
// CTA pairs (256-row tiles, half the operand traffic per SM) unless the rows
// are so few that 128-row tiles keep more SMs busy.  TG_TILE=<cta_group>x<bn>
// (e.g. "2x256") overrides the choice for tuning sweeps.
TileChoice pick_tile(int64_t rows, int64_t max_n, int sms) {
    TileChoice t;
    t.bn = max_n > 128 ? 256 : 128;
    const int64_t tiles_n = (max_n + t.bn - 1) / t.bn;
    const int64_t pair_tiles = ((rows + 255) / 256) * tiles_n;
    t.cta_group = (pair_tiles * 2 >= sms) ? 2 : 1;
    if (const char* env = std::getenv("TG_TILE")) {
        int cg = 0, bn = 0;
        if (std::sscanf(env, "%dx%d", &cg, &bn) == 2 && (cg == 1 || cg == 2) && (bn == 128 || bn == 256)) {
            t.cta_group = cg;
            t.bn = bn;
        }
    }
    return t;
}

// Raster band (N-tiles swept before stepping along M).  The tiles that run at
// once cover about units / band M-tiles of `band` N-tiles, a square-ish
// footprint, so A rows and B columns are shared in L2 (band 4 for 76 pairs).
// When A and B together do not fit in L2, A is read from DRAM once per band:
// the band then widens while its B panels (bn columns x K each) take at most
// kBandL2Bytes, so that they stay in L2 while A streams past and A is read
// tiles_n / band times.  TG_BAND=<n> overrides the choice (tuning sweeps).
constexpr int64_t kBandL2Bytes = int64_t(32) << 20;
constexpr int64_t kOperandsInL2 = int64_t(96) << 20;

int pick_band(int64_t tiles_n, int units, int bn, int64_t K, int64_t rows) {
    int band = 1;
    while (band * band * 2 <= units && band < 16) band *= 2;
    const int64_t panel = static_cast<int64_t>(bn) * K * 2;
    if ((rows + tiles_n * bn) * K * 2 > kOperandsInL2)
        while (band < 16 && 2 * band * panel <= kBandL2Bytes && 2 * band <= tiles_n) band *= 2;
    if (const char* env = std::getenv("TG_BAND")) {
        const long b = std::strtol(env, nullptr, 10);
        if (b >= 1 && b <= 64) band = static_cast<int>(b);
    }
    if (band > tiles_n) band = static_cast<int>(tiles_n);
    return band < 1 ? 1 : band;
}

tg_status fill_problem(const Prob& q, const Variant& v, int g, Problem* out) {
    std::memset(out, 0, sizeof(Problem));
    const bool ab_f16 = q.ab == TG_F16;
    const CUtensorMapDataType bf16 = ab_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    tg_status s;
    if (q.K > 0) {
        if (q.la == TG_ROW_MAJOR)
            s = make_map(&out->tma_a, bf16, q.A, q.K, q.M, q.lda * 2, 64, tg::BM, "A", g);
        else
            s = make_map(&out->tma_a, bf16, q.A, q.M, q.K, q.lda * 2, 64, 64, "A", g);
        if (s != TG_OK) return s;
        if (wide_b_ok(q.lb, q.N, v.bn_cta)) {
            // one box per k-block: {64 columns, 64 k, the CTA's BN_CTA / 64 chunks}
            s = make_map_3d(&out->tma_b, bf16, q.B, 64, q.K, q.N / 64, q.ldb * 2, 128, 64, 64, v.bn_cta / 64,
                            "B (64-column chunks)");
            out->flags |= tg::FLAG_B_WIDE;
        } else if (q.lb == TG_ROW_MAJOR)
            s = make_map(&out->tma_b, bf16, q.B, q.N, q.K, q.ldb * 2, 64, 64, "B", g);
        else
            s = make_map(&out->tma_b, bf16, q.B, q.K, q.N, q.ldb * 2, 64, v.bn_cta, "B", g);
        if (s != TG_OK) return s;
    }
    const bool f32 = q.cd == TG_F32;
    const CUtensorMapDataType c_type = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : (q.cd == TG_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    s = make_map(&out->tma_c, c_type, q.C, q.N, q.M, q.ldc * (f32 ? 4 : 2), v.cw, 32, "C", g);
    if (s != TG_OK) return s;
    out->bias = q.epi != TG_EPI_NONE ? q.bias : nullptr;
    out->row_scale = q.row_scale;
    out->idesc = tg::ptx::idesc_f32_acc(v.tile_m, v.bn, q.la == TG_COL_MAJOR, q.lb == TG_ROW_MAJOR, ab_f16);
    out->flags |= (q.cd == TG_F16 ? tg::FLAG_C_F16 : 0u) | (ab_f16 ? tg::FLAG_BIAS_F16 : 0u);
    out->M = static_cast<int32_t>(q.M);
    out->N = static_cast<int32_t>(q.N);
    out->K = static_cast<int32_t>(q.K);
    out->epi = static_cast<int32_t>(q.epi);
    out->tiles_m = static_cast<int32_t>((q.M + v.tile_m - 1) / v.tile_m);
    out->tiles_n = static_cast<int32_t>((q.N + v.bn - 1) / v.bn);
    out->k_blocks = static_cast<int32_t>((q.K + tg::BK - 1) / tg::BK);
    out->repeat = 0;
    out->replicas = 1;
    return TG_OK;
}

// Launch-wide fields every launch carries: the error record, the wait budget,
// and the test and trace hooks armed on this thread (consumed by this launch).
void base_params(Params* p, tg::ErrorRecord* err) {
    p->err = err;
    p->wait_budget_ns = static_cast<uint64_t>(budget_ms()) * 1000000ull;
    p->withhold_kb = t_withhold.kb;
    p->withhold_block = t_withhold.block;
    t_withhold = WithholdArm{};
    p->trace_tiles = t_trace.tiles;
    p->trace_tiles_cap = t_trace.tiles_cap;
    p->trace_ctas = t_trace.ctas;
    p->trace_ctas_cap = t_trace.ctas_cap;
    t_trace = TraceArm{};
}

// Launch with one CTA (pair) per work unit that has work: every resident unit,
// or fewer when there are fewer whole tiles plus stream-K ranges than units.
tg_status enqueue(const Params& p, const Variant& v, int units, cudaStream_t stream) {
    int64_t want = p.total_tiles + p.nh_tiles - p.sk_tiles;
    if (p.sk_units > want) want = p.sk_units;
    if (want > units) want = units;
    const int grid = static_cast<int>(want) * v.cta_group;
    cudaError_t e = v.launch(p, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    ++t_launches;
    return TG_OK;
}

}  // namespace

// ----------------------------------------------------------------------------------------
// Grouped GEMM that allocates nothing (tg_grouped_gemm_noalloc).
//
// Some callers may not allocate device memory once they are running: a
// serving loop that pre-reserves everything at start-up so that no request can
// fail or stall on an allocation, or an application whose device memory is
// owned by its own allocator under a fixed budget.  tg_grouped_gemm allocates a
// small stream-ordered workspace per call for the problem table; this entry
// point keeps the table in g_noalloc_table instead.  The array lives in the
// library's device image, so every GPU that loads libtg holds it (128 KiB)
// until the process exits.  All calls share it: a call overwrites the entries
// it uses, and a kernel reads only the entries its own call wrote, so nothing
// has to start at zero; two calls whose copies and kernels overlap on the GPU
// (different streams, no ordering between them) race on it.

namespace {

// The device address of g_noalloc_table on d's device, looked up once per
// device by the first no-alloc call (with that device current).  In host code
// the array's name is only a stand-in for the symbol: a kernel given it would
// read the wrong memory, so its address comes from cudaGetSymbolAddress.
tg_status noalloc_table(DeviceState* d, tg::Problem** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!d->noalloc_table) {
        tg::Problem* tab = nullptr;
        cudaError_t e = cudaGetSymbolAddress((void**)&tab, g_noalloc_table);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc problem table)");
        d->noalloc_table = tab;
    }
    *out = d->noalloc_table;
    return TG_OK;
}

// Host staging for one call's table: fixed per-thread storage, no heap.  The
// next no-alloc call on the thread overwrites it.
thread_local tg::Problem t_noalloc_host[TG_NOALLOC_MAX_PROBLEMS];

}  // namespace

namespace {
// Row statistics launched just before a dense GEMM (the fused RMS normalisation).
struct RowPass {
    const void* A;
    int64_t lda, M, K;
    float eps;
    float* r;
};

tg_status check_row_rms(const void* A, int64_t lda, int64_t M, int64_t K, float eps, const float* r) {
    if (M < 0 || K < 0) return fail(TG_ERR_INVALID_ARG, "negative size M=%lld K=%lld", (long long)M, (long long)K);
    if (M == 0) return TG_OK;
    if (!r) return fail(TG_ERR_INVALID_ARG, "r is NULL");
    if (!(eps >= 0.0f)) return fail(TG_ERR_INVALID_ARG, "eps must be a non-negative number");
    if (K > 0) {
        if (!A) return fail(TG_ERR_INVALID_ARG, "A is NULL");
        if (lda < K) return fail(TG_ERR_INVALID_ARG, "lda=%lld < K=%lld", (long long)lda, (long long)K);
        if (!aligned16(A) || (lda * 2) % 16)
            return fail(TG_ERR_UNSUPPORTED, "A must be 16-byte aligned with lda a multiple of 8");
    }
    if (reinterpret_cast<uintptr_t>(r) & 3u) return fail(TG_ERR_INVALID_ARG, "r is not 4-byte aligned");
    return TG_OK;
}

tg_status dense_gemm(const Prob& q, tg_stream_t stream, const RowPass* pre = nullptr);
}  // namespace

// ========================================================================================
// C ABI

extern "C" {

tg_status tg_gemm(const void* A, tg_layout layout_a, int64_t lda, const void* B, tg_layout layout_b, int64_t ldb,
                  void* C, tg_dtype c_dtype, int64_t ldc, int64_t M, int64_t N, int64_t K, tg_epilogue epi,
                  const void* bias, tg_stream_t stream) {
    return dense_gemm(Prob{A, layout_a, lda, B, layout_b, ldb, C, c_dtype, ldc, M, N, K, epi, bias, TG_BF16}, stream);
}

tg_status tg_row_rms(const void* A, int64_t lda, int64_t M, int64_t K, float eps, float* r, tg_stream_t stream) {
    tg_status s = check_row_rms(A, lda, M, K, eps, r);
    if (s != TG_OK || M == 0) return s;
    DeviceState* d = nullptr;
    if ((s = device_state(&d)) != TG_OK) return s;
    cudaError_t e = tg::launch_row_rms(A, lda, M, K, eps, r, d->sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "row statistics launch");
    ++t_launches;
    return TG_OK;
}

tg_status tg_gemm_rmsnorm(const void* A, int64_t lda, const void* B, tg_layout layout_b, int64_t ldb, void* C,
                          tg_dtype c_dtype, int64_t ldc, int64_t M, int64_t N, int64_t K, float eps, float* row_scale,
                          tg_epilogue epi, const void* bias, tg_stream_t stream) {
    Prob q{A, TG_ROW_MAJOR, lda, B, layout_b, ldb, C, c_dtype, ldc, M, N, K, epi, bias, TG_BF16};
    tg_status s = check(q, 0);
    if (s != TG_OK) return s;
    if (M == 0 || N == 0) return TG_OK;
    if (!row_scale) return fail(TG_ERR_INVALID_ARG, "row_scale is NULL");
    if ((s = check_row_rms(A, lda, M, K, eps, row_scale)) != TG_OK) return s;
    // with K == 0 the product is 0 whatever r is (r may be infinite when eps == 0): no scale
    q.row_scale = K > 0 ? row_scale : nullptr;
    const RowPass pre{A, lda, M, K, eps, row_scale};
    return dense_gemm(q, stream, &pre);
}

tg_status tg_gemm_ex(const tg_group_problem* problem, tg_stream_t stream) {
    if (!problem) return fail(TG_ERR_INVALID_ARG, "problem is NULL");
    return dense_gemm(prob_of(*problem), stream);
}

}  // extern "C"

namespace {

// The last, partial wave of a dense launch.  With T tiles on U units, its
// R = T mod U tiles would leave U - R units idle.  Short tiles (at most
// kHalvesMaxKb k-blocks) of 256 columns, when 2R <= U, run as 2R column halves:
// a half costs 3/4 of a whole tile's operand bytes (the A box and half of B) and
// needs no partial sums.  Longer tiles are balanced with stream-K (tg::sk_plan),
// whose partial sums cost relatively less.  TG_STREAM_K=0 turns both off (one
// unit per tile, as grouped launches); TG_STREAM_K=1 uses stream-K wherever its
// plan applies.
constexpr int kHalvesMaxKb = 96;

struct WavePlan {
    int64_t halves = 0;   // tiles run as column halves
    tg::SkPlan sk;
};

WavePlan plan_last_wave(int64_t tiles, int units, int k_blocks, int bn) {
    WavePlan wp;
    const char* env = std::getenv("TG_STREAM_K");
    if (env && env[0] == '0') return wp;
    const bool force_sk = env && env[0] == '1';
    const int64_t R = units > 0 ? tiles % units : 0;
    if (!force_sk && bn == 256 && tiles > units && R > 0 && 2 * R <= units && k_blocks <= kHalvesMaxKb) {
        wp.halves = R;
        return wp;
    }
    wp.sk = tg::sk_plan(tiles, units, k_blocks);
    return wp;
}

tg_status dense_gemm(const Prob& q, tg_stream_t stream, const RowPass* pre) {
    const tg_layout layout_a = q.la, layout_b = q.lb;
    const tg_dtype c_dtype = q.cd;
    const int64_t M = q.M, N = q.N;
    tg_status s = check(q, 0);
    if (s != TG_OK) return s;
    if (M == 0 || N == 0) return TG_OK;
    DeviceState* d = nullptr;
    if ((s = device_state(&d)) != TG_OK) return s;
    if ((s = encoder()) != TG_OK) return s;

    const TileChoice tc = pick_tile(M, N, d->sms);
    const int vi = variant_index(false, c_dtype == TG_F32, tc.cta_group, tc.bn, layout_a == TG_COL_MAJOR,
                                 layout_b == TG_ROW_MAJOR);
    const Variant& v = kVariants[vi];
    int units = 0;
    if ((s = resident(d, vi, &units)) != TG_OK) return s;

    Params p;
    std::memset(&p, 0, sizeof p);
    if ((s = fill_problem(q, v, 0, &p.dense)) != TG_OK) return s;
    p.dense.tile_begin = 0;
    p.problems = nullptr;
    p.num_problems = 1;
    const int64_t tiles = static_cast<int64_t>(p.dense.tiles_m) * p.dense.tiles_n;
    p.total_tiles = tiles;
    p.band = pick_band(p.dense.tiles_n, units, v.bn, q.K, q.M);
    base_params(&p, d->err);

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const WavePlan wp = plan_last_wave(tiles, units, p.dense.k_blocks, v.bn);
    const tg::SkPlan& sp = wp.sk;
    if (wp.halves > 0) {
        p.nh_tiles = static_cast<int32_t>(wp.halves);
        const CUtensorMapDataType bt =
            q.ab == TG_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        if (layout_b == TG_COL_MAJOR) {
            // K-major B: a second map whose box covers the half of each CTA's N rows
            if ((s = make_map(&p.b_half, bt, q.B, q.K, q.N, q.ldb * 2, 64, v.bn_cta / 2, "B (column halves)", 0)) !=
                TG_OK)
                return s;
        } else if (p.dense.flags & tg::FLAG_B_WIDE) {
            // N-major B through the wide view: halves load 64-column boxes of the plain map
            if ((s = make_map(&p.b_half, bt, q.B, q.N, q.K, q.ldb * 2, 64, 64, "B (column halves)", 0)) != TG_OK)
                return s;
        }
    }
    void* ws = nullptr;
    int n_counters = 0;
    if (sp.tiles > 0) {
        // partial sums of every piece, then one arrival counter per (tile, CTA, epilogue warp)
        // and one ready flag per (tile, piece, CTA, epilogue warp), all zeroed before the GEMM
        const size_t partial =
            static_cast<size_t>(sp.tiles) * sp.max_slices * v.tile_m * v.bn * sizeof(float);
        const int n_count = sp.tiles * v.cta_group * tg::NUM_EPI_WARPS;
        n_counters = n_count * (1 + sp.max_slices);
        cudaMemPool_t pool = nullptr;
        if ((s = device_pool(d, &pool)) != TG_OK) return s;
        cudaError_t e = cudaMallocFromPoolAsync(&ws, partial + n_counters * sizeof(uint32_t), pool, st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync(stream-K partials)");
        p.sk_tiles = sp.tiles;
        p.sk_units = sp.units;
        p.sk_max_slices = sp.max_slices;
        p.sk_partial = static_cast<float*>(ws);
        p.sk_count = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + partial);
        p.sk_flag = p.sk_count + n_count;
    }
    // the kernel before the GEMM: the row pass (which also zeroes the counters) or the counter reset;
    // the GEMM follows it as a programmatic dependent and waits for it only where it reads its output
    cudaError_t e = cudaSuccess;
    if (pre) e = tg::launch_row_rms(pre->A, pre->lda, pre->M, pre->K, pre->eps, pre->r, d->sms, st, p.sk_count,
                                    n_counters);
    else if (n_counters) e = tg::launch_clear_counters(p.sk_count, n_counters, st);
    s = e == cudaSuccess ? TG_OK : cuda_fail(e, pre ? "row statistics launch" : "counter reset launch");
    if (s == TG_OK && (pre || n_counters)) ++t_launches;
    p.pdl = (pre != nullptr || n_counters > 0) ? 1 : 0;
    if (s == TG_OK) s = enqueue(p, v, units, st);
    if (ws) {
        e = cudaFreeAsync(ws, st);   // stream-ordered: released after the GEMM has run
        if (e != cudaSuccess && s == TG_OK) s = cuda_fail(e, "cudaFreeAsync(stream-K partials)");
    }
    return s;
}

}  // namespace

extern "C" {

tg_status tg_gemm_bcast(const void* A_user, tg_layout layout_a, int64_t lda, int64_t U, int64_t repeat,
                        const void* B, tg_layout layout_b, int64_t ldb, void* C, tg_dtype c_dtype, int64_t ldc,
                        int64_t N, int64_t K, tg_epilogue epi, const void* bias, tg_stream_t stream) {
    if (repeat < 1) return fail(TG_ERR_INVALID_ARG, "repeat=%lld must be at least 1", (long long)repeat);
    if (U < 0) return fail(TG_ERR_INVALID_ARG, "negative U=%lld", (long long)U);
    if (U > 0 && repeat > kMaxDim / U)
        return fail(TG_ERR_UNSUPPORTED, "U * repeat must be below 2^31 (U=%lld, repeat=%lld)", (long long)U,
                    (long long)repeat);
    const Prob q{A_user, layout_a, lda, B, layout_b, ldb, C, c_dtype, ldc, U, N, K, epi, bias, TG_BF16};
    tg_status s = check(q, 0);
    if (s != TG_OK) return s;
    if (U == 0 || N == 0) return TG_OK;
    DeviceState* d = nullptr;
    if ((s = device_state(&d)) != TG_OK) return s;
    if ((s = encoder()) != TG_OK) return s;

    // Single-CTA tiles over the user rows; the broadcast store is what costs, so
    // each tile is recomputed by `replicas` CTAs that split its repeat indices.
    TileChoice tc = pick_tile(U, N, d->sms);
    tc.cta_group = 1;
    const int vi = variant_index(false, c_dtype == TG_F32, 1, tc.bn, layout_a == TG_COL_MAJOR, layout_b == TG_ROW_MAJOR);
    const Variant& v = kVariants[vi];
    int units = 0;
    if ((s = resident(d, vi, &units)) != TG_OK) return s;

    Params p;
    std::memset(&p, 0, sizeof p);
    if ((s = fill_problem(q, v, 0, &p.dense)) != TG_OK) return s;
    const bool f32 = c_dtype == TG_F32;
    const uint64_t row = static_cast<uint64_t>(ldc) * (f32 ? 4 : 2);
    if ((s = make_map_3d(&p.dense.tma_c, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                             : (c_dtype == TG_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                  : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16), C,
                         N, repeat, U, row, row * repeat, v.cw, 1, 32, "C (broadcast view)")) != TG_OK)
        return s;
    const int64_t tiles = static_cast<int64_t>(p.dense.tiles_m) * p.dense.tiles_n;
    int64_t replicas = units / tiles;
    if (replicas < 1) replicas = 1;
    if (replicas > repeat) replicas = repeat;
    p.dense.repeat = static_cast<int32_t>(repeat);
    p.dense.replicas = static_cast<int32_t>(replicas);
    p.dense.tile_begin = 0;
    p.num_problems = 1;
    p.total_tiles = tiles * replicas;
    p.band = pick_band(p.dense.tiles_n, units, v.bn, K, U);
    base_params(&p, d->err);
    return enqueue(p, v, units, reinterpret_cast<cudaStream_t>(stream));
}

tg_status tg_moe_gemm(const void* A, int64_t lda, int64_t T, int64_t K, const void* B, tg_layout layout_b,
                      int64_t ldb, int64_t expert_stride, int64_t G, int64_t N, void* C, tg_dtype c_dtype,
                      int64_t ldc, const int32_t* counts, tg_epilogue epi, const void* bias, tg_stream_t stream) {
    if (T < 0 || K < 0 || N < 0 || G < 0)
        return fail(TG_ERR_INVALID_ARG, "negative size T=%lld K=%lld N=%lld G=%lld", (long long)T, (long long)K,
                    (long long)N, (long long)G);
    if (T == 0 || N == 0 || G == 0) return TG_OK;
    if (G > TG_MOE_MAX_EXPERTS)
        return fail(TG_ERR_UNSUPPORTED, "G=%lld experts; the device-counts form takes at most %d", (long long)G,
                    TG_MOE_MAX_EXPERTS);
    if (!counts) return fail(TG_ERR_INVALID_ARG, "counts is NULL");
    if (reinterpret_cast<uintptr_t>(counts) & 3u) return fail(TG_ERR_INVALID_ARG, "counts is not 4-byte aligned");
    const Prob q{A, TG_ROW_MAJOR, lda, B, layout_b, ldb, C, c_dtype, ldc, T, N, K, epi, bias, TG_BF16};
    tg_status s = check(q, 0);
    if (s != TG_OK) return s;
    if (K > 0) {
        const int64_t min_stride = (layout_b == TG_ROW_MAJOR ? K : N) * ldb;
        if (expert_stride < min_stride)
            return fail(TG_ERR_INVALID_ARG, "expert_stride=%lld < %lld (one expert's B)", (long long)expert_stride,
                        (long long)min_stride);
        if ((expert_stride * 2) % 16 || expert_stride > (int64_t(1) << 38))
            return fail(TG_ERR_UNSUPPORTED, "expert_stride must be a multiple of 8 elements below 2^38 (TMA)");
    }
    DeviceState* d = nullptr;
    if ((s = device_state(&d)) != TG_OK) return s;
    if ((s = encoder()) != TG_OK) return s;

    const TileChoice tc = pick_tile(T, N, d->sms);
    const int vi = moe_variant_index(c_dtype == TG_F32, tc.cta_group, tc.bn, layout_b == TG_ROW_MAJOR);
    const Variant& v = kMoeVariants[vi];
    int units = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        units = d->moe_units[vi];
    }
    if (units <= 0) {
        cudaError_t e = v.units(&units);
        if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
        if (units <= 0) return fail(TG_ERR_UNSUPPORTED, "MoE kernel variant %d cannot be resident", vi);
        std::lock_guard<std::mutex> lock(g_mu);
        d->moe_units[vi] = units;
    }

    Params p;
    std::memset(&p, 0, sizeof p);
    if ((s = fill_problem(q, v, 0, &p.dense)) != TG_OK) return s;
    if (K > 0) {
        // B as one 3-D tensor: expert g is the outermost coordinate
        p.dense.flags &= ~tg::FLAG_B_WIDE;
        if (wide_b_ok(layout_b, N, v.bn_cta)) {
            const uint64_t dims[4] = {64, static_cast<uint64_t>(K), static_cast<uint64_t>(N / 64),
                                      static_cast<uint64_t>(G)};
            const uint64_t strides[3] = {static_cast<uint64_t>(ldb) * 2, 128, static_cast<uint64_t>(expert_stride) * 2};
            const uint32_t box[4] = {64, 64, static_cast<uint32_t>(v.bn_cta / 64), 1};
            s = make_map_4d(&p.dense.tma_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, dims, strides, box,
                            "B (experts, 64-column chunks)");
            p.dense.flags |= tg::FLAG_B_WIDE;
        } else if (layout_b == TG_ROW_MAJOR)
            s = make_map_3d(&p.dense.tma_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, N, K, G, ldb * 2, expert_stride * 2,
                            64, 64, 1, "B (experts)");
        else
            s = make_map_3d(&p.dense.tma_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, K, N, G, ldb * 2, expert_stride * 2,
                            64, v.bn_cta, 1, "B (experts)");
        if (s != TG_OK) return s;
    }
    p.num_problems = 1;
    p.total_tiles = 0;   // the kernel derives it from the device counts
    p.band = pick_band(p.dense.tiles_n, units, v.bn, 0, 0);
    p.moe_counts = counts;
    p.moe_groups = static_cast<int32_t>(G);
    p.moe_rows = T;
    base_params(&p, d->err);

    // Each expert's own A and C maps, written on the device from the counts by a small
    // kernel that the GEMM follows as a programmatic dependent (stream-ordered workspace).
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaMemPool_t pool = nullptr;
    if ((s = device_pool(d, &pool)) != TG_OK) return s;
    void* ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, static_cast<size_t>(2 * G) * sizeof(CUtensorMap), pool, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync(per-expert tensor maps)");
    p.moe_maps = static_cast<const CUtensorMap*>(ws);
    const int64_t c_esize = c_dtype == TG_F32 ? 4 : 2;
    e = tg::launch_moe_maps(p.dense.tma_a, p.dense.tma_c, counts, static_cast<int>(G), A, lda * 2, C, ldc * c_esize, T,
                            static_cast<CUtensorMap*>(ws), st);
    s = e == cudaSuccess ? TG_OK : cuda_fail(e, "per-expert tensor map launch");
    if (s == TG_OK) {
        ++t_launches;
        p.pdl = 1;
        const int grid = units * v.cta_group;
        e = v.launch(p, grid, st);
        if (e != cudaSuccess) s = cuda_fail(e, "kernel launch");
        else ++t_launches;
    }
    e = cudaFreeAsync(ws, st);   // stream-ordered: released after the GEMM has run
    if (e != cudaSuccess && s == TG_OK) s = cuda_fail(e, "cudaFreeAsync(per-expert tensor maps)");
    return s;
}

tg_status tg_grouped_gemm(const tg_group_problem* table, int G, tg_stream_t stream) {
    if (G < 0 || G > 65536) return fail(TG_ERR_INVALID_ARG, "G=%d out of range [0, 65536]", G);
    if (G == 0) return TG_OK;
    if (!table) return fail(TG_ERR_INVALID_ARG, "problem table is NULL");
    std::vector<Prob> qs(G);
    bool any = false;
    for (int g = 0; g < G; ++g) {
        const tg_group_problem& t = table[g];
        qs[g] = prob_of(t);
        tg_status s = check(qs[g], g);
        if (s != TG_OK) return s;
        any = any || (t.M > 0 && t.N > 0);
    }
    if (!any) return TG_OK;
    DeviceState* d = nullptr;
    tg_status s;
    if ((s = device_state(&d)) != TG_OK) return s;
    if ((s = encoder()) != TG_OK) return s;
    cudaMemPool_t pool = nullptr;
    if ((s = device_pool(d, &pool)) != TG_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    // One launch per (layout_a, layout_b, c_dtype) class, classes in order of first appearance.
    std::vector<std::tuple<int, int, int>> order;
    std::map<std::tuple<int, int, int>, std::vector<int>> classes;
    for (int g = 0; g < G; ++g) {
        if (qs[g].M == 0 || qs[g].N == 0) continue;
        auto key = std::make_tuple(int(qs[g].la), int(qs[g].lb), int(qs[g].cd));
        auto it = classes.find(key);
        if (it == classes.end()) { order.push_back(key); classes[key] = {g}; }
        else it->second.push_back(g);
    }
    const WithholdArm withhold = t_withhold;
    for (const auto& key : order) {
        const std::vector<int>& members = classes[key];
        int64_t max_n = 0, rows = 0;
        for (int g : members) {
            max_n = qs[g].N > max_n ? qs[g].N : max_n;
            rows += qs[g].M;
        }
        const TileChoice tc = pick_tile(rows, max_n, d->sms);
        const int vi = variant_index(true, std::get<2>(key) == TG_F32, tc.cta_group, tc.bn,
                                     std::get<0>(key) == TG_COL_MAJOR, std::get<1>(key) == TG_ROW_MAJOR);
        const Variant& v = kVariants[vi];
        int units = 0;
        if ((s = resident(d, vi, &units)) != TG_OK) return s;

        std::vector<Problem> host(members.size());
        int64_t tiles = 0, max_tiles_n = 1;
        for (size_t i = 0; i < members.size(); ++i) {
            if ((s = fill_problem(qs[members[i]], v, members[i], &host[i])) != TG_OK) return s;
            host[i].tile_begin = tiles;
            tiles += static_cast<int64_t>(host[i].tiles_m) * host[i].tiles_n;
            if (host[i].tiles_n > max_tiles_n) max_tiles_n = host[i].tiles_n;
        }
        const size_t bytes = host.size() * sizeof(Problem);
        void* ws = nullptr;
        cudaError_t e = cudaMallocFromPoolAsync(&ws, bytes, pool, st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync(problem table)");
        e = cudaMemcpyAsync(ws, host.data(), bytes, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) {
            cudaFreeAsync(ws, st);
            return cuda_fail(e, "cudaMemcpyAsync(problem table)");
        }
        Params p;
        std::memset(&p, 0, sizeof p);
        p.problems = static_cast<const Problem*>(ws);
        p.num_problems = static_cast<int32_t>(host.size());
        p.total_tiles = tiles;
        p.band = pick_band(max_tiles_n, units, v.bn, 0, 0);
        t_withhold = withhold;
        base_params(&p, d->err);
        s = enqueue(p, v, units, st);
        e = cudaFreeAsync(ws, st);
        if (s != TG_OK) return s;
        if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(problem table)");
    }
    t_withhold = WithholdArm{};
    return TG_OK;
}

tg_status tg_grouped_gemm_noalloc(const tg_group_problem* table, int G, tg_stream_t stream) {
    if (G < 0 || G > 65536) return fail(TG_ERR_INVALID_ARG, "G=%d out of range [0, 65536]", G);
    if (G == 0) return TG_OK;
    if (!table) return fail(TG_ERR_INVALID_ARG, "problem table is NULL");
    int live = 0;
    for (int g = 0; g < G; ++g) {
        const tg_group_problem& t = table[g];
        const Prob q = prob_of(t);
        tg_status s = check(q, g);
        if (s != TG_OK) return s;
        live += (t.M > 0 && t.N > 0) ? 1 : 0;
    }
    if (live == 0) return TG_OK;
    if (live > TG_NOALLOC_MAX_PROBLEMS)
        return fail(TG_ERR_UNSUPPORTED,
                    "%d non-empty problems, but the fixed no-alloc table holds at most %d; split the call or use "
                    "tg_grouped_gemm", live, TG_NOALLOC_MAX_PROBLEMS);
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // The descriptors travel from t_noalloc_host, which the thread's next call
    // overwrites: a captured copy would read it again at replay, so a stream
    // under capture is refused before anything is enqueued.
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    cudaError_t ce = cudaStreamIsCapturing(st, &capturing);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamIsCapturing");
    if (capturing != cudaStreamCaptureStatusNone)
        return fail(TG_ERR_UNSUPPORTED,
                    "tg_grouped_gemm_noalloc does not run on a stream that is being captured (its descriptor copy "
                    "reads a host buffer that the next call overwrites)");
    DeviceState* d = nullptr;
    tg_status s;
    if ((s = device_state(&d)) != TG_OK) return s;
    tg::Problem* dev_table = nullptr;
    if ((s = noalloc_table(d, &dev_table)) != TG_OK) return s;
    if ((s = encoder()) != TG_OK) return s;

    // Classes (layout_a, layout_b, c_dtype) in order of first appearance; each
    // class gets its own consecutive slice of the table and its own launch.
    auto class_of = [](const tg_group_problem& t) {
        return (t.layout_a == TG_COL_MAJOR ? 4 : 0) + (t.layout_b == TG_COL_MAJOR ? 2 : 0) +
               (t.c_dtype == TG_F32 ? 1 : 0);
    };
    int class_order[8], n_classes = 0;
    for (int g = 0; g < G; ++g) {
        const tg_group_problem& t = table[g];
        if (t.M == 0 || t.N == 0) continue;
        const int key = class_of(t);
        bool seen = false;
        for (int c = 0; c < n_classes; ++c) seen = seen || class_order[c] == key;
        if (!seen) class_order[n_classes++] = key;
    }
    const WithholdArm withhold = t_withhold;
    int offset = 0;
    for (int c = 0; c < n_classes; ++c) {
        const int key = class_order[c];
        const bool a_col = key & 4, b_col = key & 2, f32 = key & 1;
        int64_t max_n = 0, rows = 0;
        for (int g = 0; g < G; ++g) {
            const tg_group_problem& t = table[g];
            if (t.M == 0 || t.N == 0 || class_of(t) != key) continue;
            max_n = t.N > max_n ? t.N : max_n;
            rows += t.M;
        }
        const TileChoice tc = pick_tile(rows, max_n, d->sms);
        const int vi = variant_index(true, f32, tc.cta_group, tc.bn, a_col, !b_col);
        const Variant& v = kVariants[vi];
        int units = 0;
        if ((s = resident(d, vi, &units)) != TG_OK) return s;

        tg::Problem* host = t_noalloc_host + offset;
        int n = 0;
        int64_t tiles = 0, max_tiles_n = 1;
        for (int g = 0; g < G; ++g) {
            const tg_group_problem& t = table[g];
            if (t.M == 0 || t.N == 0 || class_of(t) != key) continue;
            const Prob q = prob_of(t);
            if ((s = fill_problem(q, v, g, &host[n])) != TG_OK) return s;
            host[n].tile_begin = tiles;
            tiles += static_cast<int64_t>(host[n].tiles_m) * host[n].tiles_n;
            if (host[n].tiles_n > max_tiles_n) max_tiles_n = host[n].tiles_n;
            ++n;
        }
        cudaError_t e = cudaMemcpyAsync(dev_table + offset, host, n * sizeof(tg::Problem), cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(no-alloc problem table)");
        Params p;
        std::memset(&p, 0, sizeof p);
        p.problems = dev_table + offset;
        p.num_problems = n;
        p.total_tiles = tiles;
        p.band = pick_band(max_tiles_n, units, v.bn, 0, 0);
        t_withhold = withhold;
        base_params(&p, d->err);
        if ((s = enqueue(p, v, units, st)) != TG_OK) return s;
        offset += n;
    }
    t_withhold = WithholdArm{};
    return TG_OK;
}

const char* tg_status_string(tg_status status) {
    switch (status) {
        case TG_OK: return "success";
        case TG_ERR_INVALID_ARG: return "invalid argument";
        case TG_ERR_UNSUPPORTED: return "unsupported (alignment, size limit or device)";
        case TG_ERR_CUDA: return "CUDA error";
        case TG_ERR_TIMEOUT: return "in-kernel wait timed out";
        case TG_ERR_NO_DEVICE: return "no CUDA device";
    }
    return "unknown status";
}

const char* tg_last_error_message(void) { return t_message.c_str(); }

tg_status tg_device_status(tg_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    DeviceState* d = nullptr;
    tg_status s = device_state(&d);
    if (s != TG_OK) return s;
    tg::ErrorRecord rec;
    e = cudaMemcpy(&rec, d->err, sizeof rec, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error record");
    if (rec.code == tg::ERR_NONE) return TG_OK;
    e = cudaMemset(d->err, 0, sizeof rec);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error record");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error record");
    if (rec.code == tg::ERR_COUNTS)
        return fail(TG_ERR_INVALID_ARG,
                    "device token counts are negative or sum to %lld rows, more than T; the launch computed nothing",
                    (long long)rec.tile);
    static const char* roles[] = {"?", "TMA producer", "MMA issuer", "epilogue", "abort drain"};
    return fail(TG_ERR_TIMEOUT,
                "in-kernel wait ran out: role=%s block=%u stage=%u slot=%lld waited=%.1f ms; %u abort-path "
                "drains ran out",
                rec.role < 5 ? roles[rec.role] : "?", rec.block, rec.stage, (long long)rec.tile,
                rec.waited_ns / 1e6, rec.drains);
}

tg_status tg_set_wait_budget_ms(uint32_t ms) {
    if (ms > 3600000u) return fail(TG_ERR_INVALID_ARG, "wait budget %u ms above one hour", ms);
    g_budget_ms.store(ms);
    return TG_OK;
}

tg_status tg_debug_withhold_stage_in(int64_t k_block, int32_t block) {
    if (k_block < -1) return fail(TG_ERR_INVALID_ARG, "k_block must be >= -1");
    if (block < 0) return fail(TG_ERR_INVALID_ARG, "block must be >= 0");
    t_withhold = WithholdArm{k_block, block};
    return TG_OK;
}

tg_status tg_debug_withhold_stage(int64_t k_block) { return tg_debug_withhold_stage_in(k_block, 0); }

tg_status tg_debug_trace(uint64_t* tile_records, int64_t tile_capacity, uint64_t* cta_records, int64_t cta_capacity) {
    if (tile_capacity < 0 || cta_capacity < 0) return fail(TG_ERR_INVALID_ARG, "negative trace capacity");
    if ((tile_capacity > 0 && !tile_records) || (cta_capacity > 0 && !cta_records))
        return fail(TG_ERR_INVALID_ARG, "trace buffer is NULL");
    t_trace = TraceArm{tile_capacity ? tile_records : nullptr, tile_capacity, cta_capacity ? cta_records : nullptr,
                       cta_capacity};
    return TG_OK;
}

uint32_t tg_version(void) { return (0u << 16) | 2u; }

uint64_t tg_launch_count(void) { return t_launches; }

}  // extern "C"
