// tg_kernel.cuh - the persistent, warp-specialised bf16 GEMM / grouped GEMM kernel.
//
// Structure (the producer / MMA / epilogue split and the mbarrier-guarded
// shared-memory ring of the TLX-on-Blackwell matmul listing in "How We Built
// TLX", section "Introducing TLX"; here re-designed for sm_103a, made
// persistent, with a double-buffered TMEM accumulator so the epilogue of one
// tile overlaps the main loop of the next):
//
//   warp 0      TMA producer: one thread streams A and B k-blocks into a
//               STAGES-deep ring; full[s] completes when the bytes land.
//   warp 1      MMA issuer: the converged warp waits full[s]; one lane picked by
//               elect.sync (no branch) issues BK/16 tcgen05.mma into TMEM
//               accumulator buffer b and commits empty[s] (slot free) and,
//               after the last k-block, tfull[b] (tile done).  Warp 1 also
//               allocates and frees tensor memory.
//   warps 2-5   epilogue: wait tfull[b], tcgen05.ld the fp32 accumulator,
//               release the buffer (tempty[b]), add bias / apply GELU(tanh),
//               round, stage through swizzled shared memory and TMA-store C.
//
// CTA_GROUP == 2 pairs the two CTAs of a cluster on one 256-row tile: each
// CTA loads its own 128 rows of A and its own half of the tile's B columns
// into its own shared memory, the leader CTA's MMA thread issues
// tcgen05.mma.cta_group::2 over both, and each CTA's TMEM receives its 128
// rows of the accumulator.  No TMA multicast is used.
//
// The tile scheduler is static and persistent.  CTA (pair) u of U takes whole
// tiles u, u + U, u + 2U, ... of the concatenated tile list of all problems;
// within a problem tiles are rastered in bands of `band` N-tiles so that
// concurrently running tiles share A rows and B columns in L2.  A dense launch
// whose tiles do not divide evenly over the U units is balanced with stream-K:
// the k-blocks of its first R tiles (R = tiles mod U, or all tiles when there
// are fewer than U) are cut into equal contiguous ranges, one per unit, and
// every unit runs its range (one or two tile pieces) before its whole tiles.
// Each piece writes its fp32 partial sums to a workspace; the piece that
// arrives last adds all of them in k order and runs the epilogue, while the
// unit's MMA issuer is already on its next tile.  In grouped and MoE launches
// a problem's last M-tile with at most 128 rows is a half tile (M = 128 MMAs).
//
// Every mbarrier wait is bounded (wait_budget_ns, measured with %globaltimer).
// On expiry the waiting thread records the failure in the device error
// record, raises the CTA's abort flag (and its peer's), and all roles leave
// their loops: the producer waits until the TMA loads it issued have landed
// (in a pair, the leader closes the phases the other CTA left open and waits
// for both CTAs' loads), issued MMAs are drained with a final commit, tensor
// memory is freed and the kernel returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <type_traits>

#include "tg_ptx.cuh"

namespace tg {

constexpr int BM = 128;              // accumulator rows per CTA (TMEM lanes)
constexpr int BK = 64;               // K per pipeline stage: one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;           // K per tcgen05.mma.kind::f16
constexpr int NUM_THREADS = 192;
constexpr int EPI_WARP0 = 2;         // warps 2..5 drain TMEM; warp w reads lanes 32*(w%4)..+31
constexpr int NUM_EPI_WARPS = 4;
constexpr int FIX_BUFS = 4;          // chunks in flight per warp while a unit's last piece adds up its tile
constexpr int C_STAGE_BYTES = 32 * 128;   // per-warp store staging buffer: 32 rows x 128 bytes
constexpr int SMEM_LIMIT = 232448;        // max dynamic shared memory per CTA on sm_100 family
constexpr int MOE_MAX_G = 190;            // experts per call of the device-counts MoE form (table in shared memory)
constexpr int GROUP_TABLE_MAX = 2 * (MOE_MAX_G + 1);   // grouped launches: problems whose first tiles fit that table
constexpr int SK_QUANTUM = 4;             // stream-K range boundaries fall on multiples of 4 k-blocks
constexpr int MAX_STAGES = 8;

enum : uint32_t { ERR_NONE = 0, ERR_TIMEOUT = 1, ERR_COUNTS = 2 };
enum : uint32_t { ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_EPILOGUE = 3, ROLE_DRAIN = 4 };
enum : int32_t { EPI_NONE = 0, EPI_BIAS = 1, EPI_BIAS_GELU = 2 };

struct ErrorRecord {
    uint32_t code;        // ERR_*
    uint32_t role;        // ROLE_*
    uint32_t block;       // blockIdx.x of the reporting CTA
    uint32_t stage;       // ring stage or accumulator buffer being waited on
    int64_t tile;         // work item slot
    uint64_t waited_ns;
    uint32_t drains;      // waits of the abort path (issued loads, issued MMAs) that ran out too
    uint32_t pad;
};

// One GEMM problem as the device sees it.
struct alignas(128) Problem {
    CUtensorMap tma_a;
    CUtensorMap tma_b;
    CUtensorMap tma_c;
    const void* bias;       // bf16 or fp16 [N] (FLAG_BIAS_F16)
    const float* row_scale;   // optional fp32 [M]: row i of the accumulator is multiplied by it (RMS norm)
    int64_t tile_begin;   // global index of this problem's first tile
    int32_t M, N, K;
    int32_t epi;
    int32_t tiles_m, tiles_n, k_blocks;
    // Broadcast form (repeat > 0): rows of A are U distinct "user" rows and
    // output row i * repeat + j (j < repeat) is user row i's result; tma_c is a
    // 3-D view [U][repeat][N] of C.  Each (M-tile, N-tile) is computed by
    // `replicas` CTAs, replica r storing the repeat indices
    // [r * repeat / replicas, (r + 1) * repeat / replicas).
    int32_t repeat;
    int32_t replicas;           // >= 1
    uint32_t idesc;             // tcgen05 instruction descriptor (operand types, M, N, majors)
    uint32_t flags;             // FLAG_*: 16-bit output and bias element types
};

enum : uint32_t {
    FLAG_C_F16 = 1u,      // 16-bit output is IEEE fp16 (else bf16)
    FLAG_BIAS_F16 = 2u,   // bias is fp16 (else bf16)
    // N-major B with N % 64 == 0: tma_b is the view {64 columns, k, column chunk of 64}
    // (MoE: plus the expert), so a CTA's BN_CTA columns of one k-block are a single box.
    // Each TMA instruction costs the producer about as much as a quarter of an MMA
    // k-block, so one box instead of BN_CTA / 64 keeps the ring ahead of the MMA.
    FLAG_B_WIDE = 4u,
};

struct Params {
    Problem dense;              // the problem of a dense launch (lives in parameter space)
    // Dense column halves (nh_tiles): B map whose box covers half the N rows of
    // dense.tma_b's (K-major B); N-major B loads half as many 64-column boxes instead,
    // from this map (the plain 2-D one) when dense.tma_b is the wide view (FLAG_B_WIDE).
    CUtensorMap b_half;
    const Problem* problems;    // grouped launch: device array written by the host
    int32_t num_problems;
    int32_t band;               // raster band width in N-tiles
    int64_t total_tiles;        // tiles of the launch (dense broadcast form: tiles x replicas)
    ErrorRecord* err;
    uint64_t wait_budget_ns;
    int64_t withhold_kb;        // test hook, -1 = off (see tg_debug_withhold_stage_in)
    int32_t withhold_block;
    // Timeline trace (tg_debug_trace), null when off.  trace_tiles[s] = {block,
    // first k-block ready, accumulator complete, epilogue done} for work item slot
    // s < trace_tiles_cap, where the i-th item of unit u has slot i * U + u (times
    // from %globaltimer, ns); trace_ctas[b] = {entry, set-up done, teardown start,
    // exit} for block b < trace_ctas_cap.
    uint64_t* trace_tiles;
    int64_t trace_tiles_cap;
    uint64_t* trace_ctas;
    int64_t trace_ctas_cap;
    // Device-counts MoE form: expert g owns rows [off_g, off_g + moe_counts[g]) of A and C,
    // off_g = sum of the counts before g; B is a 3-D map [G][K][N] (or [G][N][K]).
    // moe_maps[2 g] and [2 g + 1] are expert g's own A and C maps (its moe_counts[g] rows),
    // written on the device by the kernel launched just before this one (moe_maps_kernel).
    const int32_t* moe_counts;
    int32_t moe_groups;
    int64_t moe_rows;           // T: rows of A and C; the counts must sum to at most T
    const CUtensorMap* moe_maps;
    // Host side only: launch as a programmatic dependent of the kernel before it in the
    // stream (the row-statistics pass of the fused RMS norm, or the counter reset).
    // Only the reads of that kernel's output wait for it (griddepcontrol.wait); set-up
    // and main loop overlap it.
    int32_t pdl;
    // Stream-K (dense only; see the file header).  The sk_tiles * k_blocks k-blocks of
    // tiles [0, sk_tiles), in tile order, are cut into sk_units contiguous ranges, range
    // r = [sk_bound(r), sk_bound(r + 1)) belonging to unit r.  Tiles [sk_tiles,
    // total_tiles) are whole tiles: unit u takes sk_tiles + u, sk_tiles + u + U, ...
    // Column halves (dense only; exclusive with stream-K).  The last nh_tiles tiles, the
    // last partial wave, each run as two units of BN/2 columns (N = BN/2 MMAs on half the
    // B bytes; no partial sums): unit u's item index g = u, u + U, ... covers whole tile g
    // while g < total_tiles - nh_tiles, then column half (g - f) / nh_tiles of tile
    // f + (g - f) % nh_tiles, f = total_tiles - nh_tiles, for g < total_tiles + nh_tiles.
    int32_t nh_tiles;
    int32_t sk_tiles;           // 0: no stream-K
    int32_t sk_units;
    int32_t sk_max_slices;      // pieces of one tile at most (stride of the partial slabs)
    float* sk_partial;          // [sk_tiles][sk_max_slices][CTA_GROUP][4 warps][BN/4][32 lanes][4]
    uint32_t* sk_count;         // [sk_tiles][CTA_GROUP][4 warps], zero at launch
    uint32_t* sk_flag;          // [sk_tiles][sk_max_slices][CTA_GROUP][4 warps], zero at launch
};

// ----------------------------------------------------------------------------------------
// stream-K ranges (shared by the host plan and the kernel)

// First k-block of unit r's range in the stream-K space of `total` k-blocks:
// SK_QUANTUM * floor(r * G / units) with G = floor(total / SK_QUANTUM); the last
// range ends at `total`.  Ranges are non-empty when G >= units.
__host__ __device__ __forceinline__ int64_t sk_bound(int64_t r, int64_t units, int64_t total) {
    if (r >= units) return total;
    const int64_t G = total / SK_QUANTUM;
    return SK_QUANTUM * ((r * G) / units);
}

// The unit whose range holds k-block x: the largest r with sk_bound(r) <= x.
__host__ __device__ __forceinline__ int64_t sk_owner(int64_t x, int64_t units, int64_t total) {
    const int64_t G = total / SK_QUANTUM;
    const int64_t X = x / SK_QUANTUM;
    const int64_t r = ((X + 1) * units + G - 1) / G - 1;
    return r < units - 1 ? r : units - 1;
}

// One piece of a stream-K range: k-blocks [kb0, kb1) of tile t, the slice-th of
// the tile's `slices` pieces in k order (slices == 0: the range holds the whole
// tile, which then needs no partial sums).
struct SkPiece {
    int64_t t;
    int kb0, kb1;
    int slice, slices;
};

// The piece that starts at k-block `cur` of unit `unit`'s range [.., end), in the
// stream-K space of `total` = tiles * k_blocks k-blocks cut into `units` ranges.
__host__ __device__ __forceinline__ SkPiece sk_piece(int64_t cur, int64_t end, int k_blocks, int64_t units,
                                                     int64_t total, int64_t unit) {
    SkPiece q;
    q.t = cur / k_blocks;
    q.kb0 = static_cast<int>(cur - q.t * k_blocks);
    const int64_t kb1 = q.kb0 + (end - cur);
    q.kb1 = static_cast<int>(kb1 < k_blocks ? kb1 : k_blocks);
    const int64_t first = sk_owner(q.t * k_blocks, units, total);
    const int64_t last = sk_owner((q.t + 1) * k_blocks - 1, units, total);
    q.slice = static_cast<int>(unit - first);
    q.slices = last > first ? static_cast<int>(last - first + 1) : 0;
    return q;
}

// Stream-K plan of a dense launch of `tiles` tiles of `k_blocks` k-blocks on
// `units` resident units.  The R = tiles mod units tiles of the last, partial
// wave (all tiles when there are fewer than units) would leave units - R units
// idle while they run; instead their R * k_blocks k-blocks are cut into U
// ranges (U = units, fewer where ranges would drop below SK_QUANTUM k-blocks or
// a tile would be cut into more pieces than allowed: SK_MAX_PIECES when every
// tile is in pieces, SK_MAX_PIECES_WITH_WHOLE when units also run whole tiles,
// so that a tile's last piece reads back one or two partials only, while its
// unit is busy with its next tile).  A piece costs a write of its fp32 partial
// sums, so there is no stream-K when the pieces would be almost whole tiles
// (R > 3 units / 4), when a range would hold a whole tile (U <= R), or when
// tiles are short: k_blocks < 2 * SK_QUANTUM, or, when units also run whole
// tiles, k_blocks < SK_MIN_KB_WITH_WHOLE (a short tile's piece saves less than
// its partial sums cost the units around it; measured on the 131072 x 128 x 1024
// workload, 16 k-blocks per tile: 55 us without stream-K, 71 us with it).
constexpr int SK_MAX_PIECES = 8;
constexpr int SK_MAX_PIECES_WITH_WHOLE = 2;
constexpr int SK_MIN_KB_WITH_WHOLE = 32;

struct SkPlan {
    int tiles = 0;        // R: tiles [0, R) run as stream-K pieces (0: no stream-K)
    int units = 0;        // U: units that own a range
    int max_slices = 0;   // pieces of one tile at most
};

__host__ __forceinline__ SkPlan sk_plan(int64_t tiles, int64_t units, int64_t k_blocks) {
    SkPlan sp;
    if (units <= 1 || k_blocks < 2 * SK_QUANTUM || tiles <= 0) return sp;
    const int64_t R = tiles < units ? tiles : tiles % units;
    if (R == 0) return sp;
    if (tiles > units && (R * 4 > units * 3 || k_blocks < SK_MIN_KB_WITH_WHOLE)) return sp;
    const int64_t total = R * k_blocks;
    int64_t U = units;
    const int64_t max_pieces = tiles > units ? SK_MAX_PIECES_WITH_WHOLE : SK_MAX_PIECES;
    if (U > max_pieces * R) U = max_pieces * R;
    if (U > total / SK_QUANTUM) U = total / SK_QUANTUM;
    if (U <= R) return sp;
    int64_t max_slices = 1;
    for (int64_t t = 0; t < R; ++t) {
        const int64_t n = sk_owner((t + 1) * k_blocks - 1, U, total) - sk_owner(t * k_blocks, U, total) + 1;
        if (n > max_slices) max_slices = n;
    }
    sp.tiles = static_cast<int>(R);
    sp.units = static_cast<int>(U);
    sp.max_slices = static_cast<int>(max_slices);
    return sp;
}

// MODE: 0 dense (tensor maps in parameter space), 1 grouped (problem table in
// device memory), 2 MoE with device-resident token counts.
template <int BN_, int CTA_GROUP_, bool A_MN_, bool B_MN_, bool C_F32_, int MODE_>
struct Config {
    static constexpr int BN = BN_;                   // tile columns (whole pair)
    static constexpr int CTA_GROUP = CTA_GROUP_;
    static constexpr bool A_MN = A_MN_;              // A stored M-contiguous (column-major)
    static constexpr bool B_MN = B_MN_;              // B stored N-contiguous (row-major K x N)
    static constexpr bool C_F32 = C_F32_;
    static constexpr bool GROUPED = MODE_ == 1;
    static constexpr bool MOE = MODE_ == 2;
    static constexpr int BN_CTA = BN / CTA_GROUP;    // B columns each CTA loads
    static constexpr int TILE_M = BM * CTA_GROUP;    // rows per tile (pair)
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN_CTA * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int CW = C_F32 ? 32 : 64;       // output columns per 128-byte staged row
    static constexpr int TMEM_COLS = 2 * BN;         // two fp32 accumulators of BN columns
    static constexpr int C_BYTES = NUM_EPI_WARPS * 2 * C_STAGE_BYTES;
    // Prefix tables in shared memory: MoE, tiles and rows before each expert; grouped, each
    // problem's first tile (while the problems fit), so that finding a unit's problem at a
    // unit boundary reads no global memory.
    static constexpr int TABLE_BYTES = (MOE || GROUPED) ? 8 * (MOE_MAX_G + 1) : 0;
    static constexpr int FIXED = C_BYTES + TABLE_BYTES + 512 /*barriers and slots*/ + 1024 /*alignment slack*/;
    static constexpr int STAGES_FIT = (SMEM_LIMIT - FIXED) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > MAX_STAGES ? MAX_STAGES : STAGES_FIT;

    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_C = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_TABLE = OFF_C + C_BYTES;
    static constexpr int OFF_BAR = OFF_TABLE + TABLE_BYTES;
    // barriers: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int OFF_TMEM_SLOT = OFF_BAR + 8 * NUM_BARS;
    static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
    static constexpr int OFF_MOE_TOTAL = OFF_ABORT + 4;
    // The producer's record of its ring, read after an abort (by the pair's leader
    // through distributed shared memory): flag (set when final), ring positions
    // advanced, and per stage the last position loaded there and its bytes.
    static constexpr int OFF_DRAIN_FLAG = OFF_MOE_TOTAL + 4;
    static constexpr int OFF_DRAIN_POS = OFF_DRAIN_FLAG + 4;
    static constexpr int OFF_DRAIN_LAST = OFF_DRAIN_POS + 4;
    static constexpr int OFF_DRAIN_BYTES = OFF_DRAIN_LAST + 4 * MAX_STAGES;
    static constexpr int SMEM_BYTES = OFF_DRAIN_BYTES + 4 * MAX_STAGES + 1024;


    static_assert(BN == 128 || BN == 256, "tile width");
    static_assert(CTA_GROUP == 1 || CTA_GROUP == 2, "cta group");
    static_assert(STAGES >= 2, "ring too shallow");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
    static_assert(BN_CTA % 64 == 0, "MN-major B is loaded in 64-column boxes");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation is a power of two");
    static_assert(NUM_EPI_WARPS * FIX_BUFS * 32 * CW * 4 <= STAGES * STAGE_BYTES,
                  "the add-up staging of a unit's last piece must fit in the operand ring");
};

// ----------------------------------------------------------------------------------------
// scheduling helpers

struct TileCoord {
    int g;        // problem (grouped) or expert (MoE) index
    int m0;       // first accumulator row of this CTA (MoE: a row of the whole A / C)
    int n0;       // first column of the tile
    int r;        // replica index (broadcast form), else 0
    int row_end;  // MoE: first row past this expert's rows; otherwise INT32_MAX
    // Half tile (grouped and MoE pairs): a problem's last M-tile with at most 128 rows
    // left is computed by 256 x 16 x 128-row MMAs (M = 128 for the pair), which take
    // half the time of M = 256.  Each CTA then holds 64 rows; its accumulator keeps
    // columns [0, BN/2) in TMEM lanes 0-63 and [BN/2, BN) in lanes 64-127, both in
    // TMEM columns [0, BN/2).
    bool half;
    // Column half (dense): columns [n0, n0 + BN/2) only, by N = BN/2 MMAs; the
    // accumulator holds them in TMEM columns [0, BN/2) with the usual row layout.
    bool nhalf;
};

// Shared-memory prefix tables, built by every CTA at start (null when a launch has none).
// Device-counts MoE: tile_pref[g] = tiles of experts before g, row_off[g] = rows before g,
// [G + 1] each.  Grouped: tile_pref[i] = problem i's first tile.
struct MoeTable {
    const int32_t* tile_pref;
    const int32_t* row_off;
};

template <class Cfg>
__device__ __forceinline__ const Problem& problem_of(const Params& p, int g) {
    if constexpr (Cfg::GROUPED) return p.problems[g];
    else return p.dense;
}

// Grouped launches keep each problem's first tile in shared memory when the problems fit
// the table and the tile indices fit 32 bits.
__device__ __forceinline__ bool group_table_fits(const Params& p) {
    return p.num_problems <= GROUP_TABLE_MAX && p.total_tiles <= 0x7fffffffll;
}

// Problem (or expert) containing global tile t; `g` is a hint that only moves forward.
// Grouped: from the shared-memory table of first tiles when there is one (mt.tile_pref),
// else from the problem array in global memory, one dependent load per problem passed.
template <class Cfg>
__device__ __forceinline__ int find_problem(const Params& p, int64_t t, int g, const MoeTable& mt = {}) {
    if constexpr (Cfg::GROUPED) {
        if (mt.tile_pref != nullptr) {
            while (g + 1 < p.num_problems && mt.tile_pref[g + 1] <= t) ++g;
        } else {
            while (g + 1 < p.num_problems && p.problems[g + 1].tile_begin <= t) ++g;
        }
        return g;
    } else if constexpr (Cfg::MOE) {
        while (g + 1 < p.moe_groups && mt.tile_pref[g + 1] <= t) ++g;
        return g;
    } else {
        return 0;
    }
}

// Raster of one problem's tiles_m x tiles_n tiles: bands of `band` N-tiles, swept
// one M-row of the band after another; odd bands run up the M-tiles, so that the
// A rows of a band's last raster rows, still in L2, serve the next band's first.
// Tile `local` (0 <= local < tiles_m * tiles_n) is M-tile mb, N-tile nb.
__host__ __device__ __forceinline__ void raster(int64_t local, int tiles_m, int tiles_n, int band, int& mb, int& nb) {
    const int64_t per_band = static_cast<int64_t>(tiles_m) * band;
    const int b = static_cast<int>(local / per_band);
    const int r = static_cast<int>(local - static_cast<int64_t>(b) * per_band);
    const int n_first = b * band;
    const int width = band < tiles_n - n_first ? band : tiles_n - n_first;
    const int row = r / width;
    mb = (b & 1) ? tiles_m - 1 - row : row;
    nb = n_first + (r - row * width);
}

template <class Cfg>
__device__ __forceinline__ TileCoord tile_coord(const Params& p, int64_t t, int g, uint32_t rank,
                                                const MoeTable& mt = {}) {
    const Problem& pr = problem_of<Cfg>(p, g);
    int64_t local = t - pr.tile_begin;
    int tiles_m = pr.tiles_m;
    if constexpr (Cfg::MOE) {
        local = t - mt.tile_pref[g];
        tiles_m = (mt.tile_pref[g + 1] - mt.tile_pref[g]) / pr.tiles_n;
    }
    int replica = 0;
    if (pr.replicas > 1) {   // replicas of one tile are adjacent: they share A and B in L2
        replica = static_cast<int>(local % pr.replicas);
        local /= pr.replicas;
    }
    int mb, nb;
    raster(local, tiles_m, pr.tiles_n, p.band, mb, nb);
    TileCoord c;
    c.g = g;
    c.half = false;
    c.nhalf = false;
    if constexpr (Cfg::CTA_GROUP == 2 && (Cfg::GROUPED || Cfg::MOE)) {
        const int rows_left = (Cfg::MOE ? mt.row_off[g + 1] - mt.row_off[g] : pr.M) - mb * Cfg::TILE_M;
        c.half = rows_left <= BM;
    }
    c.m0 = mb * Cfg::TILE_M + static_cast<int>(rank) * (c.half ? BM / 2 : BM);
    c.n0 = nb * Cfg::BN;
    c.r = replica;
    c.row_end = INT32_MAX;
    if constexpr (Cfg::MOE) {
        c.m0 += mt.row_off[g];
        c.row_end = mt.row_off[g + 1];
    }
    return c;
}

// A work item: a whole tile, or one stream-K piece (a k-block range) of a tile.
struct Work {
    int64_t t;    // tile
    int kb0;      // k-blocks [kb0, kb1) of the tile; a whole tile uses its problem's k_blocks
    int kb1;
    int slice;    // piece: its index among the tile's pieces (k order)
    int slices;   // piece: pieces of the tile (>= 2); 0 for a whole tile
    int nh;       // column half (0 or 1), or -1
    int64_t slot; // i * U + u for the i-th item of unit u (trace index)
};

// The work items of one unit, in order: its first whole tile, its stream-K range
// (one or two pieces), then its other whole tiles.  The first whole tiles of all
// units start together on neighbouring tiles, which share their operands in L2;
// a piece's partial sums are added up while the unit works on its next tile.
struct Sched {
    int64_t cur, end;    // rest of the unit's stream-K range (k-blocks of the stream-K space)
    int64_t next_tile;   // its next whole tile
    int64_t i;           // items handed out so far
};

template <class Cfg>
__device__ __forceinline__ Sched sched_begin(const Params& p, int64_t unit) {
    Sched s{0, 0, unit, 0};
    if constexpr (!Cfg::GROUPED && !Cfg::MOE) {
        if (p.sk_tiles > 0) {
            const int64_t total = static_cast<int64_t>(p.sk_tiles) * p.dense.k_blocks;
            if (unit < p.sk_units) {
                s.cur = sk_bound(unit, p.sk_units, total);
                s.end = sk_bound(unit + 1, p.sk_units, total);
            }
            s.next_tile = p.sk_tiles + unit;
        }
    }
    return s;
}

template <class Cfg>
__device__ __forceinline__ bool sched_next(const Params& p, int64_t unit, int64_t num_units, int64_t total_tiles,
                                           Sched& s, Work& w) {
    w.slot = s.i * num_units + unit;
    if constexpr (!Cfg::GROUPED && !Cfg::MOE) {
        if (s.cur < s.end && (s.i > 0 || s.next_tile >= total_tiles)) {
            const int kbs = p.dense.k_blocks;
            const SkPiece q = sk_piece(s.cur, s.end, kbs, p.sk_units, static_cast<int64_t>(p.sk_tiles) * kbs, unit);
            w.nh = -1;
            w.t = q.t;
            w.kb0 = q.kb0;
            w.kb1 = q.kb1;
            w.slice = q.slice;
            w.slices = q.slices;
            s.cur += q.kb1 - q.kb0;
            ++s.i;
            return true;
        }
    }
    w.nh = -1;
    int64_t whole = total_tiles;
    if constexpr (!Cfg::GROUPED && !Cfg::MOE) whole -= p.nh_tiles;
    if (s.next_tile >= whole) {
        if constexpr (Cfg::GROUPED || Cfg::MOE) return false;
        const int64_t hu = s.next_tile - whole;          // column-half unit
        if (hu >= 2 * static_cast<int64_t>(p.nh_tiles)) return false;
        w.t = whole + hu % p.nh_tiles;
        w.nh = static_cast<int>(hu / p.nh_tiles);
    } else {
        w.t = s.next_tile;
    }
    w.kb0 = 0;
    w.kb1 = 0;
    w.slice = 0;
    w.slices = 0;
    s.next_tile += num_units;
    ++s.i;
    return true;
}

// The coordinates of a work item: its tile's, narrowed to one column half.
template <class Cfg>
__device__ __forceinline__ TileCoord coord_of(const Params& p, const Work& w, int g, uint32_t rank,
                                              const MoeTable& mt) {
    TileCoord c = tile_coord<Cfg>(p, w.t, g, rank, mt);
    c.nhalf = w.nh >= 0;
    if (c.nhalf) c.n0 += w.nh * (Cfg::BN / 2);
    return c;
}

// k-blocks [begin, end) of a work item on problem pr
__device__ __forceinline__ int work_kb_end(const Work& w, const Problem& pr) {
    return (w.kb1 > 0 || w.slices > 0) ? w.kb1 : pr.k_blocks;
}

// ----------------------------------------------------------------------------------------
// bounded waits

__device__ __forceinline__ void report_timeout(const Params& p, uint32_t role, int64_t tile, uint32_t stage,
                                               uint64_t waited) {
    if (role == ROLE_DRAIN) atomicAdd(&p.err->drains, 1u);
    if (atomicCAS(&p.err->code, ERR_NONE, ERR_TIMEOUT) == ERR_NONE) {
        p.err->role = role;
        p.err->block = blockIdx.x;
        p.err->stage = stage;
        p.err->tile = tile;
        p.err->waited_ns = waited;
        __threadfence();
    }
}

// Raise the abort flag of this CTA and, in a pair, of the peer CTA.
template <int CTA_GROUP>
__device__ __forceinline__ void raise_abort(uint32_t abort_addr) {
    asm volatile("st.volatile.shared::cta.u32 [%0], 1;" :: "r"(abort_addr) : "memory");
    if constexpr (CTA_GROUP == 2) {
        const uint32_t peer = ptx::mapa(abort_addr, ptx::cluster_ctarank() ^ 1u);
        asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], 1;" :: "r"(peer) : "memory");
    }
}

__device__ __forceinline__ bool abort_raised(uint32_t abort_addr) {
    uint32_t v;
    asm volatile("ld.volatile.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(abort_addr) : "memory");
    return v != 0;
}

// Wait for phase `parity` of `bar`.  false: the budget ran out (recorded) or
// another role aborted; the caller leaves its loop.
//
// SLEEP waiters (everyone but the MMA issuer) let the hardware suspend them
// inside try_wait until the phase completes (up to SLEEP_NS per call): a
// spinning warp would take issue slots from the MMA-issuing warp on the same
// SM sub-partition and leave the tensor pipe idle between instructions.  The
// hint is an immediate: taken from a kernel parameter instead, the main loops
// of the N-major-B GEMMs ran ~1 % slower per k-block.
constexpr uint32_t SLEEP_NS = 20000;

template <int CTA_GROUP, bool SLEEP = true>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Params& p, uint32_t abort_addr,
                                             uint32_t role, int64_t tile, uint32_t stage) {
    auto try_once = [&]() {
        if constexpr (SLEEP) return ptx::mbar_try_wait_sleep(bar, parity, SLEEP_NS);
        else return ptx::mbar_try_wait(bar, parity);
    };
    if (try_once()) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (try_once()) return true;
        if (SLEEP || (it & 15u) == 0u) {
            if (abort_raised(abort_addr)) return false;
            const uint64_t dt = ptx::globaltimer_ns() - t0;
            if (dt > p.wait_budget_ns) {
                report_timeout(p, role, tile, stage, dt);
                raise_abort<CTA_GROUP>(abort_addr);
                return false;
            }
        }
    }
}

// Quiet wait used while shutting down after an abort: no new error record.
__device__ __forceinline__ bool wait_quiet(uint32_t bar, uint32_t parity, uint64_t budget_ns) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > budget_ns) return false;
    }
    return true;
}

// ----------------------------------------------------------------------------------------
// epilogue math

// z/2 * (1 + tanh(sqrt(2/pi) * (z + 0.044715 z^3))), arranged for few instructions
// (the epilogue warps share issue slots with the MMA issuer):
//   u = z * (k0 + k0 k1 z^2),  gelu = h + h * tanh(u) with h = z / 2
constexpr float GELU_K0 = 0.7978845608028654f;               // sqrt(2 / pi)
constexpr float GELU_K01 = 0.7978845608028654f * 0.044715f;  // sqrt(2 / pi) * 0.044715

__device__ __forceinline__ float gelu_tanh_f32(float z) {
    const float u = z * fmaf(GELU_K01, z * z, GELU_K0);
    const float h = 0.5f * z;
    return fmaf(h, ptx::tanh_approx(u), h);
}

// gelu_tanh_f32 of two values with packed f32x2 arithmetic: the same operations in the
// same order, so each result is bit for bit that of gelu_tanh_f32; measured ~780 issue
// cycles a 64-column chunk in scalar form, the epilogue's largest cost.
__device__ __forceinline__ void gelu_tanh_f32x2(float& a, float& b) {
    const uint64_t z = ptx::f32x2_pack(a, b);
    const uint64_t poly = ptx::f32x2_fma(ptx::f32x2_pack(GELU_K01, GELU_K01), ptx::f32x2_mul(z, z),
                                         ptx::f32x2_pack(GELU_K0, GELU_K0));
    float u0, u1;
    ptx::f32x2_unpack(ptx::f32x2_mul(z, poly), u0, u1);
    const uint64_t h = ptx::f32x2_mul(ptx::f32x2_pack(0.5f, 0.5f), z);
    ptx::f32x2_unpack(ptx::f32x2_fma(h, ptx::f32x2_pack(ptx::tanh_approx(u0), ptx::tanh_approx(u1)), h), a, b);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ----------------------------------------------------------------------------------------
// shared-memory words (own CTA)

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cta.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// ----------------------------------------------------------------------------------------
// after an abort: wait until the TMA loads this CTA (pair) issued have landed
//
// Positions are k-blocks counted along the unit's work items, the same sequence
// in both CTAs of a pair; position x uses stage x % STAGES in phase (x / STAGES) & 1.
// Only the last STAGES positions can still have loads in flight: a producer
// loads position x only after the MMA released position x - STAGES, which
// needed all of its bytes.  Every load signals the full barrier of the pair's
// leader; the leader expects the bytes of both CTAs when it arrives.  So in a
// pair, a position that only one CTA loaded (the other withheld it or had not
// got there) is closed by the leader: complete_tx for the bytes that will never
// come, or its own arrival with the other CTA's bytes.  Then each such phase
// completes exactly when the issued bytes have landed, and the leader waits for
// it; the other CTA stays in the cluster barrier of the teardown until then.
template <class Cfg>
__device__ __noinline__ void drain_issued_loads(const Params& p, uint32_t base) {
    constexpr int STAGES = Cfg::STAGES;
    constexpr int CG = Cfg::CTA_GROUP;
    const uint32_t bar0 = base + Cfg::OFF_BAR;
    const uint32_t pos0 = ld_shared_u32(base + Cfg::OFF_DRAIN_POS);
    uint32_t pos1 = 0;
    uint32_t last1[STAGES], bytes1[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) last1[s] = bytes1[s] = 0xffffffffu;
    if constexpr (CG == 2) {
        // the other CTA's ring record, once it is final
        const uint32_t flag1 = ptx::mapa(base + Cfg::OFF_DRAIN_FLAG, 1);
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::ld_cluster_acquire_u32(flag1) == 0u) {
            if (ptx::globaltimer_ns() - t0 > p.wait_budget_ns) {
                report_timeout(p, ROLE_DRAIN, -1, 0, p.wait_budget_ns);
                return;
            }
        }
        pos1 = ptx::ld_cluster_u32(ptx::mapa(base + Cfg::OFF_DRAIN_POS, 1));
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            last1[s] = ptx::ld_cluster_u32(ptx::mapa(base + Cfg::OFF_DRAIN_LAST + 4 * s, 1));
            bytes1[s] = ptx::ld_cluster_u32(ptx::mapa(base + Cfg::OFF_DRAIN_BYTES + 4 * s, 1));
        }
    }
    const uint32_t top = pos0 > pos1 ? pos0 : pos1;
    bool ok = true;
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
        if (top < static_cast<uint32_t>(s) + 1u) continue;             // stage never reached
        const uint32_t x = top - 1u - ((top - 1u - s) % STAGES);        // its position in [top - STAGES, top)
        const uint32_t bar = bar0 + 8u * s;
        const bool a0 = ld_shared_u32(base + Cfg::OFF_DRAIN_LAST + 4 * s) == x;
        const bool a1 = CG == 2 && last1[s] == x;
        if constexpr (CG == 2) {
            if (a0 && !a1) ptx::mbar_complete_tx(bar, ld_shared_u32(base + Cfg::OFF_DRAIN_BYTES + 4 * s));
            else if (!a0 && a1) ptx::mbar_arrive_expect_tx(bar, bytes1[s]);
        }
        if (a0 || a1) ok = wait_quiet(bar, (x / STAGES) & 1u, p.wait_budget_ns) && ok;
    }
    if (!ok) report_timeout(p, ROLE_DRAIN, -1, 0, p.wait_budget_ns);
}

// ----------------------------------------------------------------------------------------
// the kernel

template <class Cfg>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_kernel(const __grid_constant__ Params p) {
    constexpr int STAGES = Cfg::STAGES;
    constexpr int CG = Cfg::CTA_GROUP;
    constexpr int BN = Cfg::BN;

    const uint64_t t_entry = p.trace_ctas != nullptr ? ptx::globaltimer_ns() : 0;

    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms (same offset in every CTA).
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);

    const uint32_t sA = base + Cfg::OFF_A;
    const uint32_t sB = base + Cfg::OFF_B;
    const uint32_t sC = base + Cfg::OFF_C;
    const uint32_t bar0 = base + Cfg::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    const uint32_t tmem_slot = base + Cfg::OFF_TMEM_SLOT;
    const uint32_t abort_addr = base + Cfg::OFF_ABORT;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = (CG == 2) ? ptx::cluster_ctarank() : 0u;
    const bool leader = (rank == 0);
    const int64_t unit = blockIdx.x / CG;
    const int64_t num_units = gridDim.x / CG;

    // ---- set-up: barriers, ring record, tensor memory
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);
            ptx::mbar_init(tempty_bar(b), NUM_EPI_WARPS * CG);
        }
        ptx::mbar_init(drain_bar, 1);
        st_shared_u32(abort_addr, 0u);
        st_shared_u32(base + Cfg::OFF_DRAIN_FLAG, 0u);
        st_shared_u32(base + Cfg::OFF_DRAIN_POS, 0u);
        for (int s = 0; s < MAX_STAGES; ++s) {
            st_shared_u32(base + Cfg::OFF_DRAIN_LAST + 4 * s, 0xffffffffu);
            st_shared_u32(base + Cfg::OFF_DRAIN_BYTES + 4 * s, 0u);
        }
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(tmem_slot, Cfg::TMEM_COLS);
        ptx::tmem_relinquish<CG>();
    }
    if constexpr (Cfg::MOE) {
        if (warp == EPI_WARP0) {
            // Prefix sums of the device-resident token counts: rows and tiles before each expert.
            int32_t* tile_pref = reinterpret_cast<int32_t*>(smem + Cfg::OFF_TABLE);
            int32_t* row_off = tile_pref + (MOE_MAX_G + 1);
            const int G = p.moe_groups;
            const int64_t tiles_n = p.dense.tiles_n;
            long long rows = 0, tiles = 0;
            bool bad = false;
            if (lane == 0) { tile_pref[0] = 0; row_off[0] = 0; }
            for (int base_g = 0; base_g < G; base_g += 32) {
                const int i = base_g + lane;
                long long c = (i < G) ? static_cast<long long>(__ldg(p.moe_counts + i)) : 0ll;
                bad |= c < 0;
                c = c < 0 ? 0 : c;
                long long tl = (c + Cfg::TILE_M - 1) / Cfg::TILE_M * tiles_n;
                for (int d = 1; d < 32; d <<= 1) {   // inclusive warp scan
                    const long long xc = __shfl_up_sync(0xffffffffu, c, d);
                    const long long xt = __shfl_up_sync(0xffffffffu, tl, d);
                    if (lane >= d) { c += xc; tl += xt; }
                }
                if (i < G) {
                    row_off[i + 1] = static_cast<int32_t>(min(rows + c, 0x7fffffffll));
                    tile_pref[i + 1] = static_cast<int32_t>(min(tiles + tl, 0x7fffffffll));
                }
                rows += __shfl_sync(0xffffffffu, c, 31);
                tiles += __shfl_sync(0xffffffffu, tl, 31);
            }
            bad = __any_sync(0xffffffffu, bad) || rows > p.moe_rows;
            if (lane == 0) {
                *reinterpret_cast<volatile int32_t*>(smem + Cfg::OFF_MOE_TOTAL) = bad ? 0 : static_cast<int32_t>(tiles);
                if (bad && blockIdx.x == 0 && atomicCAS(&p.err->code, ERR_NONE, ERR_COUNTS) == ERR_NONE) {
                    p.err->role = 0;
                    p.err->block = 0;
                    p.err->stage = 0;
                    p.err->tile = rows;
                    p.err->waited_ns = 0;
                }
            }
        }
    }
    if constexpr (Cfg::GROUPED) {
        if (warp == EPI_WARP0 && group_table_fits(p)) {
            int32_t* first_tile = reinterpret_cast<int32_t*>(smem + Cfg::OFF_TABLE);
            for (int i = lane; i < p.num_problems; i += 32)
                first_tile[i] = static_cast<int32_t>(p.problems[i].tile_begin);
        }
    }
    if constexpr (!Cfg::GROUPED) {
        if (threadIdx.x == 0) {
            ptx::prefetch_tensormap(&p.dense.tma_a);
            ptx::prefetch_tensormap(&p.dense.tma_b);
            ptx::prefetch_tensormap(&p.dense.tma_c);
            if (p.nh_tiles > 0) ptx::prefetch_tensormap(&p.b_half);
        }
    }
    ptx::tc_fence_before_sync();
    if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_TMEM_SLOT);
    int64_t total_tiles = p.total_tiles;
    MoeTable mt{};
    if constexpr (Cfg::MOE) {
        total_tiles = *reinterpret_cast<volatile int32_t*>(smem + Cfg::OFF_MOE_TOTAL);
        mt.tile_pref = reinterpret_cast<const int32_t*>(smem + Cfg::OFF_TABLE);
        mt.row_off = mt.tile_pref + (MOE_MAX_G + 1);
    }
    if constexpr (Cfg::GROUPED) {
        if (group_table_fits(p)) mt.tile_pref = reinterpret_cast<const int32_t*>(smem + Cfg::OFF_TABLE);
    }
    if (p.trace_ctas && threadIdx.x == 0 && blockIdx.x < p.trace_ctas_cap) {
        p.trace_ctas[4 * blockIdx.x + 0] = t_entry;
        p.trace_ctas[4 * blockIdx.x + 1] = ptx::globaltimer_ns();
    }

    if (warp == 0) {
        // ================================ TMA producer ================================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t pos = 0;            // ring positions advanced (k-blocks loaded or withheld)
            int g = 0, g_fenced = -1;
            bool aborted = false;
            bool maps_ready = !Cfg::MOE;   // MoE: the per-expert maps come from the kernel before this one
            bool withhold = (p.withhold_kb >= 0) && blockIdx.x == static_cast<uint32_t>(p.withhold_block);
            Sched sc = sched_begin<Cfg>(p, unit);
            Work w;
            while (!aborted && sched_next<Cfg>(p, unit, num_units, total_tiles, sc, w)) {
                g = find_problem<Cfg>(p, w.t, g, mt);
                const Problem& pr = problem_of<Cfg>(p, g);
                if constexpr (Cfg::GROUPED) {
                    if (g != g_fenced) {
                        ptx::fence_tensormap_acquire(&pr.tma_a);
                        ptx::fence_tensormap_acquire(&pr.tma_b);
                        g_fenced = g;
                    }
                }
                const TileCoord tc = coord_of<Cfg>(p, w, g, rank, mt);
                // first B column this CTA loads (a column half: half of each CTA's share)
                const int nb0 = tc.n0 + static_cast<int>(rank) * (tc.nhalf ? Cfg::BN_CTA / 2 : Cfg::BN_CTA);
                const int b_boxes = tc.nhalf ? Cfg::BN_CTA / 128 : Cfg::BN_CTA / 64;   // N-major B: 64-column boxes
                const uint32_t item_tx = Cfg::A_BYTES + (tc.nhalf ? Cfg::B_BYTES / 2 : Cfg::B_BYTES);
                const bool b_wide = Cfg::B_MN && (pr.flags & FLAG_B_WIDE) != 0;
                const int kb_end = work_kb_end(w, pr);
                // A rows: the problem's map at row m0, or (MoE) the expert's own map at its local row
                const CUtensorMap* map_a = &pr.tma_a;
                int a_row = tc.m0;
                if constexpr (Cfg::MOE) {
                    map_a = p.moe_maps + 2 * g;
                    a_row = tc.m0 - mt.row_off[g];
                    if (!maps_ready) {
                        ptx::grid_dependency_wait();
                        maps_ready = true;
                    }
                    if (g != g_fenced) {
                        ptx::fence_tensormap_acquire(map_a);
                        g_fenced = g;
                    }
                }
                // One k-block's loads into ring stage st (ring position `at`).
                auto load_stage = [&](int st, int kb, uint32_t at) {
                    const bool skip = withhold && kb == p.withhold_kb;
                    if (!skip) {
                        const uint32_t fb = (CG == 2) ? ptx::mapa(full_bar(st), 0) : full_bar(st);
                        if (leader) ptx::mbar_arrive_expect_tx(full_bar(st), item_tx * CG);
                        const int k0 = kb * BK;
                        const uint32_t a_dst = sA + st * Cfg::A_BYTES;
                        const uint32_t b_dst = sB + st * Cfg::B_BYTES;
                        auto load = [&](uint32_t dst, const CUtensorMap* m, int x, int y) {
                            if constexpr (CG == 2) ptx::tma_load_2d_pair(dst, m, x, y, fb);
                            else ptx::tma_load_2d(dst, m, x, y, fb);
                        };
                        if constexpr (Cfg::A_MN) {
                            load(a_dst, map_a, a_row, k0);
                            load(a_dst + 8192, map_a, a_row + 64, k0);
                        } else {
                            load(a_dst, map_a, k0, a_row);
                        }
                        if constexpr (Cfg::MOE) {
                            auto load3 = [&](uint32_t dst, int x, int y) {
                                if constexpr (CG == 2) ptx::tma_load_3d_pair(dst, &pr.tma_b, x, y, tc.g, fb);
                                else ptx::tma_load_3d(dst, &pr.tma_b, x, y, tc.g, fb);
                            };
                            if constexpr (Cfg::B_MN) {
                                if (b_wide) {
                                    if constexpr (CG == 2) ptx::tma_load_4d_pair(b_dst, &pr.tma_b, 0, k0, nb0 / 64, tc.g, fb);
                                    else ptx::tma_load_4d(b_dst, &pr.tma_b, 0, k0, nb0 / 64, tc.g, fb);
                                } else {
#pragma unroll
                                    for (int j = 0; j < Cfg::BN_CTA / 64; ++j) load3(b_dst + j * 8192, nb0 + j * 64, k0);
                                }
                            } else {
                                load3(b_dst, k0, nb0);
                            }
                        } else if constexpr (Cfg::B_MN) {
                            if (b_wide && !tc.nhalf) {
                                // box {64 columns, 64 k, BN_CTA / 64 chunks}: lands as the chunks' 8 KiB blocks in order
                                if constexpr (CG == 2) ptx::tma_load_3d_pair(b_dst, &pr.tma_b, 0, k0, nb0 / 64, fb);
                                else ptx::tma_load_3d(b_dst, &pr.tma_b, 0, k0, nb0 / 64, fb);
                            } else {
                                const CUtensorMap* mb = b_wide ? &p.b_half : &pr.tma_b;
#pragma unroll
                                for (int j = 0; j < Cfg::BN_CTA / 64; ++j)
                                    if (j < b_boxes) load(b_dst + j * 8192, mb, nb0 + j * 64, k0);
                            }
                        } else if constexpr (!Cfg::GROUPED) {
                            load(b_dst, tc.nhalf ? &p.b_half : &pr.tma_b, k0, nb0);
                        } else {
                            load(b_dst, &pr.tma_b, k0, nb0);
                        }
                        st_shared_u32(base + Cfg::OFF_DRAIN_LAST + 4 * st, at);
                        st_shared_u32(base + Cfg::OFF_DRAIN_BYTES + 4 * st, item_tx);
                    }
                };
                // One or two ring stages per iteration.  A slot is refilled as soon as the
                // MMA releases it: the producer waits for this stage's slot alone (a
                // non-blocking probe first, as a blocking wait on a barrier that has already
                // completed still costs the single issuing thread ~130 cycles), then loads
                // the next stage as well if its slot is already free.  Waiting for both
                // slots before loading either, as an earlier form did, delayed every other
                // refill by a k-block of MMA work; with 6 stages the ring's round trip
                // has no slack for that (4 stages run at ~735 cycles a k-block).
                for (int kb = w.kb0; kb < kb_end;) {
                    const int last = stage + 1 == STAGES ? 0 : stage + 1;
                    const uint32_t last_phase = stage + 1 == STAGES ? phase ^ 1u : phase;
                    if (!ptx::mbar_test_wait(empty_bar(stage), phase ^ 1u) &&
                        !wait_bounded<CG>(empty_bar(stage), phase ^ 1u, p, abort_addr, ROLE_PRODUCER, w.slot, stage)) {
                        aborted = true;
                        break;
                    }
                    const bool two = kb + 1 < kb_end && ptx::mbar_test_wait(empty_bar(last), last_phase ^ 1u);
                    load_stage(stage, kb, pos);
                    if (two) load_stage(last, kb + 1, pos + 1u);
                    const int adv = two ? 2 : 1;
                    kb += adv;
                    pos += static_cast<uint32_t>(adv);
                    stage += adv;
                    if (stage >= STAGES) { stage -= STAGES; phase ^= 1u; }
                }
                withhold = false;
            }
            if (!aborted) {
                // Tail: wait until the MMA has released every slot, so no commit
                // arrives on this CTA's barriers after it leaves.
                for (int i = 0; i < STAGES; ++i) {
                    if (!wait_bounded<CG>(empty_bar(stage), phase ^ 1u, p, abort_addr, ROLE_PRODUCER, -1, stage)) {
                        aborted = true;
                        break;
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // the ring record is final (the pair's leader reads the other CTA's after an abort)
            st_shared_u32(base + Cfg::OFF_DRAIN_POS, pos);
            ptx::st_release_cluster_u32(base + Cfg::OFF_DRAIN_FLAG, 1u);
            if (aborted && leader) drain_issued_loads<Cfg>(p, base);
        }
    } else if (warp == 1) {
        // ================================ MMA issuer ================================
        // The whole warp runs the loop, converged; lane 0 alone issues the MMAs and commits.
        if (leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int g = 0;
            bool aborted = false;
            bool any_mma = false;
            // shared-memory descriptors of stage 0 (A and B)
            const uint64_t a_desc0 = Cfg::A_MN ? ptx::smem_desc_sw128(sA, 8192, 1024) : ptx::smem_desc_sw128(sA, 16, 1024);
            const uint64_t b_desc0 = Cfg::B_MN ? ptx::smem_desc_sw128(sB, 8192, 1024) : ptx::smem_desc_sw128(sB, 16, 1024);
            // Warp-uniform bounded wait: every lane polls once; if the phase is not yet
            // complete, lane 0 runs the bounded wait and tells the others how it ended.
            auto warp_wait = [&](uint32_t bar, uint32_t par, int64_t tile, uint32_t st) -> bool {
                if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, par))) return true;
                uint32_t ok = 1;
                if (lane == 0) ok = wait_bounded<CG, false>(bar, par, p, abort_addr, ROLE_MMA, tile, st) ? 1u : 0u;
                return __shfl_sync(0xffffffffu, ok, 0) != 0;
            };
            Sched sc = sched_begin<Cfg>(p, unit);
            Work w;
            while (!aborted && sched_next<Cfg>(p, unit, num_units, total_tiles, sc, w)) {
                g = find_problem<Cfg>(p, w.t, g, mt);
                const Problem& pr = problem_of<Cfg>(p, g);
                // half tiles: M = 128 for the pair (bits 24-28 of the instruction descriptor hold M >> 4)
                // column halves: N = BN/2 (bits 17-22 hold N >> 3)
                const TileCoord tcm = coord_of<Cfg>(p, w, g, rank, mt);
                uint32_t idesc = pr.idesc;
                if (tcm.half) idesc = (idesc & ~(0x1Fu << 24)) | ((128u >> 4) << 24);
                if (tcm.nhalf) idesc = (idesc & ~(0x3Fu << 17)) | ((static_cast<uint32_t>(BN / 2) >> 3) << 17);
                if (!warp_wait(tempty_bar(acc), acc_phase ^ 1u, w.slot, 16 + acc)) {
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                const int kb_begin = w.kb0;
                const int kb_end = work_kb_end(w, pr);
                const bool trace_unit = p.trace_tiles != nullptr && w.slot < p.trace_tiles_cap;
                // One ring stage per iteration: a warp-wide check of its full barrier, then the
                // stage's four MMAs and its commit from one elected lane.  The MMAs of a
                // 256 x 256 x 64 k-block take 512 tensor cycles, and the elected issue of all
                // five instructions takes fewer, so the loop keeps the pipe fed at every tile
                // width.  (With a lane-0 guard on each instruction the issue took ~365 cycles,
                // and K-major launches handled two stages per iteration to save a barrier
                // check; with the elected issue that form measured ~1 % slower at 4096^3 and
                // 3-6 % slower with N-major B.)
                auto issue_stage = [&](int st, bool first) {
                    // stage s starts s * BYTES further on: add (s * BYTES) >> 4 to the start-address field
                    const uint64_t a_desc = a_desc0 + static_cast<uint64_t>((st * Cfg::A_BYTES) >> 4);
                    const uint64_t b_desc = b_desc0 + static_cast<uint64_t>((st * Cfg::B_BYTES) >> 4);
                    // All lanes run the issue code and elect.sync picks the lane that issues
                    // (branching on the lane and reconverging each k-block left the tensor pipe
                    // idle for ~15 % of the main loop).  Step kk of the stage: K-major, the next
                    // 16 K elements are 32 bytes further along the swizzled row; MN-major, 16
                    // rows (2048 bytes) further down.
                    static_assert(BK / UMMA_K == 4, "four MMAs per ring stage");
                    constexpr uint64_t AO = Cfg::A_MN ? 2048u >> 4 : 32u >> 4;
                    constexpr uint64_t BO = Cfg::B_MN ? 2048u >> 4 : 32u >> 4;
                    ptx::mma_stage_elect<CG>(d_tmem, a_desc, a_desc + AO, a_desc + 2 * AO, a_desc + 3 * AO,
                                             b_desc, b_desc + BO, b_desc + 2 * BO, b_desc + 3 * BO, idesc,
                                             first ? 0u : 1u, empty_bar(st));
                };
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!warp_wait(full_bar(stage), phase, w.slot, stage)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    if (lane == 0 && kb == kb_begin && trace_unit) {
                        p.trace_tiles[4 * w.slot + 0] = blockIdx.x;
                        p.trace_tiles[4 * w.slot + 1] = ptx::globaltimer_ns();
                    }
                    issue_stage(stage, kb == kb_begin);
                    any_mma = true;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (aborted) break;
                if (lane == 0) {
                    if (kb_end > kb_begin) {
                        if constexpr (CG == 2) ptx::mma_commit_pair(tfull_bar(acc), 0x3);
                        else ptx::mma_commit(tfull_bar(acc));
                    } else {
                        // K == 0: nothing to accumulate; the epilogue writes epilogue(0).
                        ptx::mbar_arrive(tfull_bar(acc));
                        if constexpr (CG == 2) ptx::mbar_arrive_cluster(ptx::mapa(tfull_bar(acc), 1));
                    }
                }
                __syncwarp();
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            if (aborted && any_mma && lane == 0) {
                // Drain: one more commit completes when every MMA issued so far has.
                if constexpr (CG == 2) ptx::mma_commit_pair(drain_bar, 0x1);
                else ptx::mma_commit(drain_bar);
                if (!wait_quiet(drain_bar, 0, p.wait_budget_ns)) report_timeout(p, ROLE_DRAIN, -1, 0, p.wait_budget_ns);
            }
            __syncwarp();
        }
    } else {
        // ================================ epilogue ================================
        const int ew = warp - EPI_WARP0;                     // 0..3
        const int q = warp % 4;                              // TMEM lane quarter this warp may read
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t c_stage0 = sC + ew * 2 * C_STAGE_BYTES;
        int acc = 0;
        uint32_t acc_phase = 0;
        int sbuf = 0;
        int g = 0, g_fenced = -1;
        bool maps_ready = !Cfg::MOE;
        const uint64_t pol_c = ptx::l2_policy_evict_first();    // C is written once
        Sched sc = sched_begin<Cfg>(p, unit);
        Work w;
        while (sched_next<Cfg>(p, unit, num_units, total_tiles, sc, w)) {
            g = find_problem<Cfg>(p, w.t, g, mt);
            const Problem& pr = problem_of<Cfg>(p, g);
            // C: the problem's map, or (MoE) the expert's own map, whose rows end where its tokens do
            const CUtensorMap* map_c = Cfg::MOE ? p.moe_maps + 2 * g + 1 : &pr.tma_c;
            const int c_row_base = Cfg::MOE ? mt.row_off[g] : 0;
            if constexpr (Cfg::GROUPED || Cfg::MOE) {
                if (lane == 0 && g != g_fenced) {
                    if (!maps_ready) {
                        ptx::grid_dependency_wait();
                        maps_ready = true;
                    }
                    ptx::fence_tensormap_acquire(map_c);
                    g_fenced = g;
                }
            }
            const TileCoord tc = coord_of<Cfg>(p, w, g, rank, mt);
            // half tiles: warps q and q + 2 share rows (q % 2) * 32 .. + 32 of this CTA's 64,
            // warp q / 2 == 1 taking columns [BN/2, BN)
            const int row0 = tc.m0 + (tc.half ? (q % 2) * 32 : q * 32);
            const int col_base = tc.half ? (q / 2) * (BN / 2) : 0;
            int row_limit = pr.M;                     // rows of C this tile may write: [.., row_limit)
            if constexpr (Cfg::MOE) row_limit = static_cast<int>(min(static_cast<int64_t>(tc.row_end), p.moe_rows));
            const bool active = row0 < row_limit;
            const int epi = pr.epi;
            const bool has_acc = work_kb_end(w, pr) > w.kb0;
            const bool f16b = (pr.flags & FLAG_BIAS_F16) != 0;

            // The tile's bias, fetched before waiting for the accumulator so its latency
            // is hidden: lane l holds the 16-bit values of columns [n0 + 8 l, n0 + 8 l + 8).
            uint4 bias8 = make_uint4(0u, 0u, 0u, 0u);
            if (epi != EPI_NONE && 8 * lane < BN) {
                const int col = tc.n0 + 8 * lane;
                const uint16_t* bg = reinterpret_cast<const uint16_t*>(pr.bias) + col +
                                     (Cfg::MOE ? static_cast<int64_t>(tc.g) * pr.N : 0);
                if (col + 8 <= pr.N && (reinterpret_cast<uintptr_t>(bg) & 15u) == 0) {
                    bias8 = __ldg(reinterpret_cast<const uint4*>(bg));
                } else {
                    uint32_t h[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) h[i] = col + i < pr.N ? __ldg(bg + i) : 0u;
                    bias8 = make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
                }
            }

            uint32_t ok = 1;
            if (lane == 0) ok = wait_bounded<CG>(tfull_bar(acc), acc_phase, p, abort_addr, ROLE_EPILOGUE, w.slot, 16 + acc) ? 1u : 0u;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ptx::tc_fence_after_sync();
            __syncwarp();
            const bool tracer = p.trace_tiles && lane == 0 && ew == 0 && leader && w.slot < p.trace_tiles_cap;
            if (tracer) p.trace_tiles[4 * w.slot + 2] = ptx::globaltimer_ns();

            // RMS normalisation of A's row: one factor per accumulator row (this lane's row)
            float rs = 1.0f;
            if (pr.row_scale) {
                ptx::grid_dependency_wait();      // the factors come from the kernel launched before this one
                if (row0 + lane < row_limit) rs = pr.row_scale[row0 + lane];
            }

            const uint32_t t_acc = tmem_base + lane_off + static_cast<uint32_t>(acc * BN);
            constexpr int CHUNKS = BN / Cfg::CW;
            const int n_chunks = (tc.half || tc.nhalf) ? CHUNKS / 2 : CHUNKS;

            // accumulator columns [c * CW, (c + 1) * CW) of this lane's row; the last chunk
            // hands the TMEM buffer back to the MMA issuer
            auto read_chunk = [&](int c, float (&v)[Cfg::CW], bool release) {
                if (has_acc && active) {
                    if constexpr (Cfg::CW == 64) {
                        uint32_t r[64];
                        ptx::tmem_ld_32x32b_x64(t_acc + c * Cfg::CW, r);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
                    } else {
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32(t_acc + c * Cfg::CW, r);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < Cfg::CW; ++i) v[i] = 0.0f;
                }
                if (release && c == n_chunks - 1) {
                    ptx::tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if (CG == 2 && !leader) ptx::mbar_arrive_cluster(ptx::mapa(tempty_bar(acc), 0));
                        else ptx::mbar_arrive(tempty_bar(acc));
                    }
                }
            };

            // row scale, bias, GELU, rounding and the store of one chunk of final values
            auto finish_chunk = [&](int c, float (&v)[Cfg::CW]) {
                const int n_chunk = tc.n0 + col_base + c * Cfg::CW;
                if (!active || n_chunk >= pr.N) return;
                if (pr.row_scale) {
#pragma unroll
                    for (int i = 0; i < Cfg::CW; ++i) v[i] *= rs;
                }

                if (epi != EPI_NONE) {
                    // bias of columns [n_chunk, n_chunk + CW): 8 columns from each of CW / 8 lanes
                    auto add_bias = [&](auto f16_tag) {
                        constexpr bool F16 = decltype(f16_tag)::value;
                        auto widen = [](uint32_t h) {
                            if constexpr (F16) return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
                            else return __uint_as_float(h << 16);
                        };
#pragma unroll
                        for (int j = 0; j < Cfg::CW / 8; ++j) {
                            const int src = (col_base + c * Cfg::CW) / 8 + j;
                            const uint32_t ws[4] = {__shfl_sync(0xffffffffu, bias8.x, src),
                                                    __shfl_sync(0xffffffffu, bias8.y, src),
                                                    __shfl_sync(0xffffffffu, bias8.z, src),
                                                    __shfl_sync(0xffffffffu, bias8.w, src)};
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                float& lo = v[8 * j + 2 * h];
                                float& hi = v[8 * j + 2 * h + 1];
                                ptx::f32x2_unpack(ptx::f32x2_add(ptx::f32x2_pack(lo, hi),
                                                                 ptx::f32x2_pack(widen(ws[h] & 0xffffu), widen(ws[h] >> 16))),
                                                  lo, hi);
                            }
                        }
                    };
                    if (f16b) add_bias(std::true_type{});
                    else add_bias(std::false_type{});
                    if (epi == EPI_BIAS_GELU) {
#pragma unroll
                        for (int i = 0; i < Cfg::CW; i += 2) gelu_tanh_f32x2(v[i], v[i + 1]);
                    }
                }

                // stage: this lane's row (128 bytes) as eight 16-byte chunks, 128-byte swizzled
                const uint32_t buf = c_stage0 + sbuf * C_STAGE_BYTES;
                if (lane == 0) ptx::bulk_wait_group_read<1>();
                __syncwarp();
                const uint32_t row_addr = buf + lane * 128;
                const bool c_f16 = (pr.flags & FLAG_C_F16) != 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t w0, w1, w2, w3;
                    if constexpr (Cfg::C_F32) {
                        w0 = __float_as_uint(v[4 * j + 0]);
                        w1 = __float_as_uint(v[4 * j + 1]);
                        w2 = __float_as_uint(v[4 * j + 2]);
                        w3 = __float_as_uint(v[4 * j + 3]);
                    } else if (c_f16) {
                        w0 = pack_f16x2(v[8 * j + 0], v[8 * j + 1]);
                        w1 = pack_f16x2(v[8 * j + 2], v[8 * j + 3]);
                        w2 = pack_f16x2(v[8 * j + 4], v[8 * j + 5]);
                        w3 = pack_f16x2(v[8 * j + 6], v[8 * j + 7]);
                    } else {
                        w0 = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
                        w1 = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
                        w2 = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
                        w3 = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
                    }
                    const uint32_t dst = row_addr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                 :: "r"(dst), "r"(w0), "r"(w1), "r"(w2), "r"(w3) : "memory");
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (pr.repeat > 0) {
                        // broadcast: the same 32 user rows go to every repeat index of this replica
                        const int j0 = static_cast<int>(static_cast<int64_t>(tc.r) * pr.repeat / pr.replicas);
                        const int j1 = static_cast<int>(static_cast<int64_t>(tc.r + 1) * pr.repeat / pr.replicas);
                        for (int j = j0; j < j1; ++j) ptx::tma_store_3d(&pr.tma_c, buf, n_chunk, j, row0);
                    } else {
                        ptx::tma_store_2d_hint(map_c, buf, n_chunk, row0 - c_row_base, pol_c);
                    }
                    ptx::bulk_commit_group();
                }
                sbuf ^= 1;
            };

            if (w.slices == 0) {
#pragma unroll 1
                for (int c = 0; c < n_chunks; ++c) {
                    float v[Cfg::CW];
                    read_chunk(c, v, true);
                    finish_chunk(c, v);
                }
            } else {
                // Stream-K piece.  Each epilogue warp first arrives on the tile's counter (zeroed
                // by the kernel launched just before this one).  Every piece but the last to
                // arrive writes its 32 x BN partial sums to its own slab - float4 [column / 4]
                // [lane], so that a warp's stores are 512 contiguous bytes - and raises its ready
                // flag; the last one adds all S in k order, its own from TMEM, the others from
                // their slabs once their flags are up.  Those pieces have arrived, so they are
                // already writing and the wait ends (it is bounded all the same).
                const int S = w.slices;
                constexpr int64_t SLAB = 32 * BN;
                auto slab = [&](int slice) {
                    return reinterpret_cast<float4*>(
                        p.sk_partial + (((w.t * p.sk_max_slices + slice) * CG + rank) * 4 + q) * SLAB);
                };
                auto flag = [&](int slice) {
                    return p.sk_flag + ((w.t * p.sk_max_slices + slice) * CG + rank) * 4 + q;
                };
                uint32_t last = 0;
                if (active) {
                    if (lane == 0) {
                        ptx::grid_dependency_wait();   // the counters were zeroed by the kernel before this one
                        const int64_t idx = (w.t * CG + rank) * 4 + q;
                        last = atomicAdd(p.sk_count + idx, 1u) == static_cast<uint32_t>(S - 1) ? 1u : 0u;
                    }
                    last = __shfl_sync(0xffffffffu, last, 0);
                }
                if (!last) {
                    // write the partial sums, hand the accumulator back, then raise the flag
                    float4* mine = slab(w.slice);
#pragma unroll 1
                    for (int c = 0; c < CHUNKS; ++c) {
                        float v[Cfg::CW];
                        read_chunk(c, v, true);
                        if (active) {
#pragma unroll
                            for (int i = 0; i < Cfg::CW / 4; ++i)
                                __stcg(mine + (c * (Cfg::CW / 4) + i) * 32 + lane,
                                       make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
                        }
                    }
                    if (active) {
                        __threadfence();
                        __syncwarp();
                        if (lane == 0) ptx::st_release_gpu_u32(flag(w.slice), 1u);
                    }
                } else {
                    // the other pieces' flags (each one's partials are then visible)
                    uint32_t ok = 1;
                    if (lane == 0) {
                        const uint64_t t0 = ptx::globaltimer_ns();
                        for (int sl = 0; sl < S && ok; ++sl) {
                            if (sl == w.slice) continue;
                            while (ptx::ld_acquire_gpu_u32(flag(sl)) == 0u) {
                                const uint64_t dt = ptx::globaltimer_ns() - t0;
                                if (dt > p.wait_budget_ns || abort_raised(abort_addr)) {
                                    if (dt > p.wait_budget_ns) {
                                        report_timeout(p, ROLE_EPILOGUE, w.slot, static_cast<uint32_t>(sl), dt);
                                        raise_abort<CG>(abort_addr);
                                    }
                                    ok = 0;
                                    break;
                                }
                            }
                        }
                    }
                    __syncwarp();
                    __threadfence();
                    // the unit's last work item: its operand ring is idle from here on
                    Sched peek = sc;
                    Work after;
                    const bool unit_done = !sched_next<Cfg>(p, unit, num_units, total_tiles, peek, after);
                    if (unit_done) {
                        // The others stream through this warp's share of the operand ring - idle, as
                        // no MMA or load of this unit is left - with cp.async, FIX_BUFS chunks in
                        // flight; each lane copies and reads back only its own float4s.
                        constexpr int CH_BYTES = 32 * Cfg::CW * 4;
                        const uint32_t region = sA + static_cast<uint32_t>(q) * FIX_BUFS * CH_BYTES;
                        const int items = CHUNKS * (S - 1);      // (chunk, other piece), chunk-major
                        auto issue = [&](int k) {
                            if (k < items) {
                                const int c = k / (S - 1), j = k % (S - 1);
                                const float4* src = slab(j < w.slice ? j : j + 1) + c * (Cfg::CW / 4) * 32 + lane;
                                const uint32_t dst = region + static_cast<uint32_t>(k % FIX_BUFS) * CH_BYTES + lane * 16u;
#pragma unroll
                                for (int i = 0; i < Cfg::CW / 4; ++i) ptx::cp_async_16(dst + i * 512u, src + i * 32);
                            }
                            ptx::cp_async_commit();              // empty groups keep the count uniform
                        };
#pragma unroll 1
                        for (int k = 0; k < FIX_BUFS - 1; ++k) issue(k);
                        int k = 0;
#pragma unroll 1
                        for (int c = 0; c < CHUNKS; ++c) {
                            float v[Cfg::CW];
#pragma unroll 1
                            for (int sl = 0; sl < S; ++sl) {
                                float x[Cfg::CW];
                                if (sl == w.slice) {
                                    read_chunk(c, x, c == CHUNKS - 1);
                                } else {
                                    ptx::cp_async_wait<FIX_BUFS - 2>();   // item k has landed
                                    const uint32_t buf = region + static_cast<uint32_t>(k % FIX_BUFS) * CH_BYTES + lane * 16u;
#pragma unroll
                                    for (int i = 0; i < Cfg::CW / 4; ++i) {
                                        const float4 y = ptx::ld_shared_f4(buf + i * 512u);
                                        x[4 * i] = y.x;
                                        x[4 * i + 1] = y.y;
                                        x[4 * i + 2] = y.z;
                                        x[4 * i + 3] = y.w;
                                    }
                                    issue(k + FIX_BUFS - 1);          // into the buffer of item k - 1
                                    ++k;
                                }
                                if (sl == 0) {
#pragma unroll
                                    for (int i = 0; i < Cfg::CW; ++i) v[i] = x[i];
                                } else {
#pragma unroll
                                    for (int i = 0; i < Cfg::CW; ++i) v[i] += x[i];
                                }
                            }
                            finish_chunk(c, v);
                        }
                        ptx::cp_async_wait<0>();
                    } else {
                        // The operand ring belongs to the unit's next work item: the others come
                        // into registers, 32 columns at a time, the next (chunk, half, other piece)
                        // item always in flight while the current one is added and the chunk stored.
                        constexpr int HALVES = Cfg::CW / 32;
                        const int items = CHUNKS * HALVES * (S - 1);
                        float4 nx[8];
                        auto load_item = [&](int k) {
                            const int j = k % (S - 1), ch = k / (S - 1);
                            const float4* src = slab(j < w.slice ? j : j + 1) + ch * 8 * 32 + lane;
#pragma unroll
                            for (int i = 0; i < 8; ++i) nx[i] = __ldcg(src + i * 32);
                        };
                        load_item(0);
                        int k = 0;
#pragma unroll 1
                        for (int c = 0; c < CHUNKS; ++c) {
                            // v = sum of the pieces in k order, accumulated in place
                            float v[Cfg::CW];
#pragma unroll
                            for (int h = 0; h < HALVES; ++h) {
#pragma unroll 1
                                for (int sl = 0; sl < S; ++sl) {
                                    if (sl == w.slice) {
                                        uint32_t r[32];
                                        ptx::tmem_ld_32x32b_x32(t_acc + c * Cfg::CW + h * 32, r);
                                        ptx::tmem_ld_wait();
#pragma unroll
                                        for (int i = 0; i < 32; ++i)
                                            v[h * 32 + i] = sl == 0 ? __uint_as_float(r[i]) : v[h * 32 + i] + __uint_as_float(r[i]);
                                    } else {
#pragma unroll
                                        for (int i = 0; i < 8; ++i) {
                                            const float4 y = nx[i];
                                            v[h * 32 + 4 * i] = sl == 0 ? y.x : v[h * 32 + 4 * i] + y.x;
                                            v[h * 32 + 4 * i + 1] = sl == 0 ? y.y : v[h * 32 + 4 * i + 1] + y.y;
                                            v[h * 32 + 4 * i + 2] = sl == 0 ? y.z : v[h * 32 + 4 * i + 2] + y.z;
                                            v[h * 32 + 4 * i + 3] = sl == 0 ? y.w : v[h * 32 + 4 * i + 3] + y.w;
                                        }
                                        if (++k < items) load_item(k);
                                    }
                                }
                            }
                            if (c == CHUNKS - 1) {
                                // this piece's accumulator is fully read: hand it back
                                ptx::tc_fence_before_sync();
                                __syncwarp();
                                if (lane == 0) {
                                    if (CG == 2 && !leader) ptx::mbar_arrive_cluster(ptx::mapa(tempty_bar(acc), 0));
                                    else ptx::mbar_arrive(tempty_bar(acc));
                                }
                            }
                            finish_chunk(c, v);
                        }
                    }
                }
            }
            if (tracer) p.trace_tiles[4 * w.slot + 3] = ptx::globaltimer_ns();
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (lane == 0) ptx::bulk_wait_group<0>();
        __syncwarp();
    }

    // ---- teardown (lanes 1-31 of warps 0 and 1 wait here for their lane 0)
    __syncwarp();
    if (p.trace_ctas && warp == EPI_WARP0 && lane == 0 && blockIdx.x < p.trace_ctas_cap)
        p.trace_ctas[4 * blockIdx.x + 2] = ptx::globaltimer_ns();
    ptx::tc_fence_before_sync();
    if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after_sync();
    if (warp == 1) ptx::tmem_dealloc<CG>(tmem_base, Cfg::TMEM_COLS);
    if (p.trace_ctas && warp == 1 && lane == 0 && blockIdx.x < p.trace_ctas_cap)
        p.trace_ctas[4 * blockIdx.x + 3] = ptx::globaltimer_ns();
}

}  // namespace tg
