/*
 * tg.h - C ABI of libtg: bf16 GEMM and grouped GEMM on NVIDIA GB300 (sm_103a).
 *
 * What is computed.  C = epilogue(A . B) with bf16 (or fp16) operands, an
 * fp32 accumulator summed over K in BLOCK_K steps, and an epilogue fused into
 * the same kernel: none, + bias, or + bias then GELU(tanh).  This is the tiled
 * matmul that "How We Built TLX: A Hardware-Native GPU Compiler for Production
 * ML at Scale" uses as its running example (section "Introducing TLX": the
 * standard Triton listing fixes the arithmetic, the TLX-on-Blackwell listing
 * the producer / MMA / epilogue split), with the bias + GELU fusion of the
 * TileGym/cuTile tutorial page.  The grouped form is the MoE expert GEMM of
 * the same TLX article's third case study ("Distributed grouped GEMM for LLM
 * pre-training"): one problem per expert, ragged M, one persistent launch.
 * Around these sit a broadcast form for repeated A rows, an MoE form whose
 * token counts stay in device memory, and an RMS-normalised form (the
 * normalisation applied as a per-row factor in the epilogue).
 *
 * Where it runs.  One persistent, warp-specialised CUDA kernel on the
 * current device: a TMA producer warp fills a shared-memory ring guarded by
 * mbarriers, one thread issues tcgen05.mma into TMEM accumulators (double
 * buffered), four epilogue warps drain TMEM, apply the epilogue and store C
 * with TMA.  There is no CPU fallback and no other backend: on a device that
 * is not sm_103 every compute call fails with TG_ERR_UNSUPPORTED.
 *
 * Conventions for every entry point below.
 *  - All matrix pointers are DEVICE pointers owned by the caller; the library
 *    never frees, keeps or reallocates them.  Calls are asynchronous on
 *    `stream` (NULL = the legacy default stream) and return after enqueue;
 *    the caller keeps A, B, C and bias alive until the stream has run.
 *  - Arguments are checked on the host before anything is enqueued; a call
 *    that returns an error has launched nothing.  tg_last_error_message()
 *    describes the most recent failure on the calling thread.
 *  - TMA addressing rules: every matrix base pointer must be 16-byte aligned
 *    and every leading dimension * element size a multiple of 16 bytes
 *    (bf16: ld % 8 == 0; fp32: ld % 4 == 0).  M, N, K and leading dimensions
 *    must be below 2^31.  Breaking these gives TG_ERR_UNSUPPORTED.
 *  - Degenerate sizes: M == 0 or N == 0 is a no-op returning TG_OK.  K == 0
 *    is the empty sum: C = epilogue(0), i.e. zeros, bias, or GELU(bias).
 *  - Results are deterministic: two identical calls write bitwise-identical C.
 *    A dense call whose tiles do not divide evenly over the SMs runs the tiles
 *    of its last, partial wave in smaller units.  Tiles of at most 96 k-blocks,
 *    when there are at most half as many of them as CTA pairs, run as two
 *    128-column halves (no partial sums: bitwise equal to whole tiles).  Other
 *    last waves run as stream-K pieces: their k-blocks are cut into ranges of
 *    equal length, one per CTA pair, each run after the pair's first whole
 *    tile; the fp32 partial sums of a tile's pieces are added in k order (an
 *    atomic counter only picks which SM does the adding), so the result does
 *    not depend on timing.  TG_STREAM_K=0 in the environment runs whole tiles
 *    only (one K order per tile, as grouped calls); TG_STREAM_K=1 uses stream-K
 *    pieces where column halves would be chosen.
 *  - Dense stream-K calls take a workspace from a library-owned stream-ordered
 *    memory pool (up to 9 x 256 KiB per stream-K tile, fewer than the resident
 *    CTA pairs; released on the stream after the launch).
 */
#ifndef TG_H
#define TG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL selects the legacy default stream. */
typedef struct CUstream_st *tg_stream_t;

typedef enum {
    TG_OK = 0,
    TG_ERR_INVALID_ARG = 1,  /* null pointer, negative size, ld too small, bad enum */
    TG_ERR_UNSUPPORTED = 2,  /* alignment / size limits, or the device is not sm_103 */
    TG_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed (message has the CUDA error) */
    TG_ERR_TIMEOUT = 4,      /* a bounded in-kernel wait ran out (reported by tg_device_status) */
    TG_ERR_NO_DEVICE = 5     /* no CUDA device / driver is available */
} tg_status;

typedef enum {
    TG_EPI_NONE = 0,       /* C = A.B */
    TG_EPI_BIAS = 1,       /* C = A.B + bias[j] */
    TG_EPI_BIAS_GELU = 2   /* C = gelu_tanh(A.B + bias[j]), gelu_tanh(z) = z/2 (1 + tanh(sqrt(2/pi)(z + 0.044715 z^3))) */
} tg_epilogue;

typedef enum {
    TG_ROW_MAJOR = 0,  /* element (r, c) at p[r * ld + c] */
    TG_COL_MAJOR = 1   /* element (r, c) at p[c * ld + r] */
} tg_layout;

typedef enum {
    TG_BF16 = 0,  /* bfloat16; as output, rounded once to nearest even from the fp32 epilogue value */
    TG_F32 = 1,   /* output only: the fp32 epilogue value itself */
    TG_F16 = 2    /* IEEE binary16 (the TLX listing's type); as output, rounded once to nearest even */
} tg_dtype;

/*
 * tg_gemm - one dense GEMM, C[M,N] = epilogue(A[M,K] . B[K,N]).
 *
 *   A, layout_a, lda : bf16 M x K.  Row-major: lda >= K.  Column-major: lda >= M.
 *   B, layout_b, ldb : bf16 K x N.  Row-major: ldb >= N.  Column-major (i.e. the
 *                      N x K matrix B^T stored row-major): ldb >= K.
 *   C, c_dtype, ldc  : M x N, always row-major, ldc >= N, bf16, fp32 or fp16.
 *   epi, bias        : bias is a device bf16[N] (2-byte aligned); required for
 *                      TG_EPI_BIAS / TG_EPI_BIAS_GELU, ignored for TG_EPI_NONE.
 *   A and B may be NULL only when K == 0.  C must not overlap A, B or bias.
 *
 * Accumulation is fp32 in tensor memory; the epilogue runs in fp32 and rounds
 * once.  Each element agrees with the exact result within
 * 1e-2 * sum_k |a_ik b_kj| (+ 1e-2 |bias_j|) + 1e-5.
 *
 * Source: "How We Built TLX", section "Introducing TLX": the standard Triton
 * matmul listing (an fp32 accumulator summed over BLOCK_K steps of A and B
 * tiles) and the TLX-on-Blackwell listing (TMA loads into a barrier-guarded
 * ring, MMAs into a tensor-memory accumulator, a separate epilogue); and the
 * tile tutorial "Guide de programmation pour la programmation GPU par tuiles
 * de NVIDIA", its fused kernel that multiplies, adds a bias and applies GELU
 * in one pass.
 */
tg_status tg_gemm(const void *A, tg_layout layout_a, int64_t lda,
                  const void *B, tg_layout layout_b, int64_t ldb,
                  void *C, tg_dtype c_dtype, int64_t ldc,
                  int64_t M, int64_t N, int64_t K,
                  tg_epilogue epi, const void *bias,
                  tg_stream_t stream);

/*
 * tg_gemm_bcast - dense GEMM whose A rows are repeated: in-kernel broadcast.
 *
 * C[U * repeat, N] = epilogue(A . B) where row i * repeat + j of A (j < repeat)
 * is row i of A_user[U, K]: each user's `repeat` candidate rows are contiguous
 * in C.  This is the in-kernel broadcast of the TLX article's second case study
 * ("In-kernel broadcast optimization for RecSys"): instead of materialising the
 * repeated user rows, the kernel consumes A_user at its own batch size and
 * broadcasts inside the kernel.  Each distinct result row is computed once per
 * replica CTA and stored `repeat` times, so A costs U*K*2 bytes of traffic
 * instead of U*repeat*K*2.  Results are bitwise identical to tg_gemm on the
 * materialised A when that call runs without stream-K pieces (always with
 * TG_STREAM_K=0), and within the stated tolerance otherwise.
 *
 *   A_user, layout_a, lda : bf16 U x K (row-major: lda >= K; column-major: lda >= U).
 *   repeat                : >= 1; U * repeat < 2^31.
 *   other arguments       : as tg_gemm, with M = U * repeat rows of C (ldc >= N).
 */
tg_status tg_gemm_bcast(const void *A_user, tg_layout layout_a, int64_t lda, int64_t U, int64_t repeat,
                        const void *B, tg_layout layout_b, int64_t ldb,
                        void *C, tg_dtype c_dtype, int64_t ldc,
                        int64_t N, int64_t K,
                        tg_epilogue epi, const void *bias,
                        tg_stream_t stream);

/*
 * tg_row_rms - r[i] = 1 / sqrt((1/K) sum_k A[i][k]^2 + eps) for a row-major bf16
 * A [M, K] (lda >= K, 16-byte aligned rows); r is a DEVICE fp32 [M].  Sums run
 * in fp32 in a fixed order (deterministic).  K == 0 gives r = 1 / sqrt(eps).
 * The row statistics of the normalisation that tg_gemm_rmsnorm fuses into the
 * GEMM (same source as tg_gemm_rmsnorm).
 */
tg_status tg_row_rms(const void *A, int64_t lda, int64_t M, int64_t K, float eps, float *r, tg_stream_t stream);

/*
 * tg_gemm_rmsnorm - C = epilogue(rmsnorm(A) . B), the normalisation fused
 * into the GEMM.  Source: the Chinese rewrite of "How We Built TLX" ("Meta 造了
 * 个 Triton 扩展 TLX ..."), section on what TLX provides: because layouts are
 * inferred, a normalisation can be fused into the GEMM and the intermediate
 * round trip through memory disappears; and the companion article it lists,
 * "Achieving Free Normalization: Fusing Norms into GEMM and Attention via TLX"
 * (title only; the pages give no formula, RMS normalisation is this library's
 * reading).
 *
 * Since rmsnorm(A) = diag(r) A, the product is computed on A as stored and
 * row i of the fp32 accumulator is scaled by r_i in the epilogue, before bias
 * and GELU; the normalised A is never written or read back.  r comes from tg_row_rms
 * (one read of A) and is left in row_scale (DEVICE fp32 [M]) for reuse.  A
 * gain vector gamma folds into B: rmsnorm_gamma(A) . B = rmsnorm(A) . diag(gamma) B.
 * A is row-major bf16; other arguments as tg_gemm.  With K == 0 the result is
 * epilogue(0) (an empty row normalises to an empty row), even when eps == 0.
 */
tg_status tg_gemm_rmsnorm(const void *A, int64_t lda, const void *B, tg_layout layout_b, int64_t ldb,
                          void *C, tg_dtype c_dtype, int64_t ldc, int64_t M, int64_t N, int64_t K,
                          float eps, float *row_scale, tg_epilogue epi, const void *bias, tg_stream_t stream);

/*
 * One problem of a grouped GEMM: C_g = epilogue_g(A_g . B_g), fields as in
 * tg_gemm.  Problems are independent and may differ in every field; a problem
 * with M == 0 or N == 0 (an expert that received no tokens) is skipped and its
 * pointers may be NULL.
 */
typedef struct tg_group_problem {
    int64_t M, N, K;
    const void *A;  int64_t lda; tg_layout layout_a;
    const void *B;  int64_t ldb; tg_layout layout_b;
    void *C;        int64_t ldc; tg_dtype c_dtype;   /* TG_BF16, TG_F32 or TG_F16 */
    tg_epilogue epi;
    const void *bias;
    tg_dtype ab_dtype;  /* element type of A, B and bias: TG_BF16 (0, the default) or TG_F16 */
} tg_group_problem;

/*
 * tg_gemm_ex - one dense GEMM described by a problem record (fields as for
 * tg_gemm), which also selects fp16 operands (ab_dtype = TG_F16, the element
 * type of the TLX listing) and an fp16 output (c_dtype = TG_F16).  The record
 * is read during the call only.  Source: as tg_gemm; the fp16 element type is
 * the one the TLX-on-Blackwell listing ("How We Built TLX", section
 * "Introducing TLX") declares for its operands and output.
 */
tg_status tg_gemm_ex(const tg_group_problem *problem, tg_stream_t stream);

/*
 * tg_grouped_gemm - G independent GEMMs in one persistent launch (one launch
 * per distinct (layout_a, layout_b, c_dtype) combination present).
 *
 * Source: "How We Built TLX", case-study table (LLM pre-training row) and
 * "Case study 3: distributed grouped GEMM for LLM pre-training": the grouped
 * matrix multiplies of a mixture-of-experts layer, one GEMM per expert with a
 * ragged number of tokens (rows), run as one persistent kernel.  This call is
 * one GPU's share of that kernel; the token exchange between GPUs is not part
 * of it.
 *
 *   table : HOST array of G problems.  It is read during the call and may be
 *           reused or freed as soon as the call returns.
 *   G     : number of problems, 0 <= G <= 65536.  G == 0 is a no-op.
 *
 * The persistent tile scheduler walks the output tiles of all non-empty
 * problems in table order (prefix sums of per-problem tile counts).  The
 * library encodes per-problem TMA descriptors on the host and copies them into
 * a stream-ordered device workspace that it allocates and frees on `stream`
 * (from a library-owned memory pool); nothing outlives the launch.
 * Errors are as for tg_gemm; a bad problem g is named in the message.
 */
tg_status tg_grouped_gemm(const tg_group_problem *table, int G, tg_stream_t stream);

/* Largest number of experts tg_moe_gemm accepts (its schedule lives in shared memory). */
#define TG_MOE_MAX_EXPERTS 190

/*
 * tg_moe_gemm - MoE expert GEMM whose per-expert token counts are in DEVICE
 * memory, as a router running on the GPU produces them: no host round trip
 * (the MoE layer of the TLX article's third case study, "Distributed grouped
 * GEMM for LLM pre-training", with counts that never leave the GPU).  A
 * one-warp kernel reads the counts and writes each expert's own A and C tensor
 * maps on the device (tensormap.replace on copies of maps over all T rows); the
 * GEMM, launched as its programmatic dependent, schedules its tiles from the
 * same counts and loads and stores through those maps, so a tile that runs
 * past an expert's rows reads zeros and writes nothing beyond them.  The maps
 * take 256 bytes per expert of a stream-ordered workspace from the library's
 * memory pool, released on the stream after the launch.
 *
 *   A, lda, T, K     : bf16 [T, K] row-major; expert g owns rows
 *                      [off_g, off_g + counts[g]), off_g = counts[0] + ... + counts[g-1].
 *   B, layout_b, ldb, expert_stride, G, N :
 *                      bf16 experts; expert g's K x N matrix starts at
 *                      B + g * expert_stride (elements) and is row-major
 *                      (ldb >= N) or column-major (ldb >= K).
 *   C, c_dtype, ldc  : [T, N] row-major, same row grouping as A.
 *   counts           : DEVICE int32[G], read by the kernel.  Rows past the sum
 *                      of the counts are not written.
 *   epi, bias        : bias is bf16 [G, N] (row g for expert g).
 *
 * Limits: G <= TG_MOE_MAX_EXPERTS; TMA alignment rules as for tg_gemm;
 * expert_stride a multiple of 8 elements.  Counts that are
 * negative or sum to more than T make the launch compute nothing and
 * tg_device_status report TG_ERR_INVALID_ARG.  Results are bitwise equal to
 * tg_grouped_gemm on the same rows.
 */
tg_status tg_moe_gemm(const void *A, int64_t lda, int64_t T, int64_t K,
                      const void *B, tg_layout layout_b, int64_t ldb, int64_t expert_stride, int64_t G, int64_t N,
                      void *C, tg_dtype c_dtype, int64_t ldc,
                      const int32_t *counts, tg_epilogue epi, const void *bias,
                      tg_stream_t stream);

/*
 * Largest number of non-empty problems tg_grouped_gemm_noalloc accepts in one
 * call: the size of its fixed device-side problem table.
 */
#define TG_NOALLOC_MAX_PROBLEMS 256

/*
 * tg_grouped_gemm_noalloc - tg_grouped_gemm for callers that may not allocate.
 *
 * The pages have no counterpart for this entry point; it exists for callers
 * that must not allocate device memory once running (serving loops that
 * reserve everything up front so a request can never stall or fail on an
 * allocation, or programs whose device memory sits under another allocator's
 * fixed budget).  It computes exactly what tg_grouped_gemm computes, with the
 * same arguments, but calls no cudaMalloc, cudaFree or other allocating
 * routine: the per-problem descriptors go into a fixed 128 KiB table compiled
 * into the library (held on every GPU that loads libtg until process exit).
 *
 *   - At most TG_NOALLOC_MAX_PROBLEMS non-empty problems per call; more gives
 *     TG_ERR_UNSUPPORTED (split the call, or use tg_grouped_gemm).
 *   - The first call on each device looks up the table's device address
 *     (cudaGetSymbolAddress) once; make that first call before any stream
 *     capture on that device.
 *   - Every call reuses the same table.  Calls ordered on one stream are safe;
 *     calls that overlap on the GPU (different streams without ordering) race
 *     and may compute with another call's descriptors.
 */
tg_status tg_grouped_gemm_noalloc(const tg_group_problem *table, int G, tg_stream_t stream);

/*
 * tg_status_string - static English description of a status code (never NULL;
 * an unknown code gives "unknown status").
 *
 * Source: "How We Built TLX", section "Lessons: advice for building a GPU
 * compiler", point "The compiler is part of the user interface": error
 * messages and debugging support weigh as much as the quality of the generated
 * code, because the engineer chasing a utilisation or synchronisation problem
 * needs plain feedback.  Every entry point therefore returns a status code
 * with a fixed meaning, and tg_last_error_message adds the detail.
 */
const char *tg_status_string(tg_status status);

/*
 * tg_last_error_message - what the most recent failing call on the calling
 * thread found (argument check, CUDA error or in-kernel timeout), naming the
 * offending value or problem index.  Same source as tg_status_string.  The
 * string is owned by the library and valid until the thread's next libtg
 * call; it is empty if no call has failed yet.
 */
const char *tg_last_error_message(void);

/*
 * tg_device_status - synchronise `stream`, then read and clear the current
 * device's error record.
 *
 * Source: "How We Built TLX", "Case study 3": at the scale of weeks-long
 * pre-training runs, reliability and debuggability count as much as peak
 * throughput; and the Chinese rewrite of the same article ("Meta 造了个 Triton
 * 扩展 TLX ..."), editor's commentary, third point: a hung warp-specialised
 * mega-kernel is hard to locate, so hang detection belongs in the test setup
 * before such a kernel is adopted.  Here every in-kernel wait is bounded and
 * its expiry is recorded on the device and reported by this call, which
 * allocates nothing.
 *
 * Returns TG_OK, TG_ERR_CUDA (the stream reported a
 * CUDA error), TG_ERR_INVALID_ARG (tg_moe_gemm found invalid device counts),
 * or TG_ERR_TIMEOUT (a kernel's bounded mbarrier wait ran out:
 * the kernel recorded the role, tile and stage, stopped, drained its own
 * in-flight copies and MMAs, freed its tensor memory and returned; the context
 * stays usable).  The record is per device and shared by all streams.
 */
tg_status tg_device_status(tg_stream_t stream);

/*
 * Wait budget of every in-kernel mbarrier wait, in milliseconds (default 1000,
 * or the TG_WAIT_BUDGET_MS environment variable read at the first call).
 * Applies to launches made after the call.  0 restores the default.
 */
tg_status tg_set_wait_budget_ms(uint32_t ms);

/*
 * Test hooks for the failure path.  The next launch made by this thread has
 * the TMA producer of CTA `block` (blockIdx.x; 0 for tg_debug_withhold_stage)
 * withhold the arrival and the loads for the k-block with index `k_block` of
 * its first work item (a k-block of a tile, counted from the tile's first), so
 * that a bounded wait on that stage runs out (in a CTA pair the MMA issuer of
 * the pair's first CTA waits for both CTAs' loads) and tg_device_status
 * reports TG_ERR_TIMEOUT.  -1 (the default) disables it; the hook disarms
 * itself after one launch.  Nothing faults: after the timeout the kernel waits
 * for the loads that were issued and returns.
 */
tg_status tg_debug_withhold_stage(int64_t k_block);
tg_status tg_debug_withhold_stage_in(int64_t k_block, int32_t block);

/*
 * Timeline trace of the next launch made by this thread (a profiling aid; off
 * by default, disarms itself after one launch).  Both buffers are DEVICE
 * memory owned by the caller; the kernel writes, with %globaltimer nanosecond
 * stamps:
 *   tile_records[4 s .. 4 s + 3] for work slot s < tile_capacity:
 *       {block index, first k-block ready for the MMA, accumulator complete,
 *        epilogue done}.  A work item is a tile, or one stream-K piece (a
 *       k-block range) of a tile; the i-th item of CTA (pair) u of U has slot
 *       i * U + u, so a unit with fewer items leaves its later slots untouched;
 *   cta_records[4 b .. 4 b + 3] for block b < cta_capacity:
 *       {kernel entry, set-up done, teardown start, exit}.
 * Capacities may be 0 to skip a buffer.  Grouped calls with several layout
 * classes trace only their first launch.
 */
tg_status tg_debug_trace(uint64_t *tile_records, int64_t tile_capacity,
                         uint64_t *cta_records, int64_t cta_capacity);

/* Library version as (major << 16) | minor. */
uint32_t tg_version(void);

/*
 * Number of CUDA kernels the calling thread has enqueued through libtg since
 * the library was loaded (GEMM launches and the small kernels some calls run
 * before them: the row statistics of tg_gemm_rmsnorm, the counter reset of a
 * dense stream-K launch).  Benchmarks report the difference over a timed region.
 */
uint64_t tg_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* TG_H */
