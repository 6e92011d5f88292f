/*
 * sdt.h -- C ABI of the shape-driven-tile library (libsdt.so) for GB300 (sm_103a).
 *
 * Two compute calls and the tile-selection calls around them:
 *
 *   gemm_f16   C = A . B, fp16 in, fp32 accumulate, fp16 out, with the CTA tile
 *              chosen from the problem shape.
 *   gemv_m1    y = W . x for a single activation row (M = 1 decode), streaming a
 *              K-major weight matrix, bf16 or q8 (int8 + one fp16 scale per 32).
 *
 * Conventions for every call in this header:
 *  - Pointers named A, B, C, x, W, scales, y are DEVICE pointers owned by the
 *    caller (typically PyTorch-allocated).  The library never frees, keeps or
 *    allocates device memory for them; it allocates no device memory at all.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream) owned by the
 *    caller.  Work is enqueued on it asynchronously; the library never
 *    synchronises on the hot path.  Kernel faults surface on the caller's next
 *    synchronising CUDA call, as with any CUDA kernel.
 *  - Layouts are tight row-major: A is MxK (row stride K), B is KxN (row stride
 *    N), C is MxN (row stride N).  W is [N][K] ("K-major": each output's K
 *    weights are contiguous), scales are [N][K/32].
 *  - Return value: SDT_OK (0) or a negative sdt_status.  Argument errors are
 *    detected on the host before anything is enqueued; the message of the last
 *    failure on the calling thread is available from sdt_last_error().
 *
 * Sources (the pages this library restates; cited by title and section):
 *  [P1] "Beating hipBLASLt on a Gaming GPU" -- sections "The result" (the
 *       pipelined fp16 GEMM) and "The part that actually mattered" (tile
 *       geometry chosen from how many blocks the grid yields).
 *  [P2] "mojo-baro" -- "Four rounds on the decode shape" (M=1, K=4096,
 *       N=12288 decode; K-major weights; q8 with a scale per 32 weights;
 *       several contiguous columns per thread with wide loads; an
 *       M=1-specialised kernel).
 *  [P3] FlyDSL pull request "Speed up the RDNA3 GEMM up to 1.85x by choosing
 *       the tile from the shape" -- "Changes" (pick_tile over feasible_tiles,
 *       opt-in measured sweep frozen into an artefact, k-loop start stagger with
 *       mask wraparound for power-of-two k-tile counts) and the third commit
 *       message (the K-scan that isolates power-of-two row strides).
 *  [P4] "Iteratively Tuning hipBLASLt TensileLite Kernels" -- "The Six Rounds"
 *       (split-K with a choice of reduction algorithm; workgroup mapping).
 */
#ifndef SDT_H
#define SDT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; declared here so this header needs no CUDA headers. */
typedef struct CUstream_st *sdt_stream_t;

typedef enum sdt_status {
    SDT_OK = 0,
    SDT_ERR_NULL = -1,               /* a required pointer is NULL */
    SDT_ERR_ALIGN = -2,              /* a pointer is not 16-byte aligned */
    SDT_ERR_SHAPE = -3,              /* negative dims, no feasible tile, N or K not a multiple of 8,
                                        q8 with K not a multiple of 32 */
    SDT_ERR_UNSUPPORTED_DEVICE = -4, /* current device is not compute capability 10.3 (sm_103) */
    SDT_ERR_LAUNCH = -5,             /* the kernel launch was rejected by the CUDA runtime */
    SDT_ERR_TIMEOUT = -6,            /* a kernel gave up a bounded wait (read by sdt_check_device_status) */
    SDT_ERR_TILE = -7,               /* unknown tile id, or the forced tile is infeasible for the shape */
    SDT_ERR_TABLE = -8,              /* tune table could not be read or parsed */
    SDT_ERR_CUDA = -9,               /* another CUDA runtime / driver call failed */
    SDT_ERR_ARG = -10                /* another invalid argument (e.g. stagger value) */
} sdt_status;

/* ------------------------------------------------------------------------ */
/* Core calls                                                                */
/* ------------------------------------------------------------------------ */

/*
 * gemm_f16 -- C[M][N] = A[M][K] . B[K][N]; fp16 (IEEE binary16) operands,
 * fp32 accumulation on the tensor cores, C rounded to fp16 (nearest even).
 * [P1 "The result"; P3 "Changes"].
 *
 * The tile is the tune-table entry for (M,N,K) when one is loaded and
 * feasible, otherwise sdt_pick_tile(M,N,K).  With SDT_AUTOTUNE=1 in the
 * environment, the first call for a shape times every feasible tile on
 * `stream` (synchronising it) and remembers the fastest for later calls.
 * The k-loop stagger follows SDT_STAGGER: "auto" (default) staggers the
 * one-CTA tiles when the k-tile count is a power of two and leaves the
 * persistent and two-CTA tiles unstaggered (measured faster on GB300); "0" and
 * "1" force it off or on.
 *
 * Requirements: A, B, C 16-byte aligned; M, N, K >= 0.  M == 0 or N == 0 is a
 * no-op; K == 0 writes C = 0.  Otherwise some tile must divide the shape
 * (M % 64, N % 64, K % 64 == 0 and K >= 128 at the least) or SDT_ERR_SHAPE is
 * returned; shapes with ragged edges are not handled.
 */
int gemm_f16(int64_t M, int64_t N, int64_t K,
             const void *A, const void *B, void *C, sdt_stream_t stream);

/*
 * gemv_m1 -- y[n] = sum_k x[k] * W[n][k] for n < N  (M = 1 decode).
 * [P2 "Four rounds on the decode shape", rounds v1-v4].
 *
 *   x       bf16 [K]
 *   W       scales == NULL: bf16 [N][K];  scales != NULL: int8 [N][K] (q8)
 *   scales  NULL, or fp16 [N][K/32]: weight k of row n is
 *           q[n][k] * scales[n][k/32]; the scale multiplies each group sum.
 *   y       fp32 [N] (written, not accumulated into)
 *
 * Requirements: x, W, y 16-byte aligned (scales 2-byte aligned); K a
 * multiple of 8 (bf16) or 32 (q8); K, N <= 2^30.  N == 0 is a no-op; K == 0
 * writes y = 0.
 *
 * Launched with programmatic dependent launch, the kernel may start while the
 * previous kernel in `stream` is still running; before it waits for that
 * kernel it only asks L2 for the first rows of W (a prefetch, which cannot
 * observe stale data: L2 is where device memory is coherent), so results still
 * reflect everything the previous kernel wrote to x, W and scales.  q8 sums
 * each group exactly in int32 after scaling the group's activations to int16
 * by a power of two (exact for activations within a factor 2^7 of the group's
 * largest; otherwise off by at most 2^-15 of it).
 */
int gemv_m1(int64_t K, int64_t N, const void *x, const void *W,
            const void *scales, float *y, sdt_stream_t stream);

/* The two arms of gemv_m1 called explicitly (same contract; the q8 arm requires scales). */
int gemv_m1_bf16(int64_t K, int64_t N, const void *x, const void *W, float *y,
                 sdt_stream_t stream);
int gemv_m1_q8(int64_t K, int64_t N, const void *x, const void *W,
               const void *scales, float *y, sdt_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Tile ladder, feasibility and selection  [P3 "Changes"; P1 tile rule]      */
/* ------------------------------------------------------------------------ */

/* Static description of one tile of the ladder. */
typedef struct sdt_tile_desc {
    int id;           /* index into the ladder, 0 .. sdt_num_tiles()-1 */
    int BM, BN, BK;   /* output rows x columns covered (by the CTA pair when cta_group == 2), k-depth */
    int cta_group;    /* 1, or 2 for a two-CTA (cluster pair) tile */
    int stages;       /* depth of the shared-memory TMA/MMA ring */
    int threads;      /* threads per CTA */
    int smem_bytes;   /* dynamic shared memory per CTA, including alignment slack */
    int tmem_cols;    /* tensor-memory columns allocated per CTA */
    char name[24];    /* e.g. "128x256", "2cta_256x128" */
} sdt_tile_desc;

/* The ladder also holds "skinny" tiles, named s<BM>x<BN> (s128x16, s128x32), for
 * problems with few rows (M up to a few tens): gemm_ex and gemm_ex_splitk run
 * them on C^T = op(B)^T . op(A)^T so that the many output columns fill the MMA's
 * 128 rows, and write C back transposed.  They need A stored M x K (K
 * contiguous); sdt_feasible_tiles, pick_tile, gemm_f16, gemm_f16_splitk and the
 * tune table never use them. */
int sdt_num_tiles(void);
/* Fills *out for tile `tile_id`; SDT_ERR_TILE for an unknown id, SDT_ERR_NULL for out == NULL. */
int sdt_tile_info(int tile_id, sdt_tile_desc *out);
/* Static name of a tile, or NULL for an unknown id. */
const char *sdt_tile_name(int tile_id);

/*
 * Feasible tiles for (M,N,K) [P3 "Changes"]: a tile is feasible when it
 * (i) divides the shape (BM | M, BN | N, BK | K), (ii) can fill the pipeline
 * (at least two k-tiles), (iii) fits on chip (its shared memory within
 * `smem_limit` bytes per block, its accumulator within 512 TMEM columns).
 * Writes up to `cap` tile ids in ladder order to `ids` (may be NULL when
 * cap == 0) and returns how many tiles are feasible (which may exceed cap),
 * or a negative status.  The `_for` form needs no GPU; the plain form uses
 * the current device's opt-in shared-memory limit.
 */
int sdt_feasible_tiles_for(int64_t M, int64_t N, int64_t K, int smem_limit,
                           int *ids, int cap);
int sdt_feasible_tiles(int64_t M, int64_t N, int64_t K, int *ids, int cap);

/*
 * pick_tile [P3 "Changes"; P1 "The part that actually mattered"]: the
 * heuristic tile for (M,N,K) on a GPU with `sm_count` SMs, chosen among the
 * feasible tiles by an estimate of each one's run time: the waves (or, for
 * the persistent and two-CTA tiles, the rounds per worker) its grid makes on
 * `sm_count` SMs, priced by per-tile launch, k-tile, per-round, operand
 * streaming and co-residency costs fitted to a measured sweep.  Needs no GPU
 * and measures nothing.  Returns a tile id, or SDT_ERR_SHAPE when no tile is
 * feasible.
 * The plain form reads the current device's SM count and shared-memory limit.
 */
int sdt_pick_tile_for(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit);
int sdt_pick_tile(int64_t M, int64_t N, int64_t K);

/*
 * The launcher rule of [P1 "The part that actually mattered"] as printed for
 * a 96-unit card and scaled to `units`: count the 128x128-equivalent blocks
 * (M/128)*(N/128); >= units -> the 128x128 tile, >= 2*units/3 -> 64x128,
 * else 64x64.  Returns that tile's id (the seed the fitted heuristic grew
 * from; kept for comparison).
 */
int sdt_seed_tile(int64_t M, int64_t N, int units);

/*
 * gemm_f16 with a forced tile (for sweeps).  `stagger`: -1 = as gemm_f16
 * (SDT_STAGGER / auto), 0 = off, 1 = on when the k-tile count is a power of
 * two (otherwise silently off) [P3 "Changes", third commit message].
 * SDT_ERR_TILE if the tile is unknown or infeasible for the shape.
 */
int gemm_f16_with_tile(int64_t M, int64_t N, int64_t K,
                       const void *A, const void *B, void *C, sdt_stream_t stream,
                       int tile_id, int stagger);

/*
 * gemm_ex -- the general form: caller row strides, transposed operands, bf16,
 * and shapes no tile divides [P3 "Changes": the row strides are taken from the
 * caller's tensors; the measured layouts are TN and NN; P3 "Performance" runs
 * bf16].  C[M][N] (row stride ldc) = op(A) . op(B) with fp32 accumulation:
 *   op(A): layout without SDT_LAYOUT_A_T: A is M x K row-major (lda >= K);
 *          with it, A is stored K x M (lda >= M), i.e. A^T is given.
 *   op(B): without SDT_LAYOUT_B_T: B is K x N row-major (ldb >= N);
 *          with it, B is stored N x K (ldb >= K), i.e. B^T is given ("TN" is
 *          SDT_LAYOUT_B_T: C = A . (B^T)^T).
 *   dtype: SDT_DTYPE_F16 or SDT_DTYPE_BF16 for A, B and C alike.
 * Any M, K >= 0; N a multiple of 8; lda, ldb, ldc multiples of 8 (16-byte
 * rows) at least the row lengths above; pointers 16-byte aligned.  Tiles
 * overhang ragged edges: the TMA reads zeros outside the operands and the
 * epilogue writes only inside C.  tile_id -1 picks with sdt_pick_tile_any_for's
 * model; a forced tile needs only to fit on chip.  The k-loop stagger follows
 * SDT_STAGGER as in gemm_f16.  Errors: SDT_ERR_SHAPE (N % 8, dims > 2^30),
 * SDT_ERR_ARG (strides, dtype, layout), SDT_ERR_ALIGN, SDT_ERR_NULL,
 * SDT_ERR_TILE.
 */
#define SDT_DTYPE_F16 0
#define SDT_DTYPE_BF16 1
#define SDT_LAYOUT_A_T 1
#define SDT_LAYOUT_B_T 2
int gemm_ex(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
            void *C, int64_t ldc, int dtype, int layout, int tile_id, sdt_stream_t stream);
/*
 * gemm_f16_ws / gemm_ex_ws -- gemm_f16 / gemm_ex with a caller workspace that lets
 * the two-CTA tiles split the contraction of their last round [P3, third commit
 * message: persistent workgroups and the grid tail when the tile count is not a
 * multiple of the slot count; P4 "The Six Rounds": splitting the contraction, and
 * Stream-K's decomposition of the iteration space, of which this is the special case
 * "whole tiles, then the last partial wave split in K"].
 *
 * A two-CTA launch runs T output tiles on P = SMs/2 pairs.  When L = T mod P tiles
 * are left for a last round (P - L pairs idle), each of them may run as S full-width
 * items over consecutive k-ranges (L*S <= P, 2 <= S <= nK) instead of gemm_f16's form
 * (whole, or two half-width items).  Split 0 takes the first k-tiles and is made
 * longer than the others (sdt_pair_tail_plan's split0_ktiles) so that it normally
 * finishes last.  An item that finishes while another split is still running writes
 * its fp32 partial to the workspace and counts its arrival; the last to finish adds
 * the S partials in split order (so the result does not depend on the order of
 * arrival) and writes C.  The form is chosen per launch by a cost estimate (on GB300
 * it splits at 4096^3 and above and keeps the half-width items at 2560^3, where 40
 * k-tiles leave too little to hide the sum); gemm_ex_ws's tail_splits forces it: -1
 * estimate, 0 never split, 2..8
 * that count (lowered to what L*S <= P, nK and the shared memory for the partials'
 * copies allow: at most 7 with the current tiles; below 2 it is not split).
 * Every other tile, and a launch with no partial last round, runs exactly as
 * gemm_f16 / gemm_ex would.  Results may differ from gemm_f16's in the last bits
 * (the split tiles add their k-ranges in another order); integer-valued products
 * are identical.
 *
 * Workspace: NULL runs exactly gemm_f16 / gemm_ex.  Otherwise device memory owned
 * by the caller, 256-byte aligned, at least sdt_gemm_workspace_bytes() bytes (the
 * 1 MiB counter region of the split-K workspaces, then one 256 x 256 fp32 slot per
 * SM pair: 20 MiB on a 152-SM GPU, for any shape).  Its counters must be zero before
 * the first call (sdt_splitk_workspace_init); every completed call leaves them zero,
 * so a workspace zeroed once serves any sequence of calls, and it may be shared with
 * the split-K calls.  Calls that share a workspace must not overlap on the GPU.
 * After a call that reported a device error (sdt_check_device_status), zero it again.
 * Arguments and errors otherwise as gemm_f16 / gemm_ex, plus SDT_ERR_ALIGN and
 * SDT_ERR_ARG for the workspace and SDT_ERR_ARG for tail_splits outside -1, 0, 2..8.
 */
int gemm_f16_ws(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C, void *workspace,
                size_t workspace_bytes, sdt_stream_t stream);
int gemm_ex_ws(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
               void *C, int64_t ldc, int dtype, int layout, int tile_id, int tail_splits, void *workspace,
               size_t workspace_bytes, sdt_stream_t stream);
/* Workspace bytes gemm_f16_ws / gemm_ex_ws accept on the current device (0 on error),
 * and on a GPU with sm_count SMs (needs no GPU). */
size_t sdt_gemm_workspace_bytes(void);
size_t sdt_gemm_workspace_bytes_for(int sm_count);
/*
 * The last-round plan of two-CTA tile `tile_id` on M x N x K with sm_count SMs and
 * smem_limit bytes of shared memory per block (needs no GPU): items [0, *tail_start)
 * are whole tiles, items [*tail_start, *num_items) the last round's, as *splits
 * k-ranges per tile (*splits >= 2; split 0 has *split0_ktiles k-tiles, the others
 * share the rest evenly) or two half-width items per tile (*splits == 0,
 * *num_items > *tail_start); *tail_start == *num_items means whole tiles throughout.
 * with_workspace != 0 plans as gemm_ex_ws with `tail_splits`, 0 as gemm_ex.
 * SDT_ERR_TILE for a tile that is not two-CTA, SDT_ERR_ARG for bad sizes.
 */
int sdt_pair_tail_plan(int64_t M, int64_t N, int64_t K, int tile_id, int sm_count, int smem_limit,
                       int with_workspace, int tail_splits, int *tail_start, int *num_items, int *splits,
                       int *split0_ktiles);
/* pick_tile's cost model over every tile for any shape (tiles may overhang); needs no GPU. */
int sdt_pick_tile_any_for(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit);
/*
 * The run-time estimate (microseconds) pick_tile gives tile `tile_id` on an M x N x K
 * problem with `sm_count` SMs (228 KiB of shared memory per SM), whether or not the
 * tile divides the shape or is a candidate; a negative status (SDT_ERR_TILE, SDT_ERR_ARG)
 * for an unknown tile or a dimension outside 1..2^30.  Needs no GPU.
 */
double sdt_tile_estimate_us(int tile_id, int64_t M, int64_t N, int64_t K, int sm_count);

/*
 * Split-K [P4 "The Six Rounds", the "Split-K" step: the contraction is split
 * across CTAs and the partial results are reduced; the page distinguishes a
 * reduction in a separate pass from one inside the single kernel].
 *
 * Output tile t of a one-CTA-per-tile ladder rung (64x64, 64x128, 128x64,
 * 128x128, 128x256) is computed by `splits` CTAs, CTA s accumulating k-tiles
 * [s*ceil(nK/splits), ...) (nK = K/64) and writing an fp32 partial tile to the
 * caller's workspace; the partials are summed in split order (independent of
 * arrival order) and rounded once to fp16:
 *   SDT_SPLITK_REDUCE_KERNEL  a second kernel sums the partials;
 *   SDT_SPLITK_IN_KERNEL      the last CTA of each tile to finish (per-tile
 *                             arrival counter in the workspace) sums them and
 *                             resets its counter to zero.
 * `splits` is rounded down to the count that leaves no split empty.
 * tile_id < 0 picks tile and splits with sdt_pick_splitk_for (then splits <= 0
 * takes the picked count).  The k-loop stagger is not applied.
 *
 * Workspace: device memory owned by the caller, 256-byte aligned, at least
 * sdt_splitk_workspace_bytes(M,N,K,tile_id,splits) bytes: a fixed 1 MiB region
 * of u32 counters (the in-kernel reduction uses one per output tile, at most
 * 262144 tiles; stream-K one per tile and TMEM lane quarter), then fp32
 * partials [splits][M][N].  The counter region has the same place and size in
 * every configuration.  The counters must be zero before the first SDT_SPLITK_IN_KERNEL call on a
 * workspace (sdt_splitk_workspace_init zeroes a workspace on `stream`); every
 * completed call leaves them zero again and writes partials only after the
 * counter region, so a workspace zeroed once serves any sequence of split-K
 * calls (any shape, tile, split count or algorithm) that fit in it.  Calls that
 * share a workspace must not overlap on the GPU.  Same operand requirements as gemm_f16 (tight row-major,
 * 16-byte aligned; tile dims divide M, N; K % 64 == 0).
 * Errors: SDT_ERR_TILE (tile without split-K form or not dividing the shape),
 * SDT_ERR_ARG (splits out of 1..nK, unknown algo, workspace too small),
 * SDT_ERR_ALIGN, SDT_ERR_NULL, as well as gemm_f16's.
 */
#define SDT_SPLITK_REDUCE_KERNEL 0
#define SDT_SPLITK_IN_KERNEL 1
#define SDT_SPLITK_STREAM 2        /* stream-K, fix-up by the last CTA to arrive; see sdt_streamk_workspace_bytes */
#define SDT_SPLITK_STREAM_REDUCE 3 /* stream-K, fix-up by a second kernel over the whole GPU */
int gemm_f16_splitk(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C,
                    void *workspace, size_t workspace_bytes, int tile_id, int splits, int algo,
                    sdt_stream_t stream);
/* Bytes of workspace gemm_f16_splitk needs (0 for an invalid combination, including a
 * dimension above 2^30 or more than 2^30 - 1 output tiles, which the launch refuses). */
size_t sdt_splitk_workspace_bytes(int64_t M, int64_t N, int64_t K, int tile_id, int splits);
/* Zero a split-K workspace on `stream` (its counters must start at zero). */
int sdt_splitk_workspace_init(void *workspace, size_t workspace_bytes, sdt_stream_t stream);
/*
 * Heuristic (tile, splits) for split-K on a GPU with `sm_count` SMs: the
 * pick_tile cost model with K shared among the splits plus the reduction's
 * fp32 traffic, minimised over the split-K tiles and 1..32 splits.  splits == 1
 * means splitting does not pay.  Needs no GPU.
 */
int sdt_pick_splitk_for(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit,
                        int *tile_id, int *splits);

/*
 * gemm_ex_splitk -- split-K in gemm_ex's general form [P4 "The Six Rounds",
 * the split-K step, with the operands of P3 "Changes"]: caller row strides, either
 * transposed operand, fp16 or bf16, and shapes no tile divides.  Arguments and
 * requirements as gemm_ex, plus the split-K arguments of gemm_f16_splitk.
 * The partial planes cover whole tiles: the 1 MiB counter region, then [splits][ceil(M/BM)*BM][ceil(N/BN)*BN] fp32; the
 * workspace (shareable with gemm_f16_splitk calls) must hold
 * sdt_splitk_ex_workspace_bytes(M,N,K,tile_id,splits) bytes (256-byte
 * aligned; counters zero before the first SDT_SPLITK_IN_KERNEL call, as for
 * gemm_f16_splitk).  The reduction writes only inside C (row stride ldc), in
 * the operands' type.  tile_id < 0 picks with sdt_pick_splitk_any_for (then
 * splits <= 0 takes the picked count).  Errors as gemm_ex and gemm_f16_splitk.
 */
int gemm_ex_splitk(int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
                   void *C, int64_t ldc, int dtype, int layout, void *workspace, size_t workspace_bytes,
                   int tile_id, int splits, int algo, sdt_stream_t stream);
/* Bytes of workspace gemm_ex_splitk needs for any shape (0 for a tile without split-K form,
 * splits outside 1..ceil(K/64), a dimension outside 1..2^30, or more than 2^30 - 1 output
 * tiles: the shapes the launch refuses). */
size_t sdt_splitk_ex_workspace_bytes(int64_t M, int64_t N, int64_t K, int tile_id, int splits);
/*
 * Stream-K [P4 "The Six Rounds", the last round "Stream-K": a fixed grid of
 * workgroups shares the whole iteration space instead of the contraction being
 * split per tile; a workgroup's share may end inside an output tile, and the
 * partial tiles are fixed up afterwards].  algo = SDT_SPLITK_STREAM in
 * gemm_f16_splitk / gemm_ex_splitk, with `splits` read as the CTA count G
 * (<= 0: one CTA per SM slot, sdt_streamk_ctas; lowered to the unit count when
 * larger).  The units are (output tile, 64-deep k-tile) pairs, tiles in banded
 * raster order and k-tiles in order; CTA g takes units
 * [floor(g*U/G), floor((g+1)*U/G)).  Whole tiles are stored directly; a CTA's
 * first and last tile may be partial: it writes an fp32 partial tile to its
 * slots (2g, 2g+1) and counts its arrival on per-(tile, TMEM lane quarter)
 * counters; the last CTA to arrive sums the tile's partials in CTA order,
 * writes C and zeroes the counter (SDT_SPLITK_STREAM), or a second kernel sums
 * every shared tile's partials in the same order (SDT_SPLITK_STREAM_REDUCE; the
 * counters are not used).  Same tiles as split-K (the one-CTA rungs
 * and the skinny tiles), any shape and layout gemm_ex takes.
 * Workspace: the 1 MiB counter region shared with split-K (zero before the
 * first call, left zero by every completed call), then 2*G fp32 tiles of
 * BM x BN: sdt_streamk_workspace_bytes(M,N,K,tile_id,G) bytes (G >= 1, taken
 * as at most the unit count; 0 for
 * a tile without stream-K form, a dimension outside 1..2^30, more than 65536
 * output tiles or more than 2^20 CTAs).
 */
size_t sdt_streamk_workspace_bytes(int64_t M, int64_t N, int64_t K, int tile_id, int ctas);
/* Default stream-K CTA count of a tile: SMs x CTAs of its kernel per SM (needs no GPU). */
int sdt_streamk_ctas_for(int tile_id, int sm_count, int smem_limit);
/* The same on the current device. */
int sdt_streamk_ctas(int tile_id);
/* sdt_pick_splitk_for's model over the split-K tiles for any shape (tiles may overhang). */
int sdt_pick_splitk_any_for(int64_t M, int64_t N, int64_t K, int sm_count, int smem_limit,
                            int *tile_id, int *splits);

/*
 * gemm_f16_splitk_noalloc -- gemm_f16_splitk (SDT_SPLITK_REDUCE_KERNEL) with its
 * workspace in a fixed 16 MiB array that the library holds in device memory,
 * so the call allocates nothing.  The pages have no counterpart; this is an
 * interface for callers that cannot allocate device memory where they
 * multiply: code that must not synchronise the device (cudaMalloc and
 * cudaFree can), plugin hosts that give a kernel library a fixed memory
 * budget and no allocator, latency-critical loops that forbid allocator calls.
 *
 * Arguments as gemm_f16_splitk, minus the workspace and the algorithm
 * (tile_id < 0 picks tile and splits).  The array holds the workspace layout
 * of gemm_f16_splitk: the 1 MiB counter region, then the fp32 partials, so
 * the partials get 15 MiB (sdt_splitk_workspace_bytes must be at most 16 MiB:
 * e.g. 1024x1024 with 3 splits, 512x512 with 15).  A given split count whose
 * workspace exceeds that is rejected with SDT_ERR_ARG and a message naming
 * the sizes; a split count the call picks itself (tile_id < 0, splits <= 0)
 * is lowered until it fits, and only a shape that does not fit unsplit is
 * rejected.  K == 0 writes C = 0 whatever tile and splits say.  The first
 * call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every GPU on which the library's module holding
 * the array is loaded keeps the 16 MiB until the process exits.  All calls
 * share the array: nothing in it has to start at zero (each call overwrites
 * the partials it reads), but calls that overlap on the GPU race on it and
 * corrupt each other's results.
 */
int gemm_f16_splitk_noalloc(int64_t M, int64_t N, int64_t K, const void *A, const void *B, void *C,
                            int tile_id, int splits, sdt_stream_t stream);

/*
 * Frozen tune table [P3 "Changes": the measured sweep can be frozen into an
 * offline artefact].  Text file, one entry per line: "M N K tile_name
 * [stagger]"; '#' starts a comment.  Loading replaces the current table.
 * Entries whose tile is infeasible for their shape are rejected
 * (SDT_ERR_TABLE, table left unchanged).  The table named by the environment
 * variable SDT_TUNE_TABLE is loaded on the first gemm_f16 call.
 * sdt_tune_table_lookup returns the tile id for a shape or -1.
 */
int sdt_load_tune_table(const char *path);
void sdt_clear_tune_table(void);
int sdt_tune_table_size(void);
int sdt_tune_table_lookup(int64_t M, int64_t N, int64_t K);

/* ------------------------------------------------------------------------ */
/* Diagnostics                                                               */
/* ------------------------------------------------------------------------ */

/* Message of the last failed call on this thread ("" if none).  Valid until the next call. */
const char *sdt_last_error(void);

/*
 * Every mbarrier wait in the kernels is bounded (by default 2 s).  A kernel
 * that gives up records a code in a device status word and returns without
 * trapping.  This call synchronises `stream`, reads and clears the word for
 * the current device, and returns SDT_OK or SDT_ERR_TIMEOUT (SDT_ERR_CUDA if
 * the stream itself reports an error).  `where` (may be NULL) receives the
 * recorded code: its low 4 bits are the site (1 producer, 2 MMA issuer,
 * 3 epilogue, 4 drain, 5 probe); the two-CTA kernels add the CTA's rank in the
 * pair at bit 4 and the loop position from bit 8.
 */
int sdt_check_device_status(sdt_stream_t stream, int *where);

/*
 * Test hook for the bounded waits: launches one CTA of the GEMM kernel's
 * wait routine on an mbarrier nothing ever arrives at, with the given limit
 * in microseconds (1 .. 10,000,000).  The kernel gives up, records code 5 and
 * returns; read it with sdt_check_device_status.
 */
int sdt_debug_timeout_probe(sdt_stream_t stream, int64_t limit_us);

/*
 * Number of TMA tensor maps encoded so far by this process (misses of the
 * tensor-map cache, whose key holds the base pointer, both extents, the row
 * stride and the box).  For tests of the cache key.
 */
int64_t sdt_debug_tensor_map_encodes(void);

/* SM count and opt-in shared memory per block of the current device. */
int sdt_device_sm_count(void);
int sdt_device_smem_optin(void);

/* ABI version of this header (bumped on incompatible changes). */
#define SDT_ABI_VERSION 1
int sdt_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDT_H */
