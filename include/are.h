/*
 * are.h — C ABI of the GB300 (sm_103a) tensor-parallel row-parallel linear
 * epilogue library (libare.so).
 *
 * The operations, with the pages that define them:
 *
 *  are_gemm_rs   R per-rank partial BF16 GEMMs P_r = A_r[M,K] x B_r[K,N]
 *                (fp32 accumulation), summed in the fixed ring order
 *                r = 0..R-1 and reduce-scattered: rank s receives rows
 *                [s*M/R, (s+1)*M/R) of bf16(sum).  DeepGEMM PR #1 "Fused ring
 *                RS: per-tile bitmask + drain-ring with owner-boundary flush",
 *                description (fused BF16 GEMM + reduce-scatter; per-tile ready
 *                bitmask instead of a per-segment flag; multi-stage partial
 *                buffer; asynchronous TMA stores not drained per tile).
 *  are_gemm_ar   The same R partial GEMMs, each rounded to a bf16 output, then
 *                all-reduced (fp32 sum in ring order, rounded to bf16) into
 *                every rank's view.  ROCm/mori PR #662 "Fuse DSV4-Pro wo_b's
 *                GEMM with its all-reduce", description (GEMM whose bf16
 *                [M, 7168] output is all-reduced across TP ranks).
 *  are_allreduce_rmsnorm
 *                All-reduce of R bf16 partials, residual add and RMSNorm in
 *                one kernel whose two phases meet through a staging buffer
 *                armed with the -0.0 sentinel (the data is its own flag).
 *                ROCm/aiter PR #4977 "Single-kernel Lamport fused all-reduce +
 *                RMSNorm", sections "Approach" and "Correctness notes".
 *
 * On one GPU the R ranks are R separate device buffers; the library emulates
 * their exchange in HBM/L2 and uses no collective.
 *
 * Conventions
 *  - All tensors are row-major and owned by the caller; every tensor pointer
 *    is a DEVICE pointer, 16-byte aligned.  Arrays of per-rank pointers
 *    (A[], B[], out[], partials[]) are HOST arrays of R device pointers; the
 *    library copies them before the call returns.
 *  - `are_bf16` is the 16-bit pattern of a bfloat16 (upper half of an IEEE
 *    binary32).  bf16 results are rounded to nearest even.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous and stream-ordered; they launch kernels
 *    and never synchronise.  A workspace must be used from one stream at a
 *    time: calls on different streams with the same workspace race on the
 *    device, and a call made while another host thread is inside the library
 *    with the same workspace returns ARE_EBUSY.
 *  - are_gemm_rs, are_gemm_ar, are_allreduce_rmsnorm, are_allreduce_add_rmsnorm
 *    and are_allreduce_rmsnorm_quant may be captured into a CUDA graph once
 *    their workspace exists: they only enqueue work on `stream` (kernels;
 *    memsets for an empty contraction), and the state they leave for the next call
 *    (tile masks at 0, staging words at -0.0) is restored inside those
 *    kernels, never by a host step, so every replay finds it as the capture
 *    did.  Workspace creation, reset and snapshots are not capturable.
 *  - Every argument is validated before anything is launched: on any error
 *    nothing is launched and nothing is written.
 *  - Device-side waits are bounded by the workspace's timeout.  A wait that
 *    expires records an error in the workspace's device status word, makes
 *    every other wait of that workspace give up, and lets the kernel return;
 *    read it with are_get_device_status().  After such an error the outputs
 *    of that call are undefined and the workspace must be re-armed with
 *    are_workspace_reset() before further use (until then every call aborts
 *    at its first wait).
 *  - The GEMM kernels and the Lamport AR+RMSNorm kernel run persistent grids
 *    no larger than what the device holds at once (co-resident CTA clusters,
 *    resp. blocks), and their waits on other CTAs' work assume that the whole
 *    grid runs together.  Kernels of other streams that occupy SMs at the
 *    same time can delay part of the grid; a wait that then expires ends the
 *    call with an error status as above, never with a hang.  For full speed,
 *    and to stay clear of that, run these calls without concurrent kernels.
 */
#ifndef ARE_H
#define ARE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ARE_API __attribute__((visibility("default")))
#else
#define ARE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t are_bf16;

typedef enum are_status {
    ARE_OK = 0,
    ARE_EINVAL = 1,   /* bad argument: NULL or misaligned pointer, size outside are_supports(), eps <= 0 ... */
    ARE_ENOMEM = 2,   /* device allocation failed (workspace creation only) */
    ARE_ECUDA = 3,    /* a CUDA runtime call or kernel launch failed */
    ARE_ETIMEOUT = 4, /* a bounded device wait expired (reported by are_get_device_status) */
    ARE_EBUSY = 5,    /* the workspace is in use by another host thread */
    ARE_ENODEV = 6,   /* the current device is not an sm_103 GPU */
    ARE_ECAPACITY = 7, /* the call exceeds the capacities the workspace (or fixed scratch) was created with */
    ARE_ECAPTURE = 8   /* a one-time set-up that cannot run inside a stream capture was needed */
} are_status;

typedef enum are_op {
    ARE_OP_GEMM_RS = 1,
    ARE_OP_GEMM_AR = 2,
    ARE_OP_ALLREDUCE_RMSNORM = 3
} are_op;

/* Workspace capacities.  Buffers are sized from these once, at creation, so
 * their layout never moves with the shapes of later calls. */
typedef struct are_caps {
    int32_t R_max;       /* largest R, 1..8 */
    int64_t M_max;       /* largest M */
    int64_t N_max;       /* largest N */
    int64_t K_max;       /* largest K; 0 = no GEMM buffers (AR+RMSNorm only) */
    uint64_t timeout_ns; /* bound of every device-side wait; 0 = 200 ms */
    uint32_t debug_flags;/* ARE_DEBUG_* */
    uint32_t reserved;
} are_caps;

/* Debug switches (default off; they change bookkeeping, never the arithmetic). */
enum {
    ARE_DEBUG_NO_REARM = 1u,      /* keep tile masks / staging words as the call left them (snapshots) */
    ARE_DEBUG_LOG_PIECES = 2u,    /* record the owner pieces stored for each GEMM+RS tile */
    ARE_DEBUG_COUNT_CANON = 4u,   /* count staged words canonicalised from -0.0 to +0.0 */
    ARE_DEBUG_SKIP_PUBLISH = 8u,  /* GEMM: work unit `debug_arg` never sets its ready bit */
    ARE_DEBUG_SKIP_STAGE = 16u,   /* AR+RMSNorm: 8-element pack `debug_arg` is never staged */
    ARE_DEBUG_SINGLE_CTA = 32u,   /* GEMM: use the one-CTA kernel even where the CTA-pair kernel applies */
    ARE_DEBUG_WAIT_PROFILE = 64u, /* GEMM (CTA-pair kernel) and AR+RMSNorm: add each role's waiting SM cycles
                                     to the counters (see ARE_SNAP_COUNTERS) */
    ARE_DEBUG_AR_ONESHOT = 128u,  /* AR+RMSNorm: take the one-shot path whatever the size (where a row fits) */
    ARE_DEBUG_AR_LAMPORT = 256u,  /* AR+RMSNorm: take the Lamport path whatever the size */
    ARE_DEBUG_PAIR_CTA = 512u,    /* GEMM: use the CTA-pair kernel whatever the size (also with a single tile
                                     row, where the pair's second tile is absent, and below one wave) */
    ARE_DEBUG_RS_RING = 1024u,    /* GEMM+RS on the CTA-pair kernel: push the running sum along the ranks
                                     whatever the size (chunked calls always do) */
    ARE_DEBUG_RS_SPLIT = 2048u    /* GEMM+RS on the CTA-pair kernel: every unit of a tile reduces its row slice
                                     (two-shot) whatever the size; not with chunking */
};

/* Device status word, see are_get_device_status(). */
typedef struct are_dev_status {
    uint32_t code;  /* ARE_DEV_* */
    uint32_t where; /* block index that recorded it */
    int32_t a;      /* MASK_TIMEOUT: tile; STAGE_TIMEOUT: row; PIPE_TIMEOUT: barrier id */
    int32_t b;      /* MASK_TIMEOUT: mask word seen; STAGE_TIMEOUT: pack in row; PIPE_TIMEOUT: unit */
} are_dev_status;

enum {
    ARE_DEV_OK = 0,
    ARE_DEV_MASK_TIMEOUT = 1,  /* a GEMM unit waited too long for a tile's ready bit(s) (a reducer, or the
                                  next rank of the GEMM+RS ring) */
    ARE_DEV_STAGE_TIMEOUT = 2, /* an RMSNorm consumer waited too long for a staged pack */
    ARE_DEV_PIPE_TIMEOUT = 3   /* a GEMM pipeline barrier wait expired */
};

/* Snapshot kinds for are_debug_snapshot(). */
enum {
    ARE_SNAP_MASKS = 1,    /* uint32 per tile (tile index in the kernel's work order) */
    ARE_SNAP_STAGING = 2,  /* fp32 staging words, row-major [M, N] of the last AR+RMSNorm call */
    ARE_SNAP_PIECES = 3,   /* int32 x 64 per tile: tile_m, tile_n, count, then (segment, begin, end) x count */
    ARE_SNAP_CHUNKS = 5,   /* uint64 x (R_max x 64): chunk completion counters, [segment][chunk], see
                              are_workspace_set_chunks() */
    ARE_SNAP_COUNTERS = 4  /* uint64 x 16: [0] canonicalised words; with ARE_DEBUG_WAIT_PROFILE, summed over
                              the CTAs, in SM cycles: [1] TMA producer waiting for a free stage, [2] MMA
                              waiting for operands, [3] MMA waiting for a free accumulator, [4] MMA thread
                              from its first wait to its last commit, [5] drain waiting for an accumulator,
                              [6] loader waiting for tile masks, [7] reduce waiting for partial sub-tiles,
                              [8] CTAs counted, and per pair, in ns of %globaltimer: [9] max and [10]
                              sum of the time from its last MMA to its end, [11] max of its span,
                              [12] sum of its time up to its last MMA.  For AR+RMSNorm: [1] producer waiting for a free stage or
                              residual slot, [2] phase A waiting for partials, [3] phase A held back by
                              its own phase B, [4] phase A waiting for a ring slot's re-arm, [5] phase B
                              spinning on staged words, [6] phase B waiting for its residual row, [7]
                              phase B span, [8] blocks counted */
};

/* Which kernel a call launched, see are_debug_last_launch(). */
typedef enum are_kernel {
    ARE_KERNEL_NONE = 0,          /* nothing launched (an empty problem) */
    ARE_KERNEL_MEMSET = 1,        /* K == 0: the outputs were zero-filled with memsets */
    ARE_KERNEL_GEMM_ONE_CTA = 2,  /* GEMM + reduce, one CTA per 128x256 tile */
    ARE_KERNEL_GEMM_PAIR = 3,     /* GEMM + reduce, CTA pairs (cta_group::2) per 256x256 block */
    ARE_KERNEL_AR_LAMPORT = 4,    /* AR+RMSNorm, two phases meeting through -0.0-armed staging words */
    ARE_KERNEL_AR_ONESHOT = 5     /* AR+RMSNorm, one-shot (no staging) */
} are_kernel;

typedef struct are_launch_info {
    int32_t kernel;       /* are_kernel */
    int32_t grid;         /* CTAs launched */
    int32_t block;        /* threads per CTA */
    int32_t cluster;      /* CTAs per cluster (1 or 2) */
    int32_t rank_block;   /* GEMM pair kernel: tile pairs per rank block, 0 = a pair's R units consecutive */
    int32_t variant;      /* AR kernels: 8-element packs per thread of a row (template variant); GEMM pair
                             kernel: 1 = every unit reduces its row slice of the tile (two-shot), 0 = the
                             GEMM+RS running sum pushed along the ranks */
    int32_t rank_group;   /* GEMM pair kernel: ranks run together inside a rank block (R = ranks innermost) */
    int32_t group_m;      /* GEMM kernels: tile(-pair) rows per raster group */
} are_launch_info;

typedef struct are_ws are_ws;

/* Library version, (major << 16) | minor. */
ARE_API int are_version(void);

/* Human-readable name of a status code (static string). */
ARE_API const char* are_status_string(are_status s);

/* The predicate every call applies before launching; ARE_OK if supported.
 * ROCm/mori PR #662 "Fuse DSV4-Pro wo_b's GEMM with its all-reduce over cco
 * SDMA", review threads: a capability query and the execution path must share
 * one predicate, so that a shape the query accepts never fails later at
 * launch, and a shape it rejects is never run.  Every operation below calls
 * this same function before it validates pointers or launches anything.
 *  GEMM_RS: 1 <= R <= 8; M, N >= 0; K >= 0; K % 8 == 0 and N % 8 == 0 (16-byte
 *           rows for TMA); M % R == 0 and (M / R) % 8 == 0 (owner segments
 *           start on 8-row boundaries).
 *  GEMM_AR: 1 <= R <= 8; K % 8 == 0; N % 8 == 0.
 *  ALLREDUCE_RMSNORM: 1 <= R <= 8; N % 8 == 0 (16-byte packs); N <= 32768.
 * K is ignored for ALLREDUCE_RMSNORM.  Pure host function: no device needed. */
ARE_API are_status are_supports(int op, int R, int64_t M, int64_t N, int64_t K);

/* Create a workspace on the current CUDA device: tile masks, the per-rank
 * partial buffer, the Lamport staging buffer (filled with the sentinel, on a
 * private stream, synchronously) and the device status word.
 * ROCm/mori PR #662, review threads: every capacity is validated before the
 * first allocation; buffer offsets are sized from the capacities, never from
 * a call's M, so the layout does not move between calls; a set-up that fails
 * part-way releases everything it acquired and returns the first (original)
 * error, not the error of the clean-up.  ROCm/aiter PR #4977, bring-up
 * commits: the staging region is private to this library and is armed here,
 * outside any stream capture, on a stream of its own (an arming captured into
 * a graph would re-arm on every replay, under the kernel's feet).
 *  caps : R_max 1..8, M_max >= 1, N_max >= 8 and N_max % 8 == 0, K_max >= 0.
 *  ws   : receives the handle; *ws is NULL on any failure.
 * Returns ARE_EINVAL for bad capacities, ARE_ENODEV if the current device is
 * not sm_103, ARE_ENOMEM / ARE_ECUDA if an allocation or the arming fails.
 * Must not be called during stream capture. */
ARE_API are_status are_workspace_create(are_ws** ws, const are_caps* caps);

/* Release a workspace: synchronise the device (so no launched kernel still
 * uses it), then free every buffer of it.  NULL is accepted.  The caller's
 * tensors are not touched.  ROCm/mori PR #662, review threads: an op that
 * owns device buffers releases them through an explicit close, never only
 * through a destructor at interpreter exit.  Returns the synchronisation's
 * error, if any (the buffers are freed either way). */
ARE_API are_status are_workspace_destroy(are_ws* ws);

/* Clear the device status word, zero every tile mask and re-arm every staging
 * word with the sentinel; synchronous.  Needed only after a device error (or
 * after a debug call made with ARE_DEBUG_NO_REARM).  Not capturable. */
ARE_API are_status are_workspace_reset(are_ws* ws);

/* Change the debug switches (ARE_DEBUG_*) and their argument for later calls. */
ARE_API are_status are_workspace_set_debug(are_ws* ws, uint32_t flags, int64_t arg);

/* Per-rank input size (M * N * 2 bytes) at or below which are_allreduce_rmsnorm
 * takes its one-shot kernel; 0 sends every call to the Lamport kernel.  The
 * default, 448 KiB, is the crossover the pages measured for a 4-GPU collective
 * (ROCm/aiter PR #4977, the commit that gates on the measured crossover).  With
 * the ranks local to one GPU there is no link traffic for the Lamport path to
 * save, and the one-shot kernel measured faster at every size, so a
 * single-GPU caller may raise it.  Returns ARE_EINVAL for a NULL workspace,
 * ARE_EBUSY if the workspace is in use by another thread. */
ARE_API are_status are_workspace_set_oneshot_max_bytes(are_ws* ws, uint64_t bytes);

/* Order of the CTA-pair GEMM kernel's work units (tuning; the results do not
 * depend on it: every tile is still summed in the order r = 0..R-1).  A unit is
 * one rank's 256x256 partial of one tile pair; the persistent grid takes units
 * in this order, wave by wave.  The pages leave the order open; DeepGEMM PR #1
 * (description) notes that a reduce epilogue that backs up stalls the MMA, and
 * ROCm/mori PR #662 (the destination-rotated order follow-ups) that the tile
 * order decides when each destination's data completes.
 *  group_m     : 256-row tile pairs per raster group (tile pairs are taken
 *                column by column inside a group of group_m pair rows);
 *                0 = the library's choice (8 for GEMM+RS on the ring, 4
 *                otherwise).
 *  block_pairs : > 0: tile pairs are taken in blocks of block_pairs, and a
 *                block's units run in rank groups (below); < 0: the R units of
 *                a tile pair run consecutively; 0 = the library's choice.
 *                GEMM+RS on the ring pushes a running sum from rank to rank,
 *                so it runs one block of all tile pairs, rank by rank (a
 *                pair's R units consecutive would make each tile's ranks wait
 *                on one another in turn), padded to one wave of pairs where
 *                the pairs fill 60-100 % of a wave and K <= 2048; chunked GEMM+RS
 *                (are_workspace_set_chunks), always on the ring, runs rank by
 *                rank in blocks that finish whole chunks (the rotated order:
 *                one order chunk of every owner segment; the raster: two
 *                waves of tile pairs).  GEMM+RS with the reduction split over
 *                a tile's units (R = 4, 8 with K <= 2048 up to 3/4 of a wave of
 *                tile pairs, otherwise up to half a wave) and
 *                GEMM+AR: consecutive.
 *  rank_group  : with block_pairs > 0, the number of ranks whose units of a
 *                block run together (1 = rank by rank, R = a pair's R units
 *                consecutive); 0 = 1.  With block_pairs = 0 the library's
 *                choice is used for both.
 * Returns ARE_EINVAL for negative group_m / rank_group or rank_group > 8. */
ARE_API are_status are_workspace_set_gemm_order(are_ws* ws, int group_m, int block_pairs, int rank_group);

/*
 * Chunked owner-segment completion for GEMM+RS.  ROCm/mori PR #662, the fused
 * GEMM -> scatter follow-ups: per-(destination, chunk) completion counters,
 * monotonic and never reset, whose modulo test elects exactly one CTA per
 * chunk, with the chunk count halved until it divides the destination's
 * M-tiles; and the destination-rotated, chunk-major tile order (and its
 * striped variant), so that every destination's first chunk completes early
 * instead of destination 0's whole slice first.  Here the destinations are the
 * owner segments: chunk c of segment s is a band of the 128-row output tiles
 * that intersect s (their count n_s split into C_s = `chunks` halved until it
 * divides n_s), and it completes once every 128x256 tile of the band has been
 * reduced and its rows stored into segment s.  The unit whose piece completes
 * the chunk (elected by the counters) publishes the chunk's generation (how
 * many calls have completed it since the workspace was created or reset) to
 * host-mapped memory, where are_chunk_wait() sees it while the kernel is
 * still running.
 *  chunks : chunks per owner segment, 0 (off, the default) .. 64.
 *  stripe : the CTA-pair kernel's tile order while chunking is on, where the
 *           owner segments are whole 256-row tile pairs (M/R % 256 == 0):
 *           0 = destination-rotated chunk-major (chunk c of every segment, all
 *           its tile columns, before chunk c+1 of any); > 0 = striped (every
 *           segment's chunk-c band of `stripe` tile columns before the next
 *           band); -1 = the library's usual order (counters only).
 * The results do not depend on either setting.  Returns ARE_EINVAL for values
 * outside these ranges, ARE_ECAPACITY for a workspace without GEMM buffers.
 */
ARE_API are_status are_workspace_set_chunks(are_ws* ws, int chunks, int stripe);

/* The generation that the last GEMM+RS call enqueued on `ws` with chunking on
 * publishes for each of its chunks when they complete: the number of such
 * calls that launched a kernel since the workspace was created or reset
 * (a call with M, N or K equal to 0 launches none and publishes nothing).
 * Replays of a captured graph are not counted here: each adds one per
 * captured call.  Host only. */
ARE_API are_status are_chunk_generation(are_ws* ws, uint64_t* generation);

/* Host-side wait for chunk `chunk` of owner segment `segment` to reach
 * `generation` (compared modulo 2^32): polls the host-mapped word that the
 * unit completing the chunk writes, so it returns while the GEMM+RS kernel
 * is still running, as soon as that chunk's rows are in device memory.  No
 * GPU-side waiter is involved.  Returns ARE_OK, ARE_ETIMEOUT after
 * `timeout_ns`, ARE_EINVAL for an index outside the workspace. */
ARE_API are_status are_chunk_wait(are_ws* ws, int segment, int chunk, uint64_t generation, uint64_t timeout_ns);

/* Synchronise the device, then copy the workspace's device status word.
 * Returns ARE_ETIMEOUT if a device wait expired, else ARE_OK. */
ARE_API are_status are_get_device_status(are_ws* ws, are_dev_status* out);

/* Host-side record of the last operation called with this workspace: which
 * kernel it launched and with which launch shape.  Reads no device memory and
 * does not synchronise.  Zeroed (ARE_KERNEL_NONE) before any call. */
ARE_API are_status are_debug_last_launch(are_ws* ws, are_launch_info* out);

/* Synchronise the device and copy `bytes` of a bookkeeping buffer (ARE_SNAP_*)
 * to host memory `host_dst`. */
ARE_API are_status are_debug_snapshot(are_ws* ws, int kind, void* host_dst, size_t bytes);

/*
 * GEMM + reduce-scatter.
 *  A[r]   : bf16 [M, K] (K contiguous), r < R
 *  B[r]   : bf16 [K, N] (N contiguous), r < R
 *  out[s] : bf16 [M/R, N], rank s's owner segment, s < R.  Passing
 *           out[s] = base + s*(M/R)*N fills one contiguous [M, N] tensor.
 *  Result : out[s][i][j] = bf16( sum_{r=0..R-1} P_r[s*M/R + i][j] ), the fp32
 *           partials added in the order r = 0, 1, ..., R-1.
 * Outputs must not alias inputs.  K == 0 writes zeros.
 */
ARE_API are_status are_gemm_rs(const are_bf16* const A[], const are_bf16* const B[], are_bf16* const out[], int R,
                       int64_t M, int64_t N, int64_t K, are_ws* ws, void* stream);

/*
 * GEMM + all-reduce.
 *  A[r], B[r] as for are_gemm_rs.
 *  out[v] : bf16 [M, N] for every rank view v < R (views may alias each other;
 *           identical pointers are written once).
 *  Result : out[v][i][j] = bf16( sum_{r=0..R-1} f32(bf16(P_r[i][j])) ), in the
 *           order r = 0..R-1: each rank's GEMM output is bf16 before the
 *           all-reduce, the sum is fp32.
 */
ARE_API are_status are_gemm_ar(const are_bf16* const A[], const are_bf16* const B[], are_bf16* const out[], int R,
                       int64_t M, int64_t N, int64_t K, are_ws* ws, void* stream);

/*
 * All-reduce + residual add + RMSNorm (one kernel).
 *  partials[r] : bf16 [M, N], r < R
 *  residual    : bf16 [M, N] or NULL (treated as zero)
 *  gamma       : fp32 [N]
 *  out         : bf16 [M, N]
 *  Result      : s = sum_{r=0..R-1} f32(partials[r]) in that order, -0.0
 *                staged as +0.0; h = s + f32(residual);
 *                out = bf16( h * rsqrt(mean_j(h_j^2) + eps) * gamma ).
 * eps must be finite and > 0.  The staging buffer must have been armed (it is
 * at creation, and every call re-arms what it consumed).
 *
 * Two kernels compute it, with the same arithmetic in the same order, so the
 * result bits do not depend on which runs (ROCm/aiter PR #4977, the commits
 * that re-baseline against the one-stage kernel and gate on the crossover):
 *  - the one-shot kernel: reads every rank's row once and stages nothing.  It
 *    runs when the per-rank input M * N * 2 bytes is at most the workspace's
 *    one-shot threshold (default 448 KiB; see
 *    are_workspace_set_oneshot_max_bytes) and (R + 1) rows of N fit one
 *    block's shared memory (R * N * 2 + N * 2 <= ~227 KB);
 *  - the Lamport kernel (two phases meeting through the -0.0-armed staging
 *    words) otherwise.
 * ARE_DEBUG_AR_ONESHOT / ARE_DEBUG_AR_LAMPORT force one path.
 */
ARE_API are_status are_allreduce_rmsnorm(const are_bf16* const partials[], const are_bf16* residual, const float* gamma,
                                 float eps, are_bf16* out, int R, int64_t M, int64_t N, are_ws* ws, void* stream);

/*
 * All-reduce + residual add + RMSNorm that also returns the updated residual.
 * (The pages name the fused kernel's other variants but port only this
 * operation's normalised output: ROCm/aiter PR #4977, "Known gaps /
 * follow-ups".)  A transformer layer feeds h, the sum of the all-reduced
 * partials and the incoming residual, to the next layer as its residual.
 *  Arguments   : as are_allreduce_rmsnorm, plus
 *  residual_out: bf16 [M, N] or NULL; receives bf16(h) (round to nearest even)
 *                with h exactly as in the RMSNorm: h = s + f32(residual), s
 *                the canonicalised fp32 ring-order sum.  It may be the same
 *                buffer as `residual` (in-place update): each row's residual
 *                is read before that row's residual_out is written, by the
 *                same block.  It must not alias a partial or `out`.
 * Both kernels (one-shot and Lamport) write it, with identical bits.
 */
ARE_API are_status are_allreduce_add_rmsnorm(const are_bf16* const partials[], const are_bf16* residual,
                                             const float* gamma, float eps, are_bf16* out, are_bf16* residual_out,
                                             int R, int64_t M, int64_t N, are_ws* ws, void* stream);

/*
 * All-reduce + residual add + RMSNorm with a quantised output: the pages list
 * the fused kernel's quantising variants without defining one (ROCm/aiter PR
 * #4977, "Known gaps / follow-ups"); this is per-row (per-token) dynamic FP8:
 *  out_q       : FP8 E4M3 codes [M, N] (OCP e4m3fn: bias 7, max finite 448)
 *  out_scale   : fp32 [M]
 *  residual_out: bf16 [M, N] or NULL, as in are_allreduce_add_rmsnorm
 *  Result      : y = h * rsqrt(mean_j(h_j^2) + eps) * gamma as in
 *                are_allreduce_rmsnorm (fp32, before its bf16 rounding);
 *                out_scale[i] = max_j |y_ij| / 448 (1 for an all-zero row);
 *                out_q[i][j]  = e4m3(y_ij / out_scale[i]), round to nearest
 *                even, saturating to +-448; both divisions correctly rounded.
 *                y_ij ~= out_q[i][j] * out_scale[i].
 * The other arguments, the two kernels and their dispatch are as for
 * are_allreduce_rmsnorm; no bf16 output is written.
 */
ARE_API are_status are_allreduce_rmsnorm_quant(const are_bf16* const partials[], const are_bf16* residual,
                                               const float* gamma, float eps, uint8_t* out_q, float* out_scale,
                                               are_bf16* residual_out, int R, int64_t M, int64_t N, are_ws* ws,
                                               void* stream);

/*
 * All-reduce + residual + RMSNorm that allocates nothing.
 *
 * The pages have no counterpart to this entry point.  It is for callers that
 * cannot let a library call cudaMalloc or cudaFree: a framework whose caching
 * allocator must own every device byte, a process held to a fixed
 * device-memory budget, or code that cannot pay the device-wide
 * synchronisation an allocation or a free can cause.  Such callers cannot
 * create a workspace, so this call needs none.
 *
 *  Arguments and result: as are_allreduce_rmsnorm, without `ws`.
 *  Scratch: a fixed array compiled into the library (8 MiB of fp32 staging
 *           words after a 256-byte status header), held by every GPU that
 *           loads the library until the process exits.
 *  Limit:   M * N <= 2,097,152 (e.g. M <= 292 at N = 7168); a larger call
 *           returns ARE_ECAPACITY and launches nothing.
 *  Set-up:  the first call on a device looks up the array's device address
 *           (once per device, with that device current); make that first
 *           call before any stream capture.  A first call made on a stream
 *           that is capturing returns ARE_ECAPTURE and enqueues nothing.
 *  Sharing: every call uses the same array and it keeps the last call's
 *           contents.  Each call therefore first clears the status word and
 *           re-arms the staging words it uses with the -0.0 sentinel, on
 *           `stream`, then runs the kernel.  Calls whose kernels can overlap
 *           on the GPU (other streams, other host threads) race on the array
 *           and give undefined results.  A device-side wait that expires
 *           (bounded at 200 ms) is recorded in the array's status word; read
 *           it with are_noalloc_device_status().
 *  Never calls cudaMalloc, cudaFree or any allocating library routine.
 */
ARE_API are_status are_allreduce_rmsnorm_noalloc(const are_bf16* const partials[], const are_bf16* residual,
                                                 const float* gamma, float eps, are_bf16* out, int R, int64_t M,
                                                 int64_t N, void* stream);

/*
 * Device status word of the allocation-free entry point on the current device.
 * The pages have no counterpart to it: it exists because callers of
 * are_allreduce_rmsnorm_noalloc have no workspace to ask.  It synchronises the
 * device, then copies the 16-byte status word at the start of the fixed array
 * to `out` with cudaMemcpy (no allocation).  Every call of the entry point
 * clears that word first, so it describes the last call only.  Returns
 * ARE_ETIMEOUT if a device wait of that call expired (its output is then
 * undefined), ARE_OK otherwise, ARE_ENODEV / ARE_ECUDA if the current device
 * cannot be set up, ARE_EINVAL for a NULL `out`.
 */
ARE_API are_status are_noalloc_device_status(are_dev_status* out);

#ifdef __cplusplus
}
#endif

#endif /* ARE_H */
