// C ABI of the library: argument validation, workspace lifecycle, launches.
//
// Lessons from the pages that shape this layer:
//  * ROCm/mori PR #662 (review threads): one predicate shared by the
//    "supports" query and the execution path; validation before any
//    allocation or launch; a failed setup releases what it acquired and
//    returns the original error; buffer offsets sized by capacity so the
//    layout never moves with M.
//  * ROCm/aiter PR #4977 (bring-up and follow-up commits): the Lamport staging
//    region is private to this kernel, armed once outside any graph capture
//    (on a private stream), and the persistent grid is clamped to the
//    co-resident block count.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "are_internal.h"

using namespace are;

struct are_ws {
    int device = 0;
    int num_sms = 0;
    are_caps caps{};
    DevStatus* d_status = nullptr;
    unsigned long long* d_counters = nullptr;
    uint32_t* d_mask = nullptr;
    size_t mask_words = 0;
    uint8_t* d_part = nullptr;
    size_t part_bytes = 0;
    int32_t* d_pieces = nullptr;
    size_t piece_words = 0;
    uint32_t* d_staging = nullptr;
    size_t staging_words = 0;
    int ar_resident[kArMaxPpt + 1] = {0};
    uint64_t oneshot_max_bytes = 0;   // set at creation
    std::mutex mu;
    uint32_t debug_flags = 0;
    int64_t debug_arg = -1;
    uint64_t timeout_ns = 0;
    int64_t last_ar_M = 0, last_ar_N = 0;
    int pair_clusters = 0;            // co-resident clusters of the pair kernel on `device`
    int order_group_m = 0;            // pair-kernel unit order overrides (0 = the library's choice)
    int order_block = 0;
    int order_rank_group = 0;
    uint32_t* d_cons = nullptr;       // GEMM+AR row-slice readers done per tile
    // chunked owner-segment completion (GEMM+RS)
    unsigned long long* d_chunk_ctr = nullptr;  // [R_max][kChunkCap] monotonic counters
    uint32_t* h_chunk_gen = nullptr;            // [R_max][kChunkCap] completed generations (mapped host memory)
    uint32_t* d_chunk_gen = nullptr;            // the same memory as the device sees it
    int chunks = 0;                             // chunks per owner segment, 0 = off
    int chunk_stripe = 0;                       // destination-rotated order: columns per rotation
    uint64_t rs_generation = 0;                 // GEMM+RS kernels launched with chunking on
    are_launch_info last{};           // what the last operation launched
};

namespace {

constexpr uint64_t kDefaultTimeoutNs = 200ull * 1000 * 1000;
// AR+RMSNorm: per-rank input bytes (M * N * 2) at or below which the one-shot
// kernel runs instead of the Lamport kernel.
constexpr uint64_t kOneShotMaxBytes = 448ull * 1024;
constexpr size_t kCounterWords = 16;

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

are_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return ARE_OK;
    if (e == cudaErrorMemoryAllocation) return ARE_ENOMEM;
    return ARE_ECUDA;
}

struct TryLock {
    std::mutex& m;
    bool ok;
    explicit TryLock(std::mutex& mm) : m(mm), ok(mm.try_lock()) {}
    ~TryLock() {
        if (ok) m.unlock();
    }
};

void free_ws(are_ws* ws) {
    if (!ws) return;
    cudaFree(ws->d_status);
    cudaFree(ws->d_counters);
    cudaFree(ws->d_mask);
    cudaFree(ws->d_part);
    cudaFree(ws->d_pieces);
    cudaFree(ws->d_staging);
    cudaFree(ws->d_chunk_ctr);
    cudaFree(ws->d_cons);
    if (ws->h_chunk_gen) cudaFreeHost(ws->h_chunk_gen);
    delete ws;
}

// Zero the bookkeeping and arm the staging buffer on a private non-blocking
// stream, then wait for it.  Never on the caller's stream (a captured arming
// would re-arm on every replay).
are_status arm_workspace(are_ws* ws) {
    cudaStream_t s = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return from_cuda(e);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws->d_status, 0, sizeof(DevStatus), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws->d_counters, 0, kCounterWords * 8, s);
    if (e == cudaSuccess && ws->d_mask) e = cudaMemsetAsync(ws->d_mask, 0, ws->mask_words * 4, s);
    if (e == cudaSuccess && ws->d_pieces) e = cudaMemsetAsync(ws->d_pieces, 0, ws->piece_words * 4, s);
    if (e == cudaSuccess && ws->d_staging) e = launch_fill_u32(ws->d_staging, kSentinelF32, ws->staging_words, s);
    if (e == cudaSuccess && ws->d_chunk_ctr)
        e = cudaMemsetAsync(ws->d_chunk_ctr, 0, (size_t)ws->caps.R_max * kChunkCap * 8, s);
    if (e == cudaSuccess && ws->d_cons) e = cudaMemsetAsync(ws->d_cons, 0, ws->mask_words * 4, s);
    cudaError_t e2 = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = e2;
    cudaStreamDestroy(s);
    if (e == cudaSuccess && ws->h_chunk_gen) {
        std::memset(ws->h_chunk_gen, 0, (size_t)ws->caps.R_max * kChunkCap * 4);
        ws->rs_generation = 0;
    }
    return from_cuda(e);
}

bool ranks_ok(int R) { return R >= 1 && R <= kMaxRanks; }

// A device pointer must be 16-byte aligned; it may be NULL only when the
// tensor it stands for has no elements.
bool ptr_ok(const void* p, int64_t elems) { return elems == 0 ? (p == nullptr || aligned16(p)) : aligned16(p); }

are_status check_gemm_ptrs(const are_bf16* const A[], const are_bf16* const B[], are_bf16* const out[], int R,
                           int64_t M, int64_t N, int64_t K, int mode) {
    if (!A || !B || !out) return ARE_EINVAL;
    const int64_t out_elems = (mode == kModeRS) ? (M / R) * N : M * N;
    for (int r = 0; r < R; ++r)
        if (!ptr_ok(A[r], M * K) || !ptr_ok(B[r], K * N) || !ptr_ok(out[r], out_elems)) return ARE_EINVAL;
    return ARE_OK;
}

are_status gemm_call(int mode, const are_bf16* const A[], const are_bf16* const B[], are_bf16* const out[], int R,
                     int64_t M, int64_t N, int64_t K, are_ws* ws, void* stream) {
    if (!ws) return ARE_EINVAL;
    const int op = (mode == kModeRS) ? ARE_OP_GEMM_RS : ARE_OP_GEMM_AR;
    are_status st = are_supports(op, R, M, N, K);
    if (st != ARE_OK) return st;
    st = check_gemm_ptrs(A, B, out, R, M, N, K, mode);
    if (st != ARE_OK) return st;
    TryLock lk(ws->mu);
    if (!lk.ok) return ARE_EBUSY;
    if (R > ws->caps.R_max || M > ws->caps.M_max || N > ws->caps.N_max || K > ws->caps.K_max || !ws->d_part)
        return ARE_ECAPACITY;
    const int64_t tiles_m = ceil_div(M, kBM), tiles_n = ceil_div(N, kBN);
    const int64_t T = tiles_m * tiles_n;
    if ((size_t)T > ws->mask_words || (size_t)(R * T) * kTilePartBytes > ws->part_bytes) return ARE_ECAPACITY;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ws->last = are_launch_info{};
    if (M == 0 || N == 0) return ARE_OK;

    // distinct output views (GEMM+AR views may alias)
    int nviews = 0;
    const are_bf16* views[kMaxRanks];
    if (mode == kModeAR) {
        for (int v = 0; v < R; ++v) {
            bool dup = false;
            for (int w = 0; w < nviews; ++w) dup |= (views[w] == out[v]);
            if (!dup) views[nviews++] = out[v];
        }
    }
    if (K == 0) {  // empty contraction: the result is zero
        ws->last.kernel = ARE_KERNEL_MEMSET;
        if (mode == kModeRS) {
            for (int r = 0; r < R; ++r) {
                cudaError_t e = cudaMemsetAsync(out[r], 0, (size_t)(M / R) * N * 2, s);
                if (e != cudaSuccess) return from_cuda(e);
            }
        } else {
            for (int v = 0; v < nviews; ++v) {
                cudaError_t e = cudaMemsetAsync(const_cast<are_bf16*>(views[v]), 0, (size_t)M * N * 2, s);
                if (e != cudaSuccess) return from_cuda(e);
            }
        }
        return ARE_OK;
    }

    GemmParams* p = new (std::nothrow) GemmParams;
    if (!p) return ARE_ENOMEM;
    std::memset(p, 0, sizeof(GemmParams));
    cudaError_t e = cudaSuccess;
    const int64_t S = (mode == kModeRS) ? M / R : M;
    int H = 128;
    if (mode == kModeRS) {
        while (S % H) H >>= 1;  // largest power of two dividing S, <= 128 (>= 8 by are_supports)
    }
    for (int r = 0; r < R && e == cudaSuccess; ++r) {
        e = make_tmap_bf16(&p->tmA[r], A[r], (uint64_t)K, (uint64_t)M, kBK, kBM);
        if (e == cudaSuccess) e = make_tmap_bf16(&p->tmB[r], B[r], (uint64_t)N, (uint64_t)K, 64, kBK);
    }
    // CTA pairs (256-row tiles) wherever there are at least two tile rows and
    // the device can co-schedule the clusters; one CTA per tile otherwise.  GEMM+AR
    // also takes the pairs with a single tile row (the pair's second tile does not
    // exist, as with any odd number of tile rows): such a problem is bound by streaming
    // B, and the pair kernel spreads the reduction over a pair's R units and keeps every
    // SM streaming (R=8, M=64, N=7168, K=2048: 58.6 against 64.5 us).
    const int clusters = ws->pair_clusters;
    const int64_t pair_units = (int64_t)((tiles_m + 1) / 2) * tiles_n * R;
    // GEMM+RS on the pair kernel: the running sum pushed along the ranks, or every unit of a tile
    // reducing its row slice (two-shot, as GEMM+AR).  The ring's R drains of a tile run one after
    // the other, which a wave or more of tile pairs (or a block padded to one, see the unit order)
    // hides and fewer pairs do not.  Measured (us per call, ring / split / one-CTA kernel; tile
    // pairs, of 76 co-resident clusters): R=4, N=4096, K=2048 at M=256 44.0 / 29.8 / 35.2 (16),
    // M=512 52.3 / 41.3 / 52.8 (32), M=768 53.2 / 52.0 (48), M=1024 54.1 (padded) / 62.6 / 88.6
    // (64), M=4096 171.5 / 192.2 / 235.0 (256); R=8, K=2048, M=256, N=7168 98.9 / 69.7 / 118.0
    // (28), M=384, N=4096 91.5 / 68.1 (32), M=256, N=8192 103.1 / 82.1 (32); R=8, N=8192,
    // K=4096, M=512 173.8 / 193.3 / 266.6 (64); R=2, N=4096, K=2048, M=256 26.8 / 27.0 / 29.1 (16:
    // a chain of two).  At 48 pairs the split still leads for R=4 and 8 (R=8, M=384, N=6144
    // 92.9 / 98.3; R=4, M=768 52.3 / 53.2) but not for R=5 and 6 (R=6, M=768 80.5 / 73.9; R=5,
    // M=640 71.6 / 62.4), whose row slices are not whole 16-row groups (more, partly empty stage
    // loads and whole-row stores instead of TMA boxes); at 32 pairs it leads for those too (R=6,
    // M=384 63.2 / 71.0).  Long units hide more of the ring's chain: at K=4096 with 56 pairs the
    // ring leads (R=8, M=384, N=7168 152.9 / 161.5), with 32 the two tie for R=8 (M=256, N=8192
    // 132.4 / 131.9) and the split leads for R=4 (M=512 67.7 / 63.2).  So: the split for R = 4
    // and 8 up to three quarters of a wave of pairs when K <= 2048, and otherwise (R = 5..7, or
    // longer K) up to half a wave; the ring beyond that; and the pair kernel (either way) rather
    // than the one-CTA kernel from two tile rows on.  Chunked calls count a tile's pieces at the
    // ring's last rank: always the ring.
    const int64_t num_pairs_all = (int64_t)((tiles_m + 1) / 2) * tiles_n;
    const bool whole_groups = kBM % (16 * R) == 0;  // R = 4, 8: every row slice is 16-row groups
    bool rs_split = mode == kModeRS && ws->chunks == 0 && R >= 4 &&
                    ((whole_groups && K <= 2048) ? 4 * num_pairs_all <= 3 * (int64_t)clusters
                                                 : 2 * num_pairs_all <= (int64_t)clusters);
    if (ws->debug_flags & ARE_DEBUG_RS_SPLIT) rs_split = mode == kModeRS && ws->chunks == 0;
    if (ws->debug_flags & ARE_DEBUG_RS_RING) rs_split = false;
    // A single tile row (the pair's second tile does not exist, as with any odd number of tile
    // rows) takes the pair kernel for GEMM+AR and for the GEMM+RS split: R=4, M=128, N=4096,
    // K=2048 29.1 against 35.8-36.1 us here and 44.9 on the ring, R=8, M=128, N=7168 62.5 against
    // 90.7 and 96.0; with R < 4 the one-CTA kernel stays ahead (R=2, M=64, N=256, K=128 14.1-14.3
    // against 16.6-17.0 us, R=2, M=128, N=1024, K=512 16.8-17.1 against 18.5-19.2).
    const bool pair_ok = (tiles_m >= 2 || mode == kModeAR || rs_split || (ws->debug_flags & ARE_DEBUG_PAIR_CTA)) &&
                         clusters > 0 && !(ws->debug_flags & ARE_DEBUG_SINGLE_CTA);
    // GEMM+AR below one wave of pairs: the one-CTA kernel (the pair kernel from one wave on, or
    // with a single tile row, see above)
    const bool use_pair = pair_ok && (pair_units > clusters || mode == kModeRS || (ws->debug_flags & ARE_DEBUG_PAIR_CTA));
    if (mode == kModeRS) {
        // owner-segment maps: H-row boxes for the ring's and the one-CTA kernel's piece stores,
        // 16-row boxes (where segments are whole 16-row groups) for the row slices' groups
        if (use_pair && rs_split && H > 16) H = 16;
        for (int r = 0; r < R && e == cudaSuccess; ++r) {
            e = make_tmap_bf16(&p->tmOut[r], out[r], (uint64_t)N, (uint64_t)S, 64, (uint32_t)H);
            p->views[r] = out[r];
        }
    }
    // GEMM+AR views: the one-CTA kernel stores whole 128-row tiles, the pair kernel 16-row
    // groups of a unit's row slice (boxes of 64 columns either way)
    for (int v = 0; v < nviews && e == cudaSuccess; ++v) {
        e = make_tmap_bf16(&p->tmOut[v], views[v], (uint64_t)N, (uint64_t)M, 64, use_pair ? 16u : (uint32_t)kBM);
        p->views[v] = const_cast<are_bf16*>(views[v]);
    }
    if (e != cudaSuccess) {
        delete p;
        return ARE_EINVAL;
    }
    p->part = ws->d_part;
    p->mask = ws->d_mask;
    p->status = ws->d_status;
    p->pieces = ws->d_pieces;
    p->counters = ws->d_counters;
    p->R = R;
    p->M = (int)M;
    p->N = (int)N;
    p->K = (int)K;
    p->S = (int)S;
    p->H = H;
    p->nviews = nviews;
    p->tiles_m = (int)tiles_m;
    p->tiles_n = (int)tiles_n;
    p->num_tiles = (int)T;
    p->num_units = (int)(T * R);
    p->num_kb = (int)ceil_div(K, kBK);
    p->pairs_m = (int)((tiles_m + 1) / 2);
    p->block_tiles = 0;
    p->num_pair_units = (int)(p->pairs_m * tiles_n * R);
    p->flags = ws->debug_flags;
    p->debug_arg = ws->debug_arg;
    p->timeout_ns = ws->timeout_ns;
    if (mode == kModeRS && ws->chunks > 0) {
        p->chunk_ctr = ws->d_chunk_ctr;
        p->chunk_host = ws->d_chunk_gen;
        p->chunks = ws->chunks;
    }
    if (use_pair) {
        // the partial slots as a 5-D map: a row slice's 16-row group of 8 sub-tiles in one load
        if (make_tmap_part(&p->tmPart, ws->d_part, (uint64_t)T, (uint64_t)R) != cudaSuccess) {
            delete p;
            return ARE_EINVAL;
        }
        p->group_m = (int)std::min<int64_t>(p->pairs_m, 4);
        const int64_t num_pairs = (int64_t)p->pairs_m * tiles_n;
        // destination-rotated order (chunked GEMM+RS): needs owner segments of whole pair
        // rows; chunk c of every segment then runs before chunk c+1 of any
        if (p->chunks > 0 && ws->chunk_stripe >= 0 && S % 256 == 0) {
            const int ps = (int)(S / 256);
            int cs = ws->chunks;
            while (cs > 1 && ps % cs) cs >>= 1;
            p->rot_ps = ps;
            p->rot_cs = cs;
            p->rot_pc = ps / cs;
            p->rot_w = ws->chunk_stripe > 0 ? std::min<int>(ws->chunk_stripe, (int)tiles_n) : (int)tiles_n;
        }
        if (mode == kModeRS && rs_split) {
            // two-shot, as GEMM+AR: a pair's R units consecutive
            p->rs_split = 1;
            p->rank_group = 1;
        } else if (mode == kModeRS) {
            // GEMM+RS pushes a running sum along the ranks (rank r adds its accumulator to rank
            // r-1's sum), so a tile's rank r+1 should run after its rank r: rank by rank over
            // blocks of tile pairs (each rank sweeps the block's tiles, as one GEMM would).
            p->rank_group = 1;
            if (!p->chunk_ctr) {
                // one block of all the tile pairs, raster groups of 8 pair rows: no padding, and
                // with at least a wave of pairs a tile's consecutive ranks are never in the same
                // wave.  Measured on the large GEMM+RS (us per call, one box): 2361 against 2362
                // (blocks of 256 pairs), 2373 (128), 2417 (76 = one wave, 320 padding units), 2452
                // (152), 2430 (4 pair-row raster) and 4831 with a pair's ranks consecutive (each
                // tile's drains then wait in a chain).
                p->block_tiles = (int)num_pairs;
                p->group_m = (int)std::min<int64_t>(p->pairs_m, 8);
                // With most of a wave of pairs but not a whole one, a tile's consecutive ranks would
                // share waves and its drains wait in a chain; a block padded to one wave runs each
                // rank in a wave of its own.  That pays where units are short (K <= 2048): R=4,
                // M=1024, N=4096, K=2048 (64 pairs) 61.7 -> 55.1 us, R=2 the same 38.0 -> 32.1,
                // R=3, M=768 (48 pairs) 45.6 -> 42.1; not with long units or a sparse wave (R=8,
                // M=512, N=8192, K=4096, 64 pairs 176.0 -> 186.7; R=2, M=256, 16 pairs 26.7 -> 30.1).
                if (num_pairs < clusters && 10 * num_pairs >= 6 * (int64_t)clusters && K <= 2048)
                    p->block_tiles = clusters;
            } else {
                // chunked GEMM+RS completes chunks early: blocks that finish whole chunks, one
                // order chunk of every segment each in the destination-rotated order, else two
                // waves of tile pairs of the raster
                p->block_tiles = p->rot_pc > 0 ? (int)((int64_t)R * p->rot_pc * tiles_n)
                                               : (int)std::min<int64_t>(num_pairs, 2 * (int64_t)clusters);
            }
        } else {
            // GEMM+AR keeps a pair's R units consecutive: its reduction is split over them (two-shot)
            p->rank_group = 1;
        }
        // caller's order overrides (are_workspace_set_gemm_order); they change the
        // order of the work units only, never the arithmetic
        if (ws->order_group_m > 0) p->group_m = (int)std::min<int64_t>(p->pairs_m, ws->order_group_m);
        if (ws->order_block > 0) {
            p->block_tiles = ws->order_block;
            p->rank_group = ws->order_rank_group > 0 ? std::min(ws->order_rank_group, R) : 1;
        } else if (ws->order_block < 0) {
            p->block_tiles = 0;
        }
        p->cons = ws->d_cons;
        if (p->block_tiles > 0) {
            const int64_t blocks = (num_pairs + p->block_tiles - 1) / p->block_tiles;
            p->num_pair_units = (int)(blocks * p->block_tiles * R);
        }
        const int grid = 2 * (int)std::min<int64_t>(p->num_pair_units, clusters);
        ws->last = are_launch_info{ARE_KERNEL_GEMM_PAIR, grid, gemm_pair_threads(), 2, p->block_tiles,
                                   (mode == kModeAR || p->rs_split) ? 1 : 0,
                                   p->block_tiles > 0 ? p->rank_group : R, p->group_m};
        e = launch_gemm_pair(*p, mode, grid, s);
    } else {
        p->group_m = (int)std::min<int64_t>(tiles_m, 8);
        // as many CTAs as keep every one busy for the same number of units: with more units
        // than SMs, the last wave no longer runs on a fraction of the SMs while the rest idle
        // (streaming-bound problems then keep the full DRAM bandwidth to the end)
        const int64_t waves = ceil_div(p->num_units, (int64_t)ws->num_sms);
        const int grid = (int)ceil_div(p->num_units, waves);
        ws->last = are_launch_info{ARE_KERNEL_GEMM_ONE_CTA, grid, kGemmThreads, 1, 0, 0, R, p->group_m};
        e = launch_gemm_reduce(*p, mode, grid, s);
    }
    if (e == cudaSuccess && p->chunk_ctr) ++ws->rs_generation;
    delete p;
    return from_cuda(e);
}

}  // namespace

extern "C" {

int are_version(void) { return (1 << 16) | 0; }

const char* are_status_string(are_status s) {
    switch (s) {
        case ARE_OK: return "ARE_OK";
        case ARE_EINVAL: return "ARE_EINVAL: invalid argument";
        case ARE_ENOMEM: return "ARE_ENOMEM: device allocation failed";
        case ARE_ECUDA: return "ARE_ECUDA: CUDA call or launch failed";
        case ARE_ETIMEOUT: return "ARE_ETIMEOUT: a bounded device wait expired";
        case ARE_EBUSY: return "ARE_EBUSY: workspace in use by another thread";
        case ARE_ENODEV: return "ARE_ENODEV: current device is not sm_103";
        case ARE_ECAPACITY: return "ARE_ECAPACITY: call exceeds workspace capacity";
        case ARE_ECAPTURE: return "ARE_ECAPTURE: one-time set-up needed inside a stream capture";
    }
    return "unknown are_status";
}

are_status are_supports(int op, int R, int64_t M, int64_t N, int64_t K) {
    const int64_t kLim = (int64_t)1 << 31;
    if (!ranks_ok(R) || M < 0 || N < 0 || M >= kLim || N >= kLim) return ARE_EINVAL;
    switch (op) {
        case ARE_OP_GEMM_RS:
            if (K < 0 || K >= kLim || K % 8 || N % 8 || M % R || (M / R) % 8) return ARE_EINVAL;
            if (ceil_div(M, kBM) * ceil_div(N, kBN) * R >= kLim) return ARE_EINVAL;
            return ARE_OK;
        case ARE_OP_GEMM_AR:
            if (K < 0 || K >= kLim || K % 8 || N % 8) return ARE_EINVAL;
            if (ceil_div(M, kBM) * ceil_div(N, kBN) * R >= kLim) return ARE_EINVAL;
            return ARE_OK;
        case ARE_OP_ALLREDUCE_RMSNORM:
            if (N % 8 || N > 32768) return ARE_EINVAL;
            return ARE_OK;
        default:
            return ARE_EINVAL;
    }
}

are_status are_workspace_create(are_ws** out, const are_caps* caps) {
    if (!out || !caps) return ARE_EINVAL;
    *out = nullptr;
    if (!ranks_ok(caps->R_max) || caps->M_max < 1 || caps->N_max < 8 || caps->N_max % 8 || caps->K_max < 0)
        return ARE_EINVAL;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ARE_ENODEV;
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return from_cuda(e);
    if (prop.major != 10 || prop.minor != 3) return ARE_ENODEV;

    are_ws* ws = new (std::nothrow) are_ws;
    if (!ws) return ARE_ENOMEM;
    ws->device = dev;
    ws->num_sms = prop.multiProcessorCount;
    ws->caps = *caps;
    ws->debug_flags = caps->debug_flags;
    ws->oneshot_max_bytes = kOneShotMaxBytes;
    ws->timeout_ns = caps->timeout_ns ? caps->timeout_ns : kDefaultTimeoutNs;

    e = cudaMalloc(&ws->d_status, sizeof(DevStatus));
    if (e == cudaSuccess) e = cudaMalloc(&ws->d_counters, kCounterWords * 8);
    if (e == cudaSuccess && caps->K_max > 0) {
        const int64_t T = ceil_div(caps->M_max, kBM) * ceil_div(caps->N_max, kBN);
        ws->mask_words = (size_t)T;
        ws->part_bytes = (size_t)caps->R_max * (size_t)T * kTilePartBytes;
        ws->piece_words = (size_t)T * kPieceWords;
        e = cudaMalloc(&ws->d_mask, ws->mask_words * 4);
        if (e == cudaSuccess) e = cudaMalloc(&ws->d_part, ws->part_bytes);
        if (e == cudaSuccess) e = cudaMalloc(&ws->d_pieces, ws->piece_words * 4);
        if (e == cudaSuccess) e = cudaMalloc(&ws->d_chunk_ctr, (size_t)caps->R_max * kChunkCap * 8);
        if (e == cudaSuccess) e = cudaMalloc(&ws->d_cons, ws->mask_words * 4);
        if (e == cudaSuccess)
            e = cudaHostAlloc(reinterpret_cast<void**>(&ws->h_chunk_gen), (size_t)caps->R_max * kChunkCap * 4,
                              cudaHostAllocMapped);
        if (e == cudaSuccess)
            e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&ws->d_chunk_gen), ws->h_chunk_gen, 0);
        if (e == cudaSuccess) e = gemm_prepare_kernels();
        if (e == cudaSuccess) ws->pair_clusters = gemm_pair_max_clusters();
    }
    if (e == cudaSuccess && caps->N_max <= 32768) {
        ws->staging_words = (size_t)caps->M_max * (size_t)caps->N_max;
        e = cudaMalloc(&ws->d_staging, ws->staging_words * 4);
    }
    if (e == cudaSuccess) {
        for (int ppt = 1; ppt <= kArMaxPpt; ++ppt) ws->ar_resident[ppt] = ar_rmsnorm_resident_blocks(ppt, ws->num_sms);
        if (e == cudaSuccess) e = ar_oneshot_prepare();
    }
    if (e != cudaSuccess) {
        are_status st = from_cuda(e);
        free_ws(ws);
        return st;
    }
    are_status st = arm_workspace(ws);
    if (st != ARE_OK) {
        free_ws(ws);
        return st;
    }
    *out = ws;
    return ARE_OK;
}

are_status are_workspace_destroy(are_ws* ws) {
    if (!ws) return ARE_OK;
    cudaError_t e = cudaDeviceSynchronize();
    free_ws(ws);
    return from_cuda(e);
}

are_status are_workspace_reset(are_ws* ws) {
    if (!ws) return ARE_EINVAL;
    TryLock lk(ws->mu);
    if (!lk.ok) return ARE_EBUSY;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return from_cuda(e);
    return arm_workspace(ws);
}

are_status are_workspace_set_debug(are_ws* ws, uint32_t flags, int64_t arg) {
    if (!ws) return ARE_EINVAL;
    TryLock lk(ws->mu);
    if (!lk.ok) return ARE_EBUSY;
    ws->debug_flags = flags;
    ws->debug_arg = arg;
    return ARE_OK;
}

are_status are_workspace_set_gemm_order(are_ws* ws, int group_m, int block_pairs, int rank_group) {
    if (!ws || group_m < 0 || rank_group < 0 || rank_group > kMaxRanks) return ARE_EINVAL;
    TryLock lk(ws->mu);
    if (!lk.ok) return ARE_EBUSY;
    ws->order_group_m = group_m;
    ws->order_block = block_pairs;
    ws->order_rank_group = rank_group;
    return ARE_OK;
}

are_status are_workspace_set_chunks(are_ws* ws, int chunks, int stripe) {
    if (!ws || chunks < 0 || chunks > kChunkCap || stripe < -1) return ARE_EINVAL;
    TryLock lk(ws->mu);
    if (!lk.ok) return ARE_EBUSY;
    if (chunks > 0 && !ws->d_chunk_ctr) return ARE_ECAPACITY;
    ws->chunks = chunks;
    ws->chunk_stripe = stripe;
    return ARE_OK;
}

are_status are_chunk_generation(are_ws* ws, uint64_t* generation) {
    if (!ws || !generation) return ARE_EINVAL;
    TryLock lk(ws->mu);
    if (!lk.ok) return ARE_EBUSY;
    *generation = ws->rs_generation;
    return ARE_OK;
}

are_status are_chunk_wait(are_ws* ws, int segment, int chunk, uint64_t generation, uint64_t timeout_ns) {
    if (!ws || !ws->h_chunk_gen || segment < 0 || segment >= ws->caps.R_max || chunk < 0 || chunk >= kChunkCap)
        return ARE_EINVAL;
    // the mapped word holds the chunk's generation modulo 2^32; compare in that ring
    const volatile uint32_t* w = ws->h_chunk_gen + (size_t)segment * kChunkCap + chunk;
    const uint32_t want = (uint32_t)generation;
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        if ((int32_t)(*w - want) >= 0) {
            std::atomic_thread_fence(std::memory_order_acquire);
            return ARE_OK;
        }
        const auto dt = std::chrono::steady_clock::now() - t0;
        if ((uint64_t)std::chrono::duration_cast<std::chrono::nanoseconds>(dt).count() > timeout_ns)
            return ARE_ETIMEOUT;
    }
}

are_status are_workspace_set_oneshot_max_bytes(are_ws* ws, uint64_t bytes) {
    if (!ws) return ARE_EINVAL;
    TryLock lk(ws->mu);
    if (!lk.ok) return ARE_EBUSY;
    ws->oneshot_max_bytes = bytes;
    return ARE_OK;
}

are_status are_get_device_status(are_ws* ws, are_dev_status* out) {
    if (!ws || !out) return ARE_EINVAL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return from_cuda(e);
    DevStatus d;
    e = cudaMemcpy(&d, ws->d_status, sizeof(d), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return from_cuda(e);
    out->code = d.code;
    out->where = d.where;
    out->a = d.a;
    out->b = d.b;
    return d.code == ARE_DEV_OK ? ARE_OK : ARE_ETIMEOUT;
}

are_status are_debug_last_launch(are_ws* ws, are_launch_info* out) {
    if (!ws || !out) return ARE_EINVAL;
    TryLock lk(ws->mu);
    if (!lk.ok) return ARE_EBUSY;
    *out = ws->last;
    return ARE_OK;
}

are_status are_debug_snapshot(are_ws* ws, int kind, void* host_dst, size_t bytes) {
    if (!ws || !host_dst) return ARE_EINVAL;
    const void* src = nullptr;
    size_t avail = 0;
    switch (kind) {
        case ARE_SNAP_MASKS: src = ws->d_mask; avail = ws->mask_words * 4; break;
        case ARE_SNAP_STAGING: src = ws->d_staging; avail = ws->staging_words * 4; break;
        case ARE_SNAP_PIECES: src = ws->d_pieces; avail = ws->piece_words * 4; break;
        case ARE_SNAP_COUNTERS: src = ws->d_counters; avail = kCounterWords * 8; break;
        case ARE_SNAP_CHUNKS: src = ws->d_chunk_ctr; avail = ws->d_chunk_ctr ? (size_t)ws->caps.R_max * kChunkCap * 8 : 0;
            break;
        default: return ARE_EINVAL;
    }
    if (!src || bytes > avail) return ARE_EINVAL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(host_dst, src, bytes, cudaMemcpyDeviceToHost);
    return from_cuda(e);
}

are_status are_gemm_rs(const are_bf16* const A[], const are_bf16* const B[], are_bf16* const out[], int R,
                       int64_t M, int64_t N, int64_t K, are_ws* ws, void* stream) {
    return gemm_call(kModeRS, A, B, out, R, M, N, K, ws, stream);
}

are_status are_gemm_ar(const are_bf16* const A[], const are_bf16* const B[], are_bf16* const out[], int R,
                       int64_t M, int64_t N, int64_t K, are_ws* ws, void* stream) {
    return gemm_call(kModeAR, A, B, out, R, M, N, K, ws, stream);
}

}  // extern "C"

namespace {

are_status allreduce_rmsnorm_call(const are_bf16* const partials[], const are_bf16* residual, const float* gamma,
                                  float eps, are_bf16* out, are_bf16* residual_out, uint8_t* out_q, float* out_scale,
                                  int R, int64_t M, int64_t N, are_ws* ws, void* stream) {
    if (!ws || !partials) return ARE_EINVAL;
    if (residual_out && !ptr_ok(residual_out, M * N)) return ARE_EINVAL;
    const bool quant = out_q != nullptr || out_scale != nullptr;
    if (quant && (!ptr_ok(out_q, M * N) || !ptr_ok(out_scale, M))) return ARE_EINVAL;
    are_status st = are_supports(ARE_OP_ALLREDUCE_RMSNORM, R, M, N, 0);
    if (st != ARE_OK) return st;
    for (int r = 0; r < R; ++r)
        if (!ptr_ok(partials[r], M * N)) return ARE_EINVAL;
    if ((residual && !aligned16(residual)) || !ptr_ok(gamma, N) || (!quant && !ptr_ok(out, M * N))) return ARE_EINVAL;
    if (!(eps > 0.f) || !std::isfinite(eps)) return ARE_EINVAL;
    TryLock lk(ws->mu);
    if (!lk.ok) return ARE_EBUSY;
    if (R > ws->caps.R_max || M > ws->caps.M_max || N > ws->caps.N_max || !ws->d_staging ||
        (size_t)M * (size_t)N > ws->staging_words)
        return ARE_ECAPACITY;
    ws->last = are_launch_info{};
    if (M == 0 || N == 0) return ARE_OK;

    ArParams p;
    std::memset(&p, 0, sizeof(p));
    for (int r = 0; r < R; ++r) p.x[r] = partials[r];
    p.residual = residual;
    p.gamma = gamma;
    p.out = out;
    p.residual_out = residual_out;
    p.out_q = out_q;
    p.out_scale = out_scale;
    p.staging = ws->d_staging;
    p.status = ws->d_status;
    p.counters = ws->d_counters;
    p.R = R;
    p.M = (int)M;
    p.N = (int)N;
    p.packs_per_row = (int)(N / 8);
    const int ppt = ar_rmsnorm_ppt(p.packs_per_row);
    const int resident = ppt > 0 ? ws->ar_resident[ppt] : 0;
    if (resident <= 0) return ARE_ECUDA;
    const int grid = std::min(resident, 2 * ws->num_sms);
    p.chunk_rows = grid;
    ar_rmsnorm_smem_plan(p);
    p.ring_slots = (M + grid - 1) / grid > kArRingSlots ? kArRingSlots : 0;
    p.num_chunks = (int)ceil_div(M, grid);
    p.eps = eps;
    p.inv_n = 1.0f / (float)N;
    p.flags = ws->debug_flags;
    p.debug_arg = ws->debug_arg;
    p.timeout_ns = ws->timeout_ns;
    ws->last_ar_M = M;
    ws->last_ar_N = N;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Small messages take the one-shot kernel (no staging), larger ones the Lamport
    // kernel; the threshold is a per-rank input size, as in the pages' dispatch.
    const bool fits = ar_oneshot_fits(R, (int)N, residual != nullptr);
    const bool oneshot = fits && !(ws->debug_flags & ARE_DEBUG_AR_LAMPORT) &&
                         ((ws->debug_flags & ARE_DEBUG_AR_ONESHOT) || (uint64_t)M * (uint64_t)N * 2 <= ws->oneshot_max_bytes);
    if (oneshot) {
        const int os_grid = (int)std::min<int64_t>(M, ws->num_sms);
        ws->last = are_launch_info{ARE_KERNEL_AR_ONESHOT, os_grid, ar_oneshot_threads(), 1, 0, ppt, 0, 0};
        return from_cuda(launch_ar_oneshot(p, ppt, os_grid, s));
    }
    ws->last = are_launch_info{ARE_KERNEL_AR_LAMPORT, grid, kArThreads, 1, 0, ppt, 0, 0};
    return from_cuda(launch_ar_rmsnorm(p, ppt, grid, s));
}

}  // namespace

extern "C" {

are_status are_allreduce_rmsnorm(const are_bf16* const partials[], const are_bf16* residual, const float* gamma,
                                 float eps, are_bf16* out, int R, int64_t M, int64_t N, are_ws* ws, void* stream) {
    return allreduce_rmsnorm_call(partials, residual, gamma, eps, out, nullptr, nullptr, nullptr, R, M, N, ws, stream);
}

are_status are_allreduce_add_rmsnorm(const are_bf16* const partials[], const are_bf16* residual, const float* gamma,
                                     float eps, are_bf16* out, are_bf16* residual_out, int R, int64_t M, int64_t N,
                                     are_ws* ws, void* stream) {
    return allreduce_rmsnorm_call(partials, residual, gamma, eps, out, residual_out, nullptr, nullptr, R, M, N, ws,
                                  stream);
}

are_status are_allreduce_rmsnorm_quant(const are_bf16* const partials[], const are_bf16* residual, const float* gamma,
                                       float eps, uint8_t* out_q, float* out_scale, are_bf16* residual_out, int R,
                                       int64_t M, int64_t N, are_ws* ws, void* stream) {
    return allreduce_rmsnorm_call(partials, residual, gamma, eps, nullptr, residual_out, out_q, out_scale, R, M, N,
                                  ws, stream);
}

}  // extern "C"
