// Internal interfaces between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/are.h"

namespace are {

constexpr int kMaxRanks = 8;

// Device status word: first error wins (code 0 = no error).
struct DevStatus {
    uint32_t code;
    uint32_t where;
    int32_t a;
    int32_t b;
};

__device__ __forceinline__ void record_error(DevStatus* st, uint32_t code, uint32_t where, int32_t a, int32_t b) {
    if (atomicCAS(&st->code, 0u, code) == 0u) {
        st->where = where;
        st->a = a;
        st->b = b;
        __threadfence();
    }
}

// ------------------------------------------------------------------ AR+RMSNorm
constexpr uint32_t kSentinelF32 = 0x80000000u;  // -0.0 as an fp32 word
constexpr int kArThreads = 512;   // 1 producer warp + 7 phase-A warps + 8 phase-B warps
constexpr int kMaxArStages = 8;   // phase-A shared-memory stages (upper bound)
constexpr int kArRingSlots = 8;   // staging ring slots (chunks) when the rows wrap

struct ArParams {
    const uint16_t* x[kMaxRanks];  // R bf16 partials [M, N]
    const uint16_t* residual;      // bf16 [M, N] or nullptr
    const float* gamma;            // fp32 [N]
    uint16_t* out;                 // bf16 [M, N]
    uint16_t* residual_out;        // bf16 [M, N] or nullptr: bf16(h), h = canon(s) + residual
    uint8_t* out_q;                // FP8 E4M3 [M, N] or nullptr (then `out` is written)
    float* out_scale;              // fp32 [M] with out_q: the per-row scale
    uint32_t* staging;             // fp32 words, armed with the sentinel (chunk rows, see ring_slots)
    DevStatus* status;
    unsigned long long* counters;  // debug counters
    int R;
    int M;
    int N;
    int packs_per_row;  // N / 8
    int chunk_rows;     // rows per pipeline chunk (<= grid)
    int num_chunks;
    int ring_slots;     // 0: chunk c's rows at c*chunk_rows; else staging slot c % ring_slots
    int stages;         // phase-A shared-memory stages (set by ar_rmsnorm_smem_plan)
    int res_in_smem;    // residual rows streamed into shared memory (set by ar_rmsnorm_smem_plan)
    int gamma_in_smem;  // gamma copied into shared memory once per block (set by ar_rmsnorm_smem_plan)
    float eps;
    float inv_n;
    uint32_t flags;
    int64_t debug_arg;
    uint64_t timeout_ns;
};

// Packs-per-thread variant for a row of `packs_per_row` 8-element packs (0 if too wide).
int ar_rmsnorm_ppt(int packs_per_row);
constexpr int kArMaxPpt = 20;
// Choose the phase-A stage count and whether residual rows go through shared
// memory (needs p.N and p.residual set).
void ar_rmsnorm_smem_plan(ArParams& p);
// Largest grid that is fully co-resident for the packs-per-thread variant `ppt`.
int ar_rmsnorm_resident_blocks(int ppt, int num_sms);
cudaError_t launch_ar_rmsnorm(const ArParams& p, int ppt, int grid, cudaStream_t stream);
// One-shot AR+RMSNorm for small messages (one row per block, no staging).
size_t ar_oneshot_smem_bytes(int R, int N, bool residual);
bool ar_oneshot_fits(int R, int N, bool residual);
cudaError_t ar_oneshot_prepare();
cudaError_t launch_ar_oneshot(const ArParams& p, int ppt, int grid, cudaStream_t stream);
int ar_oneshot_threads();
// Fill n 32-bit words with v.
cudaError_t launch_fill_u32(uint32_t* dst, uint32_t v, size_t n, cudaStream_t stream);

// ------------------------------------------------------------------ GEMM + reduce
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 3;            // mainloop shared-memory stages
constexpr int kPStages = 3;           // partial_buf stages
constexpr int kSubBytes = 16384;      // one 128-row x 128-byte sub-tile
constexpr int kTilePartBytes = 131072;  // fp32 128x256 partial (bf16 uses the first half)
constexpr int kGemmThreads = 256;
constexpr int kPieceWords = 64;       // debug piece log words per tile
constexpr int kChunkCap = 64;         // completion counters per owner segment (largest chunk count)
constexpr unsigned long long kChunkQ = 1ull << 32;  // counter advance per completed chunk

enum GemmMode : int { kModeRS = 0, kModeAR = 1 };

struct GemmParams {
    CUtensorMap tmA[kMaxRanks];
    CUtensorMap tmB[kMaxRanks];
    CUtensorMap tmOut[kMaxRanks];  // GEMM+RS: owner segments (64 x H boxes); GEMM+AR: the distinct views
                                   // (64 x 128 boxes for the one-CTA kernel, 64 x 16 for the pair kernel)
    // CTA-pair kernel: the partial slots as [R][T][16 sub-tiles][128 rows][16 words], boxes of
    // 8 sub-tiles x 16 rows (one 8 KB partial-buffer stage of a row slice's 16-row group)
    CUtensorMap tmPart;
    are_bf16* views[kMaxRanks];  // GEMM+AR: distinct output views; GEMM+RS with rs_split: the owner
                                 // segments (row groups that no box covers: st.global)
    uint8_t* part;       // [R][T][tile part bytes]
    uint32_t* mask;      // [T]
    DevStatus* status;
    int32_t* pieces;     // debug piece log [T][kPieceWords]
    unsigned long long* counters;  // debug counters (wait profile)
    int R;
    int M, N, K;
    int S;               // owner segment rows (RS)
    int H;               // output box height (RS)
    int nviews;          // distinct output views (AR)
    int tiles_m, tiles_n, num_tiles, num_units, num_kb;
    int pairs_m, num_pair_units;  // CTA-pair kernel: 256-row tile pairs, R units per pair
    int block_tiles;     // CTA-pair kernel: tile pairs per rank block (0 = ranks innermost)
    int rs_split;        // CTA-pair kernel, GEMM+RS: 1 = every unit reduces its row slice of the tile
                         // (two-shot, as GEMM+AR); 0 = the running sum is pushed along the ranks
    int rank_group;      // CTA-pair kernel: ranks run together inside a block (1 = rank by rank)
    uint32_t* cons;      // CTA-pair kernel, GEMM+AR: row-slice readers done per tile (0 between calls)
    int group_m;         // tile raster: rows of tiles (pairs) per group
    // chunked owner-segment completion (GEMM+RS; chunk_ctr == nullptr: off)
    unsigned long long* chunk_ctr;  // [R][kChunkCap] monotonic completion counters
    uint32_t* chunk_host;           // [R][kChunkCap] completed generation, host-mapped (may be null)
    int chunks;          // requested chunks per owner segment
    // destination-rotated order of the pair kernel (rot_pc == 0: raster order)
    int rot_pc;          // pair rows per order chunk
    int rot_cs;          // order chunks per owner segment
    int rot_ps;          // pair rows per owner segment
    int rot_w;           // tile columns per destination rotation (stripe)
    uint32_t flags;
    int64_t debug_arg;
    uint64_t timeout_ns;
};

size_t gemm_smem_bytes();
cudaError_t gemm_prepare_kernels();
// bf16 [outer, inner] row-major tensor map, 128B-swizzled boxes of box_inner x box_outer.
cudaError_t make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                           uint32_t box_outer);
// The pair kernel's partial slots for T tiles and R ranks as a 5-D map (see GemmParams::tmPart).
cudaError_t make_tmap_part(CUtensorMap* m, const void* part, uint64_t T, uint64_t R);
cudaError_t launch_gemm_reduce(const GemmParams& p, int mode, int grid, cudaStream_t stream);
// CTA-pair variant (cta_group::2 UMMA, 256x256 per pair); grid = 2 x clusters.
cudaError_t launch_gemm_pair(const GemmParams& p, int mode, int grid, cudaStream_t stream);
// Largest number of co-resident 2-CTA clusters of the pair kernel on the current
// device (0 if unavailable); valid after gemm_prepare_kernels() on that device.
int gemm_pair_max_clusters();
int gemm_pair_threads();

}  // namespace are
