// Per-rank partial BF16 GEMMs on the 5th-generation tensor cores, reduced
// across the R emulated ranks by a bitmask-gated epilogue.
//
// Method: DeepGEMM PR #1 "Fused ring RS: per-tile bitmask + drain-ring with
// owner-boundary flush", description.  Its three points, as built here:
//   * readiness is a per-tile bitmask (bit r of word t = rank r's partial of
//     output tile t is in memory), not one flag per owner segment, so a
//     reducer starts on a tile as soon as that tile's R-1 peer partials exist;
//   * the peer partials reach the reducer through a multi-stage shared-memory
//     partial buffer fed by its own loader warp (the page's 2-stage buffer
//     could not hide the load latency and backed up into TMEM and the MMA);
//   * outputs leave through asynchronous TMA/bulk stores that are never
//     drained per tile by the whole epilogue: each staging buffer belongs to
//     one lane, which waits only for its own bulk group before reusing it
//     (DeepEP PR #527 "Fix the MultiStages for intranode combine", one stage
//     per lane), and a producer's publish waits only in the two issuing lanes.
// The page's title also names an owner-boundary flush: a reduced tile whose
// rows span several owner segments is cut at the segment boundaries and each
// piece is stored into its owner's segment.
//
// One-GPU design.  Two kernels implement it.  gemm_pair_kernel (further down)
// runs a CTA pair per 256x256 block with cta_group::2 MMAs; it takes GEMM+RS
// from two 128-row tiles on and GEMM+AR from one wave of tile pairs on (the
// host's dispatch also picks its GEMM+RS reduction: the running sum pushed
// along the ranks, or the row slices split over a tile's units for problems
// of a few waves).  gemm_reduce_kernel (next), one CTA per 128x256 tile,
// covers the rest.  Both share the workspace layout, the mask protocol and the
// owner-piece stores, and give the same bytes.
//
// gemm_reduce_kernel.  A work unit is (rank r, output tile t), a 128x256 tile of
// P_r = A_r B_r with K = K_r.  Units are ordered tile-major with the tile's
// reducer (the owner of the tile's first row for GEMM+RS, rank t mod R for
// GEMM+AR) last among its R units; a persistent grid (one CTA per SM) walks
// the units wave by wave, CTA b taking unit i*G + (b+i) mod G of wave i, so
// every wait points at a smaller unit index and the reducers rotate over the
// CTAs.  Non-reducer units store their partial tile (fp32 for RS, bf16 for AR)
// into the workspace and release-OR their bit; the reducer keeps its own
// partial in TMEM, waits (bounded) for the peers' bits, streams their
// sub-tiles through the partial buffer and adds all R in the order
// r = 0..R-1 in fp32.
//
// Warp roles (256 threads): warp 0 TMA producer, warp 1 MMA issuer (both run
// converged, one elected lane issuing), warp 2 TMEM allocator + partial loader,
// warp 3 idle, warps 4-7 epilogue (TMEM lane = tile row).  TMEM holds two
// 128x256 fp32 accumulators (512 columns).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "are_internal.h"
#include "ptx.cuh"

namespace are {
namespace {

constexpr uint32_t kAStageBytes = kBM * kBK * 2;  // 16 KB, K-major, 128B-swizzled
constexpr uint32_t kBStageBytes = kBN * kBK * 2;  // 32 KB, 4 boxes of 64(N) x 64(K), 128B-swizzled
constexpr uint32_t kStageTx = kAStageBytes + kBStageBytes;
constexpr int kNumBars = 2 * kStages + 4 + 2 * kPStages + 1;
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * (kAStageBytes + kBStageBytes) + (size_t)kPStages * kSubBytes +
                              2 * (size_t)kSubBytes + kNumBars * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// tcgen05 instruction descriptor (kind::f16): D fp32, A bf16, B bf16, A K-major,
// B MN-major, N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

// Shared-memory matrix descriptor: 128B swizzle, tcgen05 version bit.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

struct Unit {
    int t, r, own, tm, tn;
    bool reducer;
};

__device__ __forceinline__ Unit decode(const GemmParams& p, int mode, int u) {
    Unit U;
    U.t = u / p.R;
    const int j = u - U.t * p.R;
    const int per_group = p.group_m * p.tiles_n;
    const int g = U.t / per_group;
    const int first = g * p.group_m;
    const int gm = min(p.tiles_m - first, p.group_m);
    const int in = U.t - g * per_group;
    U.tm = first + in % gm;
    U.tn = in / gm;
    U.own = (mode == kModeRS) ? (U.tm * kBM) / p.S : U.t % p.R;
    int r = U.own + 1 + j;
    while (r >= p.R) r -= p.R;
    U.r = r;
    U.reducer = (j == p.R - 1);
    return U;
}

// Unit of wave i for CTA b: i*G + (b+i) mod G (a rotation per wave).
__device__ __forceinline__ int unit_of(int b, int i, int G) { return i * G + (b + i) % G; }

// Bounded wait on an mbarrier phase; gives up when the CTA aborts or the
// workspace timeout expires (recording the error).
// Roles off the MMA's critical path pass a back-off so that their polling
// leaves the SM's issue slots to the producer and MMA warps.
// The slow path (the phase was not complete at the first try) is out of line;
// the first try is inlined at every call site, so the producer and MMA warps,
// whose waits mostly find the phase complete, make no call per k-block
// (measured: GEMM+AR 633 -> 622 us, GEMM+RS 2607 -> 2567 us at the bench shapes).
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                           const GemmParams& p, int id, int unit, uint32_t backoff_ns) {
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (backoff_ns) ptx::nanosleep(backoff_ns);
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > p.timeout_ns) {
            record_error(p.status, ARE_DEV_PIPE_TIMEOUT, blockIdx.x, id, unit);
            *abort_flag = 1u;
            return false;
        }
    }
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         const GemmParams& p, int id, int unit, uint32_t backoff_ns = 0) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, abort_flag, p, id, unit, backoff_ns);
}

// Wait for an asynchronous copy that was already issued (it completes on its
// own); bounded, ignores the abort flag.
__device__ __noinline__ void drain_bar(uint64_t* bar, uint32_t parity, const GemmParams& p) {
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - t0 > p.timeout_ns) break;
    }
}

// wait_bar that, under ARE_DEBUG_WAIT_PROFILE, adds the SM cycles spent
// waiting to `acc`.
__device__ __forceinline__ bool wait_bar_prof(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                              const GemmParams& p, int id, int unit, uint64_t& acc,
                                              uint32_t backoff_ns = 0) {
    if (!(p.flags & ARE_DEBUG_WAIT_PROFILE)) return wait_bar(bar, parity, abort_flag, p, id, unit, backoff_ns);
    const uint64_t t0 = clock64();
    const bool ok = wait_bar(bar, parity, abort_flag, p, id, unit, backoff_ns);
    acc += (uint64_t)(clock64() - t0);
    return ok;
}
__device__ __forceinline__ void prof_add(const GemmParams& p, int slot, uint64_t v) {
    if ((p.flags & ARE_DEBUG_WAIT_PROFILE) && v) atomicAdd(&p.counters[slot], (unsigned long long)v);
}

// Named barriers are .aligned: every lane of a warp must arrive together, so
// each helper first reconverges the warp (lanes that ran a single-lane branch,
// such as issuing a store or an arrive, would otherwise arrive late and be
// counted in the barrier's next phase).
__device__ __forceinline__ void epi_bar() {
    __syncwarp();
    asm volatile("bar.sync 1, 128;" ::: "memory");
}
// Epilogue-wide OR of a predicate (uniform result for all 128 threads).
__device__ __forceinline__ bool epi_bar_or(bool v) {
    __syncwarp();
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Chunked owner-segment completion (ROCm/mori PR #662, the fused GEMM ->
// scatter follow-ups: per-(destination, chunk) completion counters, monotonic,
// with a modulo election).  The destinations are the owner segments: chunk c
// of segment s is a band of the n_s tile rows that intersect s, the requested
// chunk count halved until it divides n_s.  A reducer tile stores one piece
// into every segment its rows meet; once those stores have completed it adds
// 1 to each piece's (segment, chunk) counter with release.  The counters are
// never reset: every call starts at a multiple of kChunkQ, so the low 32 bits
// count this call's pieces, and the one add that sees `pieces - 1` there is
// the chunk's last (the modulo election).  The elected thread advances the
// counter to the next multiple of kChunkQ, so the next call starts at zero
// pieces whatever its shape, and publishes the chunk's generation (counter /
// kChunkQ) to the host-mapped word a host-side waiter polls.
__device__ __noinline__ void chunk_bump_tile(const GemmParams& p, int tm) {
    const int row0 = tm * kBM;
    const int row_end = min(row0 + kBM, p.M);
    for (int r0 = row0; r0 < row_end;) {
        const int s = r0 / p.S;
        const int e = min((s + 1) * p.S, row_end);
        const int t_lo = (int)(((long long)s * p.S) / kBM);
        const int t_hi = (int)(((long long)(s + 1) * p.S - 1) / kBM);
        const int n_s = t_hi - t_lo + 1;
        int cs = p.chunks;
        while (cs > 1 && n_s % cs) cs >>= 1;
        const int per = n_s / cs;
        const int idx = s * kChunkCap + (tm - t_lo) / per;
        const unsigned long long pieces = (unsigned long long)per * (unsigned long long)p.tiles_n;
        const unsigned long long old = ptx::atom_add_release_gpu_u64(&p.chunk_ctr[idx], 1ull);
        if ((old & (kChunkQ - 1)) + 1 == pieces) {
            if (!(p.flags & ARE_DEBUG_NO_REARM)) ptx::atom_add_release_gpu_u64(&p.chunk_ctr[idx], kChunkQ - pieces);
            if (p.chunk_host) ptx::st_release_sys(&p.chunk_host[idx], (uint32_t)((old >> 32) + 1));
        }
        r0 = e;
    }
}

// One 128-byte row of a 128B-swizzled 128-row sub-tile: 16-byte chunk c of row
// `row` lives at chunk position c ^ (row & 7).
__device__ __forceinline__ void write_row_sw128(uint8_t* base, int row, const uint32_t (&w)[32]) {
    uint8_t* rp = base + row * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(rp + ((c ^ (row & 7)) << 4)) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}
__device__ __forceinline__ void read_row_sw128(const uint8_t* base, int row, uint32_t (&w)[32]) {
    const uint8_t* rp = base + row * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(rp + ((c ^ (row & 7)) << 4));
        w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
    }
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_reduce_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + kStages * kAStageBytes;
    uint8_t* sP = sB + kStages * kBStageBytes;
    uint8_t* sOut = sP + kPStages * kSubBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(sOut + 2 * kSubBytes);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* pfull = tempty + 2;
    uint64_t* pempty = pfull + kPStages;
    uint64_t* mma_done = pempty + kPStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const int b = blockIdx.x;
    const int nsub = (MODE == kModeRS) ? 8 : 4;  // 16 KB sub-tiles per partial tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) { ptx::mbar_init(&full[s], 1); ptx::mbar_init(&empty[s], 1); }
        for (int s = 0; s < 2; ++s) { ptx::mbar_init(&tfull[s], 1); ptx::mbar_init(&tempty[s], 128); }
        for (int s = 0; s < kPStages; ++s) { ptx::mbar_init(&pfull[s], 1); ptx::mbar_init(&pempty[s], 128); }
        ptx::mbar_init(mma_done, 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_shared();
    }
    if (warp == 2) {
        ptx::tmem_alloc(tmem_slot, 512);
        ptx::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        for (int r = 0; r < p.R; ++r) { ptx::prefetch_tmap(&p.tmA[r]); ptx::prefetch_tmap(&p.tmB[r]); }
    }
    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // The whole warp runs the loop; one elected lane issues (see the pair kernel).
        const bool issuer = ptx::elect_one();
        const uint64_t pol = ptx::policy_evict_normal();
        int stage = 0;
        uint32_t ph = 0;
        uint32_t issued = 0, issued_ph = 0;  // bit s: stage s has a fill in flight; its parity
        for (int i = 0;; ++i) {
            if (i * G >= p.num_units) break;
            const int u = unit_of(b, i, G);
            if (u >= p.num_units) continue;
            const Unit U = decode(p, MODE, u);
            bool ok = true;
            for (int kb = 0; kb < p.num_kb; ++kb) {
                const bool eok = wait_bar(&empty[stage], ph ^ 1u, abort_flag, p, 0, u);
                if (!__all_sync(0xFFFFFFFFu, eok)) { ok = false; break; }
                if (issuer) {
                    ptx::mbar_arrive_expect_tx(&full[stage], kStageTx);
                    ptx::tma_load_2d(sA + stage * kAStageBytes, &p.tmA[U.r], &full[stage], kb * kBK, U.tm * kBM,
                                     pol);
#pragma unroll
                    for (int q = 0; q < kBN / 64; ++q)
                        ptx::tma_load_2d(sB + stage * kBStageBytes + q * 8192, &p.tmB[U.r], &full[stage],
                                         U.tn * kBN + q * 64, kb * kBK, pol);
                }
                __syncwarp();
                issued |= 1u << stage;
                issued_ph = (issued_ph & ~(1u << stage)) | (ph << stage);
                if (++stage == kStages) { stage = 0; ph ^= 1u; }
            }
            if (!ok) break;
        }
        for (int s = 0; s < kStages; ++s)
            if (issued & (1u << s)) drain_bar(&full[s], (issued_ph >> s) & 1u, p);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop with warp-uniform descriptors; one elected
        // lane issues every MMA and every commit.
        const bool issuer = ptx::elect_one();
        int stage = 0;
        uint32_t ph = 0;
        int it = 0;
        const uint64_t adesc0 = sdesc(ptx::smem_u32(sA), 16, 1024);
        const uint64_t bdesc0 = sdesc(ptx::smem_u32(sB), 8192, 1024);
        for (int i = 0;; ++i) {
            if (i * G >= p.num_units) break;
            const int u = unit_of(b, i, G);
            if (u >= p.num_units) continue;
            const int buf = it & 1;
            const uint32_t tph = (it >> 1) & 1;
            const bool tok = wait_bar(&tempty[buf], tph ^ 1u, abort_flag, p, 1, u);
            if (!__all_sync(0xFFFFFFFFu, tok)) break;
            ptx::tc_fence_after();
            const uint32_t d = tmem_base + buf * kBN;
            bool ok = true;
            for (int kb = 0; kb < p.num_kb; ++kb) {
                const bool fok = wait_bar(&full[stage], ph, abort_flag, p, 2, u);
                if (!__all_sync(0xFFFFFFFFu, fok)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint64_t ad = adesc0 + (uint64_t)(stage * (kAStageBytes >> 4));
                const uint64_t bd = bdesc0 + (uint64_t)(stage * (kBStageBytes >> 4));
                if (issuer) {
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)  // K16 steps: +32 bytes in A's rows, +16 rows of B
                        ptx::umma_bf16(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 128), kIdesc, (kb | kk) != 0);
                    ptx::umma_commit(&empty[stage]);
                    if (kb == p.num_kb - 1) ptx::umma_commit(&tfull[buf]);
                }
                __syncwarp();
                if (++stage == kStages) { stage = 0; ph ^= 1u; }
            }
            if (!ok) break;
            ++it;
        }
        // every MMA the issuing lane issued has completed once mma_done flips
        if (issuer) ptx::umma_commit(mma_done);
        __syncwarp();
        drain_bar(mma_done, 0, p);
    } else if (warp == 2) {
        // ------------------------------------------------------------ partial loader
        if (lane == 0) {
            int ps = 0;
            uint32_t pph = 0;
            uint32_t issued = 0, issued_ph = 0;
            const uint32_t full_mask = (p.R >= 32) ? 0xFFFFFFFFu : ((1u << p.R) - 1u);
            for (int i = 0;; ++i) {
                if (i * G >= p.num_units) break;
                const int u = unit_of(b, i, G);
                if (u >= p.num_units) continue;
                const Unit U = decode(p, MODE, u);
                if (!U.reducer) continue;
                const uint32_t need = full_mask & ~(1u << U.own);
                bool ok = true;
                if (need) {
                    uint32_t seen = ptx::ld_acquire_gpu(&p.mask[U.t]);
                    if ((seen & need) != need) {
                        const uint64_t t0 = ptx::globaltimer();
                        while (true) {
                            ptx::nanosleep(100);
                            seen = ptx::ld_acquire_gpu(&p.mask[U.t]);
                            if ((seen & need) == need) break;
                            if (*abort_flag || ptx::ld_relaxed_gpu(&p.status->code) != 0u) {
                                *abort_flag = 1u;
                                ok = false;
                                break;
                            }
                            if (ptx::globaltimer() - t0 > p.timeout_ns) {
                                record_error(p.status, ARE_DEV_MASK_TIMEOUT, blockIdx.x, U.t, (int32_t)seen);
                                *abort_flag = 1u;
                                ok = false;
                                break;
                            }
                        }
                    }
                    // generic-proxy acquire above, async-proxy (bulk copy) reads below
                    ptx::fence_proxy_async_global();
                }
                if (!ok) break;
                // only the tile's rows inside M were stored (128-byte rows, a sub-tile's row r at r * 128)
                const uint32_t vbytes = (uint32_t)min(kBM, p.M - U.tm * kBM) * 128u;
                for (int j = 0; j < nsub && ok; ++j) {
                    for (int q = 0; q < p.R; ++q) {
                        if (q == U.own) continue;
                        if (!wait_bar(&pempty[ps], pph ^ 1u, abort_flag, p, 3, u)) { ok = false; break; }
                        ptx::mbar_arrive_expect_tx(&pfull[ps], vbytes);
                        const uint8_t* src =
                            p.part + ((size_t)q * p.num_tiles + U.t) * kTilePartBytes + (size_t)j * kSubBytes;
                        ptx::bulk_load(sP + ps * kSubBytes, src, vbytes, &pfull[ps]);
                        issued |= 1u << ps;
                        issued_ph = (issued_ph & ~(1u << ps)) | (pph << ps);
                        if (++ps == kPStages) { ps = 0; pph ^= 1u; }
                    }
                }
                if (!ok) break;
            }
            for (int s = 0; s < kPStages; ++s)
                if (issued & (1u << s)) drain_bar(&pfull[s], (issued_ph >> s) & 1u, p);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int row = threadIdx.x - 128;  // tile row == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
        const bool lead = (warp == 4);
        int prev_tm = -1;  // chunk counting: the last reducer tile whose stores may still be in flight
        int it = 0, ps = 0;
        uint32_t pph = 0;
        bool bad = false;
        for (int i = 0;; ++i) {
            if (i * G >= p.num_units) break;
            const int u = unit_of(b, i, G);
            if (u >= p.num_units) continue;
            const Unit U = decode(p, MODE, u);
            const int buf = it & 1;
            const uint32_t tph = (it >> 1) & 1;
            if (!wait_bar(&tfull[buf], tph, abort_flag, p, 4, u)) bad = true;
            ptx::tc_fence_after();
            __syncwarp();
            const uint32_t tacc = tmem_base + lane_base + buf * kBN;
            const int row0 = U.tm * kBM;

            if (!U.reducer) {
                // ---- producer unit: TMEM -> registers -> swizzled smem -> bulk store -> publish
                // (a sub-tile's rows past M are never read: only the rows inside M are stored)
                uint8_t* gdst = p.part + ((size_t)U.r * p.num_tiles + U.t) * kTilePartBytes;
                const uint32_t vbytes = (uint32_t)min(kBM, p.M - row0) * 128u;
                for (int j = 0; j < nsub; ++j) {
                    uint32_t w[32];
                    if (MODE == kModeRS) {
                        ptx::tmem_ld32(tacc + j * 32, w);
                    } else {
                        uint32_t v0[32], v1[32];
                        ptx::tmem_ld32(tacc + j * 64, v0);
                        ptx::tmem_ld32(tacc + j * 64 + 32, v1);
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            w[c] = pack_bf16x2(__uint_as_float(v0[2 * c]), __uint_as_float(v0[2 * c + 1]));
                            w[16 + c] = pack_bf16x2(__uint_as_float(v1[2 * c]), __uint_as_float(v1[2 * c + 1]));
                        }
                    }
                    if (j == nsub - 1) {
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(&tempty[buf]);
                    }
                    const int sb = j & 1;
                    if (lead && lane == sb) ptx::bulk_wait_read0();
                    if (epi_bar_or(bad)) { bad = true; break; }
                    write_row_sw128(sOut + sb * kSubBytes, row, w);
                    ptx::fence_proxy_async_shared();
                    epi_bar();
                    if (lead && lane == sb) {
                        ptx::bulk_store(gdst + (size_t)j * kSubBytes, sOut + sb * kSubBytes, vbytes);
                        ptx::bulk_commit();
                    }
                }
                if (bad) break;
                if (lead) {
                    if (lane < 2) {
                        ptx::bulk_wait0();
                        ptx::fence_proxy_async_global();
                        __threadfence();
                    }
                    __syncwarp();
                    if (lane == 0 && !((p.flags & ARE_DEBUG_SKIP_PUBLISH) && (int64_t)u == p.debug_arg))
                        ptx::red_release_or(&p.mask[U.t], 1u << U.r);
                }
            } else {
                // ---- reducer unit: own partial in TMEM + R-1 peers through partial_buf
                if (lead && lane == 0) ptx::red_relaxed_or(&p.mask[U.t], 1u << U.own);
                for (int c = 0; c < kBN / 64; ++c) {  // 64-column output chunks
                    uint32_t outw[32];
                    if (MODE == kModeRS) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int j = 2 * c + h;
                            float acc[32];
                            for (int q = 0; q < p.R; ++q) {
                                uint32_t v[32];
                                if (q == U.own) {
                                    __syncwarp();
                                    ptx::tmem_ld32(tacc + j * 32, v);
                                } else {
                                    if (!wait_bar(&pfull[ps], pph, abort_flag, p, 5, u)) bad = true;
                                    read_row_sw128(sP + ps * kSubBytes, row, v);
                                    ptx::mbar_arrive(&pempty[ps]);
                                    if (++ps == kPStages) { ps = 0; pph ^= 1u; }
                                }
                                if (q == 0) {
#pragma unroll
                                    for (int e = 0; e < 32; ++e) acc[e] = __uint_as_float(v[e]);
                                } else {
#pragma unroll
                                    for (int e = 0; e < 32; ++e) acc[e] = acc[e] + __uint_as_float(v[e]);
                                }
                            }
#pragma unroll
                            for (int e = 0; e < 16; ++e) outw[16 * h + e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
                        }
                    } else {
                        const int j = c;
                        float acc[64];
                        for (int q = 0; q < p.R; ++q) {
                            uint32_t v[32];  // 64 bf16
                            if (q == U.own) {
                                uint32_t t0[32], t1[32];
                                __syncwarp();
                                ptx::tmem_ld32(tacc + j * 64, t0);
                                ptx::tmem_ld32(tacc + j * 64 + 32, t1);
#pragma unroll
                                for (int e = 0; e < 16; ++e) {
                                    v[e] = pack_bf16x2(__uint_as_float(t0[2 * e]), __uint_as_float(t0[2 * e + 1]));
                                    v[16 + e] = pack_bf16x2(__uint_as_float(t1[2 * e]), __uint_as_float(t1[2 * e + 1]));
                                }
                            } else {
                                if (!wait_bar(&pfull[ps], pph, abort_flag, p, 5, u)) bad = true;
                                read_row_sw128(sP + ps * kSubBytes, row, v);
                                ptx::mbar_arrive(&pempty[ps]);
                                if (++ps == kPStages) { ps = 0; pph ^= 1u; }
                            }
                            if (q == 0) {
#pragma unroll
                                for (int e = 0; e < 32; ++e) {
                                    acc[2 * e] = __uint_as_float(v[e] << 16);
                                    acc[2 * e + 1] = __uint_as_float(v[e] & 0xFFFF0000u);
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 32; ++e) {
                                    acc[2 * e] = acc[2 * e] + __uint_as_float(v[e] << 16);
                                    acc[2 * e + 1] = acc[2 * e + 1] + __uint_as_float(v[e] & 0xFFFF0000u);
                                }
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 32; ++e) outw[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
                    }
                    if (c == kBN / 64 - 1) {
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(&tempty[buf]);
                    }
                    const int sb = c & 1;
                    if (lead && lane == sb) ptx::bulk_wait_read0();
                    if (epi_bar_or(bad)) { bad = true; break; }
                    write_row_sw128(sOut + sb * kSubBytes, row, outw);
                    ptx::fence_proxy_async_shared();
                    epi_bar();
                    if (lead && lane == sb) {
                        const int x = U.tn * kBN + c * 64;
                        if (x < p.N) {
                            if (MODE == kModeRS) {
                                // owner-boundary flush: one store per (segment piece, H-row box)
                                const int row_end = min(row0 + kBM, p.M);
                                for (int r0 = row0; r0 < row_end;) {
                                    const int s = r0 / p.S;
                                    const int e = min((s + 1) * p.S, row_end);
                                    for (int rb = r0; rb < e; rb += p.H)
                                        ptx::tma_store_2d(&p.tmOut[s], sOut + sb * kSubBytes + (rb - row0) * 128, x,
                                                          rb - s * p.S);
                                    r0 = e;
                                }
                            } else {
                                for (int v = 0; v < p.nviews; ++v)
                                    ptx::tma_store_2d(&p.tmOut[v], sOut + sb * kSubBytes, x, row0);
                            }
                            ptx::bulk_commit();
                        }
                    }
                }
                if (bad) break;
                if (MODE == kModeRS && p.chunk_ctr && lead) {
                    // count the previous reducer tile's pieces once its stores have completed:
                    // each issuing lane waits for all but its groups of this tile (chunks lane, lane+2)
                    if (lane < 2 && prev_tm >= 0) {
                        int n = 0;
                        for (int c = lane; c < kBN / 64; c += 2) n += (U.tn * kBN + c * 64 < p.N) ? 1 : 0;
                        ptx::bulk_wait_upto(n);
                    }
                    __syncwarp();
                    if (lane == 0 && prev_tm >= 0) {
                        ptx::fence_proxy_async_global();
                        chunk_bump_tile(p, prev_tm);
                    }
                    prev_tm = U.tm;
                }
                if (lead && lane == 0) {
                    if (MODE == kModeRS && (p.flags & ARE_DEBUG_LOG_PIECES)) {
                        int32_t* log = p.pieces + (size_t)U.t * kPieceWords;
                        const int row_end = min(row0 + kBM, p.M);
                        int n = 0;
                        for (int r0 = row0; r0 < row_end && n < (kPieceWords - 3) / 3;) {
                            const int s = r0 / p.S;
                            const int e = min((s + 1) * p.S, row_end);
                            log[3 + 3 * n] = s; log[4 + 3 * n] = r0; log[5 + 3 * n] = e;
                            ++n;
                            r0 = e;
                        }
                        log[0] = U.tm; log[1] = U.tn; log[2] = n;
                    }
                    // re-arm the tile's mask word for the next call
                    if (!(p.flags & ARE_DEBUG_NO_REARM)) atomicExch(&p.mask[U.t], 0u);
                }
            }
            ++it;
        }
        if (bad) *abort_flag = 1u;
        if (lead && lane < 2) ptx::bulk_wait0();
        if (MODE == kModeRS && p.chunk_ctr && lead) {
            __syncwarp();
            if (lane == 0 && prev_tm >= 0 && !bad) {
                ptx::fence_proxy_async_global();
                chunk_bump_tile(p, prev_tm);
            }
        }
    }

    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 2) {
        __syncwarp();
        ptx::tmem_dealloc(tmem_base, 512);
    }
}

// ============================================================================
// CTA-pair variant: tcgen05.mma.cta_group::2 computes a 256x256 tile per CTA
// pair (cluster of 2).  Each CTA stages its own 128 rows of A and its own 128
// columns of B (32 KB per k-block, 5 stages) and holds its 128x256 half of the
// accumulator in its own TMEM; the leader (cluster rank 0) issues the MMAs.
// Each CTA's half is one 128x256 output tile with its own mask word and
// partial slot; the pair computes the same rank r for both halves.
//
// The epilogue:
//   warps 4-7   drain: TMEM -> registers -> swizzled staging -> 8 KB bulk
//               stores into the unit's partial slot; the accumulator goes
//               back to the MMA as soon as it is read, and the unit's bit is
//               release-ORed once the two issuing lanes' stores completed.
//               GEMM+RS pushes a running sum along the ranks: rank r's drain
//               first adds S_(r-1) (fed by the loader warp into the 3-stage
//               partial buffer once bit r-1 is set) and stores S_r; the last
//               rank rounds to bf16 and stores the owner pieces with TMA.
//               Problems of a few waves, where that chain of drains would be
//               the tail, split the reduction instead (rs_split): every unit
//               stores its fp32 partial, as GEMM+AR does its bf16 partial (at
//               R = 8 without its own row slice, which stays in shared memory);
//   warps 8-11  reduce, two-shot (GEMM+AR, and GEMM+RS with rs_split): every
//               unit sums its row slice of the tile's R partials in the order
//               r = 0..R-1, fed by the loader warp, and writes it to every view
//               (GEMM+AR) or to the rows' owner segments (GEMM+RS).
// The drain never waits on a reduction (apart from GEMM+AR's bounded
// own-slice wait, see the kernel), and the MMA never waits on the exchange.
// ============================================================================
constexpr int kStages2 = 5;
constexpr int kPStages2 = 3;
// Partial sub-tile of the pair kernel: 128 rows x 64 bytes (16 fp32 or 32 bf16
// columns), 64-byte swizzled.  Small sub-tiles keep the partial buffer and the
// drain staging at 40 KB, which leaves room for five mainloop stages.
constexpr uint32_t kPSub2 = 8192;
constexpr int kAccBufs2 = 2;                         // TMEM accumulator buffers per CTA
constexpr uint32_t kTmemCols2 = 256 * kAccBufs2;
constexpr int kPairThreads = 384;
constexpr uint32_t kAHalfBytes = kBM * kBK * 2;      // 16 KB: 128 rows of A
constexpr uint32_t kBHalfBytes = (kBN / 2) * kBK * 2;  // 16 KB: 128 columns of B (two 64x64 boxes)
constexpr uint32_t kStageTx2 = kAHalfBytes + kBHalfBytes;
constexpr int kNumBars2 = 2 * kStages2 + 2 * kAccBufs2 + 2 * kPStages2 + 1 + 2;
// A/B stages, partial buffer, one reduce staging buffer, two drain staging buffers, one 8 KB buffer
// that with the reduce staging buffer's second half holds GEMM+AR's own row slices
constexpr size_t kSmemBytes2 = 1024 + (size_t)kStages2 * (kAHalfBytes + kBHalfBytes) +
                               (size_t)kPStages2 * kPSub2 + (size_t)kSubBytes + 3 * (size_t)kPSub2 +
                               kNumBars2 * 8 + 16;
static_assert(kSmemBytes2 <= 232448, "shared memory budget (pair)");
// D fp32, A/B bf16, A K-major, B MN-major, N = 256, M = 256 (pair).
constexpr uint32_t kIdesc2 = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(kBN >> 3) << 17) |
                             ((uint32_t)(256 >> 4) << 24);

struct PUnit {
    int t;        // this CTA's 128x256 tile (row-major tile index)
    int tp;       // position of the tile pair in the unit order
    int j;        // position of the unit among its pair's R units (GEMM+AR: the row slice it reduces)
    int tm, tn, r;
    bool valid;
    bool pad;     // padding unit of the last rank block: skipped by every role
};

// Pair-unit order.  block_tiles == 0: the R units of a tile pair are
// consecutive (ranks innermost).  block_tiles == B with rank_group == g: tile
// pairs are taken in blocks of B (in raster order); inside a block the ranks
// run in groups of g: for the k-th group, every pair of the block runs its
// units j = k*g .. k*g+g-1 (consecutively) before the next group starts.  g = 1
// is rank by rank (a wave streams the operands of one or two ranks), g = R is
// ranks innermost.  Units past the last pair (padding of the last block) are
// not valid.
__device__ __forceinline__ PUnit decode_pair(const GemmParams& p, int mode, int u, int q) {
    PUnit U;
    int tp, j;
    if (p.block_tiles > 0) {
        const int B = p.block_tiles;
        const int g = p.rank_group > 0 ? p.rank_group : 1;
        const int per_block = B * p.R;
        const int blk = u / per_block;
        int rem = u - blk * per_block;
        const int k = rem / (B * g);           // rank group
        const int gk = min(g, p.R - k * g);    // ranks in this group
        rem -= k * B * g;
        const int pib = rem / gk;              // pair in block
        j = k * g + (rem - pib * gk);
        tp = blk * B + pib;
    } else {
        tp = u / p.R;
        j = u - tp * p.R;
    }
    const int num_pairs = p.pairs_m * p.tiles_n;
    U.tp = tp;
    U.j = j;
    U.pad = tp >= num_pairs;
    if (U.pad) {  // padding unit: no tile
        U.t = 0; U.tm = p.tiles_m; U.tn = 0; U.r = 0;
        U.valid = false;
        return U;
    }
    int tmp;
    if (p.rot_pc > 0) {
        // destination-rotated, chunk-major order (ROCm/mori PR #662, the follow-ups on
        // the destination-rotated tile order and its striped variant): chunk c of every
        // owner segment before chunk c+1 of any; inside a chunk, every segment's band
        // of rot_w tile columns before the next band of columns
        const int Pc = p.rot_pc, W = p.rot_w, TN = p.tiles_n;
        const int per_c = p.R * Pc * TN;
        const int c = tp / per_c;
        int rem = tp - c * per_c;
        const int ngroups = (TN + W - 1) / W;
        const int gi = min(rem / (p.R * Pc * W), ngroups - 1);
        rem -= gi * p.R * Pc * W;
        const int Wg = min(W, TN - gi * W);
        const int s = rem / (Pc * Wg);
        rem -= s * Pc * Wg;
        tmp = s * p.rot_ps + c * Pc + rem % Pc;
        U.tn = gi * W + rem / Pc;
    } else {
        const int per_group = p.group_m * p.tiles_n;
        const int g = tp / per_group;
        const int first = g * p.group_m;
        const int gm = min(p.pairs_m - first, p.group_m);
        const int in = tp - g * per_group;
        tmp = first + in % gm;
        U.tn = in / gm;
    }
    // A pair runs its ranks in the order 0..R-1: GEMM+RS on the ring pushes the running sum
    // from rank to rank (rank r waits only for the same tile's rank r-1, an earlier unit), and
    // a two-shot unit (GEMM+AR, GEMM+RS with rs_split) reduces its row slice once all R units
    // have published (later units never wait on a reduction, so that wait ends too).
    U.r = j;
    U.tm = 2 * tmp + q;
    U.valid = U.tm < p.tiles_m;
    U.t = U.tm * p.tiles_n + U.tn;
    return U;
}

// Row `row` of a 128 x 64-byte sub-tile: 16-byte chunk c lives at chunk
// c ^ ((row >> 1) & 3), so the 32 rows of a warp touching one chunk column
// spread evenly over the banks (four wavefronts per 512 bytes, the minimum).
// H selects which 16 words of `w` (columns 16H..16H+15 of a 32-word row).
template <int H>
__device__ __forceinline__ void write_half_sw64(uint8_t* base, int row, const uint32_t (&w)[32]) {
    uint8_t* rp = base + row * 64;
#pragma unroll
    for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(rp + ((c ^ ((row >> 1) & 3)) << 4)) =
            make_uint4(w[16 * H + 4 * c], w[16 * H + 4 * c + 1], w[16 * H + 4 * c + 2], w[16 * H + 4 * c + 3]);
}
__device__ __forceinline__ void read_row_sw64(const uint8_t* base, int row, uint32_t (&w)[16]) {
    const uint8_t* rp = base + row * 64;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(rp + ((c ^ ((row >> 1) & 3)) << 4));
        w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
    }
}

template <int ID>
__device__ __forceinline__ void grp_bar() {
    __syncwarp();
    asm volatile("bar.sync %0, 128;" ::"n"(ID) : "memory");
}
template <int ID>
__device__ __forceinline__ bool grp_bar_or(bool v) {
    __syncwarp();
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(ID)
        : "memory");
    return r != 0;
}

// Partial slot of rank r for this CTA's 128x256 tile: every tile has its own
// slot per rank in the workspace.
__device__ __forceinline__ uint8_t* pair_slot(const GemmParams& p, const PUnit& U, int r) {
    return p.part + ((size_t)r * p.num_tiles + U.t) * kTilePartBytes;
}

template <int MODE>
__global__ void __launch_bounds__(kPairThreads, 1) gemm_pair_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + kStages2 * kAHalfBytes;
    uint8_t* sP = sB + kStages2 * kBHalfBytes;
    uint8_t* sOut = sP + kPStages2 * kPSub2;     // reduce staging (1 buffer)
    uint8_t* sDrain = sOut + kSubBytes;          // drain staging (2 buffers of kPSub2)
    // GEMM+AR at R = 8: a unit's own 16-row slice (8 sub-tiles x 16 rows x 64 bytes) stays on chip
    uint8_t* const sOwn0 = sOut + kPSub2;
    uint8_t* const sOwn1 = sDrain + 2 * kPSub2;
    uint64_t* full = reinterpret_cast<uint64_t*>(sDrain + 3 * kPSub2);
    uint64_t* empty = full + kStages2;
    uint64_t* tfull = empty + kStages2;
    uint64_t* tempty = tfull + kAccBufs2;
    uint64_t* pfull = tempty + kAccBufs2;
    uint64_t* pempty = pfull + kPStages2;
    uint64_t* mma_done = pempty + kPStages2;
    uint64_t* ownfree = mma_done + 1;           // [2]: the reduce has read an own-slice buffer
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ownfree + 2);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t q = ptx::cluster_ctarank();  // 0 = leader
    // GEMM+AR with 16-row slices (R = 8): unit j's rank is j (every pair runs ranks 0..R-1), so the
    // slice it reduces, rows [16j, 16j+16), of its own partial never needs to leave the SM: the drain
    // keeps those rows in sOwn instead of storing them, and the slice reducer adds them at rank j's
    // place in the ring-order sum.  That saves 1/R of the partial exchange's writes and reads.
    // With two sOwn buffers the drain of a CTA's n-th valid unit waits for the reduction of its
    // (n-2)-th, the one place where a drain waits on a reduction.  That wait ends when a pair's R
    // units lie within two consecutive steps of the persistent loop: the reduction at step m then
    // needs drains at steps <= m + 1 only, so by induction over the steps every wait ends.  A
    // pair's units lie in a run of `run` consecutive units (R with the ranks consecutive, else the
    // pair's rank block), and runs start at multiples of `run`; such a run spans at most two steps
    // when it is at most G + 1 units long, or exactly 2G (then it starts at a step boundary).  Larger
    // rank blocks spread a pair over more steps, and there the own slice goes through memory like
    // the other ranks' slices.
    const int own_run = (p.block_tiles == 0 || p.rank_group >= p.R) ? p.R : p.block_tiles * p.R;
    const int G2own = (int)(gridDim.x >> 1);
    const bool own_slice = (MODE == kModeAR) && p.R == 8 && p.rot_pc == 0 &&
                           (own_run <= G2own + 1 || own_run == 2 * G2own);
    const int cl = blockIdx.x >> 1;
    const int G2 = gridDim.x >> 1;
    const int nsub = (MODE == kModeRS) ? 8 : 4;  // 128-byte column chunks of a partial row
    // GEMM+RS pushes its running sum along the ranks, or (rs_split) reduces like GEMM+AR: every
    // unit sums its row slice of the tile's R partials (two-shot)
    const bool ring = (MODE == kModeRS) && !p.rs_split;
    const bool split = !ring;
    // a 16-row group of a row slice is loaded as stages of 8 partial sub-tiles (8 KB): one for
    // GEMM+AR's bf16 partial rows (512 bytes), two for GEMM+RS's fp32 rows (1 KB)
    constexpr int kHalves = (MODE == kModeRS) ? 2 : 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages2; ++s) { ptx::mbar_init(&full[s], 1); ptx::mbar_init(&empty[s], 1); }
        for (int s = 0; s < kAccBufs2; ++s) { ptx::mbar_init(&tfull[s], 1); ptx::mbar_init(&tempty[s], 2); }
        for (int s = 0; s < kPStages2; ++s) { ptx::mbar_init(&pfull[s], 1); ptx::mbar_init(&pempty[s], 128); }
        ptx::mbar_init(mma_done, 1);
        for (int s = 0; s < 2; ++s) ptx::mbar_init(&ownfree[s], 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_shared();
    }
    if (warp == 2) {
        ptx::tmem_alloc_pair(tmem_slot, kTmemCols2);
        ptx::tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        for (int r = 0; r < p.R; ++r) { ptx::prefetch_tmap(&p.tmA[r]); ptx::prefetch_tmap(&p.tmB[r]); }
    }
    __syncwarp();
    ptx::tc_fence_before();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    volatile uint64_t* t_mma_end = reinterpret_cast<volatile uint64_t*>(tmem_slot + 2);  // wait profile only
    const uint64_t t_begin = (p.flags & ARE_DEBUG_WAIT_PROFILE) ? ptx::globaltimer() : 0;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        // The whole warp runs the loop (uniform operands); one elected lane issues.
        const bool issuer = ptx::elect_one();
        // A panels are reused by every tile column of a raster group: keep them in L2 ahead of
        // the B panels, which the group's pair rows share only while they run together
        const uint64_t pol_a = ptx::policy_evict_last();
        const uint64_t pol = ptx::policy_evict_normal();
        int stage = 0;
        uint32_t ph = 0;
        uint32_t issued = 0, issued_ph = 0;
        bool aborted = false;
        uint64_t w_empty = 0;
        for (int i = 0;; ++i) {
            if (i * G2 >= p.num_pair_units) break;
            const int u = i * G2 + (cl + i) % G2;
            if (u >= p.num_pair_units) continue;
            const PUnit U = decode_pair(p, MODE, u, (int)q);
            if (U.pad) continue;
            for (int kb = 0; kb < p.num_kb; ++kb) {
                const bool ok = wait_bar_prof(&empty[stage], ph ^ 1u, abort_flag, p, 10, u, w_empty);
                if (!__all_sync(0xFFFFFFFFu, ok)) {
                    aborted = true;
                    break;
                }
                if (issuer) {
                    // both CTAs' copies complete on the leader's full barrier
                    const uint32_t fb = ptx::mapa_shared(ptx::smem_u32(&full[stage]), 0);
                    if (q == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2 * kStageTx2);
                    ptx::tma_load_2d_pair(sA + stage * kAHalfBytes, &p.tmA[U.r], fb, kb * kBK, U.tm * kBM, pol_a);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        ptx::tma_load_2d_pair(sB + stage * kBHalfBytes + h * 8192, &p.tmB[U.r], fb,
                                              U.tn * kBN + (int)q * 128 + h * 64, kb * kBK, pol);
                }
                __syncwarp();
                issued |= 1u << stage;
                issued_ph = (issued_ph & ~(1u << stage)) | (ph << stage);
                if (++stage == kStages2) { stage = 0; ph ^= 1u; }
            }
            if (aborted) break;
        }
        if (lane == 0) {
            prof_add(p, 1, w_empty);
            prof_add(p, 8, 1);
        }
        if (q == 0) {
            for (int s = 0; s < kStages2; ++s)
                if (issued & (1u << s)) drain_bar(&full[s], (issued_ph >> s) & 1u, p);
        } else if (aborted) {
            // this CTA's copies land on the leader's barriers: give them time to land
            const uint64_t t0 = ptx::globaltimer();
            while (ptx::globaltimer() - t0 < 50000) {}
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader only)
        // The whole warp runs the loop, so the descriptors are warp-uniform values;
        // one elected lane issues every MMA and every commit (a commit tracks the
        // MMAs of the thread that issues it).  Issuing from a diverged single lane
        // measured ~70 cycles per MMA against ~45 here, and commit arrivals queue
        // behind MMA issue, so the cheaper issue is what keeps the tensor pipe fed.
        if (q == 0) {
            const bool issuer = ptx::elect_one();  // the same lane issues every MMA and commit
            int stage = 0;
            uint32_t ph = 0;
            int it = 0;
            uint64_t w_full = 0, w_tempty = 0;
            const uint64_t c_start = clock64();
            // descriptor of stage 0; stage s adds s * stage bytes / 16 to the start-address field
            const uint64_t adesc0 = sdesc(ptx::smem_u32(sA), 16, 1024);
            const uint64_t bdesc0 = sdesc(ptx::smem_u32(sB), 8192, 1024);
            for (int i = 0;; ++i) {
                if (i * G2 >= p.num_pair_units) break;
                const int u = i * G2 + (cl + i) % G2;
                if (u >= p.num_pair_units) continue;
                if (decode_pair(p, MODE, u, 0).pad) continue;
                const int buf = it % kAccBufs2;
                const uint32_t tph = (uint32_t)(it / kAccBufs2) & 1u;
                const bool tok = wait_bar_prof(&tempty[buf], tph ^ 1u, abort_flag, p, 11, u, w_tempty);
                if (!__all_sync(0xFFFFFFFFu, tok)) break;
                ptx::tc_fence_after();
                const uint32_t d = tmem_base + buf * kBN;
                bool ok = true;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    const bool fok = wait_bar_prof(&full[stage], ph, abort_flag, p, 12, u, w_full);
                    if (!__all_sync(0xFFFFFFFFu, fok)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint64_t ad = adesc0 + (uint64_t)(stage * (kAHalfBytes >> 4));
                    const uint64_t bd = bdesc0 + (uint64_t)(stage * (kBHalfBytes >> 4));
                    if (issuer) {
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)  // K16 steps: +32 bytes in A's rows, +16 rows of B
                            ptx::umma_bf16_pair(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 128), kIdesc2,
                                                (kb | kk) != 0);
                        ptx::umma_commit_pair_multicast(&empty[stage], 0x3);
                        if (kb == p.num_kb - 1) ptx::umma_commit_pair_multicast(&tfull[buf], 0x3);
                    }
                    __syncwarp();
                    if (++stage == kStages2) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                ++it;
            }
            if (issuer) ptx::umma_commit_pair(mma_done);
            __syncwarp();
            drain_bar(mma_done, 0, p);
            if (lane == 0 && (p.flags & ARE_DEBUG_WAIT_PROFILE)) *t_mma_end = ptx::globaltimer();
            if (lane == 0) {
                prof_add(p, 2, w_full);
                prof_add(p, 3, w_tempty);
                prof_add(p, 4, (uint64_t)(clock64() - c_start));
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ partial loader (own tile)
        if (lane == 0) {
            int ps = 0;
            uint32_t pph = 0;
            uint32_t issued = 0, issued_ph = 0;
            const uint32_t full_mask = (p.R >= 32) ? 0xFFFFFFFFu : ((1u << p.R) - 1u);
            uint64_t w_mask = 0;
            for (int i = 0;; ++i) {
                if (i * G2 >= p.num_pair_units) break;
                const int u = i * G2 + (cl + i) % G2;
                if (u >= p.num_pair_units) continue;
                const PUnit U = decode_pair(p, MODE, u, (int)q);
                if (ring) {
                    // push ring: rank r > 0 streams S_(r-1), the running sum rank r-1 published
                    if (!U.valid || U.r == 0) continue;
                    const uint32_t bit = 1u << (U.r - 1);
                    bool ok = true;
                    uint32_t seen = ptx::ld_acquire_gpu(&p.mask[U.t]);
                    if (!(seen & bit)) {
                        const uint64_t c0 = clock64();
                        const uint64_t t0 = ptx::globaltimer();
                        while (true) {
                            ptx::nanosleep(100);
                            seen = ptx::ld_acquire_gpu(&p.mask[U.t]);
                            if (seen & bit) break;
                            if (*abort_flag || ptx::ld_relaxed_gpu(&p.status->code) != 0u) {
                                *abort_flag = 1u;
                                ok = false;
                                break;
                            }
                            if (ptx::globaltimer() - t0 > p.timeout_ns) {
                                record_error(p.status, ARE_DEV_MASK_TIMEOUT, blockIdx.x, U.t, (int32_t)seen);
                                *abort_flag = 1u;
                                ok = false;
                                break;
                            }
                        }
                        w_mask += (uint64_t)(clock64() - c0);
                    }
                    if (!ok) break;
                    ptx::fence_proxy_async_global();
                    const uint8_t* src = pair_slot(p, U, U.r - 1);
                    // S_(r-1) is read once: evict-first leaves L2 to the operand panels (large
                    // GEMM+RS 2373-2377 -> 2364-2368 us, DRAM traffic 6767 -> 6658 MB per launch)
                    const uint64_t pol_s = ptx::policy_evict_first();
                    for (int st = 0; st < 2 * nsub && ok; ++st) {
                        if (!wait_bar(&pempty[ps], pph ^ 1u, abort_flag, p, 13, u)) { ok = false; break; }
                        ptx::mbar_arrive_expect_tx(&pfull[ps], kPSub2);
                        ptx::bulk_load_hint(sP + ps * kPSub2, src + (size_t)st * kPSub2, kPSub2, &pfull[ps], pol_s);
                        issued |= 1u << ps;
                        issued_ph = (issued_ph & ~(1u << ps)) | (pph << ps);
                        if (++ps == kPStages2) { ps = 0; pph ^= 1u; }
                    }
                    if (!ok) break;
                    continue;
                }
                // two-shot: every unit loads its row slice of the pair's R partials
                if (!U.valid) continue;
                bool ok = true;
                uint32_t seen = ptx::ld_acquire_gpu(&p.mask[U.t]);
                if (seen != full_mask) {
                    const uint64_t c0 = clock64();
                    const uint64_t t0 = ptx::globaltimer();
                    while (true) {
                        ptx::nanosleep(100);
                        seen = ptx::ld_acquire_gpu(&p.mask[U.t]);
                        if (seen == full_mask) break;
                        if (*abort_flag || ptx::ld_relaxed_gpu(&p.status->code) != 0u) {
                            *abort_flag = 1u;
                            ok = false;
                            break;
                        }
                        if (ptx::globaltimer() - t0 > p.timeout_ns) {
                            record_error(p.status, ARE_DEV_MASK_TIMEOUT, blockIdx.x, U.t, (int32_t)seen);
                            *abort_flag = 1u;
                            ok = false;
                            break;
                        }
                    }
                    w_mask += (uint64_t)(clock64() - c0);
                }
                if (!ok) break;
                // generic-proxy acquire above, async-proxy (bulk copy) reads below
                ptx::fence_proxy_async_global();
                // row slice U.j: groups of up to 16 rows; a stage holds one rank's group of 8
                // sub-tiles, 1 KB per 64-byte column sub-tile (sub-tile hf * 8 + st at st * 1 KB of
                // the group's stage hf), fetched by one 5-D tile load (rows past the tile's 128 read
                // as zeros, rows past the slice are not used); each slice of a partial is read once,
                // so evict-first
                const int lo = U.j * kBM / p.R, hi = (U.j + 1) * kBM / p.R;
                const uint64_t pol_p = ptx::policy_evict_first();
                for (int g0 = lo; g0 < hi && ok; g0 += 16) {
                    for (int hf = 0; hf < kHalves && ok; ++hf) {
                        for (int r = 0; r < p.R; ++r) {
                            if (own_slice && r == U.j) continue;  // on chip (sOwn)
                            if (!wait_bar(&pempty[ps], pph ^ 1u, abort_flag, p, 13, u)) { ok = false; break; }
                            ptx::mbar_arrive_expect_tx(&pfull[ps], kPSub2);
                            ptx::tma_load_5d(sP + ps * kPSub2, &p.tmPart, &pfull[ps], 0, g0, hf * 8, U.t, r, pol_p);
                            issued |= 1u << ps;
                            issued_ph = (issued_ph & ~(1u << ps)) | (pph << ps);
                            if (++ps == kPStages2) { ps = 0; pph ^= 1u; }
                        }
                    }
                }
                if (!ok) break;
            }
            prof_add(p, 6, w_mask);
            for (int s = 0; s < kPStages2; ++s)
                if (issued & (1u << s)) drain_bar(&pfull[s], (issued_ph >> s) & 1u, p);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ drain: TMEM -> partial slot -> publish
        const int row = threadIdx.x - 128;
        const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
        const bool lead = (warp == 4) && (lane == 0);
        const uint32_t tempty_leader = ptx::mapa_shared(ptx::smem_u32(&tempty[0]), 0);
        int it = 0;
        int nvalid = 0;         // valid units drained: own-slice buffer nvalid & 1
        int dps = 0;            // push ring: partial-buffer stage this drain reads next, and its parity
        uint32_t dpph = 0;
        int prev_tm = -1;       // chunk counting: the last tile whose owner stores may still be in flight
        bool bad = false;
        uint64_t w_tfull = 0;
        for (int i = 0;; ++i) {
            if (i * G2 >= p.num_pair_units) break;
            const int u = i * G2 + (cl + i) % G2;
            if (u >= p.num_pair_units) continue;
            const PUnit U = decode_pair(p, MODE, u, (int)q);
            if (U.pad) continue;
            const int buf = it % kAccBufs2;
            const uint32_t tph = (uint32_t)(it / kAccBufs2) & 1u;
            if (!wait_bar_prof(&tfull[buf], tph, abort_flag, p, 14, u, w_tfull, 200)) bad = true;
            if (grp_bar_or<1>(bad)) { bad = true; break; }
            ptx::tc_fence_after();
            const uint32_t tacc = tmem_base + lane_base + buf * kBN;
            uint8_t* gdst = pair_slot(p, U, U.r);
            if (U.valid) {
                const int olo = U.j * 16, ohi = olo + 16;  // own slice rows (own_slice only)
                const int oslot = nvalid & 1;
                uint8_t* const own_buf = oslot ? sOwn1 : sOwn0;
                if (own_slice && nvalid >= 2) {
                    // the buffer's previous slice (two valid units ago) must have been read
                    const bool ok = wait_bar(&ownfree[oslot], (uint32_t)((nvalid >> 1) - 1) & 1u, abort_flag, p, 16, u, 200);
                    if (grp_bar_or<1>(!ok)) { bad = true; break; }
                }
                // push ring (GEMM+RS): rank r > 0 adds S_(r-1), streamed into the partial buffer by
                // the loader in sub-tile order, to its accumulator: S_r = S_(r-1) + P_r; the last
                // rank writes bf16(S_(R-1)) to the owners instead of a partial
                const bool ring_add = ring && U.r > 0;
                const bool ring_last = ring && U.r == p.R - 1;
                const int row0 = U.tm * kBM;
                uint32_t outw[32];
                for (int j = 0; j < nsub; ++j) {
                    uint32_t w[32];
                    __syncwarp();
                    if (MODE == kModeRS) {
                        ptx::tmem_ld32(tacc + j * 32, w);
                    } else {
                        uint32_t v0[32], v1[32];
                        ptx::tmem_ld32(tacc + j * 64, v0);
                        ptx::tmem_ld32(tacc + j * 64 + 32, v1);
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            w[c] = pack_bf16x2(__uint_as_float(v0[2 * c]), __uint_as_float(v0[2 * c + 1]));
                            w[16 + c] = pack_bf16x2(__uint_as_float(v1[2 * c]), __uint_as_float(v1[2 * c + 1]));
                        }
                    }
                    if (j == nsub - 1) {
                        // the accumulator is read: hand it back (one arrival per CTA on the leader's barrier)
                        ptx::tc_fence_before();
                        grp_bar<1>();
                        if (lead) ptx::mbar_arrive_cluster(tempty_leader + (uint32_t)(buf * 8));
                    }
                    if (MODE == kModeRS && ring_add) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {  // sub-tile 2j + h: columns 16h..16h+15 of w
                            uint32_t v[16];
                            if (!wait_bar(&pfull[dps], dpph, abort_flag, p, 17, u, 200)) bad = true;
                            read_row_sw64(sP + dps * kPSub2, row, v);
                            ptx::mbar_arrive(&pempty[dps]);
                            if (++dps == kPStages2) { dps = 0; dpph ^= 1u; }
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                w[16 * h + e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(w[16 * h + e]));
                        }
                    }
                    if (MODE == kModeRS && ring_last) {
                        // bf16 of 32 columns: half of the 64-column output chunk j / 2
                        if (!(j & 1)) {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                outw[e] = pack_bf16x2(__uint_as_float(w[2 * e]), __uint_as_float(w[2 * e + 1]));
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                outw[16 + e] = pack_bf16x2(__uint_as_float(w[2 * e]), __uint_as_float(w[2 * e + 1]));
                            // one staging buffer: lane 0 of warp 4 issues the chunk's stores and waits for
                            // their reads before the next chunk is staged
                            if (warp == 4 && lane == 0) ptx::bulk_wait_read0();
                            if (grp_bar_or<1>(bad)) { bad = true; break; }
                            write_row_sw128(sOut, row, outw);
                            ptx::fence_proxy_async_shared();
                            grp_bar<1>();
                            if (warp == 4 && lane == 0) {
                                const int x = U.tn * kBN + (j >> 1) * 64;
                                if (x < p.N) {
                                    // owner-boundary flush: one store per (segment piece, H-row box)
                                    const int row_end = min(row0 + kBM, p.M);
                                    for (int r0 = row0; r0 < row_end;) {
                                        const int s = r0 / p.S;
                                        const int e = min((s + 1) * p.S, row_end);
                                        for (int rb = r0; rb < e; rb += p.H)
                                            ptx::tma_store_2d(&p.tmOut[s], sOut + (rb - row0) * 128, x, rb - s * p.S);
                                        r0 = e;
                                    }
                                    ptx::bulk_commit();
                                }
                            }
                        }
                        continue;
                    }
                    // the 128-byte row chunk becomes partial sub-tiles 2j and 2j+1: swizzled smem
                    // staging -> one 8 KB bulk store each; staging buffer b belongs to lane b,
                    // which waits only for its own bulk group before refilling it.  GEMM+RS with the
                    // row-slice split alternates two pairs of buffers (the own-slice buffers are GEMM+AR's
                    // and the slice reduce stages only sOut's first half), so the stores of chunk j - 1
                    // still read their staging while chunk j is staged (R=4, N=4096, K=2048: M=256
                    // 33.5-34.2 -> 33.0-33.1 us, M=512 45.8-46.5 -> 45.0-45.7 us; R=8 unchanged)
                    if (own_slice && row >= olo && row < ohi) {
                        // the own slice's rows of sub-tiles 2j, 2j+1, laid out as a loaded stage
                        write_half_sw64<0>(own_buf + (2 * j) * 1024 - olo * 64, row, w);
                        write_half_sw64<1>(own_buf + (2 * j + 1) * 1024 - olo * 64, row, w);
                    }
                    const bool alt = (MODE == kModeRS) && split && (j & 1);
                    uint8_t* const stg0 = alt ? sOwn0 : sDrain;
                    uint8_t* const stg1 = alt ? sOwn1 : sDrain + kPSub2;
                    if (warp == 4 && lane < 2) {
                        if ((MODE == kModeRS) && split) ptx::bulk_wait_read1();
                        else ptx::bulk_wait_read0();
                    }
                    grp_bar<1>();
                    write_half_sw64<0>(stg0, row, w);
                    write_half_sw64<1>(stg1, row, w);
                    ptx::fence_proxy_async_shared();
                    grp_bar<1>();
                    if (warp == 4 && lane < 2) {
                        uint8_t* dst = gdst + (size_t)(2 * j + lane) * kPSub2;
                        const uint8_t* src = lane ? stg1 : stg0;
                        if (own_slice) {  // every row but the own slice's
                            if (olo > 0) ptx::bulk_store(dst, src, (uint32_t)(olo * 64));
                            if (ohi < kBM) ptx::bulk_store(dst + ohi * 64, src + ohi * 64, (uint32_t)((kBM - ohi) * 64));
                        } else {
                            ptx::bulk_store(dst, src, kPSub2);
                        }
                        ptx::bulk_commit();
                    }
                }
                ++nvalid;
                if (ring && grp_bar_or<1>(bad)) { bad = true; break; }
                if (MODE == kModeRS && ring_last) {
                    // the tile is complete: every earlier rank's bit was read by this unit's loader
                    // before it streamed S_(R-2), so the word can be re-armed now
                    if (warp == 4 && lane == 0) {
                        if (p.flags & ARE_DEBUG_LOG_PIECES) {
                            int32_t* log = p.pieces + (size_t)U.t * kPieceWords;
                            const int row_end = min(row0 + kBM, p.M);
                            int n = 0;
                            for (int r0 = row0; r0 < row_end && n < (kPieceWords - 3) / 3;) {
                                const int s = r0 / p.S;
                                const int e = min((s + 1) * p.S, row_end);
                                log[3 + 3 * n] = s; log[4 + 3 * n] = r0; log[5 + 3 * n] = e;
                                ++n;
                                r0 = e;
                            }
                            log[0] = U.tm; log[1] = U.tn; log[2] = n;
                        }
                        if (p.flags & ARE_DEBUG_NO_REARM) ptx::red_release_or(&p.mask[U.t], 1u << U.r);
                        else atomicExch(&p.mask[U.t], 0u);
                        if (p.chunk_ctr) {
                            // count the previous tile's pieces once its stores have completed: at most
                            // this tile's store groups (one per 64-column chunk) may still be pending
                            if (prev_tm >= 0) {
                                const int rem_cols = p.N - U.tn * kBN;
                                ptx::bulk_wait_upto(min(kBN / 64, (rem_cols + 63) / 64));
                                ptx::fence_proxy_async_global();
                                chunk_bump_tile(p, prev_tm);
                            }
                            prev_tm = U.tm;
                        }
                    }
                } else if (warp == 4) {
                    // publish once this tile's partial is in memory: only the two issuing lanes wait
                    if (lane < 2) {
                        ptx::bulk_wait0();
                        ptx::fence_proxy_async_global();
                        __threadfence();
                    }
                    __syncwarp();
                    if (lane == 0 && !((p.flags & ARE_DEBUG_SKIP_PUBLISH) && (int64_t)u == p.debug_arg))
                        ptx::red_release_or(&p.mask[U.t], 1u << U.r);
                }
            } else {
                // no such tile (odd number of tile rows): hand the accumulator back
                ptx::tc_fence_before();
                grp_bar<1>();
                if (lead) ptx::mbar_arrive_cluster(tempty_leader + (uint32_t)(buf * 8));
            }
            ++it;
        }
        if (bad) *abort_flag = 1u;
        if (lead) prof_add(p, 5, w_tfull);
        if (warp == 4 && lane < 2) ptx::bulk_wait0();
        if (MODE == kModeRS && p.chunk_ctr && warp == 4 && lane == 0 && prev_tm >= 0 && !bad) {
            ptx::fence_proxy_async_global();
            chunk_bump_tile(p, prev_tm);
        }
    } else if (warp >= 8 && split) {
        // ------------------------------------------------------------ reduce (two-shot row slices)
        const int row = threadIdx.x - 256;
        const bool lead = (warp == 8);
        int nvalid = 0;    // GEMM+AR: valid units reduced (own-slice buffer nvalid & 1, as in the drain)
        int ps = 0;
        uint32_t pph = 0;
        bool bad = false;
        uint64_t w_pfull = 0;
        for (int i = 0;; ++i) {
            if (i * G2 >= p.num_pair_units) break;
            const int u = i * G2 + (cl + i) % G2;
            if (u >= p.num_pair_units) continue;
            const PUnit U = decode_pair(p, MODE, u, (int)q);
            if (!U.pad && U.valid) {
                // ---- this unit reduces row slice U.j of its tile (two-shot: rank j sums slice j of
                // all R partials in the order r = 0..R-1, then writes it to every view, GEMM+AR, or
                // to its owner segments, GEMM+RS), so every unit of a pair takes 1/R of the tile's
                // reduction
                const int lo = U.j * kBM / p.R, hi = (U.j + 1) * kBM / p.R;
                const int st = row >> 4, rr = row & 15;  // 64-byte column sub-tile, row in the group
                const int wq = warp - 8;
                const int oslot = nvalid & 1;
                const uint8_t* const own_buf = oslot ? sOwn1 : sOwn0;
                for (int g0 = lo; g0 < hi; g0 += 16) {
                    const int nr = min(16, hi - g0);
                    const int trow = g0 + rr;  // tile row of this thread
                    // GEMM+AR: 32 bf16 columns of sub-tile st; GEMM+RS: 16 fp32 columns of sub-tiles
                    // st (acc[0..15]) and 8 + st (acc[16..31])
                    float acc[32];
                    for (int hf = 0; hf < kHalves; ++hf) {
                        for (int qq = 0; qq < p.R; ++qq) {
                            const bool mine = own_slice && qq == U.j;
                            // The own slice was written by this CTA's drain before it published the unit's
                            // mask bit; the loader acquired the full mask before filling this unit's stages,
                            // so a wait on one of them orders those writes first.  For rank 0 that is the
                            // wait on the next stage (rank 1's, not consumed here); for a later rank the
                            // waits on the stages before it already did.
                            if (!mine || qq == 0)
                                if (!wait_bar_prof(&pfull[ps], pph, abort_flag, p, 15, u, w_pfull, 200)) bad = true;
                            uint32_t v[16];
                            if (rr < nr) {
                                const uint8_t* rp = (mine ? own_buf : sP + ps * kPSub2) + st * 1024 + rr * 64;
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    const uint4 x = *reinterpret_cast<const uint4*>(rp + ((c ^ ((trow >> 1) & 3)) << 4));
                                    v[4 * c] = x.x; v[4 * c + 1] = x.y; v[4 * c + 2] = x.z; v[4 * c + 3] = x.w;
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 16; ++e) v[e] = 0u;
                            }
                            if (!mine) {
                                ptx::mbar_arrive(&pempty[ps]);
                                if (++ps == kPStages2) { ps = 0; pph ^= 1u; }
                            }
                            if (MODE == kModeRS) {
                                float* a = acc + 16 * hf;
                                if (qq == 0) {
#pragma unroll
                                    for (int e = 0; e < 16; ++e) a[e] = __uint_as_float(v[e]);
                                } else {
#pragma unroll
                                    for (int e = 0; e < 16; ++e) a[e] = a[e] + __uint_as_float(v[e]);
                                }
                            } else if (qq == 0) {
#pragma unroll
                                for (int e = 0; e < 16; ++e) {
                                    acc[2 * e] = __uint_as_float(v[e] << 16);
                                    acc[2 * e + 1] = __uint_as_float(v[e] & 0xFFFF0000u);
                                }
                            } else {
#pragma unroll
                                for (int e = 0; e < 16; ++e) {
                                    acc[2 * e] = acc[2 * e] + __uint_as_float(v[e] << 16);
                                    acc[2 * e + 1] = acc[2 * e + 1] + __uint_as_float(v[e] & 0xFFFF0000u);
                                }
                            }
                        }
                    }
                    // The group's 16 rows x 256 bf16 columns (512 bytes a row) leave in 16-byte chunks:
                    // this thread holds four, acc[8n..8n+7] for n = 0..3, at chunk k(n) of its row.
                    // A full group (16 rows, aligned to an owner segment for GEMM+RS) is staged as four
                    // 128B-swizzled boxes of 64 columns (16 rows x 128 bytes each) and written by TMA
                    // tensor stores, one box per view (GEMM+AR) or into the rows' owner segment (GEMM+RS)
                    // and 64 columns.  Any other group is staged as 16 x 512-byte rows (16-byte chunk k of
                    // row rr at position k ^ rr) and written with whole-row 16-byte stores, so no box
                    // covers rows of another unit's slice or another segment.  The issuing thread waits
                    // until the previous group's stores have read the staging buffer; the barrier then
                    // orders the rewrite.
                    const int y = U.tm * kBM + g0;
                    const bool tma_out = (nr == 16) && (MODE == kModeAR || (p.H == 16 && (g0 & 15) == 0));
                    if (lead && lane == 0) ptx::bulk_wait_read0();
                    if (grp_bar_or<2>(bad)) { bad = true; break; }
                    // every read of the own slice is done: hand its buffer back to the drain
                    if (own_slice && lead && lane == 0) ptx::mbar_arrive(&ownfree[oslot]);
#pragma unroll
                    for (int n = 0; n < 4; ++n) {
                        const int k = (MODE == kModeRS) ? ((n >> 1) * 16 + st * 2 + (n & 1)) : (st * 4 + n);
                        uint8_t* dst = tma_out ? sOut + (k >> 3) * 2048 + rr * 128 + (((k & 7) ^ (rr & 7)) << 4)
                                               : sOut + rr * 512 + ((k ^ rr) << 4);
                        *reinterpret_cast<uint4*>(dst) =
                            make_uint4(pack_bf16x2(acc[8 * n], acc[8 * n + 1]), pack_bf16x2(acc[8 * n + 2], acc[8 * n + 3]),
                                       pack_bf16x2(acc[8 * n + 4], acc[8 * n + 5]),
                                       pack_bf16x2(acc[8 * n + 6], acc[8 * n + 7]));
                    }
                    if (tma_out) {
                        ptx::fence_proxy_async_shared();
                        grp_bar<2>();
                        if (lead && lane == 0) {
                            // the outputs are read by nothing in this kernel: evict-first keeps the
                            // operand panels and partials in L2 (648 -> 645 us alone at R=8,
                            // M=4096, N=7168, K=2048)
                            const uint64_t pol_v = ptx::policy_evict_first();
                            if (MODE == kModeRS) {
                                const int sg = y / p.S;  // the group lies inside one owner segment
                                if (y < p.M) {
#pragma unroll
                                    for (int b = 0; b < 4; ++b)  // boxes past N would store nothing
                                        if (U.tn * kBN + b * 64 < p.N)
                                            ptx::tma_store_2d_hint(&p.tmOut[sg], sOut + b * 2048, U.tn * kBN + b * 64,
                                                                   y - sg * p.S, pol_v);
                                }
                            } else {
                                for (int w = 0; w < p.nviews; ++w)
#pragma unroll
                                    for (int b = 0; b < 4; ++b)  // boxes past N or M would store nothing
                                        if (U.tn * kBN + b * 64 < p.N && y < p.M)
                                            ptx::tma_store_2d_hint(&p.tmOut[w], sOut + b * 2048, U.tn * kBN + b * 64, y,
                                                                   pol_v);
                            }
                            ptx::bulk_commit();
                        }
                        continue;
                    }
                    grp_bar<2>();
                    const int gcol = U.tn * kBN + lane * 8;
#pragma unroll
                    for (int i2 = 0; i2 < 4; ++i2) {
                        const int orr = wq + 4 * i2;
                        const int grow = y + orr;
                        if (orr < nr && grow < p.M && gcol < p.N) {
                            const uint4 val = *reinterpret_cast<const uint4*>(sOut + orr * 512 + ((lane ^ orr) << 4));
                            if (MODE == kModeRS) {
                                const int sg = grow / p.S;
                                ptx::st_stream_v4(p.views[sg] + (size_t)(grow - sg * p.S) * p.N + gcol, val);
                            } else {
                                for (int w = 0; w < p.nviews; ++w)
                                    ptx::st_stream_v4(p.views[w] + (size_t)grow * p.N + gcol, val);
                            }
                        }
                    }
                }
                if (bad) break;
                if (lead && lane == 0) {
                    // the last of the tile's R slice reducers re-arms its mask word (and this count)
                    const uint32_t old = atomicAdd(&p.cons[U.t], 1u);
                    if (old == (uint32_t)p.R - 1u) {
                        atomicExch(&p.cons[U.t], 0u);
                        if (MODE == kModeRS && (p.flags & ARE_DEBUG_LOG_PIECES)) {
                            // the tile's owner pieces (its R slices were stored by its R units)
                            int32_t* log = p.pieces + (size_t)U.t * kPieceWords;
                            const int row0 = U.tm * kBM;
                            const int row_end = min(row0 + kBM, p.M);
                            int n = 0;
                            for (int r0 = row0; r0 < row_end && n < (kPieceWords - 3) / 3;) {
                                const int sg = r0 / p.S;
                                const int e = min((sg + 1) * p.S, row_end);
                                log[3 + 3 * n] = sg; log[4 + 3 * n] = r0; log[5 + 3 * n] = e;
                                ++n;
                                r0 = e;
                            }
                            log[0] = U.tm; log[1] = U.tn; log[2] = n;
                        }
                        if (!(p.flags & ARE_DEBUG_NO_REARM)) atomicExch(&p.mask[U.t], 0u);
                    }
                }
                ++nvalid;
            }
        }
        if (bad) *abort_flag = 1u;
        if (lead && lane == 0) prof_add(p, 7, w_pfull);
        if (lead && lane == 0) ptx::bulk_wait0();
    }

    __syncwarp();
    ptx::tc_fence_before();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    if (threadIdx.x == 0 && q == 0 && (p.flags & ARE_DEBUG_WAIT_PROFILE)) {
        // the pair's time after its last MMA completed (drains and reductions still
        // running), and its whole span, in ns
        const uint64_t t_end = ptx::globaltimer();
        const uint64_t tail = t_end - *t_mma_end;
        atomicMax(&p.counters[9], (unsigned long long)tail);
        atomicAdd(&p.counters[10], (unsigned long long)tail);
        atomicMax(&p.counters[11], (unsigned long long)(t_end - t_begin));
        atomicAdd(&p.counters[12], (unsigned long long)(*t_mma_end - t_begin));
    }
    if (warp == 2) {
        __syncwarp();
        ptx::tmem_dealloc_pair(tmem_base, kTmemCols2);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;

cudaError_t get_encode() {
    std::lock_guard<std::mutex> lk(g_encode_mu);
    if (g_encode) return cudaSuccess;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

}  // namespace

size_t gemm_smem_bytes() { return kSmemBytes; }

// Co-resident clusters of the pair kernel, per device (-1 = not yet queried).
constexpr int kMaxDevices = 64;
std::mutex g_pair_mu;
int g_pair_clusters[kMaxDevices];
bool g_pair_init = false;

cudaLaunchConfig_t pair_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kPairThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes2;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

cudaError_t gemm_prepare_kernels() {
    cudaError_t e = cudaFuncSetAttribute(gemm_reduce_kernel<kModeRS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_reduce_kernel<kModeAR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_pair_kernel<kModeRS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes2);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_pair_kernel<kModeAR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes2);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lk(g_pair_mu);
        if (!g_pair_init) {
            for (int d = 0; d < kMaxDevices; ++d) g_pair_clusters[d] = -1;
            g_pair_init = true;
        }
        if (g_pair_clusters[dev] < 0) {
            // co-resident clusters bound the persistent grid (every cluster must be running)
            int n_rs = 0, n_ar = 0;
            cudaLaunchAttribute attr[1];
            cudaLaunchConfig_t cfg = pair_config(2 * 1024, nullptr, attr);
            if (cudaOccupancyMaxActiveClusters(&n_rs, (void*)gemm_pair_kernel<kModeRS>, &cfg) != cudaSuccess) n_rs = 0;
            if (cudaOccupancyMaxActiveClusters(&n_ar, (void*)gemm_pair_kernel<kModeAR>, &cfg) != cudaSuccess) n_ar = 0;
            cudaGetLastError();
            g_pair_clusters[dev] = n_rs < n_ar ? n_rs : n_ar;
        }
    }
    return get_encode();
}

int gemm_pair_max_clusters() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_pair_mu);
    return (g_pair_init && g_pair_clusters[dev] > 0) ? g_pair_clusters[dev] : 0;
}

int gemm_pair_threads() { return kPairThreads; }

// bf16 [outer, inner] row-major, 128B-swizzled boxes of box_inner x box_outer.
cudaError_t make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                           uint32_t box_outer) {
    cudaError_t e = get_encode();
    if (e != cudaSuccess) return e;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_part(CUtensorMap* m, const void* part, uint64_t T, uint64_t R) {
    cudaError_t e = get_encode();
    if (e != cudaSuccess) return e;
    // 4-byte words: 16 per 64-byte sub-tile row, 128 rows, 16 sub-tiles per 128 KB slot
    cuuint64_t dims[5] = {16, 128, 16, T, R};
    cuuint64_t strides[4] = {64, (cuuint64_t)kPSub2, (cuuint64_t)kTilePartBytes, (cuuint64_t)T * kTilePartBytes};
    cuuint32_t box[5] = {16, 16, 8, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 5, const_cast<void*>(part), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_gemm_pair(const GemmParams& p, int mode, int grid, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pair_config(grid, stream, attr);
    cudaError_t e = (mode == kModeRS) ? cudaLaunchKernelEx(&cfg, gemm_pair_kernel<kModeRS>, p)
                                      : cudaLaunchKernelEx(&cfg, gemm_pair_kernel<kModeAR>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_gemm_reduce(const GemmParams& p, int mode, int grid, cudaStream_t stream) {
    if (mode == kModeRS)
        gemm_reduce_kernel<kModeRS><<<grid, kGemmThreads, kSmemBytes, stream>>>(p);
    else
        gemm_reduce_kernel<kModeAR><<<grid, kGemmThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace are
