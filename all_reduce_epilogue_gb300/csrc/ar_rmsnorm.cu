// All-reduce + residual + RMSNorm in one kernel, with Lamport (-0.0 sentinel)
// readiness between its two phases.
//
// Method: ROCm/aiter PR #4977 "Single-kernel Lamport fused all-reduce +
// RMSNorm", sections "Approach" and "Correctness notes":
//   * the staging buffer holds the sentinel -0.0 (0x80000000 per fp32 word)
//     in every word between calls;
//   * a producer canonicalises -0.0 to +0.0 before it stores, so a written
//     word can never look like the sentinel, and needs no publish fence;
//   * a consumer polls its pack and treats it as arrived only when no word of
//     it still equals the sentinel; it re-arms the pack right after reading
//     it (one consumer per pack, so the re-arm needs no extra sync);
//   * every block finishes the producer work it owes before it spins, and
//     the grid never exceeds the co-resident block count, so the spin cannot
//     wait on a block that is not running.
//
// One-GPU design.  The R "ranks" are R device buffers.  Rows are cut into
// chunks of `chunk_rows` (= grid) rows.  Each block stages a contiguous slice
// of every chunk's 8-element packs (phase A) and normalises one row of every
// chunk (phase B), a row that another block staged: row i of a chunk goes to
// block (i + grid/2) mod grid.
//
// One block per SM, warp-specialised (512 threads):
//   warp 0      producer: streams, with 1D bulk copies into shared memory,
//               the R partial slices of every phase-A sub-chunk (224 packs)
//               into a ring of `stages` buffers, and the residual row of
//               every phase-B row into a 3-slot ring;
//   warps 1-7   phase A: each thread sums one pack of the R ranks from shared
//               memory in ring order, canonicalises, and stores 8 fp32
//               staging words;
//   warps 8-15  phase B: bounded spin per 16-byte staging pack, re-arm,
//               residual add, sum of squares, reduction, scale, store.
// Phase A runs at most four chunks ahead of this block's phase B.  When the
// rows wrap, the staging words form a ring of 8 chunk slots (~35 MB at
// N = 7168) that stays in L2 and is overwritten lap after lap, so staged
// words are neither written back to nor read from DRAM; the bytes in flight
// come from the copy engine, not from registers.  The staging words
// are fp32: staging a bf16 sum would round before the residual add.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "are_internal.h"
#include "ptx.cuh"


namespace are {
namespace {

constexpr int kAThreads = 224;                // phase-A threads = packs per sub-chunk
constexpr int kBThreads = 256;                // phase-B threads
constexpr int kRankBytes = kAThreads * 16;    // one rank's slice of a sub-chunk
constexpr int kStageBytes = kMaxRanks * kRankBytes;  // 28 KB
constexpr int kResSlots = 3;
constexpr int kAhead = 4;                     // phase A may lead phase B by this many chunks
constexpr int kArStages = 4;                  // phase-A stages used (<= kMaxArStages)
static_assert(kArStages <= kMaxArStages, "stage barriers");
constexpr size_t kSmemLimit = 227 * 1024;
constexpr size_t kTailBytes = 1024;           // barriers, reduction scratch, flags

static_assert(kArThreads == 32 + kAThreads + kBThreads, "warp roles");

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

constexpr uint32_t kSentinelOdd = 0xFFFFFFFFu;  // odd laps of the staging ring
constexpr uint32_t kCanonicalNaN = 0x7FC00000u;

__device__ __forceinline__ bool has_word(const uint4& v, uint32_t s) {
    return (v.x == s) | (v.y == s) | (v.z == s) | (v.w == s);
}
__device__ __forceinline__ bool all_words(const uint4& v, uint32_t s) {
    return (v.x == s) & (v.y == s) & (v.z == s) & (v.w == s);
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Sum of the 8 warp partials that a 256-thread block wrote to red[0..7], in the
// exact order of one warp's xor-shuffle tree over them (lanes 8..31 holding
// +0.0, which adds exactly: the partials are sums of squares, never -0.0):
// offsets 16 and 8 add zeros, 4 pairs warp w with w+4, 2 pairs (w, w+4) with
// (w+2, w+6), and 1 joins the two halves.  Phase B computes it in every thread,
// after the barrier that made the partials visible, so it needs no second
// barrier; the one-shot kernel runs the shuffle tree in one warp and gets the
// same bits.
static_assert(kBThreads == 256, "the reduction tree below is for 8 warps");
__device__ __forceinline__ float sum8_tree(const float* r) {
    return ((r[0] + r[4]) + (r[2] + r[6])) + ((r[1] + r[5]) + (r[3] + r[7]));
}

__device__ __forceinline__ void b_bar() {
    __syncwarp();  // .aligned barrier: reconverge the warp first
    asm volatile("bar.sync 2, %0;" ::"n"(kBThreads) : "memory");
}

struct Shared {
    uint8_t* stage;     // stages x 28 KB
    uint8_t* res;       // kResSlots x N*2 bytes (when the residual is staged in shared memory)
    float* gam;         // N fp32 (when gamma is staged in shared memory)
    uint64_t* full;     // [stages]
    uint64_t* empty;    // [stages]
    uint64_t* rfull;    // [kResSlots]
    uint64_t* rempty;   // [kResSlots]
    float* red;         // [32]: block sums in 0..8, block maxima in 16..24
    volatile int* bdone;        // chunks phase B has finished
    volatile uint32_t* abort;   // block gave up
};

__device__ __forceinline__ Shared carve(uint8_t* base, const ArParams& p) {
    Shared s;
    s.stage = base;
    s.res = base + (size_t)p.stages * kStageBytes;
    s.gam = reinterpret_cast<float*>(s.res + (p.res_in_smem ? (size_t)kResSlots * p.N * 2 : 0));
    uint8_t* tail = reinterpret_cast<uint8_t*>(s.gam) + (p.gamma_in_smem ? (size_t)p.N * 4 : 0);
    tail = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tail) + 15) & ~uintptr_t(15));
    s.full = reinterpret_cast<uint64_t*>(tail);
    s.empty = s.full + kMaxArStages;
    s.rfull = s.empty + kMaxArStages;
    s.rempty = s.rfull + kResSlots;
    s.red = reinterpret_cast<float*>(s.rempty + kResSlots);
    s.bdone = reinterpret_cast<volatile int*>(s.red + 32);
    s.abort = reinterpret_cast<volatile uint32_t*>(s.bdone + 1);
    return s;
}

// Bounded wait on a shared-memory barrier phase; false once the block gave up.
__device__ __forceinline__ bool ar_wait(uint64_t* bar, uint32_t parity, const Shared& sh, const ArParams& p) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*sh.abort) return false;
        if (ptx::globaltimer() - t0 > p.timeout_ns) {
            record_error(p.status, ARE_DEV_PIPE_TIMEOUT, blockIdx.x, -1, -1);
            *sh.abort = 1u;
            return false;
        }
    }
}

// Rows of chunk c, and this block's slice [q0, q1) of its packs (chunk-local
// pack indices; the chunk's first pack is `base`).
struct Slice {
    int64_t base, q0, q1;
    int rows;
};
// Without a ring the chunk's packs are split evenly over the blocks.  With a
// ring every block stages exactly row blockIdx.x of every chunk (chunk_rows ==
// grid), so each staging position has the same producer in every lap: its own
// earlier write of the position then orders its check of the next lap's
// sentinel, however far the blocks drift apart.
__device__ __forceinline__ Slice slice_of(const ArParams& p, int c) {
    const int64_t row0 = (int64_t)c * p.chunk_rows;
    Slice s;
    s.rows = (int)min((int64_t)p.chunk_rows, (int64_t)p.M - row0);
    s.base = row0 * p.packs_per_row;
    if (p.ring_slots) {
        const int64_t r = blockIdx.x < s.rows ? blockIdx.x : s.rows;
        s.q0 = r * p.packs_per_row;
        s.q1 = blockIdx.x < s.rows ? s.q0 + p.packs_per_row : s.q0;
        return s;
    }
    const int64_t total = (int64_t)s.rows * p.packs_per_row;
    const int64_t per = (total + gridDim.x - 1) / gridDim.x;
    s.q0 = min(total, (int64_t)blockIdx.x * per);
    s.q1 = min(total, s.q0 + per);
    return s;
}

// First staging word of row i of chunk c: the rows of chunk c live at
// c*chunk_rows, or in ring slot c mod ring_slots when the rows wrap.
__device__ __forceinline__ uint32_t* staging_row(const ArParams& p, int c, int64_t i) {
    const int64_t r0 = p.ring_slots ? (int64_t)(c % p.ring_slots) * p.chunk_rows : (int64_t)c * p.chunk_rows;
    return p.staging + (r0 + i) * (int64_t)p.N;
}

// Ring mode (rows wrap over `ring_slots` staging slots).  Lap L of slot s is
// chunk s + L*ring_slots.  Between laps the slot's words hold the sentinel of
// the next lap: -0.0 for even laps, 0xFFFFFFFF (a NaN pattern that staged data
// never has: NaNs are canonicalised like -0.0) for odd laps; the last lap of
// every slot re-arms with -0.0, so between calls every word is -0.0 again.
//  * A consumer position is served by the same thread in every lap, so its own
//    re-arm precedes (in program order) its next read of that position.
//  * A producer overwrites a pack only after reading the lap's sentinel in
//    all of its words: its write is then ordered after the consumer's re-arm.
//    Each position also has a fixed producer (see slice_of), which wrote the
//    position two laps earlier itself, so the sentinel it reads cannot be the
//    same-parity one from before that write.
// No counter, fence or barrier couples the blocks.
__device__ __forceinline__ int lap_of(const ArParams& p, int c) { return p.ring_slots ? c / p.ring_slots : 0; }
__device__ __forceinline__ uint32_t sentinel_of(int lap) { return (lap & 1) ? kSentinelOdd : kSentinelF32; }
// Value a consumer writes back into row i of chunk c: the next lap's sentinel
// if a later chunk of this call stages that row of the slot, else -0.0.
__device__ __forceinline__ uint32_t rearm_value(const ArParams& p, int c, int i) {
    if (!p.ring_slots || c + p.ring_slots >= p.num_chunks) return kSentinelF32;
    const int64_t next_rows = min((int64_t)p.chunk_rows, (int64_t)p.M - (int64_t)(c + p.ring_slots) * p.chunk_rows);
    if (i >= next_rows) return kSentinelF32;
    return sentinel_of(c / p.ring_slots + 1);
}

__device__ __forceinline__ int consumed_row(int G) {
    int i = (int)blockIdx.x - G / 2;
    return i < 0 ? i + G : i;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// The normalised row y = h * inv * gamma leaves either as bf16 (`out`) or, in
// the quantising variant, as FP8 E4M3 codes with one fp32 scale per row
// (dynamic per-token quantisation: scale = max|y| / 448, code = e4m3(y / scale),
// round to nearest even, saturating; both divisions correctly rounded).
// NT threads hold the row's packs bt, bt + NT, ...; bar() is their barrier and
// red[16..] their scratch.
// gamma of pack pk: from the block's shared-memory copy `gsm` when there is one, else
// from global memory through L1
__device__ __forceinline__ void gamma8(const ArParams& p, const float* gsm, int pk, float4& g0, float4& g1) {
    if (gsm) {
        g0 = reinterpret_cast<const float4*>(gsm)[pk * 2];
        g1 = reinterpret_cast<const float4*>(gsm)[pk * 2 + 1];
    } else {
        g0 = __ldg(reinterpret_cast<const float4*>(p.gamma) + pk * 2);
        g1 = __ldg(reinterpret_cast<const float4*>(p.gamma) + pk * 2 + 1);
    }
}

template <int PPT, int NT, typename Bar>
__device__ __forceinline__ void store_row(const ArParams& p, int64_t row, int bt, const float (&h)[PPT][8], float inv,
                                          float* red, const float* gsm, Bar bar) {
    const int P = p.packs_per_row;
    if (!p.out_q) {
#pragma unroll
        for (int k = 0; k < PPT; ++k) {
            const int pk = bt + k * NT;
            if (pk < P) {
                float4 g0, g1;
                gamma8(p, gsm, pk, g0, g1);
                uint4 o;
                o.x = pack_bf16x2(h[k][0] * inv * g0.x, h[k][1] * inv * g0.y);
                o.y = pack_bf16x2(h[k][2] * inv * g0.z, h[k][3] * inv * g0.w);
                o.z = pack_bf16x2(h[k][4] * inv * g1.x, h[k][5] * inv * g1.y);
                o.w = pack_bf16x2(h[k][6] * inv * g1.z, h[k][7] * inv * g1.w);
                ptx::st_stream_v4(p.out + row * (int64_t)p.N + pk * 8, o);
            }
        }
        return;
    }
    // y is recomputed in the second pass (same expression, same bits) rather than
    // held in registers across the block reduction
    float am = 0.f;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int pk = bt + k * NT;
        if (pk < P) {
            float4 g0, g1;
            gamma8(p, gsm, pk, g0, g1);
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(h[k][i] * inv * g[i]));
        }
    }
    const int w = bt >> 5, lane = bt & 31;
    am = warp_max(am);
    if (lane == 0) red[16 + w] = am;
    bar();
    if (w == 0) {
        float v = lane < NT / 32 ? red[16 + lane] : 0.f;
        v = warp_max(v);
        if (lane == 0) red[16 + NT / 32] = v;
    }
    bar();
    const float amax = red[16 + NT / 32];
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    if (bt == 0) p.out_scale[row] = sc;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int pk = bt + k * NT;
        if (pk < P) {
            float4 g0, g1;
            gamma8(p, gsm, pk, g0, g1);
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            uint32_t c[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                c[i] = (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(h[k][i] * inv * g[i], sc), __NV_SATFINITE, __NV_E4M3);
            const uint2 v = make_uint2(c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24),
                                       c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24));
            ptx::st_stream_v2(p.out_q + row * (int64_t)p.N + pk * 8, v);
        }
    }
}

// ARE_DEBUG_WAIT_PROFILE: one thread of each role adds the SM cycles it spent
// waiting to the debug counters.
__device__ __forceinline__ bool prof_on(const ArParams& p) { return (p.flags & ARE_DEBUG_WAIT_PROFILE) != 0; }
__device__ __forceinline__ void prof_add(const ArParams& p, int slot, uint64_t v) {
    if (prof_on(p) && v) atomicAdd(&p.counters[slot], (unsigned long long)v);
}

// ------------------------------------------------------------------ phase B
// `rbuf` (0 or 1, alternating row by row) selects the half of the reduction
// scratch this row's warp partials go to: a thread can start the next row's
// writes while others still read this row's partials, but not the row after.
template <int PPT>
__device__ __forceinline__ void norm_row(const ArParams& p, const Shared& sh, int64_t row, uint32_t* srow, int bt,
                                         const uint8_t* res_smem, uint64_t keep, uint32_t sent, uint32_t rearm,
                                         uint64_t& w_spin, int rbuf) {
    const int P = p.packs_per_row;
    uint4 lo[PPT], hi[PPT], res[PPT];
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int pk = bt + k * kBThreads;
        if (pk < P) {
            lo[k] = ptx::ld_relaxed_gpu_v4(srow + pk * 8);
            hi[k] = ptx::ld_relaxed_gpu_v4(srow + pk * 8 + 4);
            if (p.residual && !res_smem) res[k] = ptx::ld_stream_v4(p.residual + row * (int64_t)p.N + pk * 8);
        }
    }
    bool ok = true;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int pk = bt + k * kBThreads;
        if (pk < P && (has_word(lo[k], sent) || has_word(hi[k], sent))) {
            const uint64_t c0 = clock64();
            const uint64_t t0 = ptx::globaltimer();
            while (true) {
                lo[k] = ptx::ld_relaxed_gpu_v4(srow + pk * 8);
                hi[k] = ptx::ld_relaxed_gpu_v4(srow + pk * 8 + 4);
                if (!has_word(lo[k], sent) && !has_word(hi[k], sent)) break;
                if (ptx::ld_relaxed_gpu(&p.status->code) != 0u) { ok = false; break; }
                if (ptx::globaltimer() - t0 > p.timeout_ns) {
                    record_error(p.status, ARE_DEV_STAGE_TIMEOUT, blockIdx.x, (int32_t)row, pk);
                    ok = false;
                    break;
                }
            }
            w_spin += (uint64_t)(clock64() - c0);
        }
    }
    // Re-arm every pack this thread consumed (it is the pack's only consumer).
    if (ok && !(p.flags & ARE_DEBUG_NO_REARM)) {
        const uint4 s = make_uint4(rearm, rearm, rearm, rearm);
#pragma unroll
        for (int k = 0; k < PPT; ++k) {
            const int pk = bt + k * kBThreads;
            if (pk < P) {
                ptx::st_v4_hint(srow + pk * 8, s, keep);
                ptx::st_v4_hint(srow + pk * 8 + 4, s, keep);
            }
        }
    }
    if (p.residual && res_smem) {
#pragma unroll
        for (int k = 0; k < PPT; ++k) {
            const int pk = bt + k * kBThreads;
            if (pk < P) res[k] = *reinterpret_cast<const uint4*>(res_smem + pk * 16);
        }
    }
    // h = s + residual, kept in place in the staged registers
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int pk = bt + k * kBThreads;
        if (pk < P) {
            float f[8] = {__uint_as_float(lo[k].x), __uint_as_float(lo[k].y), __uint_as_float(lo[k].z),
                          __uint_as_float(lo[k].w), __uint_as_float(hi[k].x), __uint_as_float(hi[k].y),
                          __uint_as_float(hi[k].z), __uint_as_float(hi[k].w)};
            if (p.residual) {
                float r8[8];
                unpack8(res[k], r8);
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] = f[i] + r8[i];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
            if (p.residual_out) {  // the updated residual stream, bf16(h)
                const uint4 hv = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                                            pack_bf16x2(f[6], f[7]));
                ptx::st_stream_v4(p.residual_out + row * (int64_t)p.N + pk * 8, hv);
            }
            lo[k] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                               __float_as_uint(f[3]));
            hi[k] = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                               __float_as_uint(f[7]));
        }
    }
    const int w = bt >> 5, lane = bt & 31;
    ss = warp_sum(ss);
    float* part = sh.red + 8 * rbuf;
    if (lane == 0) part[w] = ss;
    b_bar();
    const float inv = rsqrtf(sum8_tree(part) * p.inv_n + p.eps);
    float hv[PPT][8];
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        hv[k][0] = __uint_as_float(lo[k].x); hv[k][1] = __uint_as_float(lo[k].y);
        hv[k][2] = __uint_as_float(lo[k].z); hv[k][3] = __uint_as_float(lo[k].w);
        hv[k][4] = __uint_as_float(hi[k].x); hv[k][5] = __uint_as_float(hi[k].y);
        hv[k][6] = __uint_as_float(hi[k].z); hv[k][7] = __uint_as_float(hi[k].w);
    }
    store_row<PPT, kBThreads>(p, row, bt, hv, inv, sh.red, p.gamma_in_smem ? sh.gam : nullptr, [] { b_bar(); });
}

template <int PPT>
__global__ void __launch_bounds__(kArThreads, 1) ar_rmsnorm_kernel(const __grid_constant__ ArParams p) {
    extern __shared__ __align__(128) uint8_t ar_smem[];
    const Shared sh = carve(ar_smem, p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const int consume = consumed_row(G);
    const bool res_smem = p.residual != nullptr && p.res_in_smem;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            ptx::mbar_init(&sh.full[s], 1);
            ptx::mbar_init(&sh.empty[s], kAThreads / 32);  // one arrival per phase-A warp
        }
        for (int s = 0; s < kResSlots; ++s) {
            ptx::mbar_init(&sh.rfull[s], 1);
            ptx::mbar_init(&sh.rempty[s], kBThreads / 32);  // one arrival per phase-B warp
        }
        *sh.bdone = 0;
        *sh.abort = 0u;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_shared();
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t stream_pol = ptx::policy_evict_first();
            int s = 0, rs = 0;
            uint32_t ph = 0, rph = 0;
            uint32_t issued = 0, issued_ph = 0, rissued = 0, rissued_ph = 0;
            bool ok = true;
            uint64_t w_empty = 0;
            for (int c = 0; c < p.num_chunks && ok; ++c) {
                const Slice sl = slice_of(p, c);
                if (res_smem && consume < sl.rows) {  // residual row of this block's phase-B row
                    const uint64_t c0 = clock64();
                    if (!ar_wait(&sh.rempty[rs], rph ^ 1u, sh, p)) break;
                    w_empty += (uint64_t)(clock64() - c0);
                    const uint32_t bytes = (uint32_t)p.N * 2;
                    ptx::mbar_arrive_expect_tx(&sh.rfull[rs], bytes);
                    const int64_t row = (int64_t)c * p.chunk_rows + consume;
                    ptx::bulk_load_hint(sh.res + (size_t)rs * p.N * 2, p.residual + row * (int64_t)p.N, bytes,
                                        &sh.rfull[rs], stream_pol);
                    rissued |= 1u << rs;
                    rissued_ph = (rissued_ph & ~(1u << rs)) | (rph << rs);
                    if (++rs == kResSlots) { rs = 0; rph ^= 1u; }
                }
                for (int64_t q = sl.q0; q < sl.q1; q += kAThreads) {
                    const int n = (int)min((int64_t)kAThreads, sl.q1 - q);
                    const uint64_t c0 = clock64();
                    if (!ar_wait(&sh.empty[s], ph ^ 1u, sh, p)) { ok = false; break; }
                    w_empty += (uint64_t)(clock64() - c0);
                    ptx::mbar_arrive_expect_tx(&sh.full[s], (uint32_t)(p.R * n * 16));
                    for (int r = 0; r < p.R; ++r)
                        ptx::bulk_load_hint(sh.stage + (size_t)s * kStageBytes + r * kRankBytes,
                                            p.x[r] + (sl.base + q) * 8, (uint32_t)(n * 16), &sh.full[s], stream_pol);
                    issued |= 1u << s;
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    if (++s == p.stages) { s = 0; ph ^= 1u; }
                }
            }
            prof_add(p, 1, w_empty);
            prof_add(p, 8, 1);
            // every bulk copy issued must land before the block exits
            for (int i = 0; i < p.stages; ++i) {
                if (issued & (1u << i)) {
                    const uint64_t t0 = ptx::globaltimer();
                    while (!ptx::mbar_try_wait(&sh.full[i], (issued_ph >> i) & 1u))
                        if (ptx::globaltimer() - t0 > p.timeout_ns) break;
                }
            }
            for (int i = 0; i < kResSlots; ++i) {
                if (rissued & (1u << i)) {
                    const uint64_t t0 = ptx::globaltimer();
                    while (!ptx::mbar_try_wait(&sh.rfull[i], (rissued_ph >> i) & 1u))
                        if (ptx::globaltimer() - t0 > p.timeout_ns) break;
                }
            }
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------------- phase A
        const int at = threadIdx.x - 32;
        const uint64_t keep = ptx::policy_evict_last();
        int s = 0;
        uint32_t ph = 0;
        uint32_t ncanon = 0;
        uint64_t w_full = 0, w_ahead = 0, w_ring = 0;
        for (int c = 0; c < p.num_chunks; ++c) {
            if (c >= kAhead) {  // stay at most kAhead chunks ahead of this block's phase B
                const uint64_t c0 = clock64();
                const uint64_t t0 = ptx::globaltimer();
                while (*sh.bdone < c - kAhead + 1) {
                    if (*sh.abort) break;
                    if (ptx::globaltimer() - t0 > p.timeout_ns) {
                        record_error(p.status, ARE_DEV_PIPE_TIMEOUT, blockIdx.x, -2, c);
                        *sh.abort = 1u;
                        break;
                    }
                }
                w_ahead += (uint64_t)(clock64() - c0);
            }
            const Slice sl = slice_of(p, c);
            uint32_t* chunk_staging = staging_row(p, c, 0);
            const int lap = lap_of(p, c);
            const uint32_t sent = sentinel_of(lap);
            for (int64_t q = sl.q0; q < sl.q1; q += kAThreads) {
                const int n = (int)min((int64_t)kAThreads, sl.q1 - q);
                uint32_t* dst = chunk_staging + (q + at) * 8;
                // ring laps >= 1: read the target pack (its consumer's re-arm) before overwriting it;
                // issued before the wait for the partials so the two latencies overlap
                uint4 chk0 = make_uint4(sent, sent, sent, sent), chk1 = chk0;
                if (lap > 0 && at < n) {
                    chk0 = ptx::ld_relaxed_gpu_v4(dst);
                    chk1 = ptx::ld_relaxed_gpu_v4(dst + 4);
                }
                uint64_t c0 = clock64();
                const bool ready = ar_wait(&sh.full[s], ph, sh, p);
                w_full += (uint64_t)(clock64() - c0);
                const bool work = ready && at < n;
                uint32_t wv[8];
                if (work) {
                    const uint8_t* src = sh.stage + (size_t)s * kStageBytes + at * 16;
                    float acc[8];
                    unpack8(*reinterpret_cast<const uint4*>(src), acc);
#pragma unroll
                    for (int r = 1; r < kMaxRanks; ++r) {
                        if (r < p.R) {
                            float f[8];
                            unpack8(*reinterpret_cast<const uint4*>(src + r * kRankBytes), f);
#pragma unroll
                            for (int i = 0; i < 8; ++i) acc[i] = acc[i] + f[i];
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        wv[i] = __float_as_uint(acc[i]);
                        if (wv[i] == kSentinelF32) {  // producer-side canonicalisation
                            wv[i] = 0u;
                            ++ncanon;
                        }
                        if (acc[i] != acc[i]) wv[i] = kCanonicalNaN;  // never a ring sentinel
                    }
                }
                // the warp's reads of the stage are done: one lane releases it
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sh.empty[s]);
                // the ring check, loaded before the wait, is verified only now, so its L2
                // round trip overlaps the wait and the sums; the pack is written after it
                if (lap > 0 && at < n && !(all_words(chk0, sent) && all_words(chk1, sent))) {
                    c0 = clock64();
                    const uint64_t t0 = ptx::globaltimer();
                    while (true) {
                        chk0 = ptx::ld_relaxed_gpu_v4(dst);
                        chk1 = ptx::ld_relaxed_gpu_v4(dst + 4);
                        if (all_words(chk0, sent) && all_words(chk1, sent)) break;
                        if (*sh.abort || ptx::ld_relaxed_gpu(&p.status->code) != 0u) break;
                        if (ptx::globaltimer() - t0 > p.timeout_ns) {
                            record_error(p.status, ARE_DEV_PIPE_TIMEOUT, blockIdx.x, -3, c);
                            *sh.abort = 1u;
                            break;
                        }
                    }
                    w_ring += (uint64_t)(clock64() - c0);
                }
                if (work) {
                    const int64_t pack = sl.base + q + at;
                    if (!((p.flags & ARE_DEBUG_SKIP_STAGE) && pack == p.debug_arg)) {
                        ptx::st_v4_hint(dst, make_uint4(wv[0], wv[1], wv[2], wv[3]), keep);
                        ptx::st_v4_hint(dst + 4, make_uint4(wv[4], wv[5], wv[6], wv[7]), keep);
                    }
                }
                if (++s == p.stages) { s = 0; ph ^= 1u; }
            }
        }
        if (at == 0) {
            prof_add(p, 2, w_full);
            prof_add(p, 3, w_ahead);
            prof_add(p, 4, w_ring);
        }
        if (p.flags & ARE_DEBUG_COUNT_CANON) {
            uint32_t cnt = ncanon;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
            if (lane == 0 && cnt) atomicAdd(&p.counters[0], (unsigned long long)cnt);
        }
    } else {
        // ---------------------------------------------------------------- phase B
        const int bt = threadIdx.x - 256;
        const uint64_t keep = ptx::policy_evict_last();
        int rs = 0;
        uint32_t rph = 0;
        uint64_t w_spin = 0, w_res = 0;
        const uint64_t c_start = clock64();
        if (p.gamma_in_smem) {
            // every row reads all of gamma: one copy per block in shared memory instead of
            // re-reading it through L1 (which this kernel's shared-memory carve-out leaves small)
            for (int i = bt; i < p.N / 4; i += kBThreads)
                reinterpret_cast<float4*>(sh.gam)[i] = __ldg(reinterpret_cast<const float4*>(p.gamma) + i);
            b_bar();
        }
        for (int c = 0; c < p.num_chunks; ++c) {
            const int64_t row0 = (int64_t)c * p.chunk_rows;
            const int rows = (int)min((int64_t)p.chunk_rows, (int64_t)p.M - row0);
            if (consume < rows) {
                const uint8_t* res_src = nullptr;
                if (res_smem) {
                    const uint64_t c0 = clock64();
                    ar_wait(&sh.rfull[rs], rph, sh, p);
                    w_res += (uint64_t)(clock64() - c0);
                    res_src = sh.res + (size_t)rs * p.N * 2;
                }
                norm_row<PPT>(p, sh, row0 + consume, staging_row(p, c, consume), bt, res_src, keep,
                              sentinel_of(lap_of(p, c)), rearm_value(p, c, consume), w_spin, c & 1);
                if (res_smem) {
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&sh.rempty[rs]);
                    if (++rs == kResSlots) { rs = 0; rph ^= 1u; }
                }
            }
            if (bt == 0) *sh.bdone = c + 1;
        }
        if (bt == 0) {
            prof_add(p, 5, w_spin);
            prof_add(p, 6, w_res);
            prof_add(p, 7, (uint64_t)(clock64() - c_start));
        }
    }
}

// ------------------------------------------------------------------ one-shot path
// Small messages: ROCm/aiter PR #4977, the commits that re-baseline against the
// one-stage kernel.  A reduce-scatter cannot beat a kernel that reads every
// rank's input once and stages nothing when the message is small, so the fused
// operation takes the one-shot kernel below a per-rank byte threshold set at the
// measured crossover, and the Lamport kernel above it.
//
// One row per block: one thread bulk-copies the R partial rows and the residual
// row into shared memory under one mbarrier; the 256 threads sum them in ring
// order, canonicalise exactly as the Lamport producer does, add the residual and
// normalise with the same per-thread pack order and block reduction as phase B,
// so both paths return the same bits.  As soon as h is in registers the shared
// memory is handed to the next row's copies, which then overlap this row's
// reduction and stores.
constexpr int kOsThreads = 256;

__device__ __forceinline__ bool os_wait(uint64_t* bar, uint32_t parity, const ArParams& p) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - t0 > p.timeout_ns) {
            record_error(p.status, ARE_DEV_PIPE_TIMEOUT, blockIdx.x, -4, -1);
            return false;
        }
    }
    return true;
}

template <int PPT>
__global__ void __launch_bounds__(kOsThreads, 1) ar_oneshot_kernel(const __grid_constant__ ArParams p) {
    extern __shared__ __align__(128) uint8_t os_smem[];
    const int P = p.packs_per_row;
    const uint32_t row_bytes = (uint32_t)p.N * 2u;
    const int nrows = p.R + (p.residual ? 1 : 0);
    uint8_t* rows = os_smem;  // partial rows 0..R-1, then the residual row
    uint64_t* bar = reinterpret_cast<uint64_t*>(os_smem + (size_t)nrows * row_bytes);
    float* red = reinterpret_cast<float*>(bar + 1);
    const int bt = threadIdx.x, lane = bt & 31, w = bt >> 5;
    if (bt == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    const uint64_t stream_pol = ptx::policy_evict_first();
    auto issue = [&](int64_t row) {
        if (bt == 0) {
            ptx::mbar_arrive_expect_tx(bar, (uint32_t)nrows * row_bytes);
            for (int r = 0; r < p.R; ++r)
                ptx::bulk_load_hint(rows + (size_t)r * row_bytes, p.x[r] + row * (int64_t)p.N, row_bytes, bar,
                                    stream_pol);
            if (p.residual)
                ptx::bulk_load_hint(rows + (size_t)p.R * row_bytes, p.residual + row * (int64_t)p.N, row_bytes, bar,
                                    stream_pol);
        }
    };
    uint32_t ph = 0;
    int64_t row = blockIdx.x;
    if (row < p.M) issue(row);
    for (; row < p.M; row += gridDim.x) {
        if (!os_wait(bar, ph, p)) return;  // only if a copy never lands: nothing in flight is owed then
        ph ^= 1u;
        float h[PPT][8];
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < PPT; ++k) {
            const int pk = bt + k * kOsThreads;
            if (pk < P) {
                float acc[8];
                unpack8(*reinterpret_cast<const uint4*>(rows + pk * 16), acc);
#pragma unroll
                for (int r = 1; r < kMaxRanks; ++r) {
                    if (r < p.R) {
                        float f[8];
                        unpack8(*reinterpret_cast<const uint4*>(rows + (size_t)r * row_bytes + pk * 16), f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] = acc[i] + f[i];
                    }
                }
                float r8[8];
                if (p.residual) unpack8(*reinterpret_cast<const uint4*>(rows + (size_t)p.R * row_bytes + pk * 16), r8);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint32_t wv = __float_as_uint(acc[i]);
                    if (wv == kSentinelF32) wv = 0u;                  // the Lamport producer's canonicalisation
                    if (acc[i] != acc[i]) wv = kCanonicalNaN;
                    h[k][i] = p.residual ? __uint_as_float(wv) + r8[i] : __uint_as_float(wv);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) ss = fmaf(h[k][i], h[k][i], ss);
                if (p.residual_out) {  // the updated residual stream, bf16(h)
                    const uint4 hv = make_uint4(pack_bf16x2(h[k][0], h[k][1]), pack_bf16x2(h[k][2], h[k][3]),
                                                pack_bf16x2(h[k][4], h[k][5]), pack_bf16x2(h[k][6], h[k][7]));
                    ptx::st_stream_v4(p.residual_out + row * (int64_t)p.N + pk * 8, hv);
                }
            }
        }
        __syncthreads();  // every read of this row's shared copies is done
        if (row + gridDim.x < p.M) issue(row + gridDim.x);
        ss = warp_sum(ss);
        if (lane == 0) red[w] = ss;
        __syncthreads();
        if (w == 0) {  // the same sums in the same order as sum8_tree in the Lamport kernel's phase B
            float v = lane < (kOsThreads / 32) ? red[lane] : 0.f;
            v = warp_sum(v);
            if (lane == 0) red[kOsThreads / 32] = v;
        }
        __syncthreads();
        const float inv = rsqrtf(red[kOsThreads / 32] * p.inv_n + p.eps);
        store_row<PPT, kOsThreads>(p, row, bt, h, inv, red, nullptr, [] { __syncthreads(); });
        // red[] is rewritten by the next row; this barrier also keeps the warps together, which
        // measured 10 % faster than letting early warps poll for the next row's copies
        __syncthreads();
    }
}

__global__ void fill_u32_kernel(uint32_t* dst, uint32_t v, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = v;
}

template <int PPT>
int resident(int num_sms) {
    if (cudaFuncSetAttribute(ar_rmsnorm_kernel<PPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemLimit) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ar_rmsnorm_kernel<PPT>, kArThreads, kSmemLimit) !=
        cudaSuccess)
        return 0;
    return n * num_sms;
}

}  // namespace

int ar_rmsnorm_ppt(int packs_per_row) {
    static const int kPpts[] = {1, 2, 4, 8, 16};
    for (int v : kPpts)
        if (v * kBThreads >= packs_per_row) return v;
    return 0;
}

size_t ar_rmsnorm_smem_bytes(const ArParams& p);

void ar_rmsnorm_smem_plan(ArParams& p) {
    // residual rows in shared memory when three of them leave room for >= 4 stages
    const size_t res_bytes = (size_t)kResSlots * p.N * 2;
    p.res_in_smem = (p.residual != nullptr && res_bytes + 4 * (size_t)kStageBytes + kTailBytes <= kSmemLimit) ? 1 : 0;
    const size_t avail = kSmemLimit - kTailBytes - (p.res_in_smem ? res_bytes : 0);
    // Four stages (112 KB of partials in flight per SM) measured fastest: six took 6 %
    // longer at R = 8, M = 4096, N = 7168 and eight 17 % longer; two were too few.
    int st = (int)(avail / kStageBytes);
    if (st > kArStages) st = kArStages;
    p.stages = st;
    // gamma in shared memory when it fits beside the stages and the residual rows
    p.gamma_in_smem = 0;
    p.gamma_in_smem = (ar_rmsnorm_smem_bytes(p) + (size_t)p.N * 4 <= kSmemLimit) ? 1 : 0;
}

size_t ar_rmsnorm_smem_bytes(const ArParams& p) {
    return (size_t)p.stages * kStageBytes + (p.res_in_smem ? (size_t)kResSlots * p.N * 2 : 0) +
           (p.gamma_in_smem ? (size_t)p.N * 4 : 0) + kTailBytes;
}

int ar_rmsnorm_resident_blocks(int ppt, int num_sms) {
    switch (ppt) {
        case 1: return resident<1>(num_sms);
        case 2: return resident<2>(num_sms);
        case 4: return resident<4>(num_sms);
        case 8: return resident<8>(num_sms);
        case 16: return resident<16>(num_sms);
        default: return 0;
    }
}

cudaError_t launch_ar_rmsnorm(const ArParams& p, int ppt, int grid, cudaStream_t stream) {
    const size_t smem = ar_rmsnorm_smem_bytes(p);
    switch (ppt) {
        case 1: ar_rmsnorm_kernel<1><<<grid, kArThreads, smem, stream>>>(p); break;
        case 2: ar_rmsnorm_kernel<2><<<grid, kArThreads, smem, stream>>>(p); break;
        case 4: ar_rmsnorm_kernel<4><<<grid, kArThreads, smem, stream>>>(p); break;
        case 8: ar_rmsnorm_kernel<8><<<grid, kArThreads, smem, stream>>>(p); break;
        case 16: ar_rmsnorm_kernel<16><<<grid, kArThreads, smem, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

size_t ar_oneshot_smem_bytes(int R, int N, bool residual) {
    return (size_t)(R + (residual ? 1 : 0)) * (size_t)N * 2 + 8 + 32 * 4 + 64;
}

bool ar_oneshot_fits(int R, int N, bool residual) { return ar_oneshot_smem_bytes(R, N, residual) <= kSmemLimit; }

cudaError_t ar_oneshot_prepare() {
    const int lim = (int)kSmemLimit;
    cudaError_t e = cudaFuncSetAttribute(ar_oneshot_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ar_oneshot_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ar_oneshot_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ar_oneshot_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(ar_oneshot_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    return e;
}

int ar_oneshot_threads() { return kOsThreads; }

cudaError_t launch_ar_oneshot(const ArParams& p, int ppt, int grid, cudaStream_t stream) {
    const size_t smem = ar_oneshot_smem_bytes(p.R, p.N, p.residual != nullptr);
    switch (ppt) {
        case 1: ar_oneshot_kernel<1><<<grid, kOsThreads, smem, stream>>>(p); break;
        case 2: ar_oneshot_kernel<2><<<grid, kOsThreads, smem, stream>>>(p); break;
        case 4: ar_oneshot_kernel<4><<<grid, kOsThreads, smem, stream>>>(p); break;
        case 8: ar_oneshot_kernel<8><<<grid, kOsThreads, smem, stream>>>(p); break;
        case 16: ar_oneshot_kernel<16><<<grid, kOsThreads, smem, stream>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_fill_u32(uint32_t* dst, uint32_t v, size_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    size_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    fill_u32_kernel<<<(unsigned)blocks, 256, 0, stream>>>(dst, v, n);
    return cudaGetLastError();
}

}  // namespace are
