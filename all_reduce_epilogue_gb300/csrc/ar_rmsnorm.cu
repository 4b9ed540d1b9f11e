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
// One-GPU design: the R "ranks" are R device buffers.  Phase A (reduce) and
// phase B (norm) are decoupled by rows: the rows are cut into chunks of
// `chunk_rows` (<= grid) rows; in pipeline step `it` every block first stages
// its share of chunk `it` (a contiguous slice of the chunk's packs), then
// normalises one row of chunk `it-1`, the row whose packs another block
// staged (row i of a chunk goes to block (i + grid/2) mod grid).  A chunk is
// staged one step before it is consumed, so spins are short and the staged
// fp32 words are read back while they still sit in L2.  The staging words are
// fp32: staging a bf16 sum would round before the residual add.
#include <cuda_bf16.h>

#include "are_internal.h"
#include "ptx.cuh"

namespace are {
namespace {

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ bool has_sentinel(const uint4& v) {
    return (v.x == kSentinelF32) | (v.y == kSentinelF32) | (v.z == kSentinelF32) | (v.w == kSentinelF32);
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

// Phase A for one 8-element pack: ring-order fp32 sum of the R bf16 values,
// -0.0 -> +0.0, two 16-byte stores into the staging words.
__device__ __forceinline__ void stage_pack(const ArParams& p, int64_t e, int64_t pack_id, uint32_t& ncanon) {
    uint4 v[kMaxRanks];
#pragma unroll
    for (int r = 0; r < kMaxRanks; ++r)
        if (r < p.R) v[r] = ptx::ld_stream_v4(p.x[r] + e);
    float acc[8];
    unpack8(v[0], acc);
#pragma unroll
    for (int r = 1; r < kMaxRanks; ++r) {
        if (r < p.R) {
            float f[8];
            unpack8(v[r], f);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = acc[i] + f[i];
        }
    }
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        w[i] = __float_as_uint(acc[i]);
        if (w[i] == kSentinelF32) {  // producer-side canonicalisation
            w[i] = 0u;
            ++ncanon;
        }
    }
    if ((p.flags & ARE_DEBUG_SKIP_STAGE) && pack_id == p.debug_arg) return;
    uint32_t* dst = p.staging + e;
    ptx::st_v4(dst, make_uint4(w[0], w[1], w[2], w[3]));
    ptx::st_v4(dst + 4, make_uint4(w[4], w[5], w[6], w[7]));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Phase B for one row: bounded spin on the staged packs, re-arm, residual add,
// sum of squares, block reduction, scale by rsqrt(ms + eps) * gamma, store.
template <int PPT>
__device__ __forceinline__ void norm_row(const ArParams& p, int64_t row, float* red) {
    const int tid = threadIdx.x;
    const int P = p.packs_per_row;
    uint32_t* srow = p.staging + row * (int64_t)p.N;
    uint4 lo[PPT], hi[PPT], res[PPT];
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int pk = tid + k * kArThreads;
        if (pk < P) {
            lo[k] = ptx::ld_relaxed_gpu_v4(srow + pk * 8);
            hi[k] = ptx::ld_relaxed_gpu_v4(srow + pk * 8 + 4);
            if (p.residual) res[k] = ptx::ld_stream_v4(p.residual + row * (int64_t)p.N + pk * 8);
        }
    }
    bool ok = true;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int pk = tid + k * kArThreads;
        if (pk < P && (has_sentinel(lo[k]) || has_sentinel(hi[k]))) {
            const uint64_t t0 = ptx::globaltimer();
            while (true) {
                lo[k] = ptx::ld_relaxed_gpu_v4(srow + pk * 8);
                hi[k] = ptx::ld_relaxed_gpu_v4(srow + pk * 8 + 4);
                if (!has_sentinel(lo[k]) && !has_sentinel(hi[k])) break;
                if (ptx::ld_relaxed_gpu(&p.status->code) != 0u) { ok = false; break; }
                if (ptx::globaltimer() - t0 > p.timeout_ns) {
                    record_error(p.status, ARE_DEV_STAGE_TIMEOUT, blockIdx.x, (int32_t)row, pk);
                    ok = false;
                    break;
                }
            }
        }
    }
    // Re-arm every pack this thread consumed (it is the pack's only consumer).
    if (ok && !(p.flags & ARE_DEBUG_NO_REARM)) {
        const uint4 s = make_uint4(kSentinelF32, kSentinelF32, kSentinelF32, kSentinelF32);
#pragma unroll
        for (int k = 0; k < PPT; ++k) {
            const int pk = tid + k * kArThreads;
            if (pk < P) {
                ptx::st_v4(srow + pk * 8, s);
                ptx::st_v4(srow + pk * 8 + 4, s);
            }
        }
    }
    // h = s + residual, kept in place in the staged registers
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int pk = tid + k * kArThreads;
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
            lo[k] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                               __float_as_uint(f[3]));
            hi[k] = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                               __float_as_uint(f[7]));
        }
    }
    const int warp = tid >> 5, lane = tid & 31;
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (warp == 0) {
        float v = lane < (kArThreads / 32) ? red[lane] : 0.f;
        v = warp_sum(v);
        if (lane == 0) red[kArThreads / 32] = v;
    }
    __syncthreads();
    const float inv = rsqrtf(red[kArThreads / 32] * p.inv_n + p.eps);
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        const int pk = tid + k * kArThreads;
        if (pk < P) {
            const float4 g0 = __ldg(reinterpret_cast<const float4*>(p.gamma) + pk * 2);
            const float4 g1 = __ldg(reinterpret_cast<const float4*>(p.gamma) + pk * 2 + 1);
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(lo[k].x) * inv * g0.x, __uint_as_float(lo[k].y) * inv * g0.y);
            o.y = pack_bf16x2(__uint_as_float(lo[k].z) * inv * g0.z, __uint_as_float(lo[k].w) * inv * g0.w);
            o.z = pack_bf16x2(__uint_as_float(hi[k].x) * inv * g1.x, __uint_as_float(hi[k].y) * inv * g1.y);
            o.w = pack_bf16x2(__uint_as_float(hi[k].z) * inv * g1.z, __uint_as_float(hi[k].w) * inv * g1.w);
            ptx::st_stream_v4(p.out + row * (int64_t)p.N + pk * 8, o);
        }
    }
}

// Blocks per SM the register budget is tuned for (the grid is still clamped
// by the runtime's occupancy query).
template <int PPT>
struct ArMinBlocks {
    static constexpr int value = PPT <= 8 ? 2 : 1;
};

template <int PPT>
__global__ void __launch_bounds__(kArThreads, ArMinBlocks<PPT>::value) ar_rmsnorm_kernel(const __grid_constant__ ArParams p) {
    __shared__ float red[kArThreads / 32 + 1];
    const int G = gridDim.x;
    const int b = blockIdx.x;
    const int P = p.packs_per_row;
    int consume = b - G / 2;  // chunk-local row this block normalises
    if (consume < 0) consume += G;
    uint32_t ncanon = 0;

    for (int it = 0; it <= p.num_chunks; ++it) {
        if (it < p.num_chunks) {  // phase A: stage chunk `it`
            const int64_t row0 = (int64_t)it * p.chunk_rows;
            const int rows = min((int64_t)p.chunk_rows, (int64_t)p.M - row0);
            const int64_t total = (int64_t)rows * P;
            const int64_t per = (total + G - 1) / G;
            const int64_t q0 = (int64_t)b * per;
            const int64_t q1 = min(total, q0 + per);
            for (int64_t q = q0 + threadIdx.x; q < q1; q += kArThreads) {
                const int64_t qa = row0 * P + q;
                stage_pack(p, qa * 8, qa, ncanon);
            }
        }
        if (it >= 1) {  // phase B: normalise one row of chunk `it - 1`
            const int64_t row0 = (int64_t)(it - 1) * p.chunk_rows;
            const int rows = min((int64_t)p.chunk_rows, (int64_t)p.M - row0);
            if (consume < rows) norm_row<PPT>(p, row0 + consume, red);
        }
    }
    if (p.flags & ARE_DEBUG_COUNT_CANON) {
        uint32_t c = ncanon;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
        if ((threadIdx.x & 31) == 0 && c) atomicAdd(&p.counters[0], (unsigned long long)c);
    }
}

__global__ void fill_u32_kernel(uint32_t* dst, uint32_t v, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = v;
}

template <int PPT>
int resident(int num_sms) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ar_rmsnorm_kernel<PPT>, kArThreads, 0) != cudaSuccess)
        return 0;
    return n * num_sms;
}

}  // namespace

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
    switch (ppt) {
        case 1: ar_rmsnorm_kernel<1><<<grid, kArThreads, 0, stream>>>(p); break;
        case 2: ar_rmsnorm_kernel<2><<<grid, kArThreads, 0, stream>>>(p); break;
        case 4: ar_rmsnorm_kernel<4><<<grid, kArThreads, 0, stream>>>(p); break;
        case 8: ar_rmsnorm_kernel<8><<<grid, kArThreads, 0, stream>>>(p); break;
        case 16: ar_rmsnorm_kernel<16><<<grid, kArThreads, 0, stream>>>(p); break;
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
