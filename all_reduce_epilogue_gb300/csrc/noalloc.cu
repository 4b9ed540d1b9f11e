// All-reduce + residual + RMSNorm for callers that cannot allocate device
// memory.
//
// Some callers must not let a library call cudaMalloc or cudaFree: a
// framework whose caching allocator has to own every device byte, a process
// running under a fixed device-memory budget, or code that must not pay the
// device-wide synchronisation an allocation or a free can imply.  They cannot
// create a workspace, so this entry point takes its scratch (the staging words
// the two phases of the kernel meet through, and the device status word) from
// a fixed array compiled into the library.  It runs the same kernel as
// are_allreduce_rmsnorm.
//
// The array lives in every GPU that loads this library, until the process
// exits.  Every call shares it and it keeps the last call's contents.
#include <cmath>
#include <cstring>
#include <mutex>

#include "are_internal.h"

using namespace are;

namespace {

constexpr size_t kHeaderWords = 64;                   // 256 bytes: device status word + padding
constexpr size_t kStagingWords = (size_t)2 << 20;      // 8 MiB of fp32 staging words: M * N <= 2,097,152
constexpr int kMaxDevices = 64;
constexpr uint64_t kTimeoutNs = 200ull * 1000 * 1000;

// The scratch.  In host code this name is only a stand-in for the symbol, not
// a device address; the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint32_t g_noalloc_scratch[kHeaderWords + kStagingWords];

struct DeviceScratch {
    uint32_t* base = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
    int resident[kArMaxPpt + 1] = {0};
};

std::mutex g_mu;
DeviceScratch g_devices[kMaxDevices];

// Once per device, with that device current: look up the array's device
// address and the kernel's co-resident grid limits.  These runtime queries may
// not run while `stream` is being captured into a graph (a capture in global
// mode would be invalidated), so a first call made under capture is refused
// before it queries anything.
are_status setup_current_device(DeviceScratch** out, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ARE_ENODEV;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceScratch& d = g_devices[dev];
    if (d.base == nullptr) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return ARE_ECUDA;
        if (cs != cudaStreamCaptureStatusNone) return ARE_ECAPTURE;
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ARE_ECUDA;
        if (major != 10 || minor != 3) return ARE_ENODEV;
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr) return ARE_ECUDA;
        for (int ppt = 1; ppt <= kArMaxPpt; ++ppt) d.resident[ppt] = ar_rmsnorm_resident_blocks(ppt, sms);
        d.num_sms = sms;
        d.base = static_cast<uint32_t*>(ptr);
    }
    *out = &d;
    return ARE_OK;
}

bool ptr_ok(const void* p, int64_t elems) {
    const bool a16 = p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
    return elems == 0 ? (p == nullptr || a16) : a16;
}

}  // namespace

extern "C" are_status are_allreduce_rmsnorm_noalloc(const are_bf16* const partials[], const are_bf16* residual,
                                                    const float* gamma, float eps, are_bf16* out, int R, int64_t M,
                                                    int64_t N, void* stream) {
    if (!partials) return ARE_EINVAL;
    are_status st = are_supports(ARE_OP_ALLREDUCE_RMSNORM, R, M, N, 0);
    if (st != ARE_OK) return st;
    for (int r = 0; r < R; ++r)
        if (!ptr_ok(partials[r], M * N)) return ARE_EINVAL;
    if ((residual && !ptr_ok(residual, 1)) || !ptr_ok(gamma, N) || !ptr_ok(out, M * N)) return ARE_EINVAL;
    if (!(eps > 0.f) || !std::isfinite(eps)) return ARE_EINVAL;
    if ((size_t)M * (size_t)N > kStagingWords) return ARE_ECAPACITY;
    if (M == 0 || N == 0) return ARE_OK;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DeviceScratch* d = nullptr;
    st = setup_current_device(&d, s);
    if (st != ARE_OK) return st;

    ArParams p;
    std::memset(&p, 0, sizeof(p));
    for (int r = 0; r < R; ++r) p.x[r] = partials[r];
    p.residual = residual;
    p.gamma = gamma;
    p.out = out;
    p.status = reinterpret_cast<DevStatus*>(d->base);
    p.counters = reinterpret_cast<unsigned long long*>(d->base + 8);
    p.staging = d->base + kHeaderWords;
    p.R = R;
    p.M = (int)M;
    p.N = (int)N;
    p.packs_per_row = (int)(N / 8);
    const int ppt = ar_rmsnorm_ppt(p.packs_per_row);
    const int resident = ppt > 0 ? d->resident[ppt] : 0;
    if (resident <= 0) return ARE_ECUDA;
    const int grid = resident < 2 * d->num_sms ? resident : 2 * d->num_sms;
    p.chunk_rows = grid;
    ar_rmsnorm_smem_plan(p);
    p.ring_slots = (M + grid - 1) / grid > kArRingSlots ? kArRingSlots : 0;
    p.num_chunks = (int)((M + grid - 1) / grid);
    p.eps = eps;
    p.inv_n = 1.0f / (float)N;
    p.flags = 0;
    p.debug_arg = -1;
    p.timeout_ns = kTimeoutNs;

    // The array keeps the previous call's contents: clear the status word and
    // arm the staging words this call uses with the -0.0 sentinel, so a call
    // never depends on how the one before it ended.
    cudaError_t e = cudaMemsetAsync(d->base, 0, kHeaderWords * sizeof(uint32_t), s);
    if (e == cudaSuccess) e = launch_fill_u32(p.staging, kSentinelF32, (size_t)M * (size_t)N, s);
    if (e == cudaSuccess) e = launch_ar_rmsnorm(p, ppt, grid, s);
    return e == cudaSuccess ? ARE_OK : ARE_ECUDA;
}

extern "C" are_status are_noalloc_device_status(are_dev_status* out) {
    if (!out) return ARE_EINVAL;
    DeviceScratch* d = nullptr;
    are_status st = setup_current_device(&d, nullptr);
    if (st != ARE_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    DevStatus v{};
    if (e == cudaSuccess) e = cudaMemcpy(&v, d->base, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return ARE_ECUDA;
    out->code = v.code;
    out->where = v.where;
    out->a = v.a;
    out->b = v.b;
    return v.code == ARE_DEV_OK ? ARE_OK : ARE_ETIMEOUT;
}
