// gn_act_lse_noalloc: the GroupNorm -> tanh -> hardswish -> residual ->
// channel-logsumexp chain without any device allocation.
//
// gn_act_lse needs 2 * N * G floats of scratch for the per-(sample, group)
// mean and 1/sqrt(var + eps), which it takes from a stream-ordered memory pool.
// Some callers cannot allow that: a plugin or engine whose host framework has
// reserved all device memory up front and forbids its components to allocate,
// or a latency-critical path that cannot afford an allocation's cost or its
// out-of-memory failure in the middle of a step.  This entry point serves
// them: its scratch is the fixed array below, compiled into the library, so the
// call allocates nothing (no cudaMalloc, cudaFree, pool or library allocator).
//
// The array holds kNoAllocMaxGroups (n, g) pairs (512 KiB); every GPU that loads
// the library keeps it until the process exits.  Every call on a device shares
// it, and it keeps the last call's contents: the statistics kernel overwrites
// every entry a call reads before the apply kernel reads it, so nothing needs
// clearing, but calls whose kernels overlap on the GPU (concurrent streams)
// race on it and must be ordered by the caller.
#include <cstdint>
#include <mutex>

#include "../../include/lse.h"
#include "launch.h"

namespace lse {

constexpr int64_t kNoAllocMaxGroups = 65536;

// Scratch for gn_act_lse_noalloc: [2 * n*G + 0] = mean, [2 * n*G + 1] = rstd.
static __device__ __align__(256) float g_noalloc_stats[2 * kNoAllocMaxGroups];

namespace {

struct NoAllocDevice {
    bool ready = false;
    DeviceInfo info;
    float* stats = nullptr;  // device address of g_noalloc_stats on this device
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
NoAllocDevice g_dev[kMaxDevices];

// Set-up, once per device, with that device current: the device facts and the
// device address of the scratch array.  (In host code the array's name is only
// a host-side stand-in; the kernels must be given this address.)
lse_status_t noalloc_device(NoAllocDevice** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return LSE_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return LSE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    NoAllocDevice& s = g_dev[dev];
    if (!s.ready) {
        DeviceInfo d;
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
                cudaSuccess) {
            record_cuda_error(e);
            return LSE_ERR_CUDA;
        }
        if (d.cc_major != 10 || d.cc_minor != 3) return LSE_ERR_UNSUPPORTED;
        float* p = nullptr;
        e = cudaGetSymbolAddress((void**)&p, g_noalloc_stats);
        if (e != cudaSuccess) {
            record_cuda_error(e);
            return LSE_ERR_CUDA;
        }
        s.info = d;
        s.stats = p;
        s.ready = true;
    }
    *out = &s;
    return LSE_OK;
}

}  // namespace
}  // namespace lse

extern "C" lse_status_t gn_act_lse_noalloc(const float* y, const float* gamma, const float* beta,
                                           float* out, int64_t N, int64_t C, int64_t HW, int64_t G,
                                           float eps, cudaStream_t stream) {
    using namespace lse;
    // gn_act_lse's argument rules, then the limit of the fixed scratch (N and G are
    // known to be positive and N * G not to overflow once check_gn has passed)
    bool empty = false;
    lse_status_t st0 = check_gn(y, gamma, beta, out, N, C, HW, G, eps, &empty);
    if (st0 != LSE_OK) return st0;
    if (N * G > kNoAllocMaxGroups) return LSE_ERR_SIZE;
    if (empty) return LSE_OK;
    NoAllocDevice* s = nullptr;
    lse_status_t st = noalloc_device(&s);
    if (st != LSE_OK) return st;
    cudaError_t e = launch_gn_act_lse(s->info, y, gamma, beta, out, N, C, HW, G, eps, s->stats, stream);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return LSE_ERR_CUDA;
    }
    return LSE_OK;
}
