// C ABI of liblse.so: argument checks, variant choice, scratch, status.
// Declarations and the contract of each entry point are in include/lse.h.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/lse.h"
#include "launch.h"

namespace lse {

__device__ int g_device_status = 0;

namespace {

constexpr int kMaxDevices = 64;

// Copy streams and events of the host-buffer pipeline (created on first use).
constexpr int kHostBufs = 3;
struct HostPipe {
    bool ready = false;
    std::mutex mu;  // one pipeline enqueue at a time per device
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t ev_h2d[kHostBufs] = {}, ev_comp[kHostBufs] = {}, ev_d2h[kHostBufs] = {};
};

struct DeviceState {
    bool ready = false;
    DeviceInfo info;
    cudaMemPool_t pool = nullptr;
    HostPipe pipe;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
thread_local int g_last_cuda_error = 0;

lse_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return LSE_ERR_CUDA;
}

// Per-device facts, queried once with that device current.
lse_status_t device_state(DeviceState** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return LSE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        DeviceInfo d;
        d.device = dev;
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
                cudaSuccess)
            return cuda_fail(e);
        // The kernels are built for sm_103a only.
        if (d.cc_major != 10 || d.cc_minor != 3) return LSE_ERR_UNSUPPORTED;
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_device_status)) != cudaSuccess) return cuda_fail(e);
        d.status = static_cast<int*>(p);
        s.info = d;
        s.ready = true;
    }
    *out = &s;
    return LSE_OK;
}

// The library's own stream-ordered pool on this device (idle memory is kept
// until lse_release_workspace()).
lse_status_t device_pool(DeviceState* s, cudaMemPool_t* pool) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!s->pool) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = s->info.device;
        cudaError_t e = cudaMemPoolCreate(&s->pool, &props);
        if (e != cudaSuccess) {
            s->pool = nullptr;
            return cuda_fail(e);
        }
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(s->pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    *pool = s->pool;
    return LSE_OK;
}

lse_status_t host_pipe(DeviceState* s, HostPipe** out) {
    HostPipe& hp = s->pipe;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!hp.ready) {
        cudaError_t e;
        if ((e = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_fail(e);
        for (int b = 0; b < kHostBufs; ++b) {
            if ((e = cudaEventCreateWithFlags(&hp.ev_h2d[b], cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&hp.ev_comp[b], cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&hp.ev_d2h[b], cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e);
        }
        hp.ready = true;
    }
    *out = &hp;
    return LSE_OK;
}

// Stream-ordered scratch from the device pool.  LSE_TEST_FAIL_ALLOC=1 makes it
// fail as an exhausted pool would (cudaErrorMemoryAllocation), so that the
// error path of every entry point can be exercised without using up memory.
cudaError_t pool_alloc(void** p, size_t bytes, cudaMemPool_t pool, cudaStream_t stream) {
    if (env_int("LSE_TEST_FAIL_ALLOC", 0) == 1) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMallocFromPoolAsync(p, bytes, pool, stream);
}

bool mul_ok(int64_t a, int64_t b, int64_t* r) { return !__builtin_mul_overflow(a, b, r); }

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

void record_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

static bool gn_mul_ok(int64_t a, int64_t b, int64_t* r) { return !__builtin_mul_overflow(a, b, r); }

static bool gn_aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Host-side checks shared by the GroupNorm entry points (declared in launch.h).
lse_status_t check_gn(const float* y, const float* gamma, const float* beta, const float* out, int64_t N,
                      int64_t C, int64_t HW, int64_t G, float eps, bool* empty) {
    *empty = false;
    if (N < 0 || HW < 0 || C <= 0 || G <= 0 || C % G != 0) return LSE_ERR_SIZE;
    if (C > kGnMaxChannels) return LSE_ERR_SIZE;
    int64_t nchw = 0, nhw = 0, ng = 0;
    if (!gn_mul_ok(N, C, &nchw) || !gn_mul_ok(nchw, HW, &nchw) || nchw > INT64_MAX / 4 ||
        !gn_mul_ok(N, HW, &nhw) || !gn_mul_ok(N, G, &ng))
        return LSE_ERR_SIZE;
    if (!(eps >= 0.f) || eps == __builtin_inff()) return LSE_ERR_VALUE;
    if (nhw == 0) {
        *empty = true;
        return LSE_OK;
    }
    if (!y || !gamma || !beta || !out) return LSE_ERR_NULL;
    if (!gn_aligned4(y) || !gn_aligned4(gamma) || !gn_aligned4(beta) || !gn_aligned4(out)) return LSE_ERR_ALIGN;
    return LSE_OK;
}

}  // namespace lse

using namespace lse;

extern "C" {

lse_status_t lse_reduce(const float* x, float* out, int64_t outer, int64_t R, int64_t inner,
                        cudaStream_t stream) {
    if (outer < 0 || R < 0 || inner < 0) return LSE_ERR_SIZE;
    int64_t nout = 0, nin = 0;
    if (!mul_ok(outer, inner, &nout) || !mul_ok(nout, R, &nin) || nin > INT64_MAX / 4)
        return LSE_ERR_SIZE;
    if (nout == 0) return LSE_OK;
    if (R == 0) return LSE_ERR_SIZE;
    if (!x || !out) return LSE_ERR_NULL;
    if (!aligned4(x) || !aligned4(out)) return LSE_ERR_ALIGN;
    DeviceState* s = nullptr;
    lse_status_t st = device_state(&s);
    if (st != LSE_OK) return st;
    cudaError_t e;
    if (inner == 1) {
        // Contiguous reduced axis: the row statistic of form 2, one value per row.
        if (R <= kRegRowMaxCols)
            e = launch_rows_reg(s->info, x, out, outer, R, 1, stream);
        else
            e = launch_rows_stream(s->info, x, out, outer, R, 1, stream);
    } else {
        e = launch_lse_strided(s->info, x, out, outer, R, inner, stream);
    }
    return e == cudaSuccess ? LSE_OK : cuda_fail(e);
}

}  // extern "C"

namespace {

// Row-wise log_softmax (softmax = false) or softmax (true) of a (rows, cols)
// tensor, after the entry point's argument checks.
lse_status_t row_transform(const float* x, float* out, int64_t rows, int64_t cols, bool softmax,
                           cudaStream_t stream) {
    DeviceState* s = nullptr;
    lse_status_t st = device_state(&s);
    if (st != LSE_OK) return st;
    cudaError_t e;
    // LSE_LSM_VARIANT forces a kernel: 1 registers, 2 cluster shared memory,
    // 3 streaming, 4 lock-step group shared memory, 5 group with an L2 re-read,
    // 6 warp-specialised group shared memory, 7 the same with a ring of chunk slots
    // per CTA, 8 the same with its rows parked in tensor memory (the default for long
    // 16-byte-aligned rows; 6 where 8 has no plan).  softmax has the register,
    // streaming and warp-specialised kernels only.
    int force = env_int("LSE_LSM_VARIANT", 0);
    if (softmax && force != 1 && force != 3 && force != 6 && force != 7 && force != 8) force = 0;
    if ((force == 0 || force == 1) && cols <= kRegRowMaxCols) {
        e = launch_rows_reg(s->info, x, out, rows, cols, softmax ? 2 : 0, stream);
    } else {
        e = cudaErrorNotSupported;
        if (force == 2) {
            e = launch_lsm_smem_cluster(s->info, x, out, rows, cols, stream);
        } else if (force == 0 || (force >= 4 && force <= 8)) {
            GroupPlan plan;
            auto plan_kind = [&](int kind) {
                return kind == 5 ? plan_lsm_l2_group(s->info, x, out, rows, cols, &plan)
                     : kind == 6 ? plan_lsm_ws_group(s->info, x, out, rows, cols, &plan)
                     : kind == 7 ? plan_lsm_ring_group(s->info, x, out, rows, cols, &plan)
                     : kind == 8 ? plan_lsm_tmem_group(s->info, x, out, rows, cols, &plan)
                                 : plan_lsm_smem_group(s->info, x, out, rows, cols, &plan);
            };
            int kind = force == 0 ? 8 : force;
            e = plan_kind(kind);
            if (e == cudaErrorNotSupported && force == 0) e = plan_kind(kind = 6);
            if (e == cudaSuccess) {
                cudaMemPool_t pool = nullptr;
                if ((st = device_pool(s, &pool)) != LSE_OK) return st;
                void* scratch = nullptr;
                e = pool_alloc(&scratch, plan.scratch_bytes, pool, stream);
                if (e != cudaSuccess) return cuda_fail(e);
                e = kind == 5 ? launch_lsm_l2_group(s->info, x, out, rows, cols, plan, scratch, stream)
                  : kind == 6 ? launch_lsm_ws_group(s->info, x, out, rows, cols, plan, scratch, stream, softmax)
                  : kind == 7 ? launch_lsm_ring_group(s->info, x, out, rows, cols, plan, scratch, stream, softmax)
                  : kind == 8 ? launch_lsm_tmem_group(s->info, x, out, rows, cols, plan, scratch, stream, softmax)
                              : launch_lsm_smem_group(s->info, x, out, rows, cols, plan, scratch, stream);
                cudaError_t ef = cudaFreeAsync(scratch, stream);
                if (e == cudaSuccess) e = ef;
            }
        }
        if (e == cudaErrorNotSupported) {
            (void)cudaGetLastError();
            e = launch_rows_stream(s->info, x, out, rows, cols, softmax ? 2 : 0, stream);
        }
    }
    return e == cudaSuccess ? LSE_OK : cuda_fail(e);
}

// Host-side checks shared by the row entry points.
lse_status_t check_rows(const float* x, const float* out, int64_t rows, int64_t cols, bool* empty) {
    *empty = false;
    if (rows < 0 || cols < 0) return LSE_ERR_SIZE;
    int64_t n = 0;
    if (!mul_ok(rows, cols, &n) || n > INT64_MAX / 4) return LSE_ERR_SIZE;
    if (n == 0) {
        *empty = true;
        return LSE_OK;
    }
    if (!x || !out) return LSE_ERR_NULL;
    if (!aligned4(x) || !aligned4(out)) return LSE_ERR_ALIGN;
    return LSE_OK;
}

// The one-kernel GroupNorm chain with output kind out_kind (0 channel lse,
// 1 GroupNorm, 2 chain before the lse), scratch from the device pool.
// By default the channel lse takes the work queue with per-thread loads and the
// elementwise outputs the (sample, group) slabs as rows of the tensor-memory row kernel
// (the bulk-copy work queue where that does not apply).  LSE_GN_VARIANT 2 forces the
// work-queue kernel with per-thread loads, 3 the one with bulk-copy staging, 4 the
// sample-slice kernel (y read once, slices kept in shared memory; the channel lse
// only, where it applies; measured slower on GB300), 5 the tile queue with tiles
// parked in tensor memory (y read once; the channel lse only, where it applies), 6 the
// (sample, group) slabs as rows of the tensor-memory row kernel (GroupNorm and the
// chain before the lse, where it applies), 7 the whole grid on one sample at a time
// (y read once; the channel lse only, where it applies).
lse_status_t gn_fused(const float* y, const float* gamma, const float* beta, float* out, int64_t N, int64_t C,
                      int64_t HW, int64_t G, float eps, int out_kind, cudaStream_t stream) {
    DeviceState* s = nullptr;
    lse_status_t st = device_state(&s);
    if (st != LSE_OK) return st;
    cudaMemPool_t pool = nullptr;
    if ((st = device_pool(s, &pool)) != LSE_OK) return st;
    const int variant = env_int("LSE_GN_VARIANT", 0);
    if (out_kind != 0 && (variant == 6 || variant == 0)) {
        // the slabs as rows parked in tensor memory: y read once, out written once
        GroupPlan plan;
        if (plan_gn_rows(s->info, y, out, N, C, HW, G, out_kind, &plan) == cudaSuccess) {
            void* scratch = nullptr;
            cudaError_t e = pool_alloc(&scratch, plan.scratch_bytes, pool, stream);
            if (e != cudaSuccess) return cuda_fail(e);
            e = launch_gn_rows(s->info, y, gamma, beta, out, N, C, HW, G, eps, plan, scratch, stream, out_kind);
            cudaError_t ef = cudaFreeAsync(scratch, stream);
            if (e == cudaSuccess && ef == cudaSuccess) return LSE_OK;
            if (e != cudaErrorNotSupported) return cuda_fail(e != cudaSuccess ? e : ef);
            (void)cudaGetLastError();  // not launchable here: the default path below
        }
    }
    if (out_kind == 0 && variant == 7) {
        // the channel lse with y read once: the whole grid on one sample at a time
        GnSweepPlan plan;
        if (gn_sweep_plan(s->info, y, N, C, HW, G, &plan)) {
            void* scratch = nullptr;
            cudaError_t e = pool_alloc(&scratch, plan.scratch_bytes, pool, stream);
            if (e != cudaSuccess) return cuda_fail(e);
            e = launch_gn_sweep(s->info, y, gamma, beta, out, N, C, HW, G, eps, plan, scratch, stream);
            cudaError_t ef = cudaFreeAsync(scratch, stream);
            if (e == cudaSuccess && ef == cudaSuccess) return LSE_OK;
            if (e != cudaErrorNotSupported) return cuda_fail(e != cudaSuccess ? e : ef);
            (void)cudaGetLastError();  // not launchable here: the default path below
        }
    }
    if (out_kind == 0 && variant == 5) {
        // the channel lse with y read once: tiles parked in tensor memory
        GnTmemPlan plan;
        if (gn_tmem_plan(s->info, y, out, N, C, HW, G, &plan)) {
            void* scratch = nullptr;
            cudaError_t e = pool_alloc(&scratch, plan.scratch_bytes, pool, stream);
            if (e != cudaSuccess) return cuda_fail(e);
            e = launch_gn_tmem(s->info, y, gamma, beta, out, N, C, HW, G, eps, plan, scratch, stream);
            cudaError_t ef = cudaFreeAsync(scratch, stream);
            if (e == cudaSuccess && ef == cudaSuccess) return LSE_OK;
            if (e != cudaErrorNotSupported) return cuda_fail(e != cudaSuccess ? e : ef);
            (void)cudaGetLastError();  // not launchable here: the default path below
        }
    }
    if (out_kind == 0 && variant == 4) {
        // the channel lse with y read once: sample slices held in shared memory
        GnSlabPlan plan;
        if (gn_slab_plan(s->info, y, out, N, C, HW, G, &plan)) {
            void* scratch = nullptr;
            cudaError_t e = pool_alloc(&scratch, plan.scratch_bytes, pool, stream);
            if (e != cudaSuccess) return cuda_fail(e);
            e = launch_gn_slab(s->info, y, gamma, beta, out, N, C, HW, G, eps, plan, scratch, stream);
            cudaError_t ef = cudaFreeAsync(scratch, stream);
            if (e != cudaSuccess) return cuda_fail(e);
            if (ef != cudaSuccess) return cuda_fail(ef);
            return LSE_OK;
        }
    }
    const bool want_tma = variant == 3 || (variant != 2 && out_kind != 0);
    const bool tma = want_tma && gn_tma_applies(s->info, y, out, C, HW);
    void* scratch = nullptr;
    cudaError_t e = pool_alloc(&scratch, tma ? gn_tma_scratch_bytes(N, G) : gn_fused_scratch_bytes(N, G, out_kind),
                                            pool, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    if (tma)
        e = launch_gn_tma(s->info, y, gamma, beta, out, N, C, HW, G, eps, scratch, stream, out_kind);
    else
        e = launch_gn_act_lse_fused(s->info, y, gamma, beta, out, N, C, HW, G, eps, scratch, stream, out_kind);
    cudaError_t ef = cudaFreeAsync(scratch, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    if (ef != cudaSuccess) return cuda_fail(ef);
    return LSE_OK;
}

}  // namespace

extern "C" {

lse_status_t log_softmax_lastdim(const float* x, float* out, int64_t rows, int64_t cols,
                                 cudaStream_t stream) {
    bool empty = false;
    lse_status_t st = check_rows(x, out, rows, cols, &empty);
    if (st != LSE_OK || empty) return st;
    return row_transform(x, out, rows, cols, false, stream);
}

lse_status_t softmax_lastdim(const float* x, float* out, int64_t rows, int64_t cols, cudaStream_t stream) {
    bool empty = false;
    lse_status_t st = check_rows(x, out, rows, cols, &empty);
    if (st != LSE_OK || empty) return st;
    return row_transform(x, out, rows, cols, true, stream);
}

lse_status_t log_softmax_dim(const float* x, float* out, int64_t outer, int64_t R, int64_t inner,
                             cudaStream_t stream) {
    if (outer < 0 || R < 0 || inner < 0) return LSE_ERR_SIZE;
    int64_t rows = 0, n = 0;
    if (!mul_ok(outer, inner, &rows) || !mul_ok(rows, R, &n) || n > INT64_MAX / 4) return LSE_ERR_SIZE;
    if (n == 0) return LSE_OK;
    if (!x || !out) return LSE_ERR_NULL;
    if (!aligned4(x) || !aligned4(out)) return LSE_ERR_ALIGN;
    if (inner == 1) return row_transform(x, out, outer, R, false, stream);
    DeviceState* s = nullptr;
    lse_status_t st = device_state(&s);
    if (st != LSE_OK) return st;
    cudaError_t e = launch_lse_strided(s->info, x, out, outer, R, inner, stream, true);
    return e == cudaSuccess ? LSE_OK : cuda_fail(e);
}

lse_status_t conv2d_3x3(const float* x, const float* w, const float* b, float* y, int64_t N, int64_t Cin,
                        int64_t H, int64_t W, int64_t Cout, cudaStream_t stream) {
    if (N < 0 || Cin <= 0 || Cout <= 0 || H < 3 || W < 3) return LSE_ERR_SIZE;
    int64_t nin = 0, nout = 0;
    if (!mul_ok(N, Cin, &nin) || !mul_ok(nin, H, &nin) || !mul_ok(nin, W, &nin) || nin > INT64_MAX / 4 ||
        !mul_ok(N, Cout, &nout) || !mul_ok(nout, (H - 2) * (W - 2), &nout) || nout > INT64_MAX / 4 ||
        H > INT32_MAX || W > INT32_MAX)
        return LSE_ERR_SIZE;
    if (!conv_tc_supported(Cin, Cout, W)) return LSE_ERR_UNSUPPORTED;
    if (nout == 0) return LSE_OK;
    if (!x || !w || !b || !y) return LSE_ERR_NULL;
    if (!aligned4(x) || !aligned4(w) || !aligned4(b) || !aligned4(y)) return LSE_ERR_ALIGN;
    DeviceState* s = nullptr;
    lse_status_t st = device_state(&s);
    if (st != LSE_OK) return st;
    cudaError_t e = launch_conv2d_3x3(s->info, x, w, b, y, N, Cin, H, W, Cout, stream);
    return e == cudaSuccess ? LSE_OK : cuda_fail(e);
}

lse_status_t conv_gn_act_lse(const float* x, const float* w, const float* b, const float* gamma,
                             const float* beta, float* out, int64_t N, int64_t Cin, int64_t H, int64_t W,
                             int64_t Cout, int64_t G, float eps, cudaStream_t stream) {
    if (N < 0 || Cin <= 0 || Cout <= 0 || G <= 0 || H < 3 || W < 3 || Cout % G != 0) return LSE_ERR_SIZE;
    int64_t nin = 0, ny = 0;
    if (!mul_ok(N, Cin, &nin) || !mul_ok(nin, H, &nin) || !mul_ok(nin, W, &nin) || nin > INT64_MAX / 4 ||
        !mul_ok(N, Cout, &ny) || !mul_ok(ny, (H - 2) * (W - 2), &ny) || ny > INT64_MAX / 4 || H > INT32_MAX ||
        W > INT32_MAX)
        return LSE_ERR_SIZE;
    const int64_t cpg = Cout / G;
    if (!conv_tc_supported(Cin, Cout, W) || Cin != 8 || 16 % cpg != 0 || G > 64) return LSE_ERR_UNSUPPORTED;
    if (!(eps >= 0.f) || eps == __builtin_inff()) return LSE_ERR_VALUE;
    if (ny == 0) return LSE_OK;
    if (!x || !w || !b || !gamma || !beta || !out) return LSE_ERR_NULL;
    if (!aligned4(x) || !aligned4(w) || !aligned4(b) || !aligned4(gamma) || !aligned4(beta) || !aligned4(out))
        return LSE_ERR_ALIGN;
    DeviceState* s = nullptr;
    lse_status_t st = device_state(&s);
    if (st != LSE_OK) return st;
    cudaMemPool_t pool = nullptr;
    if ((st = device_pool(s, &pool)) != LSE_OK) return st;
    void* scratch = nullptr;
    cudaError_t e =
        pool_alloc(&scratch, conv_chain_scratch_bytes(N, H, W, Cout, G), pool, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_conv_gn_act_lse(s->info, x, w, b, gamma, beta, out, N, Cin, H, W, Cout, G, eps, scratch, stream);
    cudaError_t ef = cudaFreeAsync(scratch, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    if (ef != cudaSuccess) return cuda_fail(ef);
    return LSE_OK;
}

lse_status_t group_norm(const float* y, const float* gamma, const float* beta, float* out, int64_t N, int64_t C,
                        int64_t HW, int64_t G, float eps, cudaStream_t stream) {
    bool empty = false;
    lse_status_t st = check_gn(y, gamma, beta, out, N, C, HW, G, eps, &empty);
    if (st != LSE_OK || empty) return st;
    return gn_fused(y, gamma, beta, out, N, C, HW, G, eps, 1, stream);
}

lse_status_t gn_act_residual(const float* y, const float* gamma, const float* beta, float* out, int64_t N,
                             int64_t C, int64_t HW, int64_t G, float eps, cudaStream_t stream) {
    bool empty = false;
    lse_status_t st = check_gn(y, gamma, beta, out, N, C, HW, G, eps, &empty);
    if (st != LSE_OK || empty) return st;
    return gn_fused(y, gamma, beta, out, N, C, HW, G, eps, 2, stream);
}

lse_status_t gn_act_lse(const float* y, const float* gamma, const float* beta, float* out,
                        int64_t N, int64_t C, int64_t HW, int64_t G, float eps,
                        cudaStream_t stream) {
    bool empty = false;
    lse_status_t st = check_gn(y, gamma, beta, out, N, C, HW, G, eps, &empty);
    if (st != LSE_OK || empty) return st;
    // LSE_GN_VARIANT=1 selects the two-kernel path (statistics, then apply);
    // otherwise one work-queue kernel (see gn_fused).
    if (env_int("LSE_GN_VARIANT", 0) != 1) return gn_fused(y, gamma, beta, out, N, C, HW, G, eps, 0, stream);
    DeviceState* s = nullptr;
    if ((st = device_state(&s)) != LSE_OK) return st;
    cudaMemPool_t pool = nullptr;
    if ((st = device_pool(s, &pool)) != LSE_OK) return st;
    void* stats = nullptr;
    cudaError_t e = pool_alloc(&stats, (size_t)N * G * 2 * sizeof(float), pool, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_gn_act_lse(s->info, y, gamma, beta, out, N, C, HW, G, eps, static_cast<float*>(stats), stream);
    cudaError_t ef = cudaFreeAsync(stats, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    if (ef != cudaSuccess) return cuda_fail(ef);
    return LSE_OK;
}

lse_status_t log_softmax_lastdim_host(const float* x, float* out, int64_t rows, int64_t cols,
                                      cudaStream_t stream) {
    if (rows < 0 || cols < 0) return LSE_ERR_SIZE;
    int64_t n = 0;
    if (!mul_ok(rows, cols, &n) || n > INT64_MAX / 4) return LSE_ERR_SIZE;
    if (n == 0) return LSE_OK;
    if (!x || !out) return LSE_ERR_NULL;
    if (!aligned4(x) || !aligned4(out)) return LSE_ERR_ALIGN;
    DeviceState* s = nullptr;
    lse_status_t st = device_state(&s);
    if (st != LSE_OK) return st;
    cudaMemPool_t pool = nullptr;
    if ((st = device_pool(s, &pool)) != LSE_OK) return st;
    HostPipe* hp = nullptr;
    if ((st = host_pipe(s, &hp)) != LSE_OK) return st;

    // Chunks of whole rows of about LSE_HOST_CHUNK_MB (default 256) MB each,
    // three in flight: the copy in of chunk i+1, the call on chunk i and the
    // copy out of chunk i-1 overlap.
    const int64_t row_bytes = cols * 4;
    const int64_t target = (int64_t)std::max(1, env_int("LSE_HOST_CHUNK_MB", 256)) << 20;
    const int64_t chunk_rows = std::max<int64_t>(1, std::min<int64_t>(rows, target / row_bytes));
    const int64_t nchunks = (rows + chunk_rows - 1) / chunk_rows;
    const size_t buf_bytes = (size_t)((chunk_rows * row_bytes + 255) / 256 * 256);

    std::lock_guard<std::mutex> lock(hp->mu);
    void* mem = nullptr;
    cudaError_t e = pool_alloc(&mem, 2 * kHostBufs * buf_bytes, pool, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    auto din = [&](int b) { return reinterpret_cast<float*>(static_cast<char*>(mem) + (size_t)b * buf_bytes); };
    auto dout = [&](int b) {
        return reinterpret_cast<float*>(static_cast<char*>(mem) + (size_t)(kHostBufs + b) * buf_bytes);
    };
    // Order the copy streams after everything already queued on `stream`
    // (including the staging allocation).
    if ((e = cudaEventRecord(hp->start, stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->h2d, hp->start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->d2h, hp->start, 0)) != cudaSuccess)
        return cuda_fail(e);
    for (int64_t i = 0; i < nchunks; ++i) {
        const int b = (int)(i % kHostBufs);
        const int64_t r0 = i * chunk_rows;
        const int64_t nr = std::min(chunk_rows, rows - r0);
        const size_t bytes = (size_t)(nr * row_bytes);
        // buffer b is free once chunk i - kHostBufs has been copied out
        if (i >= kHostBufs && (e = cudaStreamWaitEvent(hp->h2d, hp->ev_d2h[b], 0)) != cudaSuccess)
            return cuda_fail(e);
        if ((e = cudaMemcpyAsync(din(b), x + r0 * cols, bytes, cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess ||
            (e = cudaEventRecord(hp->ev_h2d[b], hp->h2d)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(stream, hp->ev_h2d[b], 0)) != cudaSuccess)
            return cuda_fail(e);
        st = log_softmax_lastdim(din(b), dout(b), nr, cols, stream);
        if (st != LSE_OK) return st;
        if ((e = cudaEventRecord(hp->ev_comp[b], stream)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(hp->d2h, hp->ev_comp[b], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(out + r0 * cols, dout(b), bytes, cudaMemcpyDeviceToHost, hp->d2h)) != cudaSuccess ||
            (e = cudaEventRecord(hp->ev_d2h[b], hp->d2h)) != cudaSuccess)
            return cuda_fail(e);
    }
    // `stream` resumes after the last copy out; then the staging memory returns.
    for (int b = 0; b < kHostBufs && b < nchunks; ++b)
        if ((e = cudaStreamWaitEvent(stream, hp->ev_d2h[b], 0)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaFreeAsync(mem, stream)) != cudaSuccess) return cuda_fail(e);
    return LSE_OK;
}

lse_status_t lse_release_workspace(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    for (int d = 0; d < kMaxDevices; ++d) {
        if (g_dev[d].pool) {
            cudaError_t e = cudaMemPoolTrimTo(g_dev[d].pool, 0);
            if (e != cudaSuccess) return cuda_fail(e);
        }
    }
    return LSE_OK;
}

lse_status_t lse_device_status(cudaStream_t stream) {
    DeviceState* s = nullptr;
    lse_status_t st = device_state(&s);
    if (st != LSE_OK) return st;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    int v = 0;
    e = cudaMemcpy(&v, s->info.status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpy(s->info.status, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e);
        return LSE_ERR_TIMEOUT;
    }
    return LSE_OK;
}

const char* lse_status_string(lse_status_t status) {
    switch (status) {
        case LSE_OK: return "ok";
        case LSE_ERR_NULL: return "null pointer argument";
        case LSE_ERR_SIZE: return "invalid size argument";
        case LSE_ERR_ALIGN: return "pointer not 4-byte aligned";
        case LSE_ERR_CUDA: return "CUDA error (see lse_last_cuda_error)";
        case LSE_ERR_UNSUPPORTED: return "device not supported (needs sm_103a)";
        case LSE_ERR_VALUE: return "invalid scalar argument";
        case LSE_ERR_TIMEOUT: return "a kernel timed out waiting on a bulk copy";
    }
    return "unknown status";
}

int lse_last_cuda_error(void) { return g_last_cuda_error; }

int lse_version(void) { return 100; }

}  // extern "C"
