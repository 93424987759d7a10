// Internal launchers of the logsumexp kernels (host side, C++ linkage).
// lse_api.cu validates arguments and picks a variant; these only launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lse.h"

namespace lse {

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int max_smem_optin = 0;   // bytes of dynamic shared memory a block may opt in to
    int* status = nullptr;    // device address of the library's status word
};

// Form 1: out[o, i] = lse over r of x[o, r, i] (inner > 1).  With log_softmax
// set, out[o, r, i] = x[o, r, i] - that lse instead (out has x's shape).
cudaError_t launch_lse_strided(const DeviceInfo& dev, const float* x, float* out, int64_t outer,
                               int64_t R, int64_t inner, cudaStream_t stream, bool log_softmax = false);

// Form 2, rows held in registers (cols up to kRegRowMaxCols).  mode 0 writes
// log_softmax into out (rows x cols); mode 1 writes the row lse into out (rows);
// mode 2 writes softmax into out (rows x cols).
constexpr int64_t kRegRowMaxCols = 32768;
cudaError_t launch_rows_reg(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                            int64_t cols, int mode, cudaStream_t stream);

// Form 2, rows staged in the shared memory of a thread-block cluster (one bulk
// read of x).  Returns cudaErrorNotSupported when the row cannot be staged.
cudaError_t launch_lsm_smem_cluster(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                    int64_t cols, cudaStream_t stream);

// Form 2, rows staged in shared memory across a group of CTAs of a cooperative
// grid (all SMs usable, unlike clusters, which GPC boundaries constrain); the
// CTAs of a row merge their partial pairs through global memory.  plan_* sizes
// the launch and its scratch (tagged partial slots); launch_* initialises the
// slots on `stream` and launches.  cudaErrorNotSupported when the row cannot
// be staged.
struct GroupPlan {
    int threads = 0, nbuf = 1, group_size = 0, groups = 0, slice = 0, chunk = 0;
    size_t smem = 0, scratch_bytes = 0;
};
cudaError_t plan_lsm_smem_group(const DeviceInfo& dev, const float* x, const float* out, int64_t rows,
                                int64_t cols, GroupPlan* plan);
cudaError_t launch_lsm_smem_group(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                  int64_t cols, const GroupPlan& plan, void* scratch,
                                  cudaStream_t stream);

// Form 2, warp-specialised group kernel (fold warps and store warps on two
// buffers).  Same plan / scratch protocol.
cudaError_t plan_lsm_ws_group(const DeviceInfo& dev, const float* x, const float* out, int64_t rows,
                              int64_t cols, GroupPlan* plan);
cudaError_t launch_lsm_ws_group(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                int64_t cols, const GroupPlan& plan, void* scratch, cudaStream_t stream,
                                bool softmax = false);

// Form 2, the warp-specialised group kernel with a ring of chunk slots per CTA in
// place of whole-slice buffers (plan.nbuf holds the ring's slot count).  Same plan /
// scratch protocol.
cudaError_t plan_lsm_ring_group(const DeviceInfo& dev, const float* x, const float* out, int64_t rows,
                                int64_t cols, GroupPlan* plan);
cudaError_t launch_lsm_ring_group(const DeviceInfo& dev, const float* x, float* out, int64_t rows, int64_t cols,
                                  const GroupPlan& plan, void* scratch, cudaStream_t stream, bool softmax = false);

// Form 2, the warp-specialised group kernel with its rows parked in tensor memory
// while their lse is merged (shared memory holds landing chunks only); plan.nbuf holds
// 100 x landing slots + tensor-memory row buffers.  Same plan / scratch protocol.
cudaError_t plan_lsm_tmem_group(const DeviceInfo& dev, const float* x, const float* out, int64_t rows,
                                int64_t cols, GroupPlan* plan);
cudaError_t launch_lsm_tmem_group(const DeviceInfo& dev, const float* x, float* out, int64_t rows, int64_t cols,
                                  const GroupPlan& plan, void* scratch, cudaStream_t stream, bool softmax = false);

// Form 2, rows split over a group of CTAs of a cooperative grid that read their
// slices twice, the second time from L2.  Same plan / scratch protocol.
cudaError_t plan_lsm_l2_group(const DeviceInfo& dev, const float* x, const float* out, int64_t rows,
                              int64_t cols, GroupPlan* plan);
cudaError_t launch_lsm_l2_group(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                int64_t cols, const GroupPlan& plan, void* scratch, cudaStream_t stream);

// Form 2, any row length: each CTA of a cluster streams its slice of the row
// (stats pass, then for mode 0 an apply pass).  mode as for launch_rows_reg.
cudaError_t launch_rows_stream(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                               int64_t cols, int mode, cudaStream_t stream);

// Form 3: per-(n, g) statistics into `stats` (2 * N * G floats), then the fused
// normalise / tanh / hardswish / residual / channel-lse pass.
cudaError_t launch_gn_act_lse(const DeviceInfo& dev, const float* y, const float* gamma,
                              const float* beta, float* out, int64_t N, int64_t C, int64_t HW,
                              int64_t G, float eps, float* stats, cudaStream_t stream);

// The apply stage alone: per-(n, g) stats (mean, 1/sqrt(var + eps)) in, the
// normalise / tanh / hardswish / residual / channel-lse pass out.
cudaError_t launch_gn_apply(const DeviceInfo& dev, const float* y, const float* gamma, const float* beta, float* out,
                            int64_t N, int64_t C, int64_t HW, int64_t G, const float* stats, cudaStream_t stream);

// Form 3 in one cooperative kernel: statistics parts and apply tiles of the
// samples claimed from one work queue, each sample's second read close behind
// its first so that it hits L2.  Scratch: gn_fused_scratch_bytes(N, G, out_kind).
// out_kind 0 writes the channel lse (N x HW); 1 the GroupNorm output and 2 the
// chain before the lse, y + hardswish(tanh(GroupNorm(y))) (both N x C x HW).
size_t gn_fused_scratch_bytes(int64_t N, int64_t G, int out_kind);
cudaError_t launch_gn_act_lse_fused(const DeviceInfo& dev, const float* y, const float* gamma,
                                    const float* beta, float* out, int64_t N, int64_t C, int64_t HW,
                                    int64_t G, float eps, void* scratch, cudaStream_t stream,
                                    int out_kind = 0, bool reverse = false);

// Form 3 (and GroupNorm alone, and the chain before its lse) on the same
// work-queue schedule, each item staged through a ring of shared-memory slots
// by bulk copies.  Applies when HW % 4 == 0, y and out are 16-byte aligned and
// the ring fits; scratch: gn_tma_scratch_bytes(N, G).  out_kind as above.
bool gn_tma_applies(const DeviceInfo& dev, const float* y, const float* out, int64_t C, int64_t HW);
size_t gn_tma_scratch_bytes(int64_t N, int64_t G);
cudaError_t launch_gn_tma(const DeviceInfo& dev, const float* y, const float* gamma, const float* beta, float* out,
                          int64_t N, int64_t C, int64_t HW, int64_t G, float eps, void* scratch, cudaStream_t stream,
                          int out_kind);

// GroupNorm and the chain before the lse (out_kind 1 / 2) as rows of the tensor-memory
// row kernel: the N x G slabs of C / G x HW floats, each read once and written once
// (HW % 4 == 0, 16-byte aligned y and out; the default for these outputs where it
// applies).  Same plan / scratch protocol as plan_lsm_tmem_group.
cudaError_t plan_gn_rows(const DeviceInfo& dev, const float* y, const float* out, int64_t N, int64_t C, int64_t HW,
                         int64_t G, int out_kind, GroupPlan* plan);
cudaError_t launch_gn_rows(const DeviceInfo& dev, const float* y, const float* gamma, const float* beta, float* out,
                           int64_t N, int64_t C, int64_t HW, int64_t G, float eps, const GroupPlan& plan,
                           void* scratch, cudaStream_t stream, int out_kind);

// cuTensorMapEncodeTiled from the driver, found once through the runtime (the library
// does not link the driver library itself); null if unavailable.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled();

// Form 3 with y read once and each tile parked in tensor memory (the channel lse
// only): a work queue of 256-pixel tiles of all C channels, claimed in sample order;
// each tile lands in shared memory (2-D tensor copy), its per-group moments are
// folded and published, it is copied into tensor memory, and once its sample's
// statistics are complete (the last tile's CTA builds the channel table) the chain
// and the channel lse run from tensor memory.  gn_tmem_plan says whether it applies
// (HW % 4 == 0, 4 <= C <= 64 with C % 4 == 0, 16-byte aligned y and out, enough tile
// buffers for the deadlock bound) and sizes the launch and its scratch.
struct GnTmemPlan {
    int grid = 0, T = 0, TR = 0, R = 0, threads = 0;
    size_t smem = 0, scratch_bytes = 0;
};
bool gn_tmem_plan(const DeviceInfo& dev, const float* y, const float* out, int64_t N, int64_t C, int64_t HW,
                  int64_t G, GnTmemPlan* plan);
cudaError_t launch_gn_tmem(const DeviceInfo& dev, const float* y, const float* gamma, const float* beta, float* out,
                           int64_t N, int64_t C, int64_t HW, int64_t G, float eps, const GnTmemPlan& plan,
                           void* scratch, cudaStream_t stream);

// Form 3 with y read once, the whole grid on one sample at a time: CTA j holds pixel
// slice j of all C channels of each sample in a ring of shared-memory slots, the group
// statistics are grid-wide fp64 sums (the channel lse only).  gn_sweep_plan says whether
// it applies (HW % 4 == 0 with a slice of at most 256 pixels, 4 <= C <= 64 with
// C % 4 == 0, G <= 64, 16-byte aligned y, at least three slots) and sizes the launch and
// its scratch.
struct GnSweepPlan {
    int grid = 0, PB = 0, R = 0, threads = 0;
    size_t smem = 0, scratch_bytes = 0;
};
bool gn_sweep_plan(const DeviceInfo& dev, const float* y, int64_t N, int64_t C, int64_t HW, int64_t G,
                   GnSweepPlan* plan);
cudaError_t launch_gn_sweep(const DeviceInfo& dev, const float* y, const float* gamma, const float* beta, float* out,
                            int64_t N, int64_t C, int64_t HW, int64_t G, float eps, const GnSweepPlan& plan,
                            void* scratch, cudaStream_t stream);

// Form 3 with y read once: each sample split by pixels over a group of CTAs that
// keep their slices in shared memory and exchange per-group partial statistics
// through global slots (the channel lse only).  gn_slab_plan says whether it
// applies (HW % 4 == 0, 16-byte aligned y and out, C <= 256, G <= 64, a slice of
// two buffers fits) and sizes the launch and its scratch.
struct GnSlabPlan {
    int GS = 0, P = 0, NB = 0, groups = 0;
    size_t smem = 0, scratch_bytes = 0;
};
bool gn_slab_plan(const DeviceInfo& dev, const float* y, const float* out, int64_t N, int64_t C, int64_t HW,
                  int64_t G, GnSlabPlan* plan);
cudaError_t launch_gn_slab(const DeviceInfo& dev, const float* y, const float* gamma, const float* beta, float* out,
                           int64_t N, int64_t C, int64_t HW, int64_t G, float eps, const GnSlabPlan& plan,
                           void* scratch, cudaStream_t stream);

// Conv2d 3 x 3, stride 1, valid, with bias, on the tensor cores (3xTF32):
// x [N, cin, H, W] -> y [N, cout, H - 2, W - 2].  Shapes conv_tc_supported()
// accepts: 1 <= cin <= 8, cout a multiple of 16 up to 128, W <= 1024.
bool conv_tc_supported(int64_t cin, int64_t cout, int64_t W);
cudaError_t launch_conv2d_3x3(const DeviceInfo& dev, const float* x, const float* w, const float* b, float* y,
                              int64_t N, int64_t cin, int64_t H, int64_t W, int64_t cout, cudaStream_t stream);

// The chain from the convolution's input: the conv kernel writes y and, per
// 128-pixel tile, the Welford partial of each of the G channel groups; a merge
// kernel reduces them to per-(n, g) stats; launch_gn_apply finishes.  Scratch:
// conv_chain_scratch_bytes(...), y included.
size_t conv_chain_scratch_bytes(int64_t N, int64_t H, int64_t W, int64_t cout, int64_t G);
cudaError_t launch_conv_gn_act_lse(const DeviceInfo& dev, const float* x, const float* w, const float* b,
                                   const float* gamma, const float* beta, float* out, int64_t N, int64_t cin,
                                   int64_t H, int64_t W, int64_t cout, int64_t G, float eps, void* scratch,
                                   cudaStream_t stream);

// Largest C that the apply kernel's shared-memory table holds.
constexpr int64_t kGnMaxChannels = 8192;

// Host-side argument checks of the GroupNorm entry points (sizes, overflow, eps,
// NULL, alignment), before any CUDA call; *empty is set when the output has no
// elements (LSE_OK, nothing to launch).
lse_status_t check_gn(const float* y, const float* gamma, const float* beta, const float* out, int64_t N,
                      int64_t C, int64_t HW, int64_t G, float eps, bool* empty);

// Reads an integer tuning knob from the environment (default when unset).
int env_int(const char* name, int dflt);

// Stores `e` as the calling thread's lse_last_cuda_error() value.
void record_cuda_error(cudaError_t e);

}  // namespace lse
