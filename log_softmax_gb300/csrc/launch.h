// Internal launchers of the logsumexp kernels (host side, C++ linkage).
// lse_api.cu validates arguments and picks a variant; these only launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace lse {

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int max_smem_optin = 0;   // bytes of dynamic shared memory a block may opt in to
    int* status = nullptr;    // device address of the library's status word
};

// Form 1: out[o, i] = lse over r of x[o, r, i] (inner > 1).
cudaError_t launch_lse_strided(const DeviceInfo& dev, const float* x, float* out, int64_t outer,
                               int64_t R, int64_t inner, cudaStream_t stream);

// Form 2, rows held in registers (cols up to kRegRowMaxCols).  mode 0 writes
// log_softmax into out (rows x cols); mode 1 writes the row lse into out (rows).
constexpr int64_t kRegRowMaxCols = 32768;
cudaError_t launch_rows_reg(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                            int64_t cols, int mode, cudaStream_t stream);

// Form 2, rows staged in the shared memory of a thread-block cluster (one bulk
// read of x).  Returns cudaErrorNotSupported when the row cannot be staged.
cudaError_t launch_lsm_smem_cluster(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                                    int64_t cols, cudaStream_t stream);

// Form 2, any row length: each CTA of a cluster streams its slice of the row
// (stats pass, then for mode 0 an apply pass).  mode as for launch_rows_reg.
cudaError_t launch_rows_stream(const DeviceInfo& dev, const float* x, float* out, int64_t rows,
                               int64_t cols, int mode, cudaStream_t stream);

// Form 3: per-(n, g) statistics into `stats` (2 * N * G floats), then the fused
// normalise / tanh / hardswish / residual / channel-lse pass.
cudaError_t launch_gn_act_lse(const DeviceInfo& dev, const float* y, const float* gamma,
                              const float* beta, float* out, int64_t N, int64_t C, int64_t HW,
                              int64_t G, float eps, float* stats, cudaStream_t stream);

// Largest C that the apply kernel's shared-memory table holds.
constexpr int64_t kGnMaxChannels = 8192;

// Reads an integer tuning knob from the environment (default when unset).
int env_int(const char* name, int dflt);

// Stores `e` as the calling thread's lse_last_cuda_error() value.
void record_cuda_error(cudaError_t e);

}  // namespace lse
