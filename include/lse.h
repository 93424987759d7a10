/*
 * lse.h — C ABI of the GB300 (sm_103a) logsumexp library, liblse.so.
 *
 * One operation in three forms: the numerically stable log-sum-exp
 * reduction  lse(x) = max(x) + log(sum(exp(x - max(x))))  along one axis of an
 * fp32 tensor.  Definitions follow three web pages on the POPCORNBENCH site:
 *   - "FW-GLM-5-1 / l1_p29": torch.logsumexp(x, dim=0) of an (R, B, D) tensor,
 *     task analysis (max, then log of the sum of shifted exponentials);
 *   - "Kimi-K2.6 / l1_p24": LogSoftmax over dim 1 of a (4096, 393216) tensor,
 *     opening analysis (x_i - max - log sum exp(x_j - max)) and its
 *     online-softmax derivation (running max with a rescaled running sum,
 *     merged pairwise);
 *   - "Kimi-K2.6 / l2_p92": Conv2d -> GroupNorm -> Tanh -> HardSwish ->
 *     residual add -> LogSumExp over channels; the GroupNorm discussion
 *     (per-sample, per-group mean and population variance over C/G channels
 *     and H*W, (x - mean)/sqrt(var + eps), per-channel affine weight and bias)
 *     and the HardSwish definition t * min(max(t + 3, 0), 6) / 6.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers to caller-owned memory, fp32,
 *     contiguous (row-major, last index fastest).  The library never frees or
 *     keeps them.  Inputs and outputs must not overlap.
 *   - Work is enqueued asynchronously on `stream` (0 = the legacy default
 *     stream).  A return of LSE_OK means the launch was enqueued; kernel-time
 *     faults surface on the next synchronising CUDA call, as usual.
 *   - Argument errors are detected on the host before any launch and return a
 *     status; nothing is enqueued then.  The library never aborts or traps.
 *   - A call whose output has no elements returns LSE_OK and launches nothing.
 *   - Pointers need 4-byte alignment.  16-byte alignment (and a row length that
 *     keeps rows 16-byte aligned) selects the vectorised / bulk-copy kernels;
 *     otherwise a scalar kernel runs with the same results.
 *   - Special values: a NaN in the reduced set gives NaN; else a +inf gives
 *     +inf; else a set that is all -inf gives -inf; -inf entries among finite
 *     ones contribute nothing.  log_softmax is x - lse in IEEE arithmetic, so
 *     a row holding +inf gives NaN at the +inf and -inf elsewhere, and an
 *     all -inf row gives NaN throughout.
 *   - Accuracy: fp32 storage and accumulation; results agree with a double
 *     precision evaluation within |err| <= 2e-5 + 1e-6 * |ref|.
 *   - CUDA graphs: every entry point on device pointers can be captured into
 *     a graph once the same call (same entry point, sizes and alignment) has
 *     run on the device outside a capture: first calls create the library's
 *     memory pool and load kernels, which must not happen inside a capture.
 *     Scratch then becomes graph memory nodes, so replays are independent.
 *     log_softmax_lastdim_host (its own copy streams) and lse_device_status
 *     (it synchronises) are not capturable.
 *
 * Environment switches (read at each call; none is needed, every default is
 * the measured best on GB300, and every setting gives the same results within
 * the tolerance above):
 *   - Kernel choice: LSE_LSM_VARIANT (rows: 1 registers, 2 cluster shared
 *     memory, 3 streaming, 4 lock-step group, 5 group with an L2 re-read,
 *     6 warp-specialised group with whole-slice shared-memory buffers, 7 the
 *     same with a ring of chunk slots, 8 the same with the rows parked in
 *     tensor memory; default by shape: 1 up to 32768 columns, else 8, else 6,
 *     else 3), LSE_GN_VARIANT (GroupNorm
 *     forms: 1 statistics kernel then apply kernel (gn_act_lse only), 2 work
 *     queue with per-thread loads, 3 work queue with bulk-copy staging, 4 sample
 *     slices held in shared memory by groups of CTAs, y read once (gn_act_lse
 *     only, HW % 4 == 0, C <= 256, G <= 64; falls back otherwise), 5 a queue
 *     of 256-pixel tiles parked in tensor memory, y read once (gn_act_lse
 *     only, HW % 4 == 0, C % 4 == 0, C <= 64; falls back otherwise), 6 the
 *     (sample, group) slabs as rows parked in tensor memory (group_norm and
 *     gn_act_residual, HW % 4 == 0 and 16-byte aligned y and out), 7 the
 *     whole grid on one sample at a time, each CTA a pixel slice of all
 *     channels in shared memory, y read once (gn_act_lse only, HW % 4 == 0
 *     with slices of at most 256 pixels, C % 4 == 0, C <= 64, G <= 64; falls
 *     back otherwise); default 2 for gn_act_lse, 6 (else 3) for group_norm
 *     and gn_act_residual),
 *     LSE_CONV_CHAIN (conv_gn_act_lse: 1 y and its tiles' statistics from
 *     the convolution's epilogue, then merge and apply; 2 y never in memory;
 *     3 y, then the GroupNorm work queue over it; default 3), LSE_CONV_TMA
 *     (0: convolution windows loaded directly),
 *     LSE_STRIDED_ONE_WALK (0: the strided log_softmax always walks a tile
 *     twice).
 *   - Tuning: LSE_WS_GROUP / LSE_WS_NB / LSE_WS_FW / LSE_WS_SW (warp-
 *     specialised rows: CTAs per row, buffers, fold and store warps;
 *     LSE_WS_GROUP also for 7 and 8), LSE_RING_CHUNK / LSE_TMEM_CHUNK (floats
 *     per landing chunk of 7 and 8),
 *     LSE_LSM_CLUSTER / LSE_LSM_GROUP / LSE_LSM_THREADS / LSE_LSM_NBUF /
 *     LSE_LSM_CHUNK, LSE_L2_GROUP / LSE_L2_THREADS, LSE_STREAM_CLUSTER (the
 *     other row kernels), LSE_GN_THREADS / LSE_GN_PARTS / LSE_GN_LAG /
 *     LSE_GN_CTAS_PER_SM and LSE_GNT_SLOTS / LSE_GNT_LAG / LSE_GNT_CTAS_PER_SM
 *     (the two GroupNorm work queues), LSE_SLAB_GROUP / LSE_SLAB_NB (CTAs per
 *     sample and slice buffers of the sample-slice kernel), LSE_GNM_SLOTS
 *     (landing slots of the tensor-memory tile queue), LSE_GNS_SLOTS (slots
 *     of the whole-grid sweep, 3 or more), LSE_CONV_WS (0: the convolution's
 *     tile-slot kernel instead of the pipelined one), LSE_GNR_GROUP /
 *     LSE_GNR_CHUNK / LSE_GNR_SW (CTAs per slab, floats per landing chunk,
 *     store warps 4 or 8 of the slab rows), LSE_HOST_CHUNK_MB (host pipeline
 *     chunk).
 *   - LSE_VERBOSE=1 prints each launch's plan on stderr.
 *   - Test hooks, not for production: LSE_TEST_FAIL_ALLOC=1 makes every
 *     scratch allocation fail (the call returns LSE_ERR_CUDA and enqueues
 *     nothing); LSE_TEST_UNREACHABLE_WAIT=1 makes the GroupNorm work queue
 *     wait for a statistics part that never comes, so its bounded waits run
 *     out (~1 s) and lse_device_status reports LSE_ERR_TIMEOUT.
 */
#ifndef LSE_H
#define LSE_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LSE_OK = 0,
    LSE_ERR_NULL = 1,        /* a required pointer is NULL                                  */
    LSE_ERR_SIZE = 2,        /* a size is negative, zero where it must not be, inconsistent, */
                             /* or too large (element counts must fit in int64)             */
    LSE_ERR_ALIGN = 3,       /* a pointer is not 4-byte aligned                             */
    LSE_ERR_CUDA = 4,        /* a CUDA call failed; lse_last_cuda_error() has the code      */
    LSE_ERR_UNSUPPORTED = 5, /* the device cannot run the kernel (not sm_103a, no clusters) */
    LSE_ERR_VALUE = 6,       /* a scalar argument is out of range (e.g. eps < 0 or NaN)     */
    LSE_ERR_TIMEOUT = 7      /* a kernel gave up waiting on a bulk copy (device status)     */
} lse_status_t;

/*
 * lse_reduce — logsumexp over the middle axis of a contiguous (outer, R, inner)
 * tensor:   out[o, i] = lse over r of x[o, r, i].
 * The reduced axis has stride `inner` elements; logsumexp(x, dim=d) of any
 * contiguous tensor is this call with outer = prod(shape[:d]), R = shape[d],
 * inner = prod(shape[d+1:]).  The dim-0 form of "FW-GLM-5-1 / l1_p29" is
 * outer = 1, R, inner = B*D.
 *   x     [outer * R * inner] fp32, device, read only.
 *   out   [outer * inner]     fp32, device, written.
 *   outer >= 0, inner >= 0; R >= 1 when outer * inner > 0 (R = 0 would be the
 *   empty-set value -inf, which this call rejects with LSE_ERR_SIZE).
 */
lse_status_t lse_reduce(const float* x, float* out, int64_t outer, int64_t R, int64_t inner,
                        cudaStream_t stream);

/*
 * log_softmax_lastdim — row-wise log_softmax of a contiguous (rows, cols) tensor
 * ("Kimi-K2.6 / l1_p24"):   out[r, j] = x[r, j] - lse over k of x[r, k].
 *   x    [rows * cols] fp32, device, read only.
 *   out  [rows * cols] fp32, device, written (must not alias x).
 *   rows >= 0, cols >= 0.
 * Rows up to a few MB are staged on chip (registers, or shared memory of a
 * thread-block cluster) so that x is read from HBM once.
 */
lse_status_t log_softmax_lastdim(const float* x, float* out, int64_t rows, int64_t cols,
                                 cudaStream_t stream);

/*
 * log_softmax_lastdim_host — log_softmax_lastdim on HOST buffers: x and out are
 * host pointers (page-locked memory lets the copies run asynchronously and
 * overlap; pageable memory works, with staged copies).  Rows are processed in
 * chunks of about 256 MB (LSE_HOST_CHUNK_MB) through three device staging
 * buffers from the library's pool: the copy in of one chunk, the computation of
 * the previous one and the copy out of the one before overlap, on two copy
 * streams the library owns, ordered after the work already queued on `stream`.
 * `stream` resumes after the last copy out, so out is complete once `stream`
 * is; the host must keep both buffers alive and untouched until then.  Calls
 * on one device enqueue one at a time.  Same argument rules as
 * log_softmax_lastdim (sizes, 4-byte alignment, NULL).
 */
lse_status_t log_softmax_lastdim_host(const float* x, float* out, int64_t rows, int64_t cols,
                                      cudaStream_t stream);

/*
 * softmax_lastdim — row-wise softmax of a contiguous (rows, cols) tensor, the
 * non-log variant that "Kimi-K2.6 / l1_p24" describes beside log_softmax (in
 * its discussion of how the write pass differs: exp(x - max) scaled by 1/sum):
 *     out[r, j] = exp(x[r, j] - lse over k of x[r, k]),
 * which equals exp(x - max) / sum up to rounding.  It is exp of
 * log_softmax_lastdim's result, special values included: a row holding NaN,
 * +inf, or only -inf gives NaN where log_softmax does, and 0 where log_softmax
 * gives -inf.  Same arguments, layout, staging and rules as
 * log_softmax_lastdim.  Accuracy: |err| <= 2e-5 + 1e-6 * |ref|.
 */
lse_status_t softmax_lastdim(const float* x, float* out, int64_t rows, int64_t cols,
                             cudaStream_t stream);

/*
 * log_softmax_dim — log_softmax over the middle axis of a contiguous
 * (outer, R, inner) tensor, the log_softmax identity of "Kimi-K2.6 / l1_p24"
 * (opening analysis) along an axis of stride `inner`:
 *     out[o, r, i] = x[o, r, i] - lse over r' of x[o, r', i].
 * log_softmax(x, dim=d) of any contiguous tensor is this call with
 * outer = prod(shape[:d]), R = shape[d], inner = prod(shape[d+1:]); inner = 1
 * is log_softmax_lastdim.  For inner > 1 one kernel computes the lse of a tile
 * of columns (the reduction of lse_reduce) and then writes the tile, whose
 * second read is served from L2 while the tiles in flight fit there.
 *   x    [outer * R * inner] fp32, device, read only.
 *   out  [outer * R * inner] fp32, device, written (must not alias x).
 *   outer, R, inner >= 0.
 */
lse_status_t log_softmax_dim(const float* x, float* out, int64_t outer, int64_t R, int64_t inner,
                             cudaStream_t stream);

/*
 * group_norm — GroupNorm forward alone, materialised ("Kimi-K2.6 / l2_p92",
 * GroupNorm discussion), the first step of gn_act_lse's chain:
 *   out[n,c,p] = (y[n,c,p] - mean[n,g]) / sqrt(var[n,g] + eps) * gamma[c] + beta[c]
 * with mean and population variance over the C/G channels of group g of
 * sample n and all HW positions.
 *   y      [N * C * HW] fp32 NCHW, device, read only.
 *   gamma  [C], beta [C] fp32, device, read only.
 *   out    [N * C * HW] fp32, device, written (must not alias y).
 *   N >= 0, HW >= 0, 1 <= C <= 8192, G >= 1, C % G == 0; eps >= 0 and finite.
 * One cooperative kernel.  Where HW % 4 == 0 and y and out are 16-byte
 * aligned, each (sample, group) slab (C/G x HW contiguous floats) is a row
 * split over a few CTAs: read once into tensor memory, its mean and M2 merged
 * across the CTAs, then written normalised; otherwise a work queue computes a
 * sample's statistics, then its output from a second read served by L2.
 * Scratch and error rules as gn_act_lse.
 */
lse_status_t group_norm(const float* y, const float* gamma, const float* beta, float* out,
                        int64_t N, int64_t C, int64_t HW, int64_t G, float eps,
                        cudaStream_t stream);

/*
 * gn_act_residual — gn_act_lse's chain without the final reduction
 * ("Kimi-K2.6 / l2_p92"): out[n,c,p] = y[n,c,p] + hardswish(tanh(z[n,c,p])),
 * z the group_norm output.  Arguments, sizes and rules as group_norm.
 */
lse_status_t gn_act_residual(const float* y, const float* gamma, const float* beta, float* out,
                             int64_t N, int64_t C, int64_t HW, int64_t G, float eps,
                             cudaStream_t stream);

/*
 * conv2d_3x3 — the Conv2d that produces the chain's input in "Kimi-K2.6 / l2_p92"
 * (its model: Conv2d(8, 64, kernel_size=3), stride 1, no padding, with bias):
 *   y[n,co,i,j] = b[co] + sum over ci, u, v of w[co,ci,u,v] * x[n,ci,i+u,j+v]
 *   x  [N * Cin * H * W] fp32 NCHW, device, read only.
 *   w  [Cout * Cin * 3 * 3] fp32, device, read only;  b [Cout] fp32, device.
 *   y  [N * Cout * (H-2) * (W-2)] fp32, device, written (must not alias x).
 *   N >= 0, H >= 3, W >= 3; 1 <= Cin <= 8, Cout a multiple of 16 up to 128 and
 *   W <= 1024 (else LSE_ERR_UNSUPPORTED).
 * Computed on the tensor cores as nine shifted GEMMs (one per kernel tap) per
 * tile of 128 output pixels, from one staged window of the input, with every
 * operand split into two tf32 parts (three products per pair), which keeps
 * fp32 accuracy: |err| <= 2e-5 + 1e-6 * |ref| against a double evaluation for
 * data of unit scale.
 */
lse_status_t conv2d_3x3(const float* x, const float* w, const float* b, float* y, int64_t N, int64_t Cin,
                        int64_t H, int64_t W, int64_t Cout, cudaStream_t stream);

/*
 * conv_gn_act_lse — the whole chain of "Kimi-K2.6 / l2_p92" from the
 * convolution's input: y = conv2d_3x3(x, w, b), then gn_act_lse(y, ...):
 *   out[n,p] = lse over c of ( y + hardswish(tanh(GroupNorm(y))) )[n,c,p]
 *   x, w, b as conv2d_3x3; gamma, beta [Cout]; out [N * (H-2) * (W-2)] fp32,
 *   device, written.  Cin = 8 (the page's layer), Cout % G == 0 with Cout / G
 *   in {1, 2, 4, 8, 16} and G <= 64 (else LSE_ERR_UNSUPPORTED); eps >= 0 and
 *   finite; the
 *   conv2d_3x3 shape rules.  Other shapes: conv2d_3x3 then gn_act_lse.
 * The convolution writes y, then gn_act_lse's one-kernel work queue runs over
 * it, walking the samples last to first so that its first reads find the
 * convolution's last samples in L2.  Scratch (y itself, about
 * N*Cout*(H-2)*(W-2)*4 bytes, plus statistics) comes from the library's pool
 * on `stream`.  (LSE_CONV_CHAIN=1 has the convolution's epilogue compute each
 * tile's group statistics instead, merged before one apply pass over y;
 * LSE_CONV_CHAIN=2 keeps y out of memory: the convolution runs twice and the
 * second pass finishes the chain from the tensor-core accumulators.  Both
 * measured slower on GB300.)
 */
lse_status_t conv_gn_act_lse(const float* x, const float* w, const float* b, const float* gamma,
                             const float* beta, float* out, int64_t N, int64_t Cin, int64_t H, int64_t W,
                             int64_t Cout, int64_t G, float eps, cudaStream_t stream);

/*
 * gn_act_lse — GroupNorm -> tanh -> hardswish -> residual add -> logsumexp over
 * channels, keepdim ("Kimi-K2.6 / l2_p92", the chain after its Conv2d):
 *   mean[n,g], var[n,g] : population statistics of the C/G channels of group g
 *                         of sample n over all HW positions;
 *   z   = (y[n,c,p] - mean[n,g]) / sqrt(var[n,g] + eps) * gamma[c] + beta[c]
 *   r   = y[n,c,p] + hardswish(tanh(z)),  hardswish(t) = t*min(max(t+3,0),6)/6
 *   out[n,p] = lse over c of r          (out is [N, 1, H, W] with HW = H*W)
 *   y      [N * C * HW] fp32 NCHW, device, read only.
 *   gamma  [C], beta [C] fp32, device, read only.
 *   out    [N * HW] fp32, device, written.
 *   N >= 0, HW >= 0, 1 <= C <= 8192, G >= 1, C % G == 0; eps >= 0 and finite.
 *   - Special values: a NaN, +inf or -inf anywhere in a group makes that
 *     group's mean or variance NaN, hence every z of the group NaN; since the
 *     lse spans all channels, the whole sample's output is then NaN (the
 *     statistics are taken over all of the group's values, as defined above).
 *     group_norm and gn_act_residual give NaN for exactly that group.
 * The per-(n, g) statistics and a work counter need 16*N*G + 4*N + 32 bytes of
 * scratch.  The library takes them, stream-ordered, from a memory pool it owns
 * on the current device
 * (cudaMallocFromPoolAsync / cudaFreeAsync on `stream`), so concurrent calls on
 * different streams never share scratch.  lse_release_workspace() returns the
 * pool's idle memory to the device.
 */
lse_status_t gn_act_lse(const float* y, const float* gamma, const float* beta, float* out,
                        int64_t N, int64_t C, int64_t HW, int64_t G, float eps,
                        cudaStream_t stream);

/*
 * gn_act_lse_noalloc — gn_act_lse's result and arguments, for callers that must
 * not allocate device memory: a plugin or engine whose host framework has
 * reserved all device memory and forbids its components to allocate, or a
 * latency-critical path that cannot take an allocation's cost or its
 * out-of-memory failure mid-step.  (The pages have no counterpart: it is a
 * deployment variant of gn_act_lse.)
 *   - It runs the two-kernel path (a statistics kernel, then the apply kernel:
 *     what LSE_GN_VARIANT=1 selects for gn_act_lse), which reads y twice from
 *     HBM where gn_act_lse's default one-kernel work queue serves most of the
 *     second read from L2: on y[128, 64, 126, 126] about 0.179 ms against
 *     0.159 ms on GB300.  Results agree with gn_act_lse's within the tolerance
 *     above, not bit for bit (the statistics are merged in another order).
 *   - Allocates nothing: the 2*N*G floats of statistics live in a fixed array
 *     compiled into the library (512 KiB, N*G <= 65536), which every GPU that
 *     loads the library holds until the process exits.  gn_act_lse's argument
 *     rules are checked first (same status codes); then N*G > 65536 returns
 *     LSE_ERR_SIZE.
 *   - The first call on a device does a one-time set-up on that device (it looks
 *     up the array's device address with cudaGetSymbolAddress); make that first
 *     call before any stream capture.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents.  Each call overwrites every entry it reads, so nothing needs
 *     clearing, but calls whose kernels may overlap on the GPU (different streams
 *     without ordering) race on it: order them.
 */
lse_status_t gn_act_lse_noalloc(const float* y, const float* gamma, const float* beta, float* out,
                                int64_t N, int64_t C, int64_t HW, int64_t G, float eps,
                                cudaStream_t stream);

/* Returns the idle memory of the library's scratch pools to the device. */
lse_status_t lse_release_workspace(void);

/*
 * Synchronises `stream`, then reads and clears the library's device-side
 * status on the current device: LSE_OK, or LSE_ERR_TIMEOUT when a kernel gave
 * up waiting on a bulk copy (its outputs are then unspecified).  Bounded waits
 * end after about one second; nothing in the library waits without a limit.
 */
lse_status_t lse_device_status(cudaStream_t stream);

/* A static, human-readable name for a status code. */
const char* lse_status_string(lse_status_t status);

/* The cudaError_t of the most recent LSE_ERR_CUDA on the calling thread (0 if none). */
int lse_last_cuda_error(void);

/* Library version, as major * 10000 + minor * 100 + patch. */
int lse_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LSE_H */
