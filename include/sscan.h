/*
 * sscan.h -- C ABI of libsscan, the S6 selective-scan forward on NVIDIA B300 (sm_103a).
 *
 * The operation (pages cited by title and section):
 *   "Mamba：选择性状态空间模型入门教程", section "Mamba 的关键创新：选择性机制" (selective scan
 *   pseudo-code); "Mamba: Linear-Time Sequence Modeling with Selective State Spaces" (wiki notes),
 *   section "核心贡献：选择机制（S6）" (B_t, C_t of shape (B, L, N), Delta_t = tau(Delta + s(x_t)));
 *   "架构变体：Mamba/SSM", sections "离散化" (zero-order hold) and "硬件感知算法" (one fused scan,
 *   state kept on chip).
 *
 * For every batch row b, channel d and step t = 0 .. L-1, with h[b,d,:] = 0 before t = 0:
 *   dt          = softplus_flag ? log(1 + exp(delta[b,t,d] + bias[d])) : delta[b,t,d] + bias[d]
 *   h[b,d,n]    = exp(dt * A[d,n]) * h[b,d,n] + dt * B[b,t,n] * u[b,t,d]      (n = 0 .. N-1)
 *   y[b,t,d]    = sum_n C[b,t,n] * h[b,d,n] + D[d] * u[b,t,d]
 *   y[b,t,d]   *= z[b,t,d] / (1 + exp(-z[b,t,d]))                             (only if z given)
 *   h_last[b,d,n] = h[b,d,n] after step L-1
 * State and arithmetic are fp32; inputs and y are fp32 or bf16 (dtype).
 */
#ifndef SSCAN_H
#define SSCAN_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SSCAN_F32 = 0, SSCAN_BF16 = 1 } sscan_dtype_t;

/* Decay factor of one step. ZOH: exp(dt * A), the zero-order hold of "架构变体：Mamba/SSM",
 * section "离散化". EULER: 1 + dt * A, the first-order expansion of exp(dt * A) (section 3.2 of
 * "从RNN到Mamba：深入浅出图解'选择性状态空间'如何让模型学会'忘记'" prints it as (I - Delta A),
 * which grows without bound for A < 0; the sign is read as +). EULER is stable for dt |A| < 2. */
typedef enum { SSCAN_DISC_ZOH = 0, SSCAN_DISC_EULER = 1 } sscan_disc_t;

typedef enum {
  SSCAN_OK = 0,
  SSCAN_ERR_INVALID_ARG = 1,   /* null required pointer, negative size, N outside 1..16, ... */
  SSCAN_ERR_UNSUPPORTED = 2,   /* reserved: no entry point of this version returns it */
  SSCAN_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
  SSCAN_ERR_CARRY_TIMEOUT = 4, /* device side: a bounded wait (pipeline or chunk carry) ran out */
  SSCAN_ERR_SCRATCH_TOO_SMALL = 5 /* sscan_fwd_noalloc: the call needs more scratch than the
                                     library's fixed buffer holds */
} sscan_status_t;

/*
 * sscan_fwd -- selective-scan forward on device memory, asynchronous on `stream`.
 *
 * Pointers (all device memory owned by the caller; the library keeps none after returning):
 *   u, delta, z : (batch, L, dim) row-major, dim fastest, element type `dtype`
 *   A           : (dim, N) fp32 (the continuous-time diagonal state matrix, normally < 0)
 *   B, C        : (batch, L, N) row-major, N fastest, element type `dtype` (shared over dim)
 *   D           : (dim) fp32 skip weights, or NULL for no skip term
 *   z           : gate input, or NULL for no SiLU gate
 *   delta_bias  : (dim) fp32, or NULL for a zero bias
 *   y           : (batch, L, dim) output, element type `dtype`; must not alias any input
 *   h_last      : (batch, dim, N) fp32 final state, or NULL if not wanted
 * softplus_flag != 0 applies softplus to delta + bias; 0 uses delta + bias as the step.
 * Sizes: batch, L, dim >= 0; 1 <= N <= 16. batch, L or dim = 0 is a no-op that returns
 * SSCAN_OK (h_last, if given, is zeroed when L = 0).
 * Any alignment and any dim are accepted; 16-byte aligned pointers with dim a multiple of 4
 * (fp32) or 8 (bf16) take the TMA-staged fast path, anything else a plain-load path.
 *
 * Errors: argument checks are synchronous and return SSCAN_ERR_INVALID_ARG before anything is
 * launched; launch failures return SSCAN_ERR_CUDA. A device-side carry timeout (possible only
 * when the library splits one sequence across thread blocks) is recorded in a per-device status
 * word that sscan_get_device_error reports.
 * Workspace: on the fast path the library takes a stream-ordered scratch allocation
 * (cudaMallocAsync on `stream`, freed stream-ordered) when it needs one: B and C widened to fp32
 * rows of 16 states (bf16 inputs or N < 16: 128 bytes per batch row and step) and, when a long
 * sequence is split across thread blocks, the chunk-carry flags and segment summaries.
 */
sscan_status_t sscan_fwd(const void* u, const void* delta, const float* A, const void* B,
                         const void* C, const float* D, const void* z, const float* delta_bias,
                         int softplus_flag, void* y, float* h_last, int64_t batch, int64_t L,
                         int64_t dim, int64_t N, sscan_dtype_t dtype, cudaStream_t stream);

/*
 * sscan_fwd_ex -- sscan_fwd from a given initial state, with a choice of decay factor.
 *
 * The recurrent (step-by-step) mode of the scan carries nothing but the state from one step to
 * the next ("Mamba：选择性状态空间模型入门教程", "Mamba 的关键创新：选择性机制"; "Mamba:
 * Linear-Time Sequence Modeling with Selective State Spaces", "核心贡献：选择机制（S6）"), so a
 * sequence can be processed in pieces: pass one call's h_last as the next call's h0.
 *
 *   h0   : (batch, dim, N) fp32 device memory, the state before step 0, or NULL for zero. It may
 *          be the same buffer as h_last: every thread block reads its part of h0 before any
 *          part of h_last is written, so a sequence can be continued in place.
 *   disc : SSCAN_DISC_ZOH (what sscan_fwd computes) or SSCAN_DISC_EULER.
 * Everything else is as for sscan_fwd; L = 0 copies h0 (or zero) to h_last. An out-of-range
 * disc returns SSCAN_ERR_INVALID_ARG.
 */
sscan_status_t sscan_fwd_ex(const void* u, const void* delta, const float* A, const void* B,
                            const void* C, const float* D, const void* z,
                            const float* delta_bias, int softplus_flag, const float* h0,
                            sscan_disc_t disc, void* y, float* h_last, int64_t batch, int64_t L,
                            int64_t dim, int64_t N, sscan_dtype_t dtype, cudaStream_t stream);

/*
 * sscan_step -- one step of the recurrence for every (batch, channel): recurrent inference
 * (decoding), constant work per token ("Mamba：选择性状态空间模型入门教程", recurrent mode at
 * inference time; "Mamba: Linear-Time Sequence Modeling with Selective State Spaces", constant
 * memory per generated token).
 *
 *   u, delta, z : (batch, dim) this step's inputs, element type `dtype` (z nullable)
 *   B, C        : (batch, N), element type `dtype`
 *   A (dim, N), D (dim), delta_bias (dim): fp32 as for sscan_fwd (D, delta_bias nullable)
 *   h           : (batch, dim, N) fp32 device state, read and overwritten with the new state
 *   y           : (batch, dim) output, element type `dtype`
 * Computes exactly one step of sscan_fwd_ex (same dt, decay factor, skip and gate), so a prefill
 * by sscan_fwd_ex followed by steps from its h_last continues the same sequence. Asynchronous
 * on `stream`; allocates nothing; argument errors as for sscan_fwd (h must not be NULL).
 */
sscan_status_t sscan_step(const void* u, const void* delta, const float* A, const void* B,
                          const void* C, const float* D, const void* z, const float* delta_bias,
                          int softplus_flag, sscan_disc_t disc, float* h, void* y, int64_t batch,
                          int64_t dim, int64_t N, sscan_dtype_t dtype, cudaStream_t stream);

/*
 * sscan_bwd -- backward pass of sscan_fwd_ex with recomputation: gradients of
 *     Loss = sum dy * y + sum dh_last * h_last
 * with respect to every input. The intermediate states are recomputed, not stored ("Mamba:
 * Linear-Time Sequence Modeling with Selective State Spaces" notes, "第二个创新：硬件感知算法",
 * item 3; "从RNN到Mamba" 3.3, item 2); the gradient is the adjoint recurrence of the defined
 * forward.
 *
 * Forward inputs (u .. disc) exactly as passed to sscan_fwd_ex. Then:
 *   dy          : (batch, L, dim) `dtype`, gradient of the loss with respect to y
 *   dh_last     : (batch, dim, N) fp32 gradient with respect to h_last, or NULL for zero
 * Outputs (device memory, overwritten):
 *   du, ddelta  : (batch, L, dim) `dtype`
 *   dA          : (dim, N) fp32          dB, dC: (batch, L, N) fp32
 *   dD          : (dim) fp32, required when D is given (else ignored)
 *   dz          : (batch, L, dim) `dtype`, required when z is given (else ignored)
 *   ddelta_bias : (dim) fp32, required when delta_bias is given (else ignored)
 *   dh0         : (batch, dim, N) fp32 gradient with respect to the initial state, or NULL
 * Parameter gradients (dA, dB, dC, dD, ddelta_bias) are sums over the other axes, reduced in a
 * fixed order: results are deterministic. Workspace: stream-ordered (cudaMallocAsync) state
 * checkpoints every 16 steps (batch * dim * N floats each), per-channel-group partial sums of
 * dB, dC, and, when the sequence is split into time segments (fewer batch rows x 32-channel
 * groups than SMs), per-segment partials and adjoint aggregates. Argument errors are
 * synchronous (SSCAN_ERR_INVALID_ARG); a bounded wait of the recomputing forward pass that runs
 * out is reported by sscan_get_device_error, as for sscan_fwd.
 */
sscan_status_t sscan_bwd(const void* u, const void* delta, const float* A, const void* B,
                         const void* C, const float* D, const void* z, const float* delta_bias,
                         int softplus_flag, const float* h0, sscan_disc_t disc, const void* dy,
                         const float* dh_last, void* du, void* ddelta, float* dA, float* dB,
                         float* dC, float* dD, void* dz, float* ddelta_bias, float* dh0,
                         int64_t batch, int64_t L, int64_t dim, int64_t N, sscan_dtype_t dtype,
                         cudaStream_t stream);

/*
 * sscan_conv1d_silu -- causal depthwise convolution over time followed by SiLU: the step that
 * turns the Mamba block's in-projection output into the scan's input u ("Mamba: Linear-Time
 * Sequence Modeling with Selective State Spaces" notes, "架构：极简设计": Linear -> Conv1d ->
 * SiLU). For every batch row b, channel d and step t, with W = width:
 *
 *   y[b,t,d] = SiLU(bias[d] + sum_{j=0}^{W-1} w[d,j] * x[b, t-(W-1)+j, d])   (SiLU if silu_flag)
 *
 * The pages give neither the width nor the tap order; the convolution is causal (no future
 * step enters) and depthwise (channels do not mix), and w[d, W-1] weighs the current step.
 *   x, y   : (batch, L, dim) device memory, element type `dtype`; y must not alias x
 *   w      : (dim, width) fp32;  bias: (dim) fp32 or NULL
 *   x_prev : (batch, width-1, dim) `dtype`, the width-1 inputs before t = 0 (oldest first), for
 *            continuing a streamed sequence; NULL means zeros
 * 1 <= width <= 64. Asynchronous on `stream`; allocates nothing; argument errors are synchronous
 * (SSCAN_ERR_INVALID_ARG), launch errors SSCAN_ERR_CUDA; a bounded wait of the tile pipeline
 * that runs out sets the status word that sscan_get_device_error reports.
 */
sscan_status_t sscan_conv1d_silu(const void* x, const float* w, const float* bias,
                                 const void* x_prev, int silu_flag, void* y, int64_t batch,
                                 int64_t L, int64_t dim, int64_t width, sscan_dtype_t dtype,
                                 cudaStream_t stream);

/*
 * sscan_fwd_host -- the same operation on HOST buffers: copies the inputs to the current
 * device, runs sscan_fwd, copies y and h_last back and synchronizes `stream`.
 * Arguments mean what they mean for sscan_fwd but every pointer is host memory (page-locked
 * memory gives asynchronous, overlapped copies). The batch is cut into up to 8 slices of whole
 * batch rows that rotate over three streams the library owns (ordered after the work already
 * on `stream`; `stream` waits for all of them), so one slice's copy in, another's scan and a
 * third's copy out overlap; each slice is an independent sscan_fwd over its rows. With fewer
 * than 8 batch rows and at least 32768 steps the sequence is cut into up to 16 time slices
 * instead (at least 16384 steps each), copied with strided 2-D copies, and each slice's scan
 * continues from the previous one's end state (sscan_fwd_ex, in place). Device staging
 * buffers and those streams are owned by the library per device, grown or created on demand and
 * kept until sscan_release(). Calls on one device are serialised inside the library. Returns when
 * y and h_last hold the result, or with the first error (after every copy it queued has ended).
 */
sscan_status_t sscan_fwd_host(const void* u, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const float* delta_bias, int softplus_flag, void* y, float* h_last,
                              int64_t batch, int64_t L, int64_t dim, int64_t N,
                              sscan_dtype_t dtype, cudaStream_t stream);

/*
 * sscan_fwd_noalloc -- sscan_fwd for callers that must not allocate device memory.
 *
 * This entry point has no counterpart in the pages; it exists for callers that cannot call
 * cudaMalloc (or cudaMallocAsync) at the point where they run the scan: code that runs while a
 * caching allocator or a framework owns all device memory, real-time paths that cannot afford an
 * allocation's possible synchronisation, or code whose memory budget is fixed up front.
 *
 * Arguments, layouts, results and errors are those of sscan_fwd; inputs and outputs are still
 * the caller's device buffers. The only difference is the scratch sscan_fwd allocates per call
 * (B and C widened to fp32, and the chunk-carry state of a sequence split across thread blocks):
 * here it lives in a fixed 16 MiB array in device memory that every GPU which loads the library
 * keeps until the process exits. A call that would need more than that (bf16 inputs or N < 16
 * with more than about 120,000 batch rows x steps, or very long sequences split into many
 * segments) returns SSCAN_ERR_SCRATCH_TOO_SMALL before launching anything; sscan_fwd serves it.
 *
 * - The first call on a device looks up that device's copy of the array (with the device
 *   current); make that first call before any stream capture.
 * - All calls share the array and it keeps the last call's contents; each call clears the parts
 *   that must start at zero on `stream`. Calls whose kernels overlap on the GPU (on different
 *   streams, or from different host threads) race on the array: serialise them.
 * - Device-side timeouts are recorded in a status word inside the array;
 *   sscan_get_device_error (which allocates nothing either) reports and clears it together
 *   with sscan_fwd's.
 * - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
sscan_status_t sscan_fwd_noalloc(const void* u, const void* delta, const float* A, const void* B,
                                 const void* C, const float* D, const void* z,
                                 const float* delta_bias, int softplus_flag, void* y,
                                 float* h_last, int64_t batch, int64_t L, int64_t dim,
                                 int64_t N, sscan_dtype_t dtype, cudaStream_t stream);

/* Synchronizes `stream`, then reads and clears the current device's status words (set by
 * kernels on a device-side error such as SSCAN_ERR_CARRY_TIMEOUT, by any entry point's
 * kernels: the scans, the step, the backward's recomputing forward, the convolution's tile
 * pipeline, or sscan_fwd_noalloc's). Allocates nothing. Returns SSCAN_OK if clear. */
sscan_status_t sscan_get_device_error(cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* sscan_status_string(sscan_status_t status);

/* Frees the library's per-device buffers (status word, host-path staging) on the current
 * device. Call only when no sscan work is in flight on that device. */
sscan_status_t sscan_release(void);

#ifdef __cplusplus
}
#endif

#endif /* SSCAN_H */
