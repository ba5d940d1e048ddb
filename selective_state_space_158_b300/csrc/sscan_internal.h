// sscan_internal.h -- interfaces between the C ABI layer (sscan_api.cu) and the kernel
// launchers (sscan_kernels.cu). Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sscan {

enum class Io { F32 = 0, BF16 = 1 };

// Everything a launcher needs: caller pointers and sizes, already validated.
struct FwdArgs {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;       // nullable
  const void* z;        // nullable
  const float* bias;    // nullable
  int softplus;
  const float* h0 = nullptr;  // initial state (batch, dim, N) fp32, nullable
  int euler = 0;              // decay factor 1 + dt A instead of exp(dt A)
  void* y;
  float* h_last;        // nullable
  float* h_ckpt = nullptr;  // backward pass: state before every 16-step chunk, nullable
  int64_t batch, L, dim, N;
  Io io;
  cudaStream_t stream;
  unsigned int* status;  // device status word (SSCAN_ERR_* bit set on device-side errors)
  // Optional caller-provided chunk-carry scratch. When null the launcher takes stream-ordered
  // scratch with cudaMallocAsync; when set it uses this buffer and allocates nothing, failing
  // with *scratch_short = true if the launch would need more than scratch_bytes.
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  bool* scratch_short = nullptr;
};

// Layout overrides (sscan_set_tuning, include/sscan_tuning.h). Zero fields mean "choose
// automatically"; skip_publish -1 means the fault-injection hook is off.
struct Tuning {
  int states_per_lane = 0;    // K: states of one channel a lane holds (4, 8 or 16)
  int segments = 0;           // time segments run by different CTAs (chunk carry)
  int threads = 0;            // threads per CTA (multiple of 32, <= 256)
  int stages = 0;             // TMA pipeline depth
  int chunk = 0;              // steps per chunk with four lanes per channel (16 or 32)
  int force_plain = 0;        // forward: plain-load kernel only
  int bwd_segments = 0;       // backward: time segments
  int conv_plain = 0;         // Conv1d: register-window kernel only
  int ctas_per_sm = 0;        // forward: cap on resident CTAs per SM (0: no cap)
  int skip_publish = -1;      // test hook: this segment never publishes its aggregate
  int time_scan = 0;          // forward: 1 time-lane kernel, 2 never, 0 automatic
};

// The setting sscan_set_tuning installed (a copy, taken under the setting's lock).
Tuning current_tuning();

// Size checks shared by the C entry points; fills the element counts (batch*L*dim, batch*L*N).
int check_fwd_args(const void* u, const void* delta, const float* A, const void* B,
                   const void* C, const void* y, int64_t batch, int64_t L, int64_t dim,
                   int64_t N, int dtype, int64_t* n_bld, int64_t* n_bln);

// Status word of the allocation-free entry point on device `dev` (null before its first call).
unsigned int* noalloc_status_word(int dev);

// A 3-D tiled TMA map over a dense (d2, d1, d0) tensor of io elements (d0 fastest) with box
// (b0, b1, 1); false if the driver entry point is missing or rejects the map.
bool make_tensor_map_3d(CUtensorMap* m, const void* ptr, Io io, uint64_t d0, uint64_t d1,
                        uint64_t d2, uint32_t b0, uint32_t b1);

// True if the TMA-staged kernel can serve these arguments (alignment and stride rules of TMA).
bool tma_path_ok(const FwdArgs& a);

// Launchers. Return cudaSuccess or the launch error.
cudaError_t launch_simple(const FwdArgs& a);
cudaError_t launch_tma(const FwdArgs& a, const Tuning& t);
cudaError_t launch_lane(const FwdArgs& a, const Tuning& t);
// The TMA-staged kernel when the arguments (and the tuning) allow it, else the plain-load one.
cudaError_t launch_forward(const FwdArgs& a);
// One step of the recurrence for every (batch, channel); h_last is the state, read and written.
cudaError_t launch_step(const FwdArgs& a);
// y = 2^x element-wise with the accurate exponential (exp2_acc).
cudaError_t launch_exp2_accurate(const float* x, float* y, int64_t n, cudaStream_t stream);

// Causal depthwise convolution over time + SiLU (sscan_conv1d_silu), arguments validated.
struct ConvArgs {
  const void* x;       // (batch, L, dim) io
  const float* w;      // (dim, width) fp32
  const float* bias;   // (dim) fp32, nullable
  const void* x_prev;  // (batch, width - 1, dim) io, nullable
  int silu;
  void* y;             // (batch, L, dim) io
  int64_t batch, L, dim, width;
  Io io;
  cudaStream_t stream;
  unsigned int* status = nullptr;  // device status word (bounded-wait timeouts), nullable
};
cudaError_t launch_conv(const ConvArgs& a);

// Backward pass (sscan_bwd), arguments validated.
struct BwdArgs {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;       // nullable
  const void* z;        // nullable
  const float* bias;    // nullable
  int softplus;
  const float* h0;      // nullable
  int euler;
  const void* dy;       // (batch, L, dim) io
  const float* dh_last; // nullable
  const float* ckpt;    // state before every 16-step chunk [n_chunks][batch][dim][N]
  void* du;             // (batch, L, dim) io
  void* ddelta;         // (batch, L, dim) io
  float* dA;            // (dim, N)
  float* dB;            // (batch, L, N)
  float* dC;            // (batch, L, N)
  float* dD;            // (dim), required when D is given
  void* dz;             // (batch, L, dim) io, required when z is given
  float* dbias;         // (dim), required when bias is given
  float* dh0;           // (batch, dim, N), nullable
  int64_t batch, L, dim, N;
  Io io;
  cudaStream_t stream;
};
cudaError_t launch_bwd(const BwdArgs& a);

}  // namespace sscan
