// sscan_peaks.cu -- issue-rate microbenchmarks that give the compute rooflines of the scan their
// denominators on the machine at hand: how many SFU exponentials (ex2.approx.ftz.f32), scalar
// FFMAs and packed FFMA2s one SM completes per clock, alone and in the mix one state update of
// the scan issues (one arg FMA, one decay exponential, one input FMUL, one state FMA, one readout
// FMA); and the rate of the scan's step loop itself (operands from shared memory, states in
// registers) at a chosen number of warps per SM, the practical ceiling of kernels built around
// that loop. Built as its own small library (libsscan_peaks.so); the scan library does not use it.
//
// Method: 148 x k CTAs of 1024 threads, each holding 120 KB of (unused) dynamic shared memory so
// that exactly one CTA is resident per SM at a time; every thread runs
// `iters` loop trips over 8 independent dependency chains of the measured instruction(s), so that
// issue, not latency, bounds the loop. Thread 0 of every CTA reads %clock64 after a CTA barrier
// on entry and on exit; a CTA's rate is its operations / its cycles, reported per SM. Counting
// cycles on the SM makes the result independent of the clock frequency the GPU runs at.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ float ex2a(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float ffma_v(float a, float b, float c) {
  float d;
  asm volatile("fma.rn.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// kind 0: ex2 only; 1: FFMA only; 2: FFMA2 only; 3: the scan's per-update mix in packed form
// (per 2 updates: 4 FFMA2 + 2 ex2); 4: the same mix in scalar form (8 FFMA + 2 ex2).
template <int KIND>
__global__ void __launch_bounds__(1024, 1) probe_kernel(float* sink, long long* cycles,
                                                        int iters) {
  float x[8];
  float2 p[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[i] = -1e-3f * float(i + 1 + (threadIdx.x & 7));
    p[i] = make_float2(x[i], -x[i]);
  }
  const float2 m = make_float2(0.999f, 0.998f), c = make_float2(1e-7f, -1e-7f);
  __syncthreads();
  long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if constexpr (KIND == 0) {
        x[i] = ex2a(x[i]);  // saturates after a few trips; the issue rate does not depend on it
      } else if constexpr (KIND == 1) {
        x[i] = ffma_v(x[i], 0.999f, 1e-7f);
      } else if constexpr (KIND == 2) {
        p[i] = __ffma2_rn(p[i], m, c);
      } else if constexpr (KIND == 3) {
        if (i < 4) {
          p[i] = __ffma2_rn(p[i], m, c);
          p[i + 4] = __ffma2_rn(p[i + 4], m, c);
        } else {
          x[i] = ex2a(x[i]);
        }
      } else {
        x[i] = ffma_v(x[i], 0.999f, 1e-7f);
        if (i < 2) x[i + 6] = ex2a(x[i + 6]);
      }
    }
  }
  __syncthreads();
  long long t1 = clock64();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += x[i] + p[i].x + p[i].y;
  sink[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int KIND>
cudaError_t launch(int blocks, int smem, float* sink, long long* cyc, int iters) {
  cudaError_t e = cudaFuncSetAttribute(probe_kernel<KIND>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  probe_kernel<KIND><<<blocks, 1024, smem>>>(sink, cyc, iters);
  return cudaGetLastError();
}

__global__ void sfu_ex2_kernel(const float* __restrict__ x, float* __restrict__ y, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    y[i] = ex2a(x[i]);
}

// Operations per thread and loop trip, by kind: {ex2, FP32 lane-ops}.
constexpr int kEx2PerTrip[5] = {8, 0, 0, 4, 2};
constexpr int kFmaPerTrip[5] = {0, 8, 16, 16, 8};

}  // namespace

extern "C" {

// Runs probe `kind` (0-4) on `blocks` CTAs of 1024 threads for `iters` loop trips per thread and
// writes, per CTA, the SM cycles it took (cycles_out, host array of `blocks` entries). The
// operations per thread and trip are returned in *ex2_per_trip and *fma_per_trip (FP32
// lane-operations: an FFMA2 counts two). Returns 0, or the CUDA error code.
int sscan_peaks_probe(int kind, int blocks, int iters, long long* cycles_out, int* ex2_per_trip,
                      int* fma_per_trip) {
  if (kind < 0 || kind > 4 || blocks <= 0 || iters <= 0 || !cycles_out) return int(cudaErrorInvalidValue);
  float* sink = nullptr;
  long long* cyc = nullptr;
  cudaError_t e = cudaMalloc(&sink, size_t(blocks) * 1024 * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&cyc, size_t(blocks) * sizeof(long long));
  constexpr int kSmem = 120 * 1024;  // two such CTAs do not fit on one SM
  if (e == cudaSuccess) {
    switch (kind) {
      case 0: e = launch<0>(blocks, kSmem, sink, cyc, iters); break;
      case 1: e = launch<1>(blocks, kSmem, sink, cyc, iters); break;
      case 2: e = launch<2>(blocks, kSmem, sink, cyc, iters); break;
      case 3: e = launch<3>(blocks, kSmem, sink, cyc, iters); break;
      default: e = launch<4>(blocks, kSmem, sink, cyc, iters); break;
    }
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(cycles_out, cyc, size_t(blocks) * sizeof(long long), cudaMemcpyDeviceToHost);
  if (sink) cudaFree(sink);
  if (cyc) cudaFree(cyc);
  if (ex2_per_trip) *ex2_per_trip = kEx2PerTrip[kind];
  if (fma_per_trip) *fma_per_trip = kFmaPerTrip[kind];
  return int(e);
}

// y[i] = ex2.approx.ftz.f32(x[i]) for i < n (device pointers): the SFU exponential's actual
// outputs, for accuracy studies of the decay factors it produces. Returns 0 or a CUDA error.
int sscan_peaks_sfu_ex2(const float* x, float* y, long long n) {
  if (n < 0 || (n > 0 && (!x || !y))) return int(cudaErrorInvalidValue);
  if (n == 0) return 0;
  const long long blocks = (n + 255) / 256 < 148 * 64 ? (n + 255) / 256 : 148 * 64;
  sfu_ex2_kernel<<<unsigned(blocks), 256>>>(x, y, n);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return int(e);
}

}  // extern "C"

namespace {

// The scan's step loop alone, as a ceiling for kernels built around it: per lane K states in
// registers (K = 16: one lane per channel; K = 8: two lanes per channel), and per step the
// per-warp table entry (dt, dt u) and the B (and C) row of the step read from shared memory, then
// per state pair one packed arg FMA, two ex2, one packed input FMUL, one packed state FMA and,
// with the readout, one packed readout FMA into a per-step sum. 16-step chunks; two buffers of
// operands alternate between chunks (the loads cannot be hoisted out of the chunk loop). No
// global-memory traffic, no softplus, gate or store: what is left when all of that is hidden.
constexpr int kLoopTC = 16;
template <int K, bool READOUT>
__global__ void __launch_bounds__(128, 6) step_loop_kernel(float* sink, long long* cyc,
                                                           unsigned* smid, int chunks) {
  constexpr int KP = K / 2;
  __shared__ float2 tab[2][kLoopTC][32];
  __shared__ __align__(16) float Bs[2][kLoopTC][16];
  __shared__ __align__(16) float Cs[2][kLoopTC][16];
  const int lane = threadIdx.x & 31;
  const int n0 = (lane % (16 / K)) * K;
  for (int i = threadIdx.x; i < 2 * kLoopTC * 16; i += blockDim.x) {
    Bs[i / (kLoopTC * 16)][(i / 16) % kLoopTC][i % 16] = 0.5f + 1e-3f * float(i);
    Cs[i / (kLoopTC * 16)][(i / 16) % kLoopTC][i % 16] = 0.25f - 5e-4f * float(i);
  }
  for (int i = threadIdx.x; i < 2 * kLoopTC * 32; i += blockDim.x)
    tab[i / (kLoopTC * 32)][(i / 32) % kLoopTC][i % 32] =
        make_float2(0.01f + 1e-4f * float(i % 97), 3e-3f * float(i % 32 + 1));
  float2 A2[KP], h[KP];
#pragma unroll
  for (int r = 0; r < KP; ++r) {
    A2[r] = make_float2(-1.4427f * float(n0 + 2 * r + 1), -1.4427f * float(n0 + 2 * r + 2));
    h[r] = make_float2(0.f, 0.f);
  }
  float ysum = 0.f;
  __shared__ long long t_start;  // thread 0's start clock (kept out of the loop's registers)
  __syncthreads();
  if (threadIdx.x == 0) t_start = clock64();
  for (int c = 0; c < chunks; ++c) {
    const int sb = c & 1;
#pragma unroll
    for (int t = 0; t < kLoopTC; ++t) {
      const float2 sv = tab[sb][t][lane];
      const float4* Bq = reinterpret_cast<const float4*>(&Bs[sb][t][n0]);
      const float4* Cq = reinterpret_cast<const float4*>(&Cs[sb][t][n0]);
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < K / 4; ++q) {
        const float4 bq = Bq[q];
        float4 cq = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (READOUT) cq = Cq[q];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int r = 2 * q + j;
          const float2 a = __ffma2_rn(make_float2(sv.x, sv.x), A2[r], make_float2(0.f, 0.f));
          const float2 dA = make_float2(ex2a(a.x), ex2a(a.y));
          const float2 bb = j ? make_float2(bq.z, bq.w) : make_float2(bq.x, bq.y);
          h[r] = __ffma2_rn(dA, h[r], __fmul2_rn(make_float2(sv.y, sv.y), bb));
          if constexpr (READOUT) {
            const float2 cc = j ? make_float2(cq.z, cq.w) : make_float2(cq.x, cq.y);
            acc = __ffma2_rn(cc, h[r], acc);
          }
        }
      }
      ysum += acc.x + acc.y;
    }
  }
  __syncthreads();
  const long long t1 = clock64();
#pragma unroll
  for (int r = 0; r < KP; ++r) ysum += h[r].x + h[r].y;
  sink[size_t(blockIdx.x) * blockDim.x + threadIdx.x] = ysum;
  if (threadIdx.x == 0) {
    unsigned id;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
    smid[blockIdx.x] = id;
    cyc[2 * blockIdx.x] = t_start;
    cyc[2 * blockIdx.x + 1] = t1;
  }
}

}  // namespace

extern "C" {

// The step-loop probe: `blocks` CTAs of 128 threads (at most 6 resident per SM, so 148 x k CTAs
// give k x 4 warps per SM for k <= 6), each running `chunks` 16-step chunks of the scan's step loop with
// `states_per_lane` (8 or 16) states per lane, with (readout 1) or without (0) the readout FMA.
// Writes per CTA its SM id (smid_out) and its start and end SM clock (clk_out, 2 per CTA; host
// arrays). State updates per CTA: 128 x states_per_lane x 16 x chunks. Returns 0 or a CUDA error.
int sscan_peaks_step_loop(int states_per_lane, int readout, int blocks, int chunks,
                          unsigned* smid_out, long long* clk_out) {
  if ((states_per_lane != 8 && states_per_lane != 16) || blocks <= 0 || chunks <= 0 ||
      !smid_out || !clk_out)
    return int(cudaErrorInvalidValue);
  float* sink = nullptr;
  long long* cyc = nullptr;
  unsigned* sm = nullptr;
  cudaError_t e = cudaMalloc(&sink, size_t(blocks) * 128 * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&cyc, size_t(blocks) * 2 * sizeof(long long));
  if (e == cudaSuccess) e = cudaMalloc(&sm, size_t(blocks) * sizeof(unsigned));
  if (e == cudaSuccess) {
    if (states_per_lane == 16)
      readout ? step_loop_kernel<16, true><<<blocks, 128>>>(sink, cyc, sm, chunks)
              : step_loop_kernel<16, false><<<blocks, 128>>>(sink, cyc, sm, chunks);
    else
      readout ? step_loop_kernel<8, true><<<blocks, 128>>>(sink, cyc, sm, chunks)
              : step_loop_kernel<8, false><<<blocks, 128>>>(sink, cyc, sm, chunks);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(clk_out, cyc, size_t(blocks) * 2 * sizeof(long long), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess)
    e = cudaMemcpy(smid_out, sm, size_t(blocks) * sizeof(unsigned), cudaMemcpyDeviceToHost);
  if (sink) cudaFree(sink);
  if (cyc) cudaFree(cyc);
  if (sm) cudaFree(sm);
  return int(e);
}

}  // extern "C"

