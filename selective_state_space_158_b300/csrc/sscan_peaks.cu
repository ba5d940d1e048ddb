// sscan_peaks.cu -- issue-rate microbenchmarks that give the compute rooflines of the scan their
// denominators on the machine at hand: how many SFU exponentials (ex2.approx.ftz.f32), scalar
// FFMAs and packed FFMA2s one SM completes per clock, alone and in the mix one state update of
// the scan issues (one arg FMA, one decay exponential, one input FMUL, one state FMA, one readout
// FMA). Built as its own small library (libsscan_peaks.so); the scan library does not use it.
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
