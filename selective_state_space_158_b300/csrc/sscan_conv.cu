// sscan_conv.cu -- causal depthwise convolution over time followed by SiLU, the step that turns
// the Mamba block's in-projection output into the scan's input ("Mamba: Linear-Time Sequence
// Modeling with Selective State Spaces" notes, "架构：极简设计": Linear -> Conv1d -> SiLU).
//
//   y[b, t, d] = SiLU(bias[d] + sum_{j < W} w[d, j] * x[b, t - (W - 1) + j, d])
//
// with the inputs before t = 0 taken from x_prev (batch, W - 1, dim) or zero. It moves every
// input and output once, so it is bound by HBM: each thread owns four consecutive channels
// over a tile of kConvT steps and keeps the last W - 1 inputs of its channels in registers, so a
// step costs one vector load and one vector store per thread (16 bytes fp32, 8 bytes bf16),
// issued kConvU steps at a time; a tile re-reads only its W - 1 step halo.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sscan_device.cuh"
#include "sscan_internal.h"

namespace sscan {
namespace {

constexpr int kConvT = 32;  // steps per thread
constexpr int kConvU = 4;   // steps whose loads are issued together

template <typename IO>
struct Vec;  // four consecutive channels' io values as floats (16 bytes fp32, 8 bytes bf16)
template <>
struct Vec<float> {
  static constexpr int V = 4;
  __device__ static void load(const float* p, float (&v)[4]) {
    const float4 r = *reinterpret_cast<const float4*>(p);
    v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
  }
  __device__ static void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int V = 4;
  __device__ static void load(const __nv_bfloat16* p, float (&v)[4]) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    v[0] = a.x; v[1] = a.y; v[2] = c.x; v[3] = c.y;
  }
  __device__ static void store(__nv_bfloat16* p, const float (&v)[4]) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
    *reinterpret_cast<uint2*>(p) = make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                                              *reinterpret_cast<const uint32_t*>(&hi));
  }
};

__device__ __forceinline__ float silu_or_id(float a, int silu) { return silu ? silu_f(a) : a; }

// Vector path: W taps (1 .. 8), dim a multiple of 4, x / y / x_prev aligned to the vector.
// Register budget 128 (two blocks of 256 per SM), except for the widest windows.
template <int W>
__host__ __device__ constexpr int conv_min_blocks() { return W <= 6 ? 2 : 1; }

template <typename IO, int W>
__global__ void __launch_bounds__(256, conv_min_blocks<W>()) conv_vec_kernel(const IO* __restrict__ x,
                                                       const float* __restrict__ w,
                                                       const float* __restrict__ bias,
                                                       const IO* __restrict__ x_prev, int silu,
                                                       IO* __restrict__ y, int64_t batch,
                                                       int64_t L, int64_t dim) {
  constexpr int V = Vec<IO>::V;
  const int64_t groups = dim / V;
  const int64_t tiles = (L + kConvT - 1) / kConvT;
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= batch * tiles * groups) return;
  const int64_t grp = gid % groups;  // channel group fastest: neighbouring threads, adjacent bytes
  const int64_t tile = (gid / groups) % tiles;
  const int64_t b = gid / (groups * tiles);
  const int64_t d0 = grp * V;
  float wk[W][V], bs[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
#pragma unroll
    for (int j = 0; j < W; ++j) wk[j][i] = w[(d0 + i) * W + j];
    bs[i] = bias ? bias[d0 + i] : 0.f;
  }
  const int64_t t0 = tile * kConvT;
  // win[j] holds the input of step t - (W - 1) + j for the step t being computed.
  float win[W][V];
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    const int64_t s = t0 - (W - 1) + j;
    if (s >= 0) {
      Vec<IO>::load(x + (b * L + s) * dim + d0, win[j]);
    } else if (x_prev) {
      Vec<IO>::load(x_prev + (b * (W - 1) + (s + W - 1)) * dim + d0, win[j]);
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) win[j][i] = 0.f;
    }
  }
  const int64_t t_end = t0 + kConvT < L ? t0 + kConvT : L;
  // kConvU steps at a time: their loads are issued together, so each thread keeps several
  // 16-byte requests in flight.
  for (int64_t t = t0; t < t_end; t += kConvU) {
    float in[kConvU][V];
#pragma unroll
    for (int k = 0; k < kConvU; ++k)
      if (t + k < t_end) Vec<IO>::load(x + (b * L + t + k) * dim + d0, in[k]);
#pragma unroll
    for (int k = 0; k < kConvU; ++k) {
      if (t + k >= t_end) break;
#pragma unroll
      for (int i = 0; i < V; ++i) win[W - 1][i] = in[k][i];
      float out[V];
#pragma unroll
      for (int i = 0; i < V; ++i) {
        float acc = bs[i];
#pragma unroll
        for (int j = 0; j < W; ++j) acc = fmaf(wk[j][i], win[j][i], acc);
        out[i] = silu_or_id(acc, silu);
      }
      Vec<IO>::store(y + (b * L + t + k) * dim + d0, out);
#pragma unroll
      for (int j = 0; j < W - 1; ++j)
#pragma unroll
        for (int i = 0; i < V; ++i) win[j][i] = win[j + 1][i];
    }
  }
}

// Any width up to 64, any dim and alignment: one thread per (batch, channel, tile), taps read
// through the cache.
template <typename IO>
__global__ void __launch_bounds__(256) conv_scalar_kernel(const IO* __restrict__ x,
                                                          const float* __restrict__ w,
                                                          const float* __restrict__ bias,
                                                          const IO* __restrict__ x_prev, int silu,
                                                          IO* __restrict__ y, int64_t batch,
                                                          int64_t L, int64_t dim, int W) {
  const int64_t tiles = (L + kConvT - 1) / kConvT;
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= batch * tiles * dim) return;
  const int64_t d = gid % dim;
  const int64_t tile = (gid / dim) % tiles;
  const int64_t b = gid / (dim * tiles);
  const int64_t t0 = tile * kConvT;
  const int64_t t_end = t0 + kConvT < L ? t0 + kConvT : L;
  const float bs = bias ? bias[d] : 0.f;
  for (int64_t t = t0; t < t_end; ++t) {
    float acc = bs;
    for (int j = 0; j < W; ++j) {
      const int64_t s = t - (W - 1) + j;
      float v = 0.f;
      if (s >= 0)
        v = to_f32(x[(b * L + s) * dim + d]);
      else if (x_prev)
        v = to_f32(x_prev[(b * (W - 1) + (s + W - 1)) * dim + d]);
      acc = fmaf(w[d * W + j], v, acc);
    }
    store_io(y + (b * L + t) * dim + d, silu_or_id(acc, silu));
  }
}

template <typename IO>
cudaError_t launch_conv_typed(const ConvArgs& a) {
  constexpr int V = Vec<IO>::V;
  const IO* x = static_cast<const IO*>(a.x);
  const IO* xp = static_cast<const IO*>(a.x_prev);
  IO* y = static_cast<IO*>(a.y);
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) % (V * sizeof(IO))) == 0; };
  const int64_t tiles = (a.L + kConvT - 1) / kConvT;
  const int threads = 256;
  if (a.width <= 8 && a.dim % V == 0 && al(x) && al(y) && (!xp || al(xp))) {
    const int64_t n = a.batch * tiles * (a.dim / V);
    const unsigned blocks = unsigned((n + threads - 1) / threads);
#define SSCAN_CONV_W(WW)                                                                 \
  case WW:                                                                                \
    conv_vec_kernel<IO, WW><<<blocks, threads, 0, a.stream>>>(x, a.w, a.bias, xp, a.silu, y, \
                                                              a.batch, a.L, a.dim);         \
    break;
    switch (a.width) {
      SSCAN_CONV_W(1) SSCAN_CONV_W(2) SSCAN_CONV_W(3) SSCAN_CONV_W(4)
      SSCAN_CONV_W(5) SSCAN_CONV_W(6) SSCAN_CONV_W(7) SSCAN_CONV_W(8)
      default: return cudaErrorInvalidValue;
    }
#undef SSCAN_CONV_W
  } else {
    const int64_t n = a.batch * tiles * a.dim;
    const unsigned blocks = unsigned((n + threads - 1) / threads);
    conv_scalar_kernel<IO><<<blocks, threads, 0, a.stream>>>(x, a.w, a.bias, xp, a.silu, y,
                                                             a.batch, a.L, a.dim, a.width);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv(const ConvArgs& a) {
  return a.io == Io::F32 ? launch_conv_typed<float>(a) : launch_conv_typed<__nv_bfloat16>(a);
}

}  // namespace sscan
