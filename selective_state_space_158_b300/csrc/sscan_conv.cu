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

#include <algorithm>
#include <cstdlib>

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

// ---- TMA-staged streaming kernel ------------------------------------------------------------
// Work item: one tile of kTileT steps x kRowBytes of channels of one batch row. A persistent CTA
// walks its items (item c, c + grid, ...) through a kConvStages-deep pipeline: one thread loads
// each item's input tile with its W - 1 step halo by TMA (rows before t = 0 arrive zero-filled),
// all threads compute from shared memory into an output tile, and the same thread stores it by
// TMA (rows past L and channels past dim are clipped). Every input byte is read once (plus the
// halo, 3/64 of a tile for width 4, mostly from L2) and every output byte written once. Small
// CTAs (128 threads, 33 KB of shared memory) let six share an SM: measured on B300, more
// resident CTAs beat deeper pipelines (bf16 b16 L4096 D2048: 256-byte rows, 256 threads and
// four stages 145 us; this shape 120 us).
constexpr int kTileT = 64;                       // steps per tile
constexpr int kRowBytes = 128;                   // channel bytes per tile row
constexpr int kWords = kRowBytes / 4;            // 4-byte words per row: 2 bf16 or 1 fp32 channels
constexpr int kConvThreads = 128;
constexpr int kGroups = kConvThreads / kWords;   // step groups per tile
constexpr int kStepsPerThread = kTileT / kGroups;
constexpr int kConvStages = 2;
constexpr int kOutBufs = 2;                      // output tiles in flight to the TMA store
constexpr int kMaxTmaWidth = 8;

template <typename IO, int W>
struct ConvTmaSmem {
  static constexpr int rows_in = kTileT + W - 1;
  static constexpr size_t in_box = size_t(rows_in) * kRowBytes;  // bytes one load delivers
  // TMA destinations start on 128-byte boundaries: stages and tiles are rounded up to 128.
  static constexpr size_t in_stage = (in_box + 127) / 128 * 128;
  static constexpr size_t out_tile = (size_t(kTileT) * kRowBytes + 127) / 128 * 128;
  static constexpr size_t off_out = kConvStages * in_stage;
  static constexpr size_t off_bar = off_out + kOutBufs * out_tile;
  static constexpr size_t bytes = off_bar + kConvStages * 8 + 128;  // + alignment slack
};

template <typename IO> struct Word;  // one 4-byte word of a row as floats
template <> struct Word<float> {
  static constexpr int C = 1;
  __device__ static void get(const unsigned char* p, float (&v)[1]) {
    v[0] = *reinterpret_cast<const float*>(p);
  }
  __device__ static void put(unsigned char* p, const float (&v)[1]) {
    *reinterpret_cast<float*>(p) = v[0];
  }
};
template <> struct Word<__nv_bfloat16> {
  static constexpr int C = 2;
  __device__ static void get(const unsigned char* p, float (&v)[2]) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
    v[0] = f.x;
    v[1] = f.y;
  }
  __device__ static void put(unsigned char* p, const float (&v)[2]) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v[0], v[1]);
  }
};

template <typename IO, int W>
__global__ void __launch_bounds__(kConvThreads) conv_tma_kernel(
    const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
    const float* __restrict__ w, const float* __restrict__ bias, const IO* __restrict__ x_prev,
    int silu, int64_t batch, int64_t L, int64_t dim, unsigned* status) {
  using SM = ConvTmaSmem<IO, W>;
  constexpr int C = Word<IO>::C;            // channels per word
  constexpr int CT = kRowBytes / sizeof(IO);  // channels per tile
  extern __shared__ unsigned char conv_smem_raw[];
  unsigned char* smem =
      conv_smem_raw + ((128u - (smem_addr(conv_smem_raw) & 127u)) & 127u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::off_bar);
  const int tid = threadIdx.x;
  const int wd = tid % kWords, grp = tid / kWords;

  const int64_t n_cb = (dim + CT - 1) / CT, n_tt = (L + kTileT - 1) / kTileT;
  const int64_t items = batch * n_tt * n_cb;
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t n_my = first < items ? (items - first + stride - 1) / stride : 0;
  // item -> (batch row, time tile, channel block); neighbouring items are neighbouring channel
  // blocks of one time tile.
  auto coords = [&](int64_t it, int64_t& b, int64_t& t0, int64_t& c0) {
    const int64_t item = first + it * stride;
    c0 = (item % n_cb) * CT;
    t0 = ((item / n_cb) % n_tt) * kTileT;
    b = item / (n_cb * n_tt);
  };
  auto issue = [&](int64_t it) {
    int64_t b, t0, c0;
    coords(it, b, t0, c0);
    const int s = int(it % kConvStages);
    mbar_arrive_expect_tx(&full[s], uint32_t(SM::in_box));
    tma_load_3d(smem + size_t(s) * SM::in_stage, &tm_x, int(c0), int(t0 - (W - 1)), int(b),
                &full[s]);
  };
  if (tid == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_y);
    for (int s = 0; s < kConvStages; ++s) mbar_init(&full[s], 1);
    mbar_init_fence();
    for (int64_t it = 0; it < kConvStages && it < n_my; ++it) issue(it);
  }
  __syncthreads();

  bool timed_out = false;
  for (int64_t it = 0; it < n_my; ++it) {
    const int s = int(it % kConvStages), ob = int(it % kOutBufs);
    const uint32_t parity = uint32_t((it / kConvStages) & 1);
    const bool landed = mbar_wait_bounded(&full[s], parity, kWaitNs);
    if (tid == 0 && it >= kOutBufs) tma_store_wait_read<kOutBufs - 1>();  // tile reusable
    if (__syncthreads_or(!landed)) {
      timed_out = true;
      break;
    }
    int64_t b, t0, c0;
    coords(it, b, t0, c0);
    // This thread: word wd (channels c0 + C wd ..), steps t0 + grp * kStepsPerThread + i.
    const int64_t ch = c0 + int64_t(wd) * C;
    float wk[W][C], bs[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const bool ok = ch + c < dim;
#pragma unroll
      for (int j = 0; j < W; ++j) wk[j][c] = ok ? w[(ch + c) * W + j] : 0.f;
      bs[c] = (ok && bias) ? bias[ch + c] : 0.f;
    }
    const unsigned char* in = smem + size_t(s) * SM::in_stage + size_t(wd) * 4;
    unsigned char* out = smem + SM::off_out + size_t(ob) * SM::out_tile + size_t(wd) * 4;
    const int r0 = grp * kStepsPerThread;  // first input row of this thread's window
    float win[W][C];
#pragma unroll
    for (int j = 0; j < W - 1; ++j) {
      Word<IO>::get(in + size_t(r0 + j) * kRowBytes, win[j]);
      // Rows before t = 0 come from x_prev when given (the tile holds zeros there).
      if (x_prev && t0 == 0 && r0 + j < W - 1) {
#pragma unroll
        for (int c = 0; c < C; ++c)
          win[j][c] = ch + c < dim ? to_f32(x_prev[(b * (W - 1) + r0 + j) * dim + ch + c]) : 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < kStepsPerThread; ++i) {
      Word<IO>::get(in + size_t(r0 + i + W - 1) * kRowBytes, win[W - 1]);
      float o[C];
#pragma unroll
      for (int c = 0; c < C; ++c) {
        float acc = bs[c];
#pragma unroll
        for (int j = 0; j < W; ++j) acc = fmaf(wk[j][c], win[j][c], acc);
        o[c] = silu_or_id(acc, silu);
      }
      Word<IO>::put(out + size_t(r0 + i) * kRowBytes, o);
#pragma unroll
      for (int j = 0; j < W - 1; ++j)
#pragma unroll
        for (int c = 0; c < C; ++c) win[j][c] = win[j + 1][c];
    }
    fence_smem_to_async();
    __syncthreads();  // output tile complete; input stage s consumed
    if (tid == 0) {
      tma_store_3d(&tm_y, smem + SM::off_out + size_t(ob) * SM::out_tile, int(c0), int(t0),
                   int(b));
      tma_store_commit();
      if (it + kConvStages < n_my) issue(it + kConvStages);
    }
  }
  if (tid == 0) {
    tma_store_wait_all();
    if (timed_out) {
      if (status) atomicOr(status, kErrTimeout);
      // Loads still in flight get a bounded chance to land before shared memory goes away.
      for (int s = 0; s < kConvStages; ++s) mbar_wait_bounded(&full[s], 0, 100000);
    }
  }
}

template <typename IO, int W>
cudaError_t launch_conv_tma(const ConvArgs& a) {
  using SM = ConvTmaSmem<IO, W>;
  constexpr int CT = kRowBytes / sizeof(IO);
  CUtensorMap mx, my;
  if (!make_tensor_map_3d(&mx, a.x, a.io, uint64_t(a.dim), uint64_t(a.L), uint64_t(a.batch), CT,
                          SM::rows_in) ||
      !make_tensor_map_3d(&my, a.y, a.io, uint64_t(a.dim), uint64_t(a.L), uint64_t(a.batch), CT,
                          kTileT))
    return cudaErrorInvalidValue;
  auto kern = conv_tma_kernel<IO, W>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(SM::bytes));
  int dev = 0, sms = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kConvThreads, SM::bytes);
  if (e != cudaSuccess) return e;
  const int64_t items = a.batch * ((a.L + kTileT - 1) / kTileT) * ((a.dim + CT - 1) / CT);
  const unsigned grid =
      unsigned(std::max<int64_t>(1, std::min<int64_t>(items, int64_t(std::max(per_sm, 1)) * sms)));
  kern<<<grid, kConvThreads, SM::bytes, a.stream>>>(mx, my, a.w, a.bias,
                                                    static_cast<const IO*>(a.x_prev), a.silu,
                                                    a.batch, a.L, a.dim, a.status);
  return cudaGetLastError();
}

// TMA needs 16-byte aligned bases and row strides, coordinates within int32.
bool conv_tma_ok(const ConvArgs& a, int es) {
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  return a.width <= kMaxTmaWidth && (a.dim * es) % 16 == 0 && al(a.x) && al(a.y) &&
         a.dim <= INT32_MAX && a.L + kTileT < INT32_MAX && a.batch <= INT32_MAX &&
         !current_tuning().conv_plain;
}

template <typename IO>
cudaError_t launch_conv_typed(const ConvArgs& a) {
  if (conv_tma_ok(a, int(sizeof(IO)))) {
    switch (a.width) {
      case 1: return launch_conv_tma<IO, 1>(a);
      case 2: return launch_conv_tma<IO, 2>(a);
      case 3: return launch_conv_tma<IO, 3>(a);
      case 4: return launch_conv_tma<IO, 4>(a);
      case 5: return launch_conv_tma<IO, 5>(a);
      case 6: return launch_conv_tma<IO, 6>(a);
      case 7: return launch_conv_tma<IO, 7>(a);
      case 8: return launch_conv_tma<IO, 8>(a);
      default: break;
    }
  }
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
