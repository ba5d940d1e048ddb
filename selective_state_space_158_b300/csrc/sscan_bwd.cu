// sscan_bwd.cu -- backward pass of the selective scan with recomputation: the intermediate
// states are recomputed rather than stored ("Mamba: Linear-Time Sequence Modeling with Selective
// State Spaces" notes, "第二个创新：硬件感知算法", item 3; "从RNN到Mamba" 3.3, item 2).
//
// Gradients of sum(dy * y) + sum(dh_last * h_last) by the adjoint recurrence, per channel:
//   lam_t = ds_t C_t + a_{t+1} lam_{t+1}          (lam = dLoss/dh_t, ds_t = dy_t SiLU(z_t))
//   dB_t += lam_t dt_t u_t,  dC_t += ds_t h_t,  du_t = ds_t D + sum_n lam_t dt_t B_t
//   d(dt_t) = sum_n lam_t (B_t u_t + h_{t-1} da_t/d(dt)),  dA += lam_t h_{t-1} da_t/dA
//   ddelta_t = d(dt_t) sigmoid(x_t) (softplus), dz_t = dy_t s_t SiLU'(z_t), dh0 = a_0 lam_0.
//
// Three kernels:
//   1. bwd_ckpt_kernel: the forward recurrence (no readout) writing the state before every
//      16-step chunk (B * D * N floats per chunk);
//   2. bwd_chunk_kernel: four lanes per channel (four states each); chunks in reverse order: the
//      chunk's 16 steps are recomputed from its checkpoint (states kept in registers), then the
//      adjoint sweeps back through them. Per-channel sums over the four lanes use shuffles. dB
//      and dC sum over channels: each warp reduces its 8 channels with shuffles into its own
//      shared-memory slot, the CTA adds the slots in warp order, and the CTA's partial is
//      stored per channel group;
//   3. bwd_reduce_kernel: sums the partials in a fixed order (deterministic): dB, dC over channel
//      groups, dA, dD, dbias over batch rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "sscan_device.cuh"
#include "sscan_internal.h"

namespace sscan {
namespace {

constexpr int kBT = 16;      // steps per chunk
constexpr int kBG = 4;       // lanes per channel
constexpr int kBK = 4;       // states per lane (N <= 16)
constexpr int kBThreads = 256;
constexpr int kBCh = kBThreads / kBG;  // channels per CTA

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + ex2(-x * kLog2e)); }

template <bool EULER>
__device__ __forceinline__ float factor(float dt, float a2) {
  // a2 = A log2e (zero-order hold) or A (first order)
  return EULER ? fmaf(dt, a2, 1.f) : ex2(fmaf(dt, a2, kEx2ArgShift));
}

// ---- 1. checkpoints: the state before every chunk ----------------------------------------------
template <typename IO, bool EULER>
__global__ void __launch_bounds__(256) bwd_ckpt_kernel(BwdArgs a, int n_chunks,
                                                       float* __restrict__ ckpt) {
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t c = gid / kBG;  // channel b * dim + d
  const int g = int(gid % kBG);
  if (c >= a.batch * a.dim) return;
  const int64_t b = c / a.dim, d = c - b * a.dim;
  const int N = int(a.N);
  const IO* u = static_cast<const IO*>(a.u);
  const IO* dl = static_cast<const IO*>(a.delta);
  const IO* Bm = static_cast<const IO*>(a.B);
  float a2[kBK], h[kBK];
#pragma unroll
  for (int k = 0; k < kBK; ++k) {
    const int n = g * kBK + k;
    a2[k] = n < N ? a.A[d * N + n] * (EULER ? 1.f : kLog2e) : 0.f;
    h[k] = (a.h0 && n < N) ? a.h0[c * N + n] : 0.f;
  }
  const float bias = a.bias ? a.bias[d] : 0.f;
  const size_t ck_stride = size_t(a.batch) * a.dim * N;
  for (int ch = 0; ch < n_chunks; ++ch) {
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      const int n = g * kBK + k;
      if (n < N) ckpt[size_t(ch) * ck_stride + size_t(c) * N + n] = h[k];
    }
    const int64_t t0 = int64_t(ch) * kBT;
    float dts[kBT], dtu[kBT];
#pragma unroll
    for (int j = 0; j < kBT; ++j) {  // the chunk's inputs first, so the loads overlap
      const int64_t t = t0 + j;
      float x = 0.f, uu = 0.f;
      if (t < a.L) {
        const int64_t i = (b * a.L + t) * a.dim + d;
        x = to_f32(dl[i]) + bias;
        uu = to_f32(u[i]);
      }
      const float dt = t < a.L ? (a.softplus ? softplus_f(x) : x) : 0.f;
      dts[j] = dt;
      dtu[j] = dt * uu;
    }
#pragma unroll
    for (int j = 0; j < kBT; ++j) {
      const int64_t t = t0 + j;
#pragma unroll
      for (int k = 0; k < kBK; ++k) {
        const int n = g * kBK + k;
        const float bt = (t < a.L && n < N) ? to_f32(Bm[(b * a.L + t) * N + n]) : 0.f;
        h[k] = fmaf(factor<EULER>(dts[j], a2[k]), h[k], dtu[j] * bt);
      }
    }
  }
}

// ---- 2. the adjoint sweep over chunks in reverse -----------------------------------------------
template <typename IO, bool EULER>
__global__ void __launch_bounds__(kBThreads, 1) bwd_chunk_kernel(BwdArgs a, int n_chunks,
                                                                 const float* __restrict__ ckpt,
                                                                 float* __restrict__ part_dB,
                                                                 float* __restrict__ part_dC,
                                                                 float* __restrict__ part_dA,
                                                                 float* __restrict__ part_dD,
                                                                 float* __restrict__ part_db) {
  // Per-warp slots of the chunk's dB / dC sums over the warp's channels; the CTA adds the
  // slots in warp order (no atomics: the result does not depend on timing).
  __shared__ float sdB[kBThreads / 32][kBT][16], sdC[kBThreads / 32][kBT][16];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane % kBG;
  const int64_t b = blockIdx.y;
  const int cg_idx = blockIdx.x;
  const int64_t d = int64_t(cg_idx) * kBCh + tid / kBG;
  const bool live = d < a.dim;
  const int N = int(a.N);
  const int64_t c = b * a.dim + d;
  const IO* u = static_cast<const IO*>(a.u);
  const IO* dl = static_cast<const IO*>(a.delta);
  const IO* Bm = static_cast<const IO*>(a.B);
  const IO* Cm = static_cast<const IO*>(a.C);
  const IO* zz = static_cast<const IO*>(a.z);
  const IO* dy = static_cast<const IO*>(a.dy);
  float a2[kBK], Av[kBK], mu[kBK], dA[kBK];
#pragma unroll
  for (int k = 0; k < kBK; ++k) {
    const int n = g * kBK + k;
    Av[k] = (live && n < N) ? a.A[d * N + n] : 0.f;
    a2[k] = Av[k] * (EULER ? 1.f : kLog2e);
    mu[k] = (live && a.dh_last && n < N) ? a.dh_last[c * N + n] : 0.f;
    dA[k] = 0.f;
  }
  const float bias = (live && a.bias) ? a.bias[d] : 0.f;
  const float Dd = (live && a.D) ? a.D[d] : 0.f;
  float dD = 0.f, dbias = 0.f;
  const size_t ck_stride = size_t(a.batch) * a.dim * N;
  const size_t part_stride = size_t(a.batch) * a.L * 16;  // one channel group's [b][t][16]

  for (int ch = n_chunks - 1; ch >= 0; --ch) {
    const int64_t t0 = int64_t(ch) * kBT;
    // Recompute the chunk: hist[j] is the state before step t0 + j (hist[kBT]: after the last).
    float hist[kBT + 1][kBK], dts[kBT], uus[kBT], spart[kBT];
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      const int n = g * kBK + k;
      hist[0][k] = (live && n < N) ? ckpt[size_t(ch) * ck_stride + size_t(c) * N + n] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kBT; ++j) {
      const int64_t t = t0 + j;
      const bool tv = live && t < a.L;
      float x = 0.f, uu = 0.f;
      if (tv) {
        const int64_t i = (b * a.L + t) * a.dim + d;
        x = to_f32(dl[i]) + bias;
        uu = to_f32(u[i]);
      }
      const float dt = tv ? (a.softplus ? softplus_f(x) : x) : 0.f;
      dts[j] = dt;
      uus[j] = uu;
      float sp = 0.f;
#pragma unroll
      for (int k = 0; k < kBK; ++k) {
        const int n = g * kBK + k;
        const bool nv = tv && n < N;
        const float bt = nv ? to_f32(Bm[(b * a.L + t) * N + n]) : 0.f;
        const float ct = nv ? to_f32(Cm[(b * a.L + t) * N + n]) : 0.f;
        hist[j + 1][k] = fmaf(factor<EULER>(dt, a2[k]), hist[j][k], dt * uu * bt);
        sp = fmaf(ct, hist[j + 1][k], sp);
      }
      spart[j] = sp;
    }
    // The readout's state part summed over the channel's four lanes (every lane gets it).
#pragma unroll
    for (int j = 0; j < kBT; ++j) {
      spart[j] += __shfl_xor_sync(0xffffffffu, spart[j], 1);
      spart[j] += __shfl_xor_sync(0xffffffffu, spart[j], 2);
    }
    // Adjoint sweep back through the chunk.
#pragma unroll
    for (int j = kBT - 1; j >= 0; --j) {
      const int64_t t = t0 + j;
      const bool tv = live && t < a.L;
      const float dt = dts[j], uu = uus[j];
      float dyt = 0.f, zt = 0.f, x = 0.f;
      if (tv) {
        const int64_t i = (b * a.L + t) * a.dim + d;
        dyt = to_f32(dy[i]);
        if (zz) zt = to_f32(zz[i]);
        x = to_f32(dl[i]) + bias;
      }
      float ds = dyt, dzv = 0.f;
      if (zz) {
        const float sg = sigmoid_f(zt);
        ds = dyt * zt * sg;
        dzv = dyt * (spart[j] + Dd * uu) * sg * fmaf(zt, 1.f - sg, 1.f);
      }
      float ddt = 0.f, dup = 0.f, vB[kBK], vC[kBK];
#pragma unroll
      for (int k = 0; k < kBK; ++k) {
        const int n = g * kBK + k;
        const bool nv = tv && n < N;
        const float bt = nv ? to_f32(Bm[(b * a.L + t) * N + n]) : 0.f;
        const float ct = nv ? to_f32(Cm[(b * a.L + t) * N + n]) : 0.f;
        const float fa = factor<EULER>(dt, a2[k]);
        const float lam = fmaf(ds, ct, mu[k]);
        const float da = lam * hist[j][k];
        const float dfa = EULER ? da : da * fa;  // lam h_{t-1} times d(factor)/d(dt A)
        ddt = fmaf(dfa, Av[k], fmaf(lam * bt, uu, ddt));
        dA[k] = fmaf(dfa, dt, dA[k]);
        vB[k] = lam * dt * uu;
        vC[k] = ds * hist[j + 1][k];
        dup = fmaf(lam * dt, bt, dup);
        mu[k] = fa * lam;
      }
      // per channel: sum over the four lanes
      ddt += __shfl_xor_sync(0xffffffffu, ddt, 1);
      ddt += __shfl_xor_sync(0xffffffffu, ddt, 2);
      dup += __shfl_xor_sync(0xffffffffu, dup, 1);
      dup += __shfl_xor_sync(0xffffffffu, dup, 2);
      if (tv && g == 0) {
        const int64_t i = (b * a.L + t) * a.dim + d;
        const float dx = a.softplus ? ddt * sigmoid_f(x) : ddt;
        store_io(static_cast<IO*>(a.du) + i, fmaf(ds, Dd, dup));
        store_io(static_cast<IO*>(a.ddelta) + i, dx);
        if (zz) store_io(static_cast<IO*>(a.dz) + i, dzv);
        dbias += dx;
        dD = fmaf(ds, uu, dD);
      }
      // dB, dC: sum over the warp's 8 channels (lanes with the same g), then into the CTA tile
#pragma unroll
      for (int k = 0; k < kBK; ++k) {
#pragma unroll
        for (int m = 4; m < 32; m <<= 1) {
          vB[k] += __shfl_xor_sync(0xffffffffu, vB[k], m);
          vC[k] += __shfl_xor_sync(0xffffffffu, vC[k], m);
        }
      }
      if (lane < kBG) {
#pragma unroll
        for (int k = 0; k < kBK; ++k) {
          sdB[warp][j][g * kBK + k] = vB[k];
          sdC[warp][j][g * kBK + k] = vC[k];
        }
      }
    }
    __syncthreads();
    // The CTA's partial of this chunk (warp slots added in order) to its channel group's slice.
    for (int i = tid; i < kBT * 16; i += kBThreads) {
      const int j = i / 16, n = i % 16;
      const int64_t t = t0 + j;
      if (t < a.L && n < N) {
        float sb = 0.f, sc = 0.f;
#pragma unroll
        for (int w = 0; w < kBThreads / 32; ++w) {
          sb += sdB[w][j][n];
          sc += sdC[w][j][n];
        }
        const size_t o = size_t(cg_idx) * part_stride + (size_t(b) * a.L + t) * 16 + n;
        part_dB[o] = sb;
        part_dC[o] = sc;
      }
    }
    __syncthreads();  // the slots are rewritten by the next chunk
  }
  if (!live) return;
  // dh0 = a_0 lam_0; per-batch-row partials of dA, dD, dbias.
#pragma unroll
  for (int k = 0; k < kBK; ++k) {
    const int n = g * kBK + k;
    if (n < N) {
      if (a.dh0) a.dh0[c * N + n] = mu[k];
      part_dA[(size_t(b) * a.dim + d) * N + n] = dA[k];
    }
  }
  if (g == 0) {
    part_dD[size_t(b) * a.dim + d] = dD;
    part_db[size_t(b) * a.dim + d] = dbias;
  }
}

// ---- 3. fixed-order sums of the partials -------------------------------------------------------
__global__ void __launch_bounds__(256) bwd_reduce_kernel(BwdArgs a, int n_groups,
                                                         const float* __restrict__ part_dB,
                                                         const float* __restrict__ part_dC,
                                                         const float* __restrict__ part_dA,
                                                         const float* __restrict__ part_dD,
                                                         const float* __restrict__ part_db) {
  const int64_t N = a.N;
  const int64_t nbc = a.batch * a.L * N, ndn = a.dim * N;
  const size_t part_stride = size_t(a.batch) * a.L * 16;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nbc + ndn + 2 * a.dim;
       i += int64_t(gridDim.x) * blockDim.x) {
    if (i < nbc) {  // dB, dC over channel groups
      const int64_t bt = i / N, n = i % N;
      float sb = 0.f, sc = 0.f;
      for (int q = 0; q < n_groups; ++q) {
        sb += part_dB[size_t(q) * part_stride + size_t(bt) * 16 + n];
        sc += part_dC[size_t(q) * part_stride + size_t(bt) * 16 + n];
      }
      a.dB[i] = sb;
      a.dC[i] = sc;
    } else if (i < nbc + ndn) {  // dA over batch rows
      const int64_t j = i - nbc;
      float s = 0.f;
      for (int64_t b = 0; b < a.batch; ++b) s += part_dA[size_t(b) * ndn + j];
      a.dA[j] = s;
    } else {  // dD, dbias over batch rows
      const int64_t j = i - nbc - ndn;
      const bool isD = j < a.dim;
      const int64_t dd = isD ? j : j - a.dim;
      const float* p = isD ? part_dD : part_db;
      float* out = isD ? a.dD : a.dbias;
      if (!out) continue;
      float s = 0.f;
      for (int64_t b = 0; b < a.batch; ++b) s += p[size_t(b) * a.dim + dd];
      out[dd] = s;
    }
  }
}

template <typename IO, bool EULER>
cudaError_t launch_bwd_typed(const BwdArgs& a) {
  const int n_chunks = int((a.L + kBT - 1) / kBT);
  const int n_groups = int((a.dim + kBCh - 1) / kBCh);
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t ck = up(size_t(n_chunks) * a.batch * a.dim * a.N * sizeof(float));
  const size_t pbc = up(size_t(n_groups) * a.batch * a.L * 16 * sizeof(float));
  const size_t pa = up(size_t(a.batch) * a.dim * a.N * sizeof(float));
  const size_t pd = up(size_t(a.batch) * a.dim * sizeof(float));
  void* ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, ck + 2 * pbc + pa + 2 * pd, a.stream);
  if (e != cudaSuccess) return e;
  char* p = static_cast<char*>(ws);
  float* ckpt = reinterpret_cast<float*>(p);
  float* part_dB = reinterpret_cast<float*>(p + ck);
  float* part_dC = reinterpret_cast<float*>(p + ck + pbc);
  float* part_dA = reinterpret_cast<float*>(p + ck + 2 * pbc);
  float* part_dD = reinterpret_cast<float*>(p + ck + 2 * pbc + pa);
  float* part_db = reinterpret_cast<float*>(p + ck + 2 * pbc + pa + pd);
  const int64_t lanes = a.batch * a.dim * kBG;
  bwd_ckpt_kernel<IO, EULER><<<unsigned((lanes + 255) / 256), 256, 0, a.stream>>>(a, n_chunks,
                                                                                 ckpt);
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    dim3 grid(unsigned(n_groups), unsigned(a.batch));
    bwd_chunk_kernel<IO, EULER><<<grid, kBThreads, 0, a.stream>>>(a, n_chunks, ckpt, part_dB,
                                                                  part_dC, part_dA, part_dD,
                                                                  part_db);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    const int64_t total = a.batch * a.L * a.N + a.dim * a.N + 2 * a.dim;
    const unsigned blocks = unsigned(std::min<int64_t>((total + 255) / 256, 148 * 16));
    bwd_reduce_kernel<<<blocks, 256, 0, a.stream>>>(a, n_groups, part_dB, part_dC, part_dA,
                                                    part_dD, part_db);
    e = cudaGetLastError();
  }
  cudaError_t e2 = cudaFreeAsync(ws, a.stream);
  return e != cudaSuccess ? e : e2;
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs& a) {
  if (a.io == Io::F32)
    return a.euler ? launch_bwd_typed<float, true>(a) : launch_bwd_typed<float, false>(a);
  using bf = __nv_bfloat16;
  return a.euler ? launch_bwd_typed<bf, true>(a) : launch_bwd_typed<bf, false>(a);
}

}  // namespace sscan
