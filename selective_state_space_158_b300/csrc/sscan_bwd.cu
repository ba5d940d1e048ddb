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
// Steps:
//   1. checkpoints: the forward kernel (sscan_fwd_ex's path, with its h_ckpt output) writes the
//      state before every 16-step chunk (B * D * N floats per chunk);
//   2. bwd_chunk_kernel: four lanes per channel (four states each); chunks in reverse order. The
//      chunk's per-(step, channel) values (dt, u, softplus slope, dy, gate and its slope) are
//      computed once into a double-buffered shared-memory table from inputs loaded a chunk ahead;
//      the chunk's 16 states are recomputed from its checkpoint in registers, then the adjoint
//      sweeps back through them. Per-channel sums over the four lanes use shuffles. dB and dC
//      sum over channels: each warp reduces its 8 channels with a transposing shuffle
//      reduction into its own shared-memory slot, the CTA adds the slots in warp order, and the
//      CTA's partial is stored per channel group;
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
constexpr int kBThreads = 128;  // three blocks per SM under the 170-register budget
constexpr int kBCh = kBThreads / kBG;  // channels per CTA

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + ex2(-x * kLog2e)); }

template <bool EULER>
__device__ __forceinline__ float factor(float dt, float a2) {
  // a2 = A log2e (zero-order hold) or A (first order)
  return EULER ? fmaf(dt, a2, 1.f) : ex2(fmaf(dt, a2, kEx2ArgShift));
}

// ---- the adjoint sweep over chunks in reverse ------------------------------------------------
// Per (step, channel) values of a chunk, computed once and shared by the channel's four lanes.
enum { kPdt = 0, kPu, kPsx, kPdy, kPgz, kPgp, kPs, kPN };  // kPs: readout's state part
struct BwdSmem {
  static constexpr size_t slot_pro = size_t(kBT) * kBCh * kPN;   // floats
  static constexpr size_t slot_bc = size_t(kBT) * 16;             // floats, each of B and C
  static constexpr size_t slot = slot_pro + 2 * slot_bc;
  static constexpr size_t red = size_t(kBThreads / 32) * kBT * 16;  // per-warp dB / dC slots
  static constexpr size_t bytes = (2 * slot + 2 * red) * sizeof(float);
};

template <typename IO, bool EULER>
__global__ void __launch_bounds__(kBThreads, 3) bwd_chunk_kernel(BwdArgs a, int n_chunks,
                                                                 int n_groups,
                                                                 unsigned* __restrict__ tiles,
                                                                 float* __restrict__ part_dB,
                                                                 float* __restrict__ part_dC,
                                                                 float* __restrict__ part_dA,
                                                                 float* __restrict__ part_dD,
                                                                 float* __restrict__ part_db) {
  extern __shared__ __align__(16) float bsm[];
  float* slots = bsm;                          // [2][slot]
  float* sdB = bsm + 2 * BwdSmem::slot;        // [warp][kBT][16]: per-warp slots, added in warp
  float* sdC = sdB + BwdSmem::red;             // order (no atomics: timing-independent results)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane % kBG, cl = tid / kBG;
  // Persistent blocks: each takes (batch row, channel group) tiles from a counter until none
  // are left, so the last wave does not leave SMs idle.
  __shared__ unsigned s_tile;
  const unsigned n_tiles = unsigned(a.batch) * unsigned(n_groups);
  for (;;) {
  if (tid == 0) s_tile = atomicAdd(tiles, 1u);
  __syncthreads();
  const unsigned tile = s_tile;
  __syncthreads();  // every thread has read the tile before thread 0 fetches the next
  if (tile >= n_tiles) break;
  const int64_t b = tile / unsigned(n_groups);
  const int cg_idx = int(tile % unsigned(n_groups));
  const int64_t d = int64_t(cg_idx) * kBCh + cl;
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

  // Raw inputs of one chunk for this thread: its channel's own steps j = g + 4 i (delta, u, z,
  // dy) and one (step, state) element of B and C. Loaded a chunk ahead, so the loads overlap
  // the previous chunk's work.
  constexpr int kBC = kBT * 16 / kBThreads;  // B / C elements per thread and chunk
  float r_dl[kBT / kBG], r_u[kBT / kBG], r_z[kBT / kBG], r_dy[kBT / kBG], r_B[kBC], r_C[kBC];
  auto prefetch = [&](int ch) {
    const int64_t t0 = int64_t(ch) * kBT;
#pragma unroll
    for (int i = 0; i < kBT / kBG; ++i) {
      const int64_t t = t0 + g + kBG * i;
      const bool tv = live && t < a.L;
      const int64_t idx = (b * a.L + t) * a.dim + d;
      r_dl[i] = tv ? to_f32(dl[idx]) : 0.f;
      r_u[i] = tv ? to_f32(u[idx]) : 0.f;
      r_z[i] = (tv && zz) ? to_f32(zz[idx]) : 0.f;
      r_dy[i] = tv ? to_f32(dy[idx]) : 0.f;
    }
#pragma unroll
    for (int e = 0; e < kBC; ++e) {
      const int idx = tid + e * kBThreads, j = idx / 16, n = idx % 16;
      const int64_t t = t0 + j;
      const bool ok = t < a.L && n < N;
      r_B[e] = ok ? to_f32(Bm[(b * a.L + t) * N + n]) : 0.f;
      r_C[e] = ok ? to_f32(Cm[(b * a.L + t) * N + n]) : 0.f;
    }
  };
  prefetch(n_chunks - 1);

  for (int ch = n_chunks - 1; ch >= 0; --ch) {
    const int64_t t0 = int64_t(ch) * kBT;
    float* sl = slots + size_t(ch & 1) * BwdSmem::slot;
    float* P = sl;                                // [kBT][kBCh][kPN]
    float* Bs = sl + BwdSmem::slot_pro;           // [kBT][16]
    float* Cs = Bs + BwdSmem::slot_bc;
    // The chunk's per-(step, channel) values: dt, u, sigmoid(x) (softplus slope), dy, SiLU(z),
    // SiLU'(z); steps past the end get dt = 0 and dy = 0 (an identity step).
#pragma unroll
    for (int i = 0; i < kBT / kBG; ++i) {
      const int j = g + kBG * i;
      const bool tv = live && t0 + j < a.L;
      const float x = r_dl[i] + bias;
      float* pp = P + (size_t(j) * kBCh + cl) * kPN;
      pp[kPdt] = tv ? (a.softplus ? softplus_f(x) : x) : 0.f;
      pp[kPu] = r_u[i];
      pp[kPsx] = a.softplus ? sigmoid_f(x) : 1.f;
      pp[kPdy] = r_dy[i];
      if (zz) {
        const float sg = sigmoid_f(r_z[i]);
        pp[kPgz] = r_z[i] * sg;
        pp[kPgp] = sg * fmaf(r_z[i], 1.f - sg, 1.f);
      } else {
        pp[kPgz] = 1.f;
        pp[kPgp] = 0.f;
      }
    }
#pragma unroll
    for (int e = 0; e < kBC; ++e) {
      Bs[tid + e * kBThreads] = r_B[e];
      Cs[tid + e * kBThreads] = r_C[e];
    }
    __syncthreads();

    // Recompute the chunk: hist[j] is the state before step t0 + j (hist[kBT]: after the last).
    float hist[kBT + 1][kBK];
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      const int n = g * kBK + k;
      hist[0][k] = (live && n < N) ? a.ckpt[size_t(ch) * ck_stride + size_t(c) * N + n] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kBT; ++j) {
      const float* pp = P + (size_t(j) * kBCh + cl) * kPN;
      const float dt = pp[kPdt], dtu = dt * pp[kPu];
      const float4 bq = *reinterpret_cast<const float4*>(Bs + j * 16 + g * kBK);
      const float4 cq = *reinterpret_cast<const float4*>(Cs + j * 16 + g * kBK);
      const float bv[4] = {bq.x, bq.y, bq.z, bq.w}, cv[4] = {cq.x, cq.y, cq.z, cq.w};
      float sp = 0.f;
#pragma unroll
      for (int k = 0; k < kBK; ++k) {
        hist[j + 1][k] = fmaf(factor<EULER>(dt, a2[k]), hist[j][k], dtu * bv[k]);
        sp = fmaf(cv[k], hist[j + 1][k], sp);
      }
      // The readout's state part summed over the channel's four lanes, kept for the gate's
      // gradient.
      sp += __shfl_xor_sync(0xffffffffu, sp, 1);
      sp += __shfl_xor_sync(0xffffffffu, sp, 2);
      if (g == 0) P[(size_t(j) * kBCh + cl) * kPN + kPs] = sp;
    }
    __syncwarp();
    if (ch > 0) prefetch(ch - 1);  // the next chunk's inputs, overlapping the adjoint sweep
    // Adjoint sweep back through the chunk.
    float* wB = sdB + size_t(warp) * kBT * 16;
    float* wC = sdC + size_t(warp) * kBT * 16;
#pragma unroll
    for (int j = kBT - 1; j >= 0; --j) {
      const int64_t t = t0 + j;
      const bool tv = live && t < a.L;
      const float* pp = P + (size_t(j) * kBCh + cl) * kPN;
      const float dt = pp[kPdt], uu = pp[kPu], dyt = pp[kPdy];
      const float ds = dyt * pp[kPgz];
      const float4 bq = *reinterpret_cast<const float4*>(Bs + j * 16 + g * kBK);
      const float4 cq = *reinterpret_cast<const float4*>(Cs + j * 16 + g * kBK);
      const float bv[4] = {bq.x, bq.y, bq.z, bq.w}, cv[4] = {cq.x, cq.y, cq.z, cq.w};
      float ddt = 0.f, dup = 0.f, vB[kBK], vC[kBK];
#pragma unroll
      for (int k = 0; k < kBK; ++k) {
        const float fa = factor<EULER>(dt, a2[k]);
        const float lam = fmaf(ds, cv[k], mu[k]);
        const float dfa = EULER ? lam * hist[j][k] : lam * hist[j][k] * fa;
        ddt = fmaf(dfa, Av[k], fmaf(lam * bv[k], uu, ddt));
        dA[k] = fmaf(dfa, dt, dA[k]);
        vB[k] = lam * dt * uu;
        vC[k] = ds * hist[j + 1][k];
        dup = fmaf(lam * dt, bv[k], dup);
        mu[k] = fa * lam;
      }
      // per channel: sum over the four lanes
      ddt += __shfl_xor_sync(0xffffffffu, ddt, 1);
      ddt += __shfl_xor_sync(0xffffffffu, ddt, 2);
      dup += __shfl_xor_sync(0xffffffffu, dup, 1);
      dup += __shfl_xor_sync(0xffffffffu, dup, 2);
      if (tv && g == 0) {
        const int64_t i = (b * a.L + t) * a.dim + d;
        const float dx = ddt * pp[kPsx];
        store_io(static_cast<IO*>(a.du) + i, fmaf(ds, Dd, dup));
        store_io(static_cast<IO*>(a.ddelta) + i, dx);
        if (zz) store_io(static_cast<IO*>(a.dz) + i, dyt * fmaf(Dd, uu, pp[kPs]) * pp[kPgp]);
        dbias += dx;
        dD = fmaf(ds, uu, dD);
      }
      // dB, dC: sum over the warp's 8 channels (lanes with the same g) by a transposing
      // reduction: each round halves the values a lane keeps, so after three rounds lane
      // (channel bits b0 b1 b2) holds the full sum of value q = 4 b0 + 2 b1 + b2 of
      // {dB[0..3], dC[0..3]}, and writes it to the warp's slot.
      {
        const bool b0 = (lane & 4) != 0, b1 = (lane & 8) != 0, b2 = (lane & 16) != 0;
        float r1[4], r2[2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float keep = b0 ? vC[i] : vB[i], send = b0 ? vB[i] : vC[i];
          r1[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float keep = b1 ? r1[2 + i] : r1[i], send = b1 ? r1[i] : r1[2 + i];
          r2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        const float keep = b2 ? r2[1] : r2[0], send = b2 ? r2[0] : r2[1];
        const float r3 = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        (b0 ? wC : wB)[j * 16 + g * kBK + (b1 ? 2 : 0) + (b2 ? 1 : 0)] = r3;
      }
    }
    __syncthreads();
    // The CTA's partial of this chunk (warp slots added in order) to its channel group's slice.
#pragma unroll
    for (int e = 0; e < kBC; ++e) {
      const int idx = tid + e * kBThreads, j = idx / 16, n = idx % 16;
      const int64_t t = t0 + j;
      if (t < a.L && n < N) {
        float sb = 0.f, sc = 0.f;
#pragma unroll
        for (int w = 0; w < kBThreads / 32; ++w) {
          sb += sdB[(size_t(w) * kBT + j) * 16 + n];
          sc += sdC[(size_t(w) * kBT + j) * 16 + n];
        }
        const size_t o = size_t(cg_idx) * part_stride + (size_t(b) * a.L + t) * 16 + n;
        part_dB[o] = sb;
        part_dC[o] = sc;
      }
    }
    __syncthreads();  // warp slots and this chunk's table are reused two chunks on
  }
  if (live) {
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
  }  // tiles
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
  static_assert((kBT * 16) % kBThreads == 0, "whole B / C elements per thread and chunk");
  const int n_chunks = int((a.L + kBT - 1) / kBT);
  const int n_groups = int((a.dim + kBCh - 1) / kBCh);
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t pbc = up(size_t(n_groups) * a.batch * a.L * 16 * sizeof(float));
  const size_t pa = up(size_t(a.batch) * a.dim * a.N * sizeof(float));
  const size_t pd = up(size_t(a.batch) * a.dim * sizeof(float));
  void* ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, 2 * pbc + pa + 2 * pd + 256, a.stream);
  if (e != cudaSuccess) return e;
  char* p = static_cast<char*>(ws);
  float* part_dB = reinterpret_cast<float*>(p);
  float* part_dC = reinterpret_cast<float*>(p + pbc);
  float* part_dA = reinterpret_cast<float*>(p + 2 * pbc);
  float* part_dD = reinterpret_cast<float*>(p + 2 * pbc + pa);
  float* part_db = reinterpret_cast<float*>(p + 2 * pbc + pa + pd);
  unsigned* tiles = reinterpret_cast<unsigned*>(p + 2 * pbc + pa + 2 * pd);
  e = cudaMemsetAsync(tiles, 0, sizeof(unsigned), a.stream);
  auto kern = bwd_chunk_kernel<IO, EULER>;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(BwdSmem::bytes));
  int per_sm = 0, sms = 0, dev = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBThreads, BwdSmem::bytes);
  if (e == cudaSuccess) {
    const int64_t n_tiles = int64_t(n_groups) * a.batch;
    const unsigned grid = unsigned(std::max<int64_t>(
        1, std::min<int64_t>(n_tiles, int64_t(std::max(per_sm, 1)) * sms)));
    kern<<<grid, kBThreads, BwdSmem::bytes, a.stream>>>(a, n_chunks, n_groups, tiles, part_dB,
                                                        part_dC, part_dA, part_dD, part_db);
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
