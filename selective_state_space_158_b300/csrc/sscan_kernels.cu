// sscan_kernels.cu -- the selective-scan forward kernels for sm_103a and their launchers.
//
// The scan follows "Mamba：选择性状态空间模型入门教程" (selective-scan pseudo-code: B_t, C_t and
// Delta_t from the input, h_t = discretize_A(Delta) h_{t-1} + discretize_B(Delta, B) x_t,
// y_t = C h_t), with the zero-order-hold A of "架构变体：Mamba/SSM" ("离散化") and the fusion
// principle of its "硬件感知算法" section: the N-wide state of every channel lives in registers
// for the whole sequence and only inputs and outputs touch HBM.
//
// Two kernels:
//   * sscan_tma_kernel: the fast path. A CTA owns CH consecutive channels of one batch row and
//     walks the sequence in chunks of TC steps. One thread streams the chunk's u/delta/z tiles
//     and B/C rows into shared memory with TMA (double-buffered, mbarrier-tracked); all threads
//     then turn (delta, u) into (dt, dt*u) once per (step, channel); then every lane advances its
//     share of the 16 states through the chunk with ex2 on the SFU and packed f32x2 FMAs, the
//     lanes of one channel combine their partial readouts, and the gated result goes back to HBM
//     through a TMA store.
//   * sscan_simple_kernel: one thread per channel with plain loads; serves any alignment, any
//     dim and any N <= 16.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include <cudaTypedefs.h>

#include "sscan_device.cuh"
#include "sscan_internal.h"

namespace sscan {

constexpr int kNP = 16;          // states held per channel (N <= 16 is zero-padded to 16)

// ================================================================================================
// Plain-load kernel: one thread per (batch row, channel), states in registers, sequential in t.
// ================================================================================================
template <typename IO, bool EULER>
__global__ void __launch_bounds__(128) sscan_simple_kernel(
    const IO* __restrict__ u, const IO* __restrict__ delta, const float* __restrict__ A,
    const IO* __restrict__ Bm, const IO* __restrict__ Cm, const float* __restrict__ Dskip,
    const IO* __restrict__ z, const float* __restrict__ bias, int softplus,
    const float* __restrict__ h0, IO* __restrict__ y, float* __restrict__ h_last,
    float* __restrict__ h_ckpt, int64_t batch, int64_t L, int64_t dim, int N) {
  const int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= batch * dim) return;
  const int64_t b = c / dim, d = c - b * dim;
  float A2[kNP], h[kNP];
#pragma unroll
  for (int n = 0; n < kNP; ++n) {
    A2[n] = n < N ? A[d * N + n] * (EULER ? 1.f : kLog2e) : 0.f;
    h[n] = (h0 && n < N) ? h0[c * N + n] : 0.f;
  }
  const float bs = bias ? bias[d] : 0.f;
  const float Dd = Dskip ? Dskip[d] : 0.f;
  // fp32 zero-order hold: the decay over every 16-step block is re-anchored (see
  // sscan_lane_kernel): hs is the block's start state, R the product of its per-step factors,
  // S its summed step.
  constexpr bool kAnchor = std::is_same<IO, float>::value && !EULER;
  float hs[kAnchor ? kNP : 1], R[kAnchor ? kNP : 1], S = 0.f;
  for (int64_t t = 0; t < L; ++t) {
    if (kAnchor && t % 16 == 0) {
#pragma unroll
      for (int n = 0; n < (kAnchor ? kNP : 1); ++n) {
        hs[n] = h[n];
        R[n] = 1.f;
      }
      S = 0.f;
    }
    if (h_ckpt && t % 16 == 0) {  // the state before every 16-step chunk (backward pass)
      float* dst = h_ckpt + ((t / 16) * batch * dim + c) * N;
#pragma unroll
      for (int n = 0; n < kNP; ++n)
        if (n < N) dst[n] = h[n];
    }
    const int64_t idx = (b * L + t) * dim + d;
    const float x = to_f32(delta[idx]) + bs;
    const float dt = softplus ? softplus_f(x) : x;
    const float uu = to_f32(u[idx]);
    const float dtu = dt * uu;
    const IO* Bt = Bm + (b * L + t) * N;
    const IO* Ct = Cm + (b * L + t) * N;
    float acc = 0.f;
#pragma unroll
    for (int n = 0; n < kNP; ++n) {
      if (n < N) {
        const float e = EULER ? fmaf(dt, A2[n], 1.f) : ex2(dt * A2[n]);
        h[n] = fmaf(e, h[n], dtu * to_f32(Bt[n]));
        acc = fmaf(to_f32(Ct[n]), h[n], acc);
        if constexpr (kAnchor) R[n] *= e;
      }
    }
    if constexpr (kAnchor) {
      S += dt;
      if (t % 16 == 15 || t == L - 1) {  // end of a block: its decay from the summed step
#pragma unroll
        for (int n = 0; n < kNP; ++n) h[n] = fmaf(exp2_acc(A2[n] * S) - R[n], hs[n], h[n]);
      }
    }
    float yv = fmaf(Dd, uu, acc);
    if (z) yv *= silu_f(to_f32(z[idx]));
    store_io(y + idx, yv);
  }
  if (h_last) {
#pragma unroll
    for (int n = 0; n < kNP; ++n)
      if (n < N) h_last[c * N + n] = h[n];
  }
}

__host__ __device__ inline size_t align128(size_t x) { return (x + 127) & ~size_t(127); }

// ================================================================================================
// Lane-owned kernel. Every lane owns one channel's K = 16 / G states (G = 1 or 2 lanes per
// channel); a warp owns 32 / G whole channels, and does its prologue (softplus), recurrence,
// readout, skip, gate and y store for them without leaving registers. The CTA shares only the
// TMA-staged input tiles, including the fp32 B / C rows (16 states, zero-padded) that every lane
// reads as broadcast 16-byte loads. Warps never wait for each other: each counts itself out of a
// stage when it has read it, and the last warp to do so issues the stage's refill.
//
// Long sequences are split into n_seg time segments run by different CTAs ("chunk carry"). The
// scan operator (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2) is associative ("架构变体：Mamba/SSM",
// "硬件感知算法": the update can be evaluated as a tree), so a segment is summarised by its
// aggregate: the end state from a zero start, H, and its decay over the segment, 2^(A log2e SD)
// with SD its summed step (exact for a product of zero-order-hold factors). A segment CTA
//   1. runs pass 1 over its steps (no readout) to its aggregate (segment 0 from its true start
//      state h0, so its pass 1 ends on its inclusive prefix);
//   2. waits for the inclusive prefix of segment s - 1 (its true start state h_in), publishes
//      its own inclusive prefix 2^(A log2e SD) h_in + H for segment s + 1 (a decoupled
//      look-back of depth one: each segment folds exactly one aggregate onto its predecessor's
//      prefix, a fixed association, so the result is deterministic);
//   3. runs pass 2 from h_in with readout, gate and stores.
// CTAs take segment numbers from an atomic ticket in launch order, segment-major, so every CTA
// they wait on is already resident or finished, and a segment's predecessor publishes right
// after its own pass 1 and wait; every wait is bounded and reports a timeout through the device
// status word instead of hanging.
// ================================================================================================
struct LaneParams {
  const float* A;
  const float* D;
  const float* bias;
  const float* h0;       // initial state (batch, dim, N), or null for zero
  float* h_last;
  float* h_ckpt;         // state before every 16-step chunk [n_chunks][batch][dim][N], or null
  unsigned int* status;
  int L, dim, N, batch;
  int softplus, has_z;
  int n_chunks;    // chunks covering L
  int stages;      // TMA pipeline depth
  int n_cg;        // CTAs (channel groups) per batch row
  int n_seg;       // time segments (1: no chunk carry)
  int seg_chunks;  // chunks per segment
  // chunk-carry workspace (n_seg > 1)
  unsigned int* ticket;  // zero at launch
  unsigned int* flags;   // [n_seg][batch][n_cg][W] warp units: inclusive prefix published
  float* agg;            // [unit][lane][2K]: the segment's inclusive prefix (K states)
  int skip_publish;      // test hook: this segment never publishes (-1: off)
};

constexpr unsigned kFlagAgg = 1;
constexpr unsigned kErrCarry = 1u << 5;         // status bit: a look-back wait ran out
constexpr uint32_t kLookbackTries = 1u << 21;  // x ~0.5 us sleep: about a second

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
constexpr uint32_t kTsLookbackTries = 1u << 26;  // a cap beside the one-second time bound
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct LaneSmem {
  size_t tile_io, bc_f32, stage, off_stage, off_y, y_warp, off_tab, tab_warp, off_bar, total;
  // share: a per-warp [TC][CPW] table of (dt, dt u) pairs that the lanes of a channel share.
  __host__ __device__ LaneSmem(int TC, int W, int CPW, int es, int stages, bool share) {
    const int CH = W * CPW;
    tile_io = align128(size_t(TC) * CH * es);
    bc_f32 = align128(size_t(TC) * kNP * sizeof(float));
    stage = 3 * tile_io + 2 * bc_f32;  // u, delta, z (io); B, C (fp32, 16 states)
    off_stage = 0;
    y_warp = align128(size_t(TC) * CPW * es);            // one warp's y tile
    off_y = size_t(stages) * stage;
    off_tab = off_y + size_t(2) * W * y_warp;            // [2][W] y tiles
    tab_warp = share ? align128(size_t(TC) * CPW * 8) : 0;
    off_bar = off_tab + size_t(W) * tab_warp;
    total = off_bar + 8 * 8 + 8 * 4 + 16;                // full[8], done[8], ticket
  }
};

// Cross-lane transpose-reduce of per-step partial readouts: on entry every lane of a channel's
// G-lane group holds its partial sum for all TC steps; on exit lane g holds the full readout of
// the steps t = g + G k (k = 0 .. TC/G - 1) in out[k]. One shuffle per value and round.
template <int G, int TC>
__device__ __forceinline__ void reduce_transpose(const float (&ys)[TC], float (&out)[TC / G],
                                                 int g) {
  if constexpr (G == 1) {
#pragma unroll
    for (int k = 0; k < TC; ++k) out[k] = ys[k];
  } else if constexpr (G == 2) {
#pragma unroll
    for (int k = 0; k < TC / 2; ++k) {
      const float lo = ys[2 * k], hi = ys[2 * k + 1];
      out[k] = (g ? hi : lo) + __shfl_xor_sync(0xffffffffu, g ? lo : hi, 1);
    }
  } else {
    static_assert(G == 4, "G must be 1, 2 or 4");
    // The exchange with lane ^ 2 keeps the steps whose bit 1 matches g's; the one with lane ^ 1
    // the ones whose bit 0 does.
    const bool hi2 = (g & 2) != 0, hi1 = (g & 1) != 0;
    float r1[TC / 2];
#pragma unroll
    for (int m = 0; m < TC / 2; ++m) {
      const int t0 = (m >> 1) * 4 + (m & 1), t1 = t0 + 2;
      r1[m] = (hi2 ? ys[t1] : ys[t0]) + __shfl_xor_sync(0xffffffffu, hi2 ? ys[t0] : ys[t1], 2);
    }
#pragma unroll
    for (int k = 0; k < TC / 4; ++k) {
      const float lo = r1[2 * k], hi = r1[2 * k + 1];
      out[k] = (hi1 ? hi : lo) + __shfl_xor_sync(0xffffffffu, hi1 ? lo : hi, 1);
    }
  }
}

__device__ __forceinline__ unsigned atom_add_acq_rel_shared(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_addr(p)), "r"(v)
               : "memory");
  return old;
}

// Launch bounds: up to 256 threads and 255 registers with one lane per channel (its 16 states
// and the chunk's steps need them); with two or four lanes per channel there are more warps to
// keep resident: 128-thread CTAs at 128 registers (four per SM; 170 and three per SM for fp32
// io) with two lanes, at most 128
// registers with four lanes and 16-step chunks, and 128-thread CTAs at 170 registers (three per
// SM) with four lanes and 32-step chunks.
template <int G, int TC>
__host__ __device__ constexpr int lane_max_threads() {
  return ((G == 4 && TC == 32) || G == 2) ? 128 : 256;
}
template <typename IO, int G, int TC>
__host__ __device__ constexpr int lane_min_blocks() {
  // two lanes, fp32 io: the re-anchoring registers need 170 (three CTAs per SM)
  return G == 4 ? (TC == 32 ? 3 : 2) : (G == 2 ? (std::is_same<IO, float>::value ? 3 : 4) : 1);
}

template <typename IO, int G, int TC, bool EULER, bool CKPT>
__global__ void __launch_bounds__(lane_max_threads<G, TC>(), lane_min_blocks<IO, G, TC>())
    sscan_lane_kernel(
    const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
    const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
    const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_y,
    const LaneParams p) {
  constexpr int K = kNP / G;     // states per lane
  constexpr int KP = K / 2;      // float2 state registers per lane (states n, n+1 packed)
  constexpr int CPW = 32 / G;    // channels per warp
  static_assert(G == 1 || G == 2 || G == 4, "G must be 1, 2 or 4");
  static_assert(TC % 2 == 0, "chunk must be even");
  // Decay factor of one step: 2^(dt * A log2e) on the SFU (zero-order hold), or 1 + dt * A (first
  // order). A2 holds A log2e or A accordingly; kArg is the addend of the FMA.
  constexpr float kScaleA = EULER ? 1.f : kLog2e;
  constexpr float kArg = EULER ? 1.f : 0.f;
  // fp32 io with the zero-order hold re-anchors the decay every 16 steps: the state's component
  // carried in from before a 16-step window is decayed by 2^(A log2e S), S the window's summed
  // step, computed accurately on the FMA pipe (exp2_acc2), instead of by the product R of the
  // window's per-step SFU factors: h_end += (2^(A log2e S) - R) h_start. The SFU's rounding (on
  // this hardware a third of an ulp low on average for the scan's arguments) then compounds over
  // at most 16 steps, not over the state's whole memory (hundreds to thousands of steps for
  // small dt). It costs one FMUL per update (R) and one accurate exponential per state and
  // window. bf16 io keeps the plain SFU product: its tolerance admits that rounding.
  constexpr bool kAnchor = std::is_same<IO, float>::value && !EULER;
  constexpr bool kBf16Io = !std::is_same<IO, float>::value;  // shorter softplus polynomial
  constexpr int kAnchorW = 16;  // re-anchoring window, steps (TC is a multiple of it)
  static_assert(TC % kAnchorW == 0, "chunk must hold whole re-anchoring windows");
  auto decay = [](float2 arg) -> float2 {
    if constexpr (EULER)
      return arg;
    else
      return f2(ex2(arg.x), ex2(arg.y));
  };
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);

  const int tid = threadIdx.x, nthr = blockDim.x;
  const int W = nthr >> 5, CH = W * CPW;
  const int N = p.N, S = p.stages;
  const LaneSmem lay(TC, W, CPW, int(sizeof(IO)), S, G >= 2);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.off_bar);
  unsigned* done = reinterpret_cast<unsigned*>(smem + lay.off_bar + 8 * 8);
  unsigned* s_ticket = done + 8;

  // ---- which work this CTA does: channel group, batch row, time segment ----
  int cgi, b, seg;
  if (p.n_seg == 1) {
    cgi = blockIdx.x;
    b = blockIdx.y;
    seg = 0;
  } else {
    if (tid == 0) *s_ticket = atomicAdd(p.ticket, 1u);
    __syncthreads();
    const unsigned t = *s_ticket;  // segment-major: every earlier segment got an earlier ticket
    const unsigned per_seg = unsigned(p.batch) * unsigned(p.n_cg);
    seg = int(t / per_seg);
    b = int((t % per_seg) / unsigned(p.n_cg));
    cgi = int(t % unsigned(p.n_cg));
  }
  const int ch0 = cgi * CH;
  const int c_begin = seg * p.seg_chunks;
  const int c_end = min(c_begin + p.seg_chunks, p.n_chunks);
  const int nch = c_end - c_begin;
  // Pass 1 (aggregate only) runs for every segment that has a successor.
  const bool agg_pass = p.n_seg > 1 && seg + 1 < p.n_seg;
  const int passes = agg_pass ? 2 : 1;
  const int n_loads = passes * nch;

  auto stage_ptr = [&](int s, int which) -> unsigned char* {  // 0 u, 1 delta, 2 z, 3 B, 4 C
    unsigned char* base = smem + lay.off_stage + size_t(s) * lay.stage;
    return which < 3 ? base + size_t(which) * lay.tile_io
                     : base + 3 * lay.tile_io + size_t(which - 3) * lay.bc_f32;
  };
  const uint32_t tile_bytes = uint32_t(TC) * CH * sizeof(IO);
  const uint32_t bc_bytes = uint32_t(TC) * kNP * sizeof(float);
  const uint32_t stage_bytes = (p.has_z ? 3u : 2u) * tile_bytes + 2u * bc_bytes;
  // Load q (0 .. n_loads-1) brings chunk c_begin + q % nch into stage s = q % S (the caller
  // passes s; loads past the first pass wrap around to the segment's first chunk).
  auto issue_load = [&](int q, int s) {
    const int t0 = (c_begin + (q < nch ? q : q - nch)) * TC;
    mbar_arrive_expect_tx(&full[s], stage_bytes);
    tma_load_3d(stage_ptr(s, 0), &tm_u, ch0, t0, b, &full[s]);
    tma_load_3d(stage_ptr(s, 1), &tm_dl, ch0, t0, b, &full[s]);
    if (p.has_z) tma_load_3d(stage_ptr(s, 2), &tm_z, ch0, t0, b, &full[s]);
    tma_load_3d(stage_ptr(s, 3), &tm_B, 0, t0, b, &full[s]);
    tma_load_3d(stage_ptr(s, 4), &tm_C, 0, t0, b, &full[s]);
  };
  // A warp done with stage s (load q) counts itself out; the last of the W warps refills it
  // with load q + S. The acquire-release count orders every warp's reads of the stage before
  // the refill's TMA writes.
  auto release_stage = [&](int s, int q) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0 && atom_add_acq_rel_shared(&done[s], 1u) == unsigned(W - 1)) {
      done[s] = 0;
      if (q + S < n_loads) {
        fence_smem_to_async();
        issue_load(q + S, s);
      }
    }
  };
  if (tid == 0) {
    tma_prefetch_desc(&tm_u);
    tma_prefetch_desc(&tm_dl);
    if (p.has_z) tma_prefetch_desc(&tm_z);
    tma_prefetch_desc(&tm_B);
    tma_prefetch_desc(&tm_C);
    tma_prefetch_desc(&tm_y);
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      done[s] = 0;
    }
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0)
    for (int q = 0; q < S && q < n_loads; ++q) issue_load(q, q);

  const int warp = tid >> 5, lane = tid & 31;
  const int cl = warp * CPW + lane / G;  // channel within the CTA
  const int g = lane % G;                // which half of the states (G == 2)
  const int n0 = g * K;
  const int cg = ch0 + cl;               // global channel
  const bool live = cg < p.dim;
  float2 A2[KP], h[KP], hz[KP];
  // The initial state, read once before anything is written (so h0 may alias h_last). It is
  // the start state of segment 0 (of the only segment when the sequence is not split).
  const float* h0c = (p.h0 && live) ? p.h0 + (size_t(b) * p.dim + cg) * N : nullptr;
#pragma unroll
  for (int r = 0; r < KP; ++r) {
    const int n = n0 + 2 * r;
    A2[r] = f2((live && n < N) ? p.A[size_t(cg) * N + n] * kScaleA : 0.f,
               (live && n + 1 < N) ? p.A[size_t(cg) * N + n + 1] * kScaleA : 0.f);
    hz[r] = f2((h0c && n < N) ? h0c[n] : 0.f, (h0c && n + 1 < N) ? h0c[n + 1] : 0.f);
    h[r] = seg == 0 ? hz[r] : f2(0.f, 0.f);
  }
  float2 Pr[EULER ? KP : 1];  // first order: product of this segment's decay factors (pass 1)
#pragma unroll
  for (int r = 0; r < (EULER ? KP : 1); ++r) Pr[r] = f2(1.f, 1.f);
  const float bias_c = (p.bias && live) ? p.bias[cg] : 0.f;
  const float D_c = (p.D && live) ? p.D[cg] : 0.f;
  IO* ywarp0 = reinterpret_cast<IO*>(smem + lay.off_y) + size_t(warp) * (lay.y_warp / sizeof(IO));

  bool timed_out = false;
  float sd = 0.f, sd_c = 0.f;  // Kahan sum of this segment's steps (pass 1)
  int q = 0;                   // loads consumed
  int s = 0;                   // its stage, q % S
  uint32_t phase = 0;          // parity of the stage's fill, (q / S) & 1
  int ystores = 0;             // y tiles this warp has stored
  const size_t unit = ((size_t(seg) * p.batch + b) * p.n_cg + cgi) * W + warp;
  const size_t units_per_seg = size_t(p.batch) * p.n_cg * W;
  for (int pass = agg_pass ? 0 : 1; pass < 2 && !timed_out; ++pass) {
    const bool readout = pass == 1;
    if (readout && p.n_seg > 1) {
      // Chunk carry between segments. Segment 0 knows its start state (h0 or zero), so its
      // first pass ended on its true end state: its inclusive prefix. Segment s > 0 waits for
      // segment s - 1's inclusive prefix (its start state), and, if it has a successor, folds
      // its own aggregate onto it and publishes its inclusive prefix:
      //   incl_s = P_s incl_{s-1} + H_s,   P_s = 2^(A log2e SD_s) (zero-order hold; SD_s the
      //   segment's summed step) or the product of its factors (first order).
      // The association is fixed (always one segment onto its predecessor's prefix), so the
      // result is deterministic, and one wait per segment suffices.
      float2 start[KP];
      if (seg == 0) {
#pragma unroll
        for (int r = 0; r < KP; ++r) start[r] = hz[r];
      } else {
        const size_t up = unit - units_per_seg;  // the same lanes of segment s - 1
        unsigned f = 0;
        if (lane == 0) {
          for (uint32_t it = 0; it < kLookbackTries; ++it) {
            f = ld_acquire(p.flags + up);
            if (f != 0) break;
            __nanosleep(512);
          }
          if (f == 0) atomicOr(p.status, kErrCarry);
        }
        f = __shfl_sync(0xffffffffu, f, 0);
        __syncwarp();
        const float* a = p.agg + (up * 32 + lane) * (2 * K);
#pragma unroll
        for (int r = 0; r < KP; ++r)  // timed out: zero (the status word says the result is wrong)
          start[r] = f != 0 ? f2(__ldcg(a + 2 * r), __ldcg(a + 2 * r + 1)) : f2(0.f, 0.f);
      }
      if (agg_pass && !timed_out && seg != p.skip_publish) {
        float* my = p.agg + (unit * 32 + lane) * (2 * K);
#pragma unroll
        for (int r = 0; r < KP; ++r) {
          float2 incl = h[r];  // segment 0: the end state from h0 already
          if (seg > 0) {
            float2 P;
            if constexpr (EULER)
              P = Pr[r];
            else if constexpr (kAnchor)
              P = exp2_acc2(__fmul2_rn(A2[r], f2(sd, sd)));
            else
              P = f2(ex2(A2[r].x * sd), ex2(A2[r].y * sd));
            incl = __ffma2_rn(P, start[r], h[r]);
          }
          my[2 * r] = incl.x;
          my[2 * r + 1] = incl.y;
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release(p.flags + unit, kFlagAgg);
      }
#pragma unroll
      for (int r = 0; r < KP; ++r) h[r] = start[r];
    }
    for (int ci = 0; ci < nch; ++ci, ++q, s = (s + 1 == S) ? 0 : s + 1, phase ^= (s == 0)) {
      const int c = c_begin + ci;
      const int t0 = c * TC;
      const int t_valid = min(TC, p.L - t0);
      const bool landed = mbar_wait_bounded(&full[s], phase, kWaitNs);
      if (__any_sync(0xffffffffu, !landed)) {  // warp-uniform: the whole warp leaves
        timed_out = true;
        break;
      }

      if (CKPT && readout && live) {  // the state before this chunk (backward pass)
        float* dst = p.h_ckpt + ((size_t(c) * p.batch + b) * p.dim + cg) * N;
        if (KP % 2 == 0 && (N & 3) == 0) {  // 16-byte stores: n0 and N are multiples of 4
#pragma unroll
          for (int r = 0; r + 1 < KP; r += 2)
            if (n0 + 2 * r < N)
              *reinterpret_cast<float4*>(dst + n0 + 2 * r) =
                  make_float4(h[r].x, h[r].y, h[r + 1].x, h[r + 1].y);
        } else {
#pragma unroll
          for (int r = 0; r < KP; ++r) {
            const int n = n0 + 2 * r;
            if (n < N) dst[n] = h[r].x;
            if (n + 1 < N) dst[n + 1] = h[r].y;
          }
        }
      }
      const IO* u_s = reinterpret_cast<const IO*>(stage_ptr(s, 0)) + cl;
      const IO* dl_s = reinterpret_cast<const IO*>(stage_ptr(s, 1)) + cl;
      const IO* z_s = reinterpret_cast<const IO*>(stage_ptr(s, 2)) + cl;
      const float* Bs = reinterpret_cast<const float*>(stage_ptr(s, 3));
      const float* Cs = reinterpret_cast<const float*>(stage_ptr(s, 4));

      // Prologue: dt = softplus(delta + bias) and dt * u, two steps at a time in f32x2. With one
      // lane per channel the lane computes all TC steps; with G = 2 or 4 lanes, lane g computes
      // only its own steps t = g + G k and publishes them in a per-warp table that the channel's
      // lanes read. Steps past the end of the sequence get dt = 0, an identity update. uo keeps
      // u of this lane's own output steps for the skip term.
      constexpr int OWN = TC / G;
      constexpr bool kShare = G >= 2;        // lanes of a channel split the prologue
      constexpr bool kScalarArgs = G == 4;   // dt, dt u kept as scalars (registers)
      constexpr int NP = kShare ? OWN : TC;  // steps this lane computes
      float own_dt[NP], own_du[NP], own_u[NP], uo[OWN];
      auto prologue = [&](auto with_softplus, auto masked) {
#pragma unroll
        for (int k = 0; k < NP; k += 2) {
          const int ta = kShare ? g + G * k : k, tb = kShare ? ta + G : k + 1;
          const float2 u2 = f2(to_f32(u_s[ta * CH]), to_f32(u_s[tb * CH]));
          float2 d2 = __fadd2_rn(f2(to_f32(dl_s[ta * CH]), to_f32(dl_s[tb * CH])),
                                 f2(bias_c, bias_c));
          if constexpr (decltype(with_softplus)::value) d2 = softplus2<kBf16Io>(d2);
          if constexpr (decltype(masked)::value)  // the sequence's last chunk only
            d2 = f2(ta < t_valid ? d2.x : 0.f, tb < t_valid ? d2.y : 0.f);
          const float2 du = __fmul2_rn(d2, u2);
          own_dt[k] = d2.x;
          own_dt[k + 1] = d2.y;
          own_du[k] = du.x;
          own_du[k + 1] = du.y;
          own_u[k] = u2.x;
          own_u[k + 1] = u2.y;
        }
      };
      // One branch per chunk on the softplus flag and on whether the chunk runs past the end
      // of the sequence, instead of tests per step pair.
      if (t_valid == TC) {
        if (p.softplus)
          prologue(std::true_type{}, std::false_type{});
        else
          prologue(std::false_type{}, std::false_type{});
      } else {
        if (p.softplus)
          prologue(std::true_type{}, std::true_type{});
        else
          prologue(std::false_type{}, std::true_type{});
      }
      // The summed step of every re-anchoring window (kAnchorW steps): each lane sums the
      // window's steps it computed; with G lanes per channel the partial sums are combined by
      // log2 G exchanges, which give all G lanes the same value (the additions see the same
      // operands in every lane).
      constexpr int NWIN = kAnchor ? TC / kAnchorW : 1;
      float S_win[NWIN];
#pragma unroll
      for (int wi = 0; wi < NWIN; ++wi) S_win[wi] = 0.f;
      if constexpr (kAnchor) {
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          const int t = kShare ? g + G * k : k;  // the step own_dt[k] belongs to
          S_win[t / kAnchorW] += own_dt[k];
        }
        if constexpr (kShare) {
#pragma unroll
          for (int wi = 0; wi < NWIN; ++wi) {
#pragma unroll
            for (int m = 1; m < G; m <<= 1) S_win[wi] += __shfl_xor_sync(0xffffffffu, S_win[wi], m);
          }
        }
      }
      // Window-start state and product of the window's factors (re-anchoring).
      float2 hs[kAnchor ? KP : 1], Rp[kAnchor ? KP : 1];
      auto open_window = [&]() {
#pragma unroll
        for (int r = 0; r < (kAnchor ? KP : 1); ++r) {
          hs[r] = h[r];
          Rp[r] = f2(1.f, 1.f);
        }
      };
      open_window();
      // After step t: at the end of a window, decay its start state by the accurate factor.
      auto reanchor = [&](int t) {
        if constexpr (kAnchor) {
          if (t % kAnchorW == kAnchorW - 1) {
            const float S = S_win[t / kAnchorW];
#pragma unroll
            for (int r = 0; r < KP; ++r) {
              const float2 P = exp2_acc2(__fmul2_rn(A2[r], f2(S, S)));
              h[r] = __ffma2_rn(__fadd2_rn(P, __fmul2_rn(Rp[r], f2(-1.f, -1.f))), hs[r], h[r]);
            }
            open_window();
          }
        }
      };
      // With four lanes per channel dt and dt u stay scalars (scalar FMAs need no duplicated
      // pairs, which leaves registers for longer chunks); otherwise they are duplicated pairs
      // {v, v} for the packed FMAs.
      // G = 1: the lane's own dt, dt u as duplicated pairs {v, v} for the packed FMAs. G > 1:
      // lane g publishes its own steps t = g + G k in the warp's table, and every lane reads
      // each step's (dt, dt u) from it when the step comes (no register copy of the chunk).
      float2 dtp[kShare ? 1 : TC], dtup[kShare ? 1 : TC];
      const float2* tabr = nullptr;
      if constexpr (kShare) {
        float2* tab = reinterpret_cast<float2*>(smem + lay.off_tab + size_t(warp) * lay.tab_warp);
        __syncwarp();  // every lane has read the previous chunk's entries
#pragma unroll
        for (int k = 0; k < OWN; ++k) tab[(g + G * k) * CPW + lane / G] = f2(own_dt[k], own_du[k]);
        __syncwarp();
        tabr = tab + lane / G;
      } else {
#pragma unroll
        for (int t = 0; t < TC; ++t) {
          dtp[t] = f2(own_dt[t], own_dt[t]);
          dtup[t] = f2(own_du[t], own_du[t]);
        }
      }
      // (dt, dt u) of step t.
      auto step_at = [&](int t) -> float2 {
        if constexpr (kShare)
          return tabr[t * CPW];
        else
          return f2(dtp[t].x, dtup[t].x);
      };
      // dA argument and input term of state pair r at step t, given the step's (dt, dt u).
      auto arg_at = [&](float2 v, int t, int r) -> float2 {
        if constexpr (kScalarArgs)
          return f2(fmaf(v.x, A2[r].x, kArg), fmaf(v.x, A2[r].y, kArg));
        else if constexpr (kShare)
          return __ffma2_rn(f2(v.x, v.x), A2[r], f2(kArg, kArg));
        else
          return __ffma2_rn(dtp[t], A2[r], f2(kArg, kArg));
      };
      auto in_at = [&](float2 v, int t, float2 bb) -> float2 {
        if constexpr (kScalarArgs)
          return f2(v.y * bb.x, v.y * bb.y);
        else if constexpr (kShare)
          return __fmul2_rn(f2(v.y, v.y), bb);
        else
          return __fmul2_rn(dtup[t], bb);
      };
#pragma unroll
      for (int k = 0; k < OWN; ++k) {
        if constexpr (kShare || G == 1)
          uo[k] = own_u[k];
        else
          uo[k] = g ? own_u[G * k + 1] : own_u[G * k];
      }

      if (!readout) {
        // Pass 1: state from a zero start, no readout; and the segment's summed step.
        float csum = 0.f;
#pragma unroll
        for (int t = 0; t < TC; ++t) {
          const float4* Bq = reinterpret_cast<const float4*>(Bs + t * kNP + n0);
          const float2 sv = step_at(t);
          csum += sv.x;
#pragma unroll
          for (int qq = 0; qq < K / 4; ++qq) {
            const float4 bq = Bq[qq];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int r = 2 * qq + j;
              const float2 dA = decay(arg_at(sv, t, r));
              const float2 bb = j ? f2(bq.z, bq.w) : f2(bq.x, bq.y);
              h[r] = __ffma2_rn(dA, h[r], in_at(sv, t, bb));
              if constexpr (EULER) Pr[r] = __fmul2_rn(Pr[r], dA);
              if constexpr (kAnchor) Rp[r] = __fmul2_rn(Rp[r], dA);
            }
          }
          reanchor(t);
        }
        release_stage(s, q);
        const float yk = csum - sd_c;  // Kahan step
        const float tk = sd + yk;
        sd_c = (tk - sd) - yk;
        sd = tk;
        continue;
      }

      // Pass 2 (or the only pass): ZOH decay on the SFU, packed f32x2 FMAs for the state and
      // the readout.
      float ys[TC];
#pragma unroll
      for (int t = 0; t < TC; ++t) {
        const float4* Bq = reinterpret_cast<const float4*>(Bs + t * kNP + n0);
        const float4* Cq = reinterpret_cast<const float4*>(Cs + t * kNP + n0);
        const float2 sv = step_at(t);
        // One chain of packed FMAs per step for the readout: the steps of the unrolled chunk
        // are independent, so a longer chain costs no stall and saves the adds of partial sums.
        float2 acc = f2(0.f, 0.f);
#pragma unroll
        for (int qq = 0; qq < K / 4; ++qq) {
          const float4 bq = Bq[qq], cq = Cq[qq];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int r = 2 * qq + j;
            const float2 dA = decay(arg_at(sv, t, r));
            const float2 bb = j ? f2(bq.z, bq.w) : f2(bq.x, bq.y);
            const float2 cc = j ? f2(cq.z, cq.w) : f2(cq.x, cq.y);
            h[r] = __ffma2_rn(dA, h[r], in_at(sv, t, bb));
            acc = __ffma2_rn(cc, h[r], acc);
            if constexpr (kAnchor) Rp[r] = __fmul2_rn(Rp[r], dA);
          }
        }
        ys[t] = acc.x + acc.y;
        reanchor(t);
      }

      // Epilogue on this lane's own steps, two at a time: (readout + D u) * SiLU(z) into the
      // warp's y tile. With G > 1 the lanes of a channel first combine their partial readouts
      // so that lane g holds the full readout of its steps t = g + G k.
      if (lane == 0 && ystores >= 2) tma_store_wait_read<1>();  // tile of two stores ago read
      __syncwarp();
      IO* yw = ywarp0 + size_t(ystores & 1) * (size_t(W) * lay.y_warp / sizeof(IO));
      float yo[OWN];
      reduce_transpose<G, TC>(ys, yo, g);
      auto epilogue = [&](auto with_gate) {
#pragma unroll
        for (int k = 0; k < OWN; k += 2) {
          const int ta = g + G * k, tb = ta + G;  // this lane's steps
          float2 y2 = __ffma2_rn(f2(D_c, D_c), f2(uo[k], uo[k + 1]), f2(yo[k], yo[k + 1]));
          if constexpr (decltype(with_gate)::value)
            y2 = __fmul2_rn(y2, silu2(f2(to_f32(z_s[ta * CH]), to_f32(z_s[tb * CH]))));
          store_io(yw + ta * CPW + lane / G, y2.x);
          store_io(yw + tb * CPW + lane / G, y2.y);
        }
      };
      if (p.has_z)  // one branch per chunk
        epilogue(std::true_type{});
      else
        epilogue(std::false_type{});
      fence_smem_to_async();
      release_stage(s, q);  // z was the stage's last use
      if (lane == 0) {
        tma_store_3d(&tm_y, yw, ch0 + warp * CPW, t0, b);
        tma_store_commit();
      }
      ++ystores;
    }
  }

  if (timed_out) {
    if (lane == 0) atomicOr(p.status, kErrTimeout);
  } else if (p.h_last && live && seg == p.n_seg - 1) {
    float* dst = p.h_last + (size_t(b) * p.dim + cg) * N;
#pragma unroll
    for (int r = 0; r < KP; ++r) {
      const int n = n0 + 2 * r;
      if (n < N) dst[n] = h[r].x;
      if (n + 1 < N) dst[n + 1] = h[r].y;
    }
  }
  if (lane == 0) tma_store_wait_all();
  // Loads still in flight (issued for chunks that were never consumed after a timeout) get a
  // bounded chance to land before the CTA's shared memory goes away.
  const int any_timeout = __syncthreads_or(timed_out);
  if (tid == 0 && any_timeout)
    for (int s = 0; s < S && s < n_loads; ++s) mbar_wait_bounded(&full[s], 0, 100000);
}

// ================================================================================================
// Time lanes: the scan over time inside a warp. One warp scans one channel; its 32 lanes are 32
// consecutive stretches of kTsT steps of a kTsChunk-step chunk, each lane holding all 16 states.
// Per chunk:
//   1. every lane runs its kTsT steps from a zero state: its aggregate (P, H), H the end state
//      and P = 2^(A log2e S) the decay over its steps (S their summed step; the product of the
//      factors for the first order);
//   2. the 32 aggregates are composed in order with (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2)
//      ("架构变体：Mamba/SSM", "硬件感知算法": the update is associative), starting from the
//      state the warp carries into the chunk: lane n < 16 walks the 32 aggregates of state n
//      through shared memory and leaves every lane's start state there, and the chunk's end
//      state is the carry into the next chunk;
//   3. every lane runs its kTsT steps again from its true start state, with the readout, skip,
//      gate and stores.
// A CTA is kTsW warps (kTsW consecutive channels: the TMA boxes are kTsChunk steps x kTsW
// channels). Each lane reads a different step, so the staged tiles are first regrouped by the
// whole CTA into layouts where a lane's steps are contiguous (u, delta, z and y channel-major;
// B and C as [quad of states][lane][step + 1 pad] float4) and the warp's accesses hit distinct
// shared-memory banks. Long sequences with few channels are split into time segments joined by
// the same chained carry as the lane kernel: a segment with a successor first runs steps 1-2 over
// all its chunks (its aggregate), then waits for its predecessor's prefix and publishes its own.
// fp32 io composes the lanes with the accurate exponential, so the SFU's rounding compounds over
// at most kTsT steps.
// ================================================================================================
constexpr int kTsT = 8;               // steps per lane and chunk
constexpr int kTsChunk = 32 * kTsT;   // steps per chunk
constexpr int kTsW = 8;               // warps (channels) per CTA
constexpr int kTsPad = kTsT + 1;      // float4 slots per lane and quad of states (one pad)
constexpr int kTsScan = kNP + 4;      // floats per lane of the aggregate rows (16 + pad)

struct TsSmem {
  size_t tile_io, bc, stage, off_t, t_io, off_bt, bt, off_scan, scan_warp, off_y, y_tile, off_bar,
      total;
  __host__ __device__ TsSmem(int es, int stages) {
    tile_io = align128(size_t(kTsChunk) * kTsW * es);      // TMA tile [kTsChunk][kTsW] io
    bc = align128(size_t(kTsChunk) * kNP * sizeof(float));  // TMA tile [kTsChunk][16] fp32
    stage = 3 * tile_io + 2 * bc;                           // u, delta, z; B, C
    off_t = size_t(stages) * stage;                         // u, delta, z as [kTsW][kTsChunk]
    t_io = align128(size_t(kTsW) * kTsChunk * es);          // (y reuses u's: see the kernel)
    off_bt = off_t + 3 * t_io;                              // B, C as [4][32][kTsPad] float4
    bt = align128(size_t(4) * 32 * kTsPad * 4 * sizeof(float));
    off_scan = off_bt + 2 * bt;
    scan_warp = align128(2 * 32 * kTsScan * sizeof(float));  // P, H [32][kTsScan]
    off_y = off_scan + size_t(kTsW) * scan_warp;             // the y tile [kTsChunk][kTsW]
    y_tile = align128(size_t(kTsChunk) * kTsW * es);
    off_bar = off_y + y_tile;
    total = off_bar + 8 * 8;  // full[8]
  }
};

// Eight io values at a 16-byte aligned address (fp32: 32 bytes) to and from floats.
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // element 2i in the low half of word i
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);  // .x the low half
    w[i] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename IO, bool EULER>
__global__ void __launch_bounds__(kTsW * 32, 1)
    sscan_tscan_kernel(const __grid_constant__ CUtensorMap tm_u,
                       const __grid_constant__ CUtensorMap tm_dl,
                       const __grid_constant__ CUtensorMap tm_z,
                       const __grid_constant__ CUtensorMap tm_B,
                       const __grid_constant__ CUtensorMap tm_C,
                       const __grid_constant__ CUtensorMap tm_y, const LaneParams p) {
  constexpr float kScaleA = EULER ? 1.f : kLog2e;
  constexpr float kArg = EULER ? 1.f : 0.f;
  constexpr bool kAccurate = std::is_same<IO, float>::value && !EULER;
  constexpr bool kBf16Io = !std::is_same<IO, float>::value;
  constexpr int KP = kNP / 2;
  auto decay = [](float2 arg) -> float2 {
    if constexpr (EULER)
      return arg;
    else
      return f2(ex2(arg.x), ex2(arg.y));
  };
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int N = p.N, S = p.stages;
  const TsSmem lay(int(sizeof(IO)), S);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.off_bar);
  __shared__ unsigned s_ticket;

  int cgi, b, seg;
  if (p.n_seg == 1) {
    cgi = blockIdx.x;
    b = blockIdx.y;
    seg = 0;
  } else {
    if (tid == 0) s_ticket = atomicAdd(p.ticket, 1u);
    __syncthreads();
    const unsigned t = s_ticket;  // segment-major: every earlier segment got an earlier ticket
    const unsigned per_seg = unsigned(p.batch) * unsigned(p.n_cg);
    seg = int(t / per_seg);
    b = int((t % per_seg) / unsigned(p.n_cg));
    cgi = int(t % unsigned(p.n_cg));
  }
  const int ch0 = cgi * kTsW;
  const int c_begin = seg * p.seg_chunks;
  const int c_end = min(c_begin + p.seg_chunks, p.n_chunks);
  const int nch = c_end - c_begin;
  const bool agg_pass = p.n_seg > 1 && seg + 1 < p.n_seg;
  const int n_loads = (agg_pass ? 2 : 1) * nch;

  auto stage_ptr = [&](int s, int which) -> unsigned char* {  // 0 u, 1 delta, 2 z, 3 B, 4 C
    unsigned char* base = smem + size_t(s) * lay.stage;
    return which < 3 ? base + size_t(which) * lay.tile_io
                     : base + 3 * lay.tile_io + size_t(which - 3) * lay.bc;
  };
  IO* tU = reinterpret_cast<IO*>(smem + lay.off_t);  // [kTsW][kTsChunk]; also y before its store
  IO* tD = reinterpret_cast<IO*>(smem + lay.off_t + lay.t_io);
  IO* tZ = reinterpret_cast<IO*>(smem + lay.off_t + 2 * lay.t_io);
  float4* tB = reinterpret_cast<float4*>(smem + lay.off_bt);  // [4][32][kTsPad]
  float4* tC = reinterpret_cast<float4*>(smem + lay.off_bt + lay.bt);
  const uint32_t tile_bytes = uint32_t(kTsChunk) * kTsW * sizeof(IO);
  const uint32_t bc_bytes = uint32_t(kTsChunk) * kNP * sizeof(float);
  // Load q brings chunk c_begin + q % nch into stage s (the aggregate pass needs no gate z).
  auto issue_load = [&](int q, int s) {
    const bool with_z = p.has_z && !(agg_pass && q < nch);
    const int t0 = (c_begin + (q < nch ? q : q - nch)) * kTsChunk;
    mbar_arrive_expect_tx(&full[s], (with_z ? 3u : 2u) * tile_bytes + 2u * bc_bytes);
    tma_load_3d(stage_ptr(s, 0), &tm_u, ch0, t0, b, &full[s]);
    tma_load_3d(stage_ptr(s, 1), &tm_dl, ch0, t0, b, &full[s]);
    if (with_z) tma_load_3d(stage_ptr(s, 2), &tm_z, ch0, t0, b, &full[s]);
    tma_load_3d(stage_ptr(s, 3), &tm_B, 0, t0, b, &full[s]);
    tma_load_3d(stage_ptr(s, 4), &tm_C, 0, t0, b, &full[s]);
  };
  // Regroups an io tile [kTsChunk][kTsW] into [kTsW][kTsChunk]: thread r takes row r.
  auto regroup_io = [&](const IO* tile, IO* dst) {
    float v[8];
    load8(tile + tid * kTsW, v);
#pragma unroll
    for (int w = 0; w < kTsW; ++w) store_io(dst + w * kTsChunk + tid, v[w]);
  };
  // Regroups a B or C tile [kTsChunk][16] into [quad][lane][step]: float4 (row r, quad q) goes
  // to lane r / kTsT, slot r % kTsT.
  auto regroup_bc = [&](const float* tile, float4* dst) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * (kTsW * 32), r = idx >> 2, qd = idx & 3;
      dst[(qd * 32 + r / kTsT) * kTsPad + r % kTsT] = reinterpret_cast<const float4*>(tile)[idx];
    }
  };
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0)
    for (int q = 0; q < S && q < n_loads; ++q) issue_load(q, q);

  const int cg = ch0 + warp;  // this warp's channel
  const bool live = cg < p.dim;
  float2 A2[KP];
#pragma unroll
  for (int r = 0; r < KP; ++r) {
    const int n = 2 * r;
    A2[r] = f2((live && n < N) ? p.A[size_t(cg) * N + n] * kScaleA : 0.f,
               (live && n + 1 < N) ? p.A[size_t(cg) * N + n + 1] * kScaleA : 0.f);
  }
  const float bias_c = (p.bias && live) ? p.bias[cg] : 0.f;
  const float D_c = (p.D && live) ? p.D[cg] : 0.f;
  // Lane n < 16 carries state n across chunks (and segments); a_n is its A log2e (or A).
  const bool scanner = lane < kNP;
  const float a_n = (live && lane < N) ? p.A[size_t(cg) * N + lane] * kScaleA : 0.f;
  const float hz = (p.h0 && live && lane < N) ? p.h0[(size_t(b) * p.dim + cg) * N + lane] : 0.f;
  float carry = seg == 0 ? hz : 0.f;
  float* scanP = reinterpret_cast<float*>(smem + lay.off_scan + size_t(warp) * lay.scan_warp);
  float* scanH = scanP + 32 * kTsScan;
  IO* ytile = reinterpret_cast<IO*>(smem + lay.off_y);
  const float4* bq_l = tB + lane * kTsPad;  // this lane's B, C slots: quad qd at + qd 32 kTsPad
  const float4* cq_l = tC + lane * kTsPad;

  bool timed_out = false;
  float sd = 0.f, sd_c = 0.f;  // Kahan sum of the segment's steps (aggregate pass)
  float pprod = 1.f;           // first order: product of the segment's factors of state n
  int q = 0, s = 0;
  uint32_t phase = 0;
  int ystores = 0;
  const size_t unit = ((size_t(seg) * p.batch + b) * p.n_cg + cgi) * kTsW + warp;
  const size_t units_per_seg = size_t(p.batch) * p.n_cg * kTsW;
  for (int pass = agg_pass ? 0 : 1; pass < 2 && !timed_out; ++pass) {
    const bool readout = pass == 1;
    if (readout && p.n_seg > 1) {
      // Chunk carry between segments: segment s > 0 waits for segment s - 1's inclusive prefix
      // and, with a successor, publishes its own, 2^(A log2e SD_s) h_in + H_s (the product of
      // its factors for the first order). Each state's prefix is one 64-bit word, its value
      // and a valid bit, stored and read whole (zeroed before the launch), so a lane polls its
      // own word and no fence or separate flag sits on the chain from segment to segment.
      unsigned long long* words = reinterpret_cast<unsigned long long*>(p.agg);
      float start = hz;
      if (seg > 0) {
        const size_t up = unit - units_per_seg;
        bool got = !scanner;
        if (scanner) {  // bounded: about a second of polling
          const uint64_t t_begin = globaltimer_ns();
          for (uint32_t it = 0; it < kTsLookbackTries; ++it) {
            const unsigned long long v = ld_relaxed_u64(words + up * kNP + lane);
            if (v >> 32) {
              start = __uint_as_float(unsigned(v));
              got = true;
              break;
            }
            if (globaltimer_ns() - t_begin > kWaitNs) break;
            __nanosleep(64);
          }
          if (!got) start = 0.f;  // timed out: the status word says the result is wrong
        }
        if (__any_sync(0xffffffffu, !got) && lane == 0) atomicOr(p.status, kErrCarry);
      }
      if (agg_pass && seg != p.skip_publish && scanner) {
        float incl = carry;  // segment 0: the end state from h0 already
        if (seg > 0) {
          float P;
          if constexpr (EULER)
            P = pprod;
          else if constexpr (kAccurate)
            P = exp2_acc(a_n * sd);
          else
            P = ex2(a_n * sd);
          incl = fmaf(P, start, carry);
        }
        st_relaxed_u64(words + unit * kNP + lane,
                       (1ull << 32) | (unsigned long long)__float_as_uint(incl));
      }
      carry = start;
    }
    for (int ci = 0; ci < nch; ++ci, ++q, s = (s + 1 == S) ? 0 : s + 1, phase ^= (s == 0)) {
      const int t0 = (c_begin + ci) * kTsChunk;
      const bool landed = mbar_wait_bounded(&full[s], phase, kWaitNs);
      // CTA-uniform exit; it also orders every warp's reads of the regrouped tiles of the
      // previous chunk before they are overwritten.
      if (__syncthreads_or(!landed)) {
        timed_out = true;
        break;
      }
      regroup_io(reinterpret_cast<const IO*>(stage_ptr(s, 0)), tU);
      regroup_io(reinterpret_cast<const IO*>(stage_ptr(s, 1)), tD);
      if (readout && p.has_z) regroup_io(reinterpret_cast<const IO*>(stage_ptr(s, 2)), tZ);
      regroup_bc(reinterpret_cast<const float*>(stage_ptr(s, 3)), tB);
      if (readout) regroup_bc(reinterpret_cast<const float*>(stage_ptr(s, 4)), tC);
      __syncthreads();  // the stage is consumed; the regrouped tiles are complete
      if (tid == 0 && q + S < n_loads) {
        fence_smem_to_async();
        issue_load(q + S, s);
      }
      const int row0 = lane * kTsT;  // this lane's first step in the chunk
      // The lane's steps: dt = softplus(delta + bias) (0 past the sequence end), dt u, u, and
      // SiLU(z) (1 without gate) for the readout.
      float uo[kTsT], dt[kTsT], du[kTsT], sil[kTsT];
      load8(tU + warp * kTsChunk + row0, uo);
      load8(tD + warp * kTsChunk + row0, dt);
      const int tv = p.L - (t0 + row0);  // this lane's steps inside the sequence
#pragma unroll
      for (int k = 0; k < kTsT; k += 2) {
        float2 d2 = __fadd2_rn(f2(dt[k], dt[k + 1]), f2(bias_c, bias_c));
        if (p.softplus) d2 = softplus2<kBf16Io>(d2);
        d2 = f2(k < tv ? d2.x : 0.f, k + 1 < tv ? d2.y : 0.f);
        const float2 d2u = __fmul2_rn(d2, f2(uo[k], uo[k + 1]));
        dt[k] = d2.x;
        dt[k + 1] = d2.y;
        du[k] = d2u.x;
        du[k + 1] = d2u.y;
        sil[k] = 1.f;
        sil[k + 1] = 1.f;
      }
      if (readout && p.has_z) {
        float zv[kTsT];
        load8(tZ + warp * kTsChunk + row0, zv);
#pragma unroll
        for (int k = 0; k < kTsT; k += 2) {
          const float2 sz = silu2(f2(zv[k], zv[k + 1]));
          sil[k] = sz.x;
          sil[k + 1] = sz.y;
        }
      }
      // 1. The lane's steps from a zero state: its aggregate.
      float2 h[KP], Pp[EULER ? KP : 1];
#pragma unroll
      for (int r = 0; r < KP; ++r) {
        h[r] = f2(0.f, 0.f);
        if constexpr (EULER) Pp[r] = f2(1.f, 1.f);
      }
      float ssum = 0.f;
#pragma unroll
      for (int k = 0; k < kTsT; ++k) {
        ssum += dt[k];
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) {
          const float4 bq = bq_l[qd * 32 * kTsPad + k];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int r = 2 * qd + j;
            const float2 dA = decay(__ffma2_rn(f2(dt[k], dt[k]), A2[r], f2(kArg, kArg)));
            const float2 bb = j ? f2(bq.z, bq.w) : f2(bq.x, bq.y);
            h[r] = __ffma2_rn(dA, h[r], __fmul2_rn(f2(du[k], du[k]), bb));
            if constexpr (EULER) Pp[r] = __fmul2_rn(Pp[r], dA);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < KP; r += 2) {
        float2 P0, P1;
        if constexpr (EULER) {
          P0 = Pp[r];
          P1 = Pp[r + 1];
        } else if constexpr (kAccurate) {
          P0 = exp2_acc2(__fmul2_rn(A2[r], f2(ssum, ssum)));
          P1 = exp2_acc2(__fmul2_rn(A2[r + 1], f2(ssum, ssum)));
        } else {
          P0 = f2(ex2(A2[r].x * ssum), ex2(A2[r].y * ssum));
          P1 = f2(ex2(A2[r + 1].x * ssum), ex2(A2[r + 1].y * ssum));
        }
        *reinterpret_cast<float4*>(scanP + lane * kTsScan + 2 * r) =
            make_float4(P0.x, P0.y, P1.x, P1.y);
        *reinterpret_cast<float4*>(scanH + lane * kTsScan + 2 * r) =
            make_float4(h[r].x, h[r].y, h[r + 1].x, h[r + 1].y);
      }
      if (!readout) {  // the chunk's summed step (a fixed tree), into the segment's Kahan sum
        float csum = ssum;
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) csum += __shfl_xor_sync(0xffffffffu, csum, m);
        const float yk = csum - sd_c;
        const float tk = sd + yk;
        sd_c = (tk - sd) - yk;
        sd = tk;
      }
      __syncwarp();
      // 2. Compose the 32 aggregates of state n in order (lane n < 16), from the carry; every
      //    lane's start state replaces its P. (Splitting the walk into two halves of 16, the
      //    second fixed up with the first's end state, measured slower.)
      if (scanner) {
        float x = carry;
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
          const float pj = scanP[j * kTsScan + lane], hj = scanH[j * kTsScan + lane];
          scanP[j * kTsScan + lane] = x;
          x = fmaf(pj, x, hj);
          if constexpr (EULER) {
            if (!readout) pprod *= pj;
          }
        }
        carry = x;
      }
      __syncwarp();
      if (readout) {
        // 3. The lane's steps again from its start state, with the readout; y into the lane's
        //    slots of the regrouped u (read above), then regrouped into the TMA tile.
#pragma unroll
        for (int r = 0; r < KP; r += 2) {
          const float4 hv = *reinterpret_cast<const float4*>(scanP + lane * kTsScan + 2 * r);
          h[r] = f2(hv.x, hv.y);
          h[r + 1] = f2(hv.z, hv.w);
        }
        float yv[kTsT];
#pragma unroll
        for (int k = 0; k < kTsT; ++k) {
          float2 acc = f2(0.f, 0.f);
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) {
            const float4 bq = bq_l[qd * 32 * kTsPad + k], cq = cq_l[qd * 32 * kTsPad + k];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int r = 2 * qd + j;
              const float2 dA = decay(__ffma2_rn(f2(dt[k], dt[k]), A2[r], f2(kArg, kArg)));
              const float2 bb = j ? f2(bq.z, bq.w) : f2(bq.x, bq.y);
              const float2 cc = j ? f2(cq.z, cq.w) : f2(cq.x, cq.y);
              h[r] = __ffma2_rn(dA, h[r], __fmul2_rn(f2(du[k], du[k]), bb));
              acc = __ffma2_rn(cc, h[r], acc);
            }
          }
          yv[k] = fmaf(D_c, uo[k], acc.x + acc.y) * sil[k];
        }
        store8(tU + warp * kTsChunk + row0, yv);
        if (tid == 0 && ystores > 0) tma_store_wait_read<0>();  // the last tile has been read
        __syncthreads();  // every warp's y is in tU, and the y tile is free
        {
          float v[8];
#pragma unroll
          for (int w = 0; w < kTsW; ++w) v[w] = to_f32(tU[w * kTsChunk + tid]);
          store8(ytile + tid * kTsW, v);
        }
        fence_smem_to_async();  // this thread's y row before the tile's TMA store
        __syncthreads();
        if (tid == 0) {
          tma_store_3d(&tm_y, ytile, ch0, t0, b);
          tma_store_commit();
        }
        ++ystores;
      }
    }
  }

  if (timed_out) {
    if (tid == 0) atomicOr(p.status, kErrTimeout);
  } else if (p.h_last && live && scanner && lane < N && seg == p.n_seg - 1) {
    p.h_last[(size_t(b) * p.dim + cg) * N + lane] = carry;
  }
  if (tid == 0) tma_store_wait_all();
  const int any_timeout = __syncthreads_or(timed_out);
  if (tid == 0 && any_timeout)
    for (int s2 = 0; s2 < S && s2 < n_loads; ++s2) mbar_wait_bounded(&full[s2], 0, 100000);
}

// B and C widened once per call to fp32 rows of 16 states (zero-padded past N), the layout the
// scan kernel stages with TMA and reads as 16-byte vectors. One thread per (batch, step) row.
template <typename IO>
__global__ void __launch_bounds__(256) sscan_bc_widen_kernel(const IO* __restrict__ B,
                                                             const IO* __restrict__ C, int N,
                                                             int64_t rows, float* __restrict__ B16,
                                                             float* __restrict__ C16) {
  for (int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; r < rows;
       r += int64_t(gridDim.x) * blockDim.x) {
    float vb[kNP], vc[kNP];
#pragma unroll
    for (int n = 0; n < kNP; ++n) {
      vb[n] = n < N ? to_f32(B[r * N + n]) : 0.f;
      vc[n] = n < N ? to_f32(C[r * N + n]) : 0.f;
    }
    float4* ob = reinterpret_cast<float4*>(B16 + r * kNP);
    float4* oc = reinterpret_cast<float4*>(C16 + r * kNP);
#pragma unroll
    for (int k = 0; k < kNP / 4; ++k) {
      ob[k] = make_float4(vb[4 * k], vb[4 * k + 1], vb[4 * k + 2], vb[4 * k + 3]);
      oc[k] = make_float4(vc[4 * k], vc[4 * k + 1], vc[4 * k + 2], vc[4 * k + 3]);
    }
  }
}

// ================================================================================================
// Host side.
// ================================================================================================
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

bool make_tensor_map_3d(CUtensorMap* m, const void* ptr, Io io, uint64_t d0, uint64_t d1,
                        uint64_t d2, uint32_t b0, uint32_t b1) {
  auto enc = get_encode();
  if (!enc) return false;
  const uint64_t es = io == Io::F32 ? 4 : 2;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, io == Io::F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

bool make_map(CUtensorMap* m, const void* ptr, Io io, uint64_t d0, uint64_t d1, uint64_t d2,
              uint32_t b0, uint32_t b1) {
  return make_tensor_map_3d(m, ptr, io, d0, d1, d2, b0, b1);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

constexpr int kLaneTC = 16;
constexpr int64_t kSplitBelowWarps = 300;  // fewer warps than this: split the sequence

// Per-call scratch: B and C widened to fp32 rows of 16 states (unless they already are), then
// the chunk-carry ticket, flags and aggregates (carry_units warp units of 32 lanes x (K + 1)
// floats). Stream-ordered allocation, or the caller's buffer.
struct Workspace {
  const void* B16 = nullptr;
  const void* C16 = nullptr;
  unsigned* ticket = nullptr;
  unsigned* flags = nullptr;
  float* agg = nullptr;
  void* mem = nullptr;
  bool own = false;
  cudaStream_t stream = nullptr;
  cudaError_t release(cudaError_t err) {
    if (mem && own) {
      cudaError_t e2 = cudaFreeAsync(mem, stream);
      if (err == cudaSuccess) err = e2;
    }
    mem = nullptr;
    return err;
  }
};

cudaError_t prepare_workspace(const FwdArgs& a, size_t carry_units, int K, Workspace* w,
                              bool zero_carry = false) {
  w->stream = a.stream;
  const bool widen = a.io != Io::F32 || a.N != kNP;
  const size_t rows = size_t(a.batch) * size_t(a.L);
  const size_t bc_bytes = widen ? align128(rows * kNP * sizeof(float)) : 0;
  const size_t flag_bytes = carry_units ? align128(sizeof(unsigned) * (1 + carry_units)) : 0;
  const size_t carry_bytes =
      carry_units ? flag_bytes + carry_units * 32 * (2 * K) * sizeof(float) : 0;
  const size_t bytes = 2 * bc_bytes + carry_bytes;
  w->own = a.scratch == nullptr;
  cudaError_t e = cudaSuccess;
  if (bytes > 0) {
    if (w->own) {
      e = cudaMallocAsync(&w->mem, bytes, a.stream);
      if (e != cudaSuccess) return e;
    } else {
      if (bytes > a.scratch_bytes) {
        if (a.scratch_short) *a.scratch_short = true;
        return cudaErrorInvalidValue;
      }
      w->mem = a.scratch;
    }
  }
  char* wsb = static_cast<char*>(w->mem);
  w->B16 = a.B;
  w->C16 = a.C;
  if (widen) {
    float* b16 = reinterpret_cast<float*>(wsb);
    float* c16 = reinterpret_cast<float*>(wsb + bc_bytes);
    const int wthreads = 256;
    const unsigned wblocks =
        unsigned(std::min<size_t>((rows + wthreads - 1) / wthreads, size_t(148) * 64));
    if (a.io == Io::F32)
      sscan_bc_widen_kernel<float><<<wblocks, wthreads, 0, a.stream>>>(
          static_cast<const float*>(a.B), static_cast<const float*>(a.C), int(a.N), int64_t(rows),
          b16, c16);
    else
      sscan_bc_widen_kernel<__nv_bfloat16><<<wblocks, wthreads, 0, a.stream>>>(
          static_cast<const __nv_bfloat16*>(a.B), static_cast<const __nv_bfloat16*>(a.C),
          int(a.N), int64_t(rows), b16, c16);
    e = cudaGetLastError();
    if (e != cudaSuccess) return w->release(e);
    w->B16 = b16;
    w->C16 = c16;
  }
  if (carry_units) {
    char* carry = wsb + 2 * bc_bytes;
    e = cudaMemsetAsync(carry, 0, zero_carry ? carry_bytes : flag_bytes, a.stream);
    if (e != cudaSuccess) return w->release(e);
    w->ticket = reinterpret_cast<unsigned*>(carry);
    w->flags = w->ticket + 1;
    w->agg = reinterpret_cast<float*>(carry + flag_bytes);
  }
  return cudaSuccess;
}

// Common launch parameters; segments: time segments requested (0: automatic, for `units_per_seg`
// warp units of state).
LaneParams base_params(const FwdArgs& a, int CH, int stages, int segments, int64_t units_per_seg,
                       int skip_publish, int TC = kLaneTC) {
  LaneParams p;
  p.A = a.A;
  p.D = a.D;
  p.bias = a.bias;
  p.h0 = a.h0;
  p.h_last = a.h_last;
  p.h_ckpt = a.h_ckpt;
  p.status = a.status;
  p.L = int(a.L);
  p.dim = int(a.dim);
  p.N = int(a.N);
  p.batch = int(a.batch);
  p.softplus = a.softplus;
  p.has_z = a.z != nullptr;
  p.n_chunks = int((a.L + TC - 1) / TC);
  p.n_cg = int((a.dim + CH - 1) / CH);
  p.stages = stages;
  // Chunk carry: split the sequence when too few warps would run otherwise (about 2 per SM),
  // into enough segments for about 256 warps per SM in total, i.e. many short waves of resident
  // CTAs: measured on B300 for the long sequence (batch 1, L 2^20, D 1536, two lanes per
  // channel), 62 segments 12.6 ms, 123 11.6 ms, 246 11.4 ms, 492 11.25 ms, 740 11.2 ms.
  // But the prefix passes from one segment to the next in about 2.5 us (measured), so the chain
  // of n_seg segments costs n_seg x 2.5 us however few channels there are: with few channels
  // (batch 1, D 64, L 2^20: 9472 segments by the rule above, 19.8 ms; 256 segments 1.28 ms)
  // the count is capped at the larger of sqrt(L / 10) (chain and per-segment time balanced,
  // measured) and the count whose chain takes a tenth of the two passes' time at about
  // 4.8e12 updates/s.
  int n_seg = segments;
  if (n_seg <= 0) {
    n_seg = 1;
    if (units_per_seg < kSplitBelowWarps) {
      const double fill = std::ceil(148.0 * 256.0 / double(units_per_seg));
      const double two_pass_us = 2.0 * double(a.batch) * double(a.L) * double(a.dim) * kNP / 4.8e6;
      const double by_chain = std::max(std::sqrt(double(a.L) / 10.0), 0.1 * two_pass_us / 2.5);
      n_seg = int(std::max(1.0, std::min(fill, std::ceil(by_chain))));
    }
  }
  n_seg = std::max(1, std::min(n_seg, std::max(1, p.n_chunks / 4)));
  p.seg_chunks = (p.n_chunks + n_seg - 1) / n_seg;
  p.n_seg = (p.n_chunks + p.seg_chunks - 1) / p.seg_chunks;  // no empty segments
  p.skip_publish = skip_publish;
  p.ticket = p.flags = nullptr;
  p.agg = nullptr;
  return p;
}

template <typename IO, int G, int TC, bool EULER, bool CKPT>
cudaError_t launch_lane_typed(const FwdArgs& a, int threads, const Tuning& tune) {
  threads = std::min(threads, lane_max_threads<G, TC>());  // the kernel's launch bound
  int stages = tune.stages;
  const int segments = tune.segments, skip_publish = tune.skip_publish;
  constexpr int CPW = 32 / G;
  constexpr int K = kNP / G;
  const int W = threads / 32;
  const int CH = W * CPW;
  const int es = a.io == Io::F32 ? 4 : 2;
  // Two stages for the four-lane 32-step layout (its shared memory then admits seven CTAs per
  // SM), three otherwise.
  if (stages < 2 || stages > 8) stages = (G == 4 && TC == 32) ? 2 : 3;
  while (stages > 2 &&
         LaneSmem(TC, W, CPW, es, stages, G >= 2).total + 128 > size_t(227) * 1024)
    --stages;
  const LaneSmem lay(TC, W, CPW, es, stages, G >= 2);
  size_t smem_bytes = lay.total + 128;
  if (smem_bytes > size_t(227) * 1024) return cudaErrorInvalidValue;
  if (tune.ctas_per_sm > 0) {
    // At most ctas_per_sm resident CTAs per SM: reserve enough shared memory that one more does
    // not fit (228 KB per SM, 1 KB of it reserved per CTA by the system).
    const size_t cap = size_t(228) * 1024 / size_t(tune.ctas_per_sm + 1) - 1024 + 16;
    smem_bytes = std::min(std::max(smem_bytes, cap), size_t(227) * 1024);
  }
  const int64_t n_cg = (a.dim + CH - 1) / CH;
  const int64_t warps_per_seg = a.batch * n_cg * W;
  LaneParams p = base_params(a, CH, stages, segments, warps_per_seg, skip_publish, TC);

  Workspace w;
  cudaError_t e = prepare_workspace(a, p.n_seg > 1 ? size_t(p.n_seg) * warps_per_seg : 0, K, &w);
  if (e != cudaSuccess) return e;
  p.ticket = w.ticket;
  p.flags = w.flags;
  p.agg = w.agg;

  CUtensorMap mu, md, mz, mB, mC, my;
  const uint64_t dim = a.dim, L = a.L, bt = a.batch;
  bool ok = make_map(&mu, a.u, a.io, dim, L, bt, CH, TC) &&
            make_map(&md, a.delta, a.io, dim, L, bt, CH, TC) &&
            make_map(&mz, a.z ? a.z : a.u, a.io, dim, L, bt, CH, TC) &&
            make_map(&mB, w.B16, Io::F32, kNP, L, bt, kNP, TC) &&
            make_map(&mC, w.C16, Io::F32, kNP, L, bt, kNP, TC) &&
            make_map(&my, a.y, a.io, dim, L, bt, CPW, TC);
  if (!ok) return w.release(cudaErrorInvalidValue);
  auto kern = sscan_lane_kernel<IO, G, TC, EULER, CKPT>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_bytes));
  if (e != cudaSuccess) return w.release(e);
  if (p.n_seg > 1) {
    kern<<<unsigned(p.n_seg * warps_per_seg / W), threads, smem_bytes, a.stream>>>(mu, md, mz, mB,
                                                                                   mC, my, p);
  } else {
    dim3 grid(unsigned(p.n_cg), unsigned(bt), 1);
    kern<<<grid, threads, smem_bytes, a.stream>>>(mu, md, mz, mB, mC, my, p);
  }
  return w.release(cudaGetLastError());
}

// Chunk length: 32 steps with four lanes per channel (their per-chunk fixed cost is spread over
// few state updates per step), else 16; always 16 when the backward pass wants checkpoints.
template <typename IO, bool EULER>
cudaError_t launch_lane_g(const FwdArgs& a, int G, int threads, const Tuning& tune) {
  // Backward checkpoints get their own instantiations (the store code left out of the others
  // measured 0.3-1.6% faster on the forward workloads).
  const bool ck = a.h_ckpt != nullptr;
  if (G == 1)
    return ck ? launch_lane_typed<IO, 1, 16, EULER, true>(a, threads, tune)
              : launch_lane_typed<IO, 1, 16, EULER, false>(a, threads, tune);
  if (G == 2)
    return ck ? launch_lane_typed<IO, 2, 16, EULER, true>(a, threads, tune)
              : launch_lane_typed<IO, 2, 16, EULER, false>(a, threads, tune);
  const bool long_chunks = !a.h_ckpt && tune.chunk != 16 && threads <= 128;
  if (long_chunks) return launch_lane_typed<IO, 4, 32, EULER, false>(a, threads, tune);
  return ck ? launch_lane_typed<IO, 4, 16, EULER, true>(a, threads, tune)
            : launch_lane_typed<IO, 4, 16, EULER, false>(a, threads, tune);
}

// The time-lane kernel: CTAs of kTsW channels (one resident per SM); for few channels the
// sequence is split into time segments: one wave of CTAs when a segment has at most 4 CTAs, two
// waves otherwise, and at most sqrt(L / 32) segments, where the chain of segment prefixes
// (about 1 us a segment) overtakes a segment's own work. Measured on B300 (bf16, batch 1):
// D 8, L 2^20: 148 segments (one wave) 0.31 ms, 296 (two) 0.31 ms, 222 0.33 ms; D 8, L 2^16:
// 46 segments 0.068 ms; D 64, L 2^20: 37 segments 1.37 ms.
template <typename IO, bool EULER>
cudaError_t launch_tscan_typed(const FwdArgs& a, const Tuning& tune) {
  const int es = int(sizeof(IO));
  int stages = (tune.stages >= 2 && tune.stages <= 8) ? tune.stages : 3;
  while (stages > 2 && TsSmem(es, stages).total + 128 > size_t(227) * 1024) --stages;
  const TsSmem lay(es, stages);
  const size_t smem_bytes = lay.total + 128;
  if (smem_bytes > size_t(227) * 1024) return cudaErrorInvalidValue;
  const int64_t n_cg = (a.dim + kTsW - 1) / kTsW;
  const int64_t ctas_per_seg = a.batch * n_cg;
  int segments = tune.segments;
  if (segments <= 0) {
    segments = 1;
    if (ctas_per_seg < 148) {
      const double fill = ctas_per_seg <= 4 ? std::floor(148.0 / double(ctas_per_seg))
                                            : std::ceil(296.0 / double(ctas_per_seg));
      segments = int(std::max(1.0, std::min(fill, std::ceil(std::sqrt(double(a.L) / 32.0)))));
    }
  }
  LaneParams p = base_params(a, kTsW, stages, segments, 0, tune.skip_publish, kTsChunk);
  Workspace w;
  cudaError_t e = prepare_workspace(
      a, p.n_seg > 1 ? size_t(p.n_seg) * size_t(ctas_per_seg) * kTsW : 0, 1, &w, true);
  if (e != cudaSuccess) return e;
  p.ticket = w.ticket;
  p.flags = w.flags;
  p.agg = w.agg;
  CUtensorMap mu, md, mz, mB, mC, my;
  const uint64_t dim = a.dim, L = a.L, bt = a.batch;
  bool ok = make_map(&mu, a.u, a.io, dim, L, bt, kTsW, kTsChunk) &&
            make_map(&md, a.delta, a.io, dim, L, bt, kTsW, kTsChunk) &&
            make_map(&mz, a.z ? a.z : a.u, a.io, dim, L, bt, kTsW, kTsChunk) &&
            make_map(&mB, w.B16, Io::F32, kNP, L, bt, kNP, kTsChunk) &&
            make_map(&mC, w.C16, Io::F32, kNP, L, bt, kNP, kTsChunk) &&
            make_map(&my, a.y, a.io, dim, L, bt, kTsW, kTsChunk);
  if (!ok) return w.release(cudaErrorInvalidValue);
  auto kern = sscan_tscan_kernel<IO, EULER>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_bytes));
  if (e != cudaSuccess) return w.release(e);
  if (p.n_seg > 1)
    kern<<<unsigned(p.n_seg * ctas_per_seg), kTsW * 32, smem_bytes, a.stream>>>(mu, md, mz, mB,
                                                                                  mC, my, p);
  else
    kern<<<dim3(unsigned(n_cg), unsigned(bt), 1), kTsW * 32, smem_bytes, a.stream>>>(
        mu, md, mz, mB, mC, my, p);
  return w.release(cudaGetLastError());
}

}  // namespace

cudaError_t launch_lane(const FwdArgs& a, const Tuning& tune) {
  // Layout from the number of channels (batch x dim), measured on B300: one lane per channel
  // (16 states per lane, 256-thread CTAs) from about 24k channels up; two lanes (128 threads)
  // from about 16k; four lanes (64 threads, 32-step chunks) below that. When the sequence will
  // be split into time segments anyway (too few warps even with four lanes), two lanes per
  // channel.
  const int64_t chans = a.batch * a.dim;
  int G = tune.states_per_lane ? kNP / tune.states_per_lane : 0;
  if (G == 0) {
    G = chans >= 24576 ? 1 : (chans >= 16384 ? 2 : 4);
    if (chans * 4 / 32 < kSplitBelowWarps) G = 2;
  }
  int threads = tune.threads ? tune.threads : (G == 1 ? 256 : (G == 2 ? 128 : 64));
  if (!tune.threads && G >= 2 && tune.segments <= 1) {
    // Two or four lanes per channel in one wave (no time split): the CTA size that puts the
    // fewest warps on the busiest SM when the CTAs spread evenly over the 148 SMs, the larger
    // CTA on a tie. Measured on B300: wide bf16 b4 L8192 D5120 1.127 ms with 4 warps per CTA
    // (12 on the busiest SM), 1.094 ms with 3 (9); fp32 b8 L2048 D1536 0.202 ms with 2 warps
    // (12), 0.196 ms with 1 (11).
    const int CPWl = 32 / G;
    const int64_t warps = a.batch * ((a.dim + CPWl - 1) / CPWl);
    if (warps >= kSplitBelowWarps) {
      int best_w = threads / 32;
      int64_t best = INT64_MAX;
      for (int w = threads / 32; w >= 1; --w) {
        const int64_t ctas = a.batch * ((a.dim + int64_t(w) * CPWl - 1) / (int64_t(w) * CPWl));
        const int64_t busiest = (ctas + 147) / 148 * w;
        if (busiest < best) {
          best = busiest;
          best_w = w;
        }
      }
      threads = 32 * best_w;
    }
  }
  if (threads % 32 || threads < 32 || threads > 256) return cudaErrorInvalidValue;
  const int es = a.io == Io::F32 ? 4 : 2;
  if (G != 1 && G != 2 && G != 4) return cudaErrorInvalidValue;
  if (((32 / G) * es) % 16) return cudaErrorInvalidValue;
  if (a.io == Io::F32) return a.euler ? launch_lane_g<float, true>(a, G, threads, tune)
                                      : launch_lane_g<float, false>(a, G, threads, tune);
  using bf = __nv_bfloat16;
  return a.euler ? launch_lane_g<bf, true>(a, G, threads, tune)
                 : launch_lane_g<bf, false>(a, G, threads, tune);
}

bool tma_path_ok(const FwdArgs& a) {
  const int64_t es = a.io == Io::F32 ? 4 : 2;
  if (!aligned16(a.u) || !aligned16(a.delta) || !aligned16(a.B) || !aligned16(a.C) ||
      !aligned16(a.y) || (a.z && !aligned16(a.z)))
    return false;
  if ((a.dim * es) % 16 != 0) return false;  // B / C are re-laid out when not fp32 x 16
  if (a.L > INT32_MAX - 64 || a.dim > INT32_MAX || a.batch > 65535) return false;
  return get_encode() != nullptr;
}

static cudaError_t launch_tscan(const FwdArgs& a, const Tuning& tune) {
  if (a.io == Io::F32) return a.euler ? launch_tscan_typed<float, true>(a, tune)
                                      : launch_tscan_typed<float, false>(a, tune);
  using bf = __nv_bfloat16;
  return a.euler ? launch_tscan_typed<bf, true>(a, tune) : launch_tscan_typed<bf, false>(a, tune);
}

// The time-lane kernel: when asked for, or automatically for few channels, where the lane
// kernel's many short time segments are bound by the chain of segment prefixes. Measured on
// B300 (bf16, batch 1; lane kernel -> time lanes): D 32, L 2^20 1.45 -> 0.80 ms; D 64, L 2^20
// 1.45 -> 1.40 ms; D 128, L 2^16 0.29 -> 0.22 ms; D 128, L 2^18 0.75 -> 0.85 ms; D 256, L 2^14
// 0.152 -> 0.107 ms; D 256, L 2^16 0.35 -> 0.41 ms: time lanes for at most 64 channels, or at
// most 256 channels and 2^23 channel-steps. It writes no backward checkpoints, and an explicit
// lane layout (states per lane, threads, chunk) keeps the lane kernel.
static bool use_tscan(const FwdArgs& a, const Tuning& tune) {
  if (a.h_ckpt || tune.time_scan == 2) return false;
  if (tune.time_scan == 1) return true;
  if (tune.states_per_lane || tune.threads || tune.chunk) return false;
  const int64_t chans = a.batch * a.dim;
  return chans <= 64 || (chans <= 256 && chans * a.L <= (int64_t(1) << 23));
}

cudaError_t launch_tma(const FwdArgs& a, const Tuning& tune) {
  if (use_tscan(a, tune)) return launch_tscan(a, tune);
  return launch_lane(a, tune);
}

cudaError_t launch_forward(const FwdArgs& a) {
  const Tuning tune = current_tuning();
  if (!tune.force_plain && tma_path_ok(a)) return launch_tma(a, tune);
  return launch_simple(a);
}

namespace {

template <typename IO, bool EULER>
cudaError_t launch_simple_typed(const FwdArgs& a) {
  const int64_t chans = a.batch * a.dim;
  const int threads = 128;
  const unsigned blocks = unsigned((chans + threads - 1) / threads);
  sscan_simple_kernel<IO, EULER><<<blocks, threads, 0, a.stream>>>(
      static_cast<const IO*>(a.u), static_cast<const IO*>(a.delta), a.A,
      static_cast<const IO*>(a.B), static_cast<const IO*>(a.C), a.D,
      static_cast<const IO*>(a.z), a.bias, a.softplus, a.h0, static_cast<IO*>(a.y), a.h_last,
      a.h_ckpt, a.batch, a.L, a.dim, int(a.N));
  return cudaGetLastError();
}

// Four consecutive io values as floats (16-byte load for fp32, 8-byte for bf16).
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 r = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
  const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
  return make_float4(a.x, a.y, c.x, c.y);
}

// One step of the recurrence (recurrent / decode mode): four lanes per (batch, channel), lane q
// holding states 4q .. 4q + 3 of the state h (batch, dim, N), which is read and written in place.
// u, delta, z, y are (batch, dim); B, C (batch, N). The per-channel work (softplus, skip, gate)
// is repeated by the four lanes; the readout is summed with two shuffles. VEC: N a multiple of 4
// and rows aligned, so a lane moves its states, A, B and C with one vector access each (the
// state is streamed through with evict-first hints: it is read and written once per step).
template <typename IO, bool EULER, bool VEC>
__global__ void __launch_bounds__(256) sscan_step_kernel(
    const IO* __restrict__ u, const IO* __restrict__ delta, const float* __restrict__ A,
    const IO* __restrict__ Bm, const IO* __restrict__ Cm, const float* __restrict__ Dskip,
    const IO* __restrict__ z, const float* __restrict__ bias, int softplus, float* __restrict__ h,
    IO* __restrict__ y, int64_t batch, int64_t dim, int N) {
  const int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t c = gid >> 2;  // channel b * dim + d
  const int q = int(threadIdx.x & 3);
  const bool live = c < batch * dim;
  const int64_t b = live ? c / dim : 0, d = live ? c - b * dim : 0;
  float part = 0.f, uu = 0.f;
  if (live && VEC && 4 * q < N) {
    const float x = to_f32(delta[c]) + (bias ? bias[d] : 0.f);
    const float dt = softplus ? softplus_f(x) : x;
    uu = to_f32(u[c]);
    const float dtu = dt * uu;
    float4* hp = reinterpret_cast<float4*>(h + c * N + 4 * q);
    const float4 hv = __ldcs(hp);
    const float4 av = load4(A + d * N + 4 * q);
    const float4 bv = load4(Bm + b * N + 4 * q), cv = load4(Cm + b * N + 4 * q);
    auto fac = [&](float a) {
      return EULER ? fmaf(dt, a, 1.f) : ex2(dt * (a * kLog2e));
    };
    float4 hn;
    hn.x = fmaf(fac(av.x), hv.x, dtu * bv.x);
    hn.y = fmaf(fac(av.y), hv.y, dtu * bv.y);
    hn.z = fmaf(fac(av.z), hv.z, dtu * bv.z);
    hn.w = fmaf(fac(av.w), hv.w, dtu * bv.w);
    __stcs(hp, hn);
    part = fmaf(cv.x, hn.x, fmaf(cv.y, hn.y, fmaf(cv.z, hn.z, cv.w * hn.w)));
  } else if (live && !VEC) {
    const float x = to_f32(delta[c]) + (bias ? bias[d] : 0.f);
    const float dt = softplus ? softplus_f(x) : x;
    uu = to_f32(u[c]);
    const float dtu = dt * uu;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = 4 * q + i;
      if (n < N) {
        const float e = EULER ? fmaf(dt, A[d * N + n], 1.f)
                              : ex2(dt * (A[d * N + n] * kLog2e));
        const float hn = fmaf(e, h[c * N + n], dtu * to_f32(Bm[b * N + n]));
        h[c * N + n] = hn;
        part = fmaf(to_f32(Cm[b * N + n]), hn, part);
      }
    }
  }
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  if (live && q == 0) {
    float yv = Dskip ? fmaf(Dskip[d], uu, part) : part;
    if (z) yv *= silu_f(to_f32(z[c]));
    store_io(y + c, yv);
  }
}

template <typename IO, bool EULER>
cudaError_t launch_step_typed(const FwdArgs& a) {
  const int64_t lanes = a.batch * a.dim * 4;
  const int threads = 256;
  const unsigned blocks = unsigned((lanes + threads - 1) / threads);
  auto al = [](const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; };
  const bool vec = a.N % 4 == 0 && al(a.h_last, 16) && al(a.A, 16) &&
                   al(a.B, 4 * sizeof(IO)) && al(a.C, 4 * sizeof(IO));
  auto kern = vec ? sscan_step_kernel<IO, EULER, true> : sscan_step_kernel<IO, EULER, false>;
  kern<<<blocks, threads, 0, a.stream>>>(
      static_cast<const IO*>(a.u), static_cast<const IO*>(a.delta), a.A,
      static_cast<const IO*>(a.B), static_cast<const IO*>(a.C), a.D,
      static_cast<const IO*>(a.z), a.bias, a.softplus, a.h_last, static_cast<IO*>(a.y), a.batch,
      a.dim, int(a.N));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simple(const FwdArgs& a) {
  if (a.io == Io::F32)
    return a.euler ? launch_simple_typed<float, true>(a) : launch_simple_typed<float, false>(a);
  using bf = __nv_bfloat16;
  return a.euler ? launch_simple_typed<bf, true>(a) : launch_simple_typed<bf, false>(a);
}

__global__ void __launch_bounds__(256) exp2_accurate_kernel(const float* __restrict__ x,
                                                            float* __restrict__ y, int64_t n) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x)
    y[i] = exp2_acc(x[i]);
}

cudaError_t launch_exp2_accurate(const float* x, float* y, int64_t n, cudaStream_t stream) {
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 148 * 16);
  exp2_accurate_kernel<<<unsigned(blocks), 256, 0, stream>>>(x, y, n);
  return cudaGetLastError();
}

cudaError_t launch_step(const FwdArgs& a) {
  if (a.io == Io::F32)
    return a.euler ? launch_step_typed<float, true>(a) : launch_step_typed<float, false>(a);
  using bf = __nv_bfloat16;
  return a.euler ? launch_step_typed<bf, true>(a) : launch_step_typed<bf, false>(a);
}

}  // namespace sscan
