// sscan_device.cuh -- device-side building blocks of libsscan (sm_103a): inline-PTX wrappers for
// mbarriers, TMA tensor copies and the SFU exponential, io-type conversions, and the scalar
// per-(step, channel) functions (softplus, SiLU) in scalar and f32x2-paired forms.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sscan {

constexpr float kLog2e = 1.4426950408889634f;

// ---- io element conversions -------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_io(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_io(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// ---- SFU exponential: 2^x, flushing denormal results to zero ----------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- paired (f32x2) forms used per (step, channel pair) ------------------------------------
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// log1p(s)/s on [0, 1] by a polynomial from Chebyshev interpolation in double precision,
// re-expanded in powers of s and rounded to fp32 (csrc/gen_softplus_poly.py regenerates both):
// degree 9, s * p(s) within 1.6e-7 relative of log1p(s) in fp32 on the whole interval (the fp32
// io path); degree 6, within 1.5e-6 (bf16 io, where it is far inside the tolerance and saves
// three FMAs per step).
template <bool kDeg6 = false>
__device__ __forceinline__ float2 log1p_unit2(float2 s) {
  if constexpr (kDeg6) {
    constexpr float c[7] = {9.999985695e-01f, -4.998590052e-01f, 3.309752643e-01f,
                            -2.345452011e-01f, 1.482941359e-01f, -6.559030712e-02f,
                            1.387448423e-02f};
    float2 acc = f2(c[6], c[6]);
#pragma unroll
    for (int i = 5; i >= 0; --i) acc = __ffma2_rn(acc, s, f2(c[i], c[i]));
    return __fmul2_rn(s, acc);
  } else {
    constexpr float c[10] = {1.000000000e+00f, -4.999989271e-01f, 3.332971036e-01f,
                             -2.495161593e-01f, 1.966327429e-01f, -1.526966691e-01f,
                             1.054362357e-01f, -5.637361482e-02f, 1.954252832e-02f,
                             -3.176057013e-03f};
    float2 acc = f2(c[9], c[9]);
#pragma unroll
    for (int i = 8; i >= 0; --i) acc = __ffma2_rn(acc, s, f2(c[i], c[i]));
    return __fmul2_rn(s, acc);
  }
}

// 2^x on the FMA pipe, accurate to about one ulp and unbiased (the fp32 path's decay over a
// whole chunk, where the SFU's approximate exponential would otherwise enter the state once per
// step and its rounding, which leans low for small arguments, would compound over the state's
// memory). Range reduction after Cody and Waite: k = rint(x) by the 1.5 * 2^23 rounding constant
// (exact for |x| < 2^22), f = x - k in [-1/2, 1/2] exactly; 2^f by a degree-6 polynomial from
// Chebyshev interpolation (csrc/gen_exp2_poly.py regenerates it: relative error 1.04e-7 for an
// unfused fp32 evaluation, mean signed error 1.2e-9); 2^k enters through the exponent field.
// x is clamped to [-125, 125]: results below 2^-125 are not needed (they multiply a state that
// has decayed away), and no result is denormal or infinite.
__device__ __forceinline__ float2 exp2_poly2(float2 f) {
  constexpr float c[7] = {1.000000000e+00f, 6.931471825e-01f, 2.402265072e-01f,
                          5.550327152e-02f, 9.618056938e-03f, 1.340042800e-03f,
                          1.546144485e-04f};
  float2 p = f2(c[6], c[6]);
#pragma unroll
  for (int i = 5; i >= 0; --i) p = __ffma2_rn(p, f, f2(c[i], c[i]));
  return p;
}
__device__ __forceinline__ float2 exp2_acc2(float2 x) {
  constexpr float kRound = 12582912.f;  // 1.5 * 2^23
  x = f2(fminf(fmaxf(x.x, -125.f), 125.f), fminf(fmaxf(x.y, -125.f), 125.f));
  const float2 t = __fadd2_rn(x, f2(kRound, kRound));                    // rint(x) + kRound
  const float2 kf = __fadd2_rn(t, f2(-kRound, -kRound));                 // rint(x), exact
  const float2 f = __ffma2_rn(kf, f2(-1.f, -1.f), x);                    // x - rint(x), exact
  const float2 p = exp2_poly2(f);
  const int kx = __float_as_int(t.x) - __float_as_int(kRound);
  const int ky = __float_as_int(t.y) - __float_as_int(kRound);
  return f2(__int_as_float(__float_as_int(p.x) + (kx << 23)),
            __int_as_float(__float_as_int(p.y) + (ky << 23)));
}
__device__ __forceinline__ float exp2_acc(float x) { return exp2_acc2(f2(x, 0.f)).x; }

// softplus on a pair: max(x, 0) + log1p(exp(-|x|)); one SFU exponential per element.
template <bool kDeg6 = false>
__device__ __forceinline__ float2 softplus2(float2 x) {
  const float2 e = __fmul2_rn(f2(-fabsf(x.x), -fabsf(x.y)), f2(kLog2e, kLog2e));
  const float2 s = f2(ex2(e.x), ex2(e.y));
  return __fadd2_rn(f2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), log1p_unit2<kDeg6>(s));
}

// softplus(x) = log(1 + e^x), the positivity map of the step ("Mamba：选择性状态空间模型入门教程",
// selective-scan pseudo-code), scalar form of softplus2.
__device__ __forceinline__ float softplus_f(float x) {
  const float2 r = softplus2(f2(x, 0.f));
  return r.x;
}

// SiLU on a pair: z / (1 + 2^(-z log2 e)).
__device__ __forceinline__ float2 silu2(float2 z) {
  const float2 e = __fmul2_rn(z, f2(-kLog2e, -kLog2e));
  const float2 d = __fadd2_rn(f2(ex2(e.x), ex2(e.y)), f2(1.f, 1.f));
  return f2(__fdividef(z.x, d.x), __fdividef(z.y, d.y));
}

// z * sigmoid(z), the SiLU gate of the Mamba block ("Mamba: Linear-Time Sequence Modeling with
// Selective State Spaces", block diagram in "架构：极简设计").
__device__ __forceinline__ float silu_f(float z) {
  return __fdividef(z, 1.f + ex2(-z * kLog2e));
}

// ---- io pairs ---------------------------------------------------------------------------------
__device__ __forceinline__ float2 load_pair(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
__device__ __forceinline__ float2 load_pair(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void store_pair(float* p, float2 v) {
  *reinterpret_cast<float2*>(p) = v;
}
__device__ __forceinline__ void store_pair(__nv_bfloat16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __float22bfloat162_rn(v);
}

// ---- shared-memory addresses ------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ---------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait with a suspend-time hint: the thread may sleep in hardware (issuing nothing) until the
// phase completes or about `hint_ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity,
                                                   uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: returns false if the phase has not completed after `max_ns` nanoseconds of
// wall-clock time (or 2^24 sleeps, whichever comes first). Waiting warps sleep in hardware
// between polls instead of spinning, so they take no issue slots from the working warps.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t max_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0; i < (1u << 24); ++i) {
    if (mbar_try_wait_hint(bar, parity, 100000u)) return true;
    if (globaltimer_ns() - t0 > max_ns) break;
  }
  return false;
}

constexpr uint64_t kWaitNs = 1000000000ull;  // bound on one mbarrier wait: one second
constexpr unsigned kErrTimeout = 1u << 4;    // status bit: a bounded wait ran out

// ---- TMA tensor copies (3-D maps: x = fastest dimension) --------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::
          "l"(reinterpret_cast<uint64_t>(m)),
      "r"(x), "r"(y), "r"(z), "r"(smem_addr(src))
      : "memory");
}
__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later async-proxy (TMA) reads.
__device__ __forceinline__ void fence_smem_to_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace sscan
