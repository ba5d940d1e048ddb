/*
 * sscan_oracle.c -- fp64 CPU oracle for the S6 selective-scan forward.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously-correct statement of what the
 * selective scan computes. It exists so that tests, the smoke check and the benchmark's CPU
 * baseline leg can compare the CUDA library against it. Nothing in the product path may call,
 * link or load it, and it shares no code, header, table or helper with the CUDA library.
 *
 * Pages cited below, by title:
 *   [tutorial] "Mamba：选择性状态空间模型入门教程"
 *   [notes]    "Mamba: Linear-Time Sequence Modeling with Selective State Spaces" (wiki notes)
 *   [article]  "从RNN到Mamba：深入浅出图解'选择性状态空间'如何让模型学会'忘记'"
 *   [variant]  "架构变体：Mamba/SSM"
 *
 * What it computes (one channel (b, d), state size N, sequence length L), all in double:
 *
 *   h[n] = h0[b,d,n], or 0 without h0           initial state: zero as the scan in the
 *                                                 [variant] "Python 演示" demo starts from h = 0.0;
 *                                                 a given state continues a sequence in the
 *                                                 recurrent (step-by-step) inference mode,
 *                                                 [tutorial] "Mamba 的关键创新：选择性机制" and
 *                                                 [notes] "核心贡献：选择机制（S6）" (the state is
 *                                                 all that carries over between steps)
 *   for t = 0 .. L-1:
 *     x      = delta[b,t,d] + bias[d]           Delta_t = tau(Delta + s_Delta(x_t)): S6 row of
 *                                                 the algorithm table, [notes] "核心贡献：选择机制（S6）"
 *     dt     = softplus_flag ? log(1 + e^x) : x tau = softplus keeps the step positive: [tutorial]
 *                                                 "Mamba 的关键创新：选择性机制" pseudo-code;
 *                                                 [article] section 3.1
 *     for n:  h[n] = dA * h[n] + dt * B[b,t,n] * u[b,t,d]
 *             dA = exp(dt*A[d,n])               zero-order hold for A: [variant] "离散化";
 *                                                 Delta*B for the input term: [article] 3.2
 *             dA = 1 + dt*A[d,n]  (euler)       first-order variant: [article] 3.2 writes
 *                                                 (I - Delta A); with A < 0 that factor exceeds 1
 *                                                 and the state grows without bound, so the
 *                                                 reading is the first-order expansion of
 *                                                 exp(Delta A), I + Delta A
 *     y[b,t,d] = sum_n C[b,t,n] * h[n]          readout of the updated state: [tutorial]
 *                                                 selection pseudo-code, y_t = C * h_t
 *              + Dskip[d] * u[b,t,d]            the D*x term: [tutorial] "状态空间模型（SSM）的直觉"
 *     if z:  y[b,t,d] *= z / (1 + e^-z)         SiLU gate branch multiplied into the SSM
 *                                                 branch: [notes] "架构：极简设计" block diagram
 *   h_last[b,d,n] = h[n]
 *
 * Inputs are read as stored: fp32 values widen to double exactly, bf16 values (passed as their
 * 16-bit patterns) widen to fp32 and then to double exactly. Layouts:
 *   u, delta, z : (batch, L, dim), dim fastest         A      : (dim, N) fp32
 *   B, C        : (batch, L, N),   N fastest           Dskip, bias : (dim) fp32
 *   h0          : (batch, dim, N) fp32, or NULL
 *   y           : (batch, L, dim) double               h_last : (batch, dim, N) double
 *
 * The loop is sequential in t, exactly as defined; threads only split independent channels.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef SSCAN_ORACLE_MUTANT
#define SSCAN_ORACLE_MUTANT 0 /* tests compile deliberately broken copies with other values */
#endif

static double widen(const void *p, int64_t i, int io_bf16) {
  if (!io_bf16) return (double)((const float *)p)[i];
  uint32_t w = (uint32_t)((const uint16_t *)p)[i] << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* log(1 + e^x), written so that neither branch overflows. */
static double softplus(double x) {
  return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x));
}

/* One channel. Element t of u/delta/z sits at index t*t_stride; B and C rows are L x N,
 * N fastest; y element t is written at y[t*y_stride]; h (N doubles) receives the final state.
 * h0_d (N floats) is the initial state, or NULL for zero; euler selects dA = 1 + dt*A.
 * ymag, if not NULL, receives the same sum taken over absolute values (the scale that rounding
 * error in a finite-precision evaluation is proportional to). */
void sscan_oracle_channel_ex(const void *u, const void *delta, const void *z, int64_t t_stride,
                             const float *A_d, const void *Bm, const void *Cm,
                             const float *Dskip_d, const float *bias_d, int softplus_flag,
                             const float *h0_d, int euler, int64_t L, int64_t N, int io_bf16,
                             double *y, int64_t y_stride, double *h, double *ymag) {
  double *habs = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
  for (int64_t n = 0; n < N; ++n) {
#if SSCAN_ORACLE_MUTANT == 12
    h[n] = 0.0; /* mutant: initial state ignored */
#else
    h[n] = h0_d ? (double)h0_d[n] : 0.0;
#endif
    habs[n] = fabs(h[n]);
  }
  for (int64_t t = 0; t < L; ++t) {
    double x = widen(delta, t * t_stride, io_bf16) + (bias_d ? (double)*bias_d : 0.0);
#if SSCAN_ORACLE_MUTANT == 7
    double dt = x; /* mutant: softplus dropped */
    (void)softplus_flag;
#elif SSCAN_ORACLE_MUTANT == 8
    double dt = softplus_flag ? softplus(widen(delta, t * t_stride, io_bf16)) +
                                    (bias_d ? (double)*bias_d : 0.0)
                              : x; /* mutant: bias added after softplus */
#else
    double dt = softplus_flag ? softplus(x) : x;
#endif
    double ut = widen(u, t * t_stride, io_bf16);
    double acc = 0.0, mag = 0.0;
    for (int64_t n = 0; n < N; ++n) {
#if SSCAN_ORACLE_MUTANT == 2
      double dA = euler ? 1.0 + dt * (double)A_d[n]
                        : exp(-dt * (double)A_d[n]); /* mutant: sign of the exponent flipped */
#elif SSCAN_ORACLE_MUTANT == 9
      double dA = 1.0 + dt * (double)A_d[n]; /* mutant: first-order (Euler) instead of ZOH */
#elif SSCAN_ORACLE_MUTANT == 14
      double dA = euler ? 1.0 - dt * (double)A_d[n] /* mutant: Euler factor with the page's sign */
                        : exp(dt * (double)A_d[n]);
#else
      double dA = euler ? 1.0 + dt * (double)A_d[n] : exp(dt * (double)A_d[n]);
#endif
#if SSCAN_ORACLE_MUTANT == 4
      double bt = widen(Bm, (L - 1 - t) * N + n, io_bf16); /* mutant: B read at the wrong time */
#else
      double bt = widen(Bm, t * N + n, io_bf16);
#endif
      double ct = widen(Cm, t * N + n, io_bf16);
#if SSCAN_ORACLE_MUTANT == 1
      acc += ct * h[n]; /* mutant: readout taken before the state update */
      h[n] = dA * h[n] + dt * bt * ut;
#elif SSCAN_ORACLE_MUTANT == 5
      h[n] = dA * h[n] + bt * ut; /* mutant: dt missing from the input term */
      acc += ct * h[n];
#elif SSCAN_ORACLE_MUTANT == 10
      h[n] = dA * h[n] + dt * ct * ut; /* mutant: B and C swapped */
      acc += bt * h[n];
#elif SSCAN_ORACLE_MUTANT == 13
      h[n] = (t == 0 && h0_d ? 1.0 : dA) * h[n] + dt * bt * ut; /* mutant: h0 not decayed */
      acc += ct * h[n];
#else
      h[n] = dA * h[n] + dt * bt * ut;
      acc += ct * h[n];
#endif
      habs[n] = fabs(dA) * habs[n] + fabs(dt * bt * ut);
      mag += fabs(ct) * habs[n];
    }
#if SSCAN_ORACLE_MUTANT != 3
    if (Dskip_d) { /* mutant 3: skip term dropped */
      acc += (double)*Dskip_d * ut;
      mag += fabs((double)*Dskip_d * ut);
    }
#endif
    if (z) {
      double zt = widen(z, t * t_stride, io_bf16);
#if SSCAN_ORACLE_MUTANT == 6
      double g = 1.0 / (1.0 + exp(-zt)); /* mutant: sigmoid gate instead of SiLU */
#else
      double g = zt / (1.0 + exp(-zt));
#endif
      acc *= g;
      mag *= fabs(g);
    }
    y[t * y_stride] = acc;
    if (ymag) ymag[t * y_stride] = mag;
  }
  free(habs);
}

/* The zero-initial-state, zero-order-hold scan of one channel (sscan_oracle_channel_ex with
 * h0 = NULL, euler = 0). */
void sscan_oracle_channel(const void *u, const void *delta, const void *z, int64_t t_stride,
                          const float *A_d, const void *Bm, const void *Cm,
                          const float *Dskip_d, const float *bias_d, int softplus_flag,
                          int64_t L, int64_t N, int io_bf16, double *y, int64_t y_stride,
                          double *h, double *ymag) {
  sscan_oracle_channel_ex(u, delta, z, t_stride, A_d, Bm, Cm, Dskip_d, bias_d, softplus_flag,
                          NULL, 0, L, N, io_bf16, y, y_stride, h, ymag);
}

typedef struct {
  const void *u, *delta, *z, *B, *C;
  const float *A, *Dskip, *bias, *h0;
  int softplus_flag, io_bf16, euler;
  int64_t batch, L, dim, N;
  double *y, *h_last, *ymag;
  int64_t chan_begin, chan_end; /* channel index c = b*dim + d */
} job_t;

static void *run_job(void *arg) {
  job_t *j = (job_t *)arg;
  size_t es = j->io_bf16 ? 2 : 4;
  for (int64_t c = j->chan_begin; c < j->chan_end; ++c) {
    int64_t b = c / j->dim, d = c % j->dim;
#if SSCAN_ORACLE_MUTANT == 11
    int64_t bb = (b + 1) % j->batch; /* mutant: B/C rows taken from another batch */
#else
    int64_t bb = b;
#endif
    int64_t base = (b * j->L) * j->dim + d; /* element (b, 0, d) */
    const char *u = (const char *)j->u + (size_t)base * es;
    const char *dl = (const char *)j->delta + (size_t)base * es;
    const char *zz = j->z ? (const char *)j->z + (size_t)base * es : NULL;
    const char *Bm = (const char *)j->B + (size_t)(bb * j->L * j->N) * es;
    const char *Cm = (const char *)j->C + (size_t)(bb * j->L * j->N) * es;
    sscan_oracle_channel_ex(u, dl, zz, j->dim, j->A + d * j->N, Bm, Cm,
                            j->Dskip ? j->Dskip + d : NULL, j->bias ? j->bias + d : NULL,
                            j->softplus_flag, j->h0 ? j->h0 + (b * j->dim + d) * j->N : NULL,
                            j->euler, j->L, j->N, j->io_bf16, j->y + base, j->dim,
                            j->h_last + (b * j->dim + d) * j->N, j->ymag ? j->ymag + base : NULL);
  }
  return NULL;
}

/* Whole tensors, channels split over nthreads POSIX threads. h0 ((batch, dim, N) fp32) may be
 * NULL for a zero initial state; euler selects dA = 1 + dt*A. Returns 0, or -1 on bad sizes. */
int sscan_oracle_fwd_ex(const void *u, const void *delta, const float *A, const void *B,
                        const void *C, const float *Dskip, const void *z,
                        const float *delta_bias, int softplus_flag, const float *h0, int euler,
                        double *y, double *h_last, double *ymag, int64_t batch, int64_t L,
                        int64_t dim, int64_t N, int io_bf16, int nthreads) {
  if (batch < 0 || L < 0 || dim < 0 || N < 1) return -1;
  int64_t chans = batch * dim;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (chans < nthreads) nthreads = chans > 0 ? (int)chans : 1;
  job_t jobs[256];
  pthread_t tid[256];
  for (int i = 0; i < nthreads; ++i) {
    job_t *j = &jobs[i];
    j->u = u; j->delta = delta; j->z = z; j->B = B; j->C = C;
    j->A = A; j->Dskip = Dskip; j->bias = delta_bias; j->h0 = h0;
    j->softplus_flag = softplus_flag; j->io_bf16 = io_bf16; j->euler = euler;
    j->batch = batch; j->L = L; j->dim = dim; j->N = N;
    j->y = y; j->h_last = h_last; j->ymag = ymag;
    j->chan_begin = chans * i / nthreads;
    j->chan_end = chans * (i + 1) / nthreads;
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&tid[i], NULL, run_job, &jobs[i]);
  run_job(&jobs[0]);
  for (int i = 1; i < nthreads; ++i) pthread_join(tid[i], NULL);
  return 0;
}

/* The zero-initial-state, zero-order-hold scan over whole tensors (sscan_oracle_fwd_ex with
 * h0 = NULL, euler = 0). */
int sscan_oracle_fwd(const void *u, const void *delta, const float *A, const void *B,
                     const void *C, const float *Dskip, const void *z, const float *delta_bias,
                     int softplus_flag, double *y, double *h_last, double *ymag, int64_t batch,
                     int64_t L, int64_t dim, int64_t N, int io_bf16, int nthreads) {
  return sscan_oracle_fwd_ex(u, delta, A, B, C, Dskip, z, delta_bias, softplus_flag, NULL, 0, y,
                             h_last, ymag, batch, L, dim, N, io_bf16, nthreads);
}

/*
 * Causal depthwise convolution over time, then SiLU: the step that turns the in-projection's
 * output into the scan's input in the Mamba block ([notes] "架构：极简设计": Linear -> Conv1d ->
 * SiLU). Per channel d, with W = width taps and w[d, W-1] the tap of the current step:
 *
 *   acc = bias[d] + sum_{j=0}^{W-1} w[d, j] * x[b, t - (W-1) + j, d]
 *   y[b, t, d] = silu ? acc / (1 + e^-acc) : acc
 *
 * Inputs before t = 0 come from x_prev (batch, W-1, dim), oldest first, or are zero. Causal
 * (no future step enters) and depthwise (channels do not mix): the plainest reading of a
 * convolution placed ahead of a causal, per-channel recurrence. Width is a parameter (the pages
 * do not give it). Layouts: x (batch, L, dim) io; w (dim, W) fp32; bias (dim) fp32 or NULL;
 * y (batch, L, dim) double. Returns 0, or -1 on bad sizes.
 */
int sscan_oracle_conv1d(const void *x, const float *w, const float *bias, const void *x_prev,
                        int silu, double *y, int64_t batch, int64_t L, int64_t dim,
                        int64_t width, int io_bf16) {
  if (batch < 0 || L < 0 || dim < 0 || width < 1) return -1;
  for (int64_t b = 0; b < batch; ++b)
    for (int64_t d = 0; d < dim; ++d)
      for (int64_t t = 0; t < L; ++t) {
        double acc = bias ? (double)bias[d] : 0.0;
#if SSCAN_ORACLE_MUTANT == 18
        acc = 0.0; /* mutant: bias dropped */
#endif
        for (int64_t j = 0; j < width; ++j) {
#if SSCAN_ORACLE_MUTANT == 15
          int64_t s = t + j; /* mutant: future steps instead of past ones */
#elif SSCAN_ORACLE_MUTANT == 16
          int64_t s = t - j; /* mutant: taps applied in reverse order */
#else
          int64_t s = t - (width - 1) + j;
#endif
          double v = 0.0;
          if (s >= 0 && s < L)
            v = widen(x, (b * L + s) * dim + d, io_bf16);
          else if (s < 0 && x_prev)
            v = widen(x_prev, (b * (width - 1) + (s + width - 1)) * dim + d, io_bf16);
          acc += (double)w[d * width + j] * v;
        }
#if SSCAN_ORACLE_MUTANT == 17
        y[(b * L + t) * dim + d] = acc; /* mutant: SiLU dropped */
        (void)silu;
#else
        y[(b * L + t) * dim + d] = silu ? acc / (1.0 + exp(-acc)) : acc;
#endif
      }
  return 0;
}
