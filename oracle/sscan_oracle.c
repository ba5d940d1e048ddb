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
#if SSCAN_ORACLE_MUTANT != 24
      mag += fabs((double)*Dskip_d * ut); /* mutant 24: the skip term left out of the magnitude */
#endif
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

/*
 * Backward pass: gradients of  Loss = sum_{b,t,d} dy[b,t,d] * y[b,t,d] + sum dh_last * h_last
 * with respect to every input of the forward above (the same h0 and factor selector). The
 * pages fix the method's backward only as "recompute the intermediate states instead of storing
 * them" ([notes] "第二个创新：硬件感知算法", item 3; [article] 3.3, item 2); the gradient itself
 * is the derivative of the defined forward, written here as the adjoint recurrence, per channel:
 *
 *   forward, keeping every state:  h_t = a_t h_{t-1} + dt_t B_t u_t,  s_t = C_t . h_t + D u_t
 *   lam_t = dL/dh_t = ds_t C_t + a_{t+1} lam_{t+1},  lam_{L-1} = ds_{L-1} C_{L-1} + dh_last
 *   ds_t = dy_t g(z_t),  dz_t = dy_t s_t g'(z_t)      (g = SiLU, g' = sig (1 + z (1 - sig)))
 *   dC_t += ds_t h_t,  dB_t += lam_t dt_t u_t,  du_t = ds_t D + sum_n lam_t dt_t B_t
 *   d(dt_t) = sum_n lam_t (B_t u_t + h_{t-1} da_t/d(dt)),   da/d(dt) = A a (ZOH) or A (first order)
 *   dA += lam_t h_{t-1} da_t/dA,                             da/dA = dt a (ZOH) or dt (first order)
 *   ddelta_t = d(dt_t) sig(x_t) with softplus (1 without),  dbias += ddelta_t,  dD += ds_t u_t
 *   dh0 = a_0 lam_0
 *
 * Outputs (double, overwritten): du, ddelta (batch, L, dim); dz (batch, L, dim) if z; dA
 * (dim, N); dB, dC (batch, L, N); dD (dim) if Dskip; dbias (dim) if bias; dh0 (batch, dim, N)
 * if not NULL. dy is (batch, L, dim) io; dh_last (batch, dim, N) fp32 or NULL. Single-threaded
 * (the parameter gradients sum over channels). Returns 0, or -1 on bad sizes.
 *
 * mag != 0 computes, in the same outputs, each gradient's magnitude instead: the same sums with
 * every input, factor and derivative factor replaced by its absolute value, so that every term
 * enters with its size (the scale that rounding in a finite-precision evaluation of the gradient
 * is proportional to, as ymag is for y). With every input non-negative and no negative factor
 * the magnitude equals the gradient.
 */
int sscan_oracle_bwd(const void *u, const void *delta, const float *A, const void *Bm,
                     const void *Cm, const float *Dskip, const void *z, const float *bias,
                     int softplus_flag, const float *h0, int euler, const void *dy,
                     const float *dh_last, double *du, double *ddelta, double *dA, double *dB,
                     double *dC, double *dD, double *dz, double *dbias, double *dh0,
                     int64_t batch, int64_t L, int64_t dim, int64_t N, int io_bf16, int mag) {
#define M(v) (mag ? fabs(v) : (v)) /* a leaf of the gradient's terms (its size when mag) */
  if (batch < 0 || L < 0 || dim < 0 || N < 1) return -1;
  memset(dA, 0, sizeof(double) * (size_t)(dim * N));
  memset(dB, 0, sizeof(double) * (size_t)(batch * L * N));
  memset(dC, 0, sizeof(double) * (size_t)(batch * L * N));
  if (dD) memset(dD, 0, sizeof(double) * (size_t)dim);
  if (dbias) memset(dbias, 0, sizeof(double) * (size_t)dim);
  double *hs = (double *)malloc(sizeof(double) * (size_t)((L + 1) * N)); /* h_{-1} .. h_{L-1} */
  double *as = (double *)malloc(sizeof(double) * (size_t)(L * N + 1));
  double *dts = (double *)malloc(sizeof(double) * (size_t)(L + 1));
  double *xs = (double *)malloc(sizeof(double) * (size_t)(L + 1));
  double *ss = (double *)malloc(sizeof(double) * (size_t)(L + 1));
  double *mu = (double *)malloc(sizeof(double) * (size_t)N);
  for (int64_t b = 0; b < batch; ++b)
    for (int64_t d = 0; d < dim; ++d) {
      const int64_t cbase = b * L * dim + d; /* element (b, 0, d) */
      const double Dd = M(Dskip ? (double)Dskip[d] : 0.0);
      for (int64_t n = 0; n < N; ++n) hs[n] = M(h0 ? (double)h0[(b * dim + d) * N + n] : 0.0);
      for (int64_t t = 0; t < L; ++t) { /* forward, every state kept */
        const int64_t i = cbase + t * dim;
        const double x = widen(delta, i, io_bf16) + (bias ? (double)bias[d] : 0.0);
        const double dt = softplus_flag ? softplus(x) : x;
        const double ut = M(widen(u, i, io_bf16));
        double s = Dd * ut;
        for (int64_t n = 0; n < N; ++n) {
          const double a =
              M(euler ? 1.0 + dt * (double)A[d * N + n] : exp(dt * (double)A[d * N + n]));
          const double hn =
              a * hs[t * N + n] + M(dt) * M(widen(Bm, (b * L + t) * N + n, io_bf16)) * ut;
          hs[(t + 1) * N + n] = hn;
          as[t * N + n] = a;
          s += M(widen(Cm, (b * L + t) * N + n, io_bf16)) * hn;
        }
        xs[t] = x;
        dts[t] = dt;
        ss[t] = s;
      }
      for (int64_t n = 0; n < N; ++n)
        mu[n] = M(dh_last ? (double)dh_last[(b * dim + d) * N + n] : 0.0);
      for (int64_t t = L - 1; t >= 0; --t) { /* adjoint sweep */
        const int64_t i = cbase + t * dim;
        const double ut = M(widen(u, i, io_bf16)), dyt = M(widen(dy, i, io_bf16));
        const double dt = M(dts[t]);
        double ds = dyt;
        if (z) {
          const double zr = widen(z, i, io_bf16), sg = 1.0 / (1.0 + exp(-zr)), zt = M(zr);
          ds = dyt * zt * sg;
#if SSCAN_ORACLE_MUTANT == 23
          dz[i] = dyt * ss[t] * sg; /* mutant: gate derivative taken as the sigmoid alone */
#else
          dz[i] = dyt * ss[t] * sg * (1.0 + zt * (1.0 - sg));
#endif
        }
        if (dD) dD[d] += ds * ut;
        double dut = ds * Dd, ddt = 0.0;
        for (int64_t n = 0; n < N; ++n) {
          const double Bt = M(widen(Bm, (b * L + t) * N + n, io_bf16));
          const double Ct = M(widen(Cm, (b * L + t) * N + n, io_bf16));
          const double An = M((double)A[d * N + n]), a = as[t * N + n];
          const double lam = mu[n] + ds * Ct;
#if SSCAN_ORACLE_MUTANT == 21
          dC[(b * L + t) * N + n] += ds * hs[t * N + n]; /* mutant: previous state in dC */
#else
          dC[(b * L + t) * N + n] += ds * hs[(t + 1) * N + n];
#endif
          const double da = lam * hs[t * N + n];
#if SSCAN_ORACLE_MUTANT == 19
          (void)An; /* mutant: the decay's dependence on dt dropped */
#else
          ddt += euler ? da * An : da * a * An;
#endif
          dA[d * N + n] += euler ? da * dt : da * a * dt;
          ddt += lam * Bt * ut;
          dB[(b * L + t) * N + n] += lam * dt * ut;
          dut += lam * dt * Bt;
#if SSCAN_ORACLE_MUTANT == 20
          mu[n] = (t > 0 ? as[(t - 1) * N + n] : a) * lam; /* mutant: the earlier step's factor */
#else
          mu[n] = a * lam;
#endif
        }
        du[i] = dut;
#if SSCAN_ORACLE_MUTANT == 22
        const double dx = ddt; /* mutant: softplus derivative dropped */
#else
        const double dx = softplus_flag ? ddt / (1.0 + exp(-xs[t])) : ddt;
#endif
        ddelta[i] = dx;
        if (dbias) dbias[d] += dx;
      }
      if (dh0)
        for (int64_t n = 0; n < N; ++n) dh0[(b * dim + d) * N + n] = mu[n];
    }
  free(hs);
  free(as);
  free(dts);
  free(xs);
  free(ss);
  free(mu);
  return 0;
#undef M
}
