// sscan_api.cu -- the C ABI of libsscan: argument checks, path choice, per-device state and the
// host-buffer entry point. The operation itself is defined in include/sscan.h.
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "../../include/sscan.h"
#include "../../include/sscan_tuning.h"
#include "sscan_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kHostStreams = 3;      // host path: streams the batch slices rotate over
constexpr int64_t kHostSlices = 8;   // host path: at most this many batch slices per call
constexpr int64_t kHostTimeSlices = 16;     // host path, few batch rows: time slices per call
constexpr int64_t kHostMinSliceSteps = 16384;  // host path: shortest time slice

struct DeviceState {
  unsigned int* status = nullptr;  // device status word
  // host-path staging (device side), grown on demand, and the streams its slices run on
  void* stage = nullptr;
  size_t stage_bytes = 0;
  cudaStream_t host_streams[kHostStreams] = {};
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::mutex g_host_mu[kMaxDevices];  // one host-path call per device at a time

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

unsigned int* status_word(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[dev];
  if (!s.status) {
    if (cudaMalloc(&s.status, sizeof(unsigned int)) != cudaSuccess) {
      s.status = nullptr;
      return nullptr;
    }
    if (cudaMemset(s.status, 0, sizeof(unsigned int)) != cudaSuccess) return nullptr;
  }
  return s.status;
}

std::mutex g_tune_mu;
sscan::Tuning g_tune;  // sscan_set_tuning's setting, process-wide

using sscan::launch_forward;

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > INT64_MAX / a) return false;
  *out = a * b;
  return true;
}

}  // namespace

namespace sscan {

Tuning current_tuning() {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  return g_tune;
}

// Shared validation of sizes and pointer presence; fills the element counts.
int check_fwd_args(const void* u, const void* delta, const float* A, const void* B,
                   const void* C, const void* y, int64_t batch, int64_t L, int64_t dim,
                   int64_t N, int dtype, int64_t* n_bld, int64_t* n_bln) {
  if (dtype != SSCAN_F32 && dtype != SSCAN_BF16) return SSCAN_ERR_INVALID_ARG;
  if (batch < 0 || L < 0 || dim < 0 || N < 1 || N > 16) return SSCAN_ERR_INVALID_ARG;
  int64_t bl, bld, bln, bd, bdn, bytes;
  if (!mul_ok(batch, L, &bl) || !mul_ok(bl, dim, &bld) || !mul_ok(bl, N, &bln) ||
      !mul_ok(bld, 4, &bytes) || !mul_ok(batch, dim, &bd) || !mul_ok(bd, N, &bdn) ||
      !mul_ok(bdn, 4, &bytes))
    return SSCAN_ERR_INVALID_ARG;
  *n_bld = bld;
  *n_bln = bln;
  if (bd == 0 || L == 0) return SSCAN_OK;  // nothing to read
  if (!A || !u || !delta || !B || !C || !y) return SSCAN_ERR_INVALID_ARG;
  return SSCAN_OK;
}

}  // namespace sscan

namespace {

sscan_status_t check_args(const void* u, const void* delta, const float* A, const void* B,
                          const void* C, const void* y, int64_t batch, int64_t L, int64_t dim,
                          int64_t N, sscan_dtype_t dtype, int64_t* n_bld, int64_t* n_bln) {
  return static_cast<sscan_status_t>(
      sscan::check_fwd_args(u, delta, A, B, C, y, batch, L, dim, N, int(dtype), n_bld, n_bln));
}

}  // namespace

extern "C" {

sscan_status_t sscan_set_tuning(const sscan_tuning_t* t) {
  sscan::Tuning n;
  if (t) {
    const int k = t->states_per_lane;
    if ((k != 0 && k != 4 && k != 8 && k != 16) || t->segments < 0 || t->threads < 0 ||
        t->threads > 256 || t->threads % 32 != 0 || t->stages < 0 || t->stages > 8 ||
        t->stages == 1 || (t->chunk != 0 && t->chunk != 16 && t->chunk != 32) ||
        t->bwd_segments < 0 || t->test_skip_publish < -1 || t->ctas_per_sm < 0 ||
        t->ctas_per_sm > 32 || t->time_scan < 0 || t->time_scan > 2)
      return SSCAN_ERR_INVALID_ARG;
    n.states_per_lane = k;
    n.segments = t->segments;
    n.threads = t->threads;
    n.stages = t->stages;
    n.chunk = t->chunk;
    n.force_plain = t->force_plain != 0;
    n.bwd_segments = t->bwd_segments;
    n.conv_plain = t->conv_plain != 0;
    n.ctas_per_sm = t->ctas_per_sm;
    n.skip_publish = t->test_skip_publish;
    n.time_scan = t->time_scan;
  }
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tune = n;
  return SSCAN_OK;
}

sscan_status_t sscan_exp2_accurate(const float* x, float* y, int64_t n, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return SSCAN_ERR_INVALID_ARG;
  if (n == 0) return SSCAN_OK;
  if (current_device() < 0) return SSCAN_ERR_CUDA;
  return sscan::launch_exp2_accurate(x, y, n, stream) == cudaSuccess ? SSCAN_OK : SSCAN_ERR_CUDA;
}

sscan_status_t sscan_get_tuning(sscan_tuning_t* t) {
  if (!t) return SSCAN_ERR_INVALID_ARG;
  const sscan::Tuning c = sscan::current_tuning();
  t->states_per_lane = c.states_per_lane;
  t->segments = c.segments;
  t->threads = c.threads;
  t->stages = c.stages;
  t->chunk = c.chunk;
  t->force_plain = c.force_plain;
  t->bwd_segments = c.bwd_segments;
  t->conv_plain = c.conv_plain;
  t->ctas_per_sm = c.ctas_per_sm;
  t->test_skip_publish = c.skip_publish;
  t->time_scan = c.time_scan;
  return SSCAN_OK;
}

const char* sscan_status_string(sscan_status_t s) {
  switch (s) {
    case SSCAN_OK: return "SSCAN_OK";
    case SSCAN_ERR_INVALID_ARG: return "SSCAN_ERR_INVALID_ARG";
    case SSCAN_ERR_UNSUPPORTED: return "SSCAN_ERR_UNSUPPORTED";
    case SSCAN_ERR_CUDA: return "SSCAN_ERR_CUDA";
    case SSCAN_ERR_CARRY_TIMEOUT: return "SSCAN_ERR_CARRY_TIMEOUT";
    case SSCAN_ERR_SCRATCH_TOO_SMALL: return "SSCAN_ERR_SCRATCH_TOO_SMALL";
  }
  return "SSCAN_ERR_UNKNOWN";
}

sscan_status_t sscan_fwd_ex(const void* u, const void* delta, const float* A, const void* B,
                            const void* C, const float* D, const void* z,
                            const float* delta_bias, int softplus_flag, const float* h0,
                            sscan_disc_t disc, void* y, float* h_last, int64_t batch, int64_t L,
                            int64_t dim, int64_t N, sscan_dtype_t dtype, cudaStream_t stream) {
  int64_t bld = 0, bln = 0;
  if (disc != SSCAN_DISC_ZOH && disc != SSCAN_DISC_EULER) return SSCAN_ERR_INVALID_ARG;
  sscan_status_t st = check_args(u, delta, A, B, C, y, batch, L, dim, N, dtype, &bld, &bln);
  if (st != SSCAN_OK) return st;
  const int dev = current_device();
  if (dev < 0) return SSCAN_ERR_CUDA;
  if (batch == 0 || dim == 0) return SSCAN_OK;
  if (L == 0) {  // the final state is the initial state
    const size_t hb = size_t(batch * dim * N) * sizeof(float);
    if (h_last && (h0 ? cudaMemcpyAsync(h_last, h0, hb, cudaMemcpyDeviceToDevice, stream)
                      : cudaMemsetAsync(h_last, 0, hb, stream)) != cudaSuccess)
      return SSCAN_ERR_CUDA;
    return SSCAN_OK;
  }
  sscan::FwdArgs a;
  a.u = u;
  a.delta = delta;
  a.A = A;
  a.B = B;
  a.C = C;
  a.D = D;
  a.z = z;
  a.bias = delta_bias;
  a.softplus = softplus_flag != 0;
  a.h0 = h0;
  a.euler = disc == SSCAN_DISC_EULER;
  a.y = y;
  a.h_last = h_last;
  a.batch = batch;
  a.L = L;
  a.dim = dim;
  a.N = N;
  a.io = dtype == SSCAN_F32 ? sscan::Io::F32 : sscan::Io::BF16;
  a.stream = stream;
  a.status = status_word(dev);
  if (!a.status) return SSCAN_ERR_CUDA;
  return launch_forward(a) == cudaSuccess ? SSCAN_OK : SSCAN_ERR_CUDA;
}

sscan_status_t sscan_fwd(const void* u, const void* delta, const float* A, const void* B,
                         const void* C, const float* D, const void* z, const float* delta_bias,
                         int softplus_flag, void* y, float* h_last, int64_t batch, int64_t L,
                         int64_t dim, int64_t N, sscan_dtype_t dtype, cudaStream_t stream) {
  return sscan_fwd_ex(u, delta, A, B, C, D, z, delta_bias, softplus_flag, nullptr,
                      SSCAN_DISC_ZOH, y, h_last, batch, L, dim, N, dtype, stream);
}

sscan_status_t sscan_step(const void* u, const void* delta, const float* A, const void* B,
                          const void* C, const float* D, const void* z, const float* delta_bias,
                          int softplus_flag, sscan_disc_t disc, float* h, void* y, int64_t batch,
                          int64_t dim, int64_t N, sscan_dtype_t dtype, cudaStream_t stream) {
  if (disc != SSCAN_DISC_ZOH && disc != SSCAN_DISC_EULER) return SSCAN_ERR_INVALID_ARG;
  int64_t bld = 0, bln = 0;
  sscan_status_t st = check_args(u, delta, A, B, C, y, batch, 1, dim, N, dtype, &bld, &bln);
  if (st != SSCAN_OK) return st;
  if (batch * dim > 0 && !h) return SSCAN_ERR_INVALID_ARG;
  if (current_device() < 0) return SSCAN_ERR_CUDA;
  if (batch == 0 || dim == 0) return SSCAN_OK;
  sscan::FwdArgs a;
  a.u = u;
  a.delta = delta;
  a.A = A;
  a.B = B;
  a.C = C;
  a.D = D;
  a.z = z;
  a.bias = delta_bias;
  a.softplus = softplus_flag != 0;
  a.euler = disc == SSCAN_DISC_EULER;
  a.y = y;
  a.h_last = h;  // read and written in place
  a.batch = batch;
  a.L = 1;
  a.dim = dim;
  a.N = N;
  a.io = dtype == SSCAN_F32 ? sscan::Io::F32 : sscan::Io::BF16;
  a.stream = stream;
  a.status = nullptr;
  return sscan::launch_step(a) == cudaSuccess ? SSCAN_OK : SSCAN_ERR_CUDA;
}

sscan_status_t sscan_bwd(const void* u, const void* delta, const float* A, const void* B,
                         const void* C, const float* D, const void* z, const float* delta_bias,
                         int softplus_flag, const float* h0, sscan_disc_t disc, const void* dy,
                         const float* dh_last, void* du, void* ddelta, float* dA, float* dB,
                         float* dC, float* dD, void* dz, float* ddelta_bias, float* dh0,
                         int64_t batch, int64_t L, int64_t dim, int64_t N, sscan_dtype_t dtype,
                         cudaStream_t stream) {
  if (disc != SSCAN_DISC_ZOH && disc != SSCAN_DISC_EULER) return SSCAN_ERR_INVALID_ARG;
  int64_t bld = 0, bln = 0;
  sscan_status_t st = check_args(u, delta, A, B, C, dy, batch, L, dim, N, dtype, &bld, &bln);
  if (st != SSCAN_OK) return st;
  if (batch * dim > 0 && L > 0 &&
      (!du || !ddelta || !dA || !dB || !dC || (D && !dD) || (z && !dz) ||
       (delta_bias && !ddelta_bias)))
    return SSCAN_ERR_INVALID_ARG;
  if (current_device() < 0) return SSCAN_ERR_CUDA;
  if (batch == 0 || dim == 0) return SSCAN_OK;
  if (L == 0) {  // nothing depends on the sequence: parameter gradients are zero, dh0 = dh_last
    cudaError_t e = cudaSuccess;
    if (dA) e = cudaMemsetAsync(dA, 0, size_t(dim * N) * sizeof(float), stream);
    if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, size_t(dim) * sizeof(float), stream);
    if (e == cudaSuccess && ddelta_bias)
      e = cudaMemsetAsync(ddelta_bias, 0, size_t(dim) * sizeof(float), stream);
    if (e == cudaSuccess && dh0) {
      const size_t hb = size_t(batch * dim * N) * sizeof(float);
      e = dh_last ? cudaMemcpyAsync(dh0, dh_last, hb, cudaMemcpyDeviceToDevice, stream)
                  : cudaMemsetAsync(dh0, 0, hb, stream);
    }
    return e == cudaSuccess ? SSCAN_OK : SSCAN_ERR_CUDA;
  }
  // Checkpoints: the forward pass (same inputs) writes the state before every 16-step chunk;
  // its y goes to scratch. Stream-ordered workspace, released after the backward kernels.
  const int dev = current_device();
  const size_t es = dtype == SSCAN_F32 ? 4 : 2;
  const int64_t n_chunks = (L + 15) / 16;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t ck_bytes = up(size_t(n_chunks) * size_t(batch * dim * N) * sizeof(float));
  const size_t y_bytes = up(size_t(bld) * es);
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, ck_bytes + y_bytes, stream) != cudaSuccess) return SSCAN_ERR_CUDA;
  float* ckpt = static_cast<float*>(ws);
  sscan::FwdArgs f;
  f.u = u;
  f.delta = delta;
  f.A = A;
  f.B = B;
  f.C = C;
  f.D = D;
  f.z = z;
  f.bias = delta_bias;
  f.softplus = softplus_flag != 0;
  f.h0 = h0;
  f.euler = disc == SSCAN_DISC_EULER;
  f.y = static_cast<char*>(ws) + ck_bytes;
  f.h_last = nullptr;
  f.h_ckpt = ckpt;
  f.batch = batch;
  f.L = L;
  f.dim = dim;
  f.N = N;
  f.io = dtype == SSCAN_F32 ? sscan::Io::F32 : sscan::Io::BF16;
  f.stream = stream;
  f.status = status_word(dev);
  cudaError_t e = f.status ? launch_forward(f) : cudaErrorMemoryAllocation;
  sscan::BwdArgs a;
  a.u = u;
  a.delta = delta;
  a.A = A;
  a.B = B;
  a.C = C;
  a.D = D;
  a.z = z;
  a.bias = delta_bias;
  a.softplus = softplus_flag != 0;
  a.h0 = h0;
  a.euler = disc == SSCAN_DISC_EULER;
  a.dy = dy;
  a.dh_last = dh_last;
  a.du = du;
  a.ddelta = ddelta;
  a.dA = dA;
  a.dB = dB;
  a.dC = dC;
  a.dD = D ? dD : nullptr;
  a.dz = z ? dz : nullptr;
  a.dbias = delta_bias ? ddelta_bias : nullptr;
  a.dh0 = dh0;
  a.batch = batch;
  a.L = L;
  a.dim = dim;
  a.N = N;
  a.io = dtype == SSCAN_F32 ? sscan::Io::F32 : sscan::Io::BF16;
  a.stream = stream;
  a.ckpt = ckpt;
  if (e == cudaSuccess) e = sscan::launch_bwd(a);
  const cudaError_t e2 = cudaFreeAsync(ws, stream);
  return (e == cudaSuccess && e2 == cudaSuccess) ? SSCAN_OK : SSCAN_ERR_CUDA;
}

sscan_status_t sscan_conv1d_silu(const void* x, const float* w, const float* bias,
                                 const void* x_prev, int silu_flag, void* y, int64_t batch,
                                 int64_t L, int64_t dim, int64_t width, sscan_dtype_t dtype,
                                 cudaStream_t stream) {
  if (dtype != SSCAN_F32 && dtype != SSCAN_BF16) return SSCAN_ERR_INVALID_ARG;
  if (batch < 0 || L < 0 || dim < 0 || width < 1 || width > 64) return SSCAN_ERR_INVALID_ARG;
  int64_t bl, bld, bytes;
  if (!mul_ok(batch, L, &bl) || !mul_ok(bl, dim, &bld) || !mul_ok(bld, 4, &bytes) ||
      !mul_ok(dim, width, &bytes))
    return SSCAN_ERR_INVALID_ARG;
  if (bld == 0) return SSCAN_OK;
  if (!x || !w || !y || x == y) return SSCAN_ERR_INVALID_ARG;
  if (current_device() < 0) return SSCAN_ERR_CUDA;
  sscan::ConvArgs a;
  a.x = x;
  a.w = w;
  a.bias = bias;
  a.x_prev = width > 1 ? x_prev : nullptr;
  a.silu = silu_flag != 0;
  a.y = y;
  a.batch = batch;
  a.L = L;
  a.dim = dim;
  a.width = width;
  a.io = dtype == SSCAN_F32 ? sscan::Io::F32 : sscan::Io::BF16;
  a.stream = stream;
  a.status = status_word(current_device());
  if (!a.status) return SSCAN_ERR_CUDA;
  return sscan::launch_conv(a) == cudaSuccess ? SSCAN_OK : SSCAN_ERR_CUDA;
}

sscan_status_t sscan_fwd_host(const void* u, const void* delta, const float* A, const void* B,
                              const void* C, const float* D, const void* z,
                              const float* delta_bias, int softplus_flag, void* y, float* h_last,
                              int64_t batch, int64_t L, int64_t dim, int64_t N,
                              sscan_dtype_t dtype, cudaStream_t stream) {
  int64_t bld = 0, bln = 0;
  sscan_status_t st = check_args(u, delta, A, B, C, y, batch, L, dim, N, dtype, &bld, &bln);
  if (st != SSCAN_OK) return st;
  const int dev = current_device();
  if (dev < 0) return SSCAN_ERR_CUDA;
  if (batch == 0 || dim == 0) return SSCAN_OK;
  const size_t es = dtype == SSCAN_F32 ? 4 : 2;
  std::lock_guard<std::mutex> call_lock(g_host_mu[dev]);
  // Device staging layout, each piece 256-byte aligned.
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t s_bld = up(size_t(bld) * es), s_bln = up(size_t(bln) * es);
  const size_t s_A = up(size_t(dim * N) * 4), s_dim = up(size_t(dim) * 4);
  const size_t s_h = up(size_t(batch * dim * N) * 4);
  const size_t total = (3 + (z ? 1 : 0)) * s_bld + 2 * s_bln + s_A + 2 * s_dim + s_h;
  unsigned char* base = nullptr;
  cudaStream_t hs[kHostStreams];
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& ds = g_dev[dev];
    if (ds.stage_bytes < total) {
      if (ds.stage) {
        cudaDeviceSynchronize();
        cudaFree(ds.stage);
      }
      ds.stage = nullptr;
      ds.stage_bytes = 0;
      if (cudaMalloc(&ds.stage, total) != cudaSuccess) return SSCAN_ERR_CUDA;
      ds.stage_bytes = total;
    }
    for (int k = 0; k < kHostStreams; ++k) {
      if (!ds.host_streams[k] &&
          cudaStreamCreateWithFlags(&ds.host_streams[k], cudaStreamNonBlocking) != cudaSuccess) {
        ds.host_streams[k] = nullptr;
        return SSCAN_ERR_CUDA;
      }
      hs[k] = ds.host_streams[k];
    }
    base = static_cast<unsigned char*>(ds.stage);
  }
  unsigned char* p = base;
  auto take = [&](size_t n) { unsigned char* r = p; p += n; return r; };
  unsigned char* du = take(s_bld);
  unsigned char* ddl = take(s_bld);
  unsigned char* dy = take(s_bld);
  unsigned char* dz = z ? take(s_bld) : nullptr;
  unsigned char* dB = take(s_bln);
  unsigned char* dC = take(s_bln);
  float* dA = reinterpret_cast<float*>(take(s_A));
  float* dD = D ? reinterpret_cast<float*>(take(s_dim)) : nullptr;
  float* dbias = delta_bias ? reinterpret_cast<float*>(take(s_dim)) : nullptr;
  // Few batch rows and a long sequence: the sequence is cut into time slices instead, each
  // continuing from the previous one's end state (dh, always allocated then).
  const bool by_time = batch < kHostSlices && L >= 2 * kHostMinSliceSteps;
  float* dh = (h_last || by_time) ? reinterpret_cast<float*>(take(s_h)) : nullptr;
  auto copy = [](void* dst, const void* src, size_t n, cudaMemcpyKind kind, cudaStream_t s) {
    return n == 0 || cudaMemcpyAsync(dst, src, n, kind, s) == cudaSuccess;
  };
  const auto H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
  // Per-channel parameters on the caller's stream; then the batch is cut into slices that
  // rotate over the library's streams, so one slice's host-to-device copy, another's scan and
  // a third's device-to-host copy run at the same time.
  bool ok = copy(dA, A, size_t(dim * N) * 4, H2D, stream) &&
            (!D || copy(dD, D, size_t(dim) * 4, H2D, stream)) &&
            (!delta_bias || copy(dbias, delta_bias, size_t(dim) * 4, H2D, stream));
  cudaEvent_t ev_start = nullptr, ev_done[kHostStreams] = {};
  ok = ok && cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming) == cudaSuccess;
  for (int k = 0; k < kHostStreams && ok; ++k)
    ok = cudaEventCreateWithFlags(&ev_done[k], cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventRecord(ev_start, stream) == cudaSuccess;
  for (int k = 0; k < kHostStreams && ok; ++k)
    ok = cudaStreamWaitEvent(hs[k], ev_start, 0) == cudaSuccess;
  if (by_time && ok) {
    // Slice k holds steps [t0, t0 + Lk) of every batch row, staged densely as (batch, Lk, dim);
    // its scan waits for slice k - 1's (sscan_fwd_ex from its end state, in place in dh), while
    // the copies of neighbouring slices run on the other streams in both directions.
    const int64_t n_t = std::min<int64_t>(kHostTimeSlices, L / kHostMinSliceSteps);
    const int64_t Ls = (L + n_t - 1) / n_t;
    cudaEvent_t ev_scan[kHostTimeSlices] = {};
    for (int64_t k = 0; k < n_t && ok; ++k)
      ok = cudaEventCreateWithFlags(&ev_scan[k], cudaEventDisableTiming) == cudaSuccess;
    const unsigned char* hu = static_cast<const unsigned char*>(u);
    const unsigned char* hdl = static_cast<const unsigned char*>(delta);
    const unsigned char* hz = static_cast<const unsigned char*>(z);
    const unsigned char* hB = static_cast<const unsigned char*>(B);
    const unsigned char* hC = static_cast<const unsigned char*>(C);
    unsigned char* hy = static_cast<unsigned char*>(y);
    const size_t row_d = size_t(L * dim) * es, row_n = size_t(L * N) * es;  // host row pitches
    auto copy2 = [&](void* dst, size_t dp, const void* src, size_t sp, size_t w,
                     cudaMemcpyKind kind, cudaStream_t s) {
      return cudaMemcpy2DAsync(dst, dp, src, sp, w, size_t(batch), kind, s) == cudaSuccess;
    };
    for (int64_t k = 0, t0 = 0; k < n_t && t0 < L && ok; ++k, t0 += Ls) {
      const int64_t Lk = std::min(Ls, L - t0);
      cudaStream_t s = hs[k % kHostStreams];
      const size_t od = size_t(batch * t0 * dim) * es, on = size_t(batch * t0 * N) * es;
      const size_t wd = size_t(Lk * dim) * es, wn = size_t(Lk * N) * es;  // one row's slice
      const size_t hd = size_t(t0 * dim) * es, hn = size_t(t0 * N) * es;  // its host offset
      ok = copy2(du + od, wd, hu + hd, row_d, wd, H2D, s) &&
           copy2(ddl + od, wd, hdl + hd, row_d, wd, H2D, s) &&
           (!z || copy2(dz + od, wd, hz + hd, row_d, wd, H2D, s)) &&
           copy2(dB + on, wn, hB + hn, row_n, wn, H2D, s) &&
           copy2(dC + on, wn, hC + hn, row_n, wn, H2D, s);
      if (ok && k > 0) ok = cudaStreamWaitEvent(s, ev_scan[k - 1], 0) == cudaSuccess;
      if (ok) {
        st = sscan_fwd_ex(du + od, ddl + od, dA, dB + on, dC + on, dD, z ? dz + od : nullptr,
                          dbias, softplus_flag, k > 0 ? dh : nullptr, SSCAN_DISC_ZOH, dy + od,
                          dh, batch, Lk, dim, N, dtype, s);
        ok = st == SSCAN_OK;
      }
      ok = ok && cudaEventRecord(ev_scan[k], s) == cudaSuccess &&
           copy2(hy + hd, row_d, dy + od, wd, wd, D2H, s);
      if (ok && h_last && t0 + Lk == L)
        ok = copy(h_last, dh, size_t(batch * dim * N) * 4, D2H, s);
    }
    for (int k = 0; k < kHostStreams; ++k) {  // every stream done before the events go
      if (ok) ok = cudaEventRecord(ev_done[k], hs[k]) == cudaSuccess &&
                   cudaStreamWaitEvent(stream, ev_done[k], 0) == cudaSuccess;
    }
    if (ok) ok = cudaStreamSynchronize(stream) == cudaSuccess;
    if (!ok)
      for (int k = 0; k < kHostStreams; ++k) cudaStreamSynchronize(hs[k]);
    for (int64_t k = 0; k < n_t; ++k)
      if (ev_scan[k]) cudaEventDestroy(ev_scan[k]);
    if (ev_start) cudaEventDestroy(ev_start);
    for (int k = 0; k < kHostStreams; ++k)
      if (ev_done[k]) cudaEventDestroy(ev_done[k]);
    if (!ok) return st != SSCAN_OK ? st : SSCAN_ERR_CUDA;
    return SSCAN_OK;
  }
  const int64_t n_slices = batch < kHostSlices ? batch : kHostSlices;
  const int64_t rows = (batch + n_slices - 1) / n_slices;
  const unsigned char* hu = static_cast<const unsigned char*>(u);
  const unsigned char* hdl = static_cast<const unsigned char*>(delta);
  const unsigned char* hz = static_cast<const unsigned char*>(z);
  const unsigned char* hB = static_cast<const unsigned char*>(B);
  const unsigned char* hC = static_cast<const unsigned char*>(C);
  unsigned char* hy = static_cast<unsigned char*>(y);
  for (int64_t r0 = 0, i = 0; r0 < batch && ok; r0 += rows, ++i) {
    const int64_t nr = batch - r0 < rows ? batch - r0 : rows;
    cudaStream_t s = hs[i % kHostStreams];
    const size_t o = size_t(r0 * L * dim) * es, n = size_t(nr * L * dim) * es;
    const size_t ob = size_t(r0 * L * N) * es, nbc = size_t(nr * L * N) * es;
    ok = copy(du + o, hu + o, n, H2D, s) && copy(ddl + o, hdl + o, n, H2D, s) &&
         (!z || copy(dz + o, hz + o, n, H2D, s)) && copy(dB + ob, hB + ob, nbc, H2D, s) &&
         copy(dC + ob, hC + ob, nbc, H2D, s);
    float* dhs = dh ? dh + r0 * dim * N : nullptr;
    if (ok) {
      st = sscan_fwd(du + o, ddl + o, dA, dB + ob, dC + ob, dD, z ? dz + o : nullptr, dbias,
                     softplus_flag, dy + o, dhs, nr, L, dim, N, dtype, s);
      ok = st == SSCAN_OK;
    }
    ok = ok && copy(hy + o, dy + o, n, D2H, s) &&
         (!h_last || copy(h_last + r0 * dim * N, dhs, size_t(nr * dim * N) * 4, D2H, s));
  }
  for (int k = 0; k < kHostStreams; ++k) {
    if (ok) ok = cudaEventRecord(ev_done[k], hs[k]) == cudaSuccess &&
                 cudaStreamWaitEvent(stream, ev_done[k], 0) == cudaSuccess;
  }
  if (ok) ok = cudaStreamSynchronize(stream) == cudaSuccess;
  if (!ok)  // nothing may still be reading or writing the caller's buffers when this returns
    for (int k = 0; k < kHostStreams; ++k) cudaStreamSynchronize(hs[k]);
  if (ev_start) cudaEventDestroy(ev_start);
  for (int k = 0; k < kHostStreams; ++k)
    if (ev_done[k]) cudaEventDestroy(ev_done[k]);
  if (!ok) return st != SSCAN_OK ? st : SSCAN_ERR_CUDA;
  return SSCAN_OK;
}

sscan_status_t sscan_get_device_error(cudaStream_t stream) {
  const int dev = current_device();
  if (dev < 0) return SSCAN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SSCAN_ERR_CUDA;
  unsigned int* w = nullptr;  // sscan_fwd's word, if any call created it (no allocation here)
  {
    std::lock_guard<std::mutex> lk(g_mu);
    w = g_dev[dev].status;
  }
  unsigned int v = 0, v2 = 0;
  if (w && cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return SSCAN_ERR_CUDA;
  // Calls of the allocation-free entry point record device errors in its own static word.
  unsigned int* w2 = sscan::noalloc_status_word(dev);
  if (w2 && cudaMemcpy(&v2, w2, sizeof v2, cudaMemcpyDeviceToHost) != cudaSuccess)
    return SSCAN_ERR_CUDA;
  if ((v | v2) == 0) return SSCAN_OK;
  if (v && cudaMemset(w, 0, sizeof v) != cudaSuccess) return SSCAN_ERR_CUDA;
  if (v2 && cudaMemset(w2, 0, sizeof v2) != cudaSuccess) return SSCAN_ERR_CUDA;
  return SSCAN_ERR_CARRY_TIMEOUT;
}

sscan_status_t sscan_release(void) {
  const int dev = current_device();
  if (dev < 0) return SSCAN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[dev];
  cudaError_t e = cudaSuccess;
  for (int k = 0; k < kHostStreams; ++k)
    if (s.host_streams[k] && e == cudaSuccess) e = cudaStreamDestroy(s.host_streams[k]);
  if (s.status && e == cudaSuccess) e = cudaFree(s.status);
  if (s.stage && e == cudaSuccess) e = cudaFree(s.stage);
  s = DeviceState();
  return e == cudaSuccess ? SSCAN_OK : SSCAN_ERR_CUDA;
}

}  // extern "C"
