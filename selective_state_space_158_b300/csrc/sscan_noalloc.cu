// sscan_noalloc.cu -- sscan_fwd_noalloc: the selective-scan forward for callers that cannot
// allocate device memory. The chunk-carry scratch (and this entry point's device status word)
// live in a fixed static device array instead of a stream-ordered allocation.
#include <cstring>
#include <mutex>

#include "../../include/sscan.h"
#include "sscan_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB per device, held until exit
constexpr size_t kStatusBytes = 256;                // status word, then the chunk-carry scratch

// The array in device memory. In host code its name is only a host-side stand-in: the device
// address is looked up per device with cudaGetSymbolAddress (set-up below).
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's copy of the array; looked up once per device, with the
// device current. Returns null if the lookup fails.
unsigned char* scratch_for(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    g_scratch_addr[dev] = static_cast<unsigned char*>(ptr);
  }
  return g_scratch_addr[dev];
}

}  // namespace

namespace sscan {

unsigned int* noalloc_status_word(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  return reinterpret_cast<unsigned int*>(g_scratch_addr[dev]);
}

}  // namespace sscan

extern "C" sscan_status_t sscan_fwd_noalloc(const void* u, const void* delta, const float* A,
                                            const void* B, const void* C, const float* D,
                                            const void* z, const float* delta_bias,
                                            int softplus_flag, void* y, float* h_last,
                                            int64_t batch, int64_t L, int64_t dim, int64_t N,
                                            sscan_dtype_t dtype, cudaStream_t stream) {
  int64_t bld = 0, bln = 0;
  const int st = sscan::check_fwd_args(u, delta, A, B, C, y, batch, L, dim, N, int(dtype), &bld,
                                       &bln);
  if (st != SSCAN_OK) return static_cast<sscan_status_t>(st);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSCAN_ERR_CUDA;
  if (batch == 0 || dim == 0) return SSCAN_OK;
  if (L == 0) {
    if (h_last &&
        cudaMemsetAsync(h_last, 0, size_t(batch * dim * N) * sizeof(float), stream) != cudaSuccess)
      return SSCAN_ERR_CUDA;
    return SSCAN_OK;
  }
  unsigned char* base = scratch_for(dev);
  if (!base) return SSCAN_ERR_CUDA;
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
  a.y = y;
  a.h_last = h_last;
  a.batch = batch;
  a.L = L;
  a.dim = dim;
  a.N = N;
  a.io = dtype == SSCAN_F32 ? sscan::Io::F32 : sscan::Io::BF16;
  a.stream = stream;
  a.status = reinterpret_cast<unsigned int*>(base);
  bool short_scratch = false;
  a.scratch = base + kStatusBytes;
  a.scratch_bytes = kScratchBytes - kStatusBytes;
  a.scratch_short = &short_scratch;
  const cudaError_t e = sscan::launch_forward(a);  // the plain-load kernel needs no scratch
  if (short_scratch) return SSCAN_ERR_SCRATCH_TOO_SMALL;
  return e == cudaSuccess ? SSCAN_OK : SSCAN_ERR_CUDA;
}
