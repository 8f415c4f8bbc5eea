// Fast-mode scaling exponents without any device allocation.
//
// ozaki2_dgemm keeps its intermediates in a workspace that it allocates (and
// grows) with cudaMalloc on first use.  Some callers cannot allow that: code
// running inside a framework that owns all device memory through its own
// pool, latency-critical loops in which an allocation could block or
// synchronise the device, and plug-ins that are not permitted to touch the
// allocator at all.  For them this file provides ozaki2_fast_exponents_noalloc:
// the scale-statistics stage of the fast mode (per-row and per-column maximum
// magnitude and sum of squares, then the exponents alpha and beta), with its
// scratch held in a fixed array compiled into the library.
//
// The scratch array is shared by every call in the process and keeps the
// contents of the last call; each call clears the part it uses before the
// statistics kernels run.  Two calls whose kernels overlap on the GPU (for
// example, issued on different streams without ordering) race on it.
#include <mutex>

#include "oz2_internal.cuh"

namespace oz2 {
namespace {

constexpr int64_t kMaxVectors = OZ2_NOALLOC_MAX_VECTORS;  // p + r at most
constexpr int kMaxDevices = 64;

// [amax of A's rows | amax of B's columns | sums of A's rows | sums of B's columns]
static __device__ __align__(256) uint64_t g_fast_exp_scratch[2 * kMaxVectors];

std::mutex g_setup_mutex;
uint64_t* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The first call
// per device looks the symbol up (which may load the library's device code on
// that device); later calls reuse the stored address.
oz2_status scratch_address(uint64_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZ2_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return OZ2_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fast_exp_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return OZ2_ERR_CUDA;
    }
    g_scratch_addr[dev] = static_cast<uint64_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return OZ2_OK;
}

// L = M/2 - 1 for the first s greedy moduli, computed on the stack.
BoundConsts bound_consts_on_stack(int s) {
  int mods[OZ2_S_MAX];
  int n = 0;
  for (int m = 256; m >= 2 && n < s; --m) {
    bool ok = true;
    for (int k = 0; k < n && ok; ++k) {
      int a = m, b = mods[k];
      while (b) {
        const int t = a % b;
        a = b;
        b = t;
      }
      ok = (a == 1);
    }
    if (ok) mods[n++] = m;
  }
  uint32_t L[6] = {1, 0, 0, 0, 0, 0};
  for (int t = 0; t < s; ++t) {  // L <- M
    uint64_t c = 0;
    for (int k = 0; k < 6; ++k) {
      const uint64_t v = static_cast<uint64_t>(L[k]) * static_cast<uint32_t>(mods[t]) + c;
      L[k] = static_cast<uint32_t>(v);
      c = v >> 32;
    }
  }
  for (int k = 0; k < 6; ++k) L[k] = (L[k] >> 1) | (k + 1 < 6 ? (L[k + 1] << 31) : 0u);  // M/2
  for (int k = 0; k < 6; ++k) {  // minus 1
    if (L[k] != 0) {
      L[k] -= 1;
      break;
    }
    L[k] = 0xFFFFFFFFu;
  }
  int bits = 0;
  for (int k = 5; k >= 0 && bits == 0; --k)
    for (int b = 31; b >= 0; --b)
      if ((L[k] >> b) & 1u) {
        bits = 32 * k + b + 1;
        break;
      }
  uint64_t norm = 0;
  for (int i = 0; i < 64; ++i) {
    const int pos = bits - 1 - i;
    norm <<= 1;
    if (pos >= 0 && ((L[pos >> 5] >> (pos & 31)) & 1u)) norm |= 1;
  }
  BoundConsts bc;
  bc.Lbits = bits;
  bc.Lnorm = norm;
  return bc;
}

}  // namespace
}  // namespace oz2

extern "C" oz2_status ozaki2_fast_exponents_noalloc(int64_t p, int64_t q, int64_t r,
                                                    const double* A, int64_t lda, const double* B,
                                                    int64_t ldb, int s, int32_t* alpha,
                                                    int32_t* beta, void* stream) {
  using namespace oz2;
  if (p <= 0 || q <= 0 || r <= 0 || lda < p || ldb < q) return OZ2_ERR_INVALID_ARG;
  if (!A || !B || !alpha || !beta) return OZ2_ERR_INVALID_ARG;
  if (s < OZ2_S_MIN || s > OZ2_S_MAX) return OZ2_ERR_INVALID_ARG;
  if (q >= OZ2_Q_LIMIT_FAST) return OZ2_ERR_Q_TOO_LARGE;
  if (p > kMaxVectors || r > kMaxVectors || p + r > kMaxVectors) return OZ2_ERR_SCRATCH_TOO_SMALL;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZ2_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (!(major == 10 && minor == 3)) return OZ2_ERR_UNSUPPORTED_DEVICE;
  uint64_t* scratch = nullptr;
  const oz2_status e = scratch_address(&scratch);
  if (e != OZ2_OK) return e;
  uint64_t* amaxA = scratch;
  uint64_t* amaxB = scratch + p;
  uint64_t* sumA = scratch + p + r;
  uint64_t* sumB = scratch + 2 * p + r;
  ScaleArgs sa{p, q, r, lda, ldb, A, B};
  // launch_fast_exponents clears the four scratch ranges (cudaMemsetAsync)
  // before its statistics kernels accumulate into them.
  if (launch_fast_exponents(sa, bound_consts_on_stack(s), amaxA, amaxB, sumA, sumB, alpha, beta,
                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return OZ2_ERR_CUDA;
  return OZ2_OK;
}
