// CRT reconstruction and inverse scaling of Ozaki II: for every output entry,
// X = CRT_M(R_1..R_s) in [-M/2, M/2) and C = X 2^-(alpha_i + beta_j), one
// correct rounding to FP64 ("Profiling Ozaki II: The Cost Behind Fast INT8
// GEMMs" §1, red stage; §6 notes the reference implementation works in fixed
// one- or two-word precision — here the integer is kept exact in 160 bits).
//
// Integer only: w_t = R_t inv_t mod m_t (one multiply-high reduction),
// Y = sum_t w_t (M/m_t) accumulated in 64-bit limb sums, X = Y - k M with k
// estimated from the top limbs and corrected exactly, then the rounding is
// done on the bits of X and the double is assembled from its fields.
#include "oz2_internal.cuh"

namespace oz2 {
namespace {

// Bits [pos, pos + 64) of a 160-bit magnitude (pos >= 0; zeros above).
__device__ __forceinline__ uint64_t bits_at(const uint32_t (&x)[kLimbs], int pos) {
  uint64_t r = 0;
#pragma unroll
  for (int k = 0; k < kLimbs; ++k) {
    const int d = 32 * k - pos;
    const uint64_t v = x[k];
    if (d >= 0) {
      if (d < 64) r |= v << d;
    } else if (d > -32) {
      r |= v >> (-d);
    }
  }
  return r;
}

// Any bit set in positions [0, b)?
__device__ __forceinline__ bool sticky_below(const uint32_t (&x)[kLimbs], int b) {
  bool s = false;
#pragma unroll
  for (int k = 0; k < kLimbs; ++k) {
    const int lo = 32 * k;
    if (lo + 32 <= b) {
      s |= x[k] != 0;
    } else if (lo < b) {
      s |= (x[k] & ((1u << (b - lo)) - 1u)) != 0;
    }
  }
  return s;
}

// RN_even(sign * mag * 2^-k) as a double, subnormals and overflow included.
__device__ __forceinline__ double round_scaled(const uint32_t (&mag)[kLimbs], bool neg, int k) {
  int nb = 0;
#pragma unroll
  for (int i = 0; i < kLimbs; ++i)
    if (mag[i]) nb = 32 * i + (32 - __clz(static_cast<int>(mag[i])));
  if (nb == 0) return 0.0;
  int sh = nb - 53;                  // drop this many low bits for 53 significant bits
  if (k - 1074 > sh) sh = k - 1074;  // ... or more, below the subnormal threshold
  uint64_t m;
  if (sh <= 0) {
    m = bits_at(mag, 0) << (-sh);    // exact: mag < 2^53 here
  } else {
    const uint64_t q = bits_at(mag, sh);
    const bool rnd = (bits_at(mag, sh - 1) & 1ull) != 0;
    const bool st = sticky_below(mag, sh - 1);
    m = q + ((rnd && (st || (q & 1ull))) ? 1ull : 0ull);
    if (m == (1ull << 53)) {
      m = 1ull << 52;
      ++sh;
    }
  }
  uint64_t bits;
  if (m >= (1ull << 52)) {
    const int biased = sh - k + 1075;
    if (biased >= 2047) bits = 0x7FF0000000000000ull;
    else bits = (static_cast<uint64_t>(biased) << 52) | (m & ((1ull << 52) - 1));
  } else {
    bits = m;  // subnormal (sh == k - 1074)
  }
  if (neg) bits |= 1ull << 63;
  return __longlong_as_double(static_cast<long long>(bits));
}

// X >= y for X signed (top limb two's complement) and y a nonnegative constant?
__device__ __forceinline__ bool ge_const(const uint32_t (&X)[kLimbs], const uint32_t (&y)[kLimbs]) {
  int64_t c = 0;
#pragma unroll
  for (int k = 0; k < kLimbs - 1; ++k) {
    const int64_t t = static_cast<int64_t>(X[k]) - static_cast<int64_t>(y[k]) + c;
    c = t >> 32;
  }
  const int64_t top = static_cast<int64_t>(static_cast<int32_t>(X[kLimbs - 1])) -
                      static_cast<int64_t>(y[kLimbs - 1]) + c;
  return top >= 0;
}

// X += f * y (f in {-1, +1}), y a nonnegative constant.
__device__ __forceinline__ void add_scaled(uint32_t (&X)[kLimbs], const uint32_t (&y)[kLimbs], int f) {
  int64_t c = 0;
#pragma unroll
  for (int k = 0; k < kLimbs; ++k) {
    const int64_t t = static_cast<int64_t>(X[k]) + f * static_cast<int64_t>(y[k]) + c;
    X[k] = static_cast<uint32_t>(t);
    c = t >> 32;
  }
}

__global__ void __launch_bounds__(256) crt_kernel(int64_t p, int64_t r, const __grid_constant__ CrtConsts cc,
                                                  const uint8_t* __restrict__ R,
                                                  const int32_t* __restrict__ alpha,
                                                  const int32_t* __restrict__ beta,
                                                  double* __restrict__ C, int64_t ldc,
                                                  uint64_t* __restrict__ Xout) {
  const int64_t n = p * r;
  const int64_t plane = p * r;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = idx % p;
    const int64_t j = idx / p;
    const uint8_t* Rp = R + idx;  // R_t[j][i] = R[t * plane + j * p + i]
    uint64_t acc[kLimbs] = {0, 0, 0, 0, 0};
    for (int t = 0; t < cc.s; ++t) {
      const uint32_t m = static_cast<uint32_t>(cc.m[t]);
      const uint32_t x = static_cast<uint32_t>(Rp[t * plane]) * cc.inv[t];  // < 2^16
      const uint32_t w = x - __umulhi(x, cc.magic32[t]) * m;                   // x mod m
#pragma unroll
      for (int k = 0; k < kLimbs; ++k) acc[k] += static_cast<uint64_t>(w) * cc.Mt[t][k];
    }
    uint32_t Y[kLimbs];
    uint64_t carry = 0;
#pragma unroll
    for (int k = 0; k < kLimbs; ++k) {
      const uint64_t t = acc[k] + carry;
      Y[k] = static_cast<uint32_t>(t);
      carry = t >> 32;
    }
    // k = round(Y / M) from the top limbs (exactly corrected below)
    float yf = 0.0f;
    {
      const int top = cc.top;
      const float y2 = (top + 1 < kLimbs) ? static_cast<float>(Y[top + 1]) : 0.0f;
      yf = (y2 * 4294967296.0f + static_cast<float>(Y[top])) * 4294967296.0f +
           static_cast<float>(Y[top - 1]);
    }
    const int kq = static_cast<int>(floorf(yf * cc.inv_Mtop + 0.5f));
    uint32_t X[kLimbs];
    {
      int64_t c = 0;
#pragma unroll
      for (int k = 0; k < kLimbs; ++k) {
        const int64_t t = static_cast<int64_t>(Y[k]) - static_cast<int64_t>(kq) * cc.M[k] + c;
        X[k] = static_cast<uint32_t>(t);
        c = t >> 32;
      }
    }
    if (ge_const(X, cc.Mhalf)) add_scaled(X, cc.M, -1);  // X >= M/2: subtract M
    // X < -M/2  <=>  X + M/2 < 0
    {
      uint32_t Z[kLimbs];
#pragma unroll
      for (int k = 0; k < kLimbs; ++k) Z[k] = X[k];
      add_scaled(Z, cc.Mhalf, 1);
      if (static_cast<int32_t>(Z[kLimbs - 1]) < 0) add_scaled(X, cc.M, 1);
    }
    const bool neg = static_cast<int32_t>(X[kLimbs - 1]) < 0;
    if (Xout) {
      uint64_t* xo = Xout + idx * 3;
      xo[0] = (static_cast<uint64_t>(X[1]) << 32) | X[0];
      xo[1] = (static_cast<uint64_t>(X[3]) << 32) | X[2];
      xo[2] = static_cast<uint64_t>(static_cast<int64_t>(static_cast<int32_t>(X[4])));
    }
    uint32_t mag[kLimbs];
    if (neg) {
      uint64_t c = 1;
#pragma unroll
      for (int k = 0; k < kLimbs; ++k) {
        const uint64_t t = static_cast<uint64_t>(~X[k]) + c;
        mag[k] = static_cast<uint32_t>(t);
        c = t >> 32;
      }
    } else {
#pragma unroll
      for (int k = 0; k < kLimbs; ++k) mag[k] = X[k];
    }
    C[j * ldc + i] = round_scaled(mag, neg, alpha[i] + beta[j]);
  }
}

}  // namespace

cudaError_t launch_crt(int64_t p, int64_t r, int s, const CrtConsts& cc, const uint8_t* R,
                       const int32_t* alpha, const int32_t* beta, double* C, int64_t ldc,
                       uint64_t* X, cudaStream_t st) {
  (void)s;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n = p * r;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  crt_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(p, r, cc, R, alpha, beta, C, ldc, X);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace oz2
