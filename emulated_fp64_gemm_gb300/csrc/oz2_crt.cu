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

// Exact CRT of one output entry from its s residues (byte lanes of rv across
// VEC entries), accumulated in 64-bit sums of 32-bit limbs.  NL limbs hold
// every sum_t w_t M/m_t (< s M); MAXS bounds s at compile time so the
// channel loop unrolls and every constant is an immediate operand.
template <int NL>
__device__ __forceinline__ double crt_finish(uint64_t (&acc)[NL], const CrtConsts& cc, int k,
                                             uint64_t* xo) {
  uint32_t Y[NL];
  uint64_t carry = 0;
#pragma unroll
  for (int l = 0; l < NL; ++l) {
    const uint64_t t = acc[l] + carry;
    Y[l] = static_cast<uint32_t>(t);
    carry = t >> 32;
  }
  // quotient estimate from the top three limbs scaled as a float (the
  // dropped limbs change Y/M by far less than the float rounding; an estimate
  // one off is corrected exactly below)
  const float yf = static_cast<float>(Y[NL - 1]) + static_cast<float>(Y[NL - 2]) * 0x1p-32f +
                   static_cast<float>(Y[NL - 3]) * 0x1p-64f;
  const int kq = static_cast<int>(floorf(yf * cc.inv_Mtop + 0.5f));
  uint32_t X[NL];
  {
    int64_t c = 0;
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      const int64_t t = static_cast<int64_t>(Y[l]) - static_cast<int64_t>(kq) * cc.M[l] + c;
      X[l] = static_cast<uint32_t>(t);
      c = t >> 32;
    }
  }
  // exact correction into [-M/2, M/2): compare the top 64 bits, full compare on a tie
  {
    const int64_t xt = static_cast<int64_t>((static_cast<uint64_t>(X[NL - 1]) << 32) | X[NL - 2]);
    const int64_t ht = static_cast<int64_t>((static_cast<uint64_t>(cc.Mhalf[NL - 1]) << 32) | cc.Mhalf[NL - 2]);
    int fix = 0;
    if (xt > ht) fix = -1;
    else if (xt < -ht - 1) fix = 1;
    else if (xt == ht || xt == -ht - 1) {
      // tie on the top limbs: decide with all limbs (X >= M/2 or X < -M/2)
      int64_t c = 0;
      uint32_t top = 0;
#pragma unroll
      for (int l = 0; l < NL; ++l) {
        const int64_t t = static_cast<int64_t>(X[l]) - static_cast<int64_t>(cc.Mhalf[l]) + c;
        top = static_cast<uint32_t>(t);
        c = t >> 32;
      }
      if (static_cast<int32_t>(top) >= 0) fix = -1;
      c = 0;
#pragma unroll
      for (int l = 0; l < NL; ++l) {
        const int64_t t = static_cast<int64_t>(X[l]) + static_cast<int64_t>(cc.Mhalf[l]) + c;
        top = static_cast<uint32_t>(t);
        c = t >> 32;
      }
      if (static_cast<int32_t>(top) < 0) fix = 1;
    }
    if (fix) {
      int64_t c = 0;
#pragma unroll
      for (int l = 0; l < NL; ++l) {
        const int64_t t = static_cast<int64_t>(X[l]) + fix * static_cast<int64_t>(cc.M[l]) + c;
        X[l] = static_cast<uint32_t>(t);
        c = t >> 32;
      }
    }
  }
  const bool neg = static_cast<int32_t>(X[NL - 1]) < 0;
  if (xo) {
    uint32_t ext[6];
#pragma unroll
    for (int l = 0; l < 6; ++l) ext[l] = (l < NL) ? X[l] : (neg ? 0xFFFFFFFFu : 0u);
    xo[0] = (static_cast<uint64_t>(ext[1]) << 32) | ext[0];
    xo[1] = (static_cast<uint64_t>(ext[3]) << 32) | ext[2];
    xo[2] = (static_cast<uint64_t>(ext[5]) << 32) | ext[4];
  }
  // magnitude
  uint32_t mag[NL];
  {
    uint64_t c = neg ? 1u : 0u;
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      const uint64_t t = static_cast<uint64_t>(neg ? ~X[l] : X[l]) + c;
      mag[l] = static_cast<uint32_t>(t);
      c = t >> 32;
    }
  }
  // move the top nonzero limb to position NL-1
  int drop = 0;  // limbs shifted in from below
#pragma unroll
  for (int st = 0; st < NL - 1; ++st) {
    if (mag[NL - 1] == 0) {
#pragma unroll
      for (int l = NL - 1; l > 0; --l) mag[l] = mag[l - 1];
      mag[0] = 0;
      ++drop;
    }
  }
  if (mag[NL - 1] == 0) return 0.0;
  const int lz = __clz(static_cast<int>(mag[NL - 1]));
  const uint64_t hi = (static_cast<uint64_t>(mag[NL - 1]) << 32) | mag[NL - 2];
  const uint32_t l3 = mag[NL - 3];
  const uint64_t T = lz ? ((hi << lz) | (l3 >> (32 - lz))) : hi;  // top 64 bits, MSB at 63
  bool sticky = lz ? ((l3 << lz) != 0) : (l3 != 0);
#pragma unroll
  for (int l = 0; l < NL - 3; ++l) sticky |= mag[l] != 0;
  const int nb = 32 * (NL - drop) - lz;  // bit length of |X|
  int E = nb - 1 - k;                     // |X| 2^-k in [2^E, 2^(E+1))
  int d = 11;                             // bits of T dropped for 53 significant bits
  if (E < -1022) d += -1022 - E;          // subnormal result: drop more
  uint64_t m;
  bool rnd, st;
  if (d < 64) {
    m = T >> d;
    rnd = (T >> (d - 1)) & 1ull;
    st = sticky || (T & ((1ull << (d - 1)) - 1ull)) != 0;
  } else {
    m = 0;
    rnd = (d == 64) ? (T >> 63) != 0 : false;
    st = sticky || (d == 64 ? (T & ~(1ull << 63)) != 0 : T != 0);
  }
  m += (rnd && (st || (m & 1ull))) ? 1ull : 0ull;
  uint64_t bits;
  if (E >= -1022) {
    if (m == (1ull << 53)) {
      m >>= 1;
      ++E;
    }
    bits = (E + 1023 >= 2047) ? 0x7FF0000000000000ull
                              : ((static_cast<uint64_t>(E + 1023) << 52) | (m & ((1ull << 52) - 1)));
  } else {
    bits = m;  // subnormal, or the smallest normal when rounding carried into bit 52
  }
  if (neg) bits |= 1ull << 63;
  return __longlong_as_double(static_cast<long long>(bits));
}

// Output rows [row0, row0 + rows); R and X have p_total rows per column.
template <int MAXS, int NL, int VEC>
__global__ void __launch_bounds__(256) crt_kernel(int64_t row0, int64_t rows, int64_t p_total, int64_t r,
                                                  const __grid_constant__ CrtConsts cc,
                                                  const uint8_t* __restrict__ R,
                                                  const int32_t* __restrict__ alpha,
                                                  const int32_t* __restrict__ beta,
                                                  double* __restrict__ C, int64_t ldc,
                                                  uint64_t* __restrict__ Xout) {
  const int64_t pv = rows / VEC;
  const int64_t groups = pv * r;
  const int64_t plane = p_total * r;
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < groups;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t j = g / pv;
    const int64_t i0 = row0 + (g - j * pv) * VEC;
    const int64_t base = j * p_total + i0;
    uint64_t acc[VEC][NL];
#pragma unroll
    for (int v = 0; v < VEC; ++v)
#pragma unroll
      for (int l = 0; l < NL; ++l) acc[v][l] = 0;
#pragma unroll
    for (int t = 0; t < MAXS; ++t) {
      if (t < cc.s) {
        uint32_t rv;
        if (VEC == 4) rv = __ldg(reinterpret_cast<const uint32_t*>(R + t * plane + base));
        else rv = __ldg(R + t * plane + base);
        const uint32_t m = static_cast<uint32_t>(cc.m[t]);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
          const uint32_t x = ((rv >> (8 * v)) & 255u) * cc.inv[t];  // < 2^16
          const uint32_t w = x - __umulhi(x, cc.magic32[t]) * m;   // x mod m
#pragma unroll
          for (int l = 0; l < NL; ++l) acc[v][l] += static_cast<uint64_t>(w) * cc.Mt[t][l];
        }
      }
    }
    const int bj = beta[j];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      const int64_t i = i0 + v;
      C[j * ldc + i] = crt_finish<NL>(acc[v], cc, alpha[i] + bj, Xout ? Xout + (base + v) * 3 : nullptr);
    }
  }
}

}  // namespace

cudaError_t launch_crt(int64_t row0, int64_t rows, int64_t p_total, int64_t r, int s,
                       const CrtConsts& cc, const uint8_t* R, const int32_t* alpha,
                       const int32_t* beta, double* C, int64_t ldc, uint64_t* X, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool vec = (rows % 4) == 0 && (row0 % 4) == 0 && (p_total % 4) == 0;
  const int64_t groups = (vec ? rows / 4 : rows) * r;
  int64_t blocks = (groups + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const unsigned b = static_cast<unsigned>(blocks);
  const int nl = crt_limbs(s);
#define OZ2_CRT_LAUNCH(MS, NLV, V) \
  crt_kernel<MS, NLV, V><<<b, 256, 0, st>>>(row0, rows, p_total, r, cc, R, alpha, beta, C, ldc, X)
  if (nl == 3) {
    if (vec) OZ2_CRT_LAUNCH(11, 3, 4);
    else OZ2_CRT_LAUNCH(11, 3, 1);
  } else if (nl == 4) {
    if (vec) OZ2_CRT_LAUNCH(15, 4, 4);
    else OZ2_CRT_LAUNCH(15, 4, 1);
  } else {
    if (vec) OZ2_CRT_LAUNCH(20, 5, 4);
    else OZ2_CRT_LAUNCH(20, 5, 1);
  }
#undef OZ2_CRT_LAUNCH
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace oz2
