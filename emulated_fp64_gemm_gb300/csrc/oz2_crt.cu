// CRT reconstruction and inverse scaling of Ozaki II: for every output entry,
// X = CRT_M(R_1..R_s) in [-M/2, M/2) and C = X 2^-(alpha_i + beta_j), one
// correct rounding to FP64 ("Profiling Ozaki II: The Cost Behind Fast INT8
// GEMMs" §1, red stage; §6 notes the reference implementation works in fixed
// one- or two-word precision — here the integer is kept exact in up to 160
// bits).
//
// The GEMM epilogue stores the CRT coefficients w_t = R_t (M/m_t)^-1 mod m_t
// (bytes), so here
//   Y = sum_t w_t (M/m_t)
// is accumulated as byte-limb sums S_b = sum_t w_t byte_b(M/m_t) with dp4a,
// four channels per instruction (each S_b < 2^20), and gathered into NL
// unnormalised 32-bit limbs (each < 2^46).  A float estimate of Y / M gives
// k = round(Y / M), and X = Y - k M follows with exact 64-bit carries.
// Because |X| <= M/2 - 1 always (the scaling bound of the method), X is in
// range unless Y / M lies within the estimate's error (far below 2^-12) of a
// half-integer; only then is X compared with M/2 exactly and moved by M.
// The rounding takes the top 64 bits of |X| with a sticky bit for the rest,
// converts them once with the correctly rounded u64 -> double conversion
// (the sticky bit sits 10 bits below the rounding position, so the result is
// RN of |X| itself) and scales by adding to the exponent field; a subnormal or
// overflowing result takes an exact integer rounding path instead.
#include <algorithm>

#include "oz2_internal.cuh"

namespace oz2 {
namespace {

// RN_even(X 2^-k) for X in NL 32-bit two's complement words, by exact integer
// rounding of the top 64 bits of |X| with a sticky bit for the rest: the path
// for results that are subnormal or overflow.
template <int NL>
__device__ __forceinline__ double round_x_exact(const uint32_t (&x)[NL], int k) {
  const bool neg = static_cast<int32_t>(x[NL - 1]) < 0;
  uint32_t mg[NL + 1];
  {
    uint64_t c = neg ? 1u : 0u;
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      const uint64_t t = static_cast<uint64_t>(neg ? ~x[j] : x[j]) + c;
      mg[j] = static_cast<uint32_t>(t);
      c = t >> 32;
    }
    mg[NL] = 0;
  }
  constexpr int NW = (NL + 1) / 2;
  uint64_t W[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) W[w] = static_cast<uint64_t>(mg[2 * w]) | (static_cast<uint64_t>(mg[2 * w + 1]) << 32);
  uint64_t hi, lo;
  bool st = false;
  int base;
  if (NW == 3) {
    if (W[2]) {
      hi = W[2];
      lo = W[1];
      st = W[0] != 0;
      base = 128;
    } else if (W[1]) {
      hi = W[1];
      lo = W[0];
      base = 64;
    } else {
      hi = W[0];
      lo = 0;
      base = 0;
    }
  } else {
    if (W[NW - 1]) {
      hi = W[NW - 1];
      lo = W[0];
      base = 64;
    } else {
      hi = W[0];
      lo = 0;
      base = 0;
    }
  }
  if (hi == 0) return 0.0;
  const int lz = __clzll(static_cast<long long>(hi));
  const uint64_t T = lz ? ((hi << lz) | (lo >> (64 - lz))) : hi;  // MSB at bit 63
  st = st || ((lo << lz) != 0);
  const int E = base + 63 - lz - k;  // |X| 2^-k in [2^E, 2^(E+1))
  uint64_t bits;
  if (E >= -1022 && E <= 1023) {
    uint64_t m = T >> 11;
    const bool g = (T >> 10) & 1ull;
    const bool rest = st || (T & 0x3FFull) != 0;
    m += (g && (rest || (m & 1ull))) ? 1ull : 0ull;
    bits = (static_cast<uint64_t>(E + 1022) << 52) + m;  // m's leading 1 (or a carry to 2^53) bumps the field
  } else if (E > 1023) {
    bits = 0x7FF0000000000000ull;
  } else {
    const int d = 11 + (-1022 - E);  // bits of T dropped for a subnormal result
    uint64_t m;
    bool rnd, s2;
    if (d < 64) {
      m = T >> d;
      rnd = (T >> (d - 1)) & 1ull;
      s2 = st || (T & ((1ull << (d - 1)) - 1ull)) != 0;
    } else {
      m = 0;
      rnd = (d == 64) ? (T >> 63) != 0 : false;
      s2 = st || (d == 64 ? (T & ~(1ull << 63)) != 0 : T != 0);
    }
    m += (rnd && (s2 || (m & 1ull))) ? 1ull : 0ull;
    bits = m;  // subnormal, or the smallest normal when rounding carried into bit 52
  }
  if (neg) bits |= 1ull << 63;
  return __longlong_as_double(static_cast<long long>(bits));
}

// C = RN_even(X 2^-k) for X in NL 32-bit two's complement words.
template <int NL>
__device__ __forceinline__ double round_x(const uint32_t (&x)[NL], int k) {
  const bool neg = static_cast<int32_t>(x[NL - 1]) < 0;
  uint32_t mg[NL + 1];
  {
    uint64_t c = neg ? 1u : 0u;
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      const uint64_t t = static_cast<uint64_t>(neg ? ~x[j] : x[j]) + c;
      mg[j] = static_cast<uint32_t>(t);
      c = t >> 32;
    }
    mg[NL] = 0;
  }
  constexpr int NW = (NL + 1) / 2;
  uint64_t W[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) W[w] = static_cast<uint64_t>(mg[2 * w]) | (static_cast<uint64_t>(mg[2 * w + 1]) << 32);
  uint64_t hi, lo;
  bool st = false;
  int base;
  if (NW == 3) {
    if (W[2]) {
      hi = W[2];
      lo = W[1];
      st = W[0] != 0;
      base = 128;
    } else if (W[1]) {
      hi = W[1];
      lo = W[0];
      base = 64;
    } else {
      hi = W[0];
      lo = 0;
      base = 0;
    }
  } else {
    if (W[NW - 1]) {
      hi = W[NW - 1];
      lo = W[0];
      base = 64;
    } else {
      hi = W[0];
      lo = 0;
      base = 0;
    }
  }
  if (hi == 0) return 0.0;  // X == 0
  const int lz = __clzll(static_cast<long long>(hi));
  const uint64_t T = lz ? ((hi << lz) | (lo >> (64 - lz))) : hi;  // top 64 bits of |X|, MSB at bit 63
  st = st || ((lo << lz) != 0);
  // |X| = (T + f) 2^(base - lz) with 0 <= f < 1
  const uint64_t db = static_cast<uint64_t>(__double_as_longlong(__ull2double_rn(T | (st ? 1ull : 0ull))));
  const int sc = base - lz - k;
  const int e = static_cast<int>(db >> 52) - 1023 + sc;  // unbiased exponent of the result
  if (e >= -1022 && e <= 1023) {
    uint64_t bits = db + (static_cast<uint64_t>(static_cast<int64_t>(sc)) << 52);
    if (neg) bits |= 1ull << 63;
    return __longlong_as_double(static_cast<long long>(bits));
  }
  return round_x_exact<NL>(x, k);  // subnormal or overflowing result
}

// Output rows [row0, row0 + rows).  W holds the coefficients as
// [s][r4][p_total][4] (four consecutive columns of one row per word); X has
// p_total rows per column.  Thread = (row i, group of 4 columns); x walks the
// rows, y a strided set of column groups.  MAXS: the largest s the instance
// serves; NL: 32-bit limbs of Y (crt_limbs); NBC: the byte limbs of the
// largest M/m_t (s - 1 for s >= 5); the dp4a loop stops there.  Four blocks
// per SM: the kernel is latency-bound (long dependent chains per output), so
// occupancy pays even with a few spilled registers.
template <int MAXS, int NL, int NBC>
__global__ void __launch_bounds__(256, 4) crt_kernel(int64_t row0, int64_t rows, int64_t p_total,
                                                     int64_t jg0, int64_t jg1, int64_t r,
                                                     const __grid_constant__ CrtConsts cc,
                                                     const uint8_t* __restrict__ Wb,
                                                     const int32_t* __restrict__ alpha,
                                                     const int32_t* __restrict__ beta,
                                                     double* __restrict__ C, int64_t ldc,
                                                     uint64_t* __restrict__ Xout) {
  const int64_t il = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (il >= rows) return;
  const int64_t i = row0 + il;
  const int64_t r4 = (r + 3) / 4;
  const int64_t plane = r4 * p_total;  // words per channel
  const uint32_t* W = reinterpret_cast<const uint32_t*>(Wb);
  const int ai = alpha[i];
  constexpr int NG = (MAXS + 3) / 4;  // channel groups of four
  constexpr int NB = 4 * NL;          // byte limbs of Y
  static_assert(NBC <= NB, "coefficient bytes within the limbs");
  for (int64_t jg = jg0 + blockIdx.y; jg < jg1; jg += gridDim.y) {
    const int64_t base = jg * p_total + i;
    uint32_t wv[4 * NG];
#pragma unroll
    for (int t = 0; t < 4 * NG; ++t) wv[t] = (t < cc.s) ? __ldg(W + t * plane + base) : 0u;
    // 4x4 byte transpose per group: word 4g + v then holds output v's channels 4g .. 4g + 3
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const uint32_t lo01 = __byte_perm(wv[4 * g], wv[4 * g + 1], 0x5140u);
      const uint32_t hi01 = __byte_perm(wv[4 * g], wv[4 * g + 1], 0x7362u);
      const uint32_t lo23 = __byte_perm(wv[4 * g + 2], wv[4 * g + 3], 0x5140u);
      const uint32_t hi23 = __byte_perm(wv[4 * g + 2], wv[4 * g + 3], 0x7362u);
      wv[4 * g + 0] = __byte_perm(lo01, lo23, 0x5410u);
      wv[4 * g + 1] = __byte_perm(lo01, lo23, 0x7632u);
      wv[4 * g + 2] = __byte_perm(hi01, hi23, 0x5410u);
      wv[4 * g + 3] = __byte_perm(hi01, hi23, 0x7632u);
    }
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int64_t j = jg * 4 + v;
      if (j >= r) break;
      // byte-limb sums S_b = sum_t w_t byte_b(M/m_t); byte 0 of M/m_t is zero
      // for t >= 1 (256 divides it), so only the first group takes b = 0
      // (no guards on s: the words past s and the table bytes past each M/m_t
      // are zero)
      uint32_t S[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) S[b] = 0;
#pragma unroll
      for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int b = 0; b < NBC; ++b)
          if (b > 0 || g == 0) S[b] = __dp4a(wv[4 * g + v], cc.L4[g][b], S[b]);
      // unnormalised 32-bit limbs of Y (each < 2^46)
      uint64_t Y[NL];
#pragma unroll
      for (int q = 0; q < NL; ++q) {
        const uint32_t lo = S[4 * q] + (S[4 * q + 1] << 8);
        const uint32_t hi = S[4 * q + 2] + (S[4 * q + 3] << 8);
        Y[q] = (static_cast<uint64_t>(hi) << 16) + lo;
      }
      // Y / M in float from every limb that can move it by 2^-49 or more:
      // relative error a few 2^-24, far below the 2^-12 margin used below
      float ye = 0.0f;
#pragma unroll
      for (int q = 0; q < NL; ++q)
        if (q >= cc.est_lo) ye += __ull2float_rn(Y[q]) * __int_as_float((127 + 32 * (q - NL + 1)) << 23);
      const float yq = ye * cc.inv_Ms;
      const float kf = rintf(yq);
      const int kq = static_cast<int>(kf);
      uint32_t x[NL];
      {
        int64_t carry = 0;
#pragma unroll
        for (int q = 0; q < NL; ++q) {
          const int64_t z = static_cast<int64_t>(Y[q]) + carry - static_cast<int64_t>(kq) * cc.M[q];
          x[q] = static_cast<uint32_t>(z);
          carry = z >> 32;
        }
      }
      // exact correction into [-M/2, M/2), only near a half-integer Y / M
      if (fabsf(yq - kf) > 0.5f - 0x1p-12f) {
        int64_t c = 0;
        uint32_t top = 0;
#pragma unroll
        for (int l = 0; l < NL; ++l) {  // sign of X - M/2
          const int64_t t = static_cast<int64_t>(x[l]) - static_cast<int64_t>(cc.Mhalf[l]) + c;
          top = static_cast<uint32_t>(t);
          c = t >> 32;
        }
        int fix = (static_cast<int32_t>(top) >= 0) ? -1 : 0;
        c = 0;
#pragma unroll
        for (int l = 0; l < NL; ++l) {  // sign of X + M/2
          const int64_t t = static_cast<int64_t>(x[l]) + static_cast<int64_t>(cc.Mhalf[l]) + c;
          top = static_cast<uint32_t>(t);
          c = t >> 32;
        }
        if (static_cast<int32_t>(top) < 0) fix = 1;
        if (fix) {
          c = 0;
#pragma unroll
          for (int l = 0; l < NL; ++l) {
            const int64_t t = static_cast<int64_t>(x[l]) + fix * static_cast<int64_t>(cc.M[l]) + c;
            x[l] = static_cast<uint32_t>(t);
            c = t >> 32;
          }
        }
      }
      if (Xout) {
        const bool neg = static_cast<int32_t>(x[NL - 1]) < 0;
        uint32_t ext[6];
#pragma unroll
        for (int l = 0; l < 6; ++l) ext[l] = (l < NL) ? x[l] : (neg ? 0xFFFFFFFFu : 0u);
        uint64_t* xo = Xout + (j * p_total + i) * 3;
        xo[0] = (static_cast<uint64_t>(ext[1]) << 32) | ext[0];
        xo[1] = (static_cast<uint64_t>(ext[3]) << 32) | ext[2];
        xo[2] = (static_cast<uint64_t>(ext[5]) << 32) | ext[4];
      }
      C[j * ldc + i] = round_x<NL>(x, ai + beta[j]);
    }
  }
}

// Checking path: R_t[j][i] = w_t (M/m_t) mod m_t from the coefficient layout.
__global__ void w_to_r_kernel(const uint8_t* __restrict__ W, int64_t p, int64_t r, ModConsts mc,
                              uint8_t* __restrict__ R) {
  const int64_t per_plane = p * r;
  const int64_t r4 = (r + 3) / 4;
  const int64_t n = per_plane * mc.s;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(idx / per_plane);
    const int64_t rem = idx - t * per_plane;
    const int64_t j = rem / p;
    const int64_t i = rem - j * p;
    const uint32_t w = W[((t * r4 + j / 4) * p + i) * 4 + (j % 4)];
    R[idx] = static_cast<uint8_t>((w * mc.crt_c[t]) % static_cast<uint32_t>(mc.m[t]));
  }
}

}  // namespace

cudaError_t launch_crt(int64_t row0, int64_t rows, int64_t p_total, int64_t col0, int64_t cols,
                       int64_t r, int s, const CrtConsts& cc, const uint8_t* W,
                       const int32_t* alpha, const int32_t* beta, double* C, int64_t ldc,
                       uint64_t* X, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t jg0 = col0 / 4;
  const int64_t jg1 = std::min<int64_t>((col0 + cols + 3) / 4, (r + 3) / 4);
  const int64_t gx = (rows + 255) / 256;
  // about 16 blocks per SM in total; each y index walks (jg1 - jg0) / gy column groups
  int64_t gy = (static_cast<int64_t>(sms) * 16 + gx - 1) / gx;
  if (gy > jg1 - jg0) gy = jg1 - jg0;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  const dim3 b(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  const int nl = crt_limbs(s);
  // exact instances for the common channel counts (fewer groups and byte
  // limbs), else the limb-count buckets with MAXS - 1 coefficient bytes
  if (s == 8) crt_kernel<8, 3, 7><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
  else if (s == 14) crt_kernel<14, 4, 13><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
  else if (s == 18) crt_kernel<18, 5, 17><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
  else if (nl == 3) crt_kernel<11, 3, 10><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
  else if (nl == 4) crt_kernel<15, 4, 14><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
  else crt_kernel<20, 5, 19><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_w_to_r(const uint8_t* W, int64_t p, int64_t r, const ModConsts& mc, uint8_t* R,
                          cudaStream_t st) {
  w_to_r_kernel<<<1024, 256, 0, st>>>(W, p, r, mc, R);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace oz2
