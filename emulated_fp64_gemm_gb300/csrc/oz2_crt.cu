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
// four channels per instruction (each S_b < 2^20).  k = round(Y / M) comes
// from a float sum of the top byte-limb sums weighted by 2^(8b) / M, and
// X = Y - k M is carried through 16-bit limbs in 32-bit arithmetic.  Because
// |X| <= M/2 - 1 always (the scaling bound of the method), X is in range
// unless Y / M lies within the estimate's error (far below 2^-12) of a
// half-integer; only then is X compared with M/2 exactly and moved by M.
// The rounding takes a signed 64-bit window of X (sign bit, then the first
// bit that differs from it) with a sticky bit for the rest, converts it once
// with the correctly rounded signed 64-bit -> double conversion (the sticky
// bit sits 9 bits below the rounding position, so the result is RN of X
// itself) and scales by adding to the exponent field; a subnormal or
// overflowing result takes an exact integer rounding path instead.
//
// The device's FP64 pipe also executes every 64-bit integer <-> floating
// conversion and runs at a small fraction of the other pipes' rate, so the
// kernel keeps to one such conversion per output; the quotient estimate uses
// 32-bit conversions only.
#include <algorithm>

#include "oz2_internal.cuh"

namespace oz2 {
namespace {

__device__ __forceinline__ uint64_t pack64(uint32_t hi, uint32_t lo) {
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// RN_even(X 2^-k) for X in NL 32-bit two's complement words (x0 lowest; the
// words past NL are ignored), by exact integer rounding of the top 64 bits of
// |X| with a sticky bit for the rest: the path for results that are subnormal
// or overflow.  Out of line, with the words in registers.
template <int NL>
__device__ __noinline__ double round_x_exact(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3,
                                             uint32_t x4, int k) {
  const uint32_t xin[5] = {x0, x1, x2, x3, x4};
  const bool neg = static_cast<int32_t>(xin[NL - 1]) < 0;
  uint32_t mg[6] = {0, 0, 0, 0, 0, 0};
  {
    uint64_t c = neg ? 1u : 0u;
#pragma unroll
    for (int j = 0; j < NL; ++j) {
      const uint64_t t = static_cast<uint64_t>(neg ? ~xin[j] : xin[j]) + c;
      mg[j] = static_cast<uint32_t>(t);
      c = t >> 32;
    }
  }
  const uint64_t W0 = pack64(mg[1], mg[0]), W1 = pack64(mg[3], mg[2]), W2 = pack64(mg[5], mg[4]);
  uint64_t hi, lo;
  bool st = false;
  int base;
  if (W2) {
    hi = W2;
    lo = W1;
    st = W0 != 0;
    base = 128;
  } else if (W1) {
    hi = W1;
    lo = W0;
    base = 64;
  } else {
    hi = W0;
    lo = 0;
    base = 0;
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

// C = RN_even(X 2^-k) for X in NL 32-bit two's complement words.  T is a
// signed 64-bit window of X whose top bit is the sign and whose next bit is
// the first that differs from it (or all of X when it fits in 64 bits), so
// X = (T + f) 2^sh with 0 <= f < 1.  Setting bit 0 of T when f > 0 leaves the
// rounding unchanged: the rounding position of |T| >= 2^62 is bit 10, and an
// odd value 9 bits below it is never a tie nor across one from T + f.
template <int NL>
__device__ __forceinline__ double round_x(const uint32_t (&x)[NL], int k) {
  int64_t H;
  uint64_t L;
  bool st = false;
  int base = 64;
  if constexpr (NL == 3) {
    H = static_cast<int32_t>(x[2]);
    L = pack64(x[1], x[0]);
  } else if constexpr (NL == 4) {
    H = static_cast<int64_t>(pack64(x[3], x[2]));
    L = pack64(x[1], x[0]);
  } else {
    static_assert(NL == 5, "three to five words");
    const int64_t H2 = static_cast<int32_t>(x[4]);
    const uint64_t M1 = pack64(x[3], x[2]);
    const uint64_t L0 = pack64(x[1], x[0]);
    if (H2 != (static_cast<int64_t>(M1) >> 63)) {  // X needs the top word
      H = H2;
      L = M1;
      st = L0 != 0;
      base = 128;
    } else {
      H = static_cast<int64_t>(M1);
      L = L0;
    }
  }
  int64_t T;
  int sh;
  if (H == (static_cast<int64_t>(L) >> 63)) {  // the window is L itself
    T = static_cast<int64_t>(L);
    sh = base - 64;
    if (T == 0 && !st) return 0.0;
  } else {
    const int n = __clzll(H ^ (H >> 63)) - 1;  // redundant sign bits of H: 0 .. 63
    T = n ? static_cast<int64_t>((static_cast<uint64_t>(H) << n) | (L >> (64 - n))) : H;
    st = st || ((L << n) != 0);
    sh = base - n;
  }
  const uint64_t db = static_cast<uint64_t>(__double_as_longlong(__ll2double_rn(T | (st ? 1ll : 0ll))));
  const int sc = sh - k;
  const int e = static_cast<int>((db >> 52) & 0x7FF) - 1023 + sc;  // unbiased exponent of the result
  if (e >= -1022 && e <= 1023)
    return __longlong_as_double(static_cast<long long>(db + (static_cast<uint64_t>(static_cast<int64_t>(sc)) << 52)));
  return round_x_exact<NL>(x[0], x[1], x[2], NL > 3 ? x[NL > 3 ? 3 : 0] : 0u, NL > 4 ? x[NL > 4 ? 4 : 0] : 0u,
                           k);  // subnormal or overflowing result
}

// Output rows [row0, row0 + rows).  W holds the coefficients as
// [s][r4][p_total][4] (four consecutive columns of one row per word); X has
// p_total rows per column.  Thread = (row i, group of 4 columns); x walks the
// rows, y a strided set of column groups.  MAXS: the largest s the instance
// serves; NL: 32-bit words of Y (crt_limbs); NBC: the byte limbs of the
// largest M/m_t (s - 1 for s >= 5), where the dp4a loop stops; EB0: the lowest
// byte-limb sum the quotient estimate takes (below it the sums move Y / M by
// less than 2^-36 for every s the instance serves); MINB: blocks per SM (the
// kernel is issue-bound; four where the registers allow it without spills);
// WX: also write X (checking path).
template <int MAXS, int NL, int NBC, int EB0, int MINB, bool WX>
__global__ void __launch_bounds__(256, MINB) crt_kernel(int64_t row0, int64_t rows, int64_t p_total,
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
  constexpr int NL16 = 2 * NL;        // 16-bit limbs of X
  static_assert(NBC <= 2 * NL16, "coefficient bytes within the limbs");
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
      uint32_t S[2 * NL16];
#pragma unroll
      for (int b = 0; b < 2 * NL16; ++b) S[b] = 0;
#pragma unroll
      for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int b = 0; b < NBC; ++b)
          if (b > 0 || g == 0) S[b] = __dp4a(wv[4 * g + v], cc.L4[g][b], S[b]);
      // Y / M in float: each S_b < 2^20 converts exactly; the error is a few
      // 2^-20, far below the 2^-12 margin used below.  k = RN_even(Y / M) by
      // adding 1.5 2^23 (the float's integer part then sits in its low bits).
      float yq = 0.0f;
#pragma unroll
      for (int b = EB0; b < NBC; ++b) yq = __fmaf_rn(__uint2float_rn(S[b]), cc.est_f[b], yq);
      const float tq = yq + 12582912.0f;
      const int kq = __float_as_int(tq) - 0x4B400000;
      const float kf = tq - 12582912.0f;
      // X = Y - k M in 16-bit limbs: Z_q = S_2q + 2^8 S_2q+1 - k M16_q + carry
      // (|Z_q| < 2^30), carry = floor(Z_q / 2^16); the last carry is the sign
      // extension since |X| < M < 2^(32 NL - 1)
      uint32_t x[NL];
      {
        int32_t c = 0;
        int32_t Z[NL16];
#pragma unroll
        for (int q = 0; q < NL16; ++q) {
          const int32_t V = static_cast<int32_t>(S[2 * q] + (S[2 * q + 1] << 8));
          Z[q] = V - kq * static_cast<int32_t>(cc.M16[q]) + c;
          c = Z[q] >> 16;
        }
#pragma unroll
        for (int w = 0; w < NL; ++w)
          x[w] = __byte_perm(static_cast<uint32_t>(Z[2 * w]), static_cast<uint32_t>(Z[2 * w + 1]), 0x5410u);
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
      if constexpr (WX) {
        const bool neg = static_cast<int32_t>(x[NL - 1]) < 0;
        uint32_t ext[6];
#pragma unroll
        for (int l = 0; l < 6; ++l) ext[l] = (l < NL) ? x[l] : (neg ? 0xFFFFFFFFu : 0u);
        uint64_t* xo = Xout + (j * p_total + i) * 3;
        xo[0] = pack64(ext[1], ext[0]);
        xo[1] = pack64(ext[3], ext[2]);
        xo[2] = pack64(ext[5], ext[4]);
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
#define OZ2_CRT(MAXS, NL, NBC, EB0, MINB, WX) \
  crt_kernel<MAXS, NL, NBC, EB0, MINB, WX><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X)
  if (X) {
    // checking path: one instance per word count
    if (nl == 3) OZ2_CRT(11, 3, 10, 0, 4, true);
    else if (nl == 4) OZ2_CRT(15, 4, 14, 5, 4, true);
    else OZ2_CRT(20, 5, 19, 9, 3, true);
  } else if (s == 8) {
    OZ2_CRT(8, 3, 7, 1, 4, false);
  } else if (s == 14) {
    OZ2_CRT(14, 4, 13, 7, 4, false);
  } else if (s == 18) {
    OZ2_CRT(18, 5, 17, 11, 3, false);
  } else if (nl == 3) {  // the other counts: buckets by word count, MAXS - 1 coefficient bytes
    OZ2_CRT(11, 3, 10, 0, 4, false);
  } else if (nl == 4) {
    OZ2_CRT(15, 4, 14, 5, 4, false);
  } else {
    OZ2_CRT(20, 5, 19, 9, 3, false);
  }
#undef OZ2_CRT
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
