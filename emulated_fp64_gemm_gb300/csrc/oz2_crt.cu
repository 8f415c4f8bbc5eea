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
#include <algorithm>

#include "oz2_internal.cuh"

namespace oz2 {
namespace {

// Exact CRT of one output entry.  The GEMM epilogue stores the CRT
// coefficients w_t = R_t (M/m_t)^-1 mod m_t, so here Y = sum_t w_t (M/m_t) is
// accumulated carry-free: with M/m_t in 16-bit limbs every term w_t L is below
// 2^24 and each limb sum below s 2^24 < 2^29.  NL16 limbs (2 x crt_limbs(s))
// hold every Y < s M; MAXS bounds s at compile time so the channel loop
// unrolls with the constants as immediate operands.
template <int NL>
__device__ __forceinline__ double crt_round_x(uint32_t (&X)[NL], const CrtConsts& cc, int k, uint64_t* xo);

template <int NL16>
__device__ __forceinline__ double crt_finish(const uint32_t (&acc)[NL16], const CrtConsts& cc, int k,
                                             uint64_t* xo) {
  constexpr int NL = NL16 / 2;
  // quotient estimate k ~ round(Y / M) from all limbs as a float (an estimate
  // one off is corrected exactly below)
  // (the top six limbs only: below them the sum changes Y / M by < 2^-60)
  float yf = 0.0f;
#pragma unroll
  for (int l = (NL16 > 6 ? NL16 - 6 : 0); l < NL16; ++l)
    yf += static_cast<float>(acc[l]) * __int_as_float((127 + 16 * (l - NL16 + 1)) << 23);
  const int kq = static_cast<int>(floorf(yf * cc.inv_Mest + 0.5f));
  // X = Y - k M in 16-bit limbs (signed), then carries
  uint32_t X[NL];
  {
    int32_t c = 0;
    uint32_t limb[NL16];
#pragma unroll
    for (int l = 0; l < NL16; ++l) {
      const int32_t v = static_cast<int32_t>(acc[l]) - kq * static_cast<int32_t>(cc.M16[l]) + c;
      limb[l] = static_cast<uint32_t>(v) & 0xFFFFu;
      c = v >> 16;  // arithmetic: floor division by 2^16
    }
#pragma unroll
    for (int l = 0; l < NL; ++l) X[l] = limb[2 * l] | (limb[2 * l + 1] << 16);
    // the final carry is the sign extension: |X| < 2^(32 NL - 1), so the top bit of X[NL - 1] is the sign
  }
  return crt_round_x<NL>(X, cc, k, xo);
}

// X = Y - k M (two's complement in NL 32-bit words, within one M of the
// target range) -> exact correction into [-M/2, M/2), then C = RN(X 2^-k).
template <int NL>
__device__ __forceinline__ double crt_round_x(uint32_t (&X)[NL], const CrtConsts& cc, int k, uint64_t* xo) {
  // exact correction into [-M/2, M/2): compare the top 64 bits, full compare on a tie
  {
    const int64_t xt = static_cast<int64_t>((static_cast<uint64_t>(X[NL - 1]) << 32) | X[NL - 2]);
    const int64_t ht = static_cast<int64_t>((static_cast<uint64_t>(cc.Mhalf[NL - 1]) << 32) | cc.Mhalf[NL - 2]);
    int fix = 0;
    if (xt > ht) fix = -1;
    else if (xt < -ht - 1) fix = 1;
    else if (xt == ht || xt == -ht - 1) {
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
  int drop = 0;
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

// Output rows [row0, row0 + rows).  W holds the coefficients as
// [s][r4][p_total][4] (four consecutive columns of one row per word); X has
// p_total rows per column.  Thread = (row i, group of 4 columns); x walks the
// rows, y a strided set of column groups.  NBC: the byte limbs of the largest
// M/m_t for s <= MAXS (s - 1 for s >= 5); the dp4a loop stops there.
// MINB: resident blocks per SM the register allocation must allow.  The
// kernel is latency-bound (long dependent chains per output), so occupancy
// pays even with a few spilled registers: at 8192^2, s = 14 three blocks per
// SM took 707 -> 612 us, and at s = 18 four blocks 919 -> 880 us; at s = 8 the
// unconstrained allocation already fits four.
template <int MAXS, int NL16, int NBC, int MINB>
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
  for (int64_t jg = jg0 + blockIdx.y; jg < jg1; jg += gridDim.y) {
    const int64_t base = jg * p_total + i;
    constexpr int NG = (MAXS + 3) / 4;  // channel groups of four
    constexpr int NB8 = 2 * NL16;       // byte limbs of the sums
    static_assert(NBC <= NB8, "coefficient bytes within the sum's limbs");
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
    // one output column v of the four, from its coefficient word of each group
    auto one_output = [&](int v, const uint32_t (&wsel)[NG]) {
      const int64_t j = jg * 4 + v;
      // Y in byte limbs: S_b = sum_t w_t byte_b(M/m_t), four channels per dp4a (S_b < 2^20)
      uint32_t acc8[NB8];
#pragma unroll
      for (int b = 0; b < NB8; ++b) acc8[b] = 0;
      // (no guards on s: the words past s and the table bytes past each
      // M/m_t are zero, and a uniform branch per dp4a would cost more issue
      // slots than the zero products)
#pragma unroll
      for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int b = 0; b < NBC; ++b) acc8[b] = __dp4a(wsel[g], cc.L4[g][b], acc8[b]);
      // 16-bit limb sums (each below 2^29) as the finishing step expects
      uint32_t acc[NL16];
#pragma unroll
      for (int l = 0; l < NL16; ++l) acc[l] = acc8[2 * l] + (acc8[2 * l + 1] << 8);
      C[j * ldc + i] = crt_finish<NL16>(acc, cc, ai + beta[j], Xout ? Xout + (j * p_total + i) * 3 : nullptr);
    };
    if constexpr (NL16 <= 8) {
      // unrolled: the four outputs' words are compile-time indices (at 10
      // limbs the unrolled loop took 171 registers and ran slower)
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        if (jg * 4 + v >= r) break;
        uint32_t wsel[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) wsel[g] = wv[4 * g + v];
        one_output(v, wsel);
      }
    } else {
#pragma unroll 1
      for (int v = 0; v < 4; ++v) {
        if (jg * 4 + v >= r) break;
        uint32_t wsel[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          // (select this output's word without dynamic register indexing)
          uint32_t wg = wv[4 * g];
          wg = (v == 1) ? wv[4 * g + 1] : wg;
          wg = (v == 2) ? wv[4 * g + 2] : wg;
          wg = (v == 3) ? wv[4 * g + 3] : wg;
          wsel[g] = wg;
        }
        one_output(v, wsel);
      }
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
  if (s == 8) crt_kernel<8, 6, 7, 1><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
  else if (s == 14) crt_kernel<14, 8, 13, 3><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
  else if (s == 18) crt_kernel<18, 10, 17, 4><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
  else if (nl == 3) crt_kernel<11, 6, 10, 1><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
  else if (nl == 4) crt_kernel<15, 8, 14, 3><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
  else crt_kernel<20, 10, 19, 4><<<b, 256, 0, st>>>(row0, rows, p_total, jg0, jg1, r, cc, W, alpha, beta, C, ldc, X);
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
