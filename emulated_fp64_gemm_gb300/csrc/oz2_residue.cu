// Residue planes of the Ozaki-II pipeline: for every element of A (or B),
// A_t = rho_{m_t}(trunc(2^alpha_i a)) for all s channels in one pass, written
// as fp16 planes (integers in [-128, 127] are exact in fp16); plus the
// one-read kernels that also compute the fast-mode statistics and exponents.
//
// Method: "Profiling Ozaki II: The Cost Behind Fast INT8 GEMMs" §1 (green
// stage: truncate toward zero, then one centered residue per modulus), §10.1
// (convert each scaled element to an integer once, then reduce it with
// fixed-divisor integer arithmetic per modulus); centered residues: "Ozaki II
// supplement: INT8 range conditions and paper performance results" §1.2.
//
// The channel loop is specialised at compile time on a channel bucket SB
// (8, 14 or 20 channels, every s rounded up to the next bucket): the loop
// unrolls, each modulus' constants are immediate kernel-parameter operands,
// and channels past s are skipped by a uniform branch.  At the headline
// shape (8192 x 8192, s = 14, each kernel alone) this took A's residue kernel
// from 0.68 to 0.77 of the measured HBM copy peak, and B's from 0.81 to 0.89.
#include <algorithm>

#include "oz2_bits.cuh"
#include "oz2_internal.cuh"

namespace oz2 {
namespace {

// Channel bucket: the compile-time channel count of the kernel instance that
// serves s moduli (s <= bucket; the channels in between are skipped).
inline int channel_bucket(int s) { return s <= 8 ? 8 : (s <= 14 ? 14 : 20); }

// Per element: the magnitude |trunc(2^e x)| = floor(mant 2^sh), sh = E + e.
// General path: rho_m(+-floor(mant 2^sh)) for sh > 0 via (mant mod m)(2^sh mod m).
__device__ int residue_general(uint64_t mant, int sh, uint32_t neg, int t, const ModConsts& mc,
                               const uint8_t* __restrict__ pow2mod) {
  const uint32_t m = static_cast<uint32_t>(mc.m[t]);
  uint32_t r;
  if (m == 256) {
    r = (sh >= 8) ? 0u : static_cast<uint32_t>((mant << sh) & 255u);
  } else {
    // mant mod m with 21-bit limbs (unsigned), then times 2^sh mod m
    const uint32_t a0 = static_cast<uint32_t>(mant & 0x1FFFFF);
    const uint32_t a1 = static_cast<uint32_t>((mant >> 21) & 0x1FFFFF);
    const uint32_t a2 = static_cast<uint32_t>(mant >> 42);
    const uint32_t T = a0 + mc.w21[t][1] * a1 + mc.w21[t][2] * a2;  // < 2^30
    const uint32_t q = __umulhi(T, mc.magic39[t]) >> 7;
    const uint32_t rm = T - q * m;
    const int shc = sh < kPow2Max ? sh : kPow2Max - 1;
    const uint32_t x = rm * pow2mod[t * kPow2Max + shc];  // < 2^16
    r = x - __umulhi(x, mc.magic32[t]) * m;
  }
  if (neg) r = (r == 0) ? 0u : m - r;                   // nonnegative residue of the signed value
  const int h = mc.half[t];
  return static_cast<int>((r + static_cast<uint32_t>(h)) % m) - h;  // centered
}

// Plain per-element path for eight elements of which one or more has a
// scaled magnitude that does not fit the fast path's words (accu mode only);
// kept out of line so the fast path's register allocation does not carry it.
// It reloads its eight elements (src[k stride] for k < nvalid, zero beyond)
// from memory, so the caller's register copy never needs an address.
__device__ __noinline__ void residues8_general(const double* __restrict__ src, int64_t stride, int nvalid,
                                               int scale, const ModConsts& mc,
                                               const uint8_t* __restrict__ pow2mod,
                                               uint16_t* __restrict__ out, int64_t plane_stride) {
  double x[8];
  for (int k = 0; k < 8; ++k) x[k] = (k < nvalid) ? src[k * stride] : 0.0;
  for (int t = 0; t < mc.s; ++t) {
    uint32_t w[4];
    for (int e = 0; e < 8; e += 2) {
      int v[2];
      for (int h2 = 0; h2 < 2; ++h2) {
        const Dec d = decode(x[e + h2]);
        const int sh = d.E + scale;
        const uint32_t m = static_cast<uint32_t>(mc.m[t]);
        const int hh = mc.half[t];
        if (sh <= 0) {
          const uint64_t n = (sh <= -64) ? 0ull : (d.mant >> (-sh));
          uint32_t rm = static_cast<uint32_t>(n % m);
          if (d.neg) rm = (rm == 0) ? 0u : m - rm;
          v[h2] = static_cast<int>((rm + static_cast<uint32_t>(hh)) % m) - hh;
        } else {
          v[h2] = residue_general(d.mant, sh, d.neg, t, mc, pow2mod);
        }
      }
      const __half2 hv = __halves2half2(__int2half_rn(v[0]), __int2half_rn(v[1]));
      w[e >> 1] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    *reinterpret_cast<uint4*>(out + t * plane_stride) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <int NW>
__device__ __forceinline__ bool split_words(double x, int scale, uint32_t (&wd)[3], uint32_t& neg) {
  const Dec d = decode(x);
  neg = d.neg;
  const int sh = d.E + scale;
  wd[0] = wd[1] = wd[2] = 0;
  if (sh > 32 * NW - 53) return false;
  if (sh <= 0) {
    const uint64_t n = (sh <= -64) ? 0ull : (d.mant >> (-sh));
    wd[0] = static_cast<uint32_t>(n);
    wd[1] = static_cast<uint32_t>(n >> 32);
  } else {
    const uint64_t lo = d.mant << sh;  // sh <= 43 < 64
    wd[0] = static_cast<uint32_t>(lo);
    wd[1] = static_cast<uint32_t>(lo >> 32);
    if (NW == 3) wd[2] = static_cast<uint32_t>(d.mant >> (64 - sh));
  }
  return true;
}

// Residues of 8 consecutive K elements of one plane row, for every modulus.
// out points at row `row` of plane 0 (element offset l0 already applied);
// consecutive planes are plane_stride elements apart.
//
// Per element: N = |trunc(2^e x)| = floor(mant 2^sh) as NW 32-bit words
// (NW = 2 covers N < 2^64, NW = 3 N < 2^96).  The words' bytes are base-256
// digits, so for an odd modulus m
//   T = sum_k byte_k (2^(8k) mod m) + floor(m/2)   (two or three dp4a)
// is below 2^20 and congruent to N + floor(m/2); one multiply-high gives
// the exact quotient and r = T mod m = rho_m(N) + floor(m/2).  The fp16
// value rho_m(N) comes from the bit pattern 0x6400 + r and a packed
// subtraction; for x < 0 the result is negated by flipping the fp16 sign
// bit, since rho_m(-N) = -rho_m(N) for odd m.  Channel 0 is m = 256 (the
// greedy set always starts with it): rho_256 is the low byte of +-N read as
// a signed byte.  Elements whose N does not fit NW words (accu mode only)
// take residues8_general.  src / stride / nvalid locate the same eight
// elements in memory for that path.  mc must be a kernel parameter (its
// fields are then immediate operands once the channel loop unrolls).
template <int SB, int NW>
__device__ __forceinline__ void residues8(const double (&x)[8], const double* src, int64_t stride, int nvalid,
                                          int scale, const ModConsts& mc,
                                          const uint8_t* __restrict__ pow2mod,
                                          uint16_t* __restrict__ out, int64_t plane_stride) {
  uint32_t wd[8][3];
  uint32_t neg[8];
  bool fast = true;
#pragma unroll
  for (int e = 0; e < 8; ++e) fast &= split_words<NW>(x[e], scale, wd[e], neg[e]);
  if (fast) {
    uint32_t sgn[4];  // fp16 sign-bit mask of each element pair
#pragma unroll
    for (int e = 0; e < 8; e += 2) sgn[e >> 1] = (neg[e] << 15) | (neg[e + 1] << 31);
    // channel 0: m = 256, the low byte of +-N as a signed byte (+128 bias)
    {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const uint32_t r0 = ((neg[e] ? 0u - wd[e][0] : wd[e][0]) + 128u) & 255u;
        const uint32_t r1 = ((neg[e + 1] ? 0u - wd[e + 1][0] : wd[e + 1][0]) + 128u) & 255u;
        w[e >> 1] = pack_fp16_pair(r0, r1, __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
      }
      *reinterpret_cast<uint4*>(out) = make_uint4(w[0], w[1], w[2], w[3]);
    }
#pragma unroll
    for (int t = 1; t < SB; ++t) {
      if (t >= mc.s) break;  // uniform: the channels of the bucket past s
      const uint32_t m = static_cast<uint32_t>(mc.m[t]);
      const uint32_t magic = mc.magic32[t];
      const uint32_t h = static_cast<uint32_t>(mc.half[t]);
      const uint32_t b2 = mc.bias2[t];
      const __half2 bias2 = *reinterpret_cast<const __half2*>(&b2);
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        uint32_t rr[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint32_t T = __dp4a(wd[e + k][1], mc.wb[t][1], __dp4a(wd[e + k][0], mc.wb[t][0], h));
          if (NW == 3) T = __dp4a(wd[e + k][2], mc.wb[t][2], T);
          rr[k] = T - __umulhi(T, magic) * m;  // = rho_m(N) + floor(m/2), exact for T < 2^24
        }
        w[e >> 1] = pack_fp16_pair(rr[0], rr[1], bias2) ^ sgn[e >> 1];
      }
      *reinterpret_cast<uint4*>(out + t * plane_stride) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    residues8_general(src, stride, nvalid, scale, mc, pow2mod, out, plane_stride);
  }
}

// blocks per SM: 4 with the 64-bit fast path (at most 64 registers), 3 with 96 bits
template <int NW>
struct ResOcc {
  static constexpr int kMinBlocks = NW == 2 ? 4 : 3;
};

// A (column-major p x q) -> planes [s][p][qp]: each warp covers 16 rows x 16
// K elements, so every load instruction reads two full 128-byte lines and
// every row of every plane gets 32 contiguous bytes per warp store.
template <int SB, int NW>
__global__ void __launch_bounds__(256, ResOcc<NW>::kMinBlocks) residue_rows_kernel(
    const double* __restrict__ A, int64_t p, int64_t q, int64_t lda, int64_t qp, int64_t plane_rows,
    const int32_t* __restrict__ alpha, const __grid_constant__ ModConsts mc, const uint8_t* __restrict__ pow2mod,
    uint16_t* __restrict__ planes) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i = blockIdx.x * 32ll + (warp & 1) * 16 + (lane & 15);
  if (i >= p) return;
  const int ai = alpha[i];
  // y walks the 64-wide K blocks (more of them than the grid's y extent when q > 2^22)
  for (int64_t kb = blockIdx.y; kb * 64 < qp; kb += gridDim.y) {
    const int64_t l0 = kb * 64ll + (warp >> 1) * 16 + (lane >> 4) * 8;
    if (l0 >= qp) continue;
    double x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = (l0 + k < q) ? __ldg(A + (l0 + k) * lda + i) : 0.0;
    const int64_t nv = q - l0;
    residues8<SB, NW>(x, A + l0 * lda + i, lda, nv < 8 ? static_cast<int>(nv) : 8, ai, mc, pow2mod,
                      planes + i * qp + l0, plane_rows * qp);
  }
}

// B (column-major q x ncols) -> planes [s][plane_cols][qp] (B, beta and planes
// at the first column of the range): one warp per column, 8 consecutive K
// elements per lane.
template <int SB, int NW>
__global__ void __launch_bounds__(256, ResOcc<NW>::kMinBlocks) residue_cols_kernel(
    const double* __restrict__ B, int64_t q, int64_t ncols, int64_t ldb, int64_t qp, int64_t plane_cols,
    const int32_t* __restrict__ beta, const __grid_constant__ ModConsts mc, const uint8_t* __restrict__ pow2mod,
    uint16_t* __restrict__ planes) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t j = blockIdx.x * 8ll + warp;
  if (j >= ncols) return;
  const int bj = beta[j];
  // y walks the 256-wide K blocks (more of them than the grid's y extent when q > 2^24 - 2^8)
  for (int64_t kb = blockIdx.y; kb * 256 < qp; kb += gridDim.y) {
    const int64_t l0 = kb * 256ll + lane * 8;
    if (l0 >= qp) continue;
    const double* col = B + j * ldb + l0;
    double x[8];
    if (l0 + 8 <= q && (reinterpret_cast<uintptr_t>(col) & 15) == 0) {
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        const double2 v = __ldg(reinterpret_cast<const double2*>(col + k));
        x[k] = v.x;
        x[k + 1] = v.y;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = (l0 + k < q) ? __ldg(col + k) : 0.0;
    }
    const int64_t nv = q - l0;
    residues8<SB, NW>(x, col, 1, nv < 8 ? static_cast<int>(nv) : 8, bj, mc, pow2mod, planes + j * qp + l0,
                      plane_cols * qp);
  }
}

// Fast mode, statistics of B's columns in one read (2048 < q <= 8192): one
// block per column.  The column (contiguous, column-major B) is brought into
// shared memory by one bulk copy of its 16-byte aligned middle; the one
// element before it (a column starting 8 bytes past a 16-byte boundary) and
// the one after it are plain loads.  The maximum and then the sum of squares
// are taken from shared memory, so three columns per SM are in flight while
// others compute.  Writes beta_j; the residue planes follow from
// residue_cols_kernel.  Results are identical to amax_cols + sumsq_cols +
// fast_exp: the reductions are exact integer maxima and sums.  A copy that
// has not landed within kStatsWaitNs sets the timeout bit in *err, and the
// block waits (bounded again) for it before leaving.
__global__ void __launch_bounds__(256, 3) stats_cols_bulk_kernel(const double* __restrict__ B, int64_t q,
                                                                 int64_t ldb, BoundConsts bc,
                                                                 int32_t* __restrict__ beta, int* err) {
  extern __shared__ __align__(16) uint8_t col_smem[];
  __shared__ uint64_t red[8];
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t j = blockIdx.x;
  const double* col = B + j * ldb;
  const int h = static_cast<int>((reinterpret_cast<uintptr_t>(col) >> 3) & 1);  // elements before the aligned middle
  const int64_t nmid = ((q - h) / 2) * 2;                                         // elements in it (even)
  const double* buf = reinterpret_cast<const double*>(col_smem);                // column element h + l at buf[l]
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    if (nmid > 0) {
      mbar_arrive_expect_tx(smem_u32(&bar), static_cast<uint32_t>(nmid * 8));
      bulk_copy_g2s(smem_u32(col_smem), col + h, static_cast<uint32_t>(nmid * 8), smem_u32(&bar));
    } else {
      mbar_arrive(smem_u32(&bar));
    }
  }
  double xe = 0.0;  // the element outside the aligned middle, if any, for threads 0 (head) and 1 (tail)
  if (tid == 0 && h) xe = __ldg(col);
  if (tid == 1 && h + nmid < q) xe = __ldg(col + q - 1);
  const bool got = mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, kStatsWaitNs);
  if (__syncthreads_or(!got)) {
    if (tid == 0) {
      atomicOr(err, kErrTimeout);
      mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, kStatsWaitNs);  // the copy still in flight
    }
    return;
  }
  uint64_t m = static_cast<uint64_t>(__double_as_longlong(xe)) & ~(1ull << 63);
  for (int64_t l = tid; l < nmid; l += 256) {
    const uint64_t b = static_cast<uint64_t>(__double_as_longlong(buf[l])) & ~(1ull << 63);
    m = b > m ? b : m;
  }
  for (int o = 16; o; o >>= 1) {
    const uint64_t y = __shfl_xor_sync(0xffffffffu, m, o);
    m = y > m ? y : m;
  }
  if (lane == 0) red[warp] = m;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < 8; ++w) m = red[w] > m ? red[w] : m;
  __syncthreads();
  const int e = exp_of_bits(m);
  const uint32_t ce = ceil_scaled_small(static_cast<uint64_t>(__double_as_longlong(xe)), kF - e);
  uint64_t sum = static_cast<uint64_t>(ce) * ce;
  for (int64_t l = tid; l < nmid; l += 256) {
    const uint32_t cs = ceil_scaled_small(static_cast<uint64_t>(__double_as_longlong(buf[l])), kF - e);
    sum += static_cast<uint64_t>(cs) * cs;
  }
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) red[warp] = sum;
  __syncthreads();
  if (tid == 0) {
    sum = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += red[w];
    beta[j] = fast_exponent(sum, e, bc);
  }
}

// Fast mode, B side for short columns (q <= 2048) in one read of B:
// statistics, exponent beta_j and residue planes of column j of a range of
// columns (B, beta and planes point at the range's first column; plane rows
// are plane_cols apart).  One block per column; thread t holds the K
// elements [8 t, +8) in registers, so the max, the sum of squares and the
// residues all work on the same registers.  Results are identical to the
// statistics kernels followed by residue_cols_kernel.
template <int SB, int NW>
__global__ void __launch_bounds__(256, 3) fused_cols_fast_kernel(const double* __restrict__ B, int64_t q,
                                                              int64_t ldb, int64_t qp, int64_t plane_cols,
                                                              BoundConsts bc, const __grid_constant__ ModConsts mc,
                                                              const uint8_t* __restrict__ pow2mod,
                                                              int32_t* __restrict__ beta,
                                                              uint16_t* __restrict__ planes) {
  __shared__ uint64_t red[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t j = blockIdx.x;
  const double* col = B + j * ldb;
  const bool vec = (reinterpret_cast<uintptr_t>(col) & 15) == 0;
  const int64_t l0 = tid * 8ll;
  double x[8];
  if (vec && l0 + 8 <= q) {
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      const double2 v = __ldg(reinterpret_cast<const double2*>(col + l0 + k));
      x[k] = v.x;
      x[k + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = (l0 + k < q) ? __ldg(col + l0 + k) : 0.0;
  }
  // max |b| (as the bits of |b|)
  uint64_t m = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint64_t b = static_cast<uint64_t>(__double_as_longlong(x[k])) & ~(1ull << 63);
    m = b > m ? b : m;
  }
  for (int o = 16; o; o >>= 1) {
    const uint64_t y = __shfl_xor_sync(0xffffffffu, m, o);
    m = y > m ? y : m;
  }
  if (lane == 0) red[warp] = m;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < 8; ++w) m = red[w] > m ? red[w] : m;
  __syncthreads();
  // S = sum ceil(|b| 2^(F-e))^2
  const int e = exp_of_bits(m);
  uint64_t sum = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t cs = ceil_scaled_small(static_cast<uint64_t>(__double_as_longlong(x[k])), kF - e);
    sum += static_cast<uint64_t>(cs) * cs;
  }
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) red[warp] = sum;
  __syncthreads();
  sum = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) sum += red[w];
  const int bj = fast_exponent(sum, e, bc);
  if (tid == 0) beta[j] = bj;
  if (l0 < qp) {
    const int64_t nv = q - l0;
    residues8<SB, NW>(x, col + l0, 1, nv < 0 ? 0 : (nv < 8 ? static_cast<int>(nv) : 8), bj, mc, pow2mod,
                      planes + j * qp + l0, plane_cols * qp);
  }
}

// Fast mode, A side for short rows in one read of A: statistics, exponent
// alpha_i and residue planes of R rows per block.  Thread t holds row t % R's
// columns [8 s + 8 S c, +8) for c < NCH (s = t / R, S = 256 / R column slots),
// so q <= 8 S NCH; the per-row max and sum of squares reduce over the lanes
// that share a row and then over the warps, with no atomics and nothing to
// clear.  Results are identical to the per-row-block path (amax_rows,
// sumsq_rows + fast_exp, residue_rows).  R = 4 rows per block: every load
// instruction of a warp reads 32 bytes (one sector) from each of 8 columns.
template <int NCH>
struct FusedRowsOcc {
  static constexpr int kMinBlocks = NCH <= 2 ? 2 : 1;
};
template <int R, int NCH, int SB, int NW>
__global__ void __launch_bounds__(256, FusedRowsOcc<NCH>::kMinBlocks) fused_rows_fast_kernel(const double* __restrict__ A, int64_t rows,
                                                              int64_t q, int64_t lda, int64_t qp,
                                                              int64_t plane_rows, BoundConsts bc,
                                                              const __grid_constant__ ModConsts mc,
                                                              const uint8_t* __restrict__ pow2mod,
                                                              int32_t* __restrict__ alpha,
                                                              uint16_t* __restrict__ planes) {
  constexpr int S = 256 / R;  // column slots per row
  __shared__ uint64_t red[8][R];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r = tid % R, cs = tid / R;
  const int64_t i = blockIdx.x * static_cast<int64_t>(R) + r;
  const bool row_ok = i < rows;
  double x[NCH][8];
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int64_t l0 = 8ll * cs + 8ll * S * c;
#pragma unroll
    for (int k = 0; k < 8; ++k) x[c][k] = (row_ok && l0 + k < q) ? __ldg(A + (l0 + k) * lda + i) : 0.0;
  }
  // max |a| of the row (as the bits of |a|): lanes r, r + R, ... of a warp share row r
  uint64_t m = 0;
#pragma unroll
  for (int c = 0; c < NCH; ++c)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint64_t b = static_cast<uint64_t>(__double_as_longlong(x[c][k])) & ~(1ull << 63);
      m = b > m ? b : m;
    }
#pragma unroll
  for (int o = R; o < 32; o <<= 1) {
    const uint64_t y = __shfl_xor_sync(0xffffffffu, m, o);
    m = y > m ? y : m;
  }
  if (lane < R) red[warp][lane] = m;
  __syncthreads();
  m = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) m = red[w][r] > m ? red[w][r] : m;
  __syncthreads();
  // S_i = sum ceil(|a| 2^(F-e))^2
  const int e = exp_of_bits(m);
  uint64_t sum = 0;
#pragma unroll
  for (int c = 0; c < NCH; ++c)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t cs2 = ceil_scaled_small(static_cast<uint64_t>(__double_as_longlong(x[c][k])), kF - e);
      sum += static_cast<uint64_t>(cs2) * cs2;
    }
#pragma unroll
  for (int o = R; o < 32; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < R) red[warp][lane] = sum;
  __syncthreads();
  sum = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) sum += red[w][r];
  const int ai = fast_exponent(sum, e, bc);
  if (!row_ok) return;
  if (cs == 0) alpha[i] = ai;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int64_t l0 = 8ll * cs + 8ll * S * c;
    if (l0 < qp) {
      const int64_t nv = q - l0;
      residues8<SB, NW>(x[c], A + l0 * lda + i, lda, nv < 0 ? 0 : (nv < 8 ? static_cast<int>(nv) : 8), ai, mc,
                        pow2mod, planes + i * qp + l0, plane_rows * qp);
    }
  }
}

// Instance selection: (channel bucket, words) in {(8, 2), (14, 2), (20, 2),
// (20, 3)}.  Three words are needed only when |trunc(2^e x)| may pass 2^64,
// which the fast bound allows from s = 17 on (L > 2^128); accu mode's larger
// values take the general path.
#define OZ2_RES_DISPATCH(max_bits, s, LAUNCH)       \
  do {                                              \
    if ((max_bits) > 64) {                          \
      LAUNCH(20, 3);                                \
    } else {                                        \
      const int sb_ = channel_bucket(s);            \
      if (sb_ == 8) LAUNCH(8, 2);                   \
      else if (sb_ == 14) LAUNCH(14, 2);            \
      else LAUNCH(20, 2);                           \
    }                                               \
  } while (0)

}  // namespace

// ----------------------------------------------------------------- launchers
cudaError_t launch_residues_rows(const double* A, int64_t rows, int64_t q, int64_t lda, int64_t qp,
                                 int64_t plane_rows, const ModConsts& mc, const int32_t* alpha,
                                 const uint8_t* pow2mod, int max_bits, uint16_t* planes,
                                 cudaStream_t st) {
  const dim3 g(static_cast<unsigned>((rows + 31) / 32), static_cast<unsigned>(std::min<int64_t>(qp / 64, 65535)));
#define OZ2_L(SB, NW) \
  residue_rows_kernel<SB, NW><<<g, 256, 0, st>>>(A, rows, q, lda, qp, plane_rows, alpha, mc, pow2mod, planes)
  OZ2_RES_DISPATCH(max_bits, mc.s, OZ2_L);
#undef OZ2_L
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_residues_cols(const double* B, int64_t q, int64_t ncols, int64_t ldb, int64_t qp,
                                 int64_t plane_cols, const ModConsts& mc, const int32_t* beta,
                                 const uint8_t* pow2mod, int max_bits, uint16_t* planes, cudaStream_t st) {
  const dim3 g(static_cast<unsigned>((ncols + 7) / 8), static_cast<unsigned>(std::min<int64_t>((qp + 255) / 256, 65535)));
#define OZ2_L(SB, NW) \
  residue_cols_kernel<SB, NW><<<g, 256, 0, st>>>(B, q, ncols, ldb, qp, plane_cols, beta, mc, pow2mod, planes)
  OZ2_RES_DISPATCH(max_bits, mc.s, OZ2_L);
#undef OZ2_L
  count_launches(1);
  return cudaGetLastError();
}

bool rows_fused_fast_supported(int64_t q) { return q <= 2048; }

cudaError_t launch_rows_fused_fast(const double* A, int64_t rows, int64_t q, int64_t lda, int64_t qp,
                                   int64_t plane_rows, const BoundConsts& bc, const ModConsts& mc,
                                   const uint8_t* pow2mod, int max_bits, int32_t* alpha, uint16_t* planes,
                                   cudaStream_t st) {
  if (!rows_fused_fast_supported(q) || rows < 1) return cudaErrorInvalidValue;
  // four rows per block, 64 column slots of 8: 1, 2 or 4 register chunks per thread
  const int nch = qp <= 512 ? 1 : (qp <= 1024 ? 2 : 4);
  const dim3 g(static_cast<unsigned>((rows + 3) / 4));
#define OZ2_L(SB, NW)                                                                                          \
  do {                                                                                                         \
    if (nch == 1)                                                                                              \
      fused_rows_fast_kernel<4, 1, SB, NW><<<g, 256, 0, st>>>(A, rows, q, lda, qp, plane_rows, bc, mc, pow2mod, \
                                                              alpha, planes);                                 \
    else if (nch == 2)                                                                                         \
      fused_rows_fast_kernel<4, 2, SB, NW><<<g, 256, 0, st>>>(A, rows, q, lda, qp, plane_rows, bc, mc, pow2mod, \
                                                              alpha, planes);                                 \
    else                                                                                                       \
      fused_rows_fast_kernel<4, 4, SB, NW><<<g, 256, 0, st>>>(A, rows, q, lda, qp, plane_rows, bc, mc, pow2mod, \
                                                              alpha, planes);                                 \
  } while (0)
  OZ2_RES_DISPATCH(max_bits, mc.s, OZ2_L);
#undef OZ2_L
  count_launches(1);
  return cudaGetLastError();
}

bool cols_fused_fast_supported(int64_t q) { return q <= 8192; }

cudaError_t launch_cols_fused_fast(const double* B, int64_t q, int64_t ncols, int64_t ldb, int64_t qp,
                                   int64_t plane_cols, const BoundConsts& bc, const ModConsts& mc,
                                   const uint8_t* pow2mod, int max_bits, int32_t* beta, uint16_t* planes,
                                   int* err, cudaStream_t st) {
  if (!cols_fused_fast_supported(q) || ncols < 1 || ncols > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(ncols));
  if (qp <= 2048) {
    // the whole column in one block's registers: statistics and residues from one read
#define OZ2_L(SB, NW) \
  fused_cols_fast_kernel<SB, NW><<<g, 256, 0, st>>>(B, q, ldb, qp, plane_cols, bc, mc, pow2mod, beta, planes)
    OZ2_RES_DISPATCH(max_bits, mc.s, OZ2_L);
#undef OZ2_L
    count_launches(1);
    return cudaGetLastError();
  }
  // longer columns: the statistics from one read of B, then the residue kernel
  // (a second read of B; faster than one kernel that holds the column through
  // the residues, whose register footprint leaves two blocks per SM)
  const int smem = static_cast<int>(q * 8);  // <= 64 KB: the aligned middle of one column
  // (set on every launch: the attribute belongs to the current device)
  const cudaError_t attr =
      cudaFuncSetAttribute(stats_cols_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 8192 * 8);
  if (attr != cudaSuccess) return attr;
  stats_cols_bulk_kernel<<<g, 256, smem, st>>>(B, q, ldb, bc, beta, err);
  count_launches(1);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_residues_cols(B, q, ncols, ldb, qp, plane_cols, mc, beta, pow2mod, max_bits, planes, st);
}

}  // namespace oz2
