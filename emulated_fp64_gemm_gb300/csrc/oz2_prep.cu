// Preprocessing kernels of the Ozaki-II pipeline: scaling statistics,
// power-of-two exponents, accu-mode bound quantisation and the single-pass
// residue planes.
//
// Method: "Profiling Ozaki II: The Cost Behind Fast INT8 GEMMs" §1 (green
// stage), §2 (fast and accu bounds), §5.1 (row max-abs and sum of squares,
// rounded up), §10.1 (convert each scaled element to an integer once, then
// reduce it with fixed-divisor integer arithmetic per modulus).  Centered
// residues: "Ozaki II supplement: INT8 range conditions and paper performance
// results" §1.2.
//
// No floating-point arithmetic is used on the data: every double is taken
// apart into its sign, exponent and 53-bit significand, and all statistics
// and residues are exact integer computations.  This makes the exponents
// independent of the order of the reductions (the statistics are u64 sums and
// maxima) and removes the FP64 pipe from this stage.
#include <cuda_fp16.h>

#include <algorithm>

#include "oz2_internal.cuh"

namespace oz2 {
namespace {

constexpr int kF = 20;  // fractional bits of the fast-mode statistic

struct Dec {  // |x| = mant * 2^E, mant < 2^53 (0 for x == 0), neg = sign bit
  uint64_t mant;
  int E;
  uint32_t neg;
};

__device__ __forceinline__ Dec decode(double x) {
  const uint64_t b = static_cast<uint64_t>(__double_as_longlong(x));
  Dec d;
  d.neg = static_cast<uint32_t>(b >> 63);
  const int eb = static_cast<int>((b >> 52) & 0x7FF);
  d.mant = b & ((1ull << 52) - 1);
  if (eb == 0) {
    d.E = -1074;
  } else {
    d.mant |= 1ull << 52;
    d.E = eb - 1075;
  }
  return d;
}

// e = floor(log2 a) + 1 for a > 0 given as the bits of |a|; 0 for a == 0.
__device__ __forceinline__ int exp_of_bits(uint64_t abits) {
  if (abits == 0) return 0;
  const int eb = static_cast<int>(abits >> 52);
  if (eb != 0) return eb - 1022;
  const uint64_t m = abits & ((1ull << 52) - 1);
  return (63 - __clzll(static_cast<long long>(m))) - 1073;
}

// ceil(mant * 2^sh) for a result known to be < 2^63.
__device__ __forceinline__ uint64_t ceil_shift(uint64_t mant, int sh) {
  if (mant == 0) return 0;
  if (sh >= 0) return mant << sh;
  const int d = -sh;
  if (d >= 64) return 1;
  const uint64_t q = mant >> d;
  return q + ((mant & ((1ull << d) - 1)) != 0 ? 1 : 0);
}

// ceil(|x| 2^k) for a double x (bits b) whose scaled value is below 2^21,
// with 32-bit operations: |x| = m 2^E, m < 2^53; the top 32 bits of m and a
// sticky bit for the rest suffice because the result needs at most 21 bits.
__device__ __forceinline__ uint32_t ceil_scaled_small(uint64_t b, int k) {
  const uint32_t hi = static_cast<uint32_t>(b >> 32);
  const int eb = static_cast<int>((hi >> 20) & 0x7FF);
  const uint32_t lo = static_cast<uint32_t>(b);
  if (eb == 0) return static_cast<uint32_t>(ceil_shift(b & ((1ull << 52) - 1), -1074 + k));  // subnormal
  // m = 2^52 + frac; top 32 bits: m >> 21, the rest sticky
  const uint32_t m32 = ((hi & 0xFFFFF) | 0x100000u) << 11 | (lo >> 21);
  const bool st = (lo & 0x1FFFFF) != 0;
  // value = m32 2^(E + 21 + k), E = eb - 1075
  const int sh = eb - 1075 + 21 + k;  // <= 0 for results below 2^21
  const int d = -sh;
  if (d >= 32) return 1u;             // nonzero and below 1
  const uint32_t q = m32 >> d;
  const bool rem = st || (d > 0 && (m32 & ((1u << d) - 1u)) != 0);
  return q + (rem ? 1u : 0u);
}

// max { h : S * 2^h <= L } for S > 0, with L given by (Lbits, Lnorm).
__device__ __forceinline__ int max_shift_le_L(uint64_t S, const BoundConsts& bc) {
  const int sb = 64 - __clzll(static_cast<long long>(S));
  const uint64_t Snorm = S << (64 - sb);
  const int k = bc.Lbits - sb;
  return (Snorm <= bc.Lnorm) ? k : k - 1;
}

// ------------------------------------------------------------- statistics
// Row max |a| of A (column-major p x q): threads along rows, columns split over blockIdx.y.
__global__ void amax_rows_kernel(const double* __restrict__ A, int64_t p, int64_t q, int64_t lda,
                                 int64_t cols_per_block, uint64_t* __restrict__ amax) {
  const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (i >= p) return;
  const int64_t l0 = blockIdx.y * cols_per_block;
  const int64_t l1 = min(q, l0 + cols_per_block);
  uint64_t m = 0;
  int64_t l = l0;
  for (; l + 8 <= l1; l += 8) {  // eight loads in flight per thread
    uint64_t b[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) b[k] = static_cast<uint64_t>(__double_as_longlong(__ldg(A + (l + k) * lda + i)));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint64_t v = b[k] & ~(1ull << 63);
      m = v > m ? v : m;
    }
  }
  for (; l < l1; ++l) {
    const uint64_t b = static_cast<uint64_t>(__double_as_longlong(A[l * lda + i])) & ~(1ull << 63);
    m = b > m ? b : m;
  }
  if (m) atomicMax(reinterpret_cast<unsigned long long*>(amax + i), static_cast<unsigned long long>(m));
}

// Column max |b| of B (column-major q x r): one warp per (column, segment).
__global__ void amax_cols_kernel(const double* __restrict__ B, int64_t q, int64_t r, int64_t ldb,
                                 int64_t seg, uint64_t* __restrict__ amax) {
  const int lane = threadIdx.x & 31;
  const int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
  if (j >= r) return;
  const int64_t l0 = blockIdx.y * seg;
  const int64_t l1 = min(q, l0 + seg);
  uint64_t m = 0;
  int64_t l = l0 + lane;
  for (; l + 7 * 32 < l1; l += 8 * 32) {  // eight loads in flight per lane
    uint64_t b[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) b[k] = static_cast<uint64_t>(__double_as_longlong(__ldg(B + j * ldb + l + k * 32)));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint64_t v = b[k] & ~(1ull << 63);
      m = v > m ? v : m;
    }
  }
  for (; l < l1; l += 32) {
    const uint64_t b = static_cast<uint64_t>(__double_as_longlong(B[j * ldb + l])) & ~(1ull << 63);
    m = b > m ? b : m;
  }
  for (int o = 16; o; o >>= 1) {
    const uint64_t x = __shfl_xor_sync(0xffffffffu, m, o);
    m = x > m ? x : m;
  }
  if (lane == 0 && m) atomicMax(reinterpret_cast<unsigned long long*>(amax + j), static_cast<unsigned long long>(m));
}

// S = sum ceil(|a| 2^(F-e))^2 per row of A.
__global__ void sumsq_rows_kernel(const double* __restrict__ A, int64_t p, int64_t q, int64_t lda,
                                  int64_t cols_per_block, const uint64_t* __restrict__ amax,
                                  uint64_t* __restrict__ sum) {
  const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (i >= p) return;
  const int e = exp_of_bits(amax[i]);
  const int64_t l0 = blockIdx.y * cols_per_block;
  const int64_t l1 = min(q, l0 + cols_per_block);
  uint64_t s = 0;
  int64_t l = l0;
  for (; l + 8 <= l1; l += 8) {
    uint64_t b[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) b[k] = static_cast<uint64_t>(__double_as_longlong(__ldg(A + (l + k) * lda + i)));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t c = ceil_scaled_small(b[k], kF - e);
      s += static_cast<uint64_t>(c) * c;
    }
  }
  for (; l < l1; ++l) {
    const uint32_t c = ceil_scaled_small(static_cast<uint64_t>(__double_as_longlong(A[l * lda + i])), kF - e);
    s += static_cast<uint64_t>(c) * c;
  }
  if (s) atomicAdd(reinterpret_cast<unsigned long long*>(sum + i), static_cast<unsigned long long>(s));
}

__global__ void sumsq_cols_kernel(const double* __restrict__ B, int64_t q, int64_t r, int64_t ldb,
                                  int64_t seg, const uint64_t* __restrict__ amax,
                                  uint64_t* __restrict__ sum) {
  const int lane = threadIdx.x & 31;
  const int64_t j = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
  if (j >= r) return;
  const int e = exp_of_bits(amax[j]);
  const int64_t l0 = blockIdx.y * seg;
  const int64_t l1 = min(q, l0 + seg);
  uint64_t s = 0;
  int64_t l = l0 + lane;
  for (; l + 7 * 32 < l1; l += 8 * 32) {
    uint64_t b[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) b[k] = static_cast<uint64_t>(__double_as_longlong(__ldg(B + j * ldb + l + k * 32)));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t c = ceil_scaled_small(b[k], kF - e);
      s += static_cast<uint64_t>(c) * c;
    }
  }
  for (; l < l1; l += 32) {
    const uint32_t c = ceil_scaled_small(static_cast<uint64_t>(__double_as_longlong(B[j * ldb + l])), kF - e);
    s += static_cast<uint64_t>(c) * c;
  }
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0 && s) atomicAdd(reinterpret_cast<unsigned long long*>(sum + j), static_cast<unsigned long long>(s));
}

// fast exponent: U = S 4^(e-F); exp = max { a : 4^a U <= L } = floor(h/2) - e + F,
// h = max { h : S 2^h <= L }; 0 for a zero vector.
__global__ void fast_exp_kernel(const uint64_t* __restrict__ amax, const uint64_t* __restrict__ sum,
                                int64_t n, BoundConsts bc, int32_t* __restrict__ out) {
  const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (i >= n) return;
  const uint64_t S = sum[i];
  if (S == 0) {
    out[i] = 0;
    return;
  }
  const int e = exp_of_bits(amax[i]);
  const int h = max_shift_le_L(S, bc);
  out[i] = (h >> 1) - e + kF;  // arithmetic shift: floor(h/2)
}

// ------------------------------------------------------------- accu bound
// u = max { u : ceil(amax 2^u) <= 127 } (0 for a zero vector).
__device__ __forceinline__ int quant_exp(uint64_t abits) {
  if (abits == 0) return 0;
  const int e = exp_of_bits(abits);
  uint64_t m = abits & ((1ull << 52) - 1);
  if ((abits >> 52) != 0) {
    m |= 1ull << 52;
  } else {
    m <<= (53 - (64 - __clzll(static_cast<long long>(m))));  // normalise to 53 bits
  }
  // amax * 2^(7-e) = m / 2^46 lies in [64, 128): it is <= 127 iff m <= 127 * 2^46.
  return (m <= (127ull << 46)) ? 7 - e : 6 - e;
}

// Abar[i][l] = ceil(|a_il| 2^u_i) as fp16, K-major rows of length qp (zero padded).
// Thread layout as in the residue kernel for A: 16 rows x 2 eight-element K groups per warp.
__global__ void bound_quant_rows_kernel(const double* __restrict__ A, int64_t p, int64_t q,
                                        int64_t lda, int64_t qp, const uint64_t* __restrict__ amax,
                                        int32_t* __restrict__ u_out, uint16_t* __restrict__ Abar) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i = blockIdx.x * 32ll + (warp & 1) * 16 + (lane & 15);
  const int64_t l0 = blockIdx.y * 64ll + (warp >> 1) * 16 + (lane >> 4) * 8;
  if (i >= p || l0 >= qp) return;
  const int u = quant_exp(amax[i]);
  if (l0 == 0) u_out[i] = u;
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
    uint32_t c[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t l = l0 + k + h;
      c[h] = 0;
      if (l < q) {
        const Dec d = decode(A[l * lda + i]);
        c[h] = static_cast<uint32_t>(ceil_shift(d.mant, d.E + u));
      }
    }
    // fp16 of an integer c < 1024: bits 0x6400 + c encode 1024 + c; subtract 1024.
    const uint32_t word = (c[1] << 16 | c[0]) + 0x64006400u;
    __half2 hv = *reinterpret_cast<const __half2*>(&word);
    hv = __hsub2(hv, __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
    w[k >> 1] = *reinterpret_cast<uint32_t*>(&hv);
  }
  *reinterpret_cast<uint4*>(Abar + i * qp + l0) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Bbar[j][l] = ceil(|b_lj| 2^v_j): one warp per column, 8 elements per lane.
__global__ void bound_quant_cols_kernel(const double* __restrict__ B, int64_t q, int64_t r,
                                        int64_t ldb, int64_t qp, const uint64_t* __restrict__ amax,
                                        int32_t* __restrict__ v_out, uint16_t* __restrict__ Bbar) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t j = blockIdx.x * 8ll + warp;
  const int64_t l0 = blockIdx.y * 256ll + lane * 8;
  if (j >= r || l0 >= qp) return;
  const int v = quant_exp(amax[j]);
  if (l0 == 0) v_out[j] = v;
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
    uint32_t c[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t l = l0 + k + h;
      c[h] = 0;
      if (l < q) {
        const Dec d = decode(B[j * ldb + l]);
        c[h] = static_cast<uint32_t>(ceil_shift(d.mant, d.E + v));
      }
    }
    const uint32_t word = (c[1] << 16 | c[0]) + 0x64006400u;
    __half2 hv = *reinterpret_cast<const __half2*>(&word);
    hv = __hsub2(hv, __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
    w[k >> 1] = *reinterpret_cast<uint32_t*>(&hv);
  }
  *reinterpret_cast<uint4*>(Bbar + j * qp + l0) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Accu mode, B side in one read of B (q <= 8192): one block per column; thread
// t holds the column's elements [2048 c + 8 t, +8) in registers, so the column
// maximum, v_j and the quantised row of Bbar (fp16, zero padded to qp) all come
// from one read.  Results are identical to amax_cols + bound_quant_cols (an
// exact integer maximum; the elements past q are zeros, which quantise to 0).
template <int NCH>
__global__ void __launch_bounds__(256, 2) fused_cols_bound_kernel(const double* __restrict__ B, int64_t q,
                                                               int64_t ldb, int64_t qp,
                                                               uint64_t* __restrict__ amax,
                                                               int32_t* __restrict__ v_out,
                                                               uint16_t* __restrict__ Bbar) {
  __shared__ uint64_t red[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t j = blockIdx.x;
  const double* col = B + j * ldb;
  const bool vec = (reinterpret_cast<uintptr_t>(col) & 15) == 0;
  double x[NCH][8];
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int64_t l0 = c * 2048ll + tid * 8ll;
    if (vec && l0 + 8 <= q) {
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        const double2 w = __ldg(reinterpret_cast<const double2*>(col + l0 + k));
        x[c][k] = w.x;
        x[c][k + 1] = w.y;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) x[c][k] = (l0 + k < q) ? __ldg(col + l0 + k) : 0.0;
    }
  }
  uint64_t m = 0;
#pragma unroll
  for (int c = 0; c < NCH; ++c)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint64_t b = static_cast<uint64_t>(__double_as_longlong(x[c][k])) & ~(1ull << 63);
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
  const int v = quant_exp(m);
  if (tid == 0) {
    amax[j] = m;
    v_out[j] = v;
  }
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int64_t l0 = c * 2048ll + tid * 8ll;
    if (l0 < qp) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        uint32_t cq[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const Dec d = decode(x[c][k + h]);
          cq[h] = static_cast<uint32_t>(ceil_shift(d.mant, d.E + v));
        }
        // fp16 of an integer below 1024: bits 0x6400 + c encode 1024 + c; subtract 1024
        const uint32_t word = (cq[1] << 16 | cq[0]) + 0x64006400u;
        __half2 hv = *reinterpret_cast<const __half2*>(&word);
        hv = __hsub2(hv, __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
        w[k >> 1] = *reinterpret_cast<uint32_t*>(&hv);
      }
      *reinterpret_cast<uint4*>(Bbar + j * qp + l0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// accu exponents from the max keys of the bound GEMM.  A key encodes the
// dyadic value w 2^-x (w < 2^31) as ((floor(log2) + 4096) << 32) | mantissa
// normalised to 32 bits; 0 encodes zero.  The row value is
// max_j Wbar_ij 2^-v_j, so U_i = value 2^-u_i; likewise for columns.
__global__ void accu_exp_kernel(const uint64_t* __restrict__ key, const int32_t* __restrict__ qexp,
                                int64_t n, BoundConsts bc, int32_t* __restrict__ out) {
  const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (i >= n) return;
  const uint64_t k = key[i];
  if (k == 0) {
    out[i] = 0;
    return;
  }
  const int E = static_cast<int>(k >> 32) - 4096;        // value = mant32 * 2^(E - 31)
  const uint64_t mant = k & 0xffffffffull;
  const int h = max_shift_le_L(mant, bc);                // mant 2^h <= L
  // 4^a mant 2^(E - 31 - u) <= L  <=>  2a + E - 31 - u <= h
  const int num = h - E + 31 + qexp[i];
  out[i] = num >> 1;                                     // floor
}

// ------------------------------------------------------------- residues
// Per element: the magnitude |trunc(2^e x)| = floor(mant 2^sh), sh = E + e, as
// NL limbs of LB bits, each negated when x < 0.  Then, per modulus,
//   T = l0 + sum_k w_k l_k + (K_m + floor(m/2)),  w_k = 2^(LB k) mod m,
// K_m a multiple of m with K_m >= 2^30, so T is in [0, 2^31) and
// T mod m = (trunc(2^e x) + floor(m/2)) mod m = rho_m(trunc(2^e x)) + floor(m/2).
// The quotient comes from one multiply-high (magic39); the value goes to fp16
// through the bit pattern 0x6400 + v (= 1024 + v) and a packed subtraction.
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


// fp16 bits of two values v0, v1 in [0, 2048) shifted by -bias, packed (v0 low).
__device__ __forceinline__ uint32_t pack_fp16_pair(uint32_t v0, uint32_t v1, __half2 bias2) {
  const uint32_t word = (v1 << 16 | v0) + 0x64006400u;  // fp16(1024 + v)
  __half2 hv = *reinterpret_cast<const __half2*>(&word);
  hv = __hsub2(hv, bias2);                              // exact: integers below 2048
  return *reinterpret_cast<uint32_t*>(&hv);
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
// take residue_general.
// Plain per-element path for rows that contain an element whose scaled
// magnitude does not fit NW words (accu mode only); kept out of line so the
// fast path's register allocation does not carry it.  It reloads its eight
// elements (src[k stride] for k < nvalid, zero beyond) from memory, so the
// caller's register copy never needs an address.
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

// src / stride / nvalid locate the same eight elements in memory for the
// general path.
template <int NW>
__device__ __forceinline__ void residues8(const double (&x)[8], const double* src, int64_t stride, int nvalid,
                                          int scale, const ModConsts& mc,
                                          const uint8_t* __restrict__ pow2mod,
                                          uint16_t* __restrict__ out, int64_t plane_stride) {
  uint32_t wd[8][3];
  uint32_t neg[8];
  bool fast = true;
#pragma unroll
  for (int e = 0; e < 8; ++e) fast &= split_words<NW>(x[e], scale, wd[e], neg[e]);
  const int s = mc.s;
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
    for (int t = 1; t < s; ++t) {
      const uint32_t m = static_cast<uint32_t>(mc.m[t]);
      const uint32_t magic = mc.magic32[t];
      const uint32_t h = static_cast<uint32_t>(mc.half[t]);
      const uint32_t wb0 = mc.wb[t][0], wb1 = mc.wb[t][1], wb2 = mc.wb[t][2];
      const uint32_t b2 = mc.bias2[t];
      const __half2 bias2 = *reinterpret_cast<const __half2*>(&b2);
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        uint32_t rr[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint32_t T = __dp4a(wd[e + k][1], wb1, __dp4a(wd[e + k][0], wb0, h));
          if (NW == 3) T = __dp4a(wd[e + k][2], wb2, T);
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

// A (column-major p x q) -> planes [s][p][qp]: each warp covers 16 rows x 16
// K elements, so every load instruction reads two full 128-byte lines and
// every row of every plane gets 32 contiguous bytes per warp store.
template <int NW>
__global__ void __launch_bounds__(256, 3) residue_rows_kernel(const double* __restrict__ A, int64_t p,
                                                           int64_t q, int64_t lda, int64_t qp,
                                                           int64_t plane_rows,
                                                           const int32_t* __restrict__ alpha,
                                                           ModConsts mc,
                                                           const uint8_t* __restrict__ pow2mod,
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
    residues8<NW>(x, A + l0 * lda + i, lda, nv < 8 ? static_cast<int>(nv) : 8, ai, mc, pow2mod,
                  planes + i * qp + l0, plane_rows * qp);
  }
}

// B (column-major q x r) -> planes [s][r][qp]: one warp per column, 8
// consecutive K elements per lane.
template <int NW>
__global__ void __launch_bounds__(256, 3) residue_cols_kernel(const double* __restrict__ B, int64_t q,
                                                           int64_t r, int64_t ldb, int64_t qp,
                                                           const int32_t* __restrict__ beta,
                                                           ModConsts mc,
                                                           const uint8_t* __restrict__ pow2mod,
                                                           uint16_t* __restrict__ planes) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t j = blockIdx.x * 8ll + warp;
  if (j >= r) return;
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
    residues8<NW>(x, col, 1, nv < 8 ? static_cast<int>(nv) : 8, bj, mc, pow2mod, planes + j * qp + l0,
                  r * qp);
  }
}

// Fast mode, B side in one read of B: statistics, exponent beta_j and residue
// planes of column j of a range of `ncols` columns (B, beta and planes point at
// the range's first column; plane rows are plane_cols apart).  One block per column; thread t holds the K elements
// [2048 c + 8 t, +8) for c < NCH in registers (q <= 2048 NCH), so the max, the
// sum of squares and the residues all work on the same registers and B is
// read from memory once.  Results are identical to the three-kernel path
// (amax_cols, sumsq_cols + fast_exp, residue_cols): the reductions are exact
// integer maxima and sums, independent of their order.
template <int NCH, int NW>
__global__ void __launch_bounds__(256, 2) fused_cols_fast_kernel(const double* __restrict__ B, int64_t q,
                                                              int64_t ldb, int64_t qp, int64_t plane_cols,
                                                              BoundConsts bc, ModConsts mc,
                                                              const uint8_t* __restrict__ pow2mod,
                                                              int32_t* __restrict__ beta,
                                                              uint16_t* __restrict__ planes) {
  __shared__ uint64_t red[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t j = blockIdx.x;
  const double* col = B + j * ldb;
  const bool vec = (reinterpret_cast<uintptr_t>(col) & 15) == 0;
  double x[NCH][8];
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int64_t l0 = c * 2048ll + tid * 8ll;
    if (vec && l0 + 8 <= q) {
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        const double2 v = __ldg(reinterpret_cast<const double2*>(col + l0 + k));
        x[c][k] = v.x;
        x[c][k + 1] = v.y;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) x[c][k] = (l0 + k < q) ? __ldg(col + l0 + k) : 0.0;
    }
  }
  // max |b| (as the bits of |b|)
  uint64_t m = 0;
#pragma unroll
  for (int c = 0; c < NCH; ++c)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint64_t b = static_cast<uint64_t>(__double_as_longlong(x[c][k])) & ~(1ull << 63);
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
  for (int c = 0; c < NCH; ++c)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t cs = ceil_scaled_small(static_cast<uint64_t>(__double_as_longlong(x[c][k])), kF - e);
      sum += static_cast<uint64_t>(cs) * cs;
    }
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) red[warp] = sum;
  __syncthreads();
  sum = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) sum += red[w];
  const int bj = (sum == 0) ? 0 : (max_shift_le_L(sum, bc) >> 1) - e + kF;
  if (tid == 0) beta[j] = bj;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int64_t l0 = c * 2048ll + tid * 8ll;
    if (l0 < qp) {
      const int64_t nv = q - l0;
      residues8<NW>(x[c], col + l0, 1, nv < 0 ? 0 : (nv < 8 ? static_cast<int>(nv) : 8), bj, mc, pow2mod,
                    planes + j * qp + l0, plane_cols * qp);
    }
  }
}

// Fast mode, A side for short rows in one read of A: statistics, exponent
// alpha_i and residue planes of R rows per block.  Thread t holds row t % R's
// columns [8 s + 8 S c, +8) for c < 4 (s = t / R, S = 256 / R column slots), so
// q <= 8192 / R; the per-row max and sum of squares reduce over the lanes that
// share a row and then over the warps, with no atomics and nothing to clear.
// Results are identical to the per-row-block path (amax_rows, sumsq_rows +
// fast_exp, residue_rows).
template <int R, int NW>
__global__ void __launch_bounds__(256, 1) fused_rows_fast_kernel(const double* __restrict__ A, int64_t rows,
                                                              int64_t q, int64_t lda, int64_t qp,
                                                              int64_t plane_rows, BoundConsts bc, ModConsts mc,
                                                              const uint8_t* __restrict__ pow2mod,
                                                              int32_t* __restrict__ alpha,
                                                              uint16_t* __restrict__ planes) {
  constexpr int S = 256 / R;  // column slots per row
  constexpr int NCH = 4;      // 8-column chunks per thread
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
  const int ai = (sum == 0) ? 0 : (max_shift_le_L(sum, bc) >> 1) - e + kF;
  if (!row_ok) return;
  if (cs == 0) alpha[i] = ai;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int64_t l0 = 8ll * cs + 8ll * S * c;
    if (l0 < qp) {
      const int64_t nv = q - l0;
      residues8<NW>(x[c], A + l0 * lda + i, lda, nv < 0 ? 0 : (nv < 8 ? static_cast<int>(nv) : 8), ai, mc,
                    pow2mod, planes + i * qp + l0, plane_rows * qp);
    }
  }
}

__global__ void planes_to_int8_kernel(const uint16_t* __restrict__ planes, int64_t rows, int64_t q,
                                      int64_t qp, int s, int8_t* __restrict__ out) {
  const int64_t n = static_cast<int64_t>(s) * rows * q;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t l = idx % q;
    const int64_t rt = idx / q;  // t * rows + row
    const uint16_t b = planes[rt * qp + l];
    out[idx] = static_cast<int8_t>(__half2int_rn(__ushort_as_half(b)));
  }
}

// One block waits on an mbarrier that nothing completes; the bounded wait
// must give up, flag the error word and let the kernel exit.
__global__ void wait_timeout_selftest_kernel(int* err, long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, static_cast<uint64_t>(limit_ns)))
      atomicOr(err, kErrTimeout);
  }
  __syncthreads();
}

int cols_split(int64_t q, int64_t blocks_other, int num_sms) {
  // enough blocks for ~16 waves, but at least 64 elements per thread (on an
  // 8192 x 8192 A the row maximum took 0.150 ms with 4 waves, 0.130 with 16:
  // more, shorter column ranges in flight)
  int64_t want = (16ll * num_sms + blocks_other - 1) / blocks_other;
  int64_t maxs = (q + 63) / 64;
  if (want > maxs) want = maxs;
  if (want < 1) want = 1;
  if (want > 65535) want = 65535;
  return static_cast<int>(want);
}

int device_sms() {
  int dev = 0, n = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

}  // namespace

// ----------------------------------------------------------------- launchers
cudaError_t launch_fast_exponents_rows(const ScaleArgs& a, const BoundConsts& bc, uint64_t* amaxA,
                                       uint64_t* sumA, int32_t* alpha, cudaStream_t st) {
  const int sms = device_sms();
  cudaMemsetAsync(amaxA, 0, a.p * sizeof(uint64_t), st);
  cudaMemsetAsync(sumA, 0, a.p * sizeof(uint64_t), st);
  const int64_t rb = (a.p + 255) / 256;
  const int splitA = cols_split(a.q, rb, sms);
  const int64_t cpbA = (a.q + splitA - 1) / splitA;
  amax_rows_kernel<<<dim3(static_cast<unsigned>(rb), splitA), 256, 0, st>>>(a.A, a.p, a.q, a.lda, cpbA, amaxA);
  sumsq_rows_kernel<<<dim3(static_cast<unsigned>(rb), splitA), 256, 0, st>>>(a.A, a.p, a.q, a.lda, cpbA, amaxA, sumA);
  fast_exp_kernel<<<static_cast<unsigned>((a.p + 255) / 256), 256, 0, st>>>(amaxA, sumA, a.p, bc, alpha);
  count_launches(3);
  return cudaGetLastError();
}

cudaError_t launch_fast_exponents_cols(const ScaleArgs& a, const BoundConsts& bc, uint64_t* amaxB,
                                       uint64_t* sumB, int32_t* beta, cudaStream_t st) {
  const int sms = device_sms();
  cudaMemsetAsync(amaxB, 0, a.r * sizeof(uint64_t), st);
  cudaMemsetAsync(sumB, 0, a.r * sizeof(uint64_t), st);
  const int64_t cb = (a.r + 7) / 8;
  const int splitB = cols_split(a.q, cb, sms);
  const int64_t segB = (a.q + splitB - 1) / splitB;
  amax_cols_kernel<<<dim3(static_cast<unsigned>(cb), splitB), 256, 0, st>>>(a.B, a.q, a.r, a.ldb, segB, amaxB);
  sumsq_cols_kernel<<<dim3(static_cast<unsigned>(cb), splitB), 256, 0, st>>>(a.B, a.q, a.r, a.ldb, segB, amaxB, sumB);
  fast_exp_kernel<<<static_cast<unsigned>((a.r + 255) / 256), 256, 0, st>>>(amaxB, sumB, a.r, bc, beta);
  count_launches(3);
  return cudaGetLastError();
}

cudaError_t launch_fast_exponents(const ScaleArgs& a, const BoundConsts& bc, uint64_t* amaxA,
                                  uint64_t* amaxB, uint64_t* sumA, uint64_t* sumB, int32_t* alpha,
                                  int32_t* beta, cudaStream_t st) {
  cudaError_t e = launch_fast_exponents_rows(a, bc, amaxA, sumA, alpha, st);
  if (e != cudaSuccess) return e;
  return launch_fast_exponents_cols(a, bc, amaxB, sumB, beta, st);
}

cudaError_t launch_bound_quant(const ScaleArgs& a, int64_t qp, uint64_t* amaxA, uint64_t* amaxB,
                               int32_t* u, int32_t* v, uint16_t* Abar, uint16_t* Bbar,
                               cudaStream_t st) {
  const int sms = device_sms();
  cudaMemsetAsync(amaxA, 0, a.p * sizeof(uint64_t), st);
  cudaMemsetAsync(amaxB, 0, a.r * sizeof(uint64_t), st);
  const int64_t rb = (a.p + 255) / 256;
  const int splitA = cols_split(a.q, rb, sms);
  const int64_t cpbA = (a.q + splitA - 1) / splitA;
  const int64_t cb = (a.r + 7) / 8;
  const int splitB = cols_split(a.q, cb, sms);
  const int64_t segB = (a.q + splitB - 1) / splitB;
  amax_rows_kernel<<<dim3(static_cast<unsigned>(rb), splitA), 256, 0, st>>>(a.A, a.p, a.q, a.lda, cpbA, amaxA);
  // B: one read (column in registers) up to q = 8192, else maximum then quantisation
  const bool fused_b = cols_fused_fast_supported(a.q) && a.r <= 0x7FFFFFFF;
  if (fused_b) {
    const dim3 g(static_cast<unsigned>(a.r));
    const int nch = static_cast<int>((qp + 2047) / 2048);
    if (nch <= 1) fused_cols_bound_kernel<1><<<g, 256, 0, st>>>(a.B, a.q, a.ldb, qp, amaxB, v, Bbar);
    else if (nch <= 2) fused_cols_bound_kernel<2><<<g, 256, 0, st>>>(a.B, a.q, a.ldb, qp, amaxB, v, Bbar);
    else fused_cols_bound_kernel<4><<<g, 256, 0, st>>>(a.B, a.q, a.ldb, qp, amaxB, v, Bbar);
  } else {
    amax_cols_kernel<<<dim3(static_cast<unsigned>(cb), splitB), 256, 0, st>>>(a.B, a.q, a.r, a.ldb, segB, amaxB);
  }
  bound_quant_rows_kernel<<<dim3(static_cast<unsigned>((a.p + 31) / 32), static_cast<unsigned>(qp / 64)), 256, 0, st>>>(
      a.A, a.p, a.q, a.lda, qp, amaxA, u, Abar);
  if (!fused_b)
    bound_quant_cols_kernel<<<dim3(static_cast<unsigned>((a.r + 7) / 8), static_cast<unsigned>((qp + 255) / 256)), 256, 0, st>>>(
        a.B, a.q, a.r, a.ldb, qp, amaxB, v, Bbar);
  count_launches(fused_b ? 3 : 4);
  return cudaGetLastError();
}

cudaError_t launch_accu_exponents(int64_t p, int64_t r, const BoundConsts& bc,
                                  const uint64_t* rowkey, const uint64_t* colkey, const int32_t* u,
                                  const int32_t* v, int32_t* alpha, int32_t* beta, cudaStream_t st) {
  accu_exp_kernel<<<static_cast<unsigned>((p + 255) / 256), 256, 0, st>>>(rowkey, u, p, bc, alpha);
  accu_exp_kernel<<<static_cast<unsigned>((r + 255) / 256), 256, 0, st>>>(colkey, v, r, bc, beta);
  count_launches(2);
  return cudaGetLastError();
}

cudaError_t launch_residues_rows(const double* A, int64_t rows, int64_t q, int64_t lda, int64_t qp,
                                 int64_t plane_rows, const ModConsts& mc, const int32_t* alpha,
                                 const uint8_t* pow2mod, int max_bits, uint16_t* planes,
                                 cudaStream_t st) {
  const dim3 g(static_cast<unsigned>((rows + 31) / 32), static_cast<unsigned>(std::min<int64_t>(qp / 64, 65535)));
  if (max_bits <= 64)
    residue_rows_kernel<2><<<g, 256, 0, st>>>(A, rows, q, lda, qp, plane_rows, alpha, mc, pow2mod, planes);
  else
    residue_rows_kernel<3><<<g, 256, 0, st>>>(A, rows, q, lda, qp, plane_rows, alpha, mc, pow2mod, planes);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_residues_cols(const double* B, int64_t q, int64_t r, int64_t ldb, int64_t qp,
                                 const ModConsts& mc, const int32_t* beta, const uint8_t* pow2mod,
                                 int max_bits, uint16_t* planes, cudaStream_t st) {
  const dim3 g(static_cast<unsigned>((r + 7) / 8), static_cast<unsigned>(std::min<int64_t>((qp + 255) / 256, 65535)));
  if (max_bits <= 64)
    residue_cols_kernel<2><<<g, 256, 0, st>>>(B, q, r, ldb, qp, beta, mc, pow2mod, planes);
  else
    residue_cols_kernel<3><<<g, 256, 0, st>>>(B, q, r, ldb, qp, beta, mc, pow2mod, planes);
  count_launches(1);
  return cudaGetLastError();
}

bool rows_fused_fast_supported(int64_t q) { return q <= 2048; }

cudaError_t launch_rows_fused_fast(const double* A, int64_t rows, int64_t q, int64_t lda, int64_t qp,
                                   int64_t plane_rows, const BoundConsts& bc, const ModConsts& mc,
                                   const uint8_t* pow2mod, int max_bits, int32_t* alpha, uint16_t* planes,
                                   cudaStream_t st) {
  if (!rows_fused_fast_supported(q) || rows < 1) return cudaErrorInvalidValue;
  const int R = (qp <= 1024) ? 8 : 4;
  const dim3 g(static_cast<unsigned>((rows + R - 1) / R));
  if (max_bits <= 64) {
    if (R == 8) fused_rows_fast_kernel<8, 2><<<g, 256, 0, st>>>(A, rows, q, lda, qp, plane_rows, bc, mc, pow2mod, alpha, planes);
    else fused_rows_fast_kernel<4, 2><<<g, 256, 0, st>>>(A, rows, q, lda, qp, plane_rows, bc, mc, pow2mod, alpha, planes);
  } else {
    if (R == 8) fused_rows_fast_kernel<8, 3><<<g, 256, 0, st>>>(A, rows, q, lda, qp, plane_rows, bc, mc, pow2mod, alpha, planes);
    else fused_rows_fast_kernel<4, 3><<<g, 256, 0, st>>>(A, rows, q, lda, qp, plane_rows, bc, mc, pow2mod, alpha, planes);
  }
  count_launches(1);
  return cudaGetLastError();
}

bool cols_fused_fast_supported(int64_t q) { return q <= 8192; }

cudaError_t launch_cols_fused_fast(const double* B, int64_t q, int64_t ncols, int64_t ldb, int64_t qp,
                                   int64_t plane_cols, const BoundConsts& bc, const ModConsts& mc,
                                   const uint8_t* pow2mod, int max_bits, int32_t* beta, uint16_t* planes,
                                   cudaStream_t st) {
  if (!cols_fused_fast_supported(q) || ncols < 1 || ncols > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(ncols));
  const int nch = static_cast<int>((qp + 2047) / 2048);
  if (max_bits <= 64) {
    if (nch <= 1) fused_cols_fast_kernel<1, 2><<<g, 256, 0, st>>>(B, q, ldb, qp, plane_cols, bc, mc, pow2mod, beta, planes);
    else if (nch <= 2) fused_cols_fast_kernel<2, 2><<<g, 256, 0, st>>>(B, q, ldb, qp, plane_cols, bc, mc, pow2mod, beta, planes);
    else fused_cols_fast_kernel<4, 2><<<g, 256, 0, st>>>(B, q, ldb, qp, plane_cols, bc, mc, pow2mod, beta, planes);
  } else {
    if (nch <= 1) fused_cols_fast_kernel<1, 3><<<g, 256, 0, st>>>(B, q, ldb, qp, plane_cols, bc, mc, pow2mod, beta, planes);
    else if (nch <= 2) fused_cols_fast_kernel<2, 3><<<g, 256, 0, st>>>(B, q, ldb, qp, plane_cols, bc, mc, pow2mod, beta, planes);
    else fused_cols_fast_kernel<4, 3><<<g, 256, 0, st>>>(B, q, ldb, qp, plane_cols, bc, mc, pow2mod, beta, planes);
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_planes_to_int8(const uint16_t* planes, int64_t rows, int64_t q, int64_t qp,
                                  int s, int8_t* out, cudaStream_t st) {
  planes_to_int8_kernel<<<1024, 256, 0, st>>>(planes, rows, q, qp, s, out);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(int* err, long long limit_ns, cudaStream_t st) {
  wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace oz2
