// Bit-level device helpers shared by the preprocessing kernels (statistics,
// bound quantisation and residues): doubles taken apart into sign, exponent
// and significand, exact upward-rounded scalings, the exponent rule of the
// fast bound and the fp16 packing of small integers.  Integer operations
// only: no floating-point arithmetic touches the data.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

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

// fast exponent from the row/column maximum's e and the exact sum of squares S:
// U = S 4^(e-F), exponent = max { a : 4^a U <= L } = floor(h/2) - e + F; 0 for S == 0.
__device__ __forceinline__ int fast_exponent(uint64_t S, int e, const BoundConsts& bc) {
  return (S == 0) ? 0 : (max_shift_le_L(S, bc) >> 1) - e + kF;
}

// fp16 bits of two values v0, v1 in [0, 2048) shifted by -bias, packed (v0 low).
__device__ __forceinline__ uint32_t pack_fp16_pair(uint32_t v0, uint32_t v1, __half2 bias2) {
  const uint32_t word = (v1 << 16 | v0) + 0x64006400u;  // fp16(1024 + v)
  __half2 hv = *reinterpret_cast<const __half2*>(&word);
  hv = __hsub2(hv, bias2);                              // exact: integers below 2048
  return *reinterpret_cast<uint32_t*>(&hv);
}

// Bulk copy of `bytes` (a multiple of 16) from global memory to this CTA's
// shared memory, both addresses 16-byte aligned, counted on an mbarrier.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

constexpr uint64_t kStatsWaitNs = 2ull * 1000 * 1000 * 1000;  // 2 s: a 64 KB copy takes microseconds

}  // namespace
}  // namespace oz2
