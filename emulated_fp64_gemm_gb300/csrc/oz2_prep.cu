// Preprocessing kernels of the Ozaki-II pipeline: scaling statistics,
// power-of-two exponents and the accu-mode bound quantisation.  The residue
// planes are in oz2_residue.cu.
//
// Method: "Profiling Ozaki II: The Cost Behind Fast INT8 GEMMs" §1 (green
// stage), §2 (fast and accu bounds), §5.1 (row max-abs and sum of squares,
// rounded up).
//
// No floating-point arithmetic is used on the data: every double is taken
// apart into its sign, exponent and 53-bit significand, and all statistics
// are exact integer computations.  This makes the exponents independent of
// the order of the reductions (the statistics are u64 sums and maxima) and
// removes the FP64 pipe from this stage.
#include <cuda_fp16.h>

#include <algorithm>

#include "oz2_bits.cuh"
#include "oz2_internal.cuh"

namespace oz2 {
namespace {

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
  for (; l + 16 <= l1; l += 16) {  // sixteen loads in flight per thread
    uint64_t b[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) b[k] = static_cast<uint64_t>(__double_as_longlong(__ldg(A + (l + k) * lda + i)));
#pragma unroll
    for (int k = 0; k < 16; ++k) {
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
  uint64_t b[8];  // the eight elements' bits, all loads in flight first (0 past q)
#pragma unroll
  for (int k = 0; k < 8; ++k)
    b[k] = (l0 + k < q) ? static_cast<uint64_t>(__double_as_longlong(__ldg(A + (l0 + k) * lda + i))) : 0ull;
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
    // ceil(|a| 2^u) <= 127: 32-bit operations on the top significand bits and a sticky bit
    const uint32_t c[2] = {ceil_scaled_small(b[k], u), ceil_scaled_small(b[k + 1], u)};
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
  uint64_t b[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    b[k] = (l0 + k < q) ? static_cast<uint64_t>(__double_as_longlong(__ldg(B + j * ldb + l0 + k))) : 0ull;
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
    const uint32_t c[2] = {ceil_scaled_small(b[k], v), ceil_scaled_small(b[k + 1], v)};
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
        const uint32_t cq[2] = {
            ceil_scaled_small(static_cast<uint64_t>(__double_as_longlong(x[c][k])), v),
            ceil_scaled_small(static_cast<uint64_t>(__double_as_longlong(x[c][k + 1])), v)};
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

// Accu mode, B side in one read of B for 2048 < q <= 8192: one block per
// column.  The column (contiguous in column-major B) comes into shared memory
// by one bulk copy of its 16-byte aligned middle, with the one element before
// it (a column starting 8 bytes past a 16-byte boundary) and the one after it
// stored beside it, so that column element l sits at word l + 2 - h.  The
// column maximum gives v_j; each thread quantises a strided set of elements
// (conflict-free shared-memory reads), and once every thread is done the fp16
// row of Bbar is staged over the column and written with 16-byte stores.
// Results are identical to amax_cols + bound_quant_cols.  A copy that has not
// landed within kStatsWaitNs sets the timeout bit in *err, and the block
// waits (bounded again) for it before leaving.
constexpr int kBoundColsPerThread = 32;  // q <= 8192 = 256 threads x 32
__global__ void __launch_bounds__(256, 3) bound_cols_bulk_kernel(const double* __restrict__ B, int64_t q,
                                                                 int64_t ldb, int64_t qp,
                                                                 uint64_t* __restrict__ amax,
                                                                 int32_t* __restrict__ v_out,
                                                                 uint16_t* __restrict__ Bbar, int* err) {
  extern __shared__ __align__(16) uint8_t col_smem[];  // (q + 2) doubles; later qp halves
  __shared__ uint64_t red[8];
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t j = blockIdx.x;
  const double* col = B + j * ldb;
  const int h = static_cast<int>((reinterpret_cast<uintptr_t>(col) >> 3) & 1);  // elements before the aligned middle
  const int64_t nmid = ((q - h) / 2) * 2;                                         // elements in it (even)
  double* xs = reinterpret_cast<double*>(col_smem);                              // element l at xs[l + 2 - h]
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(smem_u32(&bar), static_cast<uint32_t>(nmid * 8));
    bulk_copy_g2s(smem_u32(col_smem + 16), col + h, static_cast<uint32_t>(nmid * 8), smem_u32(&bar));
  }
  const bool got = mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, kStatsWaitNs);
  if (__syncthreads_or(!got)) {
    if (tid == 0) {
      atomicOr(err, kErrTimeout);
      mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, kStatsWaitNs);  // the copy still in flight
    }
    return;
  }
  if (tid == 0 && h) xs[1] = __ldg(col);                                       // the element before the middle
  if (tid == 1 && h + nmid < q) xs[q + 1 - h] = __ldg(col + q - 1);            // the element after it
  __syncthreads();
  const double* xe = xs + 2 - h;  // xe[l] = column element l, 0 <= l < q
  uint64_t m = 0;
  for (int64_t l = tid; l < q; l += 256) {
    const uint64_t b = static_cast<uint64_t>(__double_as_longlong(xe[l])) & ~(1ull << 63);
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
  // ceil(|b_l| 2^v) <= 127 for the elements l = tid + 256 k (0 past q)
  uint32_t cq[kBoundColsPerThread];
#pragma unroll
  for (int k = 0; k < kBoundColsPerThread; ++k) {
    const int64_t l = tid + 256ll * k;
    cq[k] = (l < q) ? ceil_scaled_small(static_cast<uint64_t>(__double_as_longlong(xe[l])), v) : 0u;
  }
  __syncthreads();  // every element read: the fp16 row goes over the column
  uint16_t* hs = reinterpret_cast<uint16_t*>(col_smem);
#pragma unroll
  for (int k = 0; k < kBoundColsPerThread; ++k) {
    const int64_t l = tid + 256ll * k;
    if (l < qp) {
      // fp16 of an integer below 1024: bits 0x6400 + c encode 1024 + c; subtract 1024
      const __half hv = __hsub(__ushort_as_half(static_cast<unsigned short>(0x6400u + cq[k])), __ushort_as_half(0x6400));
      hs[l] = __half_as_ushort(hv);
    }
  }
  __syncthreads();
  const uint4* src = reinterpret_cast<const uint4*>(col_smem);
  uint4* dst = reinterpret_cast<uint4*>(Bbar + j * qp);
  for (int64_t c16 = tid; c16 < qp / 8; c16 += 256) dst[c16] = src[c16];
}

// accu exponents ("Profiling Ozaki II" §2 and §5.1: the row and column
// maxima of the bound output give the final scale exponents), with the
// maxima taken in the quantised scale: for row i, R_i = max_j Wbar_ij (from
// the bound GEMM) and alpha_i = u_i + max {a : 4^a R_i <= L}; for column j,
// beta_j = v_j + max {b : 4^b K_j <= L} with K_j = max_i Wbar_ij; 0 for a
// zero row or column.  Then 2^(alpha_i + beta_j) (|A||B|)_ij <=
// 2^(a_i + b_j) Wbar_ij <= sqrt(4^a_i R_i 4^b_j K_j) <= L.
__global__ void accu_exp_kernel(const uint64_t* __restrict__ key, const int32_t* __restrict__ qexp,
                                int64_t n, BoundConsts bc, int32_t* __restrict__ out) {
  const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (i >= n) return;
  const uint64_t k = key[i];  // the row (column) maximum of Wbar
  if (k == 0) {
    out[i] = 0;
    return;
  }
  // 4^a k <= L  <=>  k 2^(2a) <= L  <=>  2a <= h
  out[i] = qexp[i] + (max_shift_le_L(k, bc) >> 1);  // u + floor(h / 2)
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
                               int32_t* u, int32_t* v, uint16_t* Abar, uint16_t* Bbar, int* err,
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
    if (qp <= 2048) {
      fused_cols_bound_kernel<1><<<g, 256, 0, st>>>(a.B, a.q, a.ldb, qp, amaxB, v, Bbar);
    } else {
      // (set on every launch: the attribute belongs to the current device)
      const cudaError_t attr =
          cudaFuncSetAttribute(bound_cols_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (8192 + 2) * 8);
      if (attr != cudaSuccess) return attr;
      bound_cols_bulk_kernel<<<g, 256, (a.q + 2) * 8, st>>>(a.B, a.q, a.ldb, qp, amaxB, v, Bbar, err);
    }
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
