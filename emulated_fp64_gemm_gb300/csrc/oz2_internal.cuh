// Internal declarations shared by the library's translation units.
//
// Kernels receive their constants by value (small parameter structs), so no
// __constant__ symbol has to be shared across translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ozaki2.h"

namespace oz2 {

constexpr int kSMax = OZ2_S_MAX;
// Multiword integers of the CRT stage: 5 x 32-bit limbs (160 bits).  With
// s <= 20 the product M of the moduli is < 2^156 and sum_t w_t M/m_t < s M < 2^160.
constexpr int kLimbs = 5;
// Residue planes and bound planes store K (the inner dimension) padded to a
// multiple of this, zero-filled, so every plane row is 16-byte aligned and
// whole 64-wide K blocks can be fed to the tensor cores.
constexpr int kKPad = 64;
// Largest shift of the mantissa handled by the per-modulus power table.
constexpr int kPow2Max = 2304;

// Flags in the device error word.
constexpr int kErrTimeout = 1;

struct ModConsts {  // per-modulus constants, indexed by channel t
  int s;
  int m[kSMax];
  int half[kSMax];                // floor(m/2)
  uint32_t magic39[kSMax];        // ceil(2^39/m): floor(x/m) = umulhi(x, magic39) >> 7 for x < 2^31
  uint32_t magic32[kSMax];        // ceil(2^32/m): floor(x/m) = umulhi(x, magic32) for x < 2^16
  uint32_t w21[kSMax][3];         // 2^(21k) mod m, k = 0..2  (three 21-bit limbs)
  uint32_t w20[kSMax][4];         // 2^(20k) mod m, k = 0..3  (four 20-bit limbs)
  uint32_t KH[kSMax];             // K_m + floor(m/2), K_m = m ceil(2^30/m)
  uint32_t wb[kSMax][3];          // byte weights 2^(8(4w+b)) mod m, packed 4 per word (dp4a)
  uint32_t bias2[kSMax];          // fp16x2 bit pattern of (1024 + floor(m/2), 1024 + floor(m/2))
  float mf[kSMax];                // m as float
  float inv_mf[kSMax];            // fl(1/m)
  float crt_inv_f[kSMax];         // (M/m)^-1 mod m as float: the GEMM stores w = R (M/m)^-1 mod m
  uint32_t crt_c[kSMax];          // (M/m) mod m: R = w (M/m) mod m
};

constexpr int kLimbs16 = 2 * kLimbs;  // 16-bit limbs of the same 160 bits

struct CrtConsts {  // per-s CRT constants
  int s;
  int m[kSMax];
  uint32_t M[kLimbs];             // M, 32-bit limbs
  uint32_t Mhalf[kLimbs];         // M/2 (M is even: 256 is always a modulus)
  uint32_t M16[kLimbs16];         // M, 16-bit limbs (one per word)
  float est_f[2 * kLimbs16];      // 2^(8b) / M rounded to float: weight of byte-limb sum b in Y / M
  uint32_t L4[kSMax / 4][2 * kLimbs16];  // byte b of M/m_t for channels t = 4g .. 4g + 3, packed (dp4a); zero past s
};

// 32-bit limbs the CRT kernel uses for sum_t w_t M/m_t < s M: enough for
// bits(M) + 5 bits (s <= 20 < 2^5).  3 for s <= 11, 4 for s <= 15, 5 above.
inline int crt_limbs(int s) { return s <= 11 ? 3 : (s <= 15 ? 4 : 5); }

struct BoundConsts {  // L = M/2 - 1 in the form the exponent kernels compare against
  int Lbits;                      // bit length of L
  uint64_t Lnorm;                 // L scaled so its top bit is bit 63 (exact when Lbits <= 64)
};

struct HostConsts {
  ModConsts mod;
  CrtConsts crt;
  BoundConsts bound;
};

// Filled once per s (2..20) on the host.  Returns nullptr if s is out of range.
const HostConsts* host_consts(int s);
// The greedy moduli list (20 entries).
const int* greedy_moduli20();

// Counts kernel launches (reported by ozaki2_launch_count).
void count_launches(int n);

// ---------------------------------------------------------------- launchers
struct ScaleArgs {
  int64_t p, q, r, lda, ldb;
  const double* A;
  const double* B;
};

// fast mode: alpha[p], beta[r]; uses amaxA/amaxB/sumA/sumB scratch.
cudaError_t launch_fast_exponents(const ScaleArgs& a, const BoundConsts& bc, uint64_t* amaxA,
                                  uint64_t* amaxB, uint64_t* sumA, uint64_t* sumB, int32_t* alpha,
                                  int32_t* beta, cudaStream_t st);

// the same, one side at a time (rows of A / columns of B), for two streams
cudaError_t launch_fast_exponents_rows(const ScaleArgs& a, const BoundConsts& bc, uint64_t* amaxA,
                                       uint64_t* sumA, int32_t* alpha, cudaStream_t st);
cudaError_t launch_fast_exponents_cols(const ScaleArgs& a, const BoundConsts& bc, uint64_t* amaxB,
                                       uint64_t* sumB, int32_t* beta, cudaStream_t st);

// accu mode, first half: amax, quantised bound planes Abar [p][qp], Bbar [r][qp] (fp16),
// and the quantisation exponents u[p], v[r].
cudaError_t launch_bound_quant(const ScaleArgs& a, int64_t qp, uint64_t* amaxA, uint64_t* amaxB,
                               int32_t* u, int32_t* v, uint16_t* Abar, uint16_t* Bbar, int* err,
                               cudaStream_t st);
// accu mode, second half: exponents from the row / column max keys.
cudaError_t launch_accu_exponents(int64_t p, int64_t r, const BoundConsts& bc,
                                  const uint64_t* rowkey, const uint64_t* colkey, const int32_t* u,
                                  const int32_t* v, int32_t* alpha, int32_t* beta, cudaStream_t st);

// residue planes of `rows` rows of A (column-major, leading dimension lda)
// into fp16 planes [s][plane_rows][qp]; `planes` points at the first row.
cudaError_t launch_residues_rows(const double* A, int64_t rows, int64_t q, int64_t lda, int64_t qp,
                                 int64_t plane_rows, const ModConsts& mc, const int32_t* alpha,
                                 const uint8_t* pow2mod, int max_bits, uint16_t* planes,
                                 cudaStream_t st);
// residue planes of `ncols` columns of B (column-major, leading dimension ldb)
// into fp16 planes [s][plane_cols][qp]; B, beta and planes point at the first
// column.
cudaError_t launch_residues_cols(const double* B, int64_t q, int64_t ncols, int64_t ldb, int64_t qp,
                                 int64_t plane_cols, const ModConsts& mc, const int32_t* beta,
                                 const uint8_t* pow2mod, int max_bits, uint16_t* planes, cudaStream_t st);

// fast mode, B side: beta and the residue planes of `ncols` columns
// (identical to launch_fast_exponents_cols followed by launch_residues_cols);
// B, beta and planes point at the first column, plane rows are plane_cols
// apart ([s][plane_cols][qp]).  For q <= 8192 only (cols_fused_fast_supported):
// up to q = 2048 one kernel reads B once for both, above that the statistics
// take one read of B and the residues a second.
bool cols_fused_fast_supported(int64_t q);
cudaError_t launch_cols_fused_fast(const double* B, int64_t q, int64_t ncols, int64_t ldb, int64_t qp,
                                   int64_t plane_cols, const BoundConsts& bc, const ModConsts& mc,
                                   const uint8_t* pow2mod, int max_bits, int32_t* beta, uint16_t* planes,
                                   int* err, cudaStream_t st);

// fast mode, A side for short rows in one read of A: alpha and the residue
// planes of `rows` rows (identical to launch_fast_exponents_rows followed by
// launch_residues_rows); A, alpha and planes point at the first row, plane
// rows are plane_rows apart.  For q <= 2048 only (rows_fused_fast_supported).
bool rows_fused_fast_supported(int64_t q);
cudaError_t launch_rows_fused_fast(const double* A, int64_t rows, int64_t q, int64_t lda, int64_t qp,
                                   int64_t plane_rows, const BoundConsts& bc, const ModConsts& mc,
                                   const uint8_t* pow2mod, int max_bits, int32_t* alpha, uint16_t* planes,
                                   cudaStream_t st);

// GEMM epilogue kinds
enum GemmKind { kGemmMod = 0, kGemmExactP = 1, kGemmBound = 2 };

struct GemmArgs {
  int64_t p, r, qp;       // rows of output computed by this launch, rows of B planes, padded K
  int64_t row0 = 0;       // first row (of A's planes and of the output) of this launch
  int64_t p_total = 0;    // rows of A's planes and of R / P (0: same as p)
  int64_t col0 = 0;       // first output column of this launch (CTA-pair kernel only)
  int64_t ncols = 0;      // output columns of this launch (0: all r)
  int s;                  // number of channels (planes)
  const uint16_t* Aplanes;  // [s][p][qp]
  const uint16_t* Bplanes;  // [s][r][qp]
  uint8_t* R;             // kGemmMod: CRT coefficients w_t = R_t (M/m_t)^-1 mod m_t,
                          // [s][ceil(r/4)][p_total][4] (4 consecutive columns of a row per word)
  int32_t* P;             // kGemmExactP: [s][r][p]
  uint64_t* rowkey;       // kGemmBound: [p]
  uint64_t* colkey;       // kGemmBound: [r]
  const int32_t* u;       // kGemmBound: [p]
  const int32_t* v;       // kGemmBound: [r]
  int* err;               // device error word
  int num_sms;
  bool use_2sm = false;   // kGemmMod only: CTA-pair kernel (tcgen05 cta_group::2)
};

cudaError_t launch_gemm(GemmKind kind, const GemmArgs& g, const ModConsts& mc, cudaStream_t st);

// CRT + inverse scaling of output rows [row0, row0 + rows) and columns
// [col0, col0 + cols) (col0 a multiple of 4; W, X: p_total rows, r columns)
cudaError_t launch_crt(int64_t row0, int64_t rows, int64_t p_total, int64_t col0, int64_t cols,
                       int64_t r, int s, const CrtConsts& cc, const uint8_t* W,
                       const int32_t* alpha, const int32_t* beta, double* C, int64_t ldc,
                       uint64_t* X, cudaStream_t st);

// debug copies: R_t = w_t (M/m_t) mod m_t from the stored CRT coefficients w_t
cudaError_t launch_w_to_r(const uint8_t* W, int64_t p, int64_t r, const ModConsts& mc, uint8_t* R,
                          cudaStream_t st);
cudaError_t launch_planes_to_int8(const uint16_t* planes, int64_t rows, int64_t q, int64_t qp,
                                  int s, int8_t* out, cudaStream_t st);

cudaError_t launch_wait_timeout_selftest(int* err, long long limit_ns, cudaStream_t st);

}  // namespace oz2

// ------------------------------------------------------------ device helpers
#ifdef __CUDACC__
namespace oz2 {

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of the given parity to complete.  Gives up (returns
// false) after limit_ns of wall time or as soon as *abort is set, so no wait
// in this library can spin forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t addr, uint32_t parity,
                                                  volatile int* abort, uint64_t limit_ns) {
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t addr) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}\n" ::"r"(addr)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t addr, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}\n" ::"r"(addr),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

}  // namespace oz2
#endif
