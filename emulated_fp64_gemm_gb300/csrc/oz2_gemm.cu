// The s modular GEMMs P_t = A_t B_t of Ozaki II on the 5th-generation tensor
// cores (tcgen05), with the output reduction R_t = P_t mod m_t fused into the
// epilogue ("Profiling Ozaki II: The Cost Behind Fast INT8 GEMMs" §1, yellow
// and blue stages; "Ozaki II supplement ..." §1.3 for the exactness condition).
//
// sm_103a has no integer tcgen05 MMA, so the residues (integers in
// [-128, 127]) are carried exactly as fp16 and multiplied with
// tcgen05.mma.kind::f16 into fp32 accumulators in tensor memory.  Every
// product is an integer of magnitude <= 2^14 and every partial sum stays an
// integer below 2^24 in magnitude, so the fp32 accumulation is exact as long
// as a K-chunk holds at most 960 terms (1024 for the odd moduli, below):
//   * kGemmMod (the production path): after each K-chunk the epilogue warps
//     replace every accumulator D by D - m*rint(D/m), an exact fp32
//     operation leaving |D| <= 129, and the next chunk accumulates on top.
//     This is the supplement's §1.3 K-blocking (reduce each block modulo the
//     modulus, then combine) done in tensor memory; it also frees the inner
//     dimension from the INT32 bound.  The last chunk yields R_t = D mod m_t.
//   * kGemmExactP / kGemmBound: each chunk starts from zero and is drained
//     into an int32 running sum kept in tensor memory beside the
//     accumulator, giving the exact P_t (checking path) or the exact bound
//     product Wbar = Abar Bbar (accu mode), whose epilogue reduces every row
//     and column to its maximum scaled value.
//
// Structure: one persistent CTA per SM, 6 warps.  Warp 0 issues TMA loads of
// 128x64 (A) and BNx64 (B) fp16 tiles (128-byte swizzle) into a ring of
// shared-memory stages; warp 1 allocates 512 TMEM columns and one thread of
// it issues the MMAs; warps 2-5 are the epilogue.  A work unit is a pair of
// output tiles (same rows, adjacent column tiles) of one channel t; the two
// tiles own TMEM slots 0 and 1 and their K-chunks are interleaved, so while
// the tensor core works on one tile the epilogue processes the other.
// Every wait is bounded in time; a timeout sets the device error word and
// the kernel winds down instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "oz2_internal.cuh"
#include "oz2_tcgen05.cuh"

namespace oz2 {
namespace {

constexpr int BM = 128;           // tile rows (TMEM lanes)
constexpr int BK = 64;            // K per stage: 64 fp16 = one 128-byte swizzle row
constexpr int KC_BLOCKS = 15;     // K-chunk = 15 * 64 = 960 terms (< 2^24 / 2^14 - margin)
// Odd moduli (every channel but the first, m = 256): centered residues are at
// most 127 in magnitude, so products are at most 127^2 = 16129 and a chunk of
// 16 * 64 = 1024 terms on top of a reduced accumulator (|D| <= 127) stays an
// exact fp32 integer: 127 + 1024 * 16129 = 16516223 < 2^24.  The modular GEMMs
// of those channels reduce once every 1024 terms instead of every 960.
constexpr int KC_BLOCKS_ODD = 16;
constexpr int NUM_THREADS = 192;  // 6 warps
constexpr uint64_t kWaitLimitNs = 20ull * 1000 * 1000 * 1000;  // 20 s

template <int BN>
struct Cfg {
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SMEM = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256;
};

struct KParams {
  int64_t p, r;     // output rows of this launch, output columns
  int64_t row0;     // first output row (and row of A's planes) of this launch
  int64_t p_total;  // rows of R / P (their column stride)
  int64_t r4;       // ceil(r / 4): column groups of the coefficient layout
  int64_t col0;     // first output column (and row of B's planes) of this launch (CTA-pair kernel)
  int s;
  int nkb;          // K blocks (qp / 64)
  int nchunks;      // ceil(nkb / KC_BLOCKS): channel 0, and every channel of the checking and bound GEMMs
  int nchunks_odd;  // ceil(nkb / KC_BLOCKS_ODD): channels t >= 1 of the modular GEMMs
  int tiles_m, tiles_n, pairs_n;
  int64_t units;    // s * tiles_m * pairs_n
  uint8_t* R;
  int32_t* P;
  uint64_t* rowkey;
  uint64_t* colkey;
  const int32_t* u;
  const int32_t* v;
  int* err;
  float mf[kSMax];
  float inv_mf[kSMax];
  float wmul[kSMax];  // (M/m_t)^-1 mod m_t: the mod epilogue stores w_t = R_t wmul mod m_t
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major.
template <int BN>
__device__ __forceinline__ constexpr uint32_t instr_desc() {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}

// Column maxima over a warp's 32 rows: each lane holds 32 values (one per
// column).  Five exchange steps halve the columns a lane keeps (16, 8, 4, 2,
// 1 keys cross per step): at the step with offset o a lane keeps the upper
// half of its remaining columns when its own bit o is set and sends the other
// half to lane ^ o, so after the last step lane L holds the maximum of column L
// (31 exchanges instead of 5 x 32 for one full reduction per column).
__device__ __forceinline__ uint64_t warp_column_max(uint64_t (&kc)[32], int lane) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < o; ++k) {
      const uint64_t keep = up ? kc[k + o] : kc[k];
      const uint64_t send = up ? kc[k] : kc[k + o];
      const uint64_t got = __shfl_xor_sync(0xffffffffu, send, o);
      kc[k] = keep > got ? keep : got;
    }
  }
  return kc[0];
}

// Epilogue of the accu bound GEMM for one BNc-column tile slot of one thread's
// row: the chunk's fp32 sums (exact integers below 2^24) are added into the
// int32 running sums held BNc columns further on in tensor memory.  After the
// last chunk the running sums are the bound products Wbar_ij, whose row
// maximum and column maxima (over the warp's 32 rows) go to rowkey / colkey
// by atomics.  The thread handles the 32-column blocks [cb0, cb1) of the slot.
template <int BNc>
__device__ __forceinline__ void bound_epilogue_chunk(uint32_t acc_addr, int c, bool last, int64_t il, int64_t i,
                                                     int64_t j0, int lane, const KParams& kp, int cb0 = 0,
                                                     int cb1 = BNc / 32) {
  const uint32_t sum_addr = acc_addr + BNc;
  const bool row_ok = il < kp.p;
  uint64_t rmax = 0;
#pragma unroll 1
  for (int cb = cb0; cb < cb1; ++cb) {
    uint32_t v[32], sacc[32];
    tmem_ld32(acc_addr + cb * 32, v);
    if (c > 0) tmem_ld32(sum_addr + cb * 32, sacc);
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int add = __float2int_rn(__uint_as_float(v[k]));
      sacc[k] = (c > 0) ? static_cast<uint32_t>(static_cast<int>(sacc[k]) + add) : static_cast<uint32_t>(add);
    }
    if (!last) {
      tmem_st32(sum_addr + cb * 32, sacc);
    } else {
      // row: max_j Wbar_ij; column: max_i Wbar_ij
      uint64_t kc[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int64_t j = j0 + cb * 32 + k;
        const uint64_t w = (row_ok && j < kp.r) ? sacc[k] : 0u;
        rmax = w > rmax ? w : rmax;
        kc[k] = w;
      }
      const uint64_t cmax = warp_column_max(kc, lane);
      const int64_t jl = j0 + cb * 32 + lane;
      if (cmax && jl < kp.r)
        atomicMax(reinterpret_cast<unsigned long long*>(kp.colkey + jl), static_cast<unsigned long long>(cmax));
    }
  }
  if (last && rmax)
    atomicMax(reinterpret_cast<unsigned long long*>(kp.rowkey + i), static_cast<unsigned long long>(rmax));
  if (!last) tmem_wait_st();
}

// CTA-pair bound GEMM, after the last chunk: from the running sums Wbar_ij
// in registers (this thread's row i, the NB 32-column blocks starting at
// block cb0), the row maximum and the column maxima over the warp's 32 rows
// (one 32-bit warp max reduction per column), each taken into rowkey /
// colkey with one atomic.  The tensor core is already working on the next
// unit meanwhile.
template <int NB>
__device__ __forceinline__ void bound_final_keys_regs(const uint32_t (&w)[NB][32], int64_t il, int64_t i,
                                                      int64_t j0, int lane, const KParams& kp, int cb0) {
  const bool row_ok = il < kp.p;
  uint32_t rmax = 0;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int64_t jl = j0 + (cb0 + b) * 32 + lane;  // this lane's column
    uint32_t cmax = 0;                              // the maximum of column jl
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int64_t j = j0 + (cb0 + b) * 32 + k;
      const uint32_t x = (row_ok && j < kp.r) ? w[b][k] : 0u;
      rmax = x > rmax ? x : rmax;
      const uint32_t m = __reduce_max_sync(0xffffffffu, x);
      if (lane == k) cmax = m;
    }
    if (cmax != 0 && jl < kp.r)
      atomicMax(reinterpret_cast<unsigned long long*>(kp.colkey + jl), static_cast<unsigned long long>(cmax));
  }
  if (rmax != 0)
    atomicMax(reinterpret_cast<unsigned long long*>(kp.rowkey + i), static_cast<unsigned long long>(rmax));
}

// K-chunks of a unit of channel t.
__device__ __forceinline__ int unit_nchunks(int t, const KParams& kp) {
  return t == 0 ? kp.nchunks : kp.nchunks_odd;
}

// First K block of chunk c: the nkb blocks are split into nch chunks of equal
// size (+-1), each at most KC_BLOCKS (channel 0) or KC_BLOCKS_ODD long.
__device__ __forceinline__ int chunk_begin(int c, int nch, const KParams& kp) {
  return static_cast<int>((static_cast<int64_t>(c) * kp.nkb) / nch);
}

// Final epilogue of one 32-column block: from 32 fp32 accumulators D (exact
// integers, |D| < 2^24) to the CRT coefficients w = (D (M/m)^-1) mod m as
// bytes, packed four consecutive columns per 32-bit word.  FMA-pipe only:
// rr = D - m rint(D/m) (|rr| <= 129), x = rr wm (|x| < 2^15), w = x - m rint(x/m)
// moved into [0, m); the byte is the low byte of fp32(w + 2^23).
__device__ __forceinline__ void final_w_words(const uint32_t (&v)[32], float mf, float inv_m, float wm,
                                              uint32_t (&out)[8]) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    uint32_t b[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float d = __uint_as_float(v[4 * g + h]);
      const float rr = fmaf(-mf, fmaf(d, inv_m, 12582912.0f) - 12582912.0f, d);
      const float x = rr * wm;
      float w = fmaf(-mf, fmaf(x, inv_m, 12582912.0f) - 12582912.0f, x);
      w = (w < 0.0f) ? w + mf : w;
      b[h] = __float_as_uint(w + 8388608.0f);  // low byte = w
    }
    out[g] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
  }
}

// --------------------------------------------------------------------- unit decode
struct Unit {
  int t, tm, tn0, ntile;
};

__device__ __forceinline__ Unit decode_unit(int64_t u, const KParams& kp) {
  const int64_t upp = static_cast<int64_t>(kp.tiles_m) * kp.pairs_n;
  Unit U;
  U.t = static_cast<int>(u / upp);
  const int64_t w = u % upp;
  // grouped raster: groups of GM row tiles, column pairs outer within a group,
  // so the ~152 units in flight cover a compact output block whose A and B
  // tiles stay in L2 while they are reused
  constexpr int GM = 16;
  const int64_t per_group = static_cast<int64_t>(GM) * kp.pairs_n;
  const int64_t g = w / per_group;
  const int64_t idx = w % per_group;
  const int64_t left = kp.tiles_m - g * GM;
  const int rows_in_group = static_cast<int>(left < GM ? left : GM);
  U.tm = static_cast<int>(g * GM + idx % rows_in_group);
  const int pn = static_cast<int>(idx / rows_in_group);
  U.tn0 = pn * 2;
  U.ntile = (U.tn0 + 1 < kp.tiles_n) ? 2 : 1;
  return U;
}

// --------------------------------------------------------------------- the kernel
template <int BN, int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    oz2_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ KParams kp) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* full = bars;                     // [STAGES]
  uint64_t* empty = bars + C::STAGES;        // [STAGES]
  uint64_t* accf = bars + 2 * C::STAGES;     // [2]
  uint64_t* acce = accf + 2;                 // [2]
  uint64_t* drain = acce + 2;                // [1] final wait for in-flight MMAs on abort
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* issued_ctr = reinterpret_cast<int*>(tmem_slot + 2);
  int* consumed_ctr = issued_ctr + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&accf[i]), 1);
      mbar_init(smem_u32(&acce[i]), 128);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    *issued_ctr = 0;
    *consumed_ctr = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < kp.units && ok; u += gridDim.x) {
        const Unit U = decode_unit(u, kp);
        const int nch = unit_nchunks(U.t, kp);
        for (int c = 0; c < nch && ok; ++c) {
          const int kb0 = chunk_begin(c, nch, kp);
          const int kb1 = chunk_begin(c + 1, nch, kp);
          for (int sl = 0; sl < U.ntile && ok; ++sl) {
            for (int kb = kb0; kb < kb1; ++kb) {
              if (!mbar_wait_bounded(smem_u32(&empty[stage]), phase ^ 1, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
              }
              const uint32_t fb = smem_u32(&full[stage]);
              mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
              tma_load_3d(smem_u32(sA + stage * C::A_BYTES), &tmA, kb * BK,
                          static_cast<int>(kp.row0) + U.tm * BM, U.t, fb);
              tma_load_3d(smem_u32(sB + stage * C::B_BYTES), &tmB, kb * BK,
                          static_cast<int>(kp.col0) + (U.tn0 + sl) * BN, U.t, fb);
              ++issued;
              if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1;
              }
            }
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(kp.err, kErrTimeout);
      }
      *issued_ctr = issued;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc<BN>();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t use[2] = {0, 0};
      int consumed = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < kp.units && ok; u += gridDim.x) {
        const Unit U = decode_unit(u, kp);
        const int nch = unit_nchunks(U.t, kp);
        for (int c = 0; c < nch && ok; ++c) {
          const int kb0 = chunk_begin(c, nch, kp);
          const int kb1 = chunk_begin(c + 1, nch, kp);
          for (int sl = 0; sl < U.ntile && ok; ++sl) {
            if (!mbar_wait_bounded(smem_u32(&acce[sl]), (use[sl] & 1) ^ 1, abort_flag, kWaitLimitNs)) {
              ok = false;
              break;
            }
            ++use[sl];
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(sl * 256);
            for (int kb = kb0; kb < kb1; ++kb) {
              if (!mbar_wait_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
              const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {
                const bool first = (kb == kb0) && (k == 0) && (KIND != kGemmMod || c == 0);
                mma_f16(d_tmem, smem_desc(a0 + k * 32), smem_desc(b0 + k * 32), idesc, first ? 0u : 1u);
              }
              mma_commit(smem_u32(&empty[stage]));
              ++consumed;
              if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1;
              }
            }
            if (ok) mma_commit(smem_u32(&accf[sl]));
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(kp.err, kErrTimeout);
      }
      // make sure no MMA is still writing TMEM before the final dealloc
      mma_commit(smem_u32(drain));
      mbar_wait_bounded(smem_u32(drain), 0, abort_flag, kWaitLimitNs);
      *consumed_ctr = consumed;
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quad = warp & 3;            // TMEM lane quadrant this warp may access
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t use[2] = {0, 0};
    bool ok = true;
    for (int64_t u = blockIdx.x; u < kp.units && ok; u += gridDim.x) {
      const Unit U = decode_unit(u, kp);
      const int64_t il = static_cast<int64_t>(U.tm) * BM + row_in_tile;  // row within this launch
      const int64_t i = kp.row0 + il;                                       // global row
      const float mf = kp.mf[U.t];
      const float inv_m = kp.inv_mf[U.t];
      const float wm = kp.wmul[U.t];
      const int nch = unit_nchunks(U.t, kp);
      for (int c = 0; c < nch && ok; ++c) {
        const bool last = (c == nch - 1);
        for (int sl = 0; sl < U.ntile; ++sl) {
          // every lane waits; the outcome is made warp-uniform so the
          // .sync.aligned TMEM accesses below stay convergent
          const bool got = mbar_wait_bounded(smem_u32(&accf[sl]), use[sl] & 1, abort_flag, kWaitLimitNs);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          ++use[sl];
          tc_fence_after();
          const uint32_t acc_addr = tmem_base + lane_addr + static_cast<uint32_t>(sl * 256);
          const int64_t j0 = kp.col0 + static_cast<int64_t>(U.tn0 + sl) * BN;
          if (KIND == kGemmMod) {
            if (!last) {
              // in-place reduction: D <- D - m rint(D/m), exact in fp32
#pragma unroll 1
              for (int cb = 0; cb < BN / 32; ++cb) {
                uint32_t v[32];
                tmem_ld32(acc_addr + cb * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                  const float d = __uint_as_float(v[k]);
                  const float q = fmaf(d, inv_m, 12582912.0f) - 12582912.0f;
                  v[k] = __float_as_uint(fmaf(-mf, q, d));
                }
                tmem_st32(acc_addr + cb * 32, v);
              }
              tmem_wait_st();
            } else {
              // final: R = D mod m in [0, m)
              // layout [t][r4][p_total][4]: four consecutive columns of one row per word
              uint32_t* Wt = reinterpret_cast<uint32_t*>(kp.R) + static_cast<int64_t>(U.t) * kp.r4 * kp.p_total;
#pragma unroll 1
              for (int cb = 0; cb < BN / 32; ++cb) {
                uint32_t v[32];
                tmem_ld32(acc_addr + cb * 32, v);
                tmem_wait_ld();
                if (il < kp.p) {
                  uint32_t wd[8];
                  final_w_words(v, mf, inv_m, wm, wd);
                  const int64_t jg0 = (j0 + cb * 32) >> 2;
#pragma unroll
                  for (int g = 0; g < 8; ++g)
                    if (jg0 + g < kp.r4) Wt[(jg0 + g) * kp.p_total + i] = wd[g];
                }
              }
            }
          } else if (KIND == kGemmBound) {
            bound_epilogue_chunk<BN>(acc_addr, c, last, il, i, j0, lane, kp);
          } else {
            // exact P: drain the chunk into the int32 running sum at column offset +128
            const uint32_t sum_addr = acc_addr + 128;
#pragma unroll 1
            for (int cb = 0; cb < BN / 32; ++cb) {
              uint32_t v[32], sacc[32];
              tmem_ld32(acc_addr + cb * 32, v);
              if (c > 0) tmem_ld32(sum_addr + cb * 32, sacc);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                const int add = __float2int_rn(__uint_as_float(v[k]));
                sacc[k] = (c > 0) ? static_cast<uint32_t>(static_cast<int>(sacc[k]) + add)
                                  : static_cast<uint32_t>(add);
              }
              if (!last) {
                tmem_st32(sum_addr + cb * 32, sacc);
              } else {
                int32_t* Pt = kp.P + static_cast<int64_t>(U.t) * kp.p_total * kp.r;
                if (il < kp.p) {
#pragma unroll
                  for (int k = 0; k < 32; ++k) {
                    const int64_t j = j0 + cb * 32 + k;
                    if (j < kp.r) Pt[j * kp.p_total + i] = static_cast<int32_t>(sacc[k]);
                  }
                }
              }
            }
            if (!last) tmem_wait_st();
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&acce[sl]));
        }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(kp.err, kErrTimeout);
    }
  }

  __syncthreads();
  // On an abort, wait (bounded) for TMA loads still landing in shared memory.
  if (threadIdx.x == 0 && *abort_flag) {
    const int issued = *issued_ctr;
    for (int k = *consumed_ctr; k < issued; ++k) {
      const int st = k % C::STAGES;
      const uint32_t ph = static_cast<uint32_t>((k / C::STAGES) & 1);
      volatile int no_abort = 0;
      if (!mbar_wait_bounded(smem_u32(&full[st]), ph, &no_abort, 100ull * 1000 * 1000)) break;
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512)
                 : "memory");
  }
}

// ====================================================================== 2-SM variant
// A cluster of two CTAs (a CTA pair on two SMs) computes a 256 x 256 tile per
// MMA with tcgen05.mma.cta_group::2: each CTA holds 128 rows of A and 128 of
// the 256 rows of B^T in its own shared memory, and 128 rows x 256 columns of
// the fp32 accumulator in its own tensor memory.  Per SM this needs 32 KB of
// operands per 64-deep K stage instead of 48 KB, so seven stages fit and the
// pipeline covers 1.75x the load latency, and L2 reads drop by a third.
// The leader CTA (rank 0) issues every MMA; both producers signal the
// leader's "full" barriers, the MMA commits are multicast to both CTAs, and
// both epilogues signal the leader's "empty accumulator" barriers.  The chunk
// schedule and the in-place reduction are those of the single-SM kernel.
// BN2 = 256 columns per tile.  A modular GEMM unit is two tiles side by side
// (TMEM slots at columns 0 and 256), so one slot's epilogue runs while the
// tensor core works on the other.  A unit of the accu bound GEMM is one tile:
// its int32 running sum takes the other 256 columns (the accumulator in
// [0, 256), the sum in [256, 512)), so the MMA waits for each chunk's
// epilogue.  That costs less than 128-column tiles, which ran the tensor
// core at about half its rate (the modular GEMM with 128-column tiles: 14.9
// instead of 8.1 ms at n = 8192, s = 14).
template <int BN2>
struct Cfg2 {
  static constexpr int BN = BN2;                             // output columns per tile
  static constexpr int A_BYTES = BM * BK * 2;                // 16 KB: this CTA's 128 rows of A
  static constexpr int B_BYTES = (BN2 / 2) * BK * 2;         // this CTA's half of the tile's rows of B^T
  static constexpr int STAGES = (BN2 == 256) ? 7 : 9;
  static constexpr int STAGE_TX = 2 * (A_BYTES + B_BYTES);   // bytes landing per stage across the pair
  static constexpr int SMEM = 1024 + STAGES * (A_BYTES + B_BYTES) + 256;  // 230,656 bytes for BN2 = 256 (the one in use)
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr), "r"(rank));
  return out;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier that may live in the peer CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 int z, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a, uint64_t b,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// Arrive on the barrier at this shared-memory offset in both CTAs of the pair
// once every MMA issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint32_t addr, uint32_t parity,
                                                          volatile int* abort, uint64_t limit_ns) {
  if (mbar_try_wait_cluster(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(addr, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

struct Unit2 {
  int t, mp, tn0, ntile;  // channel, 256-row pair tile, first 256-column tile, tiles (1 or 2)
};

// SINGLE: one column tile per unit (kp.pairs_n then counts tiles)
template <bool SINGLE>
__device__ __forceinline__ Unit2 decode_unit2(int64_t u, const KParams& kp) {
  // kp.tiles_m counts 256-row pair tiles here
  const int64_t upp = static_cast<int64_t>(kp.tiles_m) * kp.pairs_n;
  Unit2 U;
  U.t = static_cast<int>(u / upp);
  const int64_t w = u % upp;
  constexpr int GM = 8;  // 8 pair tiles = 2048 rows per raster group
  const int64_t per_group = static_cast<int64_t>(GM) * kp.pairs_n;
  const int64_t g = w / per_group;
  const int64_t idx = w % per_group;
  const int64_t left = kp.tiles_m - g * GM;
  const int rows_in_group = static_cast<int>(left < GM ? left : GM);
  U.mp = static_cast<int>(g * GM + idx % rows_in_group);
  const int pn = static_cast<int>(idx / rows_in_group);
  U.tn0 = SINGLE ? pn : pn * 2;
  U.ntile = (!SINGLE && U.tn0 + 1 < kp.tiles_n) ? 2 : 1;
  return U;
}

// Epilogue warps of the CTA-pair kernel: four for the modular GEMMs (one per
// TMEM lane quadrant); eight for the bound GEMM, two per quadrant, each taking
// half of a slot's columns: each holds its columns' int32 running sums in
// registers (128 per thread), and its final step (column maxima by warp
// reductions, atomics) is latency-bound with one warp per scheduler.
template <int KIND>
__host__ __device__ constexpr int epi_warps2() {
  return KIND == kGemmBound ? 8 : 4;
}

template <int BN2, int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(64 + 32 * epi_warps2<KIND>(), 1)
    oz2_gemm2sm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ KParams kp) {
  using C2 = Cfg2<BN2>;
  constexpr int BN = C2::BN, A_BYTES = C2::A_BYTES, B_BYTES = C2::B_BYTES, STAGES = C2::STAGES,
                STAGE_TX = C2::STAGE_TX;
  static_assert(KIND == kGemmMod || KIND == kGemmBound, "CTA-pair epilogues: mod and bound");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * (A_BYTES + B_BYTES));
  uint64_t* full = bars;                  // [STAGES] used in the leader only
  uint64_t* empty = bars + STAGES;        // [STAGES] in both CTAs
  uint64_t* accf = bars + 2 * STAGES;     // [2] in both CTAs
  uint64_t* acce = accf + 2;              // [2] used in the leader only
  uint64_t* drain = acce + 2;             // [1] leader
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const int64_t cluster = blockIdx.x >> 1;
  const int64_t nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&accf[i]), 1);
      mbar_init(smem_u32(&acce[i]), 2 * epi_warps2<KIND>());  // one elected lane per epilogue warp, both CTAs
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // Both CTAs of the pair must be running before the collective TMEM
  // allocation: without this cluster barrier, launches that started while
  // other kernels occupied SMs occasionally never returned from the alloc.
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int64_t u = cluster; u < kp.units && ok; u += nclusters) {
        const Unit2 U = decode_unit2<KIND == kGemmBound>(u, kp);
        const int arow = static_cast<int>(kp.row0) + U.mp * 256 + static_cast<int>(rank) * 128;
        const int nch = unit_nchunks(U.t, kp);
        for (int c = 0; c < nch && ok; ++c) {
          const int kb0 = chunk_begin(c, nch, kp);
          const int kb1 = chunk_begin(c + 1, nch, kp);
          for (int sl = 0; sl < U.ntile && ok; ++sl) {
            const int brow = static_cast<int>(kp.col0) + (U.tn0 + sl) * BN + static_cast<int>(rank) * (BN / 2);
            for (int kb = kb0; kb < kb1; ++kb) {
              if (!mbar_wait_cluster_bounded(smem_u32(&empty[stage]), phase ^ 1, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
              }
              const uint32_t fb_local = smem_u32(&full[stage]);
              const uint32_t fb_leader = map_to_rank(fb_local, 0);
              if (leader) mbar_arrive_expect_tx(fb_local, STAGE_TX);
              tma_load_3d_pair(smem_u32(sA + stage * A_BYTES), &tmA, kb * BK, arow, U.t, fb_leader);
              tma_load_3d_pair(smem_u32(sB + stage * B_BYTES), &tmB, kb * BK, brow, U.t, fb_leader);
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
              }
            }
          }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(kp.err, kErrTimeout);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer (leader only)
    if (leader && lane == 0) {
      // kind::f16, D fp32, A/B fp16 K-major, N = BN, M = 256 (the pair)
      constexpr uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                 (static_cast<uint32_t>(256 >> 4) << 24);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t use[2] = {0, 0};
      int bslot = 0;  // bound GEMM: the slot of the next chunk (chunks alternate)
      bool ok = true;
      for (int64_t u = cluster; u < kp.units && ok; u += nclusters) {
        const Unit2 U = decode_unit2<KIND == kGemmBound>(u, kp);
        const int nch = unit_nchunks(U.t, kp);
        for (int c = 0; c < nch && ok; ++c) {
          const int kb0 = chunk_begin(c, nch, kp);
          const int kb1 = chunk_begin(c + 1, nch, kp);
          for (int s0 = 0; s0 < U.ntile && ok; ++s0) {
            const int sl = (KIND == kGemmBound) ? bslot : s0;
            if (!mbar_wait_cluster_bounded(smem_u32(&acce[sl]), (use[sl] & 1) ^ 1, abort_flag, kWaitLimitNs)) {
              ok = false;
              break;
            }
            ++use[sl];
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(sl * 256);
            for (int kb = kb0; kb < kb1; ++kb) {
              if (!mbar_wait_cluster_bounded(smem_u32(&full[stage]), phase, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a0 = smem_u32(sA + stage * A_BYTES);
              const uint32_t b0 = smem_u32(sB + stage * B_BYTES);
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {
                // mod: the chunks accumulate on the reduced value; bound: each chunk starts from zero
                const bool first = (kb == kb0) && (k == 0) && (KIND != kGemmMod || c == 0);
                mma_f16_pair(d_tmem, smem_desc(a0 + k * 32), smem_desc(b0 + k * 32), idesc, first ? 0u : 1u);
              }
              mma_commit_pair(smem_u32(&empty[stage]));
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
              }
            }
            if (ok) mma_commit_pair(smem_u32(&accf[sl]));
          }
          if (KIND == kGemmBound) bslot ^= 1;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(kp.err, kErrTimeout);
      }
      mma_commit_pair(smem_u32(drain));
      mbar_wait_bounded(smem_u32(drain), 0, abort_flag, kWaitLimitNs);
    }
  } else {
    // ---------------------------------------------------------- epilogue (warps 2.., both CTAs)
    const int quad = warp & 3;  // the TMEM lane quadrant this warp may access
    constexpr int NPART = epi_warps2<KIND>() / 4;
    const int part = (warp - 2) >> 2;  // column part of each slot (bound GEMM: two)
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t use[2] = {0, 0};
    int bslot = 0;  // bound GEMM: the slot of the next chunk
    // bound GEMM: this thread's int32 running sums W_ij (its row, the
    // NBLK 32-column blocks of its part of the tile)
    constexpr int NBLK = (KIND == kGemmBound) ? BN / 32 / NPART : 1;
    uint32_t bsum[NBLK][32];
    bool ok = true;
    for (int64_t u = cluster; u < kp.units && ok; u += nclusters) {
      const Unit2 U = decode_unit2<KIND == kGemmBound>(u, kp);
      const int64_t il = static_cast<int64_t>(U.mp) * 256 + rank * 128 + row_in_tile;
      const int64_t i = kp.row0 + il;
      const float mf = kp.mf[U.t];
      const float inv_m = kp.inv_mf[U.t];
      const float wm = kp.wmul[U.t];
      const int nch = unit_nchunks(U.t, kp);
      for (int c = 0; c < nch && ok; ++c) {
        const bool last = (c == nch - 1);
        for (int s0 = 0; s0 < U.ntile; ++s0) {
          const int sl = (KIND == kGemmBound) ? bslot : s0;
          const bool got = mbar_wait_cluster_bounded(smem_u32(&accf[sl]), use[sl] & 1, abort_flag, kWaitLimitNs);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          ++use[sl];
          tc_fence_after();
          const uint32_t acc_addr = tmem_base + lane_addr + static_cast<uint32_t>(sl * 256);
          const int64_t j0 = kp.col0 + static_cast<int64_t>((KIND == kGemmBound ? U.tn0 : U.tn0 + sl)) * BN;
          if (KIND == kGemmBound) {
            // every chunk, the last included: the chunk's sums (exact fp32
            // integers) of this warp's columns into the int32 running sums in
            // registers; the slot then goes back to the MMA, which is already
            // working on the next chunk in the other slot.  After the last
            // chunk the keys are taken from the running sums (= W).
            const int cb0 = part * NBLK;
#pragma unroll
            for (int b = 0; b < NBLK; ++b) {
              uint32_t v[32];
              tmem_ld32(acc_addr + (cb0 + b) * 32, v);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                const uint32_t add = static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[k])));
                bsum[b][k] = (c == 0) ? add : bsum[b][k] + add;
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(smem_u32(&acce[sl]), 0));
            if (KIND == kGemmBound) bslot ^= 1;
            if (last) bound_final_keys_regs<NBLK>(bsum, il, i, j0, lane, kp, cb0);
            continue;
          } else if (!last) {
#pragma unroll 1
            for (int cb = 0; cb < BN / 32; ++cb) {
              uint32_t v[32];
              tmem_ld32(acc_addr + cb * 32, v);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) {
                const float d = __uint_as_float(v[k]);
                const float q = fmaf(d, inv_m, 12582912.0f) - 12582912.0f;
                v[k] = __float_as_uint(fmaf(-mf, q, d));
              }
              tmem_st32(acc_addr + cb * 32, v);
            }
            tmem_wait_st();
          } else {
            // layout [t][r4][p_total][4]: four consecutive columns of one row per word
            uint32_t* Wt = reinterpret_cast<uint32_t*>(kp.R) + static_cast<int64_t>(U.t) * kp.r4 * kp.p_total;
#pragma unroll 1
            for (int cb = 0; cb < BN / 32; ++cb) {
              uint32_t v[32];
              tmem_ld32(acc_addr + cb * 32, v);
              tmem_wait_ld();
              if (il < kp.p) {
                uint32_t wd[8];
                final_w_words(v, mf, inv_m, wm, wd);
                const int64_t jg0 = (j0 + cb * 32) >> 2;
#pragma unroll
                for (int g = 0; g < 8; ++g)
                  if (jg0 + g < kp.r4) Wt[(jg0 + g) * kp.p_total + i] = wd[g];
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(map_to_rank(smem_u32(&acce[sl]), 0));
        }
      }
    }
    if (!ok) {
      *abort_flag = 1;
      atomicOr(kp.err, kErrTimeout);
    }
  }

  __syncthreads();
  cluster_sync_all();  // the leader's MMAs are done with both CTAs' shared and tensor memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_plane_map(CUtensorMap* map, const uint16_t* base, int64_t qp, int64_t rows, int s,
                    int box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(qp), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(s)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(qp * 2), static_cast<cuuint64_t>(rows * qp * 2)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, int KIND>
cudaError_t launch_impl(const GemmArgs& g, const ModConsts& mc, cudaStream_t st) {
  using C = Cfg<BN>;
  CUtensorMap ta, tb;
  const int64_t p_total = g.p_total ? g.p_total : g.p;
  if (!make_plane_map(&ta, g.Aplanes, g.qp, p_total, g.s, BM)) return cudaErrorInvalidValue;
  if (!make_plane_map(&tb, g.Bplanes, g.qp, g.r, g.s, BN)) return cudaErrorInvalidValue;
  KParams kp{};
  kp.p = g.p;
  kp.r = g.r;
  kp.row0 = g.row0;
  kp.p_total = p_total;
  kp.r4 = (g.r + 3) / 4;
  kp.s = g.s;
  kp.nkb = static_cast<int>(g.qp / BK);
  kp.nchunks = (kp.nkb + KC_BLOCKS - 1) / KC_BLOCKS;
  kp.nchunks_odd = (KIND == kGemmMod) ? (kp.nkb + KC_BLOCKS_ODD - 1) / KC_BLOCKS_ODD : kp.nchunks;
  kp.tiles_m = static_cast<int>((g.p + BM - 1) / BM);
  kp.col0 = g.col0;
  kp.tiles_n = static_cast<int>(((g.ncols ? g.ncols : g.r) + BN - 1) / BN);
  kp.pairs_n = (kp.tiles_n + 1) / 2;
  kp.units = static_cast<int64_t>(g.s) * kp.tiles_m * kp.pairs_n;
  kp.R = g.R;
  kp.P = g.P;
  kp.rowkey = g.rowkey;
  kp.colkey = g.colkey;
  kp.u = g.u;
  kp.v = g.v;
  kp.err = g.err;
  for (int t = 0; t < kSMax; ++t) {
    kp.mf[t] = mc.mf[t];
    kp.inv_mf[t] = mc.inv_mf[t];
    kp.wmul[t] = mc.crt_inv_f[t];
  }
  auto kern = oz2_gemm_kernel<BN, KIND>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(kp.units, g.num_sms);
  kern<<<static_cast<unsigned>(grid), NUM_THREADS, C::SMEM, st>>>(ta, tb, kp);
  count_launches(1);
  return cudaGetLastError();
}

template <int BN2, int KIND>
cudaError_t launch_2sm(const GemmArgs& g, const ModConsts& mc, cudaStream_t st) {
  using C2 = Cfg2<BN2>;
  CUtensorMap ta, tb;
  const int64_t p_total = g.p_total ? g.p_total : g.p;
  if (!make_plane_map(&ta, g.Aplanes, g.qp, p_total, g.s, 128)) return cudaErrorInvalidValue;
  if (!make_plane_map(&tb, g.Bplanes, g.qp, g.r, g.s, BN2 / 2)) return cudaErrorInvalidValue;
  KParams kp{};
  kp.p = g.p;
  kp.r = g.r;
  kp.row0 = g.row0;
  kp.p_total = p_total;
  kp.r4 = (g.r + 3) / 4;
  kp.s = g.s;
  kp.nkb = static_cast<int>(g.qp / BK);
  kp.nchunks = (kp.nkb + KC_BLOCKS - 1) / KC_BLOCKS;
  kp.nchunks_odd = (KIND == kGemmMod) ? (kp.nkb + KC_BLOCKS_ODD - 1) / KC_BLOCKS_ODD : kp.nchunks;
  kp.tiles_m = static_cast<int>((g.p + 255) / 256);  // 256-row pair tiles
  kp.col0 = g.col0;
  const int64_t ncols = g.ncols ? g.ncols : g.r;
  kp.tiles_n = static_cast<int>((ncols + BN2 - 1) / BN2);
  kp.pairs_n = (KIND == kGemmBound) ? kp.tiles_n : (kp.tiles_n + 1) / 2;  // bound: one tile per unit
  kp.units = static_cast<int64_t>(g.s) * kp.tiles_m * kp.pairs_n;
  kp.R = g.R;
  kp.rowkey = g.rowkey;
  kp.colkey = g.colkey;
  kp.u = g.u;
  kp.v = g.v;
  kp.err = g.err;
  for (int t = 0; t < kSMax; ++t) {
    kp.mf[t] = mc.mf[t];
    kp.inv_mf[t] = mc.inv_mf[t];
    kp.wmul[t] = mc.crt_inv_f[t];
  }
  auto kern = oz2_gemm2sm_kernel<BN2, KIND>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C2::SMEM);
  if (e != cudaSuccess) return e;
  int64_t clusters = std::min<int64_t>(kp.units, g.num_sms / 2);
  if (clusters < 1) clusters = 1;
  kern<<<static_cast<unsigned>(2 * clusters), 64 + 32 * epi_warps2<KIND>(), C2::SMEM, st>>>(ta, tb, kp);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(GemmKind kind, const GemmArgs& g, const ModConsts& mc, cudaStream_t st) {
  switch (kind) {
    case kGemmMod:
      if (g.use_2sm) return launch_2sm<256, kGemmMod>(g, mc, st);
      return launch_impl<256, kGemmMod>(g, mc, st);
    case kGemmExactP:
      return launch_impl<128, kGemmExactP>(g, mc, st);
    case kGemmBound:
      if (g.use_2sm) return launch_2sm<256, kGemmBound>(g, mc, st);
      return launch_impl<128, kGemmBound>(g, mc, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace oz2
