// C ABI of the Ozaki-II FP64 GEMM: argument checks, host-side constants,
// the library-owned workspace and the launch sequence of the pipeline
// ("Profiling Ozaki II: The Cost Behind Fast INT8 GEMMs" §1 pipeline table;
// "Ozaki II supplement: INT8 range conditions and paper performance results"
// §1.1-§1.3 for the moduli, residue range and INT32 condition).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "oz2_internal.cuh"

namespace oz2 {
namespace {

// ------------------------------------------------------------ small big-integers
constexpr int kBigLimbs = 6;
struct Big {
  uint32_t l[kBigLimbs] = {0, 0, 0, 0, 0, 0};
};

void big_mul_small(Big& a, uint32_t m) {
  uint64_t c = 0;
  for (int k = 0; k < kBigLimbs; ++k) {
    const uint64_t t = static_cast<uint64_t>(a.l[k]) * m + c;
    a.l[k] = static_cast<uint32_t>(t);
    c = t >> 32;
  }
}

uint32_t big_divmod_small(Big& a, uint32_t m) {  // a /= m, returns a mod m
  uint64_t rem = 0;
  for (int k = kBigLimbs - 1; k >= 0; --k) {
    const uint64_t cur = (rem << 32) | a.l[k];
    a.l[k] = static_cast<uint32_t>(cur / m);
    rem = cur % m;
  }
  return static_cast<uint32_t>(rem);
}

int big_bitlen(const Big& a) {
  for (int k = kBigLimbs - 1; k >= 0; --k)
    if (a.l[k]) {
      int b = 0;
      while (b < 32 && (static_cast<uint64_t>(a.l[k]) >> b) != 0) ++b;
      return 32 * k + b;
    }
  return 0;
}

bool big_bit(const Big& a, int pos) { return (a.l[pos >> 5] >> (pos & 31)) & 1u; }

int gcd(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

struct Tables {
  int moduli[kSMax];
  HostConsts hc[kSMax + 1];
  std::vector<uint8_t> pow2mod;  // [kSMax][kPow2Max]
};

const Tables& tables() {
  static Tables T;
  static std::once_flag once;
  std::call_once(once, [] {
    // greedy: walk down from 256, keep each integer coprime to all kept
    int n = 0;
    for (int m = 256; m >= 2 && n < kSMax; --m) {
      bool ok = true;
      for (int k = 0; k < n; ++k) ok = ok && gcd(m, T.moduli[k]) == 1;
      if (ok) T.moduli[n++] = m;
    }
    T.pow2mod.assign(static_cast<size_t>(kSMax) * kPow2Max, 0);
    for (int t = 0; t < kSMax; ++t) {
      uint32_t v = 1 % T.moduli[t];
      for (int k = 0; k < kPow2Max; ++k) {
        T.pow2mod[static_cast<size_t>(t) * kPow2Max + k] = static_cast<uint8_t>(v);
        v = (v * 2) % T.moduli[t];
      }
    }
    for (int s = OZ2_S_MIN; s <= kSMax; ++s) {
      HostConsts& h = T.hc[s];
      std::memset(&h, 0, sizeof(h));
      ModConsts& mc = h.mod;
      CrtConsts& cc = h.crt;
      mc.s = s;
      cc.s = s;
      Big M;
      M.l[0] = 1;
      for (int t = 0; t < s; ++t) big_mul_small(M, static_cast<uint32_t>(T.moduli[t]));
      for (int t = 0; t < s; ++t) {
        const uint32_t m = static_cast<uint32_t>(T.moduli[t]);
        mc.m[t] = static_cast<int>(m);
        mc.half[t] = static_cast<int>(m / 2);
        mc.magic39[t] = static_cast<uint32_t>(((1ull << 39) + m - 1) / m);
        mc.magic32[t] = static_cast<uint32_t>(((1ull << 32) + m - 1) / m);
        for (int k = 0; k < 3; ++k) {
          uint64_t w = 1;
          for (int b = 0; b < 21 * k; ++b) w = (w * 2) % m;
          mc.w21[t][k] = static_cast<uint32_t>(w);
        }
        for (int k = 0; k < 4; ++k) {
          uint64_t w = 1;
          for (int b = 0; b < 20 * k; ++b) w = (w * 2) % m;
          mc.w20[t][k] = static_cast<uint32_t>(w);
        }
        mc.KH[t] = static_cast<uint32_t>(m * (((1u << 30) + m - 1) / m) + m / 2);
        {
          // fp16 of 1024 + h: exponent 10 (bias 15 -> 25), mantissa h << 0 (h < 1024)
          const uint32_t hbits = (25u << 10) | (m / 2);
          mc.bias2[t] = hbits | (hbits << 16);
        }
        for (int wd = 0; wd < 3; ++wd) {
          uint32_t packed = 0;
          for (int b = 0; b < 4; ++b) {
            uint64_t w = 1;
            for (int e2 = 0; e2 < 8 * (4 * wd + b); ++e2) w = (w * 2) % m;
            packed |= static_cast<uint32_t>(w) << (8 * b);
          }
          mc.wb[t][wd] = packed;
        }
        mc.mf[t] = static_cast<float>(m);
        mc.inv_mf[t] = 1.0f / static_cast<float>(m);
        // CRT constants
        cc.m[t] = static_cast<int>(m);
        Big Mt = M;
        const uint32_t rem = big_divmod_small(Mt, m);
        (void)rem;  // M is a multiple of m
        Big tmp = Mt;
        const uint32_t mt_mod = big_divmod_small(tmp, m);
        uint32_t inv = 0;
        for (uint32_t x = 1; x < m; ++x)
          if ((static_cast<uint64_t>(mt_mod) * x) % m == 1) {
            inv = x;
            break;
          }
        mc.crt_inv_f[t] = static_cast<float>(inv);
        mc.crt_c[t] = mt_mod;
      }
      for (int k = 0; k < kLimbs; ++k) cc.M[k] = M.l[k];
      Big Mh = M;
      big_divmod_small(Mh, 2);
      for (int k = 0; k < kLimbs; ++k) cc.Mhalf[k] = Mh.l[k];
      for (int q = 0; q < kLimbs16; ++q) cc.M16[q] = (M.l[q / 2] >> (16 * (q % 2))) & 0xFFFFu;
      {
        double md = 0.0;
        for (int k = kLimbs - 1; k >= 0; --k) md = md * 4294967296.0 + static_cast<double>(M.l[k]);
        for (int b = 0; b < 2 * kLimbs16; ++b) cc.est_f[b] = static_cast<float>(std::ldexp(1.0, 8 * b) / md);
      }
      // byte limbs of M/m_t, four channels per word
      for (int t = 0; t < s; ++t) {
        Big Mt = M;
        big_divmod_small(Mt, static_cast<uint32_t>(T.moduli[t]));
        for (int b = 0; b < 2 * kLimbs16; ++b) {
          const uint32_t byte = (Mt.l[b / 4] >> (8 * (b % 4))) & 0xFFu;
          cc.L4[t / 4][b] |= byte << (8 * (t % 4));
        }
      }
      // L = M/2 - 1
      Big L = Mh;
      for (int k = 0; k < kBigLimbs; ++k) {  // subtract 1
        if (L.l[k] != 0) {
          L.l[k] -= 1;
          break;
        }
        L.l[k] = 0xFFFFFFFFu;
      }
      const int lb = big_bitlen(L);
      h.bound.Lbits = lb;
      uint64_t norm = 0;
      for (int b = 0; b < 64; ++b) {
        const int pos = lb - 1 - b;
        norm <<= 1;
        if (pos >= 0 && big_bit(L, pos)) norm |= 1;
      }
      h.bound.Lnorm = norm;
    }
  });
  return T;
}

// ------------------------------------------------------------ per-device state
struct DeviceState {
  int* err = nullptr;          // device error word
  uint8_t* pow2mod = nullptr;  // [kSMax][kPow2Max]
  int num_sms = 0;
  bool supported = false;
};

constexpr int kMaxBlocks = 8;  // row blocks of the overlapped schedule
constexpr int kMaxParts = 4;   // column parts of its first (and, host entry point, last) row block
constexpr int kMaxTasks = kMaxBlocks + 2 * kMaxParts;  // GEMM launches

struct Workspace {
  size_t bytes = 0;
  uint8_t* base = nullptr;
  // second stream and events of the overlapped schedule (created on first use)
  cudaStream_t aux = nullptr;
  // the overlapped schedule's GEMM launches, at the device's greatest stream
  // priority, so that the block scheduler places a GEMM's CTAs before the
  // blocks of a side kernel that became ready at the same moment
  cudaStream_t gemm = nullptr;
  cudaEvent_t ev_gemm_go = nullptr;
  cudaEvent_t ev_ready = nullptr;
  cudaEvent_t ev_res[kMaxBlocks] = {};
  cudaEvent_t ev_gemm[kMaxTasks] = {};
  cudaEvent_t ev_bpart[kMaxParts] = {};  // B's planes of each first-block column part made
  cudaEvent_t ev_done = nullptr;
  cudaEvent_t ev_start = nullptr;
  cudaEvent_t ev_bready = nullptr;
  // host entry point: uploads of A's row blocks and B's column parts on their own stream
  cudaStream_t up = nullptr;
  cudaEvent_t ev_io = nullptr;
  cudaEvent_t ev_upA[kMaxBlocks] = {};
  cudaEvent_t ev_upB[kMaxParts] = {};
};

std::mutex g_mutex;
std::atomic<uint64_t> g_launches{0};

struct Profile {
  bool on = false;
  int max_calls = 0;
  std::vector<cudaEvent_t> ev;  // 6 per recorded call
  int used = 0;
};
Profile g_prof;
std::map<int, DeviceState> g_dev;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

oz2_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZ2_ERR_CUDA;
  auto it = g_dev.find(dev);
  if (it == g_dev.end()) {
    DeviceState ds;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&ds.num_sms, cudaDevAttrMultiProcessorCount, dev);
    ds.supported = (major == 10 && minor == 3);
    if (ds.supported) {
      if (cudaMalloc(&ds.err, sizeof(int)) != cudaSuccess) return OZ2_ERR_NO_MEMORY;
      if (cudaMemset(ds.err, 0, sizeof(int)) != cudaSuccess) return OZ2_ERR_CUDA;
      const auto& T = tables();
      if (cudaMalloc(&ds.pow2mod, T.pow2mod.size()) != cudaSuccess) return OZ2_ERR_NO_MEMORY;
      if (cudaMemcpy(ds.pow2mod, T.pow2mod.data(), T.pow2mod.size(), cudaMemcpyHostToDevice) != cudaSuccess)
        return OZ2_ERR_CUDA;
    }
    it = g_dev.emplace(dev, ds).first;
  }
  *out = &it->second;
  return it->second.supported ? OZ2_OK : OZ2_ERR_UNSUPPORTED_DEVICE;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  size_t alpha, beta, amaxA, amaxB, sumA, sumB, u, v, rowkey, colkey, planesA, planesB, R;
  size_t stageA, stageB, stageC;
  size_t total;
};

Layout make_layout(int64_t p, int64_t q, int64_t r, int s, int64_t qp, bool staging) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.alpha = take(p * 4);
  L.beta = take(r * 4);
  L.amaxA = take(p * 8);
  L.amaxB = take(r * 8);
  L.sumA = take(p * 8);
  L.sumB = take(r * 8);
  L.u = take(p * 4);
  L.v = take(r * 4);
  L.rowkey = take(p * 8);
  L.colkey = take(r * 8);
  L.planesA = take(static_cast<size_t>(s) * p * qp * 2);
  L.planesB = take(static_cast<size_t>(s) * r * qp * 2);
  L.R = take(static_cast<size_t>(s) * p * ((r + 3) / 4) * 4);  // coefficient words, 4 columns each
  if (staging) {
    L.stageA = take(static_cast<size_t>(p) * q * 8);
    L.stageB = take(static_cast<size_t>(q) * r * 8);
    L.stageC = take(static_cast<size_t>(p) * r * 8);
  }
  L.total = off;
  (void)q;
  return L;
}

oz2_status workspace_sync_objects(Workspace& w) {
  if (w.aux) return OZ2_OK;
  if (cudaStreamCreateWithFlags(&w.aux, cudaStreamNonBlocking) != cudaSuccess) return OZ2_ERR_CUDA;
  if (cudaStreamCreateWithFlags(&w.up, cudaStreamNonBlocking) != cudaSuccess) return OZ2_ERR_CUDA;
  int least = 0, greatest = 0;
  if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return OZ2_ERR_CUDA;
  if (cudaStreamCreateWithPriority(&w.gemm, cudaStreamNonBlocking, greatest) != cudaSuccess) return OZ2_ERR_CUDA;
  auto mk = [](cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
  bool ok = mk(&w.ev_ready) && mk(&w.ev_done) && mk(&w.ev_start) && mk(&w.ev_bready) && mk(&w.ev_io) && mk(&w.ev_gemm_go);
  for (int b = 0; b < kMaxBlocks; ++b) ok = ok && mk(&w.ev_res[b]) && mk(&w.ev_upA[b]);
  for (int c = 0; c < kMaxParts; ++c) ok = ok && mk(&w.ev_upB[c]) && mk(&w.ev_bpart[c]);
  for (int t = 0; t < kMaxTasks; ++t) ok = ok && mk(&w.ev_gemm[t]);
  return ok ? OZ2_OK : OZ2_ERR_CUDA;
}

// Streams and events of a workspace (the device's work on them must be finished).
void destroy_sync_objects(Workspace& w) {
  if (!w.aux) return;
  auto ev = [](cudaEvent_t& e) {
    if (e) cudaEventDestroy(e);
    e = nullptr;
  };
  ev(w.ev_ready);
  ev(w.ev_done);
  ev(w.ev_start);
  ev(w.ev_bready);
  ev(w.ev_io);
  ev(w.ev_gemm_go);
  for (auto& e : w.ev_res) ev(e);
  for (auto& e : w.ev_upA) ev(e);
  for (auto& e : w.ev_upB) ev(e);
  for (auto& e : w.ev_bpart) ev(e);
  for (auto& e : w.ev_gemm) ev(e);
  for (cudaStream_t* sp : {&w.aux, &w.up, &w.gemm}) {
    if (*sp) cudaStreamDestroy(*sp);
    *sp = nullptr;
  }
}

oz2_status get_workspace(cudaStream_t st, size_t bytes, uint8_t** base, Workspace** wout = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZ2_ERR_CUDA;
  Workspace& w = g_ws[std::make_pair(dev, st)];
  if (wout) *wout = &w;
  if (w.bytes < bytes) {
    if (w.base) {
      cudaDeviceSynchronize();
      cudaFree(w.base);
      w.base = nullptr;
      w.bytes = 0;
    }
    if (std::getenv("OZ2_FAIL_ALLOC") != nullptr) return OZ2_ERR_NO_MEMORY;  // host-side fault injection
    if (cudaMalloc(&w.base, bytes) != cudaSuccess) {
      cudaGetLastError();
      w.base = nullptr;
      return OZ2_ERR_NO_MEMORY;
    }
    w.bytes = bytes;
  }
  *base = w.base;
  return OZ2_OK;
}

oz2_status check_args(int64_t p, int64_t q, int64_t r, const void* A, int64_t lda, const void* B,
                      int64_t ldb, const void* C, int64_t ldc, int s, int mode) {
  if (p <= 0 || q <= 0 || r <= 0) return OZ2_ERR_INVALID_ARG;
  if (lda < p || ldb < q || ldc < p) return OZ2_ERR_INVALID_ARG;
  if (!A || !B || !C) return OZ2_ERR_INVALID_ARG;
  if (s < OZ2_S_MIN || s > OZ2_S_MAX) return OZ2_ERR_INVALID_ARG;
  if (mode != OZ2_FAST && mode != OZ2_ACCU) return OZ2_ERR_INVALID_ARG;
  if (q >= (mode == OZ2_FAST ? OZ2_Q_LIMIT_FAST : OZ2_Q_LIMIT_ACCU)) return OZ2_ERR_Q_TOO_LARGE;
  if (p > (int64_t(1) << 31) - 1024 || r > (int64_t(1) << 31) - 1024) return OZ2_ERR_INVALID_ARG;
  return OZ2_OK;
}

struct Outputs {  // optional checking outputs
  int32_t* alpha = nullptr;
  int32_t* beta = nullptr;
  int8_t* Ares = nullptr;
  int8_t* Bres = nullptr;
  int32_t* P = nullptr;
  uint8_t* R = nullptr;
  uint64_t* X = nullptr;
};

#define OZ2_CU(call)                                 \
  do {                                               \
    if ((call) != cudaSuccess) return OZ2_ERR_CUDA;  \
  } while (0)

// Host buffers of the host-memory entry point: A and B are uploaded into the
// device staging copies the pipeline reads, C is downloaded from its device copy.
struct HostIO {
  const double* A;
  int64_t lda;
  const double* B;
  int64_t ldb;
  double* C;
  int64_t ldc;
};

// The pipeline.  ev (optional, 6 events) is recorded at the stage boundaries.
// io (optional): the host-memory entry point.  A (lda = p) and B (ldb = q)
// are then device staging buffers that the pipeline fills from io->A and
// io->B itself, piece by piece in the order the overlapped schedule consumes
// them, and each finished part of C is copied to io->C as soon as its CRT is
// done.
oz2_status run_pipeline(int64_t p, int64_t q, int64_t r, const double* A, int64_t lda,
                        const double* B, int64_t ldb, double* C, int64_t ldc, int s, oz2_mode mode,
                        cudaStream_t st, const Outputs* dbg, cudaEvent_t* ev, uint8_t** ws_out,
                        Layout* lay_out, bool pipelined, const HostIO* io = nullptr) {
  double* hostC = io ? io->C : nullptr;
  const int64_t ldc_host = io ? io->ldc : 0;
  DeviceState* ds = nullptr;
  oz2_status e = device_state(&ds);
  if (e != OZ2_OK) return e;
  const HostConsts* hc = host_consts(s);
  const int64_t qp = (q + kKPad - 1) / kKPad * kKPad;
  const Layout L = make_layout(p, q, r, s, qp, lay_out != nullptr);
  uint8_t* ws = nullptr;
  Workspace* wsp = nullptr;
  e = get_workspace(st, L.total, &ws, &wsp);
  if (e != OZ2_OK) return e;
  if (ws_out) *ws_out = ws;
  if (lay_out) *lay_out = L;
  auto at = [&](size_t off) { return ws + off; };
  int32_t* alpha = reinterpret_cast<int32_t*>(at(L.alpha));
  int32_t* beta = reinterpret_cast<int32_t*>(at(L.beta));
  uint64_t* amaxA = reinterpret_cast<uint64_t*>(at(L.amaxA));
  uint64_t* amaxB = reinterpret_cast<uint64_t*>(at(L.amaxB));
  uint16_t* planesA = reinterpret_cast<uint16_t*>(at(L.planesA));
  uint16_t* planesB = reinterpret_cast<uint16_t*>(at(L.planesB));
  uint8_t* Rw = at(L.R);
  ScaleArgs sa{p, q, r, lda, ldb, A, B};

  // Row blocks of the overlapped schedule: residues of block b+1 and the CRT
  // of block b run on a second stream while the tensor cores work on the
  // GEMMs of block b (the grouped-overlap idea of the profiling study, §10.2,
  // applied to row blocks so that the CRT overlaps too).
  int64_t block_rows = (p + 3) / 4;
  block_rows = (block_rows + 255) / 256 * 256;  // whole 256-row pair tiles
  if (block_rows < 1024) block_rows = 1024;
  // Small products run as one block: below about 2^35 multiply-adds in fast
  // mode (2^32 in accu mode) the extra launches and cross-stream waits of the
  // overlapped schedule cost more than the work they hide (measured 3-15 %
  // on 1536- to 4096-row shapes).  The host entry point keeps its blocks,
  // which also stage its uploads.
  const double work = static_cast<double>(p) * static_cast<double>(q) * static_cast<double>(r);
  if (io == nullptr && work < (mode == OZ2_FAST ? 0x1p35 : 0x1p32)) block_rows = p;
  const int nb = static_cast<int>((p + block_rows - 1) / block_rows);
  const bool overlap = pipelined && dbg == nullptr && nb > 1 && nb <= kMaxBlocks;
  // one row block, fast mode, both sides in one read each: the two kernels run side by side
  const bool side_by_side = pipelined && dbg == nullptr && nb == 1 && mode == OZ2_FAST &&
                            rows_fused_fast_supported(q) && cols_fused_fast_supported(q);
  if (overlap || side_by_side) {
    e = workspace_sync_objects(*wsp);
    if (e != OZ2_OK) return e;
  }
  const int max_bits = (hc->bound.Lbits + 1) / 2;
  bool b_side_done = false;   // B's exponents and residue planes already enqueued (on aux)
  bool b_planes_done = false;  // B's residue planes already enqueued on `stream`
  // fast mode: B's statistics, exponents and residue planes in one read of B,
  // and, for short rows, A's likewise
  const bool fused_b = (mode == OZ2_FAST) && cols_fused_fast_supported(q);
  const bool fused_a = (mode == OZ2_FAST) && rows_fused_fast_supported(q);
  bool a_planes_done = false;  // A's residue planes already enqueued on `stream` (sequential path)
  auto rows_block = [&](int64_t r0, int64_t rows) { return ScaleArgs{rows, q, r, lda, ldb, A + r0, B}; };
  // Column parts of the first row block's GEMM in the overlapped schedule: it
  // starts once B's first part is ready, and the rest of B is made beside it.
  // Parts are whole multiples of 512 columns (pairs of 256-column tiles); at
  // most `want` of them.  (In the device entry point, splitting the last block
  // too, so that the CRT of its first parts overlaps the GEMM of the rest,
  // measured slower: the extra GEMM launches cost more than the hidden CRT.)
  auto col_parts = [&](int want, int64_t* c) {
    c[0] = 0;
    c[1] = r;
    if (want > r / 1024) want = static_cast<int>(r / 1024);  // parts of at least 1024 columns
    if (want < 2) return 1;
    const int64_t w = (r / want + 511) / 512 * 512;
    int n = 0;
    for (int64_t c0 = 0; c0 < r; c0 += w) c[n++] = c0;
    c[n] = r;
    return n;
  };
  int64_t cfirst[kMaxParts + 1], clast[kMaxParts + 1];
  // (host entry point: four parts, so that the first GEMM waits for a quarter
  // of B's upload instead of half)
  const int nfirst = col_parts(fused_b ? (io ? 4 : 2) : 1, cfirst);
  // With host buffers the last row block's GEMM is split too (four parts): the
  // CRT and the download of each part then run beside the GEMM of the next,
  // which leaves a quarter of a block's download after the last GEMM.
  const int nlast = col_parts(io ? 4 : 1, clast);
  auto rows_of = [&](int b) { return std::min<int64_t>(block_rows, p - b * block_rows); };

  // Host entry point: uploads into the staging copies A, B.  In the overlapped
  // fast schedule they go on their own stream in the order the schedule
  // consumes them (A's row block 0, B's column parts, A's later row blocks),
  // each followed by an event its consumers wait for; otherwise all first.
  const bool staged = io != nullptr && mode == OZ2_FAST && overlap;
  auto upload_rows = [&](int64_t r0, int64_t rows, cudaStream_t s2) {  // A rows [r0, r0 + rows)
    return cudaMemcpy2DAsync(const_cast<double*>(A) + r0, lda * 8, io->A + r0, io->lda * 8, rows * 8, q,
                             cudaMemcpyHostToDevice, s2);
  };
  auto upload_cols = [&](int64_t c0, int64_t cols, cudaStream_t s2) {  // B columns [c0, c0 + cols)
    double* dst = const_cast<double*>(B) + c0 * ldb;
    const double* src = io->B + c0 * io->ldb;
    if (io->ldb == q && ldb == q) return cudaMemcpyAsync(dst, src, q * cols * 8, cudaMemcpyHostToDevice, s2);
    return cudaMemcpy2DAsync(dst, ldb * 8, src, io->ldb * 8, q * 8, cols, cudaMemcpyHostToDevice, s2);
  };
  if (io && !staged) {
    OZ2_CU(upload_rows(0, p, st));
    OZ2_CU(upload_cols(0, r, st));
  } else if (staged) {
    cudaStream_t up = wsp->up;
    OZ2_CU(cudaEventRecord(wsp->ev_io, st));  // after this stream's earlier work on the staging copies
    OZ2_CU(cudaStreamWaitEvent(up, wsp->ev_io, 0));
    OZ2_CU(upload_rows(0, rows_of(0), up));
    OZ2_CU(cudaEventRecord(wsp->ev_upA[0], up));
    for (int c = 0; c < nfirst; ++c) {
      OZ2_CU(upload_cols(cfirst[c], cfirst[c + 1] - cfirst[c], up));
      OZ2_CU(cudaEventRecord(wsp->ev_upB[c], up));
    }
    for (int b = 1; b < nb; ++b) {
      OZ2_CU(upload_rows(b * block_rows, rows_of(b), up));
      OZ2_CU(cudaEventRecord(wsp->ev_upA[b], up));
    }
  }

  if (ev) OZ2_CU(cudaEventRecord(ev[0], st));
  if (mode == OZ2_FAST && overlap) {
    // A side on `stream` (statistics of row block 0 only: alpha_i depends on
    // row i alone, so later blocks get theirs on the second stream), then the
    // B side (statistics, exponents, residue planes) on the second stream
    // A's first-block statistics run alone first: beside B's one-read kernel
    // (which fills every SM's registers) their blocks would hardly be scheduled
    if (staged) OZ2_CU(cudaStreamWaitEvent(st, wsp->ev_upA[0], 0));
    if (fused_a)
      OZ2_CU(launch_rows_fused_fast(A, rows_of(0), q, lda, qp, p, hc->bound, hc->mod, ds->pow2mod, max_bits, alpha,
                                    planesA, st));
    else
      OZ2_CU(launch_fast_exponents_rows(rows_block(0, std::min<int64_t>(block_rows, p)), hc->bound, amaxA,
                                        reinterpret_cast<uint64_t*>(at(L.sumA)), alpha, st));
    OZ2_CU(cudaEventRecord(wsp->ev_start, st));
    OZ2_CU(cudaStreamWaitEvent(wsp->aux, wsp->ev_start, 0));
    if (fused_b) {
      for (int c = 0; c < nfirst; ++c) {
        const int64_t c0 = cfirst[c];
        if (staged) OZ2_CU(cudaStreamWaitEvent(wsp->aux, wsp->ev_upB[c], 0));
        OZ2_CU(launch_cols_fused_fast(B + c0 * ldb, q, cfirst[c + 1] - c0, ldb, qp, r, hc->bound, hc->mod,
                                      ds->pow2mod, max_bits, beta + c0, planesB + c0 * qp, ds->err, wsp->aux));
        OZ2_CU(cudaEventRecord(wsp->ev_bpart[c], wsp->aux));
      }
    } else {
      if (staged) OZ2_CU(cudaStreamWaitEvent(wsp->aux, wsp->ev_upB[0], 0));  // one part: all of B
      OZ2_CU(launch_fast_exponents_cols(sa, hc->bound, amaxB, reinterpret_cast<uint64_t*>(at(L.sumB)), beta,
                                        wsp->aux));
      OZ2_CU(launch_residues_cols(B, q, r, ldb, qp, r, hc->mod, beta, ds->pow2mod, max_bits, planesB, wsp->aux));
    }
    OZ2_CU(cudaEventRecord(wsp->ev_bready, wsp->aux));
    b_side_done = true;
    if (ev) OZ2_CU(cudaEventRecord(ev[1], st));
    if (ev) OZ2_CU(cudaEventRecord(ev[2], st));
  } else if (side_by_side) {
    OZ2_CU(cudaEventRecord(wsp->ev_start, st));
    OZ2_CU(cudaStreamWaitEvent(wsp->aux, wsp->ev_start, 0));
    OZ2_CU(launch_cols_fused_fast(B, q, r, ldb, qp, r, hc->bound, hc->mod, ds->pow2mod, max_bits, beta, planesB,
                                  ds->err, wsp->aux));
    OZ2_CU(cudaEventRecord(wsp->ev_bready, wsp->aux));
    OZ2_CU(launch_rows_fused_fast(A, p, q, lda, qp, p, hc->bound, hc->mod, ds->pow2mod, max_bits, alpha, planesA,
                                  st));
    OZ2_CU(cudaStreamWaitEvent(st, wsp->ev_bready, 0));
    a_planes_done = b_planes_done = true;
    if (ev) OZ2_CU(cudaEventRecord(ev[1], st));
    if (ev) OZ2_CU(cudaEventRecord(ev[2], st));
  } else if (mode == OZ2_FAST) {
    if (fused_a) {
      OZ2_CU(launch_rows_fused_fast(A, p, q, lda, qp, p, hc->bound, hc->mod, ds->pow2mod, max_bits, alpha, planesA,
                                    st));
      a_planes_done = true;
    } else {
      OZ2_CU(launch_fast_exponents_rows(sa, hc->bound, amaxA, reinterpret_cast<uint64_t*>(at(L.sumA)), alpha, st));
    }
    if (fused_b) {
      OZ2_CU(launch_cols_fused_fast(B, q, r, ldb, qp, r, hc->bound, hc->mod, ds->pow2mod, max_bits, beta, planesB,
                                    ds->err, st));
      b_planes_done = true;
    } else {
      OZ2_CU(launch_fast_exponents_cols(sa, hc->bound, amaxB, reinterpret_cast<uint64_t*>(at(L.sumB)), beta,
                                        st));
    }
    if (ev) OZ2_CU(cudaEventRecord(ev[1], st));
    if (ev) OZ2_CU(cudaEventRecord(ev[2], st));
  } else {
    int32_t* u = reinterpret_cast<int32_t*>(at(L.u));
    int32_t* v = reinterpret_cast<int32_t*>(at(L.v));
    uint64_t* rowkey = reinterpret_cast<uint64_t*>(at(L.rowkey));
    uint64_t* colkey = reinterpret_cast<uint64_t*>(at(L.colkey));
    // the bound planes live in the first plane of each residue buffer: they
    // are consumed by the bound GEMM before the residue kernels overwrite them
    uint16_t* Abar = planesA;
    uint16_t* Bbar = planesB;
    OZ2_CU(launch_bound_quant(sa, qp, amaxA, amaxB, u, v, Abar, Bbar, ds->err, st));
    if (ev) OZ2_CU(cudaEventRecord(ev[1], st));
    OZ2_CU(cudaMemsetAsync(rowkey, 0, p * 8, st));
    OZ2_CU(cudaMemsetAsync(colkey, 0, r * 8, st));
    GemmArgs g{};
    g.p = p;
    g.r = r;
    g.qp = qp;
    g.s = 1;
    g.Aplanes = Abar;
    g.Bplanes = Bbar;
    g.rowkey = rowkey;
    g.colkey = colkey;
    g.u = u;
    g.v = v;
    g.err = ds->err;
    g.num_sms = ds->num_sms;
    g.use_2sm = std::getenv("OZ2_GEMM_1SM") == nullptr;  // CTA-pair kernel, 128-column tiles
    OZ2_CU(launch_gemm(kGemmBound, g, hc->mod, st));
    OZ2_CU(launch_accu_exponents(p, r, hc->bound, rowkey, colkey, u, v, alpha, beta, st));
    if (ev) OZ2_CU(cudaEventRecord(ev[2], st));
  }
  // (max_bits: |trunc(2^alpha a)| <= sqrt(L) in fast mode; accu entries beyond the limbs take the general path)
  GemmArgs g{};
  g.r = r;
  g.qp = qp;
  g.s = s;
  g.p_total = p;
  g.Aplanes = planesA;
  g.Bplanes = planesB;
  g.R = Rw;
  g.err = ds->err;
  g.num_sms = ds->num_sms;
  // CTA-pair GEMM (tcgen05 cta_group::2) unless OZ2_GEMM_1SM selects the single-SM kernel
  g.use_2sm = std::getenv("OZ2_GEMM_1SM") == nullptr;
  if (!overlap) {
    if (!a_planes_done)
      OZ2_CU(launch_residues_rows(A, p, q, lda, qp, p, hc->mod, alpha, ds->pow2mod, max_bits, planesA, st));
    if (!b_planes_done)
      OZ2_CU(launch_residues_cols(B, q, r, ldb, qp, r, hc->mod, beta, ds->pow2mod, max_bits, planesB, st));
    if (ev) OZ2_CU(cudaEventRecord(ev[3], st));
    g.p = p;
    g.row0 = 0;
    OZ2_CU(launch_gemm(kGemmMod, g, hc->mod, st));
    if (ev) OZ2_CU(cudaEventRecord(ev[4], st));
    OZ2_CU(launch_crt(0, p, p, 0, r, r, s, hc->crt, Rw, alpha, beta, C, ldc, dbg ? dbg->X : nullptr, st));
    if (hostC)
      OZ2_CU(cudaMemcpy2DAsync(hostC, ldc_host * 8, C, ldc * 8, p * 8, r, cudaMemcpyDeviceToHost, st));
    if (ev) OZ2_CU(cudaEventRecord(ev[5], st));
  } else {
    cudaStream_t aux = wsp->aux;
    if (!b_side_done)
      OZ2_CU(launch_residues_cols(B, q, r, ldb, qp, r, hc->mod, beta, ds->pow2mod, max_bits, planesB, st));
    if (!fused_a)  // (with fused_a block 0's planes came with its statistics)
      OZ2_CU(launch_residues_rows(A, rows_of(0), q, lda, qp, p, hc->mod, alpha, ds->pow2mod, max_bits,
                                  planesA, st));
    OZ2_CU(cudaEventRecord(wsp->ev_ready, st));
    OZ2_CU(cudaStreamWaitEvent(aux, wsp->ev_ready, 0));
    for (int b = 1; b < nb; ++b) {
      const int64_t r0 = b * block_rows;
      if (staged) OZ2_CU(cudaStreamWaitEvent(aux, wsp->ev_upA[b], 0));
      if (fused_a) {
        OZ2_CU(launch_rows_fused_fast(A + r0, rows_of(b), q, lda, qp, p, hc->bound, hc->mod, ds->pow2mod, max_bits,
                                      alpha + r0, planesA + r0 * qp, aux));
      } else {
        if (mode == OZ2_FAST)
          OZ2_CU(launch_fast_exponents_rows(rows_block(r0, rows_of(b)), hc->bound, amaxA + r0,
                                            reinterpret_cast<uint64_t*>(at(L.sumA)) + r0, alpha + r0, aux));
        OZ2_CU(launch_residues_rows(A + r0, rows_of(b), q, lda, qp, p, hc->mod, alpha + r0, ds->pow2mod,
                                    max_bits, planesA + r0 * qp, aux));
      }
      OZ2_CU(cudaEventRecord(wsp->ev_res[b], aux));
    }
    // GEMM launches, (row block, column part), on the greatest-priority
    // stream.  When a GEMM launch ends, the next one and the CRT of the one
    // that ended become ready together; at equal priority the CRT's blocks
    // could take every SM first, and the next GEMM's CTAs (which need almost
    // all of an SM's shared memory) then waited for the whole CRT.
    cudaStream_t gs = wsp->gemm;
    OZ2_CU(cudaEventRecord(wsp->ev_gemm_go, st));  // after block 0's residues (and statistics)
    OZ2_CU(cudaStreamWaitEvent(gs, wsp->ev_gemm_go, 0));
    struct Task {
      int64_t row0, rows, col0, cols;
    };
    Task tasks[kMaxTasks];
    int ntask = 0;
    for (int b = 0; b < nb; ++b) {
      const int np = (b == 0) ? nfirst : (b == nb - 1 ? nlast : 1);
      const int64_t* cp = (b == 0) ? cfirst : clast;
      for (int c = 0; c < np; ++c) {
        const int64_t c0 = (np == 1) ? 0 : cp[c];
        const int64_t c1 = (np == 1) ? r : cp[c + 1];
        if (b > 0 && c == 0) OZ2_CU(cudaStreamWaitEvent(gs, wsp->ev_res[b], 0));
        // block 0's part c waits for B's part c (one part: for all of B)
        if (b_side_done && b == 0)
          OZ2_CU(cudaStreamWaitEvent(gs, (fused_b && nfirst > 1) ? wsp->ev_bpart[c] : wsp->ev_bready, 0));
        if (ntask == 0 && ev) OZ2_CU(cudaEventRecord(ev[3], gs));
        g.row0 = b * block_rows;
        g.p = rows_of(b);
        g.col0 = c0;
        g.ncols = c1 - c0;
        OZ2_CU(launch_gemm(kGemmMod, g, hc->mod, gs));
        OZ2_CU(cudaEventRecord(wsp->ev_gemm[ntask], gs));
        tasks[ntask++] = Task{g.row0, g.p, c0, c1 - c0};
      }
    }
    if (ev) OZ2_CU(cudaEventRecord(ev[4], gs));
    // CRT (and download) of each launch's output on the second stream
    for (int t = 0; t < ntask; ++t) {
      const Task& k = tasks[t];
      OZ2_CU(cudaStreamWaitEvent(aux, wsp->ev_gemm[t], 0));
      OZ2_CU(launch_crt(k.row0, k.rows, p, k.col0, k.cols, r, s, hc->crt, Rw, alpha, beta, C, ldc, nullptr, aux));
      if (hostC)
        OZ2_CU(cudaMemcpy2DAsync(hostC + k.row0 + k.col0 * ldc_host, ldc_host * 8, C + k.row0 + k.col0 * ldc,
                                 ldc * 8, k.rows * 8, k.cols, cudaMemcpyDeviceToHost, aux));
    }
    OZ2_CU(cudaEventRecord(wsp->ev_done, aux));
    OZ2_CU(cudaStreamWaitEvent(st, wsp->ev_done, 0));
    if (ev) OZ2_CU(cudaEventRecord(ev[5], st));
  }

  if (dbg) {
    if (dbg->alpha) OZ2_CU(cudaMemcpyAsync(dbg->alpha, alpha, p * 4, cudaMemcpyDeviceToDevice, st));
    if (dbg->beta) OZ2_CU(cudaMemcpyAsync(dbg->beta, beta, r * 4, cudaMemcpyDeviceToDevice, st));
    if (dbg->R) OZ2_CU(launch_w_to_r(Rw, p, r, hc->mod, dbg->R, st));
    if (dbg->Ares) OZ2_CU(launch_planes_to_int8(planesA, p, q, qp, s, dbg->Ares, st));
    if (dbg->Bres) OZ2_CU(launch_planes_to_int8(planesB, r, q, qp, s, dbg->Bres, st));
    if (dbg->P) {
      GemmArgs g{};
      g.p = p;
      g.r = r;
      g.qp = qp;
      g.s = s;
      g.Aplanes = planesA;
      g.Bplanes = planesB;
      g.P = dbg->P;
      g.err = ds->err;
      g.num_sms = ds->num_sms;
      OZ2_CU(launch_gemm(kGemmExactP, g, hc->mod, st));
    }
  }
  return OZ2_OK;
}

}  // namespace

void count_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }

const HostConsts* host_consts(int s) {
  if (s < OZ2_S_MIN || s > kSMax) return nullptr;
  return &tables().hc[s];
}

const int* greedy_moduli20() { return tables().moduli; }

}  // namespace oz2

// =================================================================== C ABI
using namespace oz2;

extern "C" {

oz2_status ozaki2_dgemm(int64_t p, int64_t q, int64_t r, const double* A, int64_t lda,
                        const double* B, int64_t ldb, double* C, int64_t ldc, int s, oz2_mode mode,
                        void* stream) {
  oz2_status e = check_args(p, q, r, A, lda, B, ldb, C, ldc, s, mode);
  if (e != OZ2_OK) return e;
  std::lock_guard<std::mutex> lk(g_mutex);
  cudaEvent_t* ev = nullptr;
  if (g_prof.on && g_prof.used < g_prof.max_calls) ev = &g_prof.ev[static_cast<size_t>(g_prof.used++) * 6];
  return run_pipeline(p, q, r, A, lda, B, ldb, C, ldc, s, mode, static_cast<cudaStream_t>(stream),
                      nullptr, ev, nullptr, nullptr, true);
}

oz2_status ozaki2_profile_begin(int max_calls) {
  if (max_calls < 1 || max_calls > 100000) return OZ2_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mutex);
  for (auto& e : g_prof.ev) cudaEventDestroy(e);
  g_prof.ev.assign(static_cast<size_t>(max_calls) * 6, nullptr);
  for (auto& e : g_prof.ev)
    if (cudaEventCreate(&e) != cudaSuccess) return OZ2_ERR_CUDA;
  g_prof.max_calls = max_calls;
  g_prof.used = 0;
  g_prof.on = true;
  return OZ2_OK;
}

oz2_status ozaki2_profile_end(float* stage_ms_sum, int* ncalls) {
  if (!stage_ms_sum || !ncalls) return OZ2_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mutex);
  for (int k = 0; k < 6; ++k) stage_ms_sum[k] = 0.0f;
  oz2_status res = OZ2_OK;
  for (int c = 0; c < g_prof.used; ++c) {
    cudaEvent_t* e = &g_prof.ev[static_cast<size_t>(c) * 6];
    if (cudaEventSynchronize(e[5]) != cudaSuccess) {
      res = OZ2_ERR_CUDA;
      break;
    }
    for (int k = 0; k < 5; ++k) {
      float ms = 0.0f;
      cudaEventElapsedTime(&ms, e[k], e[k + 1]);
      stage_ms_sum[k] += ms;
    }
    float tot = 0.0f;
    cudaEventElapsedTime(&tot, e[0], e[5]);
    stage_ms_sum[5] += tot;
  }
  *ncalls = g_prof.used;
  for (auto& e : g_prof.ev) cudaEventDestroy(e);
  g_prof.ev.clear();
  g_prof.on = false;
  g_prof.used = 0;
  return res;
}

uint64_t ozaki2_launch_count(void) { return g_launches.load(); }

oz2_status ozaki2_dgemm_debug(int64_t p, int64_t q, int64_t r, const double* A, int64_t lda,
                              const double* B, int64_t ldb, double* C, int64_t ldc, int s, oz2_mode mode,
                              void* stream, int32_t* alpha, int32_t* beta, int8_t* Ares,
                              int8_t* Bres, int32_t* P, uint8_t* R, uint64_t* X) {
  oz2_status e = check_args(p, q, r, A, lda, B, ldb, C, ldc, s, mode);
  if (e != OZ2_OK) return e;
  if (P && q >= OZ2_Q_LIMIT_P) return OZ2_ERR_Q_TOO_LARGE;  // |P_t| <= q 2^14 must fit int32
  std::lock_guard<std::mutex> lk(g_mutex);
  Outputs o;
  o.alpha = alpha;
  o.beta = beta;
  o.Ares = Ares;
  o.Bres = Bres;
  o.P = P;
  o.R = R;
  o.X = X;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = run_pipeline(p, q, r, A, lda, B, ldb, C, ldc, s, mode, st, &o, nullptr, nullptr, nullptr, false);
  if (e != OZ2_OK) return e;
  if (cudaStreamSynchronize(st) != cudaSuccess) return OZ2_ERR_CUDA;
  return OZ2_OK;
}

oz2_status ozaki2_dgemm_stages(int64_t p, int64_t q, int64_t r, const double* A, int64_t lda,
                               const double* B, int64_t ldb, double* C, int64_t ldc, int s, oz2_mode mode,
                               void* stream, float* stage_ms) {
  oz2_status e = check_args(p, q, r, A, lda, B, ldb, C, ldc, s, mode);
  if (e != OZ2_OK) return e;
  if (!stage_ms) return OZ2_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mutex);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaEvent_t ev[6];
  for (auto& x : ev)
    if (cudaEventCreate(&x) != cudaSuccess) return OZ2_ERR_CUDA;
  e = run_pipeline(p, q, r, A, lda, B, ldb, C, ldc, s, mode, st, nullptr, ev, nullptr, nullptr, false);
  if (e == OZ2_OK) {
    if (cudaEventSynchronize(ev[5]) != cudaSuccess) e = OZ2_ERR_CUDA;
    for (int k = 0; k < 5 && e == OZ2_OK; ++k) cudaEventElapsedTime(&stage_ms[k], ev[k], ev[k + 1]);
    if (e == OZ2_OK) cudaEventElapsedTime(&stage_ms[5], ev[0], ev[5]);
  }
  for (auto& x : ev) cudaEventDestroy(x);
  return e;
}

oz2_status ozaki2_dgemm_host(int64_t p, int64_t q, int64_t r, const double* A, int64_t lda,
                             const double* B, int64_t ldb, double* C, int64_t ldc, int s, oz2_mode mode,
                             void* stream) {
  oz2_status e = check_args(p, q, r, A, lda, B, ldb, C, ldc, s, mode);
  if (e != OZ2_OK) return e;
  std::lock_guard<std::mutex> lk(g_mutex);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceState* ds = nullptr;
  e = device_state(&ds);
  if (e != OZ2_OK) return e;
  const int64_t qp = (q + kKPad - 1) / kKPad * kKPad;
  const Layout L = make_layout(p, q, r, s, qp, true);
  uint8_t* ws = nullptr;
  e = get_workspace(st, L.total, &ws);
  if (e != OZ2_OK) return e;
  double* dA = reinterpret_cast<double*>(ws + L.stageA);
  double* dB = reinterpret_cast<double*>(ws + L.stageB);
  double* dC = reinterpret_cast<double*>(ws + L.stageC);
  // the pipeline uploads A and B itself, piece by piece as its schedule needs
  // them, and returns C row block by row block as each CRT finishes
  const HostIO io{A, lda, B, ldb, C, ldc};
  Layout L2;
  e = run_pipeline(p, q, r, dA, p, dB, q, dC, p, s, mode, st, nullptr, nullptr, nullptr, &L2, true, &io);
  if (e != OZ2_OK) return e;
  OZ2_CU(cudaStreamSynchronize(st));
  return OZ2_OK;
}

int ozaki2_moduli(int s, int32_t* out) {
  if (s < OZ2_S_MIN || s > OZ2_S_MAX || !out) return -1;
  const int* m = greedy_moduli20();
  for (int t = 0; t < s; ++t) out[t] = m[t];
  return s;
}

oz2_status ozaki2_last_error(void) {
  std::lock_guard<std::mutex> lk(g_mutex);
  oz2_status res = OZ2_OK;
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_dev) {
    if (!kv.second.err) continue;
    cudaSetDevice(kv.first);
    int v = 0;
    if (cudaMemcpy(&v, kv.second.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
      res = OZ2_ERR_CUDA;
      continue;
    }
    if (v & kErrTimeout) {
      res = OZ2_ERR_DEVICE_TIMEOUT;
      cudaMemset(kv.second.err, 0, sizeof(int));
    }
  }
  cudaSetDevice(cur);
  return res;
}

void ozaki2_workspace_release(void) {
  std::lock_guard<std::mutex> lk(g_mutex);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_ws) {
    cudaSetDevice(kv.first.first);
    cudaDeviceSynchronize();
    if (kv.second.base) cudaFree(kv.second.base);
    destroy_sync_objects(kv.second);  // the second, upload and GEMM streams and their events
  }
  g_ws.clear();
  cudaSetDevice(cur);
}

const char* ozaki2_status_string(oz2_status status) {
  switch (status) {
    case OZ2_OK: return "ok";
    case OZ2_ERR_INVALID_ARG: return "invalid argument";
    case OZ2_ERR_Q_TOO_LARGE: return "inner dimension q at or above its mode's limit";
    case OZ2_ERR_NO_MEMORY: return "workspace allocation failed";
    case OZ2_ERR_CUDA: return "CUDA error";
    case OZ2_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case OZ2_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103";
    case OZ2_ERR_SCRATCH_TOO_SMALL: return "problem exceeds the fixed no-allocation scratch";
  }
  return "unknown status";
}

oz2_status ozaki2_selftest_wait_timeout(int limit_us) {
  if (limit_us < 1 || limit_us > 1000000) return OZ2_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mutex);
  DeviceState* ds = nullptr;
  oz2_status e = device_state(&ds);
  if (e != OZ2_OK) return e;
  int* err = nullptr;
  if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return OZ2_ERR_NO_MEMORY;
  cudaMemset(err, 0, sizeof(int));
  if (launch_wait_timeout_selftest(err, static_cast<long long>(limit_us) * 1000, nullptr) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(err);
    return OZ2_ERR_CUDA;
  }
  int v = 0;
  cudaMemcpy(&v, err, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(err);
  return (v & kErrTimeout) ? OZ2_ERR_DEVICE_TIMEOUT : OZ2_OK;
}

}  // extern "C"
