/*
 * oz2_oracle.c -- a plain, threaded CPU oracle of Ozaki Scheme II.
 *
 * TEST INFRASTRUCTURE ONLY.  It is the native twin of ozaki2_oracle.py and,
 * like it, the independent reference the CUDA library is checked against:
 * only the tests, the smoke check and the benchmark's CPU-baseline and
 * reference legs load it.  It shares no code, header, table or constant
 * with the library (it includes only the C standard library and pthreads),
 * and the library never loads it.
 *
 * What it computes, step by step as the pages state the method:
 *   "Profiling Ozaki II: The Cost Behind Fast INT8 GEMMs" (cited [P]) §1
 *   pipeline table, §2 the fast and accu bounds, §5.1 statistics; and
 *   "Ozaki II supplement: INT8 range conditions and paper performance
 *   results" (cited [S]) §1.1 pipeline, §1.2 centered residues, §1.3 the
 *   INT32 condition, §2 Eq. (18).
 *   O0  moduli: walk down from 256, keep each integer coprime to every one
 *       kept; M = prod m_t, L = M/2 - 1.
 *   O2  exponents.  fast: e = floor(log2 max|x|) + 1,
 *       S = sum ceil(|x| 2^(20 - e))^2 (exact), alpha = max {a : 4^a S 4^(e-20) <= L}.
 *       accu: u = max {u : ceil(max|x| 2^u) <= 127}, Abar = ceil(|A| 2^u),
 *       Bbar likewise with v, Wbar = Abar Bbar (exact); R_i = max_j Wbar_ij,
 *       K_j = max_i Wbar_ij (maxima of the bound in the quantised scale),
 *       alpha_i = u_i + max {a : 4^a R_i <= L}, beta_j = v_j + max {b : 4^b K_j <= L}.
 *   O3  A' = trunc(2^alpha A), B' = trunc(B 2^beta), toward zero.
 *   O4  rho_m(x) = ((x + floor(m/2)) mod m) - floor(m/2) for every modulus.
 *   O5  P_t = A_t B_t exactly (64-bit sums).
 *   O6  R_t = P_t mod m_t in [0, m_t).
 *   O7  w_t = R_t (M/m_t)^-1 mod m_t, Y = sum w_t M/m_t mod M,
 *       X = Y - M if 2Y >= M else Y, so X in [-M/2, M/2).
 *   O8  C = RN_even(X 2^-(alpha_i + beta_j)), one correct rounding, with
 *       subnormals and overflow to +-Inf.
 * All integer stages are exact: multiword integers of 32-bit limbs, 64- and
 * 128-bit sums.  The only arrangement beyond the definition is in the
 * integer matrix products, which are evaluated over blocks of rows, columns
 * and inner index for cache reuse and split across threads; integer sums do
 * not depend on their order.
 *
 * It also holds an exact dot product (a fixed-point accumulator spanning
 * every product of two doubles) for the accuracy report: (AB)_ij, (|A||B|)_ij
 * and C_hat_ij - (AB)_ij, each rounded once to double.
 *
 * Entry points (plain C; pointers are host memory; matrices column-major):
 *   int oz2o_moduli(int s, int32_t* out);
 *   int oz2o_exponents(p, q, r, A, lda, B, ldb, s, mode, nthreads,
 *                      alpha, beta);                        O2
 *   int oz2o_residues(p, q, r, A, lda, B, ldb, s, mode, nthreads,
 *                     alpha, beta, Ares, Bres);             O2-O4
 *   int oz2o_products(p, q, r, s, nthreads, Ares, Bres, R);   O5-O6
 *   int oz2o_crt(p, r, s, nthreads, R, alpha, beta, X, C, ldc); O7-O8
 *   int oz2o_dgemm(p, q, r, A, lda, B, ldb, s, mode, nthreads,
 *                  alpha, beta, Ares, Bres, R, X, C, ldc);    all of them
 *   int oz2o_entries(p, q, r, A, lda, B, ldb, s, alpha, beta, n, ii, jj,
 *                    nthreads, R, X, C);            O3-O8 at sampled entries
 *   int oz2o_exact_entries(p, q, r, A, lda, B, ldb, n, ii, jj, nc, Chat,
 *                          exact, absprod, err, nthreads);
 * They return 0, or a negative code for bad arguments (-1), a bound the
 * method needs that does not hold (-2) or an allocation failure (-3).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SMAX 20
#define FBITS 20   /* fractional bits of the fast statistic */
#define QMAX8 127  /* largest upward-quantised bound entry */
#define NW 8       /* 32-bit limbs of a multiword integer: 256 bits */

/* ------------------------------------------------------------------ multiword */
typedef struct {
  uint32_t w[NW];
} big;

static void big_zero(big* a) { memset(a, 0, sizeof(*a)); }

static void big_from_u128(big* a, unsigned __int128 v) {
  big_zero(a);
  for (int k = 0; k < 4; ++k) a->w[k] = (uint32_t)(v >> (32 * k));
}

static void big_mul_u32(big* a, uint32_t m) {
  uint64_t c = 0;
  for (int k = 0; k < NW; ++k) {
    uint64_t t = (uint64_t)a->w[k] * m + c;
    a->w[k] = (uint32_t)t;
    c = t >> 32;
  }
}

/* a <- floor(a / m); returns a mod m */
static uint32_t big_divmod_u32(big* a, uint32_t m) {
  uint64_t rem = 0;
  for (int k = NW - 1; k >= 0; --k) {
    uint64_t cur = (rem << 32) | a->w[k];
    a->w[k] = (uint32_t)(cur / m);
    rem = cur % m;
  }
  return (uint32_t)rem;
}

static int big_cmp(const big* a, const big* b) {
  for (int k = NW - 1; k >= 0; --k)
    if (a->w[k] != b->w[k]) return a->w[k] < b->w[k] ? -1 : 1;
  return 0;
}

static void big_add(big* a, const big* b) {
  uint64_t c = 0;
  for (int k = 0; k < NW; ++k) {
    uint64_t t = (uint64_t)a->w[k] + b->w[k] + c;
    a->w[k] = (uint32_t)t;
    c = t >> 32;
  }
}

/* a <- a - b, for a >= b */
static void big_sub(big* a, const big* b) {
  int64_t c = 0;
  for (int k = 0; k < NW; ++k) {
    int64_t t = (int64_t)a->w[k] - (int64_t)b->w[k] + c;
    a->w[k] = (uint32_t)t;
    c = t < 0 ? -1 : 0;
  }
}

static int big_bitlen(const big* a) {
  for (int k = NW - 1; k >= 0; --k)
    if (a->w[k]) {
      int b = 32;
      while (!((a->w[k] >> (b - 1)) & 1u)) --b;
      return 32 * k + b;
    }
  return 0;
}

static int big_bit(const big* a, int pos) {
  if (pos < 0 || pos >= 32 * NW) return 0;
  return (int)((a->w[pos >> 5] >> (pos & 31)) & 1u);
}

/* a <- a * 2^k, k >= 0 (the caller keeps the result below 2^(32 NW)) */
static void big_shl(big* a, int k) {
  big r;
  big_zero(&r);
  for (int pos = 32 * NW - 1; pos >= k; --pos)
    if (big_bit(a, pos - k)) r.w[pos >> 5] |= 1u << (pos & 31);
  *a = r;
}

static int is_zero(const big* a) {
  for (int k = 0; k < NW; ++k)
    if (a->w[k]) return 0;
  return 1;
}

/* max { h in Z : S 2^h <= L } for S > 0 */
static int max_shift_le(const big* S, const big* L) {
  int k = big_bitlen(L) - big_bitlen(S);
  big a = *S, b = *L;
  if (k >= 0) big_shl(&a, k);
  else big_shl(&b, -k);
  return big_cmp(&a, &b) <= 0 ? k : k - 1;
}

static int floor_div2(int x) { return (x >= 0) ? x / 2 : -((-x + 1) / 2); }

/* ------------------------------------------------------------------ constants */
typedef struct {
  int s;
  int m[SMAX];
  big M, L, Mhalf;
  big Mt[SMAX];       /* M / m_t */
  uint32_t inv[SMAX]; /* (M/m_t)^-1 mod m_t */
} consts;

static int gcd_int(int a, int b) {
  while (b) {
    int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

static int greedy_moduli(int s, int* out) {
  int n = 0;
  for (int m = 256; m >= 2 && n < s; --m) {
    int ok = 1;
    for (int k = 0; k < n; ++k)
      if (gcd_int(m, out[k]) != 1) ok = 0;
    if (ok) out[n++] = m;
  }
  return n;
}

static int make_consts(int s, consts* c) {
  if (s < 1 || s > SMAX) return -1;
  memset(c, 0, sizeof(*c));
  c->s = s;
  if (greedy_moduli(s, c->m) != s) return -1;
  big_zero(&c->M);
  c->M.w[0] = 1;
  for (int t = 0; t < s; ++t) big_mul_u32(&c->M, (uint32_t)c->m[t]);
  c->Mhalf = c->M;
  big_divmod_u32(&c->Mhalf, 2);
  c->L = c->Mhalf;
  {
    big one;
    big_zero(&one);
    one.w[0] = 1;
    big_sub(&c->L, &one);
  }
  for (int t = 0; t < s; ++t) {
    c->Mt[t] = c->M;
    big_divmod_u32(&c->Mt[t], (uint32_t)c->m[t]);
    big tmp = c->Mt[t];
    uint32_t r = big_divmod_u32(&tmp, (uint32_t)c->m[t]);
    uint32_t inv = 0;
    for (uint32_t x = 1; x < (uint32_t)c->m[t]; ++x)
      if (((uint64_t)r * x) % (uint32_t)c->m[t] == 1) {
        inv = x;
        break;
      }
    c->inv[t] = inv;
  }
  return 0;
}

/* ------------------------------------------------------------------ doubles */
/* |x| = mant 2^E exactly, mant < 2^53 (mant = 0 for x = 0) */
static void decompose(double x, int* neg, uint64_t* mant, int* E) {
  uint64_t b;
  memcpy(&b, &x, 8);
  *neg = (int)(b >> 63);
  int eb = (int)((b >> 52) & 0x7FF);
  uint64_t f = b & ((1ull << 52) - 1);
  if (eb == 0) {
    *mant = f;
    *E = -1074;
  } else {
    *mant = f | (1ull << 52);
    *E = eb - 1075;
  }
}

/* e = floor(log2 |x|) + 1 for x != 0, 0 for x == 0 */
static int exp_plus1(double x) {
  int e = 0;
  if (x == 0.0) return 0;
  frexp(x, &e);
  return e;
}

/* ceil(mant 2^sh) for a result known to be below 2^63 */
static uint64_t ceil_shift(uint64_t mant, int sh) {
  if (mant == 0) return 0;
  if (sh >= 0) return mant << sh;
  int d = -sh;
  if (d >= 64) return 1;
  uint64_t q = mant >> d;
  return q + ((mant & ((1ull << d) - 1)) ? 1 : 0);
}

/* |trunc(mant 2^sh)| mod m, for sh of any sign (exact) */
static uint32_t trunc_mod(uint64_t mant, int sh, uint32_t m) {
  if (mant == 0) return 0;
  if (sh <= 0) {
    int d = -sh;
    uint64_t n = (d >= 64) ? 0 : (mant >> d);
    return (uint32_t)(n % m);
  }
  /* mant 2^sh mod m = (mant mod m)(2^sh mod m) mod m */
  uint64_t base = 2 % m, p2 = 1 % m;
  for (int e = sh; e > 0; e >>= 1) {
    if (e & 1) p2 = (p2 * base) % m;
    base = (base * base) % m;
  }
  return (uint32_t)(((mant % m) * p2) % m);
}

static int centered(int64_t x, int m) {
  int64_t h = m / 2;
  int64_t v = (x + h) % m;
  if (v < 0) v += m;
  return (int)(v - h);
}

/* ------------------------------------------------------------------ rounding */
/* RN_even(+-mag 2^e0) for a magnitude given as nd little-endian 32-bit digits */
static double round_digits(const uint32_t* mag, int nd, int e0, int neg) {
  int top = nd - 1;
  while (top >= 0 && mag[top] == 0) --top;
  if (top < 0) return 0.0;
  int nb = 32 * top + 32;
  while (!((mag[top] >> ((nb - 1) & 31)) & 1u)) --nb;
  /* value = mag 2^e0 in [2^E, 2^(E+1)), E = nb - 1 + e0 */
  long E = (long)nb - 1 + e0;
  long keep = (E >= -1022) ? 53 : E + 1075; /* significand bits the format holds there */
  double r;
  if (keep <= 0) {
    /* below 2^-1074: only the value above half of the smallest subnormal rounds up */
    int above_half = 0;
    if (keep == 0) { /* value in [2^-1075, 2^-1074): above half unless exactly 2^-1075 */
      for (int k = 0; k < nd && !above_half; ++k) {
        uint32_t w = mag[k];
        if (k == (nb - 1) / 32) w &= ~(1u << ((nb - 1) & 31));
        if (w) above_half = 1;
      }
    }
    r = above_half ? ldexp(1.0, -1074) : 0.0;
  } else {
    long drop = nb - keep;
    uint64_t sig = 0;
    if (drop <= 0) {
      for (int pos = nb - 1; pos >= 0; --pos) sig = (sig << 1) | ((mag[pos >> 5] >> (pos & 31)) & 1u);
      r = ldexp((double)sig, e0);
    } else {
      for (long pos = nb - 1; pos >= drop; --pos) sig = (sig << 1) | ((mag[pos >> 5] >> (pos & 31)) & 1u);
      int guard = (int)((mag[(drop - 1) >> 5] >> ((drop - 1) & 31)) & 1u);
      int sticky = 0;
      for (long pos = 0; pos < drop - 1 && !sticky; ++pos)
        if ((mag[pos >> 5] >> (pos & 31)) & 1u) sticky = 1;
      if (guard && (sticky || (sig & 1u))) sig += 1;
      /* sig <= 2^keep <= 2^53: exact in double; the scaling is exact or overflows to inf */
      r = ldexp((double)sig, (int)(drop + e0));
    }
  }
  return neg ? -r : r;
}

/* ------------------------------------------------------------------ threads */
typedef void (*task_fn)(void* ctx, int64_t task);
typedef struct {
  task_fn fn;
  void* ctx;
  int64_t ntask;
  int64_t next;
  pthread_mutex_t mu;
} pool;

static void* pool_worker(void* arg) {
  pool* P = (pool*)arg;
  for (;;) {
    pthread_mutex_lock(&P->mu);
    int64_t t = P->next++;
    pthread_mutex_unlock(&P->mu);
    if (t >= P->ntask) break;
    P->fn(P->ctx, t);
  }
  return NULL;
}

static void run_tasks(task_fn fn, void* ctx, int64_t ntask, int nthreads) {
  pool P;
  P.fn = fn;
  P.ctx = ctx;
  P.ntask = ntask;
  P.next = 0;
  pthread_mutex_init(&P.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int k = 1; k < nthreads; ++k)
    if (pthread_create(&th[started], NULL, pool_worker, &P) == 0) ++started;
  pool_worker(&P);
  for (int k = 0; k < started; ++k) pthread_join(th[k], NULL);
  pthread_mutex_destroy(&P.mu);
}

/* ------------------------------------------------------------------ exponents */
typedef struct {
  int64_t p, q, r, lda, ldb;
  const double* A;
  const double* B;
  const consts* c;
  int32_t* alpha;
  int32_t* beta;
  /* accu */
  int32_t* u;
  int32_t* v;
  uint8_t* Abar; /* [p][q] */
  uint8_t* Bbar; /* [r][q] */
  int32_t* W;    /* [r][p]: Wbar column-major */
} expctx;

/* element l of vector k: a row of A (side 0) or a column of B (side 1) */
static double vec_elem(const expctx* x, int side, int64_t k, int64_t l) {
  return side == 0 ? x->A[l * x->lda + k] : x->B[k * x->ldb + l];
}

/* fast bound ([P] §2, §5.1) for one vector */
static int32_t fast_exponent(const expctx* x, int side, int64_t k) {
  double amax = 0.0;
  for (int64_t l = 0; l < x->q; ++l) {
    double a = fabs(vec_elem(x, side, k, l));
    if (a > amax) amax = a;
  }
  if (amax == 0.0) return 0;
  int e = exp_plus1(amax);
  unsigned __int128 S = 0;
  for (int64_t l = 0; l < x->q; ++l) {
    int neg, E;
    uint64_t mant;
    decompose(vec_elem(x, side, k, l), &neg, &mant, &E);
    uint64_t t = ceil_shift(mant, E + FBITS - e); /* ceil(|x| 2^(F - e)) <= 2^F */
    S += (unsigned __int128)(t * t);
  }
  if (S == 0) return 0;
  big Sb;
  big_from_u128(&Sb, S);
  /* 4^a S 4^(e - F) <= L  <=>  S 2^(2a + 2e - 2F) <= L  <=>  2a <= h - 2e + 2F */
  int h = max_shift_le(&Sb, &x->c->L);
  return floor_div2(h - 2 * e + 2 * FBITS);
}

static void fast_task(void* ctx, int64_t task) {
  expctx* x = (expctx*)ctx;
  if (task < x->p) x->alpha[task] = fast_exponent(x, 0, task);
  else x->beta[task - x->p] = fast_exponent(x, 1, task - x->p);
}

/* u = max {u : ceil(amax 2^u) <= 127}, 0 for a zero vector */
static int32_t quant_exponent(double amax) {
  if (amax == 0.0) return 0;
  int neg, E;
  uint64_t mant;
  decompose(amax, &neg, &mant, &E);
  int u = 6 - exp_plus1(amax); /* amax 2^u in [32, 64) */
  while (ceil_shift(mant, E + u + 1) <= QMAX8) ++u;
  while (ceil_shift(mant, E + u) > QMAX8) --u;
  return u;
}

static void bound_quant_task(void* ctx, int64_t task) {
  expctx* x = (expctx*)ctx;
  int side = task < x->p ? 0 : 1;
  int64_t k = side == 0 ? task : task - x->p;
  double amax = 0.0;
  for (int64_t l = 0; l < x->q; ++l) {
    double a = fabs(vec_elem(x, side, k, l));
    if (a > amax) amax = a;
  }
  int32_t u = quant_exponent(amax);
  uint8_t* out = side == 0 ? x->Abar + k * x->q : x->Bbar + k * x->q;
  for (int64_t l = 0; l < x->q; ++l) {
    int neg, E;
    uint64_t mant;
    decompose(vec_elem(x, side, k, l), &neg, &mant, &E);
    out[l] = (uint8_t)ceil_shift(mant, E + u);
  }
  if (side == 0) x->u[k] = u;
  else x->v[k] = u;
}

/* max {a : 4^a w <= L} for an integer w > 0 (0 for w == 0) */
static int32_t pow4_exponent_of(const consts* c, int64_t w) {
  /* 4^a w <= L  <=>  w 2^(2a) <= L  <=>  2a <= h */
  if (w == 0) return 0;
  big Wb;
  big_from_u128(&Wb, (unsigned __int128)w);
  return floor_div2(max_shift_le(&Wb, &c->L));
}

/* alpha_i = u_i + max {a : 4^a R_i <= L} with R_i = max_j Wbar_ij, the row
 * maximum of the bound product in the quantised scale; beta_j likewise with
 * v_j and K_j = max_i Wbar_ij.  0 for a zero row or column of Wbar. */
static void accu_exp_task(void* ctx, int64_t task) {
  expctx* x = (expctx*)ctx;
  if (task < x->p) {
    int64_t i = task, R = 0;
    for (int64_t j = 0; j < x->r; ++j)
      if (x->W[j * x->p + i] > R) R = x->W[j * x->p + i];
    x->alpha[i] = R ? x->u[i] + pow4_exponent_of(x->c, R) : 0;
  } else {
    int64_t j = task - x->p, K = 0;
    for (int64_t i = 0; i < x->p; ++i)
      if (x->W[j * x->p + i] > K) K = x->W[j * x->p + i];
    x->beta[j] = K ? x->v[j] + pow4_exponent_of(x->c, K) : 0;
  }
}

/* ------------------------------------------------------------------ integer products */
/*
 * out[j * p + i] = sum_l a[i * q + l] b[j * q + l] for int8 (or uint8 when
 * is_unsigned) rows: an exact integer matrix product, evaluated over blocks
 * for cache reuse.  Sums are 64-bit; each inner chunk of KC terms stays below
 * 2^31 in 32 bits (KC 2^16 <= 2^31 for |a b| <= 2^16).
 */
#define KC 4096
#define BI 64
#define BJ 64
typedef struct {
  int64_t p, q, r;
  const int8_t* a;
  const int8_t* b;
  int64_t* out; /* [r][p] */
} mmctx;

static void mm_task(void* ctx, int64_t task) {
  mmctx* x = (mmctx*)ctx;
  int64_t nbi = (x->p + BI - 1) / BI;
  int64_t i0 = (task % nbi) * BI, j0 = (task / nbi) * BJ;
  int64_t i1 = i0 + BI < x->p ? i0 + BI : x->p;
  int64_t j1 = j0 + BJ < x->r ? j0 + BJ : x->r;
  for (int64_t j = j0; j < j1; ++j)
    for (int64_t i = i0; i < i1; ++i) x->out[j * x->p + i] = 0;
  for (int64_t l0 = 0; l0 < x->q; l0 += KC) {
    int64_t n = x->q - l0 < KC ? x->q - l0 : KC;
    for (int64_t j = j0; j < j1; ++j) {
      const int8_t* bj = x->b + j * x->q + l0;
      for (int64_t i = i0; i < i1; ++i) {
        const int8_t* ai = x->a + i * x->q + l0;
        int32_t s = 0;
        for (int64_t l = 0; l < n; ++l) s += (int32_t)ai[l] * (int32_t)bj[l];
        x->out[j * x->p + i] += s;
      }
    }
  }
}

typedef struct {
  int64_t p, q, r;
  const uint8_t* a;
  const uint8_t* b;
  int32_t* out; /* [r][p] */
} bmmctx;

static void bmm_task(void* ctx, int64_t task) {
  bmmctx* x = (bmmctx*)ctx;
  int64_t nbi = (x->p + BI - 1) / BI;
  int64_t i0 = (task % nbi) * BI, j0 = (task / nbi) * BJ;
  int64_t i1 = i0 + BI < x->p ? i0 + BI : x->p;
  int64_t j1 = j0 + BJ < x->r ? j0 + BJ : x->r;
  for (int64_t j = j0; j < j1; ++j)
    for (int64_t i = i0; i < i1; ++i) {
      const uint8_t* ai = x->a + i * x->q;
      const uint8_t* bj = x->b + j * x->q;
      uint32_t s = 0; /* q 127^2 < 2^31: exact */
      for (int64_t l = 0; l < x->q; ++l) s += (uint32_t)ai[l] * (uint32_t)bj[l];
      x->out[j * x->p + i] = (int32_t)s;
    }
}

/* ------------------------------------------------------------------ residues */
typedef struct {
  int64_t p, q, r, lda, ldb;
  const double* A;
  const double* B;
  const consts* c;
  const int32_t* alpha;
  const int32_t* beta;
  int8_t* Ares; /* [s][p][q] */
  int8_t* Bres; /* [s][r][q] */
} resctx;

static void res_task(void* ctx, int64_t task) {
  resctx* x = (resctx*)ctx;
  int side = task < x->p ? 0 : 1;
  int64_t k = side == 0 ? task : task - x->p;
  int32_t ex = side == 0 ? x->alpha[k] : x->beta[k];
  int64_t nvec = side == 0 ? x->p : x->r;
  int8_t* planes = side == 0 ? x->Ares : x->Bres;
  for (int64_t l = 0; l < x->q; ++l) {
    double a = side == 0 ? x->A[l * x->lda + k] : x->B[k * x->ldb + l];
    int neg, E;
    uint64_t mant;
    decompose(a, &neg, &mant, &E);
    for (int t = 0; t < x->c->s; ++t) {
      uint32_t m = (uint32_t)x->c->m[t];
      int64_t n = (int64_t)trunc_mod(mant, E + ex, m); /* |trunc(2^ex a)| mod m */
      planes[((int64_t)t * nvec + k) * x->q + l] = (int8_t)centered(neg ? -n : n, (int)m);
    }
  }
}

/* ------------------------------------------------------------------ CRT + rounding */
typedef struct {
  int64_t p, r, ldc;
  const consts* c;
  const uint8_t* R; /* [s][r][p] */
  const int32_t* alpha;
  const int32_t* beta;
  uint64_t* X; /* [r][p][3] or NULL */
  double* C;   /* column-major, ldc, or NULL */
} crtctx;

static void crt_task(void* ctx, int64_t j) {
  crtctx* x = (crtctx*)ctx;
  const consts* c = x->c;
  for (int64_t i = 0; i < x->p; ++i) {
    big Y;
    big_zero(&Y);
    for (int t = 0; t < c->s; ++t) {
      uint32_t Rt = x->R[((int64_t)t * x->r + j) * x->p + i];
      uint32_t w = (uint32_t)(((uint64_t)Rt * c->inv[t]) % (uint32_t)c->m[t]);
      big term = c->Mt[t];
      big_mul_u32(&term, w);
      big_add(&Y, &term);
    }
    while (big_cmp(&Y, &c->M) >= 0) big_sub(&Y, &c->M); /* Y mod M */
    int neg = big_cmp(&Y, &c->Mhalf) >= 0;            /* 2Y >= M */
    big mag = Y;
    if (neg) { /* |X| = M - Y */
      mag = c->M;
      big_sub(&mag, &Y);
    }
    if (x->X) {
      /* 192-bit two's complement, little-endian 64-bit limbs */
      uint32_t tw[6];
      for (int k = 0; k < 6; ++k) tw[k] = mag.w[k];
      if (neg) {
        uint64_t cy = 1;
        for (int k = 0; k < 6; ++k) {
          uint64_t t = (uint64_t)(uint32_t)~tw[k] + cy;
          tw[k] = (uint32_t)t;
          cy = t >> 32;
        }
      }
      uint64_t* o = x->X + (j * x->p + i) * 3;
      for (int k = 0; k < 3; ++k) o[k] = (uint64_t)tw[2 * k] | ((uint64_t)tw[2 * k + 1] << 32);
    }
    if (x->C) {
      int k = x->alpha[i] + x->beta[j];
      x->C[j * x->ldc + i] = is_zero(&mag) ? 0.0 : round_digits(mag.w, NW, -k, neg);
    }
  }
}

/* ------------------------------------------------------------------ products -> R */
typedef struct {
  int64_t p, q, r;
  int t, m;
  const int8_t* a;
  const int8_t* b;
  int64_t* P; /* [r][p] scratch */
  uint8_t* R; /* plane t of [s][r][p] */
} rctx;

static void r_task(void* ctx, int64_t j) {
  rctx* x = (rctx*)ctx;
  for (int64_t i = 0; i < x->p; ++i) {
    int64_t v = x->P[j * x->p + i] % x->m;
    if (v < 0) v += x->m;
    x->R[j * x->p + i] = (uint8_t)v;
  }
}

/* ------------------------------------------------------------------ entry points */
int oz2o_moduli(int s, int32_t* out) {
  int m[SMAX];
  if (s < 1 || s > SMAX || !out) return -1;
  if (greedy_moduli(s, m) != s) return -1;
  for (int t = 0; t < s; ++t) out[t] = m[t];
  return s;
}

/* O2: the exponents alpha [p], beta [r] */
int oz2o_exponents(int64_t p, int64_t q, int64_t r, const double* A, int64_t lda, const double* B, int64_t ldb,
                   int s, int mode, int nthreads, int32_t* alpha, int32_t* beta) {
  if (p <= 0 || q <= 0 || r <= 0 || lda < p || ldb < q || !A || !B || !alpha || !beta) return -1;
  if (mode != 0 && mode != 1) return -1;
  if (mode == 0 && q >= (1 << 24)) return -2;                        /* the exact statistic: q 2^40 < 2^64 */
  if (mode == 1 && (int64_t)q * 127 * 127 >= (1ll << 31)) return -2; /* Wbar in INT32 */
  consts c;
  if (make_consts(s, &c) != 0) return -1;
  expctx ex = {p, q, r, lda, ldb, A, B, &c, alpha, beta, NULL, NULL, NULL, NULL, NULL};
  if (mode == 0) {
    run_tasks(fast_task, &ex, p + r, nthreads);
    return 0;
  }
  int rc = 0;
  ex.u = (int32_t*)malloc(sizeof(int32_t) * p);
  ex.v = (int32_t*)malloc(sizeof(int32_t) * r);
  ex.Abar = (uint8_t*)malloc((size_t)p * q);
  ex.Bbar = (uint8_t*)malloc((size_t)r * q);
  ex.W = (int32_t*)malloc(sizeof(int32_t) * p * r);
  if (ex.u && ex.v && ex.Abar && ex.Bbar && ex.W) {
    run_tasks(bound_quant_task, &ex, p + r, nthreads);
    bmmctx bm = {p, q, r, ex.Abar, ex.Bbar, ex.W};
    run_tasks(bmm_task, &bm, ((p + BI - 1) / BI) * ((r + BJ - 1) / BJ), nthreads);
    run_tasks(accu_exp_task, &ex, p + r, nthreads);
  } else {
    rc = -3;
  }
  free(ex.u);
  free(ex.v);
  free(ex.Abar);
  free(ex.Bbar);
  free(ex.W);
  return rc;
}

/* O2-O4: exponents and residue planes (all four outputs required) */
int oz2o_residues(int64_t p, int64_t q, int64_t r, const double* A, int64_t lda, const double* B, int64_t ldb,
                  int s, int mode, int nthreads, int32_t* alpha, int32_t* beta, int8_t* Ares, int8_t* Bres) {
  if (!Ares || !Bres) return -1;
  int rc = oz2o_exponents(p, q, r, A, lda, B, ldb, s, mode, nthreads, alpha, beta);
  if (rc != 0) return rc;
  consts c;
  make_consts(s, &c);
  resctx rs = {p, q, r, lda, ldb, A, B, &c, alpha, beta, Ares, Bres};
  run_tasks(res_task, &rs, p + r, nthreads);
  return 0;
}

/* O5/O6: R_t = (A_t B_t) mod m_t for every channel, from the residue planes */
int oz2o_products(int64_t p, int64_t q, int64_t r, int s, int nthreads, const int8_t* Ares, const int8_t* Bres,
                  uint8_t* R) {
  if (p <= 0 || q <= 0 || r <= 0 || !Ares || !Bres || !R) return -1;
  consts c;
  if (make_consts(s, &c) != 0) return -1;
  int64_t* P = (int64_t*)malloc(sizeof(int64_t) * p * r);
  if (!P) return -3;
  for (int t = 0; t < s; ++t) {
    mmctx mm = {p, q, r, Ares + (int64_t)t * p * q, Bres + (int64_t)t * r * q, P};
    run_tasks(mm_task, &mm, ((p + BI - 1) / BI) * ((r + BJ - 1) / BJ), nthreads);
    rctx rr = {p, q, r, t, c.m[t], NULL, NULL, P, R + (int64_t)t * p * r};
    run_tasks(r_task, &rr, r, nthreads);
  }
  free(P);
  return 0;
}

/* O7/O8: X and C from the output residues R [s][r][p] (either output may be NULL) */
int oz2o_crt(int64_t p, int64_t r, int s, int nthreads, const uint8_t* R, const int32_t* alpha,
             const int32_t* beta, uint64_t* X, double* C, int64_t ldc) {
  if (p <= 0 || r <= 0 || !R || !alpha || !beta) return -1;
  if (C && ldc < p) return -1;
  consts c;
  if (make_consts(s, &c) != 0) return -1;
  crtctx cc = {p, r, ldc, &c, R, alpha, beta, X, C};
  if (X || C) run_tasks(crt_task, &cc, r, nthreads);
  return 0;
}

/* every stage in C; any output may be NULL */
int oz2o_dgemm(int64_t p, int64_t q, int64_t r, const double* A, int64_t lda, const double* B, int64_t ldb,
               int s, int mode, int nthreads, int32_t* alpha_out, int32_t* beta_out, int8_t* Ares_out,
               int8_t* Bres_out, uint8_t* R_out, uint64_t* X_out, double* C_out, int64_t ldc) {
  if (p <= 0 || q <= 0 || r <= 0 || lda < p || ldb < q || !A || !B) return -1;
  if (C_out && ldc < p) return -1;
  int rc = -3;
  int32_t* alpha = alpha_out ? alpha_out : (int32_t*)malloc(sizeof(int32_t) * p);
  int32_t* beta = beta_out ? beta_out : (int32_t*)malloc(sizeof(int32_t) * r);
  int8_t* Ares = Ares_out ? Ares_out : (int8_t*)malloc((size_t)s * p * q);
  int8_t* Bres = Bres_out ? Bres_out : (int8_t*)malloc((size_t)s * r * q);
  uint8_t* R = R_out ? R_out : (uint8_t*)malloc((size_t)s * p * r);
  if (alpha && beta && Ares && Bres && R) {
    rc = oz2o_residues(p, q, r, A, lda, B, ldb, s, mode, nthreads, alpha, beta, Ares, Bres);
    if (rc == 0) rc = oz2o_products(p, q, r, s, nthreads, Ares, Bres, R);
    if (rc == 0) rc = oz2o_crt(p, r, s, nthreads, R, alpha, beta, X_out, C_out, ldc);
  }
  if (!alpha_out) free(alpha);
  if (!beta_out) free(beta);
  if (!Ares_out) free(Ares);
  if (!Bres_out) free(Bres);
  if (!R_out) free(R);
  return rc;
}

/* O3-O8 at sampled outputs (ii[k], jj[k]) only, given the exponents: the
 * residues of row i of A and column j of B are formed on the fly, then
 * P_t = sum_l rho(a'_il) rho(b'_lj), R_t, X and C as above.  Outputs:
 * R [n][s] (may be NULL), X [n][3], C [n]. */
typedef struct {
  int64_t q, lda, ldb;
  const double* A;
  const double* B;
  const consts* c;
  const int32_t* alpha;
  const int32_t* beta;
  const int64_t* ii;
  const int64_t* jj;
  uint8_t* R;
  uint64_t* X;
  double* C;
} entctx;

static void entry_task(void* ctx, int64_t k) {
  entctx* x = (entctx*)ctx;
  const consts* c = x->c;
  int64_t i = x->ii[k], j = x->jj[k];
  int64_t P[SMAX] = {0};
  for (int64_t l = 0; l < x->q; ++l) {
    int na, nb, Ea, Eb;
    uint64_t ma, mb;
    decompose(x->A[l * x->lda + i], &na, &ma, &Ea);
    decompose(x->B[j * x->ldb + l], &nb, &mb, &Eb);
    for (int t = 0; t < c->s; ++t) {
      uint32_t m = (uint32_t)c->m[t];
      int64_t ra = (int64_t)trunc_mod(ma, Ea + x->alpha[i], m);
      int64_t rb = (int64_t)trunc_mod(mb, Eb + x->beta[j], m);
      P[t] += (int64_t)centered(na ? -ra : ra, (int)m) * centered(nb ? -rb : rb, (int)m);
    }
  }
  uint8_t Rk[SMAX];
  for (int t = 0; t < c->s; ++t) {
    int64_t v = P[t] % c->m[t];
    Rk[t] = (uint8_t)(v < 0 ? v + c->m[t] : v);
    if (x->R) x->R[k * c->s + t] = Rk[t];
  }
  /* the CRT of one entry: the same steps as crt_task on a one-entry R */
  crtctx one = {1, 1, 1, c, Rk, x->alpha + i, x->beta + j, x->X + k * 3, x->C + k};
  crt_task(&one, 0);
}

int oz2o_entries(int64_t p, int64_t q, int64_t r, const double* A, int64_t lda, const double* B, int64_t ldb,
                 int s, const int32_t* alpha, const int32_t* beta, int64_t n, const int64_t* ii,
                 const int64_t* jj, int nthreads, uint8_t* R, uint64_t* X, double* C) {
  if (p <= 0 || q <= 0 || r <= 0 || lda < p || ldb < q || !A || !B || !alpha || !beta) return -1;
  if (n < 0 || (n > 0 && (!ii || !jj || !X || !C))) return -1;
  for (int64_t k = 0; k < n; ++k)
    if (ii[k] < 0 || ii[k] >= p || jj[k] < 0 || jj[k] >= r) return -1;
  consts c;
  if (make_consts(s, &c) != 0) return -1;
  entctx e = {q, lda, ldb, A, B, &c, alpha, beta, ii, jj, R, X, C};
  run_tasks(entry_task, &e, n, nthreads);
  return 0;
}

/* ------------------------------------------------------------------ exact dot products */
/*
 * Fixed-point accumulator: digit k has weight 2^(KBASE + 32 k).  Every
 * product of two doubles is m 2^e with m < 2^106 and e >= -2148, and below
 * 2^2048; a sum of up to 2^24 of them stays below 2^2072.  Digits hold
 * signed 64-bit partial sums of 32-bit pieces, so no carry is needed until
 * the end.
 */
#define KBASE (-2208)
#define KDIG 142

typedef struct {
  int64_t d[KDIG];
} kacc;

static void kacc_add_piece(kacc* a, int pos, unsigned __int128 v, int neg) {
  /* add +-v 2^(KBASE + pos) */
  int dg = pos >> 5, off = pos & 31;
  uint64_t lo = (uint64_t)v, hi = (uint64_t)(v >> 64);
  unsigned __int128 l2 = (unsigned __int128)lo << off; /* < 2^96 */
  unsigned __int128 h2 = (unsigned __int128)hi << off; /* < 2^(64 - 22 + 31) */
  int64_t sg = neg ? -1 : 1;
  a->d[dg] += sg * (int64_t)(uint32_t)l2;
  a->d[dg + 1] += sg * (int64_t)(uint32_t)(l2 >> 32);
  a->d[dg + 2] += sg * (int64_t)(uint32_t)(l2 >> 64);
  a->d[dg + 2] += sg * (int64_t)(uint32_t)h2;
  a->d[dg + 3] += sg * (int64_t)(uint32_t)(h2 >> 32);
  a->d[dg + 4] += sg * (int64_t)(uint32_t)(h2 >> 64);
}

static void kacc_add_prod(kacc* a, double x, double y, int absval) {
  int nx, ny, ex, ey;
  uint64_t mx, my;
  decompose(x, &nx, &mx, &ex);
  decompose(y, &ny, &my, &ey);
  if (mx == 0 || my == 0) return;
  kacc_add_piece(a, ex + ey - KBASE, (unsigned __int128)mx * my, absval ? 0 : (nx ^ ny));
}

static void kacc_add_double(kacc* a, double x) {
  int n, e;
  uint64_t m;
  decompose(x, &n, &m, &e);
  if (m == 0) return;
  kacc_add_piece(a, e - KBASE, (unsigned __int128)m, n);
}

static double kacc_round(const kacc* a) {
  int64_t d[KDIG];
  memcpy(d, a->d, sizeof(d));
  for (int k = 0; k < KDIG - 1; ++k) { /* carries: digits into [0, 2^32) */
    int64_t cy = d[k] >> 32;             /* arithmetic: floor division */
    d[k] -= cy * ((int64_t)1 << 32);
    d[k + 1] += cy;
  }
  int neg = d[KDIG - 1] < 0;
  uint32_t mag[KDIG];
  if (neg) { /* magnitude = -(value): two's complement in base 2^32 */
    int64_t cy = 1;
    for (int k = 0; k < KDIG; ++k) {
      int64_t t = (int64_t)(uint32_t)~(uint32_t)d[k] + cy;
      mag[k] = (uint32_t)t;
      cy = t >> 32;
    }
  } else {
    for (int k = 0; k < KDIG; ++k) mag[k] = (uint32_t)d[k];
  }
  return round_digits(mag, KDIG, KBASE, neg);
}

typedef struct {
  int64_t p, q, r, lda, ldb;
  const double* A;
  const double* B;
  const int64_t* ii;
  const int64_t* jj;
  int64_t n;
  int nc;
  const double* Chat; /* [nc][n] */
  double* exact;      /* [n] */
  double* absprod;    /* [n] */
  double* err;        /* [nc][n] */
} exctx;

static void exact_task(void* ctx, int64_t k) {
  exctx* x = (exctx*)ctx;
  int64_t i = x->ii[k], j = x->jj[k];
  kacc acc, aab;
  memset(&acc, 0, sizeof(acc));
  memset(&aab, 0, sizeof(aab));
  for (int64_t l = 0; l < x->q; ++l) {
    double a = x->A[l * x->lda + i], b = x->B[j * x->ldb + l];
    kacc_add_prod(&acc, a, b, 0);
    kacc_add_prod(&aab, a, b, 1);
  }
  x->exact[k] = kacc_round(&acc);
  x->absprod[k] = kacc_round(&aab);
  for (int c = 0; c < x->nc; ++c) {
    kacc d = acc; /* C_hat - AB, exactly, then one rounding */
    for (int m = 0; m < KDIG; ++m) d.d[m] = -d.d[m];
    kacc_add_double(&d, x->Chat[(int64_t)c * x->n + k]);
    x->err[(int64_t)c * x->n + k] = kacc_round(&d);
  }
}

int oz2o_exact_entries(int64_t p, int64_t q, int64_t r, const double* A, int64_t lda, const double* B,
                       int64_t ldb, int64_t n, const int64_t* ii, const int64_t* jj, int nc,
                       const double* Chat, double* exact, double* absprod, double* err, int nthreads) {
  if (p <= 0 || q <= 0 || r <= 0 || lda < p || ldb < q || !A || !B || n < 0) return -1;
  if (q >= (1 << 24)) return -2;
  if (n && (!ii || !jj || !exact || !absprod)) return -1;
  if (nc < 0 || (nc > 0 && (!Chat || !err))) return -1;
  for (int64_t k = 0; k < n; ++k)
    if (ii[k] < 0 || ii[k] >= p || jj[k] < 0 || jj[k] >= r) return -1;
  exctx x = {p, q, r, lda, ldb, A, B, ii, jj, n, nc, Chat, exact, absprod, err};
  run_tasks(exact_task, &x, n, nthreads);
  return 0;
}
