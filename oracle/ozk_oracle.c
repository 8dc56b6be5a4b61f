/*
 * CPU oracle for Ozaki-scheme-II FP64 GEMM emulation.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the library.  Shares no code with the
 * CUDA path.  Plain and slow on purpose: every output is computed by the
 * method's steps in the order the Ozaki-II "Day 12" page (ithelp.ithome.com.tw,
 * section "Profile 不能只看 Tensor Core") lists them, with no blocking, fusion
 * or reordering of the arithmetic.  OpenMP only splits independent outputs.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off (no FMA contraction: the Dot2
 * reference depends on separately rounded products and sums).
 */
#include "ozk_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Moduli, in the order the method consumes them (reading R1: the first n of
 * this pairwise-coprime list of integers <= 256). */
static const int32_t MODULI[OZK_REF_NMAX] = {256, 255, 253, 251, 247, 241, 239,
                                             233, 229, 227, 223, 217, 211, 199,
                                             197, 193, 191, 181, 179, 173};

/* ------------------------------------------------------------------------- */
/* Signed wide integers: OZK_REF_LIMBS little-endian 32-bit limbs, two's      */
/* complement.  256 bits hold every value the method produces (|X| < 2^161).  */
/* ------------------------------------------------------------------------- */
#define L OZK_REF_LIMBS
typedef struct {
  uint32_t w[L];
} bigi;

static void big_set_u32(bigi* x, uint32_t v) {
  memset(x, 0, sizeof *x);
  x->w[0] = v;
}

static int big_is_negative(const bigi* x) { return (x->w[L - 1] >> 31) != 0; }

static void big_add(bigi* r, const bigi* a, const bigi* b) {
  uint64_t c = 0;
  for (int l = 0; l < L; ++l) {
    c += (uint64_t)a->w[l] + (uint64_t)b->w[l];
    r->w[l] = (uint32_t)c;
    c >>= 32;
  }
}

static void big_negate(bigi* r, const bigi* a) {
  uint64_t c = 1;
  for (int l = 0; l < L; ++l) {
    c += (uint64_t)(uint32_t)~a->w[l];
    r->w[l] = (uint32_t)c;
    c >>= 32;
  }
}

static void big_sub(bigi* r, const bigi* a, const bigi* b) {
  bigi nb;
  big_negate(&nb, b);
  big_add(r, a, &nb);
}

/* r = a * m + add, for non-negative a. */
static void big_muladd_u32(bigi* r, const bigi* a, uint32_t m, uint32_t add) {
  uint64_t c = add;
  for (int l = 0; l < L; ++l) {
    c += (uint64_t)a->w[l] * m;
    r->w[l] = (uint32_t)c;
    c >>= 32;
  }
}

/* Signed comparison: -1, 0, +1.  Values stay far below 2^255, so a - b
 * cannot wrap. */
static int big_cmp(const bigi* a, const bigi* b) {
  bigi d;
  big_sub(&d, a, b);
  if (big_is_negative(&d)) return -1;
  for (int l = 0; l < L; ++l)
    if (d.w[l]) return 1;
  return 0;
}

/* Position of the highest set bit of a non-negative value, -1 for zero. */
static int big_msb(const bigi* a) {
  for (int l = L - 1; l >= 0; --l)
    if (a->w[l]) return 32 * l + 31 - __builtin_clz(a->w[l]);
  return -1;
}

static int big_bit(const bigi* a, int64_t pos) {
  if (pos < 0 || pos >= 32 * L) return 0;
  return (int)((a->w[pos >> 5] >> (pos & 31)) & 1u);
}

/* Product of two signed integers below 2^127 in magnitude. */
static void big_mul_i128(bigi* r, __int128 a, __int128 b) {
  int neg = (a < 0) != (b < 0);
  unsigned __int128 ua = a < 0 ? -(unsigned __int128)a : (unsigned __int128)a;
  unsigned __int128 ub = b < 0 ? -(unsigned __int128)b : (unsigned __int128)b;
  uint32_t la[4], lb[4], res[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int l = 0; l < 4; ++l) {
    la[l] = (uint32_t)(ua >> (32 * l));
    lb[l] = (uint32_t)(ub >> (32 * l));
  }
  for (int i = 0; i < 4; ++i) {
    uint64_t carry = 0;
    for (int j = 0; j < 4; ++j) {
      uint64_t t = (uint64_t)la[i] * lb[j] + res[i + j] + carry;
      res[i + j] = (uint32_t)t;
      carry = t >> 32;
    }
    res[i + 4] = (uint32_t)carry;
  }
  bigi m;
  for (int l = 0; l < L; ++l) m.w[l] = l < 8 ? res[l] : 0u;
  if (neg)
    big_negate(r, &m);
  else
    *r = m;
}

static void big_product_of_moduli(bigi* P, int n) {
  big_set_u32(P, 1);
  for (int k = 0; k < n; ++k) big_muladd_u32(P, P, (uint32_t)MODULI[k], 0);
}

/* ------------------------------------------------------------------------- */
/* Step 0: the moduli and the bit budget                                     */
/* ------------------------------------------------------------------------- */
int ozk_ref_moduli(int n, int32_t* out) {
  if (n < 1 || n > OZK_REF_NMAX || !out) return OZK_REF_EINVAL;
  for (int k = 0; k < n; ++k) out[k] = MODULI[k];
  return OZK_REF_OK;
}

static int ceil_log2_i64(int64_t K) {
  int c = 0;
  while (c < 62 && ((int64_t)1 << c) < K) ++c;
  return c;
}

/* Reading R2: |a'|, |b'| <= 2^beta gives |sum_k a'b'| <= K 2^(2 beta); choosing
 * 2 beta <= floor(log2 P) - 1 - ceil(log2 K) makes that at most
 * 2^floor(log2 P) / 2 < P/2 (P is never a power of two), so the symmetric
 * CRT lift recovers the product exactly. */
int ozk_ref_beta(int64_t K, int n) {
  if (n < 2 || n > OZK_REF_NMAX) return OZK_REF_EUNSUPPORTED;
  if (K < 1) K = 1;
  bigi P;
  big_product_of_moduli(&P, n);
  int num = big_msb(&P) - 1 - ceil_log2_i64(K);
  int beta = num >= 0 ? num / 2 : -((-num + 1) / 2);
  return beta >= 1 ? beta : OZK_REF_EUNSUPPORTED;
}

/* ------------------------------------------------------------------------- */
/* Step 1: exponent scan ("scale / exponent scan")                           */
/* ------------------------------------------------------------------------- */
static int32_t scale_of(const double* x, int64_t len, int64_t stride, int beta) {
  double amax = 0.0;
  for (int64_t k = 0; k < len; ++k) {
    double v = x[k * stride];
    if (!isfinite(v)) return OZK_REF_NONFINITE;
    if (fabs(v) > amax) amax = fabs(v);
  }
  if (amax == 0.0) return 0;
  int E;
  (void)frexp(amax, &E); /* amax = f * 2^E, f in [0.5, 1) */
  return beta - E;
}

int ozk_ref_scale(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                  const double* B, int64_t ldb, int n, int32_t* s, int32_t* t) {
  if (M < 0 || N < 0 || K < 0) return OZK_REF_EINVAL;
  int beta = ozk_ref_beta(K, n);
  if (beta < 0) return beta;
  for (int64_t i = 0; i < M; ++i) s[i] = scale_of(A + i * lda, K, 1, beta);
  for (int64_t j = 0; j < N; ++j) t[j] = scale_of(B + j, K, ldb, beta);
  return OZK_REF_OK;
}

/* ------------------------------------------------------------------------- */
/* Step 1, sharper: scaling from a computed norm bound (reading R15).        */
/* By Cauchy-Schwarz, sum_k |a'_ik||b'_kj| <= ||a'_i||_2 ||b'_j||_2, so it is */
/* enough that every scaled row of A and column of B has 2-norm at most      */
/* 2^gamma (plus the rounding slack), instead of every entry being below     */
/* 2^beta with K entries at the bound.  The norm bound is computed exactly   */
/* (integers only, so any summation order gives the same scales):           */
/*   h(x) = floor(2 log2 |x|), so x^2 < 2^(h(x) + 1);                        */
/*   H = max h over the row, W = OZK_REF_NORM_WINDOW;                        */
/*   S = sum over the nonzero entries of 2^max(h - H + W, 0), an integer;    */
/*   then ||x||^2 < S 2^(H + 1 - W), and                                     */
/*   s = floor((2 gamma - (H + 1 - W) - ceil(log2 S)) / 2)                   */
/* keeps 2^(2s) S 2^(H + 1 - W) <= 2^(2 gamma).                              */
/* ------------------------------------------------------------------------- */

/* gamma = floor((floor(log2 P) - 2) / 2), usable when sqrt(K) <= 2^(gamma - 2):
 * then |a'_ik| <= 2^s |a_ik| + 1/2 gives ||a'_i|| <= 2^gamma + sqrt(K)/2
 * <= 2^gamma (1 + 1/8), and 2 ||a'_i|| ||b'_j|| <= 2 (81/64) 2^(2 gamma)
 * <= (81/128) 2^floor(log2 P) < P: the symmetric lift stays exact. */
int ozk_ref_gamma(int64_t K, int n) {
  if (n < 2 || n > OZK_REF_NMAX) return OZK_REF_EUNSUPPORTED;
  if (K < 1) K = 1;
  bigi P;
  big_product_of_moduli(&P, n);
  int gamma = (big_msb(&P) - 2) / 2;
  if (gamma < 1 || ceil_log2_i64(K) > 2 * gamma - 4) return OZK_REF_EUNSUPPORTED;
  return gamma;
}

/* floor(2 log2 |x|) for finite nonzero x: |x| = f 2^E with f in [0.5, 1), so
 * 2 log2 |x| = 2 (E - 1) + 2 log2(2f), and 2 log2(2f) >= 1 exactly when
 * (2f)^2 >= 2, i.e. m^2 >= 2^105 for the integer significand m = f 2^53. */
static int half_octave(double x) {
  int E;
  double f = frexp(fabs(x), &E);
  uint64_t m = (uint64_t)ldexp(f, 53);
  unsigned __int128 mm = (unsigned __int128)m * m;
  return 2 * (E - 1) + (mm >= ((unsigned __int128)1 << 105) ? 1 : 0);
}

static int32_t scale_norm_of(const double* x, int64_t len, int64_t stride, int gamma) {
  int H = INT32_MIN;
  for (int64_t k = 0; k < len; ++k) {
    double v = x[k * stride];
    if (!isfinite(v)) return OZK_REF_NONFINITE;
    if (v != 0.0) {
      int h = half_octave(v);
      if (h > H) H = h;
    }
  }
  if (H == INT32_MIN) return 0; /* an all-zero row or column */
  uint64_t S = 0;
  for (int64_t k = 0; k < len; ++k) {
    double v = x[k * stride];
    if (v == 0.0) continue;
    int d = half_octave(v) - H + OZK_REF_NORM_WINDOW;
    S += (uint64_t)1 << (d > 0 ? d : 0);
  }
  int c = 0; /* ceil(log2 S) */
  while (((uint64_t)1 << c) < S) ++c;
  int num = 2 * gamma - (H + 1 - OZK_REF_NORM_WINDOW) - c;
  return num >= 0 ? num / 2 : -((-num + 1) / 2);
}

int ozk_ref_scale_norm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                       const double* B, int64_t ldb, int n, int32_t* s, int32_t* t) {
  if (M < 0 || N < 0 || K < 0) return OZK_REF_EINVAL;
  int gamma = ozk_ref_gamma(K, n);
  if (gamma < 0) return gamma;
  for (int64_t i = 0; i < M; ++i) s[i] = scale_norm_of(A + i * lda, K, 1, gamma);
  for (int64_t j = 0; j < N; ++j) t[j] = scale_norm_of(B + j, K, ldb, gamma);
  return OZK_REF_OK;
}

/* ------------------------------------------------------------------------- */
/* Step 2: exponent scaling and rounding to integers ("exponent scaling,     */
/* round"; reading: to nearest, ties to even)                                */
/* ------------------------------------------------------------------------- */
static double round_scaled_int(double x, int32_t sc) {
  if (sc == OZK_REF_NONFINITE) return 0.0;
  /* |x 2^sc| < 2^beta: the scaling is exact wherever the result is >= 1/2,
   * and anything smaller rounds to 0 whatever ldexp rounds it to.  nearbyint
   * rounds in the default mode: to nearest, ties to even. */
  return nearbyint(ldexp(x, sc));
}

int ozk_ref_integers(int64_t rows, int64_t cols, const double* X, int64_t ld,
                     const int32_t* scale, int by_row, double* out) {
  if (rows < 0 || cols < 0) return OZK_REF_EINVAL;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] = round_scaled_int(X[r * ld + c], by_row ? scale[r] : scale[c]);
  return OZK_REF_OK;
}

/* ------------------------------------------------------------------------- */
/* Step 3: residues ("mod, balanced int8 conversion"; reading R4)            */
/* ------------------------------------------------------------------------- */
static int sym_residue(double xp, int32_t p) {
  __int128 v = (__int128)xp; /* exact: xp is an integer below 2^73 */
  int r = (int)(v % p);      /* C remainder carries the dividend's sign */
  if (r < 0) r += p;         /* canonical, [0, p) */
  if (r >= (p + 1) / 2) r -= p; /* balanced, [-floor(p/2), ceil(p/2) - 1] */
  return r;
}

int ozk_ref_residues(int64_t count, const double* xp, int n, int8_t* out) {
  if (count < 0 || n < 1 || n > OZK_REF_NMAX) return OZK_REF_EINVAL;
  for (int k = 0; k < n; ++k)
    for (int64_t e = 0; e < count; ++e) out[k * count + e] = (int8_t)sym_residue(xp[e], MODULI[k]);
  return OZK_REF_OK;
}

/* ------------------------------------------------------------------------- */
/* Steps 4-5: one integer GEMM per modulus, then mod reduction               */
/* ------------------------------------------------------------------------- */
/* The residue c = acc mod p comes from the exact int64 sum for every K (the
 * sums of K >= 2^17 terms are split into int32-exact chunks on the GPU, and
 * a sum of chunk residues mod p is the same residue).  Only the raw int32 sum,
 * when a caller asks for it, must fit int32; otherwise it is reported as 0
 * with OZK_REF_ES32. */
static int reduce_checked(int64_t acc, int32_t p, int32_t* raw, uint8_t* cmod) {
  int64_t c = acc % p;
  if (c < 0) c += p;
  *cmod = (uint8_t)c;
  if (acc >= ((int64_t)1 << 31) || acc < -((int64_t)1 << 31)) {
    if (raw) *raw = 0;
    return raw ? OZK_REF_ES32 : OZK_REF_OK;
  }
  if (raw) *raw = (int32_t)acc;
  return OZK_REF_OK;
}

int ozk_ref_gemm_mod(int64_t M, int64_t N, int64_t K, const int8_t* ra,
                     const int8_t* rb, int n, int32_t* raw, uint8_t* cmod) {
  if (M < 0 || N < 0 || K < 0 || n < 1 || n > OZK_REF_NMAX) return OZK_REF_EINVAL;
  int err = OZK_REF_OK;
  for (int k = 0; k < n; ++k) {
    const int8_t* a = ra + (int64_t)k * M * K;
    const int8_t* b = rb + (int64_t)k * K * N;
    for (int64_t i = 0; i < M; ++i)
      for (int64_t j = 0; j < N; ++j) {
        int64_t acc = 0;
        for (int64_t q = 0; q < K; ++q) acc += (int64_t)a[i * K + q] * (int64_t)b[q * N + j];
        int64_t o = (int64_t)k * M * N + i * N + j;
        if (reduce_checked(acc, MODULI[k], raw ? raw + o : NULL, cmod + o)) err = OZK_REF_ES32;
      }
  }
  return err;
}

/* ------------------------------------------------------------------------- */
/* Step 6: CRT reconstruction (Garner's mixed-radix form) and symmetric lift */
/* ------------------------------------------------------------------------- */
static int inverse_mod(int a, int p) {
  a %= p;
  for (int x = 1; x < p; ++x)
    if ((a * x) % p == 1) return x;
  return -1; /* not reached: the moduli are pairwise coprime */
}

static void crt_one(int n, const int* c, bigi* X) {
  int v[OZK_REF_NMAX]; /* mixed-radix digits, X = v0 + v1 p0 + v2 p0 p1 + ... */
  v[0] = c[0];
  for (int k = 1; k < n; ++k) {
    int pk = MODULI[k];
    int t = v[k - 1] % pk; /* (digits so far, as an integer) mod pk, by Horner */
    for (int j = k - 2; j >= 0; --j) t = (t * (MODULI[j] % pk) + v[j]) % pk;
    int q = 1; /* p0 ... p(k-1) mod pk */
    for (int j = 0; j < k; ++j) q = (q * (MODULI[j] % pk)) % pk;
    int d = ((c[k] - t) % pk + pk) % pk;
    v[k] = (d * inverse_mod(q, pk)) % pk;
  }
  big_set_u32(X, (uint32_t)v[n - 1]);
  for (int k = n - 2; k >= 0; --k) big_muladd_u32(X, X, (uint32_t)MODULI[k], (uint32_t)v[k]);
  bigi P, twoX;
  big_product_of_moduli(&P, n);
  big_add(&twoX, X, X);
  if (big_cmp(&twoX, &P) >= 0) big_sub(X, X, &P); /* X >= P/2 stands for X - P */
}

int ozk_ref_crt(int64_t count, int n, const uint8_t* cmod, uint32_t* X) {
  if (count < 0 || n < 2 || n > OZK_REF_NMAX) return OZK_REF_EINVAL;
  for (int64_t e = 0; e < count; ++e) {
    int c[OZK_REF_NMAX];
    for (int k = 0; k < n; ++k) c[k] = cmod[k * count + e];
    bigi x;
    crt_one(n, c, &x);
    memcpy(X + e * L, x.w, sizeof x.w);
  }
  return OZK_REF_OK;
}

/* ------------------------------------------------------------------------- */
/* The exact integer product the CRT must reproduce                          */
/* ------------------------------------------------------------------------- */
int ozk_ref_direct(int64_t M, int64_t N, int64_t K, const double* Ap,
                   const double* Bp, uint32_t* X) {
  if (M < 0 || N < 0 || K < 0) return OZK_REF_EINVAL;
  for (int64_t i = 0; i < M; ++i)
    for (int64_t j = 0; j < N; ++j) {
      bigi acc, prod;
      big_set_u32(&acc, 0);
      for (int64_t q = 0; q < K; ++q) {
        big_mul_i128(&prod, (__int128)Ap[i * K + q], (__int128)Bp[q * N + j]);
        big_add(&acc, &acc, &prod);
      }
      memcpy(X + (i * N + j) * L, acc.w, sizeof acc.w);
    }
  return OZK_REF_OK;
}

/* ------------------------------------------------------------------------- */
/* Step 7: undo scaling, write double (reading R8: one RN-even rounding)     */
/* ------------------------------------------------------------------------- */
static double round_scaled(const bigi* X, int32_t S) {
  int neg = big_is_negative(X);
  bigi m;
  if (neg)
    big_negate(&m, X);
  else
    m = *X;
  int h = big_msb(&m);
  if (h < 0) return 0.0;
  /* Lowest kept bit: 53 significant bits, fewer below 2^-1022 (the result is
   * then a multiple of 2^-1074). */
  int64_t lo = (int64_t)h - 52;
  if ((int64_t)S - 1074 > lo) lo = (int64_t)S - 1074;
  uint64_t q = 0;
  for (int64_t b = h; b >= lo; --b) q = (q << 1) | (uint64_t)big_bit(&m, b);
  int round_bit = big_bit(&m, lo - 1);
  int sticky = 0;
  for (int64_t b = lo - 2; b >= 0 && !sticky; --b) sticky = big_bit(&m, b);
  if (round_bit && (sticky || (q & 1u))) q += 1;
  /* q <= 2^53 and the exponent is >= -1074: ldexp is exact, or overflows to
   * infinity exactly when the rounded value reaches 2^1024. */
  double mag = ldexp((double)q, (int)(lo - S));
  return neg ? -mag : mag;
}

int ozk_ref_round(int64_t count, const uint32_t* X, const int32_t* S, double* out) {
  if (count < 0) return OZK_REF_EINVAL;
  for (int64_t e = 0; e < count; ++e) {
    bigi x;
    memcpy(x.w, X + e * L, sizeof x.w);
    out[e] = round_scaled(&x, S[e]);
  }
  return OZK_REF_OK;
}

/* ------------------------------------------------------------------------- */
/* The whole method                                                          */
/* ------------------------------------------------------------------------- */
/* rule 0: the scales of reading R2 (ozk_ref_scale); rule 1: those of the
 * computed norm bound, reading R15 (ozk_ref_scale_norm). */
static int dgemm_rule(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                      const double* B, int64_t ldb, double* C, int64_t ldc, int n, int rule) {
  if (M < 0 || N < 0 || K < 0) return OZK_REF_EINVAL;
  int budget = rule ? ozk_ref_gamma(K, n) : ozk_ref_beta(K, n);
  if (budget < 0) return budget;
  if (M == 0 || N == 0) return OZK_REF_OK;
  int32_t* s = malloc(sizeof(int32_t) * (size_t)M);
  int32_t* t = malloc(sizeof(int32_t) * (size_t)N);
  double* Ap = malloc(sizeof(double) * (size_t)(M * K + 1));
  double* Bt = malloc(sizeof(double) * (size_t)(N * K + 1)); /* b'_kj stored at [j][k] */
  int8_t* ra = malloc((size_t)(n * M * K + 1));
  int8_t* rbt = malloc((size_t)(n * N * K + 1)); /* residues of b'_kj at [p][j][k] */
  int err = OZK_REF_OK;
  if (!s || !t || !Ap || !Bt || !ra || !rbt) {
    err = OZK_REF_EINVAL;
    goto done;
  }
  if (rule)
    ozk_ref_scale_norm(M, N, K, A, lda, B, ldb, n, s, t);
  else
    ozk_ref_scale(M, N, K, A, lda, B, ldb, n, s, t);
  ozk_ref_integers(M, K, A, lda, s, 1, Ap);
  for (int64_t j = 0; j < N; ++j)
    for (int64_t q = 0; q < K; ++q) Bt[j * K + q] = round_scaled_int(B[q * ldb + j], t[j]);
  ozk_ref_residues(M * K, Ap, n, ra);
  ozk_ref_residues(N * K, Bt, n, rbt);

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      int c[OZK_REF_NMAX];
      for (int k = 0; k < n; ++k) {
        const int8_t* a = ra + (int64_t)k * M * K + i * K;
        const int8_t* b = rbt + (int64_t)k * N * K + j * K;
        int64_t acc = 0;
        for (int64_t q = 0; q < K; ++q) acc += (int64_t)a[q] * (int64_t)b[q];
        uint8_t cm;
        reduce_checked(acc, MODULI[k], NULL, &cm);
        c[k] = cm;
      }
      bigi xc, xd, prod;
      crt_one(n, c, &xc);
      big_set_u32(&xd, 0);
      for (int64_t q = 0; q < K; ++q) {
        big_mul_i128(&prod, (__int128)Ap[i * K + q], (__int128)Bt[j * K + q]);
        big_add(&xd, &xd, &prod);
      }
      if (big_cmp(&xc, &xd) != 0) {
#pragma omp atomic write
        err = OZK_REF_ECRT;
      }
      if (s[i] == OZK_REF_NONFINITE || t[j] == OZK_REF_NONFINITE)
        C[i * ldc + j] = NAN;
      else
        C[i * ldc + j] = round_scaled(&xc, s[i] + t[j]);
    }
  }
done:
  free(s);
  free(t);
  free(Ap);
  free(Bt);
  free(ra);
  free(rbt);
  return err;
}

int ozk_ref_dgemm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                  const double* B, int64_t ldb, double* C, int64_t ldc, int n) {
  return dgemm_rule(M, N, K, A, lda, B, ldb, C, ldc, n, 0);
}

int ozk_ref_dgemm_norm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                       const double* B, int64_t ldb, double* C, int64_t ldc, int n) {
  return dgemm_rule(M, N, K, A, lda, B, ldb, C, ldc, n, 1);
}

static int sample_rule(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                       const double* B, int64_t ldb, int n, int64_t npairs,
                       const int64_t* ii, const int64_t* jj, double* C, int32_t* raw,
                       uint8_t* cmod, uint32_t* X, int rule) {
  if (M < 0 || N < 0 || K < 0 || npairs < 0) return OZK_REF_EINVAL;
  int budget = rule ? ozk_ref_gamma(K, n) : ozk_ref_beta(K, n);
  if (budget < 0) return budget;
  for (int64_t q = 0; q < npairs; ++q)
    if (ii[q] < 0 || ii[q] >= M || jj[q] < 0 || jj[q] >= N) return OZK_REF_EINVAL;
  int err = OZK_REF_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t q = 0; q < npairs; ++q) {
    const double* arow = A + ii[q] * lda;
    const double* bcol = B + jj[q];
    int32_t si = rule ? scale_norm_of(arow, K, 1, budget) : scale_of(arow, K, 1, budget);
    int32_t tj = rule ? scale_norm_of(bcol, K, ldb, budget) : scale_of(bcol, K, ldb, budget);
    int64_t acc[OZK_REF_NMAX] = {0};
    bigi xd, prod, xc;
    big_set_u32(&xd, 0);
    for (int64_t k = 0; k < K; ++k) {
      double ap = round_scaled_int(arow[k], si);
      double bp = round_scaled_int(bcol[k * ldb], tj);
      for (int p = 0; p < n; ++p)
        acc[p] += (int64_t)sym_residue(ap, MODULI[p]) * (int64_t)sym_residue(bp, MODULI[p]);
      big_mul_i128(&prod, (__int128)ap, (__int128)bp);
      big_add(&xd, &xd, &prod);
    }
    int c[OZK_REF_NMAX];
    for (int p = 0; p < n; ++p) {
      int32_t r;
      uint8_t cm;
      if (reduce_checked(acc[p], MODULI[p], raw ? &r : NULL, &cm)) {
#pragma omp atomic write
        err = OZK_REF_ES32;
      }
      c[p] = cm;
      if (raw) raw[q * n + p] = r;
      if (cmod) cmod[q * n + p] = cm;
    }
    crt_one(n, c, &xc);
    if (big_cmp(&xc, &xd) != 0) {
#pragma omp atomic write
      err = OZK_REF_ECRT;
    }
    if (X) memcpy(X + q * L, xc.w, sizeof xc.w);
    if (si == OZK_REF_NONFINITE || tj == OZK_REF_NONFINITE)
      C[q] = NAN;
    else
      C[q] = round_scaled(&xc, si + tj);
  }
  return err;
}

int ozk_ref_sample(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                   const double* B, int64_t ldb, int n, int64_t npairs,
                   const int64_t* ii, const int64_t* jj, double* C, int32_t* raw,
                   uint8_t* cmod, uint32_t* X) {
  return sample_rule(M, N, K, A, lda, B, ldb, n, npairs, ii, jj, C, raw, cmod, X, 0);
}

int ozk_ref_sample_norm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                        const double* B, int64_t ldb, int n, int64_t npairs,
                        const int64_t* ii, const int64_t* jj, double* C, int32_t* raw,
                        uint8_t* cmod, uint32_t* X) {
  return sample_rule(M, N, K, A, lda, B, ldb, n, npairs, ii, jj, C, raw, cmod, X, 1);
}

/* ------------------------------------------------------------------------- */
/* Compensated reference DGEMM: Dot2 (Ogita, Rump, Oishi, "Accurate sum and  */
/* dot product", SIAM J. Sci. Comput. 26(6), 2005, Algorithm 5.3).  Its      */
/* result is as accurate as if computed in twice the working precision.      */
/* ------------------------------------------------------------------------- */
static void two_sum(double a, double b, double* s, double* e) {
  double x = a + b;
  double z = x - a;
  *e = (a - (x - z)) + (b - z);
  *s = x;
}

static void two_product(double a, double b, double* p, double* e) {
  double x = a * b;
  *e = fma(a, b, -x);
  *p = x;
}

static double dot2(const double* x, int64_t sx, const double* y, int64_t sy, int64_t K,
                   double* absdot) {
  double s = 0.0, c = 0.0, ab = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    double p, ep, es;
    two_product(x[k * sx], y[k * sy], &p, &ep);
    two_sum(s, p, &s, &es);
    c += ep + es;
    ab += fabs(x[k * sx]) * fabs(y[k * sy]);
  }
  if (absdot) *absdot = ab;
  return s + c;
}

int ozk_ref_dot2(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                 const double* B, int64_t ldb, double* R) {
  if (M < 0 || N < 0 || K < 0) return OZK_REF_EINVAL;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i)
    for (int64_t j = 0; j < N; ++j) R[i * N + j] = dot2(A + i * lda, 1, B + j, ldb, K, NULL);
  return OZK_REF_OK;
}

int ozk_ref_dot2_sample(int64_t K, const double* A, int64_t lda, const double* B,
                        int64_t ldb, int64_t npairs, const int64_t* ii,
                        const int64_t* jj, double* R, double* absAB) {
  if (K < 0 || npairs < 0) return OZK_REF_EINVAL;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t q = 0; q < npairs; ++q)
    R[q] = dot2(A + ii[q] * lda, 1, B + jj[q], ldb, K, absAB ? absAB + q : NULL);
  return OZK_REF_OK;
}

int ozk_ref_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
