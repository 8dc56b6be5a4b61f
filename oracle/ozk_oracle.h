/*
 * CPU oracle for Ozaki-scheme-II FP64 GEMM emulation (INT8-range residues,
 * Chinese-Remainder reconstruction).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant generator with the CUDA path.
 *
 * Source of the method: ithelp.ithome.com.tw "Day 12" (the Ozaki-II INT8/CRT
 * page), section "Profile 不能只看 Tensor Core", which lists the pipeline
 * stages in order: scale / exponent scan, residue quantization, INT8 GEMM,
 * mod reduction, CRT reconstruction, undo scaling, write double output.
 * The same page, section "為什麼 tile-local prologue 沒有直接贏", spells out
 * the quantisation step: double load, exponent scaling, round, mod, balanced
 * int8 conversion.  Everything the page leaves open is fixed by the readings
 * stated next to each function below.
 *
 * Conventions: A is M x K row-major with leading dimension lda, B is K x N
 * row-major with leading dimension ldb, C = A*B.  n is the moduli count
 * (2..20).  All functions return 0 on success and a negative code on error.
 */
#ifndef OZK_ORACLE_H
#define OZK_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

#define OZK_REF_NMAX 20
#define OZK_REF_LIMBS 8 /* signed wide integers: 8 x 32-bit limbs, two's complement */
#define OZK_REF_NONFINITE INT32_MIN /* scale of a row/column holding Inf or NaN */

enum {
  OZK_REF_OK = 0,
  OZK_REF_EINVAL = -1,      /* bad argument */
  OZK_REF_EUNSUPPORTED = -2, /* bit budget too small for K, or n outside 2..20 */
  OZK_REF_ES32 = -3,        /* a requested raw int32 per-modulus sum left the int32 range */
  OZK_REF_ECRT = -4         /* CRT-lifted integer differs from the direct product */
};

/* The first n entries of the moduli list. */
int ozk_ref_moduli(int n, int32_t* out);

/* Bit budget beta per operand (reading R2): the largest even split of
 * floor(log2 P) - 1 - ceil(log2 K) bits, so that 2*K*2^(2*beta) < P.
 * Returns beta, or OZK_REF_EUNSUPPORTED when beta < 1. */
int ozk_ref_beta(int64_t K, int n);

/* Exponent scan: s[i] = beta - E_i with max_k |a_ik| = f * 2^E_i, f in [0.5,1);
 * t[j] likewise over the columns of B.  Zero rows/columns get 0; a row or
 * column holding Inf/NaN gets OZK_REF_NONFINITE. */
int ozk_ref_scale(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                  const double* B, int64_t ldb, int n, int32_t* s, int32_t* t);

/* x * 2^scale rounded to the nearest integer, ties to even (the page's
 * "exponent scaling, round").  by_row != 0: scale[r] applies to row r;
 * otherwise scale[c] applies to column c.  out is rows x cols dense.
 * Entries whose scale is OZK_REF_NONFINITE give 0. */
int ozk_ref_integers(int64_t rows, int64_t cols, const double* X, int64_t ld,
                     const int32_t* scale, int by_row, double* out);

/* Balanced residues: out[p*count + e] = sym(xp[e] mod p_p), in
 * [-floor(p/2), ceil(p/2)-1]. */
int ozk_ref_residues(int64_t count, const double* xp, int n, int8_t* out);

/* One integer GEMM per modulus plus the mod reduction.
 * ra: n x M x K, rb: n x K x N (both residues).  raw (optional): n x M x N exact
 * int32 sums; cmod: n x M x N canonical residues in [0, p). */
int ozk_ref_gemm_mod(int64_t M, int64_t N, int64_t K, const int8_t* ra,
                     const int8_t* rb, int n, int32_t* raw, uint8_t* cmod);

/* CRT reconstruction (Garner mixed radix) plus symmetric lift.  cmod: n x count.
 * X: count x OZK_REF_LIMBS limbs. */
int ozk_ref_crt(int64_t count, int n, const uint8_t* cmod, uint32_t* X);

/* Direct wide integer product X = sum_k a'_ik b'_kj.  Ap: M x K, Bp: K x N,
 * holding exact integers.  X: M*N x OZK_REF_LIMBS. */
int ozk_ref_direct(int64_t M, int64_t N, int64_t K, const double* Ap,
                   const double* Bp, uint32_t* X);

/* Undo scaling: out[e] = RN-even(X[e] * 2^-S[e]), one rounding. */
int ozk_ref_round(int64_t count, const uint32_t* X, const int32_t* S, double* out);

/* Whole method, stage by stage, asserting CRT == direct product for every
 * output.  C: M x N with leading dimension ldc.  Uses OpenMP over rows. */
int ozk_ref_dgemm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                  const double* B, int64_t ldb, double* C, int64_t ldc, int n);

/* The method evaluated at chosen outputs only (for sizes too large to compute
 * in full).  For pair q = (ii[q], jj[q]): C[q], raw[q*n + p], cmod[q*n + p] and
 * X[q*LIMBS ...].  Any of raw, cmod, X may be NULL. */
int ozk_ref_sample(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                   const double* B, int64_t ldb, int n, int64_t npairs,
                   const int64_t* ii, const int64_t* jj, double* C, int32_t* raw,
                   uint8_t* cmod, uint32_t* X);

/* Compensated reference DGEMM (Ogita-Rump-Oishi Dot2) for error measurement.
 * R: M x N dense. */
int ozk_ref_dot2(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                 const double* B, int64_t ldb, double* R);

/* Dot2 at chosen outputs only. */
int ozk_ref_dot2_sample(int64_t K, const double* A, int64_t lda, const double* B,
                        int64_t ldb, int64_t npairs, const int64_t* ii,
                        const int64_t* jj, double* R, double* absAB);

/* Sharper scaling from a computed norm bound (reading R15; the survey's
 * "sharper scaling" next step).  gamma = floor((floor(log2 P) - 2) / 2), or
 * OZK_REF_EUNSUPPORTED when sqrt(K) > 2^(gamma - 2). */
#define OZK_REF_NORM_WINDOW 30 /* half-octaves below a row's largest entry counted exactly */
int ozk_ref_gamma(int64_t K, int n);

/* s[i] = floor((2 gamma - (H_i + 1 - W) - ceil(log2 S_i)) / 2) with
 * H_i = max_k floor(2 log2 |a_ik|) over the nonzero entries of row i,
 * S_i = sum over them of 2^max(floor(2 log2 |a_ik|) - H_i + W, 0) (an exact
 * integer, W = OZK_REF_NORM_WINDOW), so that 2^s_i ||a_i||_2 < 2^gamma; t[j]
 * likewise over the columns of B.  0 for an all-zero row/column, NONFINITE
 * for one holding Inf/NaN. */
int ozk_ref_scale_norm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                       const double* B, int64_t ldb, int n, int32_t* s, int32_t* t);

/* ozk_ref_dgemm and ozk_ref_sample with the scales of ozk_ref_scale_norm;
 * every other step is the same. */
int ozk_ref_dgemm_norm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                       const double* B, int64_t ldb, double* C, int64_t ldc, int n);
int ozk_ref_sample_norm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                        const double* B, int64_t ldb, int n, int64_t npairs,
                        const int64_t* ii, const int64_t* jj, double* C, int32_t* raw,
                        uint8_t* cmod, uint32_t* X);

/* Threads OpenMP will use (for reporting). */
int ozk_ref_threads(void);

#ifdef __cplusplus
}
#endif
#endif
