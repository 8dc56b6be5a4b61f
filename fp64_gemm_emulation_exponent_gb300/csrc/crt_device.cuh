// Device code of the CRT combine: CRT reconstruction, symmetric lift, undo
// scaling and FP64 write (the last three stages of the Ozaki-II pipeline on
// the "Day 12" page, section "Profile 不能只看 Tensor Core").  That page's
// section "Combine kernel 的瓶頸又不一樣" measures its own combine at ~85% of
// the FP64 pipe and warns that more registers per thread made it slower; on
// GB300 the FP64 pipe is slow, so this kernel is integer-only:
//
//   X = S - q P  (mod 2^(32 NL)),   S = sum_k c_k e_k,   q = round(S / P),
//
// with e_k the CRT basis vectors (e_k = 1 mod p_k, 0 mod the other moduli).
// S is built column by column in 16-bit limbs: every column sum
// sum_k c_k (limb l of e_k) is below n 2^24, so the byte residues are taken
// two at a time by a two-way 16x8-bit dot product (dp2a) against the packed
// limbs of two basis vectors, with no modular reduction and no 64-bit
// multiply-accumulate.  q comes from the same dot products over the ratios
// e_k / P = w_k / p_k in 0.32 fixed point (error below 2^-20); the rare
// outputs whose estimate lies within 2^-19 of a rounding boundary get an
// exact symmetric lift.  The 16-bit residues of moduli pairs (the GEMM's pair
// output) enter the same way, as two bytes with the bases E_j and 256 E_j.
// The lifted X in [-P/2, P/2) is then scaled by 2^-(s_i + t_j) and rounded to
// nearest-even in integer arithmetic (a short path for normal results, a
// general one for subnormals and overflow).
#pragma once

#include "ozk_internal.h"

namespace ozk {
namespace {

constexpr uint64_t kQuietNaN = 0x7FF8000000000000ull;
constexpr uint64_t kInfBits = 0x7FF0000000000000ull;

__device__ __forceinline__ uint32_t mod_p(int32_t x, uint32_t p, uint32_t magic, uint32_t bias) {
  const uint32_t u = static_cast<uint32_t>(x) + bias;
  const uint32_t q = __umulhi(u, magic);
  int32_t r = static_cast<int32_t>(u - q * p);
  r += r < 0 ? static_cast<int32_t>(p) : 0;
  return static_cast<uint32_t>(r);
}

// a += P, or a -= P when subtract (two's complement, NL limbs).
template <int NL>
__device__ __forceinline__ void add_signed_P(uint32_t (&a)[NL], const CrtConst& K, bool subtract) {
  uint64_t carry = subtract ? 1u : 0u;
#pragma unroll
  for (int l = 0; l < NL; ++l) {
    const uint32_t pl = subtract ? ~K.P[l] : K.P[l];
    const uint64_t v = static_cast<uint64_t>(a[l]) + pl + carry;
    a[l] = static_cast<uint32_t>(v);
    carry = v >> 32;
  }
}

template <int NL>
__device__ __forceinline__ bool is_negative(const uint32_t (&a)[NL]) {
  return (a[NL - 1] >> 31) != 0;
}

// Exact symmetric lift for outputs whose quotient estimate was ambiguous:
// move X into [-P/2, P/2) by one P if needed.
template <int NL>
__device__ __forceinline__ void exact_lift(uint32_t (&X)[NL], const CrtConst& K) {
  uint32_t t[NL];  // 2X
#pragma unroll
  for (int l = 0; l < NL; ++l) {
    const uint32_t hi = l ? (X[l - 1] >> 31) : 0u;
    t[l] = (X[l] << 1) | hi;
  }
  // 2X - P >= 0  <=>  X >= P/2
  uint32_t t2[NL];
#pragma unroll
  for (int l = 0; l < NL; ++l) t2[l] = t[l];
  add_signed_P<NL>(t2, K, true);
  if (!is_negative<NL>(t2)) {
    add_signed_P<NL>(X, K, true);
    return;
  }
  // t = 2X + P: X < -P/2  <=>  t < 0
  add_signed_P<NL>(t, K, false);
  if (is_negative<NL>(t)) add_signed_P<NL>(X, K, false);
}

// RN-even double of X * 2^-S for a two's-complement NL-limb integer X,
// handled as up to three 64-bit words.
template <int NL>
__device__ __forceinline__ uint64_t round_scaled_bits(const uint32_t (&X)[NL], int S) {
  constexpr int NW = (NL + 1) / 2;
  uint64_t w[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const uint32_t lo = X[2 * i];
    const uint32_t hi = (2 * i + 1 < NL) ? X[2 * i + 1] : ((X[NL - 1] >> 31) ? 0xFFFFFFFFu : 0u);
    w[i] = (static_cast<uint64_t>(hi) << 32) | lo;
  }
  const bool neg = (w[NW - 1] >> 63) != 0;
  if (neg) {  // magnitude
    uint64_t c = 1;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const uint64_t v = ~w[i] + c;
      c = (c && v == 0) ? 1u : 0u;
      w[i] = v;
    }
  }
  uint64_t hi, mid, lo;
  int base;
  if (NW == 3 && w[NW - 1] != 0) {
    hi = w[NW - 1];
    mid = w[NW > 1 ? NW - 2 : 0];
    lo = w[0];
    base = 128;
  } else if (NW >= 2 && w[NW >= 2 ? 1 : 0] != 0) {
    hi = w[NW >= 2 ? 1 : 0];
    mid = w[0];
    lo = 0;
    base = 64;
  } else {
    hi = w[0];
    mid = 0;
    lo = 0;
    base = 0;
  }
  if (hi == 0) return 0ull;  // exact zero: +0
  const int lz = __clzll(static_cast<long long>(hi));
  const uint64_t win = lz ? (hi << lz) | (mid >> (64 - lz)) : hi;
  const bool sticky = ((lz ? (mid << lz) : mid) | lo) != 0;  // bits below the window
  const int h = base + 63 - lz;                              // leading bit of |X|
  const int e = h - S;                                       // |X| 2^-S in [2^e, 2^(e+1))
  uint64_t bits;
  if (e > 1023) {
    bits = kInfBits;
  } else {
    // drop sh >= 11 bits of the window: 53 significant bits, fewer below 2^-1022
    const int sh = e >= -1022 ? 11 : 11 + (-1022 - e);
    uint64_t q;
    uint32_t rb, st;
    if (sh >= 65) {
      q = 0;
      rb = 0;
      st = 1;
    } else if (sh == 64) {
      q = 0;
      rb = static_cast<uint32_t>(win >> 63);
      st = ((win << 1) != 0) | sticky;
    } else {
      q = win >> sh;
      rb = static_cast<uint32_t>(win >> (sh - 1)) & 1u;
      st = ((win & ((1ull << (sh - 1)) - 1)) != 0) | sticky;
    }
    q += rb & (st | static_cast<uint32_t>(q & 1u));
    // lowest kept bit has weight 2^(e + sh - 63); the biased exponent field
    // base is e + sh + 1011 (0 in the subnormal range); a rounding carry
    // into bit 53 bumps the exponent by itself
    const uint64_t E0 = static_cast<uint64_t>(e + sh + 1011);
    bits = (E0 << 52) + q;
    if (bits >= kInfBits) bits = kInfBits;
  }
  return bits | (static_cast<uint64_t>(neg) << 63);
}

// Fast path of round_scaled_bits for |X| >= 2^(32(NL-2)) with a normal
// result: a 64-bit window from the top two nonzero-headed limbs, 53 bits
// kept, round to nearest even with the bits below as sticky.  Branch-free:
// always writes *out, and returns false when that value is not the answer
// (the slow path must decide).
template <int NL>
__device__ __forceinline__ bool round_scaled_fast(const uint32_t (&X)[NL], int S, uint64_t* out) {
  const uint32_t sgn = X[NL - 1] >> 31;
  const uint32_t flip = 0u - sgn;
  uint32_t m[NL];
  if constexpr (NL == 4) {  // |X| = (X ^ flip) + sgn, one carry chain
    asm("{\n\t"
        "add.cc.u32 %0, %4, %8;\n\t"
        "addc.cc.u32 %1, %5, 0;\n\t"
        "addc.cc.u32 %2, %6, 0;\n\t"
        "addc.u32 %3, %7, 0;\n\t}"
        : "=r"(m[0]), "=r"(m[1]), "=r"(m[2]), "=r"(m[3])
        : "r"(X[0] ^ flip), "r"(X[1] ^ flip), "r"(X[2] ^ flip), "r"(X[3] ^ flip), "r"(sgn));
  } else {
    uint32_t c = sgn;
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      const uint32_t x = X[l] ^ flip;
      m[l] = x + c;
      c = (c && m[l] == 0u) ? 1u : 0u;
    }
  }
  const bool top = m[NL - 1] != 0u;
  const uint32_t t2 = top ? m[NL - 1] : m[NL - 2];
  const uint32_t t1 = top ? m[NL - 2] : m[NL - 3];
  uint32_t t0, st;
  if constexpr (NL >= 4) {
    uint32_t below = 0;  // OR of the limbs under t0 when the top limb leads
#pragma unroll
    for (int l = 0; l + 3 < NL; ++l) below |= m[l];
    uint32_t below2 = 0;  // same when limb NL-2 leads
#pragma unroll
    for (int l = 0; l + 4 < NL; ++l) below2 |= m[l];
    t0 = top ? m[NL - 3] : m[NL - 4];
    st = top ? below : below2;
  } else {
    t0 = top ? m[0] : 0u;
    st = 0u;
  }
  const int lz = __clz(t2);  // 32 when t2 = 0: then the result is discarded
  const uint32_t hi = __funnelshift_l(t1, t2, lz);
  const uint32_t mid = __funnelshift_l(t0, t1, lz);
  const uint32_t lo = t0 << (lz & 31);
  const int e = (top ? 32 * (NL - 1) : 32 * (NL - 2)) + 31 - lz - S;  // |X| 2^-S in [2^e, 2^(e+1))
  const uint32_t sig_lo = __funnelshift_r(mid, hi, 11);
  const uint32_t sig_hi = hi >> 11;
  const uint32_t rb = (mid >> 10) & 1u;
  const uint32_t sticky = ((mid & 0x3FFu) | lo | st) != 0u ? 1u : 0u;
  const uint32_t inc = rb & (sticky | (sig_lo & 1u));
  // the significand carries the leading one at bit 52: exponent field e + 1022
  // plus one; a rounding carry into bit 53 bumps it once more (to Inf at the top)
  if constexpr (NL >= 4) {
    // exponent field and sign into the high word by funnel shifts (the ALU's
    // shifter, off the multiply pipe the combine is bound by from four limbs
    // up); a rounding carry out of the low word by the 64-bit add
    const uint32_t hi_word = __funnelshift_l(0u, static_cast<uint32_t>(e + 1022), 20) + sig_hi;
    const uint64_t bits = ((static_cast<uint64_t>(hi_word) << 32) | sig_lo) + inc;
    *out = bits | (static_cast<uint64_t>(__funnelshift_l(0u, sgn, 31)) << 32);
  } else {
    const uint64_t bits = (static_cast<uint64_t>(e + 1022) << 52) +
                          ((static_cast<uint64_t>(sig_hi) << 32) | sig_lo) + inc;
    *out = bits | (static_cast<uint64_t>(sgn) << 63);
  }
  return t2 != 0u && e >= -1022 && e <= 1023;
}

__device__ __forceinline__ void store4_f64(double* dst, const uint64_t (&b)[4]) {
  asm volatile("st.global.cs.v4.b64 [%0], {%1, %2, %3, %4};" ::"l"(dst), "l"(b[0]), "l"(b[1]), "l"(b[2]),
               "l"(b[3])
               : "memory");
}

// w[x] for a run-time x below G, by selects (no local-memory indexing).
template <int G>
__device__ __forceinline__ uint32_t pick(const uint32_t (&w)[G], int x) {
  uint32_t r = w[0];
#pragma unroll
  for (int y = 1; y < G; ++y) r = x == y ? w[y] : r;
  return r;
}

template <int G>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t (&w)[G]) {
  if constexpr (G == 1) {
    w[0] = __ldcs(reinterpret_cast<const unsigned int*>(p));
  } else if constexpr (G == 2) {
    const uint2 v = __ldcs(reinterpret_cast<const uint2*>(p));
    w[0] = v.x;
    w[1] = v.y;
  } else {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  }
}

// Below this distance (in units of 2^-32) of a rounding boundary the
// quotient estimate q = round(S / P) may be off by one; the estimate's error
// is at most n * 255 * 2^-33 < 2^-20 (fractions rounded to 0.32 fixed
// point), so such outputs get the exact symmetric lift.
constexpr uint32_t kLiftMargin = 1u << 13;





// One thread per 4G consecutive columns of one row, in G groups of 4, each
// group in two halves of two outputs.  For a half, the two byte digits of a
// modulus pair (or the two bytes of a pair residue) sit side by side for both
// outputs in one word: a byte permute of the two moduli's loaded words, or
// the loaded uint16 pair residues as they are.  A two-way dot product then
// adds both digits times limb l of their bases into column l of one output
// (dp2a lo for the first output, hi for the second); two more columns gather
// round(2^32 b_t / P) in 16-bit halves for q.  Columns stay below 2^29.5, so
// 32-bit sums are exact.  X = S - q P is assembled from the columns (plus
// q times the 16-bit limbs of 2^(32 NL) - P) into NL 32-bit limbs.
// NFIX > 0 fixes the moduli count at compile time (it must equal K.n); those
// kernels are held to five 256-thread blocks per SM at three limbs (48
// registers: 8192^2 at 8 moduli 317 -> 304 us against four blocks), four at
// four limbs (five spilled there: 456 -> 494 us) and three beyond.
//  IN_KIND 0: uint8 residues, modulus k at in + k * plane, row i at + i * ldi;
//  IN_KIND 1: int32 partial sums, split sp and modulus k at (sp * n + k) * plane.
// All residue words are loaded before any arithmetic so that the loads of a
// thread are in flight together.
template <int NL, int IN_KIND, bool LIMBS, int G, int NFIX>
__global__ void __launch_bounds__(256, NFIX ? (NL <= 3 ? 5 : (NL <= 4 ? 4 : 3)) : 1)
    crt_kernel(const void* __restrict__ in, int64_t ldi, int64_t plane, int64_t M, int64_t N, int splits,
               const int32_t* __restrict__ s, const int32_t* __restrict__ t, double* __restrict__ C, int64_t ldc,
               uint32_t* __restrict__ Xout, const __grid_constant__ CrtConst K, const FastDiv rd) {
  grid_dependency_sync();
  constexpr int W = 4 * G;  // columns per thread
  static_assert(IN_KIND != 2, "pair residues take crt_pairs_kernel");
  // columns of a four-column group accumulated together: four share each
  // basis constant; two keep the wider accumulators of five or six limbs small
  constexpr int kPassCols = NL <= 4 ? 4 : 2;
  // 16-bit limbs of the bases (a run-time count takes the most its limb count allows)
  constexpr int NC = NFIX ? crt_cols16(NFIX) : (2 * NL < kMaxCols16 ? 2 * NL : kMaxCols16);
  static_assert(NC <= 2 * NL, "the accumulator holds every basis limb");
  const int64_t groups = (N + W - 1) / W;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= M * groups) return;
  int64_t i, jt;
  if (M * groups <= 0x7FFFFFFF) {
    const uint32_t g32 = static_cast<uint32_t>(gid), gr = static_cast<uint32_t>(groups);
    const uint32_t i32 = div_fast(g32, rd);  // g32 / gr
    i = i32;
    jt = static_cast<int64_t>(g32 - i32 * gr) * W;
  } else {
    i = gid / groups;
    jt = (gid - i * groups) * W;
  }
  const int n = NFIX ? NFIX : K.n;  // a compile-time moduli count lets every loop unroll exactly

  // cw[k][g] holds the 4 byte residues of modulus k for columns 4g .. 4g + 3
  uint32_t cw[kMaxModuli][G];
  if constexpr (IN_KIND == 0) {
    const uint8_t* base = static_cast<const uint8_t*>(in) + i * ldi + jt;
    static_for<0, kMaxModuli>([&](auto kc) {
      constexpr int k = decltype(kc)::value;
      if (k < n) {
        if constexpr (NL >= 4) {  // plane by plane with adds, off the multiply pipe (see assemble)
          load_words<G>(base, cw[k]);
          base += plane;
        } else {
          load_words<G>(base + k * plane, cw[k]);
        }
      }
    });
  } else {
    static_for<0, kMaxModuli>([&](auto kc) {
      constexpr int k = decltype(kc)::value;
      if (k < n) {
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          // each partial is an exact int32 sum; their residues are added up
          // (at most 64 * 255) so that K beyond one int32-exact sum stays exact
          int32_t sum[4] = {0, 0, 0, 0};
          for (int sp = 0; sp < splits; ++sp) {
            const int4 v = __ldcs(reinterpret_cast<const int4*>(static_cast<const int32_t*>(in) +
                                                                (static_cast<int64_t>(sp) * n + k) * plane +
                                                                i * ldi + jt + 4 * gg));
            sum[0] += static_cast<int32_t>(mod_p(v.x, K.p[k], K.magic[k], K.bias[k]));
            sum[1] += static_cast<int32_t>(mod_p(v.y, K.p[k], K.magic[k], K.bias[k]));
            sum[2] += static_cast<int32_t>(mod_p(v.z, K.p[k], K.magic[k], K.bias[k]));
            sum[3] += static_cast<int32_t>(mod_p(v.w, K.p[k], K.magic[k], K.bias[k]));
          }
          cw[k][gg] = mod_p(sum[0], K.p[k], K.magic[k], K.bias[k]) |
                      (mod_p(sum[1], K.p[k], K.magic[k], K.bias[k]) << 8) |
                      (mod_p(sum[2], K.p[k], K.magic[k], K.bias[k]) << 16) |
                      (mod_p(sum[3], K.p[k], K.magic[k], K.bias[k]) << 24);
        }
      }
    });
  }
  const int32_t si = LIMBS ? 0 : s[i];

#pragma unroll 1
  for (int gg = 0; gg < G; ++gg) {
    const int64_t j0 = jt + 4 * gg;
    if (j0 >= N) break;
    int32_t tj[4] = {0, 0, 0, 0};
    if constexpr (!LIMBS) {
      if (j0 + 3 < N) {
        const int4 t4 = *reinterpret_cast<const int4*>(t + j0);
        tj[0] = t4.x;
        tj[1] = t4.y;
        tj[2] = t4.z;
        tj[3] = t4.w;
      } else {
#pragma unroll
        for (int o = 0; o < 4; ++o) tj[o] = (j0 + o < N) ? t[j0 + o] : 0;
      }
    }
    uint64_t outbits[4] = {0, 0, 0, 0};
    // the four columns of the group in kPassCols passes; a pass keeps its
    // columns' accumulators live and takes each basis constant once
#pragma unroll
    for (int pass = 0; pass < 4 / kPassCols; ++pass) {
      uint32_t col[kPassCols][2 * NL];
      uint32_t qh[kPassCols], ql[kPassCols];
#pragma unroll
      for (int o = 0; o < kPassCols; ++o) {
        qh[o] = ql[o] = 0;
#pragma unroll
        for (int l = 0; l < 2 * NL; ++l) col[o][l] = 0;
      }
      static_for<0, kMaxModuli / 2>([&](auto jc) {
        constexpr int j = decltype(jc)::value;
        if (2 * j < n) {
          // b[h]: digits of the pair for columns 2h, 2h+1 of the pass: bytes
          // (first, second) of the first column, then of the second
          uint32_t b[kPassCols / 2];
#pragma unroll
          for (int h = 0; h < kPassCols / 2; ++h) {
            const int sub = pass * (kPassCols / 2) + h;  // half of the group: columns 2 sub, 2 sub + 1
            const uint32_t wa = pick<G>(cw[2 * j], gg);
            const uint32_t wb = 2 * j + 1 < n ? pick<G>(cw[2 * j + 1 < kMaxModuli ? 2 * j + 1 : 0], gg) : 0u;
            b[h] = __byte_perm(wa, wb, sub ? 0x7362 : 0x5140);
          }
#pragma unroll
          for (int l = 0; l < NC; ++l) {
            const uint32_t bl = K.bt[j][l];
#pragma unroll
            for (int h = 0; h < kPassCols / 2; ++h) {
              col[2 * h][l] = __dp2a_lo(bl, b[h], col[2 * h][l]);
              col[2 * h + 1][l] = __dp2a_hi(bl, b[h], col[2 * h + 1][l]);
            }
          }
          const uint32_t fh = K.bfh[j];
          const uint32_t fl = K.bfl[j];
#pragma unroll
          for (int h = 0; h < kPassCols / 2; ++h) {
            qh[2 * h] = __dp2a_lo(fh, b[h], qh[2 * h]);
            qh[2 * h + 1] = __dp2a_hi(fh, b[h], qh[2 * h + 1]);
            ql[2 * h] = __dp2a_lo(fl, b[h], ql[2 * h]);
            ql[2 * h + 1] = __dp2a_hi(fl, b[h], ql[2 * h + 1]);
          }
        }
      });
      // q = round(S / P) from qh 2^16 + ql (32.32 fixed point) plus one
      // half, then X = S + q (2^(32 NL) - P) mod 2^(32 NL) from the 16-bit
      // columns (limb l = c_2l + c_2l+1 2^16 + the carry of limb l - 1);
      // returns the fraction of S / P + 1/2 (0.32 fixed point)
      // The 16-bit moves of the assembly are byte permutes from four limbs
      // up: the kernel is bound by the pipe of its dot products and
      // multiplies, which shifts may be given (measured: 8192^2, 14 moduli,
      // 481 -> 471 us; 20 moduli 759 -> 723 us; three limbs are faster with
      // the shifts, 321 against 330 us at 8 moduli).
      auto assemble = [&](int o, uint32_t (&X)[NL]) -> uint32_t {
        uint32_t q, frac;
        if constexpr (NL >= 4) {
          asm("{\n\t.reg .u32 t;\n\t"
              "prmt.b32 t, %2, 0, 0x1044;\n\t"  // qh << 16
              "add.cc.u32 t, t, %3;\n\t"
              "addc.u32 %0, 0, 0;\n\t"
              "add.cc.u32 %1, t, 0x80000000;\n\t"
              "addc.u32 %0, %0, 0;\n\t}"
              : "=r"(q), "=r"(frac)
              : "r"(qh[o]), "r"(ql[o]));
          q += __byte_perm(qh[o], 0, 0x4432);  // qh >> 16
        } else {
          asm("{\n\t.reg .u32 t;\n\t"
              "shl.b32 t, %2, 16;\n\t"
              "add.cc.u32 t, t, %3;\n\t"
              "addc.u32 %0, 0, 0;\n\t"
              "add.cc.u32 %1, t, 0x80000000;\n\t"
              "addc.u32 %0, %0, 0;\n\t}"
              : "=r"(q), "=r"(frac)
              : "r"(qh[o]), "r"(ql[o]));
          q += qh[o] >> 16;
        }
        uint32_t carry = 0;
#pragma unroll
        for (int l = 0; l < NL; ++l) {
          const uint32_t c0 = col[o][2 * l] + q * K.pn16[2 * l];
          const uint32_t c1 = col[o][2 * l + 1] + q * K.pn16[2 * l + 1];
          uint32_t x, nc;
          if constexpr (NL >= 4)
            asm("{\n\t.reg .u32 t, h;\n\t"
                "prmt.b32 h, %3, 0, 0x4432;\n\t"  // c1 >> 16
                "prmt.b32 t, %3, 0, 0x1044;\n\t"  // c1 << 16
                "add.cc.u32 t, t, %2;\n\t"
                "addc.u32 h, h, 0;\n\t"
                "add.cc.u32 %0, t, %4;\n\t"
                "addc.u32 %1, h, 0;\n\t}"
                : "=r"(x), "=r"(nc)
                : "r"(c0), "r"(c1), "r"(carry));
          else
            asm("{\n\t.reg .u32 t, h;\n\t"
                "shr.u32 h, %3, 16;\n\t"
                "shl.b32 t, %3, 16;\n\t"
                "add.cc.u32 t, t, %2;\n\t"
                "addc.u32 h, h, 0;\n\t"
                "add.cc.u32 %0, t, %4;\n\t"
                "addc.u32 %1, h, 0;\n\t}"
                : "=r"(x), "=r"(nc)
                : "r"(c0), "r"(c1), "r"(carry));
          X[l] = x;
          carry = nc;
        }
        return frac;
      };
      // With four outputs per pass the common case takes no branch: the fast
      // unscale of every output; outputs that need the exact lift, have a
      // non-finite scale or fall outside the fast unscale are marked and
      // redone after the pass.  (Wider X, two outputs per pass: each output
      // takes its own branches, which measured faster there.)
      constexpr bool kDeferRare = kPassCols == 4;
      uint32_t rare = 0;
#pragma unroll
      for (int o = 0; o < kPassCols; ++o) {
        const int oc = pass * kPassCols + o;  // output column j0 + oc
        uint32_t X[NL];
        const uint32_t frac = assemble(o, X);
        const bool lift = frac < kLiftMargin || frac > ~kLiftMargin;
        if constexpr (LIMBS) {
          if (lift) exact_lift<NL>(X, K);
          if (j0 + oc < N) {
            uint32_t* dst = Xout + (i * N + j0 + oc) * OZK_LIMBS;
            const uint32_t ext = is_negative<NL>(X) ? 0xFFFFFFFFu : 0u;
#pragma unroll
            for (int l = 0; l < OZK_LIMBS; ++l) dst[l] = l < NL ? X[l] : ext;
          }
        } else if constexpr (kDeferRare) {
          const bool ok = round_scaled_fast<NL>(X, si + tj[oc], &outbits[oc]);
          rare |= (lift || !ok || si == OZK_SCALE_NONFINITE || tj[oc] == OZK_SCALE_NONFINITE) ? 1u << o : 0u;
        } else {
          if (lift) exact_lift<NL>(X, K);
          if (si == OZK_SCALE_NONFINITE || tj[oc] == OZK_SCALE_NONFINITE)
            outbits[oc] = kQuietNaN;
          else if (!round_scaled_fast<NL>(X, si + tj[oc], &outbits[oc]))
            outbits[oc] = round_scaled_bits<NL>(X, si + tj[oc]);
        }
      }
      if constexpr (!LIMBS && kDeferRare) {
        if (rare) {
#pragma unroll
          for (int o = 0; o < kPassCols; ++o) {
            if (!((rare >> o) & 1u)) continue;
            const int oc = pass * kPassCols + o;
            uint32_t X[NL];
            const uint32_t frac = assemble(o, X);
            if (frac < kLiftMargin || frac > ~kLiftMargin) exact_lift<NL>(X, K);
            if (si == OZK_SCALE_NONFINITE || tj[oc] == OZK_SCALE_NONFINITE)
              outbits[oc] = kQuietNaN;
            else if (!round_scaled_fast<NL>(X, si + tj[oc], &outbits[oc]))
              outbits[oc] = round_scaled_bits<NL>(X, si + tj[oc]);
          }
        }
      }
    }
    if constexpr (!LIMBS) {
      double* dst = C + i * ldc + j0;
      if (j0 + 3 < N && (reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
        store4_f64(dst, outbits);
      } else {
#pragma unroll
        for (int o = 0; o < 4; ++o)
          if (j0 + o < N) __stcs(reinterpret_cast<unsigned long long*>(dst + o), outbits[o]);
      }
    }
  }
}

// The combine from the uint16 residues r_j of the moduli pairs (the GEMM's
// pair output; an odd last plane holds c_n-1): S = sum_j r_j E_j in 32-bit
// limbs, each product r_j (limb l of E_j) accumulated in 64 bits without
// carries (the top limb in 32 bits: only its value mod 2^32 matters), and
// q = round(sum_j r_j W_j / m_j) from round(2^32 W_j / m_j) in 32.32 fixed
// point (error below 10 * 2^16 * 2^-33 < 2^-13); outputs within 2^-12 of a
// rounding boundary get the exact lift.  One thread per 4G consecutive
// columns of one row; pair j's residues at in + j * plane + i * ldi.
template <int NL, bool LIMBS, int G, int NFIX>
__global__ void __launch_bounds__(256, NFIX ? (NL <= 4 ? 4 : 3) : 1)
    crt_pairs_kernel(const void* __restrict__ in, int64_t ldi, int64_t plane, int64_t M, int64_t N,
                     const int32_t* __restrict__ s, const int32_t* __restrict__ t, double* __restrict__ C,
                     int64_t ldc, uint32_t* __restrict__ Xout, const __grid_constant__ CrtConst K,
                     const FastDiv rd) {
  grid_dependency_sync();
  constexpr int W = 4 * G;
  constexpr uint32_t kPairLiftMargin = 1u << 20;
  const int64_t groups = (N + W - 1) / W;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= M * groups) return;
  int64_t i, jt;
  if (M * groups <= 0x7FFFFFFF) {
    const uint32_t g32 = static_cast<uint32_t>(gid), gr = static_cast<uint32_t>(groups);
    const uint32_t i32 = div_fast(g32, rd);  // g32 / gr
    i = i32;
    jt = static_cast<int64_t>(g32 - i32 * gr) * W;
  } else {
    i = gid / groups;
    jt = (gid - i * groups) * W;
  }
  const int n = NFIX ? NFIX : K.n;
  // pw[j][x]: word x (the residues of columns 2x, 2x + 1) of pair j's plane
  uint32_t pw[kMaxModuli / 2][2 * G];
  const uint16_t* base = static_cast<const uint16_t*>(in) + i * ldi + jt;
  static_for<0, kMaxModuli / 2>([&](auto jc) {
    constexpr int j = decltype(jc)::value;
    if (2 * j < n) load_words<2 * G>(reinterpret_cast<const uint8_t*>(base + j * plane), pw[j]);
  });
  const int32_t si = LIMBS ? 0 : s[i];

#pragma unroll 1
  for (int gg = 0; gg < G; ++gg) {
    const int64_t j0 = jt + 4 * gg;
    if (j0 >= N) break;
    int32_t tj[4] = {0, 0, 0, 0};
    if constexpr (!LIMBS) {
      if (j0 + 3 < N) {
        const int4 t4 = *reinterpret_cast<const int4*>(t + j0);
        tj[0] = t4.x;
        tj[1] = t4.y;
        tj[2] = t4.z;
        tj[3] = t4.w;
      } else {
#pragma unroll
        for (int o = 0; o < 4; ++o) tj[o] = (j0 + o < N) ? t[j0 + o] : 0;
      }
    }
    uint64_t acc[4][NL - 1];
    uint32_t acctop[4];
    uint64_t qacc[4];
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      qacc[o] = 0;
      acctop[o] = 0;
#pragma unroll
      for (int l = 0; l < NL - 1; ++l) acc[o][l] = 0;
    }
    static_for<0, kMaxModuli / 2>([&](auto jc) {
      constexpr int j = decltype(jc)::value;
      if (2 * j < n) {
        const bool pair = 2 * j + 1 < n;
        const uint32_t w01 = pick<2 * G>(pw[j], 2 * gg), w23 = pick<2 * G>(pw[j], 2 * gg + 1);
#pragma unroll
        for (int o = 0; o < 4; ++o) {
          const uint32_t r = ((o < 2 ? w01 : w23) >> (16 * (o & 1))) & 0xFFFFu;
          qacc[o] += static_cast<uint64_t>(r) * (pair ? K.pfrac[j] : K.flast);
#pragma unroll
          for (int l = 0; l < NL - 1; ++l)
            acc[o][l] += static_cast<uint64_t>(r) * (pair ? K.pe[j][l] : K.elast[l]);
          acctop[o] += r * (pair ? K.pe[j][NL - 1] : K.elast[NL - 1]);
        }
      }
    });
    uint64_t outbits[4] = {0, 0, 0, 0};
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      const uint64_t shifted = qacc[o] + 0x80000000ull;
      const uint32_t q = static_cast<uint32_t>(shifted >> 32);
      const uint32_t frac = static_cast<uint32_t>(shifted);
      uint32_t X[NL];
      uint64_t carry = 0;
#pragma unroll
      for (int l = 0; l < NL - 1; ++l) {
        const uint64_t v = acc[o][l] + static_cast<uint64_t>(q) * K.pn[l] + carry;
        X[l] = static_cast<uint32_t>(v);
        carry = v >> 32;
      }
      X[NL - 1] = acctop[o] + q * K.pn[NL - 1] + static_cast<uint32_t>(carry);
      if (frac < kPairLiftMargin || frac > ~kPairLiftMargin) exact_lift<NL>(X, K);
      if constexpr (LIMBS) {
        if (j0 + o < N) {
          uint32_t* dst = Xout + (i * N + j0 + o) * OZK_LIMBS;
          const uint32_t ext = is_negative<NL>(X) ? 0xFFFFFFFFu : 0u;
#pragma unroll
          for (int l = 0; l < OZK_LIMBS; ++l) dst[l] = l < NL ? X[l] : ext;
        }
      } else {
        if (si == OZK_SCALE_NONFINITE || tj[o] == OZK_SCALE_NONFINITE)
          outbits[o] = kQuietNaN;
        else if (!round_scaled_fast<NL>(X, si + tj[o], &outbits[o]))
          outbits[o] = round_scaled_bits<NL>(X, si + tj[o]);
      }
    }
    if constexpr (!LIMBS) {
      double* dst = C + i * ldc + j0;
      if (j0 + 3 < N && (reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
        store4_f64(dst, outbits);
      } else {
#pragma unroll
        for (int o = 0; o < 4; ++o)
          if (j0 + o < N) __stcs(reinterpret_cast<unsigned long long*>(dst + o), outbits[o]);
      }
    }
  }
}

}  // namespace
}  // namespace ozk
