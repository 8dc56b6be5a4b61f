// Exponent scan and residue quantisation (the first two stages of the
// Ozaki-II pipeline on the "Day 12" page, section "Profile 不能只看 Tensor
// Core": "scale / exponent scan", "residue quantization"; the quantisation
// steps are the ones its section "為什麼 tile-local prologue 沒有直接贏" lists:
// double load, exponent scaling, round, mod, balanced int8 conversion).
//
// All arithmetic on the operands is integer work on IEEE-754 bit patterns:
// GB300's FP64 pipe is slow, and rounding m * 2^sh to an integer is a shift
// plus a rounding increment.  The scan and the quantisation each cover A and
// B in one launch; a third kernel scans and quantises rows of A in one pass
// where a row fits one block.
#include <map>
#include <mutex>

#include "ozk_internal.h"

namespace ozk {
namespace {

constexpr uint64_t kAbsMask = 0x7FFFFFFFFFFFFFFFull;
constexpr uint64_t kInfBits = 0x7FF0000000000000ull;
constexpr int kScanThreads = 256;
constexpr int kQThreads = 256;
constexpr int kQK = 16;  // K elements per quantisation thread: one 32-byte store per modulus
constexpr int kMaxBudget = 94;  // |a'| <= 2^94 fits the three-word form

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = umax64(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 32 bytes (four doubles' bit patterns) from a 32-byte aligned address.
__device__ __forceinline__ void load4_u64(const double* p, uint64_t (&v)[4]) {
  asm volatile("ld.global.nc.L1::no_allocate.v4.u64 {%0, %1, %2, %3}, [%4];"
               : "=l"(v[0]), "=l"(v[1]), "=l"(v[2]), "=l"(v[3])
               : "l"(p));
}

__device__ __forceinline__ uint64_t load1_u64(const double* p) {
  return static_cast<uint64_t>(__double_as_longlong(__ldg(p)));
}

// ---------------------------------------------------------------------------
// Exponent scan.  For non-negative doubles the bit pattern orders like the
// value, so max |x| is a max over 63-bit integers; Inf/NaN sort above every
// finite value.  Blocks [0, a_blocks) scan rows of A (one warp per row
// segment), the rest scan columns of B (32 threads of 1 or 4 columns each, 8
// row groups over a row segment, reduced in shared memory); partial maxima
// meet in amax through 64-bit atomicMax.
//
// The norm pass (NORM, the scaling from a computed 2-norm bound) runs the
// same walk once the maxima are in: every nonzero entry adds
// 2^max(h - H + W, 0) with h = floor(2 log2 |x|) and H that of the row's
// (column's) largest entry, an exact integer sum (at most 2^30 per entry,
// 2^52 per row), gathered with 64-bit atomicAdd into nsum.  Integers only, so
// the sum, and the scale derived from it, do not depend on the order.
// ---------------------------------------------------------------------------
constexpr int kNormWindow = 30;  // half-octaves below the largest entry that are counted exactly
constexpr uint64_t kFracMask = (1ull << 52) - 1;
// 1 + f / 2^52 >= sqrt(2) exactly when the 52 fraction bits f reach this value:
// (2^52 + f)^2 >= 2^105, and 2^105 is not a square
constexpr uint64_t kHalfOctaveFrac = 0x6A09E667F3BCDull;
static_assert((static_cast<unsigned __int128>(kHalfOctaveFrac + (1ull << 52)) * (kHalfOctaveFrac + (1ull << 52)) >
               (static_cast<unsigned __int128>(1) << 105)) &&
                  (static_cast<unsigned __int128>(kHalfOctaveFrac - 1 + (1ull << 52)) *
                       (kHalfOctaveFrac - 1 + (1ull << 52)) <
                   (static_cast<unsigned __int128>(1) << 105)),
              "the half-octave threshold is the first significand at or above sqrt(2)");

// floor(2 log2 |x|) for the bit pattern b of a finite nonzero |x|: with
// |x| = 1.f 2^e, 2e plus one when 1.f >= sqrt(2) (subnormals normalised first).
__device__ __forceinline__ int half_octave(uint64_t b) {
  const int ex = static_cast<int>(b >> 52);
  int e;
  uint64_t frac;
  if (ex) {
    e = ex - 1023;
    frac = b & kFracMask;
  } else {
    const int lz = __clzll(static_cast<long long>(b));
    e = (63 - lz) - 1074;
    frac = (b << (lz - 11)) & kFracMask;
  }
  return 2 * e + (frac >= kHalfOctaveFrac ? 1 : 0);
}

// An entry's part of the norm sum, given H of its row's (column's) maximum.
__device__ __forceinline__ uint64_t norm_part(uint64_t b, int H) {
  if (b == 0) return 0;
  const int d = half_octave(b) - H + kNormWindow;  // at most kNormWindow for a finite row
  return 1ull << (d > 0 ? (d < 62 ? d : 62) : 0);  // (a row with Inf/NaN ignores its sum)
}

struct ScanParams {
  const double* A;
  const double* B;
  int64_t lda, ldb, M, N, K;
  int64_t a_seg, a_segs, a_blocks;  // rows: 8 per block, a_segs segments of a_seg
  int64_t b_seg, b_segs, b_cols;    // columns per block = 32 * b_cols, rows per block = b_seg
  int a_vec, b_vec;                 // 32-byte loads possible
  uint64_t* amax;                   // [M + N]
  uint64_t* nsum;                   // [M + N], the norm pass only
};

// max of abs bit patterns, or (NORM) the sum of the entries' norm parts
template <bool NORM>
__device__ __forceinline__ uint64_t fold(uint64_t acc, uint64_t bits, int H) {
  return NORM ? acc + norm_part(bits & kAbsMask, H) : umax64(acc, bits & kAbsMask);
}

template <bool NORM>
__device__ __forceinline__ uint64_t warp_fold(uint64_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = NORM ? v + w : umax64(v, w);
  }
  return v;
}

// H of a row or column from its scanned maximum (unused for an all-zero or
// non-finite one: their scale does not depend on the sum)
__device__ __forceinline__ int max_half_octave(uint64_t amax) {
  return (amax == 0 || amax >= kInfBits) ? 0 : half_octave(amax);
}

template <bool NORM>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const ScanParams sp) {
  grid_dependency_sync();
  const int64_t bid = blockIdx.x;
  if (bid < sp.a_blocks) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (bid / sp.a_segs) * 8 + warp;
    if (row >= sp.M) return;
    const int H = NORM ? max_half_octave(sp.amax[row]) : 0;
    const int64_t k0 = (bid % sp.a_segs) * sp.a_seg;
    const int64_t k1 = min(sp.K, k0 + sp.a_seg);
    const double* a = sp.A + row * sp.lda;
    uint64_t m = 0;
    if (sp.a_vec) {  // a_seg is a multiple of 4: every group of 4 starts 32-byte aligned
      const int64_t g1 = k1 >> 2;
#pragma unroll 8  // eight 32-byte loads in flight per lane
      for (int64_t g = (k0 >> 2) + lane; g < g1; g += 32) {
        uint64_t v[4];
        load4_u64(a + 4 * g, v);
        m = fold<NORM>(fold<NORM>(m, v[0], H), v[1], H);
        m = fold<NORM>(fold<NORM>(m, v[2], H), v[3], H);
      }
      for (int64_t k = (g1 << 2) + lane; k < k1; k += 32) m = fold<NORM>(m, load1_u64(a + k), H);
    } else {
#pragma unroll 4
      for (int64_t k = k0 + lane; k < k1; k += 32) m = fold<NORM>(m, load1_u64(a + k), H);
    }
    m = warp_fold<NORM>(m);
    if (lane == 0 && m) {
      if (NORM)
        atomicAdd(reinterpret_cast<unsigned long long*>(sp.nsum + row), m);
      else
        atomicMax(reinterpret_cast<unsigned long long*>(sp.amax + row), m);
    }
  } else {
    // A block of B: 32 column threads (b_cols columns each) x 8 row groups
    // over a row segment; the row groups meet in shared memory, so each
    // column takes one atomic per block.
    __shared__ uint64_t red[kScanThreads / 32][32 * 4];
    const int64_t b = bid - sp.a_blocks;
    const int64_t cgrp = b / sp.b_segs;
    const int64_t k0 = (b % sp.b_segs) * sp.b_seg;
    const int64_t k1 = min(sp.K, k0 + sp.b_seg);
    const int lane = threadIdx.x & 31, rg = threadIdx.x >> 5;
    constexpr int kRowGroups = kScanThreads / 32;
    const int64_t c = (cgrp * 32 + lane) * sp.b_cols;
    uint64_t m[4] = {0, 0, 0, 0};
    int H[4] = {0, 0, 0, 0};
    if (NORM) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < sp.b_cols && c + j < sp.N) H[j] = max_half_octave(sp.amax[sp.M + c + j]);
    }
    if (c < sp.N) {
      if (sp.b_vec && c + 3 < sp.N) {
#pragma unroll 8  // eight 32-byte loads in flight per thread (4 measured 10% slower at 4096^3)
        for (int64_t k = k0 + rg; k < k1; k += kRowGroups) {
          uint64_t v[4];
          load4_u64(sp.B + k * sp.ldb + c, v);
#pragma unroll
          for (int j = 0; j < 4; ++j) m[j] = fold<NORM>(m[j], v[j], H[j]);
        }
      } else {
        for (int j = 0; j < 4 && j < sp.b_cols && c + j < sp.N; ++j) {
#pragma unroll 4
          for (int64_t k = k0 + rg; k < k1; k += kRowGroups)
            m[j] = fold<NORM>(m[j], load1_u64(sp.B + k * sp.ldb + c + j), H[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) red[rg][lane * 4 + j] = m[j];
    __syncthreads();
    if (rg == 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint64_t v = red[0][lane * 4 + j];
#pragma unroll
        for (int g = 1; g < kRowGroups; ++g) v = NORM ? v + red[g][lane * 4 + j] : umax64(v, red[g][lane * 4 + j]);
        if (v && j < sp.b_cols && c + j < sp.N) {
          if (NORM)
            atomicAdd(reinterpret_cast<unsigned long long*>(sp.nsum + sp.M + c + j), v);
          else
            atomicMax(reinterpret_cast<unsigned long long*>(sp.amax + sp.M + c + j), v);
        }
      }
    }
  }
}

// s = beta - E with max|x| = f 2^E, f in [0.5, 1) (frexp's exponent, read off
// the bits of the maximum b; subnormals via the leading-zero count).
__device__ __forceinline__ int32_t scale_of_max(uint64_t b, int beta) {
  if (b >= kInfBits) return OZK_SCALE_NONFINITE;
  if (b == 0) return 0;
  const int ex = static_cast<int>(b >> 52);
  const int E = ex ? ex - 1022 : (63 - __clzll(static_cast<long long>(b))) - 1073;
  return beta - E;
}

// The scale of the norm rule from the row's (column's) maximum and norm sum S:
// ||x||^2 < S 2^(H + 1 - W), and s = floor((2 gamma - (H + 1 - W) - ceil(log2 S)) / 2)
// keeps 2^(2s) S 2^(H + 1 - W) <= 2^(2 gamma).
__device__ __forceinline__ int32_t scale_of_norm(uint64_t amax, uint64_t S, int gamma) {
  if (amax >= kInfBits) return OZK_SCALE_NONFINITE;
  if (amax == 0) return 0;
  const int H = half_octave(amax);
  const int c = S <= 1 ? 0 : 64 - __clzll(static_cast<long long>(S - 1));  // ceil(log2 S)
  const int num = 2 * gamma - (H + 1 - kNormWindow) - c;
  return num >= 0 ? num / 2 : -((-num + 1) / 2);
}

// budget is beta (largest-entry rule) or, with nsum, gamma (norm rule)
__device__ __forceinline__ int32_t scale_of(const uint64_t* amax, const uint64_t* nsum, int64_t idx, int budget) {
  return nsum ? scale_of_norm(amax[idx], nsum[idx], budget) : scale_of_max(amax[idx], budget);
}

__global__ void finalize_scales_kernel(const uint64_t* __restrict__ amax, const uint64_t* __restrict__ nsum,
                                       int64_t M, int64_t N, int budget, int32_t* __restrict__ s,
                                       int32_t* __restrict__ t) {
  grid_dependency_sync();
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= M + N) return;
  const int32_t r = scale_of(amax, nsum, idx, budget);
  if (idx < M)
    s[idx] = r;
  else
    t[idx - M] = r;
}

// ---------------------------------------------------------------------------
// Quantisation.  x = (-1)^neg m 2^e exactly (m < 2^53); with sh = e + s the
// integer is a' = (-1)^neg round(m 2^sh), rounded to nearest with ties to
// even (a shift and a rounding increment), |a'| <= 2^beta.  a' is kept offset
// to a non-negative integer, a'' = a' + 2^(32 NL - 1) < 2^(32 NL), as NL
// 32-bit words: the two's complement of a' modulo 2^(32 NL) with its top bit
// flipped (NL = 2 for beta <= 62, NL = 3 for beta <= 94, every budget there
// is).  Then, for every modulus,
//   a' + h = sum_b byte_b(a'') (2^8b mod p) + (h - 2^(32 NL - 1))   (mod p),
// with the bytes taken four at a time by 4-byte dot products (dp4a): one
// integer x < 4 NL * 255 * 254 + 2 p < 2^20, which a multiply-high by
// ceil(2^32 / p) divides exactly; x mod p minus h is the balanced residue.
// ---------------------------------------------------------------------------

template <int NL>
__device__ __forceinline__ void scale_round(uint64_t bits, int32_t sc, uint32_t (&l)[NL]) {
  const uint32_t ex = static_cast<uint32_t>(bits >> 52) & 0x7FFu;
  uint64_t m = bits & 0xFFFFFFFFFFFFFull;
  if (ex) m |= 1ull << 52;
  const int sh = static_cast<int>(ex ? ex : 1u) - 1075 + sc;
  uint64_t lo;
  uint32_t hi = 0;
  if (sh < 0) {
    if (sh > -64) {
      // round(m / 2^r), ties to even: add half - 1 and the kept lowest bit, shift
      const int r = -sh;
      const uint64_t lsb = (m >> r) & 1u;
      lo = (m + ((1ull << (r - 1)) - 1u) + lsb) >> r;
    } else {  // m 2^sh < 2^-11 rounds to 0
      lo = 0;
    }
  } else if (sh == 0) {
    lo = m;
  } else if (sh < 64) {
    lo = m << sh;
    hi = static_cast<uint32_t>(m >> (64 - sh));
  } else {
    lo = 0;
    hi = static_cast<uint32_t>(m << (sh - 64));
  }
  if (bits >> 63) {  // two's complement of the (hi:lo) magnitude
    hi = ~hi + (lo == 0 ? 1u : 0u);
    lo = 0ull - lo;
  }
  static_assert(NL == 2 || NL == 3, "two or three 32-bit words");
  l[0] = static_cast<uint32_t>(lo);
  l[1] = static_cast<uint32_t>(lo >> 32);
  if constexpr (NL == 2) {  // |a'| <= 2^62: the low word of the two's complement, + 2^63
    l[1] ^= 1u << 31;
  } else {  // |a'| <= 2^94: the 96-bit two's complement, + 2^95
    l[2] = hi ^ (1u << 31);
  }
}

// The four residues 2^(8 (b0 + i)) mod p, one per byte.
__host__ __device__ constexpr uint32_t byte_weights(int b0, uint32_t p) {
  return pow2_mod(8 * b0, p) | (pow2_mod(8 * b0 + 8, p) << 8) | (pow2_mod(8 * b0 + 16, p) << 16) |
         (pow2_mod(8 * b0 + 24, p) << 24);
}

// Canonical residue of a' + h for the k-th modulus (h = floor(p/2); the
// balanced residue is this minus h).
template <int k, int NL>
__device__ __forceinline__ uint32_t shifted_residue(const uint32_t (&l)[NL]) {
  constexpr uint32_t p = modulus_at(k);
  if constexpr (p == 256u) {
    return (l[0] ^ 0x80u) & 0xFFu;  // (a' + 128) mod 256 from the low byte
  } else {
    constexpr uint32_t h = (p - 1) / 2;
    // x = the bytes of a'' against 2^8b mod p, plus h - 2^(32 NL - 1) mod p:
    // x < 4 NL * 255 * 254 + 2 p < 2^20, where umulhi by ceil(2^32/p) is exact
    constexpr uint32_t off = (p - pow2_mod(32 * NL - 1, p)) % p + h;
    constexpr uint32_t m32 = static_cast<uint32_t>(((1ull << 32) + p - 1) / p);
    uint32_t x = __dp4a(l[1], byte_weights(4, p), __dp4a(l[0], byte_weights(0, p), off));
    if constexpr (NL == 3) x = __dp4a(l[2], byte_weights(8, p), x);
    return x - __umulhi(x, m32) * p;
  }
}

// fp16 bits 0x6600 + v are the value 1536 + v for |v| < 512 (fp16 steps by 1
// in [1024, 2048)); subtracting 1536 leaves v exactly.
constexpr uint32_t kHalfMagicBits = 0x6600u;
constexpr uint32_t kNegHalfMagic2 = 0xE600E600u;  // (-1536, -1536) as f16x2

// Two canonical residues of the k-th modulus to a packed pair of fp16
// balanced residues (exact integers in [-128, 127]).
template <int k>
__device__ __forceinline__ uint32_t pack_f16x2(uint32_t rlo, uint32_t rhi) {
  constexpr uint32_t p = modulus_at(k);
  constexpr uint32_t h = p == 256u ? 128u : (p - 1) / 2;
  constexpr uint32_t bias = (kHalfMagicBits - h) * 0x10001u;
  const uint32_t w = __byte_perm(rlo, rhi, 0x5410) + bias;  // (rhi << 16) | rlo, both < 2^16
  uint32_t out;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(out) : "r"(w), "r"(kNegHalfMagic2));
  return out;
}

__device__ __forceinline__ void store8_u32(uint16_t* dst, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

struct QuantParams {
  const double* A;
  const double* B;
  int32_t* s;  // scales of the rows of A: read, or written when a_amax is set
  int32_t* t;  // scales of the columns of B: read, or written when b_amax is set
  const uint64_t* a_amax;  // scanned maxima of the rows of A (the scale is derived here), or null
  const uint64_t* b_amax;  // the same for the columns of B
  const uint64_t* a_nsum;  // norm sums of the rows of A (the norm rule), or null (largest-entry rule)
  const uint64_t* b_nsum;  // the same for the columns of B
  int budget;              // beta, or gamma for the norm rule
  uint16_t* a_out;  // modulus k, row i at a_out + k * a_plane + i * kpad
  uint16_t* b_out;  // modulus k, column j at b_out + k * b_plane + j * kpad
  int64_t a_plane, b_plane;
  int64_t lda, ldb, M, N, K, kpad;
  int64_t groups;     // kpad / 16
  int64_t a_threads;  // M * groups
  int64_t a_span;     // a_threads rounded up to whole blocks; B threads follow
  int64_t b_threads;  // cgroups * ceil(groups / warps per block) blocks of threads
  int64_t cgroups;    // groups of 32 columns of B
  int n;
  int a_vec;  // rows of A are 32-byte aligned
};

// One thread: 16 consecutive K entries of one row of A (thread order: k fastest,
// so loads and stores of a warp are contiguous) or of one column of B.  For B
// a block is 32 columns x 8 consecutive 16-entry K groups, a warp 8 of the
// columns (lane % 8) x 4 consecutive K groups (lane / 8): each of its 16 row
// loads reads 64 contiguous bytes of 4 rows, and each store writes one whole
// 128-byte L2 line of each of its 8 columns' slice rows (a store of 32 columns
// x one K group, 32 pieces of 32 bytes, measured 2-4% slower over the stage at
// 4096^3 and 8192^3); consecutive blocks take the next 32 columns of the same
// 128 rows.  Each thread writes one 32-byte run of every modulus' slice.
template <int NL>
__global__ void __launch_bounds__(kQThreads) quantize_kernel(const QuantParams qp) {
  grid_dependency_sync();
  const int64_t g = static_cast<int64_t>(blockIdx.x) * kQThreads + threadIdx.x;
  uint64_t v[kQK];
  int64_t row, k0, plane;
  int32_t sc;
  uint16_t* out;
  if (g < qp.a_span) {
    if (g >= qp.a_threads) return;
    row = g / qp.groups;
    k0 = (g - row * qp.groups) * kQK;
    plane = qp.a_plane;
    out = qp.a_out;
    if (qp.a_amax) {  // the scale from the row's scanned maximum; the first thread of the row stores it
      sc = scale_of(qp.a_amax, qp.a_nsum, row, qp.budget);
      if (k0 == 0) qp.s[row] = sc;
    } else {
      sc = qp.s[row];
    }
    const double* a = qp.A + row * qp.lda + k0;
    if (qp.a_vec && k0 + kQK <= qp.K) {
#pragma unroll
      for (int e = 0; e < kQK / 4; ++e) {
        uint64_t w[4];
        load4_u64(a + 4 * e, w);
        v[4 * e] = w[0];
        v[4 * e + 1] = w[1];
        v[4 * e + 2] = w[2];
        v[4 * e + 3] = w[3];
      }
    } else {
#pragma unroll
      for (int e = 0; e < kQK; ++e) v[e] = (k0 + e < qp.K) ? load1_u64(a + e) : 0ull;
    }
  } else {
    const int64_t gb = g - qp.a_span;
    if (gb >= qp.b_threads) return;
    constexpr int kWarps = kQThreads / 32;
    const int64_t blk = gb / kQThreads;
    const int64_t cg = blk % qp.cgroups;
    const int t = static_cast<int>(gb % kQThreads), lane = t & 31, warp = t >> 5;
    const int64_t kg = (blk / qp.cgroups) * kWarps + (warp / 4) * 4 + lane / 8;
    row = cg * 32 + (warp % 4) * 8 + lane % 8;  // column j of B
    if (row >= qp.N || kg >= qp.groups) return;
    k0 = kg * kQK;
    plane = qp.b_plane;
    out = qp.b_out;
    if (qp.b_amax) {
      sc = scale_of(qp.b_amax, qp.b_nsum, row, qp.budget);
      if (k0 == 0) qp.t[row] = sc;
    } else {
      sc = qp.t[row];
    }
    const double* b = qp.B + k0 * qp.ldb + row;
#pragma unroll
    for (int e = 0; e < kQK; ++e) v[e] = (k0 + e < qp.K) ? load1_u64(b + e * qp.ldb) : 0ull;
  }
  if (sc == OZK_SCALE_NONFINITE) {
#pragma unroll
    for (int e = 0; e < kQK; ++e) v[e] = 0;
  }
  uint32_t x[kQK][NL];
#pragma unroll
  for (int e = 0; e < kQK; ++e) scale_round<NL>(v[e], sc, x[e]);
  uint16_t* dst = out + row * qp.kpad + k0;
  const int n = qp.n;
  static_for<0, kMaxModuli>([&](auto kc) {
    constexpr int k = decltype(kc)::value;
    if (k < n) {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        w[e] = pack_f16x2<k>(shifted_residue<k, NL>(x[2 * e]), shifted_residue<k, NL>(x[2 * e + 1]));
      store8_u32(dst + k * plane, w);
    }
  });
}

// Rows of A with the exponent scan fused in: one block per row (K up to
// kRowsMaxK), kQK consecutive entries per thread.  The row's max |a| is
// reduced in the block and turned into its scale while the entries are
// still in registers, so A is read once instead of twice; the quantisation
// itself is quantize_kernel's.
constexpr int kRowsMaxThreads = 256;
static_assert(kRowsMaxThreads % 32 == 0 && kRowsMaxThreads <= 1024, "whole warps");

template <int NL, bool NORM>
__global__ void __launch_bounds__(kRowsMaxThreads) quantize_rows_kernel(const QuantParams qp, int budget,
                                                                        int32_t* __restrict__ s_out) {
  grid_dependency_sync();
  __shared__ uint64_t wmax[kRowsMaxThreads / 32];
  const int64_t row = blockIdx.x;
  const int64_t k0 = static_cast<int64_t>(threadIdx.x) * kQK;
  const bool active = k0 < qp.kpad;  // the block is rounded up to whole warps
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t v[kQK];
  const double* a = qp.A + row * qp.lda + k0;
  if (active && qp.a_vec && k0 + kQK <= qp.K) {
#pragma unroll
    for (int e = 0; e < kQK / 4; ++e) {
      uint64_t w[4];
      load4_u64(a + 4 * e, w);
      v[4 * e] = w[0];
      v[4 * e + 1] = w[1];
      v[4 * e + 2] = w[2];
      v[4 * e + 3] = w[3];
    }
  } else {
#pragma unroll
    for (int e = 0; e < kQK; ++e) v[e] = (active && k0 + e < qp.K) ? load1_u64(a + e) : 0ull;
  }
  uint64_t m = 0;
#pragma unroll
  for (int e = 0; e < kQK; ++e) m = umax64(m, v[e] & kAbsMask);
  m = warp_max_u64(m);
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  m = 0;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) m = umax64(m, wmax[w]);
  int32_t sc;
  if constexpr (NORM) {  // the row's norm sum, reduced the same way
    const int H = max_half_octave(m);
    uint64_t part = 0;
#pragma unroll
    for (int e = 0; e < kQK; ++e) part += norm_part(v[e] & kAbsMask, H);
#pragma unroll
    for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    __syncthreads();  // every thread has read the maxima
    if (lane == 0) wmax[warp] = part;
    __syncthreads();
    uint64_t S = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) S += wmax[w];
    sc = scale_of_norm(m, S, budget);
  } else {
    sc = scale_of_max(m, budget);
  }
  if (threadIdx.x == 0) s_out[row] = sc;
  if (!active) return;
  if (sc == OZK_SCALE_NONFINITE) {
#pragma unroll
    for (int e = 0; e < kQK; ++e) v[e] = 0;
  }
  uint32_t x[kQK][NL];
#pragma unroll
  for (int e = 0; e < kQK; ++e) scale_round<NL>(v[e], sc, x[e]);
  uint16_t* dst = qp.a_out + row * qp.kpad + k0;
  const int n = qp.n;
  static_for<0, kMaxModuli>([&](auto kc) {
    constexpr int k = decltype(kc)::value;
    if (k < n) {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        w[e] = pack_f16x2<k>(shifted_residue<k, NL>(x[2 * e]), shifted_residue<k, NL>(x[2 * e + 1]));
      store8_u32(dst + k * qp.a_plane, w);
    }
  });
}

}  // namespace

cudaError_t launch_scan(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
                        int64_t ldb, uint64_t* amax, uint64_t* nsum, cudaStream_t stream) {
  if (M + N == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint64_t) * static_cast<size_t>(M + N), stream);
  if (e != cudaSuccess) return e;
  if (nsum && (e = cudaMemsetAsync(nsum, 0, sizeof(uint64_t) * static_cast<size_t>(M + N), stream)) != cudaSuccess)
    return e;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = kNumSmsFallback;
  ScanParams sp;
  sp.A = A;
  sp.B = B;
  sp.lda = lda;
  sp.ldb = ldb;
  sp.M = M;
  sp.N = N;
  sp.K = K;
  sp.amax = amax;
  sp.nsum = nsum;
  sp.a_vec = (reinterpret_cast<uintptr_t>(A) % 32 == 0) && (lda % 4 == 0);
  sp.b_vec = (reinterpret_cast<uintptr_t>(B) % 32 == 0) && (ldb % 4 == 0);
  sp.a_seg = sp.a_segs = sp.a_blocks = 0;
  sp.b_seg = sp.b_segs = 1;
  sp.b_cols = sp.b_vec ? 4 : 1;
  int64_t b_blocks = 0;
  if (K > 0 && M > 0) {
    const int64_t target_warps = static_cast<int64_t>(sms) * 64;
    int64_t segs = (target_warps + M - 1) / M;
    int64_t seg = (K + segs - 1) / segs;
    seg = ((seg + 255) / 256) * 256;
    sp.a_seg = seg;
    sp.a_segs = (K + seg - 1) / seg;
    sp.a_blocks = ((M + 7) / 8) * sp.a_segs;
  }
  if (K > 0 && N > 0) {
    const int64_t cgroups = (N + 32 * sp.b_cols - 1) / (32 * sp.b_cols);
    int64_t segs = (static_cast<int64_t>(sms) * 4 + cgroups - 1) / cgroups;
    int64_t seg = (K + segs - 1) / segs;
    seg = seg < 64 ? 64 : ((seg + 7) / 8) * 8;
    sp.b_seg = seg;
    sp.b_segs = (K + seg - 1) / seg;
    b_blocks = cgroups * sp.b_segs;
  }
  const int64_t blocks = sp.a_blocks + b_blocks;
  if (blocks > 0) {
    if ((e = launch_dependent(scan_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(kScanThreads), 0, stream,
                              sp)) != cudaSuccess)
      return e;
    if (nsum &&  // the norm pass, once every maximum is in
        (e = launch_dependent(scan_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(kScanThreads), 0, stream,
                              sp)) != cudaSuccess)
      return e;
  }
  return cudaSuccess;
}

cudaError_t launch_scale(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                         const double* B, int64_t ldb, int budget, int32_t* s, int32_t* t,
                         uint64_t* amax, uint64_t* nsum, cudaStream_t stream) {
  if (M + N == 0) return cudaSuccess;
  cudaError_t e = launch_scan(M, N, K, A, lda, B, ldb, amax, nsum, stream);
  if (e != cudaSuccess) return e;
  return launch_dependent(finalize_scales_kernel, dim3(static_cast<unsigned>((M + N + 255) / 256)), dim3(256), 0,
                          stream, amax, nsum, M, N, budget, s, t);
}

cudaError_t launch_quantize(int64_t M, int64_t N, int64_t K, int64_t kpad, const double* A,
                            int64_t lda, const double* B, int64_t ldb, int32_t* s, int32_t* t,
                            const uint64_t* a_amax, const uint64_t* b_amax, const uint64_t* a_nsum,
                            const uint64_t* b_nsum, int n, int budget, uint16_t* a_out, int64_t a_plane,
                            uint16_t* b_out, int64_t b_plane, cudaStream_t stream) {
  if (kpad == 0 || (M == 0 && N == 0)) return cudaSuccess;
  QuantParams qp;
  qp.A = A;
  qp.B = B;
  qp.s = s;
  qp.t = t;
  qp.a_amax = a_amax;
  qp.b_amax = b_amax;
  qp.a_nsum = a_nsum;
  qp.b_nsum = b_nsum;
  qp.budget = budget;
  qp.a_out = a_out;
  qp.b_out = b_out;
  qp.a_plane = a_plane;
  qp.b_plane = b_plane;
  qp.lda = lda;
  qp.ldb = ldb;
  qp.M = A ? M : 0;
  qp.N = B ? N : 0;
  qp.K = K;
  qp.kpad = kpad;
  qp.groups = kpad / kQK;
  qp.a_threads = qp.M * qp.groups;
  qp.a_span = (qp.a_threads + kQThreads - 1) / kQThreads * kQThreads;
  qp.cgroups = (qp.N + 31) / 32;
  qp.b_threads = qp.cgroups * ((qp.groups + kQThreads / 32 - 1) / (kQThreads / 32)) * kQThreads;
  qp.n = n;
  qp.a_vec = A && (reinterpret_cast<uintptr_t>(A) % 32 == 0) && (lda % 4 == 0);
  const int64_t threads = qp.a_span + qp.b_threads;
  if (threads == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((threads + kQThreads - 1) / kQThreads);
  // |a'| <= 2^budget: two 32-bit words of two's complement for a budget of
  // at most 62, three beyond
  if (budget > kMaxBudget) return cudaErrorInvalidValue;
  if (budget <= 62) return launch_dependent(quantize_kernel<2>, dim3(blocks), dim3(kQThreads), 0, stream, qp);
  return launch_dependent(quantize_kernel<3>, dim3(blocks), dim3(kQThreads), 0, stream, qp);
}

bool quantize_rows_fits(int64_t kpad) { return kpad / kQK <= kRowsMaxThreads; }

cudaError_t launch_quantize_rows(int64_t M, int64_t K, int64_t kpad, const double* A, int64_t lda, int n,
                                 int budget, bool norm, int32_t* s, uint16_t* a_out, int64_t a_plane,
                                 cudaStream_t stream) {
  if (M == 0 || kpad == 0) return cudaSuccess;
  if (!quantize_rows_fits(kpad) || M > 0x7FFFFFFF) return cudaErrorInvalidValue;
  QuantParams qp = {};
  qp.A = A;
  qp.a_out = a_out;
  qp.a_plane = a_plane;
  qp.lda = lda;
  qp.M = M;
  qp.K = K;
  qp.kpad = kpad;
  qp.n = n;
  qp.a_vec = (reinterpret_cast<uintptr_t>(A) % 32 == 0) && (lda % 4 == 0);
  const unsigned threads = static_cast<unsigned>((kpad / kQK + 31) / 32 * 32);
  const unsigned blocks = static_cast<unsigned>(M);
  if (budget > kMaxBudget) return cudaErrorInvalidValue;
  const dim3 grid(blocks), block(threads);
  if (budget <= 62)
    return norm ? launch_dependent(quantize_rows_kernel<2, true>, grid, block, 0, stream, qp, budget, s)
                : launch_dependent(quantize_rows_kernel<2, false>, grid, block, 0, stream, qp, budget, s);
  return norm ? launch_dependent(quantize_rows_kernel<3, true>, grid, block, 0, stream, qp, budget, s)
              : launch_dependent(quantize_rows_kernel<3, false>, grid, block, 0, stream, qp, budget, s);
}

}  // namespace ozk

// ---------------------------------------------------------------------------
// The exponent scan without caller-provided scratch.
//
// ozk_scale needs (M + N) uint64 of device scratch for the running maxima.
// Some callers cannot hand over device memory they did not plan for: a
// library embedded in a host application whose allocator owns every device
// byte, or a latency-critical loop that must not call cudaMalloc (which can
// synchronise the device).  ozk_scale_noalloc keeps that scratch in a
// fixed array compiled into the library instead.  Every GPU that loads the
// library holds the array (2 MiB) until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint64_t g_noalloc_amax[OZK_SCALE_NOALLOC_MAX];

namespace ozk {
namespace {

std::mutex g_noalloc_mutex;
std::map<int, uint64_t*> g_noalloc_ptr;  // device -> device address of g_noalloc_amax

// The device address of the fixed scratch on the current device.  The name
// g_noalloc_amax in host code is only a host-side stand-in; the address is
// looked up once per device, with that device current.
int noalloc_scratch(uint64_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  auto it = g_noalloc_ptr.find(dev);
  if (it == g_noalloc_ptr.end()) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_amax) != cudaSuccess || p == nullptr) return OZK_ERR_CUDA;
    it = g_noalloc_ptr.emplace(dev, static_cast<uint64_t*>(p)).first;
  }
  *out = it->second;
  return OZK_OK;
}

}  // namespace
}  // namespace ozk

extern "C" int ozk_scale_noalloc(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                                 const double* B, int64_t ldb, int n_moduli, int32_t* s, int32_t* t,
                                 ozk_stream_t stream) {
  using namespace ozk;
  if (M < 0 || N < 0 || K < 0) return OZK_ERR_INVALID_ARG;
  const int beta = beta_for(K, n_moduli);
  if (beta < 1 || K > OZK_MAX_K) return OZK_ERR_UNSUPPORTED;
  // beyond the fixed scratch (compared without forming M + N, which could overflow)
  if (M > OZK_SCALE_NOALLOC_MAX || N > OZK_SCALE_NOALLOC_MAX - M) return OZK_ERR_WORKSPACE;
  if (M + N == 0) return OZK_OK;
  if ((M && !s) || (N && !t)) return OZK_ERR_INVALID_ARG;
  if (K > 0 && ((M && (!A || lda < K)) || (N && (!B || ldb < N)))) return OZK_ERR_INVALID_ARG;
  int rc = current_device_supported(nullptr);
  if (rc) return rc;
  uint64_t* amax = nullptr;
  if ((rc = noalloc_scratch(&amax))) return rc;
  // launch_scale zeroes the M + N maxima it uses before the scan, so the
  // contents left by an earlier call do not matter
  if (launch_scale(M, N, K, A, lda, B, ldb, beta, s, t, amax, nullptr, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return OZK_ERR_CUDA;
  return OZK_OK;
}
