// CRT reconstruction, symmetric lift, undo scaling and FP64 write (the last
// three stages of the Ozaki-II pipeline on the "Day 12" page, section
// "Profile 不能只看 Tensor Core").  That page's section "Combine kernel
// 的瓶頸又不一樣" measures its own combine at ~85% of the FP64 pipe and warns
// that more registers per thread made it slower; on GB300 the FP64 pipe is
// slow, so this kernel is integer-only:
//
//   X = sum_k c_k e_k - q P,  e_k = (P/p_k) ((P/p_k)^-1 mod p_k),
//
// with the column sums of c_k e_k accumulated in 64 bits without carries, and
// q = round(sum_k c_k w_k / p_k) estimated in 32.32 fixed point (error below
// 2^12 / 2^32); the rare outputs whose estimate lies within 2^14 / 2^32 of a
// rounding boundary get an exact correction.  The lifted X in [-P/2, P/2) is
// then scaled by 2^-(s_i + t_j) and rounded to nearest-even in integer
// arithmetic (subnormals and overflow included).
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

// RN-even double of X * 2^-S for a two's-complement NL-limb integer X.
template <int NL>
__device__ __forceinline__ uint64_t round_scaled_bits(const uint32_t (&X)[NL], int S) {
  const bool neg = is_negative<NL>(X);
  uint32_t m[NL];
  uint64_t c = 1;
#pragma unroll
  for (int l = 0; l < NL; ++l) {
    if (neg) {
      const uint64_t v = static_cast<uint64_t>(~X[l]) + c;
      m[l] = static_cast<uint32_t>(v);
      c = v >> 32;
    } else {
      m[l] = X[l];
    }
  }
  int top = -1;
#pragma unroll
  for (int l = 0; l < NL; ++l)
    if (m[l]) top = l;
  if (top < 0) return 0ull;  // exact zero: +0
  uint32_t w2 = 0, w1 = 0, w0 = 0, below = 0;
#pragma unroll
  for (int l = 0; l < NL; ++l) {
    w2 = (l == top) ? m[l] : w2;
    w1 = (l == top - 1) ? m[l] : w1;
    w0 = (l == top - 2) ? m[l] : w0;
    below |= (l < top - 2) ? m[l] : 0u;
  }
  const int lz = __clz(w2);
  const uint64_t hi = (static_cast<uint64_t>(w2) << 32) | w1;
  const uint64_t win = lz ? (hi << lz) | (static_cast<uint64_t>(w0) >> (32 - lz)) : hi;
  uint32_t sticky = below | (lz ? (w0 << lz) : w0);  // bits below the 64-bit window
  const int h = 32 * top + 31 - lz;                   // leading bit of |X|
  const int e = h - S;                                // |X| 2^-S in [2^e, 2^(e+1))
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
      st = ((win << 1) != 0) | (sticky != 0);
    } else {
      q = win >> sh;
      rb = static_cast<uint32_t>(win >> (sh - 1)) & 1u;
      st = ((win & ((1ull << (sh - 1)) - 1)) != 0) | (sticky != 0);
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

__device__ __forceinline__ void store4_f64(double* dst, const uint64_t (&b)[4]) {
  asm volatile("st.global.cs.v4.b64 [%0], {%1, %2, %3, %4};" ::"l"(dst), "l"(b[0]), "l"(b[1]), "l"(b[2]),
               "l"(b[3])
               : "memory");
}

// One thread per 4 consecutive columns of one row.
//  IN_KIND 0: uint8 residues [n][M][ldi];  1: int32 partial sums [splits][n][M][ldi].
// All residue words are loaded before any arithmetic so that the loads of a
// thread are in flight together.
template <int NL, int IN_KIND, bool LIMBS>
__global__ void __launch_bounds__(256) crt_kernel(const void* __restrict__ in, int64_t ldi,
                                                  int64_t M, int64_t N, int splits,
                                                  const int32_t* __restrict__ s,
                                                  const int32_t* __restrict__ t,
                                                  double* __restrict__ C, int64_t ldc,
                                                  uint32_t* __restrict__ Xout, const CrtConst K) {
  const int64_t groups = (N + 3) >> 2;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= M * groups) return;
  const int64_t i = g / groups;
  const int64_t j0 = (g - i * groups) * 4;
  const int n = K.n;

  // canonical residues of the 4 outputs, 4 bytes per modulus
  uint32_t cw[kMaxModuli];
  if constexpr (IN_KIND == 0) {
    const uint8_t* base = static_cast<const uint8_t*>(in) + i * ldi + j0;
    const int64_t plane = M * ldi;
    static_for<0, kMaxModuli>([&](auto kc) {
      constexpr int k = decltype(kc)::value;
      if (k < n) cw[k] = __ldcs(reinterpret_cast<const unsigned int*>(base + k * plane));
    });
  } else {
    static_for<0, kMaxModuli>([&](auto kc) {
      constexpr int k = decltype(kc)::value;
      if (k < n) {
        int32_t sum[4] = {0, 0, 0, 0};
        for (int sp = 0; sp < splits; ++sp) {
          const int4 v = __ldcs(reinterpret_cast<const int4*>(static_cast<const int32_t*>(in) +
                                                              ((static_cast<int64_t>(sp) * n + k) * M + i) * ldi + j0));
          sum[0] += v.x;
          sum[1] += v.y;
          sum[2] += v.z;
          sum[3] += v.w;
        }
        cw[k] = mod_p(sum[0], K.p[k], K.magic[k], K.bias[k]) |
                (mod_p(sum[1], K.p[k], K.magic[k], K.bias[k]) << 8) |
                (mod_p(sum[2], K.p[k], K.magic[k], K.bias[k]) << 16) |
                (mod_p(sum[3], K.p[k], K.magic[k], K.bias[k]) << 24);
      }
    });
  }
  int32_t si = 0;
  int32_t tj[4] = {0, 0, 0, 0};
  if constexpr (!LIMBS) {
    si = s[i];
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
#pragma unroll
  for (int o = 0; o < 4; ++o) {
    // S = sum_k c_k e_k (64-bit column sums, carries later) and
    // q ~ S / P = sum_k c_k w_k / p_k in 32.32 fixed point
    uint64_t acc[NL];
#pragma unroll
    for (int l = 0; l < NL; ++l) acc[l] = 0;
    uint64_t qacc = 0;
    static_for<0, kMaxModuli>([&](auto kc) {
      constexpr int k = decltype(kc)::value;
      if (k < n) {
        const uint32_t c = __byte_perm(cw[k], 0u, 0x4440 + o);
        qacc += static_cast<uint64_t>(c) * K.frac[k];
#pragma unroll
        for (int l = 0; l < NL; ++l) acc[l] += static_cast<uint64_t>(c) * K.e[k][l];
      }
    });
    uint32_t X[NL];
    uint64_t carry = 0;
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      const uint64_t v = acc[l] + carry;
      X[l] = static_cast<uint32_t>(v);
      carry = v >> 32;
    }
    // X = S - q P with q = round(S / P); the estimate is off by less than
    // 2^12 / 2^32, so only outputs within 2^14 / 2^32 of a rounding boundary
    // need the exact check
    const uint64_t shifted = qacc + 0x80000000ull;
    const uint32_t q = static_cast<uint32_t>(shifted >> 32);
    const uint32_t frac = static_cast<uint32_t>(shifted);
    uint64_t borrow = 0;
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      const uint64_t sub = static_cast<uint64_t>(q) * K.P[l] + borrow;
      const uint32_t lo = static_cast<uint32_t>(sub);
      borrow = (sub >> 32) + (X[l] < lo ? 1u : 0u);
      X[l] -= lo;
    }
    if (frac < (1u << 14) || frac > ~(1u << 14)) exact_lift<NL>(X, K);

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
      else
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

template <int NL>
cudaError_t launch_nl(int64_t M, int64_t N, const void* in, int in_kind, int64_t ldi, int splits,
                      const int32_t* s, const int32_t* t, double* C, int64_t ldc, uint32_t* X,
                      const CrtConst& K, cudaStream_t stream) {
  const int64_t threads = M * ((N + 3) / 4);
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  if (in_kind == 0) {
    if (X)
      crt_kernel<NL, 0, true><<<blocks, 256, 0, stream>>>(in, ldi, M, N, splits, s, t, C, ldc, X, K);
    else
      crt_kernel<NL, 0, false><<<blocks, 256, 0, stream>>>(in, ldi, M, N, splits, s, t, C, ldc, X, K);
  } else {
    if (X)
      crt_kernel<NL, 1, true><<<blocks, 256, 0, stream>>>(in, ldi, M, N, splits, s, t, C, ldc, X, K);
    else
      crt_kernel<NL, 1, false><<<blocks, 256, 0, stream>>>(in, ldi, M, N, splits, s, t, C, ldc, X, K);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_crt(int64_t M, int64_t N, int n, const void* in, int in_kind, int64_t ldi,
                       int splits, const int32_t* s, const int32_t* t, double* C, int64_t ldc,
                       uint32_t* X, cudaStream_t stream) {
  if (M == 0 || N == 0) return cudaSuccess;
  const CrtConst& K = crt_const(n);
  switch (crt_limbs(n)) {
    case 3: return launch_nl<3>(M, N, in, in_kind, ldi, splits, s, t, C, ldc, X, K, stream);
    case 4: return launch_nl<4>(M, N, in, in_kind, ldi, splits, s, t, C, ldc, X, K, stream);
    case 5: return launch_nl<5>(M, N, in, in_kind, ldi, splits, s, t, C, ldc, X, K, stream);
    case 6: return launch_nl<6>(M, N, in, in_kind, ldi, splits, s, t, C, ldc, X, K, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ozk
