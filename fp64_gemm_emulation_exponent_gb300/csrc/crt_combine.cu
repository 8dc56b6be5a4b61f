// CRT reconstruction, symmetric lift, undo scaling and FP64 write (the last
// three stages of the Ozaki-II pipeline on the "Day 12" page, section
// "Profile 不能只看 Tensor Core").  That page's section "Combine kernel
// 的瓶頸又不一樣" measures its own combine at ~85% of the FP64 pipe and warns
// that more registers per thread made it slower; on GB300 the FP64 pipe is
// slow, so this kernel is integer-only:
//
//   X = sum_k y_k (P/p_k) - q P,  y_k = c_k w_k,  w_k = (P/p_k)^-1 mod p_k,
//
// with y_k left unreduced (< 2^16), the limb sums accumulated in 64 bits
// without carries, and q = round(sum_k y_k / p_k) estimated in 32.32 fixed
// point (error < 2^20 / 2^32); the rare outputs whose estimate lies within
// 2^21 of a rounding boundary get an exact correction.  The lifted X in
// [-P/2, P/2) is then scaled by 2^-(s_i + t_j) and rounded to nearest-even in
// integer arithmetic (subnormals and overflow included).
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

// One thread per 4 consecutive columns of one row.
//  IN_KIND 0: uint8 residues [n][M][ldi];  1: int32 partial sums [splits][n][M][ldi].
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

  uint64_t acc[4][NL];
  uint64_t qacc[4];
#pragma unroll
  for (int o = 0; o < 4; ++o) {
    qacc[o] = 0;
#pragma unroll
    for (int l = 0; l < NL; ++l) acc[o][l] = 0;
  }

  static_for<0, kMaxModuli>([&](auto kc) {
    constexpr int k = decltype(kc)::value;
    if (k < n) {
      uint32_t c[4];
      if constexpr (IN_KIND == 0) {
        const uint8_t* plane = static_cast<const uint8_t*>(in) + (static_cast<int64_t>(k) * M + i) * ldi + j0;
        const uint32_t w4 = __ldcs(reinterpret_cast<const unsigned int*>(plane));
#pragma unroll
        for (int o = 0; o < 4; ++o) c[o] = (w4 >> (8 * o)) & 0xFFu;
      } else {
        int32_t sum[4] = {0, 0, 0, 0};
        for (int sp = 0; sp < splits; ++sp) {
          const int32_t* row = static_cast<const int32_t*>(in) +
                               ((static_cast<int64_t>(sp) * n + k) * M + i) * ldi + j0;
          const int4 v = __ldcs(reinterpret_cast<const int4*>(row));
          sum[0] += v.x;
          sum[1] += v.y;
          sum[2] += v.z;
          sum[3] += v.w;
        }
#pragma unroll
        for (int o = 0; o < 4; ++o) c[o] = mod_p(sum[o], K.p[k], K.magic[k], K.bias[k]);
      }
#pragma unroll
      for (int o = 0; o < 4; ++o) {
        const uint32_t y = c[o] * K.w[k];  // < 2^16
        qacc[o] += static_cast<uint64_t>(y) * K.r32[k];
#pragma unroll
        for (int l = 0; l < NL; ++l) acc[o][l] += static_cast<uint64_t>(y) * K.Mk[k][l];
      }
    }
  });

  const int32_t si = s ? s[i] : 0;
#pragma unroll
  for (int o = 0; o < 4; ++o) {
    const int64_t j = j0 + o;
    if (j >= N) break;
    // S = sum_k y_k P/p_k as NL 32-bit limbs
    uint32_t X[NL];
    uint64_t carry = 0;
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      const uint64_t v = acc[o][l] + carry;
      X[l] = static_cast<uint32_t>(v);
      carry = v >> 32;
    }
    // q = round(S / P) from the fixed-point estimate; X = S - q P
    const uint64_t shifted = qacc[o] + 0x80000000ull;
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
    if (frac < (1u << 21) || frac > ~(1u << 21)) exact_lift<NL>(X, K);

    if constexpr (LIMBS) {
      uint32_t* dst = Xout + (i * N + j) * OZK_LIMBS;
      const uint32_t ext = is_negative<NL>(X) ? 0xFFFFFFFFu : 0u;
#pragma unroll
      for (int l = 0; l < OZK_LIMBS; ++l) dst[l] = l < NL ? X[l] : ext;
    } else {
      const int32_t tj = t[j];
      uint64_t bits;
      if (si == OZK_SCALE_NONFINITE || tj == OZK_SCALE_NONFINITE)
        bits = kQuietNaN;
      else
        bits = round_scaled_bits<NL>(X, si + tj);
      __stcs(reinterpret_cast<unsigned long long*>(C + i * ldc + j), bits);
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
