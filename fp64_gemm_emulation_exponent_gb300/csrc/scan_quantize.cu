// Exponent scan and residue quantisation (the first two stages of the
// Ozaki-II pipeline on the "Day 12" page, section "Profile 不能只看 Tensor
// Core": "scale / exponent scan", "residue quantization"; the quantisation
// steps are the ones its section "為什麼 tile-local prologue 沒有直接贏" lists:
// double load, exponent scaling, round, mod, balanced int8 conversion).
//
// All arithmetic on the operands is integer work on IEEE-754 bit patterns:
// GB300's FP64 pipe is slow, and rounding m * 2^sh to an integer is a shift
// plus a rounding increment.
#include "ozk_internal.h"

namespace ozk {
namespace {

constexpr uint64_t kAbsMask = 0x7FFFFFFFFFFFFFFFull;
constexpr uint64_t kInfBits = 0x7FF0000000000000ull;

__device__ __forceinline__ uint64_t abs_bits(double x) {
  return static_cast<uint64_t>(__double_as_longlong(x)) & kAbsMask;
}

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = umax64(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// The scan reads A and B first; the quantisation re-reads them for the last
// time, so only its loads are marked evict-first.
__device__ __forceinline__ double2 load_keep2(const double* p) {
  return __ldg(reinterpret_cast<const double2*>(p));
}

__device__ __forceinline__ double2 load_stream2(const double* p) {
  return __ldcs(reinterpret_cast<const double2*>(p));
}

// ---------------------------------------------------------------------------
// Exponent scan.  For non-negative doubles the bit pattern orders like the
// value, so max |x| is a max over 63-bit integers; Inf/NaN sort above every
// finite value.
// ---------------------------------------------------------------------------

// One warp per (row of A, K segment).  VEC: rows start 16-byte aligned.
template <bool VEC>
__global__ void __launch_bounds__(256) scan_rows_kernel(const double* __restrict__ A, int64_t lda,
                                                        int64_t M, int64_t K, int64_t seg,
                                                        uint64_t* __restrict__ amax) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp;
  if (row >= M) return;
  const int64_t k0 = static_cast<int64_t>(blockIdx.y) * seg;
  const int64_t k1 = min(K, k0 + seg);
  const double* a = A + row * lda;
  uint64_t m = 0;
  if (VEC) {  // seg is even, so k0 is even and a + k0 is 16-byte aligned
    const int64_t q1 = k1 >> 1;
#pragma unroll 4
    for (int64_t q = (k0 >> 1) + lane; q < q1; q += 32) {
      double2 v = load_keep2(a + 2 * q);
      m = umax64(m, umax64(abs_bits(v.x), abs_bits(v.y)));
    }
    if ((k1 & 1) && lane == 0) m = umax64(m, abs_bits(a[k1 - 1]));
  } else {
#pragma unroll 4
    for (int64_t k = k0 + lane; k < k1; k += 32) m = umax64(m, abs_bits(__ldg(a + k)));
  }
  m = warp_max_u64(m);
  if (lane == 0 && m) atomicMax(reinterpret_cast<unsigned long long*>(amax + row), m);
}

// One thread per column pair (VEC) or column, over a K segment of B.
template <bool VEC>
__global__ void __launch_bounds__(256) scan_cols_kernel(const double* __restrict__ B, int64_t ldb,
                                                        int64_t K, int64_t N, int64_t seg,
                                                        uint64_t* __restrict__ amax) {
  const int64_t c = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) * (VEC ? 2 : 1);
  if (c >= N) return;
  const int64_t k0 = static_cast<int64_t>(blockIdx.y) * seg;
  const int64_t k1 = min(K, k0 + seg);
  uint64_t m0 = 0, m1 = 0;
  if (VEC && c + 1 < N) {
#pragma unroll 4
    for (int64_t k = k0; k < k1; ++k) {
      double2 v = load_keep2(B + k * ldb + c);
      m0 = umax64(m0, abs_bits(v.x));
      m1 = umax64(m1, abs_bits(v.y));
    }
  } else {
#pragma unroll 4
    for (int64_t k = k0; k < k1; ++k) m0 = umax64(m0, abs_bits(__ldg(B + k * ldb + c)));
  }
  if (m0) atomicMax(reinterpret_cast<unsigned long long*>(amax + c), m0);
  if (VEC && m1) atomicMax(reinterpret_cast<unsigned long long*>(amax + c + 1), m1);
}

// s = beta - E with max|x| = f 2^E, f in [0.5, 1) (frexp's exponent, read off
// the bits; subnormals via the leading-zero count).
__global__ void finalize_scales_kernel(const uint64_t* __restrict__ amax, int64_t M, int64_t N,
                                       int beta, int32_t* __restrict__ s,
                                       int32_t* __restrict__ t) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= M + N) return;
  const uint64_t b = amax[idx];
  int32_t r;
  if (b >= kInfBits) {
    r = OZK_SCALE_NONFINITE;
  } else if (b == 0) {
    r = 0;
  } else {
    const int ex = static_cast<int>(b >> 52);
    const int E = ex ? ex - 1022 : (63 - __clzll(static_cast<long long>(b))) - 1073;
    r = beta - E;
  }
  if (idx < M)
    s[idx] = r;
  else
    t[idx - M] = r;
}

// ---------------------------------------------------------------------------
// Quantisation.  x = (-1)^neg m 2^e exactly (m < 2^53); with sh = e + s the
// integer is |a'| = m 2^sh rounded to nearest, ties to even (a shift and a
// rounding increment), |a'| <= 2^beta <= 2^72, held as five 16-bit limbs.
// Its residue mod p is sum_j L_j (2^16j mod p) reduced once.
// ---------------------------------------------------------------------------
struct Scaled {
  uint32_t l0, l1, l2, l3, l4;  // |a'| = l0 + l1 2^16 + l2 2^32 + l3 2^48 + l4 2^64
  uint32_t neg;
};

__device__ __forceinline__ Scaled scale_round(double x, int32_t sc) {
  const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(x));
  const uint32_t ex = static_cast<uint32_t>(bits >> 52) & 0x7FFu;
  uint64_t m = bits & 0xFFFFFFFFFFFFFull;
  if (ex) m |= 1ull << 52;
  const int sh = static_cast<int>(ex ? ex : 1u) - 1075 + sc;
  uint64_t lo;
  uint32_t hi;
  if (sh >= 64) {
    lo = 0;
    hi = static_cast<uint32_t>(m << (sh - 64));
  } else if (sh > 0) {
    lo = m << sh;
    hi = static_cast<uint32_t>(m >> (64 - sh));
  } else if (sh == 0) {
    lo = m;
    hi = 0;
  } else if (sh > -64) {
    const int r = -sh;  // 1..63 dropped bits
    const uint64_t q = m >> r;
    const uint64_t rem = m & ((1ull << r) - 1);
    const uint64_t half = 1ull << (r - 1);
    lo = q + ((rem > half || (rem == half && (q & 1u))) ? 1u : 0u);
    hi = 0;
  } else {  // m 2^sh < 2^-11: rounds to 0
    lo = 0;
    hi = 0;
  }
  Scaled r;
  r.l0 = static_cast<uint32_t>(lo) & 0xFFFFu;
  r.l1 = static_cast<uint32_t>(lo >> 16) & 0xFFFFu;
  r.l2 = static_cast<uint32_t>(lo >> 32) & 0xFFFFu;
  r.l3 = static_cast<uint32_t>(lo >> 48);
  r.l4 = hi;
  r.neg = static_cast<uint32_t>(bits >> 63);
  return r;
}

// Balanced residue of (-1)^neg |a'| modulo the k-th modulus, in [-128, 127].
// x below stays under 2^16 + 3 * 2^16 * 255 + 2^9 * 255 < 2^26.
template <int k>
__device__ __forceinline__ int balanced_residue(const Scaled& a) {
  constexpr uint32_t p = modulus_at(k);
  if constexpr (p == 256u) {
    // two's-complement low byte of the signed integer, read as int8
    const uint32_t lowbyte = a.neg ? (0u - a.l0) : a.l0;
    return static_cast<int>(static_cast<int8_t>(lowbyte & 0xFFu));
  } else {
    constexpr uint32_t c1 = pow2_mod(16, p), c2 = pow2_mod(32, p), c3 = pow2_mod(48, p),
                       c4 = pow2_mod(64, p), mg = magic_of(p);
    const uint32_t x = a.l0 + a.l1 * c1 + a.l2 * c2 + a.l3 * c3 + a.l4 * c4;
    const uint32_t q = __umulhi(x, mg);
    int r = static_cast<int>(x - q * p);
    r += r < 0 ? static_cast<int>(p) : 0;                        // |a'| mod p
    r -= r > static_cast<int>((p - 1) / 2) ? static_cast<int>(p) : 0;  // balanced (p odd)
    return a.neg ? -r : r;
  }
}

// bfloat16 bits of a small integer (|r| <= 256 is exact in bf16).
__device__ __forceinline__ uint32_t bf16_bits_of_small_int(int r) {
  const float f = __int_as_float(0x4B400000 + r) - 12582912.0f;  // exact: |r| < 2^22
  return __float_as_uint(f) >> 16;
}

__device__ __forceinline__ uint32_t pack_bf16x2(int lo, int hi) {
  return bf16_bits_of_small_int(lo) | (bf16_bits_of_small_int(hi) << 16);
}

// One thread per 8 consecutive K elements of one row of A.
template <bool VEC>
__global__ void __launch_bounds__(256) quantize_a_kernel(const double* __restrict__ A, int64_t lda,
                                                         int64_t M, int64_t K, int64_t kpad,
                                                         const int32_t* __restrict__ s, int n,
                                                         uint16_t* __restrict__ out) {
  const int64_t groups = kpad >> 3;
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= M * groups) return;
  const int64_t row = g / groups;
  const int64_t k0 = (g - row * groups) * 8;
  const int32_t sc = s[row];
  const double* a = A + row * lda + k0;
  double v[8];
  if (sc == OZK_SCALE_NONFINITE) {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.0;
  } else if (VEC && k0 + 8 <= K) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      double2 d = load_stream2(a + 2 * e);
      v[2 * e] = d.x;
      v[2 * e + 1] = d.y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = (k0 + e < K) ? __ldcs(a + e) : 0.0;
  }
  Scaled x[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] = scale_round(v[e], sc);
  uint4* dst = reinterpret_cast<uint4*>(out + row * kpad + k0);
  const int64_t plane = (M * kpad) >> 3;  // uint4 per modulus slice
  static_for<0, kMaxModuli>([&](auto kc) {
    constexpr int k = decltype(kc)::value;
    if (k < n) {
      uint4 w;
      w.x = pack_bf16x2(balanced_residue<k>(x[0]), balanced_residue<k>(x[1]));
      w.y = pack_bf16x2(balanced_residue<k>(x[2]), balanced_residue<k>(x[3]));
      w.z = pack_bf16x2(balanced_residue<k>(x[4]), balanced_residue<k>(x[5]));
      w.w = pack_bf16x2(balanced_residue<k>(x[6]), balanced_residue<k>(x[7]));
      dst[k * plane] = w;
    }
  });
}

// B (K x N, row-major) to K-major slices [n][N][kpad]: a 64 (k) x 32 (j) tile
// is read with coalesced row segments, quantised, transposed through shared
// memory and written as 128-byte rows.
constexpr int kQbK = 64, kQbJ = 32, kQbRow = kQbK + 2;  // +2 bf16: conflict-free columns

__global__ void __launch_bounds__(256) quantize_b_kernel(const double* __restrict__ B, int64_t ldb,
                                                         int64_t K, int64_t N, int64_t kpad,
                                                         const int32_t* __restrict__ t, int n,
                                                         uint16_t* __restrict__ out) {
  extern __shared__ uint16_t tile[];  // [n][kQbJ][kQbRow]
  const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kQbJ;
  const int64_t k0 = static_cast<int64_t>(blockIdx.y) * kQbK;
  const int jl = threadIdx.x & 31, kr = threadIdx.x >> 5;
  const int64_t j = j0 + jl;
  const int32_t sc = j < N ? t[j] : 0;
  const bool live = j < N && sc != OZK_SCALE_NONFINITE;
  Scaled x[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int64_t k = k0 + kr + 8 * r;
    const double v = (live && k < K) ? __ldcs(B + k * ldb + j) : 0.0;
    x[r] = scale_round(v, sc);
  }
  static_for<0, kMaxModuli>([&](auto kc) {
    constexpr int k = decltype(kc)::value;
    if (k < n) {
      uint16_t* row = tile + (k * kQbJ + jl) * kQbRow + kr;
#pragma unroll
      for (int r = 0; r < 8; ++r)
        row[8 * r] = static_cast<uint16_t>(bf16_bits_of_small_int(balanced_residue<k>(x[r])));
    }
  });
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = n * kQbJ;
  for (int q = warp; q < rows; q += 8) {
    const int p = q / kQbJ, jj = q - p * kQbJ;
    if (j0 + jj >= N) continue;
    const uint32_t w = *reinterpret_cast<const uint32_t*>(tile + q * kQbRow + 2 * lane);
    uint32_t* dst = reinterpret_cast<uint32_t*>(out + (p * N + j0 + jj) * kpad + k0);
    dst[lane] = w;
  }
}

}  // namespace

cudaError_t launch_scale(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                         const double* B, int64_t ldb, int beta, int32_t* s, int32_t* t,
                         uint64_t* amax, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(uint64_t) * static_cast<size_t>(M + N), stream);
  if (e != cudaSuccess) return e;
  int sms = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = kNumSmsFallback;
  const int64_t target_warps = static_cast<int64_t>(sms) * 48;
  if (M > 0 && K > 0) {
    int64_t segs = (target_warps + M - 1) / M;
    int64_t seg = (K + segs - 1) / segs;
    seg = ((seg + 255) / 256) * 256;  // even, and long enough to amortise the atomics
    segs = (K + seg - 1) / seg;
    const bool vec = (reinterpret_cast<uintptr_t>(A) % 16 == 0) && (lda % 2 == 0);
    dim3 grid(static_cast<unsigned>((M + 7) / 8), static_cast<unsigned>(segs));
    if (vec)
      scan_rows_kernel<true><<<grid, 256, 0, stream>>>(A, lda, M, K, seg, amax);
    else
      scan_rows_kernel<false><<<grid, 256, 0, stream>>>(A, lda, M, K, seg, amax);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (N > 0 && K > 0) {
    const bool vec = (reinterpret_cast<uintptr_t>(B) % 16 == 0) && (ldb % 2 == 0);
    const int64_t cols_per_block = vec ? 512 : 256;
    const int64_t bx = (N + cols_per_block - 1) / cols_per_block;
    int64_t segs = (static_cast<int64_t>(sms) * 6 + bx - 1) / bx;
    int64_t seg = (K + segs - 1) / segs;
    if (seg < 32) seg = 32;
    segs = (K + seg - 1) / seg;
    dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(segs));
    if (vec)
      scan_cols_kernel<true><<<grid, 256, 0, stream>>>(B, ldb, K, N, seg, amax + M);
    else
      scan_cols_kernel<false><<<grid, 256, 0, stream>>>(B, ldb, K, N, seg, amax + M);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (M + N > 0) {
    const int64_t blocks = (M + N + 255) / 256;
    finalize_scales_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(amax, M, N, beta, s, t);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_quantize_a(int64_t M, int64_t K, int64_t kpad, const double* A, int64_t lda,
                              const int32_t* s, int n, uint16_t* out, cudaStream_t stream) {
  if (M == 0 || kpad == 0) return cudaSuccess;
  const int64_t threads = M * (kpad / 8);
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  const bool vec = (reinterpret_cast<uintptr_t>(A) % 16 == 0) && (lda % 2 == 0);
  if (vec)
    quantize_a_kernel<true><<<blocks, 256, 0, stream>>>(A, lda, M, K, kpad, s, n, out);
  else
    quantize_a_kernel<false><<<blocks, 256, 0, stream>>>(A, lda, M, K, kpad, s, n, out);
  return cudaGetLastError();
}

cudaError_t launch_quantize_b(int64_t K, int64_t N, int64_t kpad, const double* B, int64_t ldb,
                              const int32_t* t, int n, uint16_t* out, cudaStream_t stream) {
  if (N == 0 || kpad == 0) return cudaSuccess;
  const size_t smem = sizeof(uint16_t) * static_cast<size_t>(n) * kQbJ * kQbRow;
  // the attribute belongs to the current device's copy of the kernel
  cudaError_t e = cudaFuncSetAttribute(quantize_b_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(uint16_t) * kMaxModuli * kQbJ * kQbRow));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((N + kQbJ - 1) / kQbJ), static_cast<unsigned>(kpad / kQbK));
  quantize_b_kernel<<<grid, 256, smem, stream>>>(B, ldb, K, N, kpad, t, n, out);
  return cudaGetLastError();
}

}  // namespace ozk
