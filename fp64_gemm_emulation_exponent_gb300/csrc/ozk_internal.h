// Internal declarations shared by the CUDA translation units of libozk.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>
#include <utility>

#include "ozk.h"

namespace ozk {

constexpr int kMaxModuli = 20;
constexpr int kKBlock = 64;  // K elements (fp16) per smem row: 128 bytes, one swizzle row
constexpr int kNumSmsFallback = 148;

// Moduli in the order they are consumed: pairwise coprime integers <= 256,
// so every balanced residue lies in [-128, 127].
__host__ __device__ constexpr uint32_t modulus_at(int k) {
  constexpr uint32_t t[kMaxModuli] = {256, 255, 253, 251, 247, 241, 239, 233, 229, 227,
                                      223, 217, 211, 199, 197, 193, 191, 181, 179, 173};
  return t[k];
}

// q = __umulhi(u, magic) is floor(u/p) or floor(u/p)+1 for every u < 2^32,
// because magic*p = 2^32 + e with 1 <= e <= p.  One conditional add fixes r.
__host__ __device__ constexpr uint32_t magic_of(uint32_t p) {
  return static_cast<uint32_t>(0x100000000ull / p) + 1u;
}

// A multiple of p in [2^31, 2^31 + p): x + bias maps every int32 |x| < 2^31 - 2^14
// to [0, 2^32) without changing its class mod p.
__host__ __device__ constexpr uint32_t bias_of(uint32_t p) {
  return static_cast<uint32_t>(((0x80000000ull + p - 1) / p) * p);
}

__host__ __device__ constexpr uint32_t pow2_mod(int e, uint32_t p) {
  uint32_t r = 1u % p;
  for (int i = 0; i < e; ++i) r = (r * 2u) % p;
  return r;
}

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialisation allowed and starts, in every
// thread, by waiting for the grid before it in the stream to complete and
// its writes to be visible (so that completing implies the predecessor's
// completion, which keeps the order transitive), then lets the grid after
// it launch: its blocks take the SM room this grid's last blocks leave and
// wait there, instead of being launched only once this grid has ended.
__device__ __forceinline__ void grid_dependency_sync() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// floor(g / d) for every g < 2^31 by one multiply-high, d fixed per launch
// (the combine's column groups per row, the GEMM's tile and split counts):
// with l = ceil(log2 d) and m = ceil(2^(31 + l) / d) < 2^32, g m / 2^(31 + l)
// exceeds g / d by less than g / 2^(31 + l) < 2^-l <= 1/d, which cannot carry
// it past the next integer, so floor(g / d) = umulhi(g, m) >> (l - 1); d = 1
// has s = -1.
struct FastDiv {
  uint32_t m;
  int s;
};
inline FastDiv fast_div(int64_t d) {
  if (d <= 1) return {0u, -1};
  int l = 0;
  while ((int64_t{1} << l) < d) ++l;
  const uint64_t num = uint64_t{1} << (31 + l);
  return {static_cast<uint32_t>((num + static_cast<uint64_t>(d) - 1) / static_cast<uint64_t>(d)), l - 1};
}
__device__ __forceinline__ uint32_t div_fast(uint32_t g, const FastDiv& r) {
  return r.s < 0 ? g : __umulhi(g, r.m) >> r.s;
}

template <int I, int N, typename F>
__host__ __device__ __forceinline__ void static_for(F&& f) {
  if constexpr (I < N) {
    f(std::integral_constant<int, I>{});
    static_for<I + 1, N>(f);
  }
}

// Limb count of the CRT accumulator for n moduli: S = sum_t d_t b_t with
// digits d_t < 256 and bases b_t < P <= 2^(8n) stays below n 2^(8n + 8) <
// 2^(8n + 14); it is held modulo 2^(32 NL).  At least 3.
__host__ __device__ constexpr int crt_limbs(int n) {
  return (8 * n + 14 + 31) / 32 < 3 ? 3 : (8 * n + 14 + 31) / 32;
}
constexpr int kMaxCrtLimbs = 6;

// Bit length of the product of the first n moduli.
__host__ __device__ constexpr int modulus_product_bits(int n) {
  uint32_t w[kMaxCrtLimbs] = {1, 0, 0, 0, 0, 0};
  for (int k = 0; k < n; ++k) {
    uint64_t c = 0;
    for (int l = 0; l < kMaxCrtLimbs; ++l) {
      c += static_cast<uint64_t>(w[l]) * modulus_at(k);
      w[l] = static_cast<uint32_t>(c);
      c >>= 32;
    }
  }
  for (int l = kMaxCrtLimbs - 1; l >= 0; --l)
    for (int b = 31; b >= 0; --b)
      if ((w[l] >> b) & 1u) return 32 * l + b + 1;
  return 0;
}
// 16-bit limbs of a CRT basis vector (a number below P) for n moduli.
__host__ __device__ constexpr int crt_cols16(int n) { return (modulus_product_bits(n) + 15) / 16; }
constexpr int kMaxCols16 = 10;  // the product of all 20 moduli is below 2^157
static_assert(2 * kMaxCrtLimbs >= kMaxCols16, "the accumulator holds every basis limb");

// Constants of the CRT combine for one moduli count (built on the host).
// e_k = (P/p_k) w_k with w_k = (P/p_k)^-1 mod p_k is the CRT basis vector of
// modulus k (e_k = 1 mod p_k, 0 mod the others, e_k < P); e_k / P = w_k / p_k.
//  * Byte residues c_k: S = sum_k c_k e_k is formed column by column in
//    16-bit limbs, the moduli taken in pairs (2j, 2j+1) by two-way 16x8-bit
//    dot products (dp2a): bt[j][l] = limb l of e_2j | limb l of e_2j+1 << 16
//    (an odd last modulus alone).  q = round(S / P) from the ratios e_k / P
//    in 0.32 fixed point, split into 16-bit halves packed the same way:
//    bfh (high halves), bfl (low halves).
//  * 16-bit residues r_j of the pair moduli m_j = p_2j p_2j+1 (the GEMM's pair
//    output): S = sum_j r_j E_j with E_j = (P/m_j) W_j, W_j = (P/m_j)^-1 mod
//    m_j, in 32-bit limbs (pe) with 64-bit multiply-accumulates, and q from
//    round(2^32 W_j / m_j) (pfrac); an odd last modulus enters as c_n-1 e_n-1
//    (elast, flast).
struct CrtConst {
  uint32_t p[kMaxModuli];
  uint32_t magic[kMaxModuli];
  uint32_t bias[kMaxModuli];
  uint32_t P[kMaxCrtLimbs];              // P, little-endian 32-bit limbs
  uint32_t pn[kMaxCrtLimbs];             // 2^(32 NL) - P (NL = crt_limbs(n)), 32-bit limbs
  uint32_t pn16[2 * kMaxCrtLimbs];       // the same in 16-bit limbs
  uint32_t bt[kMaxModuli / 2][kMaxCols16];
  uint32_t bfh[kMaxModuli / 2], bfl[kMaxModuli / 2];
  uint32_t pe[kMaxModuli / 2][kMaxCrtLimbs];
  uint32_t pfrac[kMaxModuli / 2];
  uint32_t elast[kMaxCrtLimbs], flast;
  int n;
};

// Host-side method constants (ozk_api.cu).
int beta_for(int64_t K, int n);   // -1 when unsupported
int gamma_for(int64_t K, int n);  // the norm rule's budget; -1 when unsupported
// OZK_OK when the current device is an sm_103 GPU (its SM count in *sms when not null).
int current_device_supported(int* sms);
const CrtConst& crt_const(int n);

// Launchers; each returns the first CUDA error it meets.
// Exponent scan: the abs-bit maxima of the rows of A and the columns of B
// into amax[0..M) and amax[M..M+N) (zeroed first); with nsum not null also
// the norm sums of the norm rule, nsum[0..M+N); then the scales s, t
// (budget: beta of the largest-entry rule, or gamma of the norm rule).
cudaError_t launch_scale(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                         const double* B, int64_t ldb, int budget, int32_t* s, int32_t* t,
                         uint64_t* amax, uint64_t* nsum, cudaStream_t stream);
// The scan alone (maxima and, with nsum, norm sums; no scales):
// launch_quantize then derives the scales and stores them.
cudaError_t launch_scan(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
                        int64_t ldb, uint64_t* amax, uint64_t* nsum, cudaStream_t stream);
// Per-modulus planes (residue slices, residue or partial-sum planes) sit
// `plane` elements apart; the workspace spaces them an odd number of 256-byte
// units apart so that the n streams of a kernel do not fall on the same DRAM
// channels at the same time.
//
// Quantises A (when A is not null) and B (when B is not null) in one launch;
// slices and plane strides must be 32-byte aligned.  With a_amax (b_amax) not
// null the scales are derived from the scanned maxima (and, with a_nsum
// (b_nsum), the norm sums: the norm rule) and stored in s (t); otherwise
// s (t) are read.  budget is beta, or gamma for the norm rule; it also sets
// the integer width (|a'| <= 2^budget).
cudaError_t launch_quantize(int64_t M, int64_t N, int64_t K, int64_t kpad, const double* A,
                            int64_t lda, const double* B, int64_t ldb, int32_t* s, int32_t* t,
                            const uint64_t* a_amax, const uint64_t* b_amax, const uint64_t* a_nsum,
                            const uint64_t* b_nsum, int n, int budget, uint16_t* a_out, int64_t a_plane,
                            uint16_t* b_out, int64_t b_plane, cudaStream_t stream);
// Rows of A scanned and quantised in one pass (one block per row): writes
// s[0..M) and A's slices as launch_scale + launch_quantize would.  Only for
// K up to 4096 (quantize_rows_fits(kpad)); cudaErrorInvalidValue beyond.
bool quantize_rows_fits(int64_t kpad);
cudaError_t launch_quantize_rows(int64_t M, int64_t K, int64_t kpad, const double* A, int64_t lda, int n,
                                 int budget, bool norm, int32_t* s, uint16_t* a_out, int64_t a_plane,
                                 cudaStream_t stream);
cudaError_t launch_residue_gemm(int64_t M, int64_t N, int64_t kpad, const uint16_t* a_slices,
                                int64_t a_plane, const uint16_t* b_slices, int64_t b_plane, int n,
                                int out_kind, void* out, int64_t ldo, int64_t out_plane, int splits,
                                int num_sms, cudaStream_t stream);
// The single-CTA residue GEMM (byte residues, one split; K below 2048) with
// every pipeline wait limited to timeout_ns and the copy of k-block
// withhold_kb of CTA 0's first unit never issued: the MMA issuer's wait for
// it runs out, the kernel latches OZK_ERR_TIMEOUT and every role stops.
// cudaErrorInvalidValue where the CTA-pair kernel would run or the k-block
// does not exist.
cudaError_t launch_residue_gemm_withheld(int64_t M, int64_t N, int64_t kpad, const uint16_t* a_slices,
                                         int64_t a_plane, const uint16_t* b_slices, int64_t b_plane, int n,
                                         void* out, int64_t ldo, int64_t out_plane, int num_sms,
                                         uint64_t timeout_ns, int withhold_kb, cudaStream_t stream);
// The same for in_kind 0 or 2 and an FP64 output, through a kernel compiled
// for this moduli count (crt_fixed.cu).
cudaError_t launch_crt_fixed(int64_t M, int64_t N, const void* in, int in_kind, int64_t ldi, int64_t plane,
                             const int32_t* s, const int32_t* t, double* C, int64_t ldc, const CrtConst& K,
                             cudaStream_t stream);
cudaError_t launch_crt(int64_t M, int64_t N, int n, const void* in, int in_kind, int64_t ldi,
                       int64_t plane, int splits, const int32_t* s, const int32_t* t, double* C,
                       int64_t ldc, uint32_t* X, cudaStream_t stream);

// Device status word latched by kernels (residue_gemm.cu).
int take_device_status(cudaStream_t stream, int* status);

// Tile sizes of the residue GEMM, exposed for the host's split-K choice.
constexpr int kTileM = 128;
constexpr int kTileN = 256;
int choose_splits(int64_t M, int64_t N, int64_t kpad, int n, int num_sms);

}  // namespace ozk
