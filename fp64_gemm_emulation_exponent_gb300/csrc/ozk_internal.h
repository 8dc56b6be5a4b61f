// Internal declarations shared by the CUDA translation units of libozk.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

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

template <int I, int N, typename F>
__host__ __device__ __forceinline__ void static_for(F&& f) {
  if constexpr (I < N) {
    f(std::integral_constant<int, I>{});
    static_for<I + 1, N>(f);
  }
}

// Limb count of the CRT accumulator for n moduli: S = sum_k c_k e_k with
// c_k < 256, e_k < P <= 2^(8n) stays below n 2^(8n + 8) < 2^(8n + 14).  At least 3.
__host__ __device__ constexpr int crt_limbs(int n) {
  return (8 * n + 14 + 31) / 32 < 3 ? 3 : (8 * n + 14 + 31) / 32;
}
constexpr int kMaxCrtLimbs = 6;

// Constants of the CRT combine for one moduli count (built on the host).
// e_k = (P/p_k) w_k with w_k = (P/p_k)^-1 mod p_k is the CRT basis vector of
// modulus k (e_k = 1 mod p_k, 0 mod the others, e_k < P); e_k / P = w_k / p_k.
struct CrtConst {
  uint32_t p[kMaxModuli];
  uint32_t magic[kMaxModuli];
  uint32_t bias[kMaxModuli];
  uint32_t frac[kMaxModuli];  // round(2^32 w_k / p_k): e_k / P in 0.32 fixed point
  uint32_t e[kMaxModuli][kMaxCrtLimbs];  // e_k, little-endian 32-bit limbs
  uint32_t P[kMaxCrtLimbs];
  // Moduli taken in pairs (2j, 2j+1) with m_j = p_2j p_2j+1: the pair's
  // residue r_j = (c_2j u_j0 + c_2j+1 u_j1) mod m_j (u_j0 = 1 mod p_2j and 0 mod
  // p_2j+1, u_j1 the other way round) has CRT basis vector E_j = e_2j + e_2j+1
  // (mod P), and E_j / P = w_j / m_j.
  uint32_t pm[kMaxModuli / 2];
  uint32_t pu[kMaxModuli / 2][2];
  uint32_t pmagic[kMaxModuli / 2];  // ceil(2^42 / m_j): floor(t / m_j) = umulhi(t, pmagic) >> 10 for t < 2^25
  uint32_t pfrac[kMaxModuli / 2];   // round(2^32 w_j / m_j)
  uint32_t pe[kMaxModuli / 2][kMaxCrtLimbs];
  int n;
};

// Host-side method constants (ozk_api.cu).
int beta_for(int64_t K, int n);  // -1 when unsupported
// OZK_OK when the current device is an sm_103 GPU (its SM count in *sms when not null).
int current_device_supported(int* sms);
const CrtConst& crt_const(int n);

// Launchers; each returns the first CUDA error it meets.
cudaError_t launch_scale(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                         const double* B, int64_t ldb, int beta, int32_t* s, int32_t* t,
                         uint64_t* amax, cudaStream_t stream);
// Per-modulus planes (residue slices, residue or partial-sum planes) sit
// `plane` elements apart; the workspace spaces them an odd number of 256-byte
// units apart so that the n streams of a kernel do not fall on the same DRAM
// channels at the same time.
//
// Quantises A (when A is not null) and B (when B is not null) in one launch;
// slices and plane strides must be 32-byte aligned.
cudaError_t launch_quantize(int64_t M, int64_t N, int64_t K, int64_t kpad, const double* A,
                            int64_t lda, const double* B, int64_t ldb, const int32_t* s,
                            const int32_t* t, int n, int beta, uint16_t* a_out, int64_t a_plane,
                            uint16_t* b_out, int64_t b_plane, cudaStream_t stream);
// Rows of A scanned and quantised in one pass (one block per row): writes
// s[0..M) and A's slices as launch_scale + launch_quantize would.  Only for
// K up to 4096 (quantize_rows_fits(kpad)); cudaErrorInvalidValue beyond.
bool quantize_rows_fits(int64_t kpad);
cudaError_t launch_quantize_rows(int64_t M, int64_t K, int64_t kpad, const double* A, int64_t lda, int n,
                                 int beta, int32_t* s, uint16_t* a_out, int64_t a_plane,
                                 cudaStream_t stream);
cudaError_t launch_residue_gemm(int64_t M, int64_t N, int64_t kpad, const uint16_t* a_slices,
                                int64_t a_plane, const uint16_t* b_slices, int64_t b_plane, int n,
                                int out_kind, void* out, int64_t ldo, int64_t out_plane, int splits,
                                int num_sms, cudaStream_t stream);
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
