// Launchers of the CRT combine (the arithmetic is in crt_device.cuh): the
// kernels with a runtime moduli count for byte residues, split-K int32
// partial sums, pair residues, the exact-integer (limb) output and narrow
// outputs, and the dispatch to the compile-time-count kernels of
// crt_fixed.cu for the common case (byte or pair residues, FP64 output, wide).
#include "crt_device.cuh"

namespace ozk {
namespace {

// Runtime moduli count, 4 columns per thread.
template <int NL>
cudaError_t launch_nl_g(int64_t M, int64_t N, const void* in, int in_kind, int64_t ldi, int64_t plane,
                        int splits, const int32_t* s, const int32_t* t, double* C, int64_t ldc, uint32_t* X,
                        const CrtConst& K, cudaStream_t stream) {
  constexpr int G = 1;
  const int64_t threads = M * ((N + 4 * G - 1) / (4 * G));
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  const FastDiv rd = fast_div((N + 4 * G - 1) / (4 * G));
  const dim3 grid(blocks), block(256);
  if (in_kind == 0)
    return X ? launch_dependent(crt_kernel<NL, 0, true, G, 0>, grid, block, 0, stream, in, ldi, plane, M, N, splits,
                                s, t, C, ldc, X, K, rd)
             : launch_dependent(crt_kernel<NL, 0, false, G, 0>, grid, block, 0, stream, in, ldi, plane, M, N,
                                splits, s, t, C, ldc, X, K, rd);
  if (in_kind == 1)
    return X ? launch_dependent(crt_kernel<NL, 1, true, G, 0>, grid, block, 0, stream, in, ldi, plane, M, N, splits,
                                s, t, C, ldc, X, K, rd)
             : launch_dependent(crt_kernel<NL, 1, false, G, 0>, grid, block, 0, stream, in, ldi, plane, M, N,
                                splits, s, t, C, ldc, X, K, rd);
  return X ? launch_dependent(crt_pairs_kernel<NL, true, G, 0>, grid, block, 0, stream, in, ldi, plane, M, N, s, t,
                              C, ldc, X, K, rd)
           : launch_dependent(crt_pairs_kernel<NL, false, G, 0>, grid, block, 0, stream, in, ldi, plane, M, N, s, t,
                              C, ldc, X, K, rd);
}

// The FP64 output from byte or pair residues (what the GEMM path writes) on
// outputs wide enough to give every SM several blocks of 8-column threads runs
// the kernel compiled for its moduli count; everything else the runtime-count one.
template <int NL>
cudaError_t launch_nl(int64_t M, int64_t N, const void* in, int in_kind, int64_t ldi, int64_t plane, int splits,
                      const int32_t* s, const int32_t* t, double* C, int64_t ldc, uint32_t* X,
                      const CrtConst& K, cudaStream_t stream) {
  constexpr int64_t kWideThreads = 152 * 256 * 4;
  if (M * ((N + 7) / 8) >= kWideThreads && in_kind != 1 && X == nullptr)
    return launch_crt_fixed(M, N, in, in_kind, ldi, plane, s, t, C, ldc, K, stream);
  return launch_nl_g<NL>(M, N, in, in_kind, ldi, plane, splits, s, t, C, ldc, X, K, stream);
}

}  // namespace

cudaError_t launch_crt(int64_t M, int64_t N, int n, const void* in, int in_kind, int64_t ldi,
                       int64_t plane, int splits, const int32_t* s, const int32_t* t, double* C,
                       int64_t ldc, uint32_t* X, cudaStream_t stream) {
  if (M == 0 || N == 0) return cudaSuccess;
  const CrtConst& K = crt_const(n);
  switch (crt_limbs(n)) {
    case 3: return launch_nl<3>(M, N, in, in_kind, ldi, plane, splits, s, t, C, ldc, X, K, stream);
    case 4: return launch_nl<4>(M, N, in, in_kind, ldi, plane, splits, s, t, C, ldc, X, K, stream);
    case 5: return launch_nl<5>(M, N, in, in_kind, ldi, plane, splits, s, t, C, ldc, X, K, stream);
    case 6: return launch_nl<6>(M, N, in, in_kind, ldi, plane, splits, s, t, C, ldc, X, K, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ozk
