// The CRT combine kernels with the moduli count fixed at compile time, one
// instantiation per count and input (byte residues, or the 16-bit residues of
// moduli pairs), for the FP64 output: with the count known, the pair loop,
// the accumulator set-up and the limb count are resolved by the compiler.
// The run-time-count kernels in crt_combine.cu serve the other cases.
#include "crt_device.cuh"

namespace ozk {
namespace {

template <int NM>
cudaError_t launch_fixed(int64_t M, int64_t N, const void* in, int in_kind, int64_t ldi, int64_t plane,
                         const int32_t* s, const int32_t* t, double* C, int64_t ldc, const CrtConst& K,
                         cudaStream_t stream) {
  constexpr int G = 1;
  const int64_t threads = M * ((N + 4 * G - 1) / (4 * G));
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  if (in_kind == 2)
    return launch_dependent(crt_pairs_kernel<crt_limbs(NM), false, 2, NM>,
                            dim3(static_cast<unsigned>((M * ((N + 7) / 8) + 255) / 256)), dim3(256), 0, stream, in,
                            ldi, plane, M, N, s, t, C, ldc, nullptr, K, fast_div((N + 7) / 8));
  return launch_dependent(crt_kernel<crt_limbs(NM), 0, false, G, NM>, dim3(blocks), dim3(256), 0, stream, in, ldi,
                          plane, M, N, 1, s, t, C, ldc, nullptr, K, fast_div((N + 4 * G - 1) / (4 * G)));
}

template <int NM>
cudaError_t dispatch(int n, int64_t M, int64_t N, const void* in, int in_kind, int64_t ldi, int64_t plane,
                     const int32_t* s, const int32_t* t, double* C, int64_t ldc, const CrtConst& K,
                     cudaStream_t stream) {
  if constexpr (NM > kMaxModuli) {
    return cudaErrorInvalidValue;
  } else {
    if (n == NM) return launch_fixed<NM>(M, N, in, in_kind, ldi, plane, s, t, C, ldc, K, stream);
    return dispatch<NM + 1>(n, M, N, in, in_kind, ldi, plane, s, t, C, ldc, K, stream);
  }
}

}  // namespace

cudaError_t launch_crt_fixed(int64_t M, int64_t N, const void* in, int in_kind, int64_t ldi, int64_t plane,
                             const int32_t* s, const int32_t* t, double* C, int64_t ldc, const CrtConst& K,
                             cudaStream_t stream) {
  if (K.n < 2 || K.n > kMaxModuli || (in_kind != 0 && in_kind != 2)) return cudaErrorInvalidValue;
  return dispatch<2>(K.n, M, N, in, in_kind, ldi, plane, s, t, C, ldc, K, stream);
}

}  // namespace ozk
