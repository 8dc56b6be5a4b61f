// C-ABI of libozk: argument checks, method constants, workspace layout and the
// stage sequence of the Ozaki-II pipeline (the "Day 12" page, section
// "Profile 不能只看 Tensor Core": scale / exponent scan, residue quantization,
// INT8 GEMM, mod reduction, CRT reconstruction, undo scaling, write double).
#include <cuda_runtime.h>

#include <cstring>
#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "ozk_internal.h"

namespace ozk {
namespace {

constexpr int kSplitSms = 152;  // SM count the split-K choice plans for (GB300)
constexpr int64_t kMaxDim = INT32_MAX / 2;  // rows/columns the kernels index with int

// ---- small unsigned multi-limb integers for the host-side constants -------
struct Limbs {
  uint32_t w[8];
};

void limbs_set(Limbs& a, uint32_t v) {
  std::memset(a.w, 0, sizeof a.w);
  a.w[0] = v;
}

void limbs_mul_small(Limbs& a, uint32_t m) {
  uint64_t c = 0;
  for (int l = 0; l < 8; ++l) {
    c += static_cast<uint64_t>(a.w[l]) * m;
    a.w[l] = static_cast<uint32_t>(c);
    c >>= 32;
  }
}

int limbs_msb(const Limbs& a) {
  for (int l = 7; l >= 0; --l)
    if (a.w[l]) return 32 * l + 31 - __builtin_clz(a.w[l]);
  return -1;
}

int ceil_log2(int64_t K) {
  int c = 0;
  while (c < 62 && (int64_t{1} << c) < K) ++c;
  return c;
}

// x^-1 mod m for x coprime to m (small m: a scan).
uint32_t inverse_mod(uint64_t x, uint32_t m) {
  x %= m;
  for (uint32_t y = 1; y < m; ++y)
    if (x * y % m == 1u) return y;
  return 0;
}

// (P / m) * w as limbs, and round(2^32 w / m): a CRT basis vector of a
// modulus m dividing P, and its ratio to P in 0.32 fixed point.
void basis_of(int n, uint64_t m, uint32_t w, Limbs* b, uint32_t* frac) {
  limbs_set(*b, w);
  for (int i = 0; i < n; ++i)
    if (m % modulus_at(i) != 0) limbs_mul_small(*b, modulus_at(i));
  *frac = static_cast<uint32_t>(((static_cast<uint64_t>(w) << 32) + m / 2) / m);
}

// (P / m)^-1 mod m.
uint32_t cofactor_inverse(int n, uint32_t m) {
  uint64_t r = 1;
  for (int i = 0; i < n; ++i)
    if (m % modulus_at(i) != 0) r = r * (modulus_at(i) % m) % m;
  return inverse_mod(r, m);
}

uint32_t limb16(const Limbs& a, int l) { return (a.w[l / 2] >> (16 * (l % 2))) & 0xFFFFu; }

CrtConst build_crt_const(int n) {
  CrtConst K;
  std::memset(&K, 0, sizeof K);
  K.n = n;
  const int NL = crt_limbs(n);
  const int NC = crt_cols16(n);
  Limbs P;
  limbs_set(P, 1);
  for (int k = 0; k < n; ++k) limbs_mul_small(P, modulus_at(k));
  for (int l = 0; l < kMaxCrtLimbs; ++l) K.P[l] = P.w[l];
  Limbs Pn;  // 2^(32 NL) - P
  {
    uint64_t c = 1;
    std::memset(Pn.w, 0, sizeof Pn.w);
    for (int l = 0; l < NL; ++l) {
      c += static_cast<uint64_t>(~P.w[l]);
      Pn.w[l] = static_cast<uint32_t>(c);
      c >>= 32;
    }
  }
  for (int l = 0; l < NL; ++l) K.pn[l] = Pn.w[l];
  for (int l = 0; l < 2 * NL; ++l) K.pn16[l] = limb16(Pn, l);
  for (int k = 0; k < n; ++k) {
    const uint32_t p = modulus_at(k);
    K.p[k] = p;
    K.magic[k] = magic_of(p);
    K.bias[k] = bias_of(p);
  }
  for (int j = 0; 2 * j < n; ++j) {
    // byte residues: e_2j and e_2j+1 (an odd last modulus alone)
    Limbs e[2];
    uint32_t f[2] = {0, 0};
    limbs_set(e[1], 0);
    for (int h = 0; h < 2 && 2 * j + h < n; ++h) {
      const uint32_t p = modulus_at(2 * j + h);
      basis_of(n, p, cofactor_inverse(n, p), &e[h], &f[h]);
    }
    for (int l = 0; l < NC; ++l) K.bt[j][l] = limb16(e[0], l) | (limb16(e[1], l) << 16);
    K.bfh[j] = (f[0] >> 16) | (f[1] & 0xFFFF0000u);
    K.bfl[j] = (f[0] & 0xFFFFu) | (f[1] << 16);
    // pair residues: E_j (an odd last modulus is its own residue, base e_n-1)
    if (2 * j + 1 < n) {
      const uint32_t m = modulus_at(2 * j) * modulus_at(2 * j + 1);
      Limbs E;
      basis_of(n, m, cofactor_inverse(n, m), &E, &K.pfrac[j]);
      for (int l = 0; l < kMaxCrtLimbs; ++l) K.pe[j][l] = E.w[l];
    } else {
      for (int l = 0; l < kMaxCrtLimbs; ++l) K.elast[l] = e[0].w[l];
      K.flast = f[0];
    }
  }
  return K;
}

CrtConst g_crt[kMaxModuli + 1];
std::once_flag g_crt_once;

// ---- per-device state -----------------------------------------------------
std::mutex g_mutex;
struct DevInfo {
  int checked = 0;  // 0 unknown, 1 ok, -1 wrong architecture
  int sms = 0;
};
std::map<int, DevInfo> g_dev;
std::map<std::pair<int, cudaStream_t>, std::pair<void*, size_t>> g_ws;  // cached workspaces
// Per device: the device copies of the host operands, the copy streams and
// events of the host path, and a lock held for a whole host call (one host
// call per device at a time).
constexpr int kMaxHostBlocks = 4;
// Device copies of host operands for ozk_dgemm_host(_async).  Two slots, used
// in turn, so that one call's inputs can move in while the previous call
// computes.  A slot's A and B take new inputs once the stages of the call
// that used them last are done (`computed`); its C takes a new result once
// that call has copied C out (`free`).
constexpr int kHostSlots = 2;
struct HostSlot {
  double* A = nullptr;
  double* B = nullptr;
  double* C = nullptr;
  size_t a = 0, b = 0, c = 0;
  cudaEvent_t computed = nullptr;
  cudaEvent_t free = nullptr;
};
struct HostBufs {
  HostSlot slot[kHostSlots];
  int next = 0;
  cudaStream_t in = nullptr, out = nullptr;                     // host-to-device and device-to-host copies
  cudaStream_t comp = nullptr;                                  // the stages of every call, in call order
  cudaEvent_t computed = nullptr;                               // the last call's stages are done
  cudaEvent_t ev_in[2 * kMaxHostBlocks] = {};                  // a block of A or B has arrived
  cudaEvent_t ev_out[kMaxHostBlocks * kMaxHostBlocks] = {};    // a piece of C is computed
  std::mutex call;                                             // enqueueing is serialised per device
};
std::map<int, HostBufs> g_host;

int check_device(int* sms_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DevInfo& d = g_dev[dev];
  if (d.checked == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return OZK_ERR_CUDA;
    d.checked = (major == 10 && minor == 3) ? 1 : -1;
    d.sms = sms;
  }
  if (d.checked < 0) return OZK_ERR_DEVICE;
  if (sms_out) *sms_out = d.sms;
  return OZK_OK;
}

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool ranges_overlap(const void* a, size_t abytes, const void* b, size_t bbytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

size_t span_bytes(int64_t rows, int64_t cols, int64_t ld) {
  if (rows <= 0 || cols <= 0) return 0;
  return sizeof(double) * static_cast<size_t>((rows - 1) * ld + cols);
}

int validate(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
             int64_t ldb, const double* C, int64_t ldc, int n, int rule = 0) {
  if (M < 0 || N < 0 || K < 0) return OZK_ERR_INVALID_ARG;
  if (n < 2 || n > kMaxModuli) return OZK_ERR_UNSUPPORTED;
  if (K > OZK_MAX_K || M > kMaxDim || N > kMaxDim) return OZK_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return OZK_OK;
  if (!C || ldc < N) return OZK_ERR_INVALID_ARG;
  if (K == 0) return OZK_OK;
  if (!A || !B || lda < K || ldb < N) return OZK_ERR_INVALID_ARG;
  if ((rule ? gamma_for(K, n) : beta_for(K, n)) < 1) return OZK_ERR_UNSUPPORTED;
  const size_t cb = span_bytes(M, N, ldc);
  if (ranges_overlap(C, cb, A, span_bytes(M, K, lda)) || ranges_overlap(C, cb, B, span_bytes(K, N, ldb)))
    return OZK_ERR_INVALID_ARG;
  return OZK_OK;
}

// Workspace layout (byte offsets), shared by ozk_workspace_size and the run.
struct Layout {
  size_t amax, s, t, a, b, out, total;
  int64_t kpad, ldo;
  int64_t a_plane, b_plane, out_plane;  // elements between consecutive moduli's planes
  int splits, planes, kind;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Plane stride in bytes: at least `bytes`, an odd multiple of 256.
size_t skewed_plane(size_t bytes) {
  size_t units = (bytes + 255) / 256;
  if (units % 2 == 0) ++units;
  return units * 256;
}

Layout layout_for(int64_t M, int64_t N, int64_t K, int n) {
  Layout L;
  L.kpad = ozk_kpad(K);
  L.splits = choose_splits(M, N, L.kpad, n, kSplitSms);
  // one split: byte residues (kind 0); split-K: int32 sums (kind 1).  The
  // uint16 residues of moduli pairs (kind 2, the first CRT step in the GEMM's
  // epilogue) measured slower end to end at every K once the byte planes were
  // reduced in fp32 and stored by TMA (e.g. 2048^2 x 32768: 8 moduli 1954 ->
  // 1798 us, 20 moduli 4470 -> 4296 us with byte planes; 14 moduli within
  // 0.3% either way), so ozk_dgemm does not use them; the stage entry points
  // still write and read them.
  L.kind = L.splits > 1 ? 1 : 0;
  L.ldo = L.kind == 1 ? round_up(N, 4) : round_up(N, 16);
  L.planes = L.kind == 1 ? n * L.splits : (L.kind == 2 ? (n + 1) / 2 : n);
  size_t off = 0;
  L.amax = off;  // the maxima, then the norm sums of the norm rule
  off = align_up(off + 2 * sizeof(uint64_t) * static_cast<size_t>(M + N), 256);
  L.s = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(M), 256);
  L.t = off;
  off = align_up(off + sizeof(int32_t) * static_cast<size_t>(N), 1024);
  const size_t a_plane = skewed_plane(2u * static_cast<size_t>(M) * L.kpad);
  const size_t b_plane = skewed_plane(2u * static_cast<size_t>(N) * L.kpad);
  const size_t esize = L.kind == 0 ? 1 : (L.kind == 2 ? 2 : 4);
  const size_t o_plane = skewed_plane(esize * static_cast<size_t>(M) * L.ldo);
  L.a_plane = static_cast<int64_t>(a_plane / 2);
  L.b_plane = static_cast<int64_t>(b_plane / 2);
  L.out_plane = static_cast<int64_t>(o_plane / esize);
  L.a = off;
  off = align_up(off + a_plane * static_cast<size_t>(n), 1024);
  L.b = off;
  off = align_up(off + b_plane * static_cast<size_t>(n), 1024);
  L.out = off;
  off = align_up(off + o_plane * static_cast<size_t>(L.planes), 256);
  L.total = off;
  return L;
}

// The workspace cached for (current device, stream), grown to `need` bytes.
int cached_workspace(cudaStream_t st, size_t need, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  auto& slot = g_ws[{dev, st}];
  if (slot.second < need) {
    if (slot.first) {
      if (cudaStreamSynchronize(st) != cudaSuccess) return OZK_ERR_CUDA;
      cudaFree(slot.first);
      slot = {nullptr, 0};
    }
    if (cudaMalloc(&slot.first, need) != cudaSuccess) {
      slot = {nullptr, 0};
      return OZK_ERR_WORKSPACE;
    }
    slot.second = need;
  }
  *out = slot.first;
  return OZK_OK;
}

// The regions of one call's workspace (caller-provided or cached).
struct WsViews {
  uint64_t* amax;
  int32_t* s;
  int32_t* t;
  uint16_t* as;
  uint16_t* bs;
  uint8_t* out;
  size_t esize;  // bytes per element of the residue or partial-sum planes
};

WsViews views_of(void* ws, const Layout& L) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  return {reinterpret_cast<uint64_t*>(base + L.amax), reinterpret_cast<int32_t*>(base + L.s),
          reinterpret_cast<int32_t*>(base + L.t),     reinterpret_cast<uint16_t*>(base + L.a),
          reinterpret_cast<uint16_t*>(base + L.b),    base + L.out,
          static_cast<size_t>(L.kind == 0 ? 1 : (L.kind == 2 ? 2 : 4))};
}

int record(ozk_event_t* ev, int idx, cudaStream_t stream) {
  if (!ev) return OZK_OK;
  return cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[idx]), stream) == cudaSuccess ? OZK_OK
                                                                                          : OZK_ERR_CUDA;
}

#define OZK_CUDA(expr)                   \
  do {                                   \
    if ((expr) != cudaSuccess) return OZK_ERR_CUDA; \
  } while (0)

// Scan the rows of A inside their quantisation (one block per row, A read
// once) when a row fits one block and there are enough rows to fill the GPU;
// small products keep the separate scan, which spreads rows over more threads.
bool fuse_rows(int64_t M, int64_t kpad) {
  return quantize_rows_fits(kpad) && M <= 0x7FFFFFFF && M * kpad >= (int64_t{1} << 22);
}

// rule 0: scales from each row's (column's) largest entry; rule 1: from the
// computed 2-norm bound (OZK_SCALING_NORM).
int run_dgemm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
              int64_t ldb, double* C, int64_t ldc, int n, void* ws, size_t ws_bytes,
              cudaStream_t stream, ozk_event_t* ev, int rule = 0) {
  int rc = validate(M, N, K, A, lda, B, ldb, C, ldc, n, rule);
  if (rc) return rc;
  if (M == 0 || N == 0) return OZK_OK;
  int sms = 0;
  if ((rc = check_device(&sms))) return rc;
  if (K == 0) {
    OZK_CUDA(cudaMemset2DAsync(C, sizeof(double) * ldc, 0, sizeof(double) * N, M, stream));
    return OZK_OK;
  }
  const Layout L = layout_for(M, N, K, n);
  if (!ws || ws_bytes < L.total || reinterpret_cast<uintptr_t>(ws) % 256) return OZK_ERR_WORKSPACE;
  const auto [amax, s, t, as, bs, out, esize] = views_of(ws, L);
  (void)esize;
  const int budget = rule ? gamma_for(K, n) : beta_for(K, n);
  uint64_t* nsum = rule ? amax + (M + N) : nullptr;  // the norm sums follow the maxima

  if ((rc = record(ev, 0, stream))) return rc;
  if (fuse_rows(M, L.kpad)) {
    // K up to 4096: each row of A is scanned inside its own quantisation
    // (read once); only B's columns need the separate scan, and B's
    // quantisation derives t from the scanned maxima (and norm sums)
    OZK_CUDA(launch_scan(0, N, K, nullptr, 0, B, ldb, amax + M, nsum ? nsum + M : nullptr, stream));
    if ((rc = record(ev, 1, stream))) return rc;
    OZK_CUDA(launch_quantize_rows(M, K, L.kpad, A, lda, n, budget, rule != 0, s, as, L.a_plane, stream));
    OZK_CUDA(launch_quantize(0, N, K, L.kpad, nullptr, 0, B, ldb, nullptr, t, nullptr, amax + M, nullptr,
                             nsum ? nsum + M : nullptr, n, budget, nullptr, 0, bs, L.b_plane, stream));
  } else {
    OZK_CUDA(launch_scan(M, N, K, A, lda, B, ldb, amax, nsum, stream));
    if ((rc = record(ev, 1, stream))) return rc;
    OZK_CUDA(launch_quantize(M, N, K, L.kpad, A, lda, B, ldb, s, t, amax, amax + M, nsum,
                             nsum ? nsum + M : nullptr, n, budget, as, L.a_plane, bs, L.b_plane, stream));
  }
  if ((rc = record(ev, 2, stream))) return rc;
  OZK_CUDA(launch_residue_gemm(M, N, L.kpad, as, L.a_plane, bs, L.b_plane, n, L.kind, out, L.ldo, L.out_plane,
                               L.splits, sms, stream));
  if ((rc = record(ev, 3, stream))) return rc;
  OZK_CUDA(launch_crt(M, N, n, out, L.kind, L.ldo, L.out_plane, L.splits, s, t, C, ldc, nullptr, stream));
  if ((rc = record(ev, 4, stream))) return rc;
  return OZK_OK;
}

}  // namespace

int beta_for(int64_t K, int n) {
  if (n < 2 || n > kMaxModuli) return -1;
  if (K < 1) K = 1;
  Limbs P;
  limbs_set(P, 1);
  for (int k = 0; k < n; ++k) limbs_mul_small(P, modulus_at(k));
  const int num = limbs_msb(P) - 1 - ceil_log2(K);
  const int beta = num >= 0 ? num / 2 : -((-num + 1) / 2);
  return beta >= 1 ? beta : -1;
}

int gamma_for(int64_t K, int n) {
  if (n < 2 || n > kMaxModuli) return -1;
  if (K < 1) K = 1;
  Limbs P;
  limbs_set(P, 1);
  for (int k = 0; k < n; ++k) limbs_mul_small(P, modulus_at(k));
  const int gamma = (limbs_msb(P) - 2) / 2;
  // the rounding slack sqrt(K)/2 of the scaled norms must stay below 2^(gamma - 3)
  if (gamma < 1 || ceil_log2(K) > 2 * gamma - 4) return -1;
  return gamma;
}

int current_device_supported(int* sms) { return check_device(sms); }

const CrtConst& crt_const(int n) {
  std::call_once(g_crt_once, [] {
    for (int k = 2; k <= kMaxModuli; ++k) g_crt[k] = build_crt_const(k);
  });
  return g_crt[n];
}

}  // namespace ozk

using namespace ozk;

extern "C" {

const char* ozk_status_string(int status) {
  switch (status) {
    case OZK_OK: return "ok";
    case OZK_ERR_INVALID_ARG: return "invalid argument";
    case OZK_ERR_UNSUPPORTED: return "unsupported size or moduli count";
    case OZK_ERR_WORKSPACE: return "workspace missing, too small, misaligned or not allocatable";
    case OZK_ERR_CUDA: return "CUDA runtime error";
    case OZK_ERR_TIMEOUT: return "a kernel pipeline wait timed out";
    case OZK_ERR_DEVICE: return "device is not sm_103 (GB300)";
    default: return "unknown status";
  }
}

int ozk_moduli(int n_moduli, int32_t* out) {
  if (n_moduli < 1 || n_moduli > kMaxModuli || !out) return OZK_ERR_INVALID_ARG;
  for (int k = 0; k < n_moduli; ++k) out[k] = static_cast<int32_t>(modulus_at(k));
  return OZK_OK;
}

int ozk_beta(int64_t K, int n_moduli) {
  const int b = beta_for(K, n_moduli);
  return b >= 1 ? b : -OZK_ERR_UNSUPPORTED;
}

int64_t ozk_kpad(int64_t K) { return K <= 0 ? 0 : (K + kKBlock - 1) / kKBlock * kKBlock; }

int ozk_moduli_for_bits(int64_t K, int target_bits) {
  if (target_bits < 1) return -OZK_ERR_INVALID_ARG;
  for (int n = 2; n <= kMaxModuli; ++n)
    if (beta_for(K, n) >= target_bits) return n;
  return -OZK_ERR_UNSUPPORTED;
}

int ozk_dgemm_bits(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
                   int64_t ldb, double* C, int64_t ldc, int target_bits, ozk_stream_t stream) {
  const int n = K == 0 ? 2 : ozk_moduli_for_bits(K, target_bits);
  if (n < 0) return -n;
  return ozk_dgemm(M, N, K, A, lda, B, ldb, C, ldc, n, stream);
}

size_t ozk_workspace_size(int64_t M, int64_t N, int64_t K, int n_moduli) {
  if (M <= 0 || N <= 0 || K <= 0 || K > OZK_MAX_K) return 0;
  if (M > kMaxDim || N > kMaxDim || beta_for(K, n_moduli) < 1) return 0;
  return layout_for(M, N, K, n_moduli).total;
}

int ozk_workspace_layout(int64_t M, int64_t N, int64_t K, int n_moduli, ozk_workspace_info* info) {
  if (!info) return OZK_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0) return OZK_ERR_INVALID_ARG;
  if (K > OZK_MAX_K || M > kMaxDim || N > kMaxDim || n_moduli < 2 || n_moduli > kMaxModuli ||
      beta_for(K, n_moduli) < 1)
    return OZK_ERR_UNSUPPORTED;
  const Layout L = layout_for(M, N, K, n_moduli);
  info->total_bytes = L.total;
  info->maxima_offset = L.amax;
  info->s_offset = L.s;
  info->t_offset = L.t;
  info->a_slices_offset = L.a;
  info->b_slices_offset = L.b;
  info->planes_offset = L.out;
  info->kpad = L.kpad;
  info->a_plane = L.a_plane;
  info->b_plane = L.b_plane;
  info->planes_kind = L.kind;
  info->planes_ld = L.ldo;
  info->planes_plane = L.out_plane;
  info->splits = L.splits;
  return OZK_OK;
}

int ozk_gamma(int64_t K, int n_moduli) {
  const int g = gamma_for(K, n_moduli);
  return g >= 1 ? g : -OZK_ERR_UNSUPPORTED;
}

int ozk_dgemm_norm_ws(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
                      int64_t ldb, double* C, int64_t ldc, int n_moduli, void* workspace, size_t workspace_bytes,
                      ozk_stream_t stream) {
  return run_dgemm(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, workspace, workspace_bytes,
                   reinterpret_cast<cudaStream_t>(stream), nullptr, 1);
}

int ozk_dgemm_norm_ws_timed(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
                            int64_t ldb, double* C, int64_t ldc, int n_moduli, void* workspace,
                            size_t workspace_bytes, ozk_stream_t stream, ozk_event_t* events) {
  return run_dgemm(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, workspace, workspace_bytes,
                   reinterpret_cast<cudaStream_t>(stream), events, 1);
}

int ozk_dgemm_norm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
                   int64_t ldb, double* C, int64_t ldc, int n_moduli, ozk_stream_t stream) {
  int rc = validate(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, 1);
  if (rc) return rc;
  if (M == 0 || N == 0) return OZK_OK;
  if ((rc = check_device(nullptr))) return rc;
  const size_t need = K > 0 ? layout_for(M, N, K, n_moduli).total : 0;
  void* ws = nullptr;
  if (need && (rc = cached_workspace(reinterpret_cast<cudaStream_t>(stream), need, &ws))) return rc;
  return run_dgemm(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, ws, need, reinterpret_cast<cudaStream_t>(stream),
                   nullptr, 1);
}

int ozk_dgemm_ws_timed(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                       const double* B, int64_t ldb, double* C, int64_t ldc, int n_moduli,
                       void* workspace, size_t workspace_bytes, ozk_stream_t stream,
                       ozk_event_t* events) {
  return run_dgemm(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, workspace, workspace_bytes,
                   reinterpret_cast<cudaStream_t>(stream), events);
}

int ozk_dgemm_ws(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
                 int64_t ldb, double* C, int64_t ldc, int n_moduli, void* workspace,
                 size_t workspace_bytes, ozk_stream_t stream) {
  return run_dgemm(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, workspace, workspace_bytes,
                   reinterpret_cast<cudaStream_t>(stream), nullptr);
}

int ozk_dgemm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
              int64_t ldb, double* C, int64_t ldc, int n_moduli, ozk_stream_t stream) {
  int rc = validate(M, N, K, A, lda, B, ldb, C, ldc, n_moduli);
  if (rc) return rc;
  if (M == 0 || N == 0) return OZK_OK;
  if ((rc = check_device(nullptr))) return rc;
  const size_t need = K > 0 ? layout_for(M, N, K, n_moduli).total : 0;
  void* ws = nullptr;
  if (need && (rc = cached_workspace(reinterpret_cast<cudaStream_t>(stream), need, &ws))) return rc;
  return run_dgemm(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, ws, need,
                   reinterpret_cast<cudaStream_t>(stream), nullptr);
}

// Enqueues C = A B for host A, B, C (the work of ozk_dgemm_host_async).
static int host_enqueue(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B, int64_t ldb,
                 double* C, int64_t ldc, int n_moduli, ozk_stream_t stream) {
  int rc = validate(M, N, K, A, lda, B, ldb, C, ldc, n_moduli);
  if (rc) return rc;
  if (M == 0 || N == 0) return OZK_OK;
  int sms = 0;
  if ((rc = check_device(&sms))) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZK_ERR_CUDA;
  HostBufs* hp;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    hp = &g_host[dev];
  }
  HostBufs& h = *hp;
  std::lock_guard<std::mutex> call_lock(h.call);
  HostSlot& sl = h.slot[h.next];
  h.next = (h.next + 1) % kHostSlots;
  auto grow = [&](double*& p, size_t& have, size_t need) -> bool {
    if (have >= need) return true;
    if (p) {
      cudaDeviceSynchronize();  // a call in flight may still use the old buffer
      cudaFree(p);
    }
    p = nullptr;
    have = 0;
    if (need && cudaMalloc(&p, need) != cudaSuccess) return false;
    have = need;
    return true;
  };
  if (!grow(sl.A, sl.a, sizeof(double) * static_cast<size_t>(M * K)) ||
      !grow(sl.B, sl.b, sizeof(double) * static_cast<size_t>(K * N)) ||
      !grow(sl.C, sl.c, sizeof(double) * static_cast<size_t>(M * N)))
    return OZK_ERR_WORKSPACE;
  if (!h.in) {
    if (cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&h.comp, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&h.computed, cudaEventDisableTiming) != cudaSuccess)
      return OZK_ERR_CUDA;
    for (auto& e : h.ev_in)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return OZK_ERR_CUDA;
    for (auto& e : h.ev_out)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return OZK_ERR_CUDA;
    for (auto& x : h.slot)
      if (cudaEventCreateWithFlags(&x.free, cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&x.computed, cudaEventDisableTiming) != cudaSuccess)
        return OZK_ERR_CUDA;
  }
  double *dA = sl.A, *dB = sl.B, *dC = sl.C;
  // Copies in on h.in, the stages on h.comp (every host-buffer call of the
  // device in call order), copies out on h.out.  The call reads and writes
  // only host memory and the library's own buffers, so nothing in it waits
  // for the caller's stream: the copies in start once the stages of the
  // call that used this slot last are done, the stages once that call has
  // copied its C out (a never-recorded event does not hold a stream).  Is a
  // previous call still computing?  Then this call's stages start after it,
  // by which time its copies in are done.
  const cudaError_t q = cudaEventQuery(h.computed);
  if (q != cudaSuccess && q != cudaErrorNotReady) return OZK_ERR_CUDA;
  if (q == cudaErrorNotReady) (void)cudaGetLastError();  // "not ready" is no error
  const bool pipelined = q == cudaErrorNotReady;
  OZK_CUDA(cudaStreamWaitEvent(h.in, sl.computed, 0));
  OZK_CUDA(cudaStreamWaitEvent(h.comp, sl.free, 0));
  cudaStream_t cs = h.comp;
  if (K > 0 && pipelined) {
    // Behind another call: copy A and B in whole, run the stages on the
    // whole product (the fastest schedule once the inputs are there), and
    // combine and copy C out in row blocks, so that most of C is on its way
    // back before the last block is combined.
    const Layout L = layout_for(M, N, K, n_moduli);
    void* ws = nullptr;
    if ((rc = cached_workspace(cs, L.total, &ws))) return rc;
    const auto [amax, s, t, as, bs, out, esize] = views_of(ws, L);
    const int beta = beta_for(K, n_moduli);
    OZK_CUDA(cudaMemcpy2DAsync(dA, sizeof(double) * K, A, sizeof(double) * lda, sizeof(double) * K, M,
                               cudaMemcpyHostToDevice, h.in));
    OZK_CUDA(cudaMemcpy2DAsync(dB, sizeof(double) * N, B, sizeof(double) * ldb, sizeof(double) * N, K,
                               cudaMemcpyHostToDevice, h.in));
    OZK_CUDA(cudaEventRecord(h.ev_in[0], h.in));
    OZK_CUDA(cudaStreamWaitEvent(cs, h.ev_in[0], 0));
    if (fuse_rows(M, L.kpad)) {
      OZK_CUDA(launch_scan(0, N, K, nullptr, 0, dB, N, amax + M, nullptr, cs));
      OZK_CUDA(launch_quantize_rows(M, K, L.kpad, dA, K, n_moduli, beta, false, s, as, L.a_plane, cs));
      OZK_CUDA(launch_quantize(0, N, K, L.kpad, nullptr, 0, dB, N, nullptr, t, nullptr, amax + M, nullptr, nullptr,
                               n_moduli, beta, nullptr, 0, bs, L.b_plane, cs));
    } else {
      OZK_CUDA(launch_scan(M, N, K, dA, K, dB, N, amax, nullptr, cs));
      OZK_CUDA(launch_quantize(M, N, K, L.kpad, dA, K, dB, N, s, t, amax, amax + M, nullptr, nullptr, n_moduli, beta,
                               as, L.a_plane, bs, L.b_plane, cs));
    }
    OZK_CUDA(launch_residue_gemm(M, N, L.kpad, as, L.a_plane, bs, L.b_plane, n_moduli, L.kind, out, L.ldo,
                                 L.out_plane, L.splits, sms, cs));
    const int64_t rows = M >= 2048 ? round_up((M + 7) / 8, 256) : M;  // at most 8 <= kMaxHostBlocks^2 pieces
    int piece = 0;
    for (int64_t r0 = 0; r0 < M; r0 += rows) {
      const int64_t mr = std::min(rows, M - r0);
      OZK_CUDA(launch_crt(mr, N, n_moduli, out + static_cast<size_t>(r0 * L.ldo) * esize, L.kind, L.ldo,
                          L.out_plane, L.splits, s + r0, t, dC + r0 * N, N, nullptr, cs));
      cudaEvent_t done = h.ev_out[piece++];
      OZK_CUDA(cudaEventRecord(done, cs));
      OZK_CUDA(cudaStreamWaitEvent(h.out, done, 0));
      OZK_CUDA(cudaMemcpy2DAsync(C + r0 * ldc, sizeof(double) * ldc, dC + r0 * N, sizeof(double) * N,
                                 sizeof(double) * N, mr, cudaMemcpyDeviceToHost, h.out));
    }
  } else if (K > 0) {
    // Nothing ahead (the latency case): A moves in row blocks and B in
    // column blocks, interleaved (B_0, A_0, A_1, B_1, A_2, B_2, ...); each
    // block is scanned and quantised as soon as it has arrived, the part of
    // C it completes is computed next and goes back while later blocks are
    // still on their way in.  Stage by stage that part is run_dgemm on a
    // rectangle of rows and columns, sharing the scales and slices of its
    // blocks.
    const Layout L = layout_for(M, N, K, n_moduli);
    void* ws = nullptr;
    if ((rc = cached_workspace(cs, L.total, &ws))) return rc;
    const auto [amax, s, t, as, bs, out, esize] = views_of(ws, L);
    const int beta = beta_for(K, n_moduli);
    // blocks of whole 256-row / 256-column tiles (the CTA-pair GEMM's tile),
    // four per dimension once it is long enough to keep every tile's GEMM busy
    const int64_t rows = M >= 2048 ? round_up((M + 3) / 4, 256) : M;
    const int64_t cols = N >= 2048 ? round_up((N + 3) / 4, 256) : N;
    const int nbr = static_cast<int>((M + rows - 1) / rows);  // <= kMaxHostBlocks
    const int nbc = static_cast<int>((N + cols - 1) / cols);  // <= kMaxHostBlocks
    int order[2 * kMaxHostBlocks];  // copy order: +1 + i for A_i, -1 - j for B_j
    int no = 0;
    order[no++] = -1;
    order[no++] = 1;
    for (int i = 1, j = 1; i < nbr || j < nbc; ++i, ++j) {
      if (i < nbr) order[no++] = 1 + i;
      if (j < nbc) order[no++] = -1 - j;
    }
    for (int k = 0; k < no; ++k) {
      if (order[k] > 0) {
        const int64_t r0 = (order[k] - 1) * rows, mr = std::min(rows, M - r0);
        OZK_CUDA(cudaMemcpy2DAsync(dA + r0 * K, sizeof(double) * K, A + r0 * lda, sizeof(double) * lda,
                                   sizeof(double) * K, mr, cudaMemcpyHostToDevice, h.in));
      } else {
        const int64_t c0 = (-order[k] - 1) * cols, nc = std::min(cols, N - c0);
        OZK_CUDA(cudaMemcpy2DAsync(dB + c0, sizeof(double) * N, B + c0, sizeof(double) * ldb, sizeof(double) * nc,
                                   K, cudaMemcpyHostToDevice, h.in));
      }
      OZK_CUDA(cudaEventRecord(h.ev_in[k], h.in));
    }
    // Blocks of each matrix arrive in order, so the blocks in form a prefix
    // of the rows (or columns): the tiles a new block completes make one
    // rectangle.  It is computed in pieces of up to `span` tiles, one GEMM
    // and one CRT launch each: merged where a tile is little work (fewer
    // launches), one tile at a time where it is much (each tile's copy back
    // overlaps the next one's computation, which shortens the tail).
    const double tile_work = static_cast<double>(rows) * static_cast<double>(cols) * static_cast<double>(K);
    const int64_t span = std::max<int64_t>(1, static_cast<int64_t>(1.0e10 / tile_work));
    int64_t rows_in = 0, cols_in = 0;
    int piece = 0;
    for (int k = 0; k < no; ++k) {
      OZK_CUDA(cudaStreamWaitEvent(cs, h.ev_in[k], 0));
      const bool is_a = order[k] > 0;
      const int blk = is_a ? order[k] - 1 : -order[k] - 1;
      int64_t r0, mr, c0, nc;  // the rectangle of C this block completes
      if (is_a) {
        r0 = blk * rows;
        mr = std::min(rows, M - r0);
        if (fuse_rows(mr, L.kpad)) {
          OZK_CUDA(launch_quantize_rows(mr, K, L.kpad, dA + r0 * K, K, n_moduli, beta, false, s + r0,
                                        as + r0 * L.kpad, L.a_plane, cs));
        } else {
          OZK_CUDA(launch_scan(mr, 0, K, dA + r0 * K, K, nullptr, 0, amax + r0, nullptr, cs));
          OZK_CUDA(launch_quantize(mr, 0, K, L.kpad, dA + r0 * K, K, nullptr, 0, s + r0, nullptr, amax + r0, nullptr,
                                   nullptr, nullptr, n_moduli, beta,
                                   as + r0 * L.kpad, L.a_plane, nullptr, 0, cs));
        }
        rows_in = r0 + mr;
        c0 = 0;
        nc = cols_in;
      } else {
        c0 = blk * cols;
        nc = std::min(cols, N - c0);
        OZK_CUDA(launch_scan(0, nc, K, nullptr, 0, dB + c0, N, amax + M + c0, nullptr, cs));
        OZK_CUDA(launch_quantize(0, nc, K, L.kpad, nullptr, 0, dB + c0, N, nullptr, t + c0, nullptr, amax + M + c0,
                                 nullptr, nullptr, n_moduli, beta, nullptr,
                                 0, bs + c0 * L.kpad, L.b_plane, cs));
        cols_in = c0 + nc;
        r0 = 0;
        mr = rows_in;
      }
      // pieces along the rectangle's long side (the blocks already in)
      const int64_t step = is_a ? span * cols : span * rows;
      for (int64_t p0 = 0; p0 < (is_a ? nc : mr); p0 += step) {
        const int64_t pr0 = is_a ? r0 : p0, pmr = is_a ? mr : std::min(step, mr - p0);
        const int64_t pc0 = is_a ? p0 : c0, pnc = is_a ? std::min(step, nc - p0) : nc;
        void* ob = out + static_cast<size_t>(pr0 * L.ldo + pc0) * esize;
        OZK_CUDA(launch_residue_gemm(pmr, pnc, L.kpad, as + pr0 * L.kpad, L.a_plane, bs + pc0 * L.kpad, L.b_plane,
                                     n_moduli, L.kind, ob, L.ldo, L.out_plane, L.splits, sms, cs));
        OZK_CUDA(launch_crt(pmr, pnc, n_moduli, ob, L.kind, L.ldo, L.out_plane, L.splits, s + pr0, t + pc0,
                            dC + pr0 * N + pc0, N, nullptr, cs));
        cudaEvent_t done = h.ev_out[piece++];
        OZK_CUDA(cudaEventRecord(done, cs));
        OZK_CUDA(cudaStreamWaitEvent(h.out, done, 0));
        OZK_CUDA(cudaMemcpy2DAsync(C + pr0 * ldc + pc0, sizeof(double) * ldc, dC + pr0 * N + pc0, sizeof(double) * N,
                                   sizeof(double) * pnc, pmr, cudaMemcpyDeviceToHost, h.out));
      }
    }
  } else {
    OZK_CUDA(cudaMemset2DAsync(dC, sizeof(double) * N, 0, sizeof(double) * N, M, cs));
    OZK_CUDA(cudaEventRecord(h.ev_out[0], cs));
    OZK_CUDA(cudaStreamWaitEvent(h.out, h.ev_out[0], 0));
    OZK_CUDA(cudaMemcpy2DAsync(C, sizeof(double) * ldc, dC, sizeof(double) * N, sizeof(double) * N, M,
                               cudaMemcpyDeviceToHost, h.out));
  }
  OZK_CUDA(cudaEventRecord(h.computed, cs));
  OZK_CUDA(cudaEventRecord(sl.computed, cs));
  // the call is complete, in the caller's stream order, once C is in host memory
  OZK_CUDA(cudaEventRecord(sl.free, h.out));
  OZK_CUDA(cudaStreamWaitEvent(st, sl.free, 0));
  return OZK_OK;
}

int ozk_dgemm_host(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
                   int64_t ldb, double* C, int64_t ldc, int n_moduli, ozk_stream_t stream) {
  const int rc = host_enqueue(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, stream);
  if (rc || M == 0 || N == 0) return rc;  // an empty C: nothing was enqueued
  return cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? OZK_OK : OZK_ERR_CUDA;
}

int ozk_dgemm_host_async(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
                         int64_t ldb, double* C, int64_t ldc, int n_moduli, ozk_stream_t stream) {
  return host_enqueue(M, N, K, A, lda, B, ldb, C, ldc, n_moduli, stream);
}

int ozk_stream_status(ozk_stream_t stream) {
  int status = 0;
  const int rc = take_device_status(reinterpret_cast<cudaStream_t>(stream), &status);
  if (rc) return rc;
  return status ? OZK_ERR_TIMEOUT : OZK_OK;
}

int ozk_release_cached(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZK_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return OZK_ERR_CUDA;
  HostBufs* hp = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = g_host.find(dev);
    if (it != g_host.end()) hp = &it->second;
  }
  if (hp) {  // the entry stays (a call may be waiting on its lock); what it holds goes
    HostBufs& h = *hp;
    std::lock_guard<std::mutex> call_lock(h.call);
    for (auto& sl : h.slot) {
      cudaFree(sl.A);
      cudaFree(sl.B);
      cudaFree(sl.C);
      sl.A = sl.B = sl.C = nullptr;
      sl.a = sl.b = sl.c = 0;
    }
    if (h.in) {
      cudaStreamDestroy(h.in);
      cudaStreamDestroy(h.out);
      cudaStreamDestroy(h.comp);
      cudaEventDestroy(h.computed);
      for (auto& e : h.ev_in) cudaEventDestroy(e);
      for (auto& e : h.ev_out) cudaEventDestroy(e);
      for (auto& sl : h.slot) {
        cudaEventDestroy(sl.free);
        cudaEventDestroy(sl.computed);
      }
      h.in = h.out = h.comp = nullptr;
    }
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  for (auto it = g_ws.begin(); it != g_ws.end();) {
    if (it->first.first == dev) {
      cudaFree(it->second.first);
      it = g_ws.erase(it);
    } else {
      ++it;
    }
  }
  return OZK_OK;
}

int ozk_scale(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
              int64_t ldb, int n_moduli, int32_t* s, int32_t* t, uint64_t* scratch,
              ozk_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return OZK_ERR_INVALID_ARG;
  const int beta = beta_for(K, n_moduli);
  if (beta < 1 || K > OZK_MAX_K || M > kMaxDim || N > kMaxDim) return OZK_ERR_UNSUPPORTED;
  if (M + N == 0) return OZK_OK;
  if (!scratch || (M && !s) || (N && !t)) return OZK_ERR_INVALID_ARG;
  if (K > 0 && ((M && (!A || lda < K)) || (N && (!B || ldb < N)))) return OZK_ERR_INVALID_ARG;
  int rc = check_device(nullptr);
  if (rc) return rc;
  OZK_CUDA(launch_scale(M, N, K, A, lda, B, ldb, beta, s, t, scratch, nullptr,
                        reinterpret_cast<cudaStream_t>(stream)));
  return OZK_OK;
}

int ozk_scale_norm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda, const double* B,
                   int64_t ldb, int n_moduli, int32_t* s, int32_t* t, uint64_t* scratch, ozk_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return OZK_ERR_INVALID_ARG;
  const int gamma = gamma_for(K, n_moduli);
  if (gamma < 1 || K > OZK_MAX_K || M > kMaxDim || N > kMaxDim) return OZK_ERR_UNSUPPORTED;
  if (M + N == 0) return OZK_OK;
  if (!scratch || (M && !s) || (N && !t)) return OZK_ERR_INVALID_ARG;
  if (K > 0 && ((M && (!A || lda < K)) || (N && (!B || ldb < N)))) return OZK_ERR_INVALID_ARG;
  int rc = check_device(nullptr);
  if (rc) return rc;
  OZK_CUDA(launch_scale(M, N, K, A, lda, B, ldb, gamma, s, t, scratch, scratch + (M + N),
                        reinterpret_cast<cudaStream_t>(stream)));
  return OZK_OK;
}

int ozk_quantize_a(int64_t M, int64_t K, const double* A, int64_t lda, const int32_t* s, int n_moduli,
                   uint16_t* a_slices, ozk_stream_t stream) {
  if (M < 0 || K < 0) return OZK_ERR_INVALID_ARG;
  if (n_moduli < 2 || n_moduli > kMaxModuli || K > OZK_MAX_K) return OZK_ERR_UNSUPPORTED;
  if (M == 0 || K == 0) return OZK_OK;
  if (!A || lda < K || !s || !a_slices || reinterpret_cast<uintptr_t>(a_slices) % 32)
    return OZK_ERR_INVALID_ARG;
  const int beta = beta_for(K, n_moduli);
  if (beta < 1) return OZK_ERR_UNSUPPORTED;
  int rc = check_device(nullptr);
  if (rc) return rc;
  // integers wide enough for the scales of either rule (|a'| <= 2^gamma, gamma >= beta)
  const int width = std::max(beta, gamma_for(K, n_moduli));
  OZK_CUDA(launch_quantize(M, 0, K, ozk_kpad(K), A, lda, nullptr, 0, const_cast<int32_t*>(s), nullptr, nullptr,
                           nullptr, nullptr, nullptr, n_moduli, width,
                           a_slices, M * ozk_kpad(K), nullptr, 0, reinterpret_cast<cudaStream_t>(stream)));
  return OZK_OK;
}

int ozk_quantize_b(int64_t K, int64_t N, const double* B, int64_t ldb, const int32_t* t, int n_moduli,
                   uint16_t* b_slices, ozk_stream_t stream) {
  if (N < 0 || K < 0) return OZK_ERR_INVALID_ARG;
  if (n_moduli < 2 || n_moduli > kMaxModuli || K > OZK_MAX_K) return OZK_ERR_UNSUPPORTED;
  if (N == 0 || K == 0) return OZK_OK;
  if (!B || ldb < N || !t || !b_slices || reinterpret_cast<uintptr_t>(b_slices) % 32)
    return OZK_ERR_INVALID_ARG;
  const int beta = beta_for(K, n_moduli);
  if (beta < 1) return OZK_ERR_UNSUPPORTED;
  int rc = check_device(nullptr);
  if (rc) return rc;
  const int width = std::max(beta, gamma_for(K, n_moduli));
  OZK_CUDA(launch_quantize(0, N, K, ozk_kpad(K), nullptr, 0, B, ldb, nullptr, const_cast<int32_t*>(t), nullptr,
                           nullptr, nullptr, nullptr, n_moduli, width,
                           nullptr, 0, b_slices, N * ozk_kpad(K), reinterpret_cast<cudaStream_t>(stream)));
  return OZK_OK;
}

int ozk_residue_gemm(int64_t M, int64_t N, int64_t K, const uint16_t* a_slices,
                     const uint16_t* b_slices, int n_moduli, int out_kind, void* out, int64_t ldo,
                     int splits, ozk_stream_t stream) {
  if (M < 0 || N < 0 || K < 0) return OZK_ERR_INVALID_ARG;
  if (n_moduli < 2 || n_moduli > kMaxModuli || K > OZK_MAX_K) return OZK_ERR_UNSUPPORTED;
  if (M > kMaxDim || N > kMaxDim) return OZK_ERR_UNSUPPORTED;
  if (M == 0 || N == 0 || K == 0) return OZK_OK;
  const int64_t kpad = ozk_kpad(K);
  if (!a_slices || !b_slices || !out) return OZK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(a_slices) % 16 || reinterpret_cast<uintptr_t>(b_slices) % 16 ||
      reinterpret_cast<uintptr_t>(out) % 16)
    return OZK_ERR_INVALID_ARG;
  if (out_kind == 0) {
    if (splits != 1 || ldo < N || ldo % 16) return OZK_ERR_INVALID_ARG;
    if (K >= (int64_t{1} << 17)) return OZK_ERR_INVALID_ARG;  // one int32-exact sum over all of K
  } else if (out_kind == 1) {
    if (splits < 1 || splits > 64 || splits > kpad / kKBlock || ldo < N || ldo % 4)
      return OZK_ERR_INVALID_ARG;
    // each split's K (whole 64-blocks) must keep its int32 sums exact
    if ((kpad / kKBlock + splits - 1) / splits * kKBlock > OZK_SPLIT_MAX_K) return OZK_ERR_INVALID_ARG;
  } else if (out_kind == 2) {
    if (splits != 1 || ldo < N || ldo % 8) return OZK_ERR_INVALID_ARG;
    if (K >= (int64_t{1} << 17)) return OZK_ERR_INVALID_ARG;
  } else {
    return OZK_ERR_INVALID_ARG;
  }
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  OZK_CUDA(launch_residue_gemm(M, N, kpad, a_slices, M * kpad, b_slices, N * kpad, n_moduli, out_kind,
                               out, ldo, M * ldo, splits, sms, reinterpret_cast<cudaStream_t>(stream)));
  return OZK_OK;
}

int ozk_residue_gemm_withheld(int64_t M, int64_t N, int64_t K, const uint16_t* a_slices,
                              const uint16_t* b_slices, int n_moduli, uint8_t* out, int64_t ldo,
                              int withhold_kb, uint32_t timeout_us, ozk_stream_t stream) {
  if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim) return OZK_ERR_INVALID_ARG;
  if (n_moduli < 2 || n_moduli > kMaxModuli) return OZK_ERR_UNSUPPORTED;
  const int64_t kpad = ozk_kpad(K);
  if (kpad >= 2048 || withhold_kb < 0 || withhold_kb >= kpad / kKBlock) return OZK_ERR_INVALID_ARG;
  if (timeout_us < 1 || timeout_us > 1000000) return OZK_ERR_INVALID_ARG;
  if (!a_slices || !b_slices || !out || ldo < N || ldo % 16) return OZK_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(a_slices) % 16 || reinterpret_cast<uintptr_t>(b_slices) % 16 ||
      reinterpret_cast<uintptr_t>(out) % 16)
    return OZK_ERR_INVALID_ARG;
  int sms = 0;
  int rc = check_device(&sms);
  if (rc) return rc;
  OZK_CUDA(launch_residue_gemm_withheld(M, N, kpad, a_slices, M * kpad, b_slices, N * kpad, n_moduli, out, ldo,
                                        M * ldo, sms, 1000ull * timeout_us, withhold_kb,
                                        reinterpret_cast<cudaStream_t>(stream)));
  return OZK_OK;
}

static int check_crt_args(int64_t M, int64_t N, int n_moduli, const void* in, int in_kind,
                          int64_t ldi, int splits) {
  if (M < 0 || N < 0) return OZK_ERR_INVALID_ARG;
  if (n_moduli < 2 || n_moduli > kMaxModuli) return OZK_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return OZK_OK;
  if (!in || reinterpret_cast<uintptr_t>(in) % 16) return OZK_ERR_INVALID_ARG;
  if (in_kind == 0) {
    if (splits != 1 || ldi < N || ldi % 16) return OZK_ERR_INVALID_ARG;
  } else if (in_kind == 1) {
    if (splits < 1 || splits > 64 || ldi < N || ldi % 4) return OZK_ERR_INVALID_ARG;
  } else if (in_kind == 2) {
    if (splits != 1 || ldi < N || ldi % 8) return OZK_ERR_INVALID_ARG;
  } else {
    return OZK_ERR_INVALID_ARG;
  }
  return OZK_OK;
}

int ozk_crt_combine(int64_t M, int64_t N, int n_moduli, const void* in, int in_kind, int64_t ldi,
                    int splits, const int32_t* s, const int32_t* t, double* C, int64_t ldc,
                    ozk_stream_t stream) {
  int rc = check_crt_args(M, N, n_moduli, in, in_kind, ldi, splits);
  if (rc || M == 0 || N == 0) return rc;
  if (!s || !t || !C || ldc < N) return OZK_ERR_INVALID_ARG;
  if ((rc = check_device(nullptr))) return rc;
  OZK_CUDA(launch_crt(M, N, n_moduli, in, in_kind, ldi, M * ldi, splits, s, t, C, ldc, nullptr,
                      reinterpret_cast<cudaStream_t>(stream)));
  return OZK_OK;
}

int ozk_crt_lift(int64_t M, int64_t N, int n_moduli, const void* in, int in_kind, int64_t ldi,
                 int splits, uint32_t* X, ozk_stream_t stream) {
  int rc = check_crt_args(M, N, n_moduli, in, in_kind, ldi, splits);
  if (rc || M == 0 || N == 0) return rc;
  if (!X) return OZK_ERR_INVALID_ARG;
  if ((rc = check_device(nullptr))) return rc;
  OZK_CUDA(launch_crt(M, N, n_moduli, in, in_kind, ldi, M * ldi, splits, nullptr, nullptr, nullptr, 0, X,
                      reinterpret_cast<cudaStream_t>(stream)));
  return OZK_OK;
}

int ozk_event_create(ozk_event_t* ev) {
  if (!ev) return OZK_ERR_INVALID_ARG;
  cudaEvent_t e;
  if (cudaEventCreate(&e) != cudaSuccess) return OZK_ERR_CUDA;
  *ev = reinterpret_cast<ozk_event_t>(e);
  return OZK_OK;
}

int ozk_event_destroy(ozk_event_t ev) {
  return cudaEventDestroy(reinterpret_cast<cudaEvent_t>(ev)) == cudaSuccess ? OZK_OK : OZK_ERR_CUDA;
}

int ozk_event_record(ozk_event_t ev, ozk_stream_t stream) {
  return cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev), reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? OZK_OK
             : OZK_ERR_CUDA;
}

int ozk_event_elapsed(ozk_event_t start, ozk_event_t stop, float* ms) {
  if (!ms) return OZK_ERR_INVALID_ARG;
  if (cudaEventSynchronize(reinterpret_cast<cudaEvent_t>(stop)) != cudaSuccess) return OZK_ERR_CUDA;
  return cudaEventElapsedTime(ms, reinterpret_cast<cudaEvent_t>(start),
                              reinterpret_cast<cudaEvent_t>(stop)) == cudaSuccess
             ? OZK_OK
             : OZK_ERR_CUDA;
}

int ozk_device_sm_count(void) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return sms;
}

}  // extern "C"
