/*
 * ozk — FP64 GEMM emulated with exact integer residue GEMMs on GB300 tensor
 * cores and Chinese-Remainder reconstruction (Ozaki scheme II).
 *
 * Method source: the "Day 12" page on ithelp.ithome.com.tw (Ozaki-II
 * INT8/CRT FP64 GEMM emulation).  Its section "Profile 不能只看 Tensor Core"
 * lists the pipeline this library implements, stage by stage:
 *   scale / exponent scan -> residue quantization -> integer GEMM per modulus
 *   -> mod reduction -> CRT reconstruction -> undo scaling -> write double.
 * Its section "先定義公平比較" fixes the boundary: double in, double out.
 *
 * Conventions for every entry point:
 *  - A is M x K, B is K x N, C is M x N, all row-major double, leading
 *    dimensions in elements (lda >= K, ldb >= N, ldc >= N).  C = A * B.
 *  - n_moduli (2..20) selects the first n of the moduli
 *    {256,255,253,251,247,241,239,233,229,227,223,217,211,199,197,193,191,181,179,173}.
 *    14 gives about a 53-bit product, 8 about 26 bits per operand.
 *  - Device pointers belong to the caller; the library never frees them.
 *  - ozk_stream_t is a cudaStream_t (NULL = legacy default stream).  Work is
 *    stream-ordered and asynchronous unless stated otherwise.  The library's
 *    kernels allow programmatic dependent launch: each waits for the work
 *    before it, and lets the kernel after it launch early.  A caller kernel
 *    launched after a call with programmatic stream serialisation allowed
 *    must itself wait (griddepcontrol.wait, cudaGridDependencySynchronize)
 *    before it reads the call's results; ordinary launches, copies and
 *    events are ordered as usual.
 *  - Argument errors are returned synchronously before anything is launched.
 *    Launch failures return OZK_ERR_CUDA.  Faults detected inside a kernel
 *    (a pipeline wait that ran out) are latched on the device and reported by
 *    ozk_stream_status().
 *  - Sizes M, N or K equal to 0 are valid: nothing is computed, and for K = 0
 *    (with M, N > 0) C is filled with zeros.
 *  - Requires a GB300-class GPU (sm_103a); other devices give OZK_ERR_DEVICE.
 */
#ifndef OZK_H
#define OZK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ozk_stream_t; /* identical to cudaStream_t */
typedef struct CUevent_st* ozk_event_t;   /* identical to cudaEvent_t */

typedef enum {
  OZK_OK = 0,
  OZK_ERR_INVALID_ARG = 1, /* bad pointer, size, leading dimension or overlap */
  OZK_ERR_UNSUPPORTED = 2, /* K > OZK_MAX_K, M or N > 2^30 - 1, n_moduli outside 2..20, or too few moduli for K */
  OZK_ERR_WORKSPACE = 3,   /* caller workspace too small, or allocation failed */
  OZK_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  OZK_ERR_TIMEOUT = 5,     /* a kernel's bounded pipeline wait ran out (device-side) */
  OZK_ERR_DEVICE = 6       /* current device is not sm_103 */
} ozk_status;

#define OZK_MAX_MODULI 20
#define OZK_MAX_K 4194304          /* K = 2^22; the workspace holds 2 n (M + N) K bytes of slices */
#define OZK_SPLIT_MAX_K 131008     /* K of one int32-exact partial sum: 2^14 * K < 2^31, whole 64-blocks */
#define OZK_SCALE_NONFINITE INT32_MIN
#define OZK_LIMBS 8                /* lifted integers: 8 x uint32, two's complement */

/* ------------------------------------------------------------------ */
/* Host-only helpers (no CUDA calls).                                  */
/* ------------------------------------------------------------------ */

/* Human-readable text for a status code.  Never NULL. */
const char* ozk_status_string(int status);

/* Writes the first n_moduli moduli to out[0..n-1].  Returns OZK_OK or
 * OZK_ERR_INVALID_ARG. */
int ozk_moduli(int n_moduli, int32_t* out);

/* Bits per operand beta for inner dimension K: the largest even split of
 * floor(log2 P) - 1 - ceil(log2 K) bits, P the product of the moduli, so that
 * the symmetric CRT lift of sum_k a'_ik b'_kj is exact.  Returns beta >= 1,
 * or -OZK_ERR_UNSUPPORTED when the moduli cannot cover K. */
int ozk_beta(int64_t K, int n_moduli);

/* The moduli count for a target precision: the smallest n_moduli in 2..20
 * with ozk_beta(K, n_moduli) >= target_bits, i.e. every element of A and B
 * keeps at least target_bits bits below the largest magnitude of its row of A
 * or column of B (the fixed-mantissa contract of the "Day 12" page's
 * precision-contract list, "先定義公平比較": target mantissa bits beside the
 * modulus count).  Returns the count, -OZK_ERR_INVALID_ARG when
 * target_bits < 1, or -OZK_ERR_UNSUPPORTED when 20 moduli do not reach it. */
int ozk_moduli_for_bits(int64_t K, int target_bits);

/* Norm budget gamma of the norm scaling rule (ozk_dgemm_norm):
 * floor((floor(log2 P) - 2) / 2), so that two scaled vectors of 2-norm at
 * most 2^gamma (plus the rounding slack sqrt(K)/2, required to stay below
 * 2^(gamma - 3)) keep the symmetric CRT lift of their dot product exact.
 * Returns gamma, or -OZK_ERR_UNSUPPORTED. */
int ozk_gamma(int64_t K, int n_moduli);

/* Row length of the residue slices: K rounded up to a multiple of 64. */
int64_t ozk_kpad(int64_t K);

/* Bytes of device workspace ozk_dgemm_ws needs for this problem (0 when
 * nothing is computed).  Returns 0 as well for unsupported arguments, which
 * ozk_dgemm_ws then reports. */
size_t ozk_workspace_size(int64_t M, int64_t N, int64_t K, int n_moduli);

/* Where one ozk_dgemm_ws call keeps each stage's results in its workspace,
 * for reading them back after the call (the intermediate buffers of a real
 * call in its own launch configuration: scales, residue slices, residue
 * planes).  Offsets are in bytes from the workspace start; plane strides
 * in elements of the region's type.  The layout is an implementation
 * detail of this library version: use it for inspection, not storage. */
typedef struct {
  size_t total_bytes;       /* = ozk_workspace_size */
  size_t maxima_offset;     /* uint64 abs-bit maxima: rows of A, then columns of B */
  size_t s_offset;          /* int32 s[M] */
  size_t t_offset;          /* int32 t[N] */
  size_t a_slices_offset;   /* fp16 [n][M][kpad], modulus planes a_plane elements apart */
  size_t b_slices_offset;   /* fp16 [n][N][kpad] (B transposed), b_plane elements apart */
  size_t planes_offset;     /* the residue GEMM's output, in the layout of planes_kind */
  int64_t kpad;
  int64_t a_plane, b_plane;
  int planes_kind;          /* 0: uint8 residues, 1: int32 split-K sums (the out_kind of
                               ozk_residue_gemm; its kind 2, pair residues, is not chosen here) */
  int64_t planes_ld;        /* row stride of a plane, elements */
  int64_t planes_plane;     /* elements between consecutive planes */
  int splits;               /* K splits (planes_kind 1) */
} ozk_workspace_info;

/* Fills *info for ozk_dgemm_ws(M, N, K, ..., n_moduli).  OZK_ERR_INVALID_ARG
 * for a null info or an empty product, OZK_ERR_UNSUPPORTED as ozk_dgemm. */
int ozk_workspace_layout(int64_t M, int64_t N, int64_t K, int n_moduli, ozk_workspace_info* info);

/* ------------------------------------------------------------------ */
/* The GEMM.                                                           */
/* ------------------------------------------------------------------ */

/* ozk_dgemm with n_moduli = ozk_moduli_for_bits(K, target_bits); errors of
 * that choice are returned as positive status codes.  K = 0 (nothing to
 * reduce) uses 2 moduli. */
int ozk_dgemm_bits(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                   const double* B, int64_t ldb, double* C, int64_t ldc,
                   int target_bits, ozk_stream_t stream);

/* C = A * B with n_moduli residue GEMMs.  A, B, C are device pointers.
 * C must not overlap A or B (OZK_ERR_INVALID_ARG).  Rows of A or columns of
 * B that hold an Inf or NaN give NaN rows/columns of C.  Uses a workspace the
 * library allocates on first use and caches per (device, stream); calls on
 * different streams therefore never share scratch memory. */
int ozk_dgemm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
              const double* B, int64_t ldb, double* C, int64_t ldc,
              int n_moduli, ozk_stream_t stream);

/* As ozk_dgemm, with caller-provided device workspace of at least
 * ozk_workspace_size(M, N, K, n_moduli) bytes (256-byte aligned).  The
 * library allocates nothing.  Calls that share a workspace must be ordered
 * on one stream.  After one call of the same shape on the device (which
 * sets up the kernels), a call only enqueues work on `stream`: it neither
 * synchronises nor allocates, so it can be captured into a CUDA graph
 * (worth it for small products, where launch latency is a large share). */
int ozk_dgemm_ws(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                 const double* B, int64_t ldb, double* C, int64_t ldc,
                 int n_moduli, void* workspace, size_t workspace_bytes,
                 ozk_stream_t stream);

/* As ozk_dgemm_ws, recording events[0..4] on the stream at the stage
 * boundaries (before scan, before quantize, before the residue GEMM,
 * before the CRT combine, after it) when events is not NULL.  The events are
 * the caller's (create them with ozk_event_create). */
int ozk_dgemm_ws_timed(int64_t M, int64_t N, int64_t K, const double* A,
                       int64_t lda, const double* B, int64_t ldb, double* C,
                       int64_t ldc, int n_moduli, void* workspace,
                       size_t workspace_bytes, ozk_stream_t stream,
                       ozk_event_t* events);

/* ozk_dgemm with the sharper scaling rule: the scale of row i of A is the
 * largest s_i with 2^s_i ||a_i||_2 <= 2^gamma (ozk_gamma), from an exactly
 * computed bound on the row's 2-norm (ozk_scale_norm), and likewise t_j for
 * the columns of B.  By Cauchy-Schwarz, sum_k |a'_ik||b'_kj| <=
 * ||a'_i|| ||b'_j|| then stays below P/2, so the method is as exact as with
 * the largest-entry rule while each operand keeps more bits wherever a row's
 * entries are not all near its largest (about 1.2 more bits per operand for
 * Gaussian data at K = 4096); the same precision contract can then be met
 * with fewer moduli.  The pages' precision-contract list (the "Day 12" page,
 * section "先定義公平比較") sets moduli count against target bits; this rule
 * is the library's reading of its "sharper scaling" step, not the pages'.
 * Costs one more pass over the operands whose rows are scanned separately (B,
 * and A when its rows are longer than 4096).  Same arguments, workspace and
 * errors as ozk_dgemm / ozk_dgemm_ws; OZK_ERR_UNSUPPORTED when ozk_gamma
 * rejects K. */
int ozk_dgemm_norm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                   const double* B, int64_t ldb, double* C, int64_t ldc,
                   int n_moduli, ozk_stream_t stream);
int ozk_dgemm_norm_ws(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                      const double* B, int64_t ldb, double* C, int64_t ldc,
                      int n_moduli, void* workspace, size_t workspace_bytes,
                      ozk_stream_t stream);
/* ozk_dgemm_norm_ws with the stage events of ozk_dgemm_ws_timed. */
int ozk_dgemm_norm_ws_timed(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                            const double* B, int64_t ldb, double* C, int64_t ldc,
                            int n_moduli, void* workspace, size_t workspace_bytes,
                            ozk_stream_t stream, ozk_event_t* events);

/* C = A * B for HOST matrices (pinned memory gives the fastest copies and
 * the overlap).  A goes to the device in row blocks and B in column blocks
 * (four of each once M, resp. N, reaches 2048), interleaved on a copy
 * stream of the library; each block is scanned and quantised on `stream` as
 * soon as it has arrived, each tile of C as soon as its two blocks are in,
 * and the tile goes back on a second copy stream while later blocks are
 * still moving.  Returns after C is complete in host memory; C is the same,
 * bit for bit, as ozk_dgemm's.  Device buffers, streams and events are
 * cached per device; concurrent calls on one device are serialised. */
int ozk_dgemm_host(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                   const double* B, int64_t ldb, double* C, int64_t ldc,
                   int n_moduli, ozk_stream_t stream);

/* ozk_dgemm_host without the wait: returns once the copies and stages are
 * enqueued.  The call is complete, in `stream`'s order, when C is in host
 * memory: synchronise `stream` (or an event recorded on it after the call)
 * before reading C, and keep A and B unchanged and C untouched until then.
 * Only the completion is ordered on `stream`: the call touches no device
 * memory of the caller, and its copies of A and B start at once, so A and B
 * must hold their values when the call is made (device work that writes
 * them must have finished).
 * The library keeps two sets of device buffers per device and uses them in
 * turn, so the next call's A and B move in while this call computes; a
 * third call's copies wait on the device (not on the host) until the first
 * call's C has been copied out.  The stages of all host-buffer calls of a
 * device run in call order on a stream of the library: a call made while
 * an earlier one is still
 * computing copies A and B in whole and runs the stages on the whole
 * product (its inputs are in by the time it starts), then combines and
 * copies C out in row blocks; a call with nothing ahead of it uses the
 * blocked schedule of ozk_dgemm_host.  Calls made on one stream complete in order;
 * concurrent calls on one device are serialised while they enqueue.  Host
 * memory should be pinned: with pageable memory the copies (and so the
 * call) are synchronous.  Same arguments, results and errors as
 * ozk_dgemm_host; device faults are reported by ozk_stream_status. */
int ozk_dgemm_host_async(int64_t M, int64_t N, int64_t K, const double* A,
                         int64_t lda, const double* B, int64_t ldb, double* C,
                         int64_t ldc, int n_moduli, ozk_stream_t stream);

/* Synchronises the stream, then reports and clears a fault latched by a
 * kernel (OZK_ERR_TIMEOUT), or OZK_ERR_CUDA if the stream reported an error. */
int ozk_stream_status(ozk_stream_t stream);

/* Releases the cached workspaces and host-copy buffers of the current device. */
int ozk_release_cached(void);

/* ------------------------------------------------------------------ */
/* Stage entry points (the same kernels ozk_dgemm runs, one at a time). */
/* All pointers are device pointers.                                   */
/* ------------------------------------------------------------------ */

/* Exponent scan ("scale / exponent scan").  s[i] = beta - E_i where
 * max_k |a_ik| = f 2^E_i with f in [0.5, 1); t[j] likewise over the columns
 * of B.  0 for an all-zero row/column, OZK_SCALE_NONFINITE when it holds an
 * Inf or NaN.  scratch: (M + N) uint64 of device scratch memory, overwritten. */
int ozk_scale(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
              const double* B, int64_t ldb, int n_moduli, int32_t* s, int32_t* t,
              uint64_t* scratch, ozk_stream_t stream);

/* The exponent scan of ozk_scale for callers that cannot give the library
 * device memory: a library embedded in an application whose allocator owns
 * all device memory, or a latency-critical loop that must not call
 * cudaMalloc (which may synchronise the device).  The method's pages have
 * no such entry point; it is the same scan with its (M + N) uint64 of scratch held
 * in a fixed 2 MiB array compiled into the library (each GPU that loads the
 * library keeps it until the process exits), so it allocates nothing.
 * Same arguments and results as ozk_scale without `scratch`.
 *  - M + N above OZK_SCALE_NOALLOC_MAX returns OZK_ERR_WORKSPACE (nothing runs).
 *  - The first call on a device looks up the array's device address (a
 *    one-time set-up, no allocation); make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one array: calls whose kernels may
 *    overlap on the GPU (different streams without ordering) race and give
 *    wrong scales.  Each call clears the part of the array it uses. */
#define OZK_SCALE_NOALLOC_MAX 262144
int ozk_scale_noalloc(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                      const double* B, int64_t ldb, int n_moduli, int32_t* s, int32_t* t,
                      ozk_stream_t stream);

/* The scales of the norm rule: with H_i = max_k floor(2 log2 |a_ik|) and
 * S_i = sum over the nonzero entries of 2^max(floor(2 log2 |a_ik|) - H_i + 30, 0)
 * (an exact integer, the same for any summation order; ||a_i||_2^2 <
 * S_i 2^(H_i - 29)), s_i = floor((2 gamma - (H_i - 29) - ceil(log2 S_i)) / 2);
 * t_j likewise over the columns of B.  0 for an all-zero row/column,
 * OZK_SCALE_NONFINITE when it holds an Inf or NaN.  scratch: 2 (M + N)
 * uint64 of device scratch memory, overwritten. */
int ozk_scale_norm(int64_t M, int64_t N, int64_t K, const double* A, int64_t lda,
                   const double* B, int64_t ldb, int n_moduli, int32_t* s, int32_t* t,
                   uint64_t* scratch, ozk_stream_t stream);

/* Residue quantisation of A ("double load, exponent scaling, round, mod,
 * balanced int8 conversion").  For each modulus p and element:
 * a'_ik = a_ik 2^s_i rounded to the nearest integer (ties to even) and
 * r = sym(a' mod p) in [-floor(p/2), ceil(p/2)-1],
 * stored as IEEE binary16 (fp16; exact for these integers) at
 * a_slices[(p * M + i) * kpad + k]; columns K..kpad-1 are zero.
 * kpad = ozk_kpad(K); a_slices must be 32-byte aligned.  Rows with
 * s_i = OZK_SCALE_NONFINITE are zero.  The scales may come from ozk_scale or
 * ozk_scale_norm.  Returns OZK_ERR_UNSUPPORTED when
 * ozk_beta(K, n_moduli) < 1. */
int ozk_quantize_a(int64_t M, int64_t K, const double* A, int64_t lda,
                   const int32_t* s, int n_moduli, uint16_t* a_slices,
                   ozk_stream_t stream);

/* Residue quantisation of B, transposed to K-major: the residue of b'_kj is
 * stored at b_slices[(p * N + j) * kpad + k]; rows K..kpad-1 are zero;
 * b_slices must be 32-byte aligned. */
int ozk_quantize_b(int64_t K, int64_t N, const double* B, int64_t ldb,
                   const int32_t* t, int n_moduli, uint16_t* b_slices,
                   ozk_stream_t stream);

/* One integer GEMM per modulus ("INT8 GEMM", run on fp16 tensor cores: every
 * product and every partial sum of up to 1024 terms is an exact fp32 integer)
 * with the mod reduction fused into its epilogue.
 *  out_kind 0: out is uint8 [n][M][ldo], c = (sum_k ra rb) mod p in [0, p);
 *              ldo >= N, a multiple of 16; splits must be 1 and K < 2^17
 *              (one int32-exact sum).
 *  out_kind 1: out is int32 [splits][n][M][ldo], the exact partial sums over
 *              the split'th share of K, ceil(kpad/64/splits) blocks of 64
 *              (their sum is the exact dot product); ldo >= N, a multiple of 4;
 *              each share must hold at most OZK_SPLIT_MAX_K terms, so K beyond
 *              that needs at least ceil(kpad / OZK_SPLIT_MAX_K) splits.
 *  out_kind 2: out is uint16 [(n+1)/2][M][ldo]: plane j holds the residue of
 *              the moduli pair (2j, 2j+1), the unique r < p_2j p_2j+1 with
 *              r = c_2j mod p_2j and r = c_2j+1 mod p_2j+1 (the first CRT step,
 *              done in the epilogue); for odd n the last plane holds c_n-1.
 *              ldo >= N, a multiple of 8; splits must be 1 and K < 2^17.
 * K is the inner dimension the slices were quantised with (kpad = ozk_kpad(K)).
 * splits in 1..64 and at most kpad/64; violations return OZK_ERR_INVALID_ARG. */
int ozk_residue_gemm(int64_t M, int64_t N, int64_t K, const uint16_t* a_slices,
                     const uint16_t* b_slices, int n_moduli, int out_kind,
                     void* out, int64_t ldo, int splits, ozk_stream_t stream);

/* CRT reconstruction with symmetric lift, undo scaling, FP64 write:
 * C_ij = RN-even(X_ij 2^-(s_i + t_j)) with X_ij the unique integer in
 * [-P/2, P/2) congruent to the residues; NaN where s_i or t_j is
 * OZK_SCALE_NONFINITE.  in / in_kind / ldi / splits as ozk_residue_gemm's out
 * (in_kind 0, 1 or 2); int32 partial sums are reduced mod p one by one before
 * they are added. */
int ozk_crt_combine(int64_t M, int64_t N, int n_moduli, const void* in,
                    int in_kind, int64_t ldi, int splits, const int32_t* s,
                    const int32_t* t, double* C, int64_t ldc, ozk_stream_t stream);

/* The lifted integers themselves, X[(i * N + j) * OZK_LIMBS + l] (limb l of
 * a two's-complement 256-bit value, least significant first).  For checking
 * the integer stage. */
int ozk_crt_lift(int64_t M, int64_t N, int n_moduli, const void* in, int in_kind,
                 int64_t ldi, int splits, uint32_t* X, ozk_stream_t stream);

/* ------------------------------------------------------------------ */
/* Test hook of the failure path.                                      */
/* ------------------------------------------------------------------ */

/* ozk_residue_gemm (out_kind 0, one split) on the single-CTA kernel with
 * every pipeline wait limited to timeout_us microseconds (1..10^6) and the
 * copy of k-block withhold_kb (0 .. kpad/64 - 1) of the first tile of CTA 0
 * never issued.  The wait of that CTA's MMA issuer for the missing stage runs
 * out: the kernel latches OZK_ERR_TIMEOUT, every role of the CTA stops, the
 * copies and MMAs in flight drain, TMEM is freed and the kernel returns; the
 * other CTAs finish their tiles.  Nothing faults or hangs, so the context
 * stays usable.  Every pipeline wait of the library is bounded because a
 * wrong mbarrier phase or arrive count leaves a wait hanging (the async
 * Tensor Core article on yfxerp.com, section 6.1); this call is how a test
 * reaches that bound.  Returns OZK_OK once launched (ozk_stream_status then reports
 * OZK_ERR_TIMEOUT); OZK_ERR_INVALID_ARG for K with kpad >= 2048 (the CTA-pair
 * kernel), a k-block or time limit out of range, or the arguments
 * ozk_residue_gemm rejects.  The planes of the withheld CTA's tiles are not
 * written. */
int ozk_residue_gemm_withheld(int64_t M, int64_t N, int64_t K, const uint16_t* a_slices,
                              const uint16_t* b_slices, int n_moduli, uint8_t* out, int64_t ldo,
                              int withhold_kb, uint32_t timeout_us, ozk_stream_t stream);

/* ------------------------------------------------------------------ */
/* Timing helpers (thin wrappers of the CUDA runtime).                 */
/* ------------------------------------------------------------------ */
int ozk_event_create(ozk_event_t* ev);
int ozk_event_destroy(ozk_event_t ev);
int ozk_event_record(ozk_event_t ev, ozk_stream_t stream);
/* Milliseconds between two recorded events (synchronises on the second). */
int ozk_event_elapsed(ozk_event_t start, ozk_event_t stop, float* ms);

/* Number of SMs of the current device (for sizing), or -1 on error. */
int ozk_device_sm_count(void);

#ifdef __cplusplus
}
#endif
#endif /* OZK_H */
