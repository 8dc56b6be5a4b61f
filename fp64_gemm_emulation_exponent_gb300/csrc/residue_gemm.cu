// One integer GEMM per modulus with the mod reduction fused into the epilogue
// (the "INT8 GEMM" and "mod reduction" stages of the Ozaki-II pipeline on the
// "Day 12" page, section "Profile 不能只看 Tensor Core"; its section
// "一次 NCU 結果怎麼解讀" shows a register-starved mma.sync kernel, 218
// registers per thread and the Tensor pipe at 7.5%).
//
// GB300 (sm_103a) has no tcgen05 kind::i8, so the residues (integers in
// [-128, 127]) are fed to the fp16 tensor cores, where they are exact: every
// product is an integer of magnitude at most 2^14, so every fp32 partial sum
// of a 1024-term chunk is an integer of magnitude at most 2^24 and the fp32
// accumulator in TMEM holds the chunk's exact integer sum.  For residues
// the epilogue warps stay in fp32, two outputs per packed instruction: one
// chunk is reduced mod p directly; several are each cut to a small remainder
// and added up, then reduced once.  For exact sums (split-K shares, and pair
// residues over eight or more chunks, where that is cheaper per chunk) they
// convert each chunk exactly (cvt.rni) and add it into int32 registers
// (exact for K < 2^17).
// Outputs: the residues mod p as uint8 planes (out_kind 0); the exact int32
// sums of a K split (1); or, with the two moduli of a pair run back to back
// on one tile, the uint16 residue of the pair modulus p_2j p_2j+1 (2, the
// first CRT step), the first modulus's residues parked in shared memory.
//
// Two kernels, chosen by the K of a split:
//  * K >= 2048: CTA pairs (clusters of two).  The even CTA issues
//    tcgen05.mma.cta_group::2 (M=256, N=256, K=16): each CTA stages its 128
//    rows of A and half of the B tile, so a stage is 32 KB per SM, the ring is
//    6 deep and the shared-memory traffic per MMA is a third lower than with
//    one CTA per tile.  Both CTAs drain their own 128 accumulator rows.
//  * K < 2048: one CTA per 128 x 256 tile, 4-stage ring.  Up to K = 1024
//    the tile's sums are one chunk: the epilogue loads all of its 128
//    columns, hands the accumulator back to the MMA issuer at once and
//    reduces in fp32 while the next tile accumulates (at short K the
//    epilogue, not the tensor core, set the pace of the int32 form).
//
// Structure of both: persistent CTAs (one per SM), warp-specialised.
//   warp 0      TMA producer: A and B slice tiles into the smem ring (128-byte
//               swizzle), one mbarrier pair per stage; one lane walks the
//               schedule.
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators);
//               one lane waits and issues the MMAs (the even CTA of a pair).
//   warps 2, 3  idle (they complete warpgroup 0, which hands its registers
//               to the epilogue through setmaxnreg).
//   warps 4..11 epilogue: TMEM -> registers -> residues mod p in fp32 (or
//               exact int32 sums) -> HBM, residue planes by TMA stores.
// Every mbarrier wait is bounded (2 s); a wait that runs out latches
// OZK_ERR_TIMEOUT on the device, makes all roles of the CTA stop, drains
// in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>

#include "ozk_internal.h"

namespace ozk {

__device__ int g_status;  // latched device-side faults, read by ozk_stream_status

namespace {

constexpr int BM = kTileM, BN = kTileN;
constexpr int BK = 64;       // K elements (fp16) per pipeline stage: one swizzle row
constexpr int kStages = 4;   // smem ring depth
static_assert(kKBlock % BK == 0, "slices are padded to whole stages");
constexpr int kSwizzleBytes = BK * 2;                  // 128-byte or 64-byte swizzle
constexpr uint64_t kLayoutType = kSwizzleBytes == 128 ? 2 : 4;  // descriptor swizzle code
// k-blocks per exact chunk: 1024 terms, every partial sum |x| <= 2^24
constexpr int kChunkKB = 1024 / BK;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 128 + 32 * kEpiWarps;  // warpgroup 0: control, 1-2: epilogue
// Register split between the warpgroups (setmaxnreg).  The kernel launches
// with kLaunchRegs per thread; warpgroup 0 gives registers back, the two
// epilogue warpgroups take them: 128 * 56 + 256 * 224 = 384 * 168.
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 56;
constexpr int kEpiRegs = 224;
static_assert(128 * kCtrlRegs + 256 * kEpiRegs <= kThreads * kLaunchRegs, "register split exceeds the pool");
constexpr uint32_t kABytes = BM * BK * 2;
constexpr uint32_t kBBytes = BN * BK * 2;
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr int kCols = BN / 2;  // accumulator columns per epilogue thread (two warps per TMEM lane quadrant)
static_assert(kCols % 32 == 0, "the drain moves 32 columns per tcgen05.ld");
// two BN-column fp32 accumulators, allocated as a power of two >= 32 columns
constexpr uint32_t kTmemCols = (2 * BN <= 256) ? 256u : 512u;
static_assert(2 * BN <= static_cast<int>(kTmemCols), "two accumulators fit the allocation");
// mbarriers after the ring: full and empty per stage, two accumulator-full,
// two accumulator-empty, one drain; then the TMEM address and the abort flag
constexpr int kNumBars = 2 * kStages + 5;
constexpr size_t kBarBytes = 1024;  // keeps the stash after it 1024-byte aligned (128-byte swizzle)
static_assert(8 * kNumBars + 8 <= static_cast<int>(kBarBytes), "barrier block overflows");
constexpr size_t kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes;
// CTA-pair kernel: each CTA holds 128 rows of A and half of the B tile per
// stage (32 KB), so the ring is 6 deep in the same shared memory.
constexpr int kPairMinK = 2048;  // K per split from which CTA pairs run (two long chunks)
constexpr int kPairM = 2 * BM;  // a CTA pair computes a kPairM x BN tile
constexpr int kBHalf = BN / 2;  // B rows (tile columns) each CTA of the pair loads
constexpr int kPairStages = 6;
constexpr uint32_t kPairBBytes = kBHalf * BK * 2;
constexpr uint32_t kPairStageBytes = kABytes + kPairBBytes;
constexpr int kPairNumBars = 2 * kPairStages + 5;
static_assert(8 * kPairNumBars + 8 <= static_cast<int>(kBarBytes), "barrier block overflows");
constexpr size_t kPairSmemBytes = 1024 + kPairStages * kPairStageBytes + kBarBytes;
// out_kind 2: each epilogue thread parks the residues of the first modulus of
// a pair (kCols bytes) in shared memory until the second modulus is done.
// out_kind 0 from one chunk: the same bytes stage each warp's 32 x kCols
// residue block for one TMA store (rows of kCols = 128 bytes, 128-byte
// swizzle).
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr size_t kStashBytes = static_cast<size_t>(kEpiThreads) * kCols;
static_assert(kCols == 128, "a staged residue row is one 128-byte swizzle row");
constexpr uint32_t kStageOutBytes = 32 * kCols;  // one warp's block
static_assert(kSmemBytes + kStashBytes <= 232448 && kPairSmemBytes + kStashBytes <= 232448,
              "ring, barriers and stash exceed the shared memory of a CTA");
constexpr uint64_t kTimeoutNs = 2000000000ull;  // limit of every pipeline wait in normal runs
constexpr uint64_t kDrainNs = 50000000ull;

// 1.5 * 2^23: y + 1.5 * 2^23 for |y| <= 2^22 is rounded to an integer (ulp
// 1), and for an integer y holds y in its low mantissa bits, exactly.
constexpr float kMagic = 12582912.0f;

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B fp16 (bits 7-9 and 10-12 = 0), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) |
                            (static_cast<uint32_t>(BN >> 3) << 17) |
                            (static_cast<uint32_t>(BM >> 4) << 24);
constexpr uint32_t kPairIdesc = (1u << 4) |  // M of the whole pair
                                (static_cast<uint32_t>(BN >> 3) << 17) |
                                (static_cast<uint32_t>(kPairM >> 4) << 24);

// Per modulus: p, 1/p rounded up to fp32, and the constants of mod_p.  Per
// pair of moduli (2j, 2j+1)
// with m = p_2j p_2j+1: u0 = 1 mod p_2j and 0 mod p_2j+1, u1 the other way
// round, so (c_2j u0 + c_2j+1 u1) mod m is the residue of the pair modulus;
// t < 2^25 is divided exactly as umulhi(t, ceil(2^42 / m)) >> 10.
struct ModTable {
  uint32_t p[kMaxModuli], magic[kMaxModuli], bias[kMaxModuli];
  float inv_up[kMaxModuli];
  uint32_t pu0[kMaxModuli / 2], pu1[kMaxModuli / 2], pm[kMaxModuli / 2], pmagic[kMaxModuli / 2];
};

// 1/p rounded up to fp32 (p <= 256): the nearest value, raised by one ulp
// when it lies below 1/p.
__host__ __device__ constexpr float inverse_up(uint32_t p) {
  const float inv = 1.0f / static_cast<float>(p);
  if (static_cast<double>(inv) * p >= 1.0) return inv;
  float ulp = 1.0f;
  while (ulp > inv) ulp *= 0.5f;  // the power of two at or below inv
  return inv + ulp * (1.0f / 8388608.0f);
}

__host__ __device__ constexpr uint32_t inverse_mod(uint32_t a, uint32_t p) {
  for (uint32_t x = 1; x < p; ++x)
    if ((a % p) * x % p == 1u) return x;
  return 0;
}

__host__ __device__ constexpr ModTable make_mod_table() {
  ModTable t{};
  for (int k = 0; k < kMaxModuli; ++k) {
    t.p[k] = modulus_at(k);
    t.magic[k] = magic_of(t.p[k]);
    t.bias[k] = bias_of(t.p[k]);
    t.inv_up[k] = inverse_up(t.p[k]);
  }
  for (int j = 0; j < kMaxModuli / 2; ++j) {
    const uint32_t pa = modulus_at(2 * j), pb = modulus_at(2 * j + 1);
    t.pu0[j] = pb * inverse_mod(pb, pa);
    t.pu1[j] = pa * inverse_mod(pa, pb);
    t.pm[j] = pa * pb;
    t.pmagic[j] = static_cast<uint32_t>(((uint64_t{1} << 42) + pa * pb - 1) / (pa * pb));
  }
  return t;
}

__constant__ ModTable c_mod = make_mod_table();

struct GemmParams {
  int M, N, n, kblocks, tiles_m, tiles_n, splits, kb_per_split, out_kind;
  // the limit of every mbarrier wait, and (single-CTA kernel only; -1 in
  // normal runs) a k-block of CTA 0's first unit whose copy the producer
  // withholds, so that the MMA issuer's wait for it runs out: the test of the
  // timeout path
  uint64_t timeout_ns;
  int withhold_kb;
  int mod_units;           // n, or ceil(n/2) pairs of moduli for out_kind 2
  int64_t ldo, out_plane;  // row stride and per-(split, modulus) plane stride, in elements
  void* out;
  // the unit decode's divisors: tiles per modulus and split, tiles per group
  // of tile rows, tile rows of the last (shorter) group, splits
  FastDiv div_tiles, div_group, div_tail, div_splits;
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of the given parity to complete.  Returns false when
// another role has aborted, or after timeout_ns (then latches the fault and
// tells the other roles to stop).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > timeout_ns) {
        *abort_flag = 1;
        atomicOr(&g_status, 1);
        return false;
      }
    }
  }
}

// Every lane of the warp waits; the outcome is made warp-uniform so that the
// .sync.aligned tcgen05 instructions after it see a converged warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns) {
  const bool got = mbar_wait(bar, parity, abort_flag, timeout_ns);
  return __all_sync(0xffffffffu, got);
}

// Bounded wait used only while shutting down after an abort.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_test(bar, parity))
    if (globaltimer() - t0 > kDrainNs) return;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// TMA store of a box from shared memory (bulk-group completion), and the
// waits on this thread's bulk groups: until their shared-memory source has
// been read, or until their writes are done.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Makes this thread's generic-proxy writes to shared memory visible to the
// async proxy (a following TMA store).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

// Shared-memory matrix descriptor, K-major operand with a swizzle as wide as
// one BK row: start address >> 4 (bits 0-13), leading byte offset 16 B
// (unused for this layout), stride byte offset between 8-row groups
// (bits 32-45), descriptor version 1 (bit 46), swizzle mode (bits 61-63:
// 2 = 128B, 4 = 64B).
__device__ __forceinline__ uint64_t smem_desc_swizzled(uint32_t addr) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (1ull << 16) |
         (static_cast<uint64_t>((8 * kSwizzleBytes) >> 4) << 32) | (1ull << 46) | (kLayoutType << 61);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier when every tcgen05.mma issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
template <int R>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}

// Waits for this thread's tcgen05.ld to land.  The loaded registers are
// operands, so no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
                 "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
                 "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]),
                 "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]),
                 "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}


// ---- CTA-pair (cta_group::2) forms ----
// Arrival on an mbarrier of any CTA of the cluster (shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The shared::cluster address of `local` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs of the pair.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Tile into this CTA's shared memory; completion is signalled on `bar`, an
// mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// TMEM of the CTA pair: one warp of each CTA executes these together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

// One pair MMA (M=256 across the two CTAs), issued by the even CTA.
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier at offset `bar` of both CTAs of the pair when
// every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// As above, on this CTA's mbarrier only.
__device__ __forceinline__ void mma_commit_local(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}


// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// One work unit: a tile (mt, nt) of split sk for one modulus p, or for
// out_kind 2 the two moduli p, p+1 of pair q one after the other (passes).
struct Unit {
  int p, q, passes, sk, mt, nt, kb0, kb1;
};

// Within one modulus (and split) the tiles run in groups of kGroupM tile
// rows, column by column: the units of one persistent wave then share a few
// tile rows of A and a band of B columns, which stay in L2, instead of
// sweeping every column tile of B (the whole slice, 134 MB per modulus at
// N = K = 8192) once per couple of tile rows.
constexpr int kGroupM = 8;
static_assert((kGroupM & (kGroupM - 1)) == 0, "a whole group's tile row and column by mask and shift");

// Every role of every CTA decodes each of its units.  In the single-CTA
// kernel, whose units are short (a 128 x 256 tile over at most 1024 of K),
// the divisions are multiplies by the reciprocals the host computed for the
// launch (a run-time divide is a long dependent chain): 8192^2 x 512 at 14
// moduli 618 -> 601 us.  The CTA-pair kernel's units are long, and there the
// reciprocals held in its control warps' 56 registers spilled more and cost
// 0.3% at 4096^3, so it divides.
template <bool PAIRS, bool FAST>
__device__ __forceinline__ Unit decode_unit(int u, const GemmParams& prm) {
  Unit r;
  if constexpr (!FAST) {
    const int tiles = prm.tiles_m * prm.tiles_n;
    const int idx = u % tiles;
    u /= tiles;
    const int first = idx / (kGroupM * prm.tiles_n) * kGroupM;  // first tile row of the group
    const int gm = min(prm.tiles_m - first, kGroupM);            // tile rows in the group
    const int in = idx - first * prm.tiles_n;
    r.mt = first + in % gm;
    r.nt = in / gm;
    r.sk = u % prm.splits;
    r.q = u / prm.splits;
  } else {
    const uint32_t tiles = static_cast<uint32_t>(prm.tiles_m * prm.tiles_n);
    const uint32_t uq = div_fast(static_cast<uint32_t>(u), prm.div_tiles);
    const uint32_t idx = static_cast<uint32_t>(u) - uq * tiles;
    const int first = static_cast<int>(div_fast(idx, prm.div_group)) * kGroupM;  // first tile row of the group
    const uint32_t in = idx - static_cast<uint32_t>(first * prm.tiles_n);
    if (prm.tiles_m - first >= kGroupM) {  // kGroupM tile rows in the group
      r.mt = first + static_cast<int>(in & (kGroupM - 1));
      r.nt = static_cast<int>(in / kGroupM);
    } else {  // the last group, tiles_m mod kGroupM rows
      const uint32_t nt = div_fast(in, prm.div_tail);
      r.mt = first + static_cast<int>(in - nt * static_cast<uint32_t>(prm.tiles_m - first));
      r.nt = static_cast<int>(nt);
    }
    const uint32_t q = div_fast(uq, prm.div_splits);
    r.sk = static_cast<int>(uq - q * static_cast<uint32_t>(prm.splits));
    r.q = static_cast<int>(q);
  }
  if (PAIRS) {  // out_kind 2
    r.p = 2 * r.q;
    r.passes = min(2, prm.n - r.p);
  } else {
    r.p = r.q;
    r.passes = 1;
  }
  r.kb0 = r.sk * prm.kb_per_split;
  r.kb1 = min(prm.kblocks, r.kb0 + prm.kb_per_split);
  if (r.kb1 < r.kb0) r.kb1 = r.kb0;
  return r;
}

// acc[base .. base+31] += the 32 exact chunk sums held as fp32 in v.
__device__ __forceinline__ void add_chunk(int32_t (&acc)[kCols], int base, const uint32_t (&v)[32]) {
#pragma unroll
  for (int e = 0; e < 32; ++e) acc[base + e] += __float2int_rn(__uint_as_float(v[e]));
}

// Adds this thread's kCols chunk sums from TMEM into acc, one block of 32
// columns per tcgen05.ld, loaded after the previous block is added up (the
// registers go to the conversions).
template <int Q>
__device__ __forceinline__ void drain_chunk(int32_t (&acc)[kCols], uint32_t taddr, uint32_t (&cur)[32]) {
  add_chunk(acc, 32 * Q, cur);
  if constexpr (Q + 1 < kCols / 32) {
    tmem_ld32(taddr + 32 * (Q + 1), cur);
    tmem_wait_ld(cur);
    drain_chunk<Q + 1>(acc, taddr, cur);
  }
}

// Packed fp32 pairs (f32x2: one instruction for two lanes of data).
__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ uint64_t pack2f(float v) {
  return pack2(__float_as_uint(v), __float_as_uint(v));
}
__device__ __forceinline__ uint64_t fma2_rn(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fma2_rm(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2_rn(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Per-modulus constants of the residue steps, each in both halves of a
// pair: 1/p rounded up, 1.5 * 2^23 and its negation, -p.
struct ResidueConsts {
  uint64_t inv, magic, neg_magic, neg_p;
};
__device__ __forceinline__ ResidueConsts residue_consts(int p) {
  return {pack2f(c_mod.inv_up[p]), pack2f(kMagic), pack2f(-kMagic), pack2f(-static_cast<float>(c_mod.p[p]))};
}

// Cuts two fp32 chunk sums (integers, |x| <= 2^24) to r = x - q p with
// q = rint(x * (1/p)), from one fma with the 1.5 * 2^23 add (ulp 1 there):
// x * (1/p) lies within |x| p^-1 2^-23 < 0.012 of x / p, so q is x / p
// rounded up or down, |r| < 0.512 p, and the fma forms r exactly.  q_shift
// is -(1.5 * 2^23 + s): r comes out s p higher.
__device__ __forceinline__ uint64_t cut2(uint64_t x, const ResidueConsts& c, uint64_t q_shift) {
  return fma2_rn(add2_rn(fma2_rn(x, c.inv, c.magic), q_shift), c.neg_p, x);
}

// The residues mod p of two integers 0 <= R < 2^22, each as the low byte of
// its half of the result: k = floor(R * (1/p)) by an fma with the
// 1.5 * 2^23 add rounding toward minus infinity.  With 1/p rounded up,
// R * (1/p) is at least R / p and exceeds it by less than R 2^-23 / p, which
// stays below the distance 1/p from R / p to the next integer while
// R < 2^23; so k = floor(R / p), R - k p (exact, by an fma) is the residue,
// and adding 1.5 * 2^23 puts it in the low mantissa bits.  For -p < R < 0
// the same steps give k = -1 and again the residue.
__device__ __forceinline__ uint64_t floor_residues2(uint64_t R, const ResidueConsts& c) {
  const uint64_t k = add2_rn(fma2_rm(R, c.inv, c.magic), c.neg_magic);
  return add2_rn(fma2_rn(k, c.neg_p, R), c.magic);
}

// Low bytes of the four fp32 words in a and b, in order.
__device__ __forceinline__ uint32_t low_bytes4(uint64_t a, uint64_t b) {
  const uint32_t lo = __byte_perm(static_cast<uint32_t>(a), static_cast<uint32_t>(a >> 32), 0x0040);
  const uint32_t hi = __byte_perm(static_cast<uint32_t>(b), static_cast<uint32_t>(b >> 32), 0x0040);
  return __byte_perm(lo, hi, 0x5410);
}

// Residue words (bytes of columns 4i .. 4i+3 in words[i]) of one chunk:
// r from cut2 lies in (-p, p), where floor_residues2 applies.
__device__ __forceinline__ void one_chunk_words(const uint32_t (&x)[kCols / 32][32], uint32_t (&words)[kCols / 4],
                                                const ResidueConsts& c) {
#pragma unroll
  for (int i = 0; i < kCols / 4; ++i) {
    const uint32_t* xs = &x[(4 * i) / 32][(4 * i) % 32];
    words[i] = low_bytes4(floor_residues2(cut2(pack2(xs[0], xs[1]), c, c.neg_magic), c),
                          floor_residues2(cut2(pack2(xs[2], xs[3]), c, c.neg_magic), c));
  }
}

// Several chunks: each chunk's sums are cut (cut2) and the cut values added
// up in fp32 pairs R.  The first chunk's quotient is lowered by the number of
// chunks nc, which adds nc p to R, so R ends in (0.48 nc p, 1.52 nc p): a
// positive integer below 2^22 (nc <= 128, K < 2^17), exact in fp32, and
// floor_residues2 reduces it.  This adds the 32 columns of block Q (loaded
// in cur) and loads and adds the blocks after it.
template <bool FIRST, int Q>
__device__ __forceinline__ void cut_chunk(uint64_t (&R)[kCols / 2], uint32_t taddr, uint32_t (&cur)[32],
                                          const ResidueConsts& c, uint64_t first_shift) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint64_t r = cut2(pack2(cur[2 * e], cur[2 * e + 1]), c, FIRST ? first_shift : c.neg_magic);
    R[16 * Q + e] = FIRST ? r : add2_rn(R[16 * Q + e], r);
  }
  if constexpr (Q + 1 < kCols / 32) {
    tmem_ld32(taddr + 32 * (Q + 1), cur);
    tmem_wait_ld(cur);
    cut_chunk<FIRST, Q + 1>(R, taddr, cur, c, first_shift);
  }
}

__device__ __forceinline__ void chunk_words(const uint64_t (&R)[kCols / 2], uint32_t (&words)[kCols / 4],
                                            const ResidueConsts& c) {
#pragma unroll
  for (int i = 0; i < kCols / 4; ++i)
    words[i] = low_bytes4(floor_residues2(R[2 * i], c), floor_residues2(R[2 * i + 1], c));
}

// out_kind 1: the exact int32 sums of this thread's kCols columns gj0.. of
// row gi, in plane (sk, p).
__device__ __forceinline__ void store_sums(const int32_t (&acc)[kCols], const Unit& w, int ps, int64_t gi,
                                           int64_t gj0, const GemmParams& prm) {
  if (gi >= prm.M) return;
  int32_t* dst = static_cast<int32_t*>(prm.out) +
                 (static_cast<int64_t>(w.sk) * prm.n + w.p + ps) * prm.out_plane + gi * prm.ldo + gj0;
#pragma unroll
  for (int v = 0; v < kCols / 4; ++v)
    if (gj0 + 4 * v < prm.ldo)
      *reinterpret_cast<int4*>(dst + 4 * v) = make_int4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
}

// x mod p in [0, p) for an exact int32 dot product (|x| < 2^31 - 2^14).
__device__ __forceinline__ uint32_t mod_p(int32_t x, uint32_t p, uint32_t magic, uint32_t bias) {
  const uint32_t u = static_cast<uint32_t>(x) + bias;
  const uint32_t q = __umulhi(u, magic);
  int32_t r = static_cast<int32_t>(u - q * p);
  r += r < 0 ? static_cast<int32_t>(p) : 0;
  return static_cast<uint32_t>(r);
}

// Combines the residues of the moduli of pair q into the pair residue:
// (c_2j u0 + c_2j+1 u1) mod p_2j p_2j+1 (< 2^25 before the reduction).
__device__ __forceinline__ uint32_t pair_residue(uint32_t c0, uint32_t c1, uint32_t u0, uint32_t u1, uint32_t m,
                                                 uint32_t pmg) {
  const uint32_t t = c0 * u0 + c1 * u1;
  return t - (__umulhi(t, pmg) >> 10) * m;
}

// out_kind 2 from exact int32 sums (several chunks: the int32 drain is the
// cheaper one per chunk once a split holds about six or more): pass 0 of a
// pair parks the residues mod p in the thread's stash slots
// (stash[v * kEpiThreads]); pass 1 combines them with its own into the pair
// residue, written as uint16 in plane q (an odd last modulus writes its own
// residue there).
__device__ __forceinline__ void store_pair_sums(const int32_t (&acc)[kCols], const Unit& w, int ps, int64_t gi,
                                                int64_t gj0, const GemmParams& prm, uint4* stash) {
  const int p = w.p + ps;
  const uint32_t pp = c_mod.p[p], mg = c_mod.magic[p], bs = c_mod.bias[p];
  if (ps == 0 && w.passes == 2) {
#pragma unroll
    for (int v = 0; v < kCols / 16; ++v) {
      uint32_t word[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int e = 16 * v + 4 * b;
        word[b] = mod_p(acc[e], pp, mg, bs) | (mod_p(acc[e + 1], pp, mg, bs) << 8) |
                  (mod_p(acc[e + 2], pp, mg, bs) << 16) | (mod_p(acc[e + 3], pp, mg, bs) << 24);
      }
      stash[v * kEpiThreads] = make_uint4(word[0], word[1], word[2], word[3]);
    }
    return;
  }
  if (gi >= prm.M) return;
  uint16_t* dst = static_cast<uint16_t*>(prm.out) + static_cast<int64_t>(w.q) * prm.out_plane + gi * prm.ldo + gj0;
  const bool pair = w.passes == 2;
  const uint32_t u0 = c_mod.pu0[w.q], u1 = c_mod.pu1[w.q], m = c_mod.pm[w.q], pmg = c_mod.pmagic[w.q];
#pragma unroll
  for (int v = 0; v < kCols / 16; ++v) {
    const uint4 first = pair ? stash[v * kEpiThreads] : make_uint4(0, 0, 0, 0);
    const uint32_t fw[4] = {first.x, first.y, first.z, first.w};
    uint32_t r[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t c = mod_p(acc[16 * v + e], pp, mg, bs);
      r[e] = pair ? pair_residue((fw[e >> 2] >> (8 * (e & 3))) & 0xFFu, c, u0, u1, m, pmg) : c;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (gj0 + 16 * v + 8 * h < prm.ldo)
        *reinterpret_cast<uint4*>(dst + 16 * v + 8 * h) =
            make_uint4(r[8 * h] | (r[8 * h + 1] << 16), r[8 * h + 2] | (r[8 * h + 3] << 16),
                       r[8 * h + 4] | (r[8 * h + 5] << 16), r[8 * h + 6] | (r[8 * h + 7] << 16));
  }
}

// Writes the residue words of pass ps of unit w, for this thread's kCols
// columns gj0.. of row row0 + lane (row0: the warp's first row).
//  out_kind 0 (!PAIRS): a TMA store.  The warp's 32 x kCols bytes go into its
//    staging block (16-byte chunk v of row r at chunk v ^ (r & 7), the
//    128-byte swizzle; rewritten only after the previous store has read it),
//    then lane 0 stores the block as one 128 x 32 box at (gj0, row0, p); the
//    map clips rows >= M and columns >= ldo, and a box wholly outside is
//    not stored.
//  out_kind 2 (PAIRS): pass 0 of a pair parks the residues in the thread's
//    stash slots (stash[v * kEpiThreads]); pass 1 combines them with its own
//    into the pair residue, written as uint16 in plane q (an odd last modulus
//    writes its own residue there).
template <bool PAIRS>
__device__ __forceinline__ void store_words(const uint32_t (&words)[kCols / 4], const Unit& w, int ps, int64_t row0,
                                            int lane, int64_t gj0, const GemmParams& prm, uint4* stash,
                                            uint32_t stage, const CUtensorMap* tmO) {
  if constexpr (!PAIRS) {
    if (gj0 >= prm.ldo || row0 >= prm.M) return;  // the same for the whole warp
    if (lane == 0) bulk_wait_read();
    __syncwarp();
    const uint32_t row = stage + static_cast<uint32_t>(lane) * kCols;
#pragma unroll
    for (int v = 0; v < kCols / 16; ++v)
      st_shared_v4(row + static_cast<uint32_t>((v ^ (lane & 7)) * 16), words[4 * v], words[4 * v + 1],
                   words[4 * v + 2], words[4 * v + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tma_store_3d(tmO, stage, static_cast<int>(gj0), static_cast<int>(row0), w.p + ps);
  } else {
    if (ps == 0 && w.passes == 2) {
#pragma unroll
      for (int v = 0; v < kCols / 16; ++v)
        stash[v * kEpiThreads] = make_uint4(words[4 * v], words[4 * v + 1], words[4 * v + 2], words[4 * v + 3]);
      return;
    }
    const int64_t gi = row0 + lane;
    if (gi >= prm.M) return;
    uint16_t* dst = static_cast<uint16_t*>(prm.out) + static_cast<int64_t>(w.q) * prm.out_plane + gi * prm.ldo + gj0;
    const bool pair = w.passes == 2;
    const uint32_t u0 = c_mod.pu0[w.q], u1 = c_mod.pu1[w.q], m = c_mod.pm[w.q], pmg = c_mod.pmagic[w.q];
#pragma unroll
    for (int v = 0; v < kCols / 16; ++v) {
      const uint4 first = pair ? stash[v * kEpiThreads] : make_uint4(0, 0, 0, 0);
      const uint32_t fw[4] = {first.x, first.y, first.z, first.w};
      uint32_t r[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint32_t c = (words[4 * v + (e >> 2)] >> (8 * (e & 3))) & 0xFFu;
        r[e] = pair ? pair_residue((fw[e >> 2] >> (8 * (e & 3))) & 0xFFu, c, u0, u1, m, pmg) : c;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if (gj0 + 16 * v + 8 * h < prm.ldo)
          *reinterpret_cast<uint4*>(dst + 16 * v + 8 * h) =
              make_uint4(r[8 * h] | (r[8 * h + 1] << 16), r[8 * h + 2] | (r[8 * h + 3] << 16),
                         r[8 * h + 4] | (r[8 * h + 5] << 16), r[8 * h + 6] | (r[8 * h + 7] << 16));
    }
  }
}

// One pass of one unit in an epilogue warp: takes the pass's nchunks
// accumulators from TMEM (tbase: this warp's lanes and columns of buffer 0),
// waiting on the accumulator-full barrier and handing each buffer back
// through release(ab), and writes the pass's output.  Returns false if a wait
// ran out.
//  out_kind 1, and 2 over several chunks: exact int32 sums (cvt.rni and
//    int32 adds per chunk).
//  out_kind 0, and 2 from one chunk: residues in fp32 throughout (one chunk:
//    one_chunk_words; several: cut_chunk and chunk_words).
template <bool LONG, int KIND, typename Release>
__device__ __forceinline__ bool epilogue_pass(const Unit& w, int ps, int nchunks, int64_t row0, int lane,
                                              int64_t gj0, const GemmParams& prm, uint4* stash, uint32_t out_stage,
                                              const CUtensorMap* tmO, uint32_t tbase, uint32_t accf0,
                                              volatile int* abort_flag, int& ab, uint32_t& aphase,
                                              Release release) {
  auto acquire = [&]() -> bool {
    if (!warp_wait(accf0 + 8 * ab, aphase, abort_flag, prm.timeout_ns)) return false;
    tc_fence_after();
    return true;
  };
  auto handback = [&]() {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) release(ab);
    ab ^= 1;
    if (ab == 0) aphase ^= 1u;
  };
  // one chunk: all kCols sums at once, the buffer handed back before the
  // arithmetic (zeros for an empty split)
  auto load_all = [&](uint32_t (&x)[kCols / 32][32]) -> bool {
    if (nchunks == 0) {
#pragma unroll
      for (int q = 0; q < kCols / 32; ++q)
#pragma unroll
        for (int e = 0; e < 32; ++e) x[q][e] = 0u;
      return true;
    }
    if (!acquire()) return false;
    const uint32_t taddr = tbase + static_cast<uint32_t>(ab * BN);
#pragma unroll
    for (int q = 0; q < kCols / 32; ++q) tmem_ld32(taddr + 32 * q, x[q]);
#pragma unroll
    for (int q = 0; q < kCols / 32; ++q) tmem_wait_ld(x[q]);
    handback();
    return true;
  };
  if constexpr (KIND == 1 || (KIND == 2 && LONG)) {
    int32_t acc[kCols];
    if constexpr (LONG) {
#pragma unroll
      for (int e = 0; e < kCols; ++e) acc[e] = 0;
      for (int c = 0; c < nchunks; ++c) {
        if (!acquire()) return false;
        const uint32_t taddr = tbase + static_cast<uint32_t>(ab * BN);
        uint32_t va[32];
        tmem_ld32(taddr, va);
        tmem_wait_ld(va);
        drain_chunk<0>(acc, taddr, va);
        handback();
      }
    } else {
      uint32_t x[kCols / 32][32];
      if (!load_all(x)) return false;
#pragma unroll
      for (int e = 0; e < kCols; ++e) acc[e] = __float2int_rn(__uint_as_float(x[e / 32][e % 32]));
    }
    if constexpr (KIND == 1)
      store_sums(acc, w, ps, row0 + lane, gj0, prm);
    else
      store_pair_sums(acc, w, ps, row0 + lane, gj0, prm, stash);
    return true;
  } else {
    const ResidueConsts rc = residue_consts(w.p + ps);
    uint32_t words[kCols / 4];
    if constexpr (LONG) {
      uint64_t R[kCols / 2];
      const uint64_t first_shift = pack2f(-(kMagic + static_cast<float>(nchunks)));
      for (int c = 0; c < nchunks; ++c) {
        if (!acquire()) return false;
        const uint32_t taddr = tbase + static_cast<uint32_t>(ab * BN);
        uint32_t va[32];
        tmem_ld32(taddr, va);
        tmem_wait_ld(va);
        if (c == 0)
          cut_chunk<true, 0>(R, taddr, va, rc, first_shift);
        else
          cut_chunk<false, 0>(R, taddr, va, rc, first_shift);
        handback();
      }
      chunk_words(R, words, rc);
    } else {
      uint32_t x[kCols / 32][32];
      if (!load_all(x)) return false;
      one_chunk_words(x, words, rc);
    }
    store_words<KIND == 2>(words, w, ps, row0, lane, gj0, prm, stash, out_stage, tmO);
    return true;
  }
}

template <bool LONG, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    residue_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO, const GemmParams prm) {
  grid_dependency_sync();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);  // swizzle-atom aligned tiles
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * kStages;
  const uint32_t accf0 = empty0 + 8 * kStages;
  const uint32_t acce0 = accf0 + 16;
  const uint32_t drain = acce0 + 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const int units = prm.mod_units * prm.splits * prm.tiles_m * prm.tiles_n;

  if (warp < 4) regs_dec<kCtrlRegs>();
  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    // One thread walks the schedule, waits and issues the copies.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued_parity[kStages];
      for (int s = 0; s < kStages; ++s) issued_parity[s] = -1;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = decode_unit<KIND == 2, true>(u, prm);
        for (int ps = 0; ps < w.passes && ok; ++ps) {
          for (int kb = w.kb0; kb < w.kb1; ++kb) {
            if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, prm.timeout_ns)) {
              ok = false;
              break;
            }
            if (prm.withhold_kb >= 0 && blockIdx.x == 0 && u == 0 && ps == 0 && kb == w.kb0 + prm.withhold_kb) {
              // the timeout test: this stage's copy is never issued (its full
              // barrier never completes), the ring moves on
              if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
              }
              continue;
            }
            mbar_expect_tx(full0 + 8 * stage, kStageBytes);
            tma_load_3d(smem_u32(sA + stage * kABytes), &tmA, kb * BK, w.mt * BM, w.p + ps, full0 + 8 * stage);
            tma_load_3d(smem_u32(sB + stage * kBBytes), &tmB, kb * BK, w.nt * BN, w.p + ps, full0 + 8 * stage);
            issued_parity[stage] = static_cast<int>(phase);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {  // let copies still in flight land before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (issued_parity[s] >= 0) mbar_wait_drain(full0 + 8 * s, static_cast<uint32_t>(issued_parity[s]));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    // One thread walks the schedule, waits and issues the MMAs.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int ab = 0;
      uint32_t aphase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = decode_unit<KIND == 2, true>(u, prm);
        for (int ps = 0; ps < w.passes && ok; ++ps)
        for (int c0 = w.kb0; c0 < w.kb1 && ok; c0 += kChunkKB) {
          const int c1 = min(w.kb1, c0 + kChunkKB);
          if (!mbar_wait(acce0 + 8 * ab, aphase ^ 1u, abort_flag, prm.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(ab * BN);
          for (int kb = c0; kb < c1; ++kb) {
            if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, prm.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t da = smem_desc_swizzled(smem_u32(sA + stage * kABytes));
            const uint64_t db = smem_desc_swizzled(smem_u32(sB + stage * kBBytes));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)  // K = 16 fp16 = 32 bytes per MMA
              mma_f16(d, da + 2ull * kk, db + 2ull * kk, kIdesc, (kb > c0 || kk > 0) ? 1u : 0u);
            mma_commit(empty0 + 8 * stage);  // frees the stage once these MMAs are done
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(accf0 + 8 * ab);  // chunk sum ready in TMEM buffer ab
          ab ^= 1;
          if (ab == 0) aphase ^= 1u;
        }
      }
      mma_commit(drain);  // every issued MMA has finished before TMEM is freed
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------ epilogue ------------------------------
    regs_inc<kEpiRegs>();
    const int ew = warp - 4;
    const int quad = warp & 3;  // TMEM lanes this warp may access: 32*quad .. 32*quad+31
    const int half = ew >> 2;   // which kCols of the BN tile columns
    int ab = 0;
    uint32_t aphase = 0;
    bool ok = true;
    uint4* stash = reinterpret_cast<uint4*>(smem + kStages * kStageBytes + kBarBytes) + (threadIdx.x - 128);
    const uint32_t out_stage =
        smem_u32(smem + kStages * kStageBytes + kBarBytes) + static_cast<uint32_t>(ew) * kStageOutBytes;
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(half * kCols);
    auto release = [&](int b) { mbar_arrive(acce0 + 8 * b); };
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const Unit w = decode_unit<KIND == 2, true>(u, prm);
      const int nchunks = (w.kb1 - w.kb0 + kChunkKB - 1) / kChunkKB;
      const int64_t row0 = static_cast<int64_t>(w.mt) * BM + quad * 32;
      const int64_t gj0 = static_cast<int64_t>(w.nt) * BN + half * kCols;
      for (int ps = 0; ps < w.passes && ok; ++ps)
        ok = epilogue_pass<LONG, KIND>(w, ps, nchunks, row0, lane, gj0, prm, stash, out_stage, &tmO, tbase, accf0,
                                        abort_flag, ab, aphase, release);
    }
    // the residue stores in flight finish before the CTA's shared memory goes
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

constexpr int kPairChunkKB = kChunkKB;

// The CTA-pair kernel: tcgen05.mma.cta_group::2 (M=256, N=256) issued by the
// even CTA of a cluster of two; long (1024-term) chunks only.
template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    residue_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmO, const GemmParams prm) {
  grid_dependency_sync();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);  // swizzle-atom aligned tiles
  uint8_t* sA = smem;
  uint8_t* sB = smem + kPairStages * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPairStages * kPairStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kPairNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: leader of the pair (issues the MMAs), 1: peer
  const bool leader = rank == 0;
  const uint32_t full0 = smem_u32(bars);           // leader: both CTAs' tiles of a stage landed
  const uint32_t empty0 = full0 + 8 * kPairStages;     // both: the MMAs released a stage
  const uint32_t accf0 = empty0 + 8 * kPairStages;     // both: a chunk sum is in TMEM
  const uint32_t acce0 = accf0 + 16;               // leader: both epilogues drained a buffer
  const uint32_t drain = acce0 + 16;               // leader: all MMAs finished

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 2 * kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {  // one warp of each CTA allocates the pair's TMEM together
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const int units = prm.mod_units * prm.splits * prm.tiles_m * prm.tiles_n;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int npairs = static_cast<int>(gridDim.x >> 1);

  if (warp < 4) regs_dec<kCtrlRegs>();
  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    // Each CTA loads its 128 rows of A and its half of B into its own ring;
    // both signal the leader's full barrier, which the leader arms with the
    // bytes of the two CTAs.  One thread walks the schedule.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued_parity[kPairStages];
      for (int s = 0; s < kPairStages; ++s) issued_parity[s] = -1;
      bool ok = true;
      for (int u = pair; u < units && ok; u += npairs) {
        const Unit w = decode_unit<KIND == 2, false>(u, prm);
        for (int ps = 0; ps < w.passes && ok; ++ps)
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, prm.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t full_leader = cluster_addr(full0 + 8 * stage, 0);
          if (leader) mbar_expect_tx(full0 + 8 * stage, 2 * kPairStageBytes);
          tma_load_3d_pair(smem_u32(sA + stage * kABytes), &tmA, kb * BK,
                      w.mt * kPairM + static_cast<int>(rank) * BM, w.p + ps, full_leader);
          tma_load_3d_pair(smem_u32(sB + stage * kPairBBytes), &tmB, kb * BK,
                      w.nt * BN + static_cast<int>(rank) * kBHalf, w.p + ps, full_leader);
          issued_parity[stage] = static_cast<int>(phase);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {  // let copies still in flight land before the pair exits
        for (int s = 0; s < kPairStages; ++s)
          if (issued_parity[s] >= 0) mbar_wait_drain(full0 + 8 * s, static_cast<uint32_t>(issued_parity[s]));
      }
    }
    __syncwarp();
  } else if (warp == 1 && leader) {
    // ------------------------------ MMA issuer (leader) ------------------------------
    // One thread issues M=256 MMAs that read A and B from both CTAs' rings and
    // accumulate into both TMEMs.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int ab = 0;
      uint32_t aphase = 0;
      bool ok = true;
      for (int u = pair; u < units && ok; u += npairs) {
        const Unit w = decode_unit<KIND == 2, false>(u, prm);
        for (int ps = 0; ps < w.passes && ok; ++ps)
        for (int c0 = w.kb0; c0 < w.kb1 && ok; c0 += kPairChunkKB) {
          const int c1 = min(w.kb1, c0 + kPairChunkKB);
          if (!mbar_wait(acce0 + 8 * ab, aphase ^ 1u, abort_flag, prm.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + static_cast<uint32_t>(ab * BN);
          for (int kb = c0; kb < c1; ++kb) {
            if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, prm.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t da = smem_desc_swizzled(smem_u32(sA + stage * kABytes));
            const uint64_t db = smem_desc_swizzled(smem_u32(sB + stage * kPairBBytes));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_f16_pair(d, da + 2ull * kk, db + 2ull * kk, kPairIdesc, (kb > c0 || kk > 0) ? 1u : 0u);
            mma_commit_both(empty0 + 8 * stage);  // frees the stage in both CTAs
            if (++stage == kPairStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit_both(accf0 + 8 * ab);  // chunk sum ready in both TMEMs
          ab ^= 1;
          if (ab == 0) aphase ^= 1u;
        }
      }
      mma_commit_local(drain);  // every issued MMA has finished before TMEM is freed
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------ epilogue ------------------------------
    regs_inc<kEpiRegs>();
    const int ew = warp - 4;
    const int quad = warp & 3;  // TMEM lanes this warp may access: 32*quad .. 32*quad+31
    const int half = ew >> 2;   // which kCols of the BN tile columns
    int ab = 0;
    uint32_t aphase = 0;
    bool ok = true;
    uint4* stash = reinterpret_cast<uint4*>(smem + kPairStages * kPairStageBytes + kBarBytes) + (threadIdx.x - 128);
    const uint32_t out_stage =
        smem_u32(smem + kPairStages * kPairStageBytes + kBarBytes) + static_cast<uint32_t>(ew) * kStageOutBytes;
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(half * kCols);
    auto release = [&](int b) { mbar_arrive_cluster(cluster_addr(acce0 + 8 * b, 0)); };
    for (int u = pair; u < units && ok; u += npairs) {
      const Unit w = decode_unit<KIND == 2, false>(u, prm);
      const int nchunks = (w.kb1 - w.kb0 + kPairChunkKB - 1) / kPairChunkKB;
      const int64_t row0 = static_cast<int64_t>(w.mt) * kPairM + static_cast<int64_t>(rank) * BM + quad * 32;
      const int64_t gj0 = static_cast<int64_t>(w.nt) * BN + half * kCols;
      for (int ps = 0; ps < w.passes && ok; ++ps)
        ok = epilogue_pass<true, KIND>(w, ps, nchunks, row0, lane, gj0, prm, stash, out_stage, &tmO, tbase, accf0,
                                        abort_flag, ab, aphase, release);
    }
    // the residue stores in flight finish before the CTA's shared memory goes
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the leader's MMAs are done with the peer's ring and TMEM
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// 3-D view of fp16 slices (row stride kpad, modulus stride plane elements),
// box BK (k) x box_rows x 1.
bool make_slice_map(CUtensorMap* map, const uint16_t* base, int64_t rows, int64_t kpad,
                    int64_t plane, int n, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kpad), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(n)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kpad) * 2, static_cast<cuuint64_t>(plane) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             kSwizzleBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of the uint8 residue planes (row stride ldo, plane stride
// out_plane bytes) for TMA stores of one warp's 128 x 32 block.
bool make_out_map(CUtensorMap* map, void* base, int64_t rows, int64_t ldo, int64_t out_plane, int n) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(ldo), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(n)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldo), static_cast<cuuint64_t>(out_plane)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kCols), 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Split-K choice.  A split multiplies the units (tile, modulus) by s and
// shortens each unit's K by s, so it fills SMs that one wave would leave idle;
// it costs the int32 partial sums (4 B per output, modulus and split, written
// here and read by the combine) and each unit's fixed cost.  The count is the
// one of least modelled time: waves x (k-blocks per unit + kUnitKBlocks) at
// kKBlockUs each, at least the HBM time of reading every slice once, plus the
// partial sums at HBM speed.  The constants are fitted to measurements on a
// GB300 (CTA pairs, 512^2 x 65536 at 8, 14, 17 and 20 moduli, 1024^2 x 65536,
// 2048^2 x 32768, 256^2 x 262144, every split count up to 24): the GEMM and
// combine time of the count chosen is within 0.7% of the best count's over
// those shapes (the earlier rule, which split only what filled less than one
// wave and weighed nothing but the wave fill, was 2-31% slower on four of
// them).
constexpr double kKBlockUs = 0.30;          // one 64-deep k-block of a 256 x 256 tile on one SM pair
constexpr double kUnitKBlocks = 32.0;       // a unit's fixed cost, in k-blocks
constexpr double kHbmBytesPerUs = 6.2e6;    // HBM bytes per microsecond the GEMM streams its slices at

int choose_splits(int64_t M, int64_t N, int64_t kpad, int n, int num_sms) {
  // K of at least kPairMinK runs on CTA pairs (kPairM x BN tiles, one per SM
  // pair); every split keeps at least that much K, so the choice holds
  const bool pairs = kpad >= kPairMinK;
  const int64_t min_blocks = pairs ? kPairMinK / kKBlock : 16;
  const int64_t tm = pairs ? kPairM : BM;
  const int64_t tiles = static_cast<int64_t>(n) * ((M + tm - 1) / tm) * ((N + BN - 1) / BN);
  if (pairs) num_sms /= 2;
  const int64_t kblocks = kpad / kKBlock;  // split shares are whole 64-element blocks
  // K beyond one int32-exact sum (2^14 K < 2^31) needs at least this many splits
  const int64_t min_s = (kblocks + OZK_SPLIT_MAX_K / kKBlock - 1) / (OZK_SPLIT_MAX_K / kKBlock);
  if (min_s == 1 && kblocks < 2 * min_blocks) return 1;
  const double floor_us = 2.0 * n * static_cast<double>(M + N) * static_cast<double>(kpad) / kHbmBytesPerUs;
  auto cost = [&](int64_t s) {
    const int64_t waves = (tiles * s + num_sms - 1) / num_sms;
    const double mma = static_cast<double>(waves) *
                       (static_cast<double>((kblocks + s - 1) / s) + kUnitKBlocks) * kKBlockUs;
    const double partial = s > 1 ? 8.0 * s * n * static_cast<double>(M) * static_cast<double>(N) / kHbmBytesPerUs
                                 : 0.0;
    return std::max(mma, floor_us) + partial;
  };
  int best = static_cast<int>(min_s);
  double best_cost = cost(min_s);
  for (int64_t s = min_s + 1; s <= 64 && kblocks / s >= min_blocks; ++s) {
    const double c = cost(s);
    if (c < 0.99 * best_cost) {  // a split must pay for itself by a margin
      best = static_cast<int>(s);
      best_cost = c;
    }
  }
  return best;
}

namespace {

// Cluster launch of the CTA-pair kernel: clusters of two CTAs.
void pair_launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, size_t smem, cudaStream_t stream) {
  cfg->blockDim = dim3(kThreads, 1, 1);
  cfg->gridDim = dim3(2, 1, 1);
  cfg->dynamicSmemBytes = smem;
  cfg->stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

// Once per device and kernel: the dynamic shared-memory opt-in, the check
// that the compiled launch register count covers the setmaxnreg split
// exactly (setmaxnreg.inc waits until the pool has the registers, so a
// mismatch is refused rather than launched), and for the CTA-pair kernel the
// number of co-resident clusters.  Cached so that a call issuing many
// launches (the blocked host path) does not query the driver for each.
cudaError_t kernel_setup(const void* kernel, size_t smem, bool pairs, int* resident) {
  struct Setup {
    cudaError_t err;
    int resident;
  };
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, Setup> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find({dev, kernel});
  if (it == done.end()) {
    Setup su{cudaSuccess, 0};
    cudaFuncAttributes fa;
    if ((su.err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem))) == cudaSuccess &&
        (su.err = cudaFuncGetAttributes(&fa, kernel)) == cudaSuccess) {
      if (fa.numRegs != kLaunchRegs) {
        su.err = cudaErrorInvalidKernelImage;
      } else if (pairs) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        pair_launch_config(&cfg, attr, smem, nullptr);
        su.err = cudaOccupancyMaxActiveClusters(&su.resident, kernel, &cfg);
        if (su.err == cudaSuccess && su.resident < 1) su.err = cudaErrorInvalidConfiguration;
      }
    }
    it = done.emplace(std::make_pair(dev, kernel), su).first;
  }
  *resident = it->second.resident;
  return it->second.err;
}

}  // namespace

namespace {

cudaError_t launch_gemm(int64_t M, int64_t N, int64_t kpad, const uint16_t* a_slices, int64_t a_plane,
                        const uint16_t* b_slices, int64_t b_plane, int n, int out_kind, void* out, int64_t ldo,
                        int64_t out_plane, int splits, int num_sms, uint64_t timeout_ns, int withhold_kb,
                        cudaStream_t stream) {
  if (M == 0 || N == 0) return cudaSuccess;
  GemmParams prm;
  prm.timeout_ns = timeout_ns;
  prm.withhold_kb = withhold_kb;
  prm.M = static_cast<int>(M);
  prm.N = static_cast<int>(N);
  prm.n = n;
  prm.kblocks = static_cast<int>(kpad / BK);  // kpad is a multiple of kKBlock
  prm.tiles_n = static_cast<int>((N + BN - 1) / BN);
  prm.splits = splits;
  prm.kb_per_split = static_cast<int>((kpad / kKBlock + splits - 1) / splits) * (kKBlock / BK);
  prm.out_kind = out_kind;
  prm.mod_units = out_kind == 2 ? (n + 1) / 2 : n;
  prm.ldo = ldo;
  prm.out_plane = out_plane;
  prm.out = out;
  // CTA pairs with long chunks once every split holds kPairMinK terms;
  // single CTAs otherwise
  const bool pairs = static_cast<int64_t>(prm.kb_per_split) * BK >= kPairMinK;
  prm.tiles_m = static_cast<int>(pairs ? (M + kPairM - 1) / kPairM : (M + BM - 1) / BM);
  prm.div_tiles = fast_div(static_cast<int64_t>(prm.tiles_m) * prm.tiles_n);
  prm.div_group = fast_div(static_cast<int64_t>(kGroupM) * prm.tiles_n);
  prm.div_tail = fast_div(prm.tiles_m % kGroupM);
  prm.div_splits = fast_div(splits);
  CUtensorMap tmA, tmB;
  if (!make_slice_map(&tmA, a_slices, M, kpad, a_plane, n, BM) ||
      !make_slice_map(&tmB, b_slices, N, kpad, b_plane, n, pairs ? kBHalf : BN))
    return cudaErrorInvalidValue;
  const int64_t units = static_cast<int64_t>(prm.mod_units) * splits * prm.tiles_m * prm.tiles_n;
  // several 1024-term chunks per split (int32 sums), or one (fp32 epilogue)
  const bool long_chunks = static_cast<int64_t>(prm.kb_per_split) * BK > 1024;
  // residue planes are written by TMA stores (the callers give a 16-byte
  // aligned base, ldo and plane stride)
  CUtensorMap tmO;
  memset(&tmO, 0, sizeof(tmO));
  if (out_kind == 0 && !make_out_map(&tmO, out, M, ldo, out_plane, n)) return cudaErrorInvalidValue;
  // one instantiation per output kind: each holds only its own epilogue
  auto pick = [out_kind](auto k0, auto k1, auto k2) { return out_kind == 0 ? k0 : (out_kind == 1 ? k1 : k2); };
  auto kernel = pairs ? pick(residue_gemm_pair_kernel<0>, residue_gemm_pair_kernel<1>, residue_gemm_pair_kernel<2>)
                : long_chunks
                    ? pick(residue_gemm_kernel<true, 0>, residue_gemm_kernel<true, 1>, residue_gemm_kernel<true, 2>)
                    : pick(residue_gemm_kernel<false, 0>, residue_gemm_kernel<false, 1>, residue_gemm_kernel<false, 2>);
  const size_t smem = (pairs ? kPairSmemBytes : kSmemBytes) + kStashBytes;
  if (withhold_kb >= 0 && (pairs || withhold_kb >= prm.kb_per_split)) return cudaErrorInvalidValue;
  int resident = 0;
  cudaError_t e = kernel_setup(reinterpret_cast<const void*>(kernel), smem, pairs, &resident);
  if (e != cudaSuccess) return e;
  if (!pairs) {
    const unsigned grid = static_cast<unsigned>(units < num_sms ? units : num_sms);
    return launch_dependent(kernel, dim3(grid), dim3(kThreads), smem, stream, tmA, tmB, tmO, prm);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  pair_launch_config(&cfg, attr, smem, stream);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see grid_dependency_sync
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  // persistent: one CTA pair per co-resident cluster slot, at most one per SM pair
  int64_t npairs = num_sms / 2;
  if (resident < npairs) npairs = resident;
  if (units < npairs) npairs = units;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * npairs), 1, 1);  // clusters of two CTAs
  e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmO, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_residue_gemm(int64_t M, int64_t N, int64_t kpad, const uint16_t* a_slices,
                                int64_t a_plane, const uint16_t* b_slices, int64_t b_plane, int n,
                                int out_kind, void* out, int64_t ldo, int64_t out_plane, int splits,
                                int num_sms, cudaStream_t stream) {
  return launch_gemm(M, N, kpad, a_slices, a_plane, b_slices, b_plane, n, out_kind, out, ldo, out_plane, splits,
                     num_sms, kTimeoutNs, -1, stream);
}

cudaError_t launch_residue_gemm_withheld(int64_t M, int64_t N, int64_t kpad, const uint16_t* a_slices,
                                         int64_t a_plane, const uint16_t* b_slices, int64_t b_plane, int n,
                                         void* out, int64_t ldo, int64_t out_plane, int num_sms,
                                         uint64_t timeout_ns, int withhold_kb, cudaStream_t stream) {
  if (withhold_kb < 0 || timeout_ns == 0 || timeout_ns > kTimeoutNs) return cudaErrorInvalidValue;
  return launch_gemm(M, N, kpad, a_slices, a_plane, b_slices, b_plane, n, 0, out, ldo, out_plane, 1, num_sms,
                     timeout_ns, withhold_kb, stream);
}

int take_device_status(cudaStream_t stream, int* status) {
  *status = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return OZK_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return OZK_ERR_CUDA;
  if (v) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return OZK_ERR_CUDA;
  }
  *status = v;
  return OZK_OK;
}

}  // namespace ozk
