// HSTU jagged causal attention forward for GB300 (sm_103a).
//
//   out[t,h,:] = inv_n * sum_{j <= t, same sequence} silu(alpha q[t,h,:].k[j,h,:]) v[j,h,:]
//
// (ai6s.net "HSTU fused operator" post: section 1 formula; section 2.2 block
// tiling with the score tile kept on chip; section 3.2 in-kernel mask -- key
// blocks above the diagonal are skipped, the diagonal block is triangular;
// section 4.2 jagged values + offsets.  HSTU paper section 3.2: the
// attention becomes grouped GEMMs of different sizes over ragged sequences.)
//
// Design (one persistent CTA per SM, 24 warps -- 16 with the output stage
// or at d = 128 -- warp-specialised).  A work
// item is one 128-row query block of one (sequence, head); it walks the key
// blocks 0..qt.  Step t is the t-th key block the CTA processes.
//   warp 4        K producer (one thread): each item's Q block, then its K
//                 blocks, by bulk-tensor copies into 128B-swizzled
//                 shared-memory rings.
//   warp 6        V producer (one thread): V blocks into their own ring.
//   warp 5        QK issuer (one thread, owns TMEM): S = Q K^T
//                 (tcgen05.mma kind::f16, fp32 accumulate) of step t into
//                 TMEM S buffer t mod 3, up to three steps ahead of PV.
//   warps 8-23    four "SiLU" warpgroups in two pairs taking alternate
//                 steps, each warpgroup of a pair 64 of the block's 128 key
//                 columns (with the output stage or at d = 128: warps
//                 8-15, two warpgroups taking alternate steps, all
//                 columns).  Thread r
//                 owns score row r: tcgen05.ld S (the next 16 or 32 columns
//                 load while the current ones are computed),
//                 p = h + h tanh(h) with h = alpha s / 2
//                 (= alpha s sigmoid(alpha s)), tril select on the diagonal
//                 block, split p = bf16(p) + bf16(p - bf16(p)), tcgen05.st
//                 both halves over the S columns just read.
//   warp 7        PV issuer (one thread): O += P_hi V + P_lo V with P read
//                 from TMEM, as soon as the SiLU warpgroup has written P.
//   warps 0-3     epilogue: reads a finished item's O, scales by inv_n,
//                 rounds to bf16 and stores the valid rows with 16-byte
//                 stores.
// The roles overlap the way the post's three-stage pipeline does (section
// 5.2): QK of later blocks, SiLU of the current one and PV of an earlier
// one run at the same time.
//
// TMEM columns (512 allocated): three S buffers of 128 columns, then the O
// accumulator (d columns), double-buffered where TMEM has room (d <= 64).
// P of a block overwrites its own S buffer, two bf16 per 32-bit column:
// with four SiLU warpgroups, 16-key step k's P_hi goes to columns
// 16k+[0,8) and its P_lo to 16k+[8,16); with two, the 32-key chunk c's P_hi
// goes to 32c+[0,16) and its P_lo to 32c+[16,32).
//
// The diagonal key block of a sequence's last query block, when the sequence
// ends inside it, computes only keys < n rounded up to 16: its QK uses
// N = that width and its PV stops at the last 16-key step holding a key < n.
//
// Every mbarrier wait is bounded by a %globaltimer limit.  A wait that runs
// out records a status word, raises a CTA-wide abort flag that every other
// wait checks, and the CTA drains its own TMA copies and MMAs, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <type_traits>

#include "hstu_internal.h"

namespace hstu {

__device__ unsigned int g_dev_status;
__device__ unsigned int g_dev_site;

// Trace buffer for kDebugTrace: per warp of CTA 0 (up to 24 warps),
// kTracePerWarp events of two 64-bit words; g_trace_n[w] counts warp w's
// events.
constexpr int kTraceWarps = 24;
constexpr int kTracePerWarp = 2048;
__device__ unsigned long long g_trace[kTraceWarps * kTracePerWarp * 2];
__device__ unsigned int g_trace_n[kTraceWarps];

namespace {

constexpr int kBM = 128;  // query rows per item == TMEM lanes
constexpr int kBN = 128;  // keys per K/V block
constexpr int kEpiWarp0 = 0;
constexpr int kTmaWarpK = 4;  // Q and K blocks
constexpr int kMmaWarpQK = 5;  // QK products; owns TMEM
constexpr int kMmaWarpPV = 7;  // PV products
constexpr int kTmaWarpV = 6;  // V blocks
constexpr int kEwWarp0 = 8;
constexpr uint32_t kTmemCols = 512;

// wait-site codes reported through g_dev_site
enum : int {
  kSiteQEmpty = 1, kSiteKEmpty, kSiteVEmpty, kSiteQFull, kSiteKFull, kSitePFull, kSiteOEmpty,
  kSiteVFull, kSiteSFull, kSiteOFull, kSiteUnsignalled, kSiteSFree, kSiteCheckIn
};

// Instruction descriptor, tcgen05.mma kind::f16: D fp32, A and B bf16,
// A K-major, B K-major (0) or MN-major (1), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ----------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of a phase: the result is consumed later, so its latency
// overlaps whatever the thread issues in between.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct WaitCtx {
  unsigned long long limit_ns;
  volatile int* abort_flag;
};

__device__ __noinline__ void signal_timeout(const WaitCtx& w, int site) {
  atomicOr(&g_dev_status, 1u);
  atomicCAS(&g_dev_site, 0u, (unsigned)site);
  *w.abort_flag = 1;
}

// Bounded wait by one thread; false if the CTA aborted or the limit ran out.
// A non-blocking test comes first: a try_wait on a phase that is already
// complete still holds the thread for a few hundred cycles.
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 3u) == 0) {
      if (*w.abort_flag) return false;
      if (globaltimer() - t0 > w.limit_ns) {
        signal_timeout(w, site);
        return false;
      }
    }
  }
}

// Whole-warp bounded wait with a warp-uniform result: lane 0 polls, the
// other lanes wait at the shuffle.  The caller's tcgen05.fence::
// after_thread_sync then orders every lane's TMEM accesses after the wait.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_one(bar, parity, w, site);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Wait used only while draining after an abort: ignores the abort flag.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 2000000000ull) return;
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05): start >> 4 at bit 0, leading
// byte offset >> 4 at bit 16, stride byte offset >> 4 at bit 32, version 1
// at bit 46, layout type at bit 61.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint64_t layout) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (layout << 61);
}

// The value of x, materialised in a register at this point and hidden from
// the optimiser.  A burst of tcgen05.mma issues at about half the rate when
// its operands are computed between the instructions (measured on GB300:
// ~104 against ~50 cycles per M=128 N=64 product), so every operand of a
// burst is pinned before its first product.
__device__ __forceinline__ uint64_t pin64(uint64_t x) {
  asm volatile("mov.b64 %0, %0;" : "+l"(x));
  return x;
}
__device__ __forceinline__ uint32_t pin32(uint32_t x) {
  asm volatile("mov.b32 %0, %0;" : "+r"(x));
  return x;
}

// tcgen05.mma kind::f16, M = 128, with enable-input-d fixed at compile time
// (ACC = 0 overwrites the accumulator, 1 accumulates).  _ss: A and B from
// shared-memory descriptors; _ts: A from TMEM (the P operand), B from shared.
template <int ACC>
__device__ __forceinline__ void mma_ss_c(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc) {
  if (ACC)
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 1;" ::"r"(d_tmem), "l"(a),
                 "l"(b), "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, 0;" ::"r"(d_tmem), "l"(a),
                 "l"(b), "r"(idesc)
                 : "memory");
}

template <int ACC>
__device__ __forceinline__ void mma_ts_c(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc) {
  if (ACC)
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b), "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 0;" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b), "r"(idesc)
                 : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// 32 consecutive fp32 TMEM columns of this thread's lane; waits for completion.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Same load without the wait: the registers are not valid until
// tmem_wait_ld(r) below, which ties them to the wait so that no use of them
// can be scheduled before it.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// 16 consecutive fp32 TMEM columns of this thread's lane, without the wait
// (tmem_wait_ld16 below ties the registers to it).
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 -> bf16x2 (round to nearest even); `lo` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Trace event codes.
enum : unsigned {
  kEvQkIssue = 1,  // MMA warp: QK of block index issued
  kEvPvIssue,      // MMA warp: PV of block index issued (after its waits)
  kEvSiluStart,    // SiLU warp: S of block index ready
  kEvSiluEnd,      // SiLU warp: P of block index written
  kEvEpiStart,     // epilogue warp: O of item ready
  kEvEpiEnd,       // epilogue warp: rows of item stored
  kEvLoadK,        // producer: K block load issued
  kEvLoadV,        // producer: V block load issued
  kEvLoadQ,        // producer: Q block load issued
  kEvMmaKReady,    // MMA warp: K block index present
  kEvMmaQkDone,    // MMA warp: QK instructions and commits of block index issued
  kEvMmaPReady,    // MMA warp: P of block index present
  kEvMmaPvDone,    // MMA warp: PV instructions and commits of block index issued
};

// Per-warp trace slot counters live in shared memory (set by the kernel).
__device__ __forceinline__ uint32_t* trace_counters();

// One trace event from lane 0 of the calling warp, CTA 0 only: a plain
// store into this warp's region, so the warp does not wait on it.
__device__ __forceinline__ void trace(const FwdArgs& a, unsigned ev, unsigned idx) {
  if (!(a.debug_flags & kDebugTrace) || blockIdx.x != 0 || (threadIdx.x & 31) != 0) return;
  const unsigned warp = threadIdx.x >> 5;
  uint32_t* cnt = trace_counters() + warp;
  const unsigned slot = *cnt;
  if (slot < (unsigned)kTracePerWarp) {
    *cnt = slot + 1;
    unsigned long long* dst = g_trace + 2 * ((size_t)warp * kTracePerWarp + slot);
    dst[0] = clock64();
    dst[1] = ((unsigned long long)ev << 48) | ((unsigned long long)warp << 40) | idx;
  }
}

__device__ __forceinline__ uint32_t* trace_counters() {
  __shared__ uint32_t counters[kTraceWarps];
  return counters;
}

__device__ __forceinline__ int item_index(int it, int cta, int grid) {
  // serpentine over the longest-first list: even rounds left to right, odd
  // rounds right to left, so that CTAs even out the cost of their items.
  const int base = it * grid;
  return (it & 1) ? base + (grid - 1 - cta) : base + cta;
}

// ------------------------------------------------------------------ roles
template <int D>
struct Cfg {
  static constexpr int CHUNK = D < 64 ? D : 64;  // elements per swizzled row
  static constexpr int NCHUNK = D / CHUNK;
  static constexpr int ROWB = CHUNK * 2;          // bytes per swizzled row: 128 or 64
  static constexpr int ATOMB = 8 * ROWB;          // 8-row swizzle atom
  static constexpr int CHUNKB = kBM * ROWB;       // 128 rows of one chunk
  static constexpr int TILEB = kBM * D * 2;       // one 128 x D bf16 block
  // S buffers in TMEM, K-ring and V-ring slots all have the period P, so
  // that "QK of step t done" frees K slot t mod P and "PV of step t done"
  // frees V slot t mod P: the MMA issuer's loop, unrolled by P, sees every
  // buffer and slot as a compile-time constant.
  static constexpr int P = 3;
  static constexpr int QS = D == 128 ? 1 : 2;  // Q slots (d = 128: shared memory is full)
  // O accumulators (d columns each): double-buffered when TMEM has room.
  static constexpr int OB = 128 * P + 2 * D <= (int)kTmemCols ? 2 : 1;
  static constexpr uint64_t LAYOUT = ROWB == 128 ? 2 : 4;  // descriptor layout: 128B / 64B swizzle
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + QS * TILEB;
  static constexpr int V_OFF = K_OFF + P * TILEB;
  static constexpr int BAR_OFF = V_OFF + P * TILEB;
  static constexpr int B_QFULL = 0;
  static constexpr int B_QEMPTY = B_QFULL + QS;    // an item's last QK done: Q slot free
  // QK-ready j, phase k: K of step t = P k + j landed and PV(t - P), which
  // read P from S buffer j, done (for k = 0 an arrival at set-up stands in).
  static constexpr int B_QKREADY = B_QEMPTY + QS;
  static constexpr int B_VFULL = B_QKREADY + P;
  static constexpr int B_SFULL = B_VFULL + P;      // QK done: S written, K slot free
  static constexpr int B_PFULL = B_SFULL + P;      // SiLU done: P written
  static constexpr int B_OFULL = B_PFULL + P;      // an item's last PV done
  static constexpr int B_OEMPTY = B_OFULL + OB;
  static constexpr int B_DRAIN = B_OEMPTY + OB;  // [2]: the two MMA issuers' drains
  static constexpr int NBARS = B_DRAIN + 2;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag
  static constexpr int USED = MISC_OFF + 16;
  static constexpr int SMEM = ((USED + 1023) / 1024) * 1024 + 1024;  // + realignment slack
  // Ask for more than half an SM's shared memory so that exactly one CTA
  // (and one 512-column TMEM allocation) lives on each SM.
  static constexpr int SMEM_LAUNCH = SMEM < 120 * 1024 ? 120 * 1024 : SMEM;
  // TMEM columns: S buffer j at 128 j; O buffer ob at 128 P + ob d.
  static constexpr uint32_t O_COL = 128u * P;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(128 * P + OB * D <= (int)kTmemCols, "TMEM budget");
  // Arrivals that complete a phase of barrier i: every thread of the SiLU
  // warpgroup (P-full; both warpgroups of a pair when `wide`), one per
  // epilogue warp (O-empty), the K copy's and the PV commit's (QK-ready),
  // else one.
  __host__ __device__ static constexpr uint32_t arrivals(int i, bool wide) {
    return (i >= B_PFULL && i < B_PFULL + P)       ? (wide ? 256u : 128u)
           : (i >= B_OEMPTY && i < B_OEMPTY + OB)   ? 4u
           : (i >= B_QKREADY && i < B_QKREADY + P) ? 2u
                                                   : 1u;
  }
};

// A work item decoded: query block qt of one (sequence, head).
struct Block {
  int s0, n, h, qt;
  __device__ __forceinline__ int rows() const {  // valid query rows (1..128)
    const int r = n - kBM * qt;
    return r < kBM ? r : kBM;
  }
  // Keys of key block kt that a valid row can see: 128, except for the
  // diagonal block of the sequence's last query block when the sequence ends
  // inside it (rounded up to the 16-key MMA step).
  __device__ __forceinline__ int cols(int kt) const {
    if (kt != qt) return kBN;
    const int r = n - kBN * kt;
    return r >= kBN ? kBN : ((r + 15) & ~15);
  }
};

// An item of the candidate mask, with its history length.
struct BlockTgt : Block {
  int hist;  // history tokens of the sequence
  int nk;    // key blocks the item walks (see load_block)
  // The ki-th key block the item walks: 0 .. nk - 2, then the diagonal qt.
  __device__ __forceinline__ int key_block(int ki) const { return ki == nk - 1 ? qt : ki; }
  // No key of block kt is masked: an off-diagonal block of history keys only.
  __device__ __forceinline__ bool unmasked(int kt) const {
    return kt != qt && kBN * kt + kBN <= hist;
  }
};

template <bool TGT>
using BlockOf = typename std::conditional<TGT, BlockTgt, Block>::type;

// Kernel variants, one instantiation each so that the plain causal kernel
// carries none of the others' bookkeeping: the candidate mask (items carry
// a history length), the output stage (Norm(O) (.) U; the epilogue writes
// fp32 rows and moments) and the relative attention bias (in the SiLU
// stage).
constexpr int kVarTargets = 1, kVarNorm = 2, kVarRab = 4;
template <int VAR>
constexpr bool has_targets = (VAR & kVarTargets) != 0;
template <int VAR>
constexpr bool has_norm = (VAR & kVarNorm) != 0;
template <int VAR>
constexpr bool has_rab = (VAR & kVarRab) != 0;
// Without the output stage and at d <= 64 the kernel runs four SiLU
// warpgroups in two pairs: a pair takes alternate blocks and each of its
// warpgroups 64 of the block's 128 key columns (the bias: two of its four
// 32-key chunks), so that four SiLU warps share each SMSP.  This P layout
// puts each 16-key step's P_hi and P_lo in that step's own 16 columns.  The
// others (d = 128: 768 threads leave 80 registers a thread, and its
// epilogue spills; the output stage: measured 1.3% slower on dense with
// four) run two warpgroups, each taking whole alternate blocks.
template <int D, int VAR>
constexpr bool kWideSilu = !has_norm<VAR> && D <= 64;
template <int D, int VAR>
constexpr int kFwdThreadsOf = kWideSilu<D, VAR> ? 768 : kFwdThreads;

// TGT: items carry a history length (the candidate mask); otherwise every
// item walks key blocks 0 .. qt.
template <int VAR>
__device__ __forceinline__ bool load_block(const FwdArgs& a, int it, BlockOf<has_targets<VAR>>& b) {
  constexpr bool TGT = has_targets<VAR>;
  const int idx = item_index(it, blockIdx.x, gridDim.x);
  if (idx >= a.n_items) return false;
  const Item x = __ldg(&a.items[idx]);
  b.s0 = x.x;
  b.n = x.y;
  b.h = x.z;
  b.qt = x.w;
  if constexpr (TGT) {
    // Key blocks the item walks (HSTU paper Appendix H, the M-FALCON mask):
    // the blocks that hold history keys, 0 .. min(qt, KH) - 1 with
    // KH = ceil(hist / 128), then the diagonal block qt.  A block between
    // them holds only keys of other candidates.
    b.hist = __ldg(&a.item_hist[idx]);
    const int kh = (b.hist + kBN - 1) / kBN;
    b.nk = (b.qt < kh ? b.qt : kh) + 1;
  }
  return true;
}

// A cursor over the CTA's key-block steps: item `it` (block b) at its
// ki-th key block kt; tc counts the steps.  The next item's block is fetched one item ahead
// so that crossing into it does not wait on a global load.
template <int VAR>
struct Cursor {
  static constexpr bool TGT = has_targets<VAR>;
  int it, kt, ki;  // ki: index of the step among the item's key blocks; kt = b.key_block(ki)
  uint32_t tc;
  BlockOf<TGT> b, nb;
  bool valid, nvalid;
  // The item's first key block: 0, except for a candidate item that walks
  // its diagonal block alone (no history keys before it).
  __device__ __forceinline__ int first_kt() const {
    if constexpr (TGT) return b.nk == 1 ? b.qt : 0;
    return 0;
  }
  __device__ __forceinline__ void start(const FwdArgs& a) {
    it = 0;
    ki = 0;
    tc = 0;
    valid = load_block<VAR>(a, 0, b);
    kt = valid ? first_kt() : 0;
    nvalid = valid && load_block<VAR>(a, 1, nb);
  }
  __device__ __forceinline__ void advance(const FwdArgs& a) {
    ++tc;
    bool next_item;
    if constexpr (TGT) {
      next_item = ++ki >= b.nk;
      if (!next_item) kt = ki == b.nk - 1 ? b.qt : ki;
    } else {
      next_item = ++kt > b.qt;
      ki = kt;
    }
    if (next_item) {
      ki = 0;
      ++it;
      valid = nvalid;
      b = nb;
      kt = valid ? first_kt() : 0;
      nvalid = valid && load_block<VAR>(a, it + 1, nb);
    }
  }
};

// ------------------------------------------------------------------ roles
// Runs f(integral_constant<int, I>) for I = 0, 1, ..., U-1, 0, 1, ... until
// it returns false: the step function of a role sees the step's position in
// the unroll period as a compile-time constant.
template <int I, int U, class F>
__device__ __forceinline__ bool unrolled_steps(F& f) {
  if constexpr (I == U) {
    return true;
  } else {
    if (!f(std::integral_constant<int, I>{})) return false;
    return unrolled_steps<I + 1, U>(f);
  }
}
template <int U, class F>
__device__ __forceinline__ void run_unrolled(F& f) {
  while (unrolled_steps<0, U>(f)) {
  }
}

// Waits after an abort for the last phase armed on each of `slots` full
// barriers that `count` copies were issued on, so that no copy is still
// landing when the CTA exits.
__device__ __forceinline__ void drain_copies(uint32_t full0, int slots, uint32_t count) {
  for (int s = 0; s < slots; ++s) {
    if (count > (uint32_t)s) {
      const uint32_t uses = (count - 1u - (uint32_t)s) / (uint32_t)slots + 1u;
      wait_drain(full0 + 8u * (uint32_t)s, (uses - 1u) & 1u);
    }
  }
}

// TMA producers (one thread each).  A single thread's bulk-tensor copies
// are processed one box at a time, so the K stream (with each item's Q
// block) and the V stream have separate issuing threads in separate warps.
// K slot t mod P is free once QK(t-P) has completed (S-full); the K copy
// lands on QK-ready.  V slot t mod P is free once PV(t-P) has completed,
// which QK-ready of step t includes.  A Q slot is free once the item's last
// QK has completed (Q-empty).
template <int D, bool KQ, int VAR>
__device__ void role_producer(const CUtensorMap* tm_a, const CUtensorMap* tm_q, const FwdArgs& a,
                              uint32_t base, const WaitCtx& w) {
  using C = Cfg<D>;
  constexpr bool TGT = has_targets<VAR>;
  constexpr int FULL = KQ ? C::B_QKREADY : C::B_VFULL;
  constexpr int OFF = KQ ? C::K_OFF : C::V_OFF;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  uint32_t c = 0, qc = 0;
  bool ok = true;
  BlockOf<TGT> b;
  for (int it = 0; ok && load_block<VAR>(a, it, b); ++it) {
    if (KQ) {
      const int qs = (int)(qc % C::QS);
      if (!(ok = wait_one(bar(C::B_QEMPTY + qs), ((qc / C::QS) & 1u) ^ 1u, w, kSiteQEmpty))) break;
      trace(a, kEvLoadQ, qc);
      mbar_arrive_expect_tx(bar(C::B_QFULL + qs), C::TILEB);
#pragma unroll
      for (int ch = 0; ch < C::NCHUNK; ++ch)
        tma_load_3d(base + C::Q_OFF + qs * C::TILEB + ch * C::CHUNKB, tm_q, bar(C::B_QFULL + qs),
                    ch * C::CHUNK, b.h, b.s0 + kBM * b.qt);
      ++qc;
    }
    int nk = b.qt + 1;
    if constexpr (TGT) nk = b.nk;
    for (int ki = 0; ki < nk; ++ki) {
      int kt = ki;
      if constexpr (TGT) kt = b.key_block(ki);
      const int slot = (int)(c % C::P);
      // A parity wait is exact only while the barrier is at most one phase
      // short of the awaited one.  K(c) waits for phase c/P - 1 of S-full
      // (its first use passes at once).  V(c) waits for phase c/P of
      // QK-ready, the first uses included: phase 0 (K landed) must be seen
      // complete before phase 1 is awaited, or a barrier still in phase 0
      // would pass the wait for phase 1.
      ok = KQ ? wait_one(bar(C::B_SFULL + slot), ((c / C::P) & 1u) ^ 1u, w, kSiteKEmpty)
              : wait_one(bar(C::B_QKREADY + slot), (c / C::P) & 1u, w, kSiteVEmpty);
      if (!ok) break;
      trace(a, KQ ? kEvLoadK : kEvLoadV, c);
      mbar_arrive_expect_tx(bar(FULL + slot), C::TILEB);
#pragma unroll
      for (int ch = 0; ch < C::NCHUNK; ++ch)
        tma_load_3d(base + OFF + slot * C::TILEB + ch * C::CHUNKB, tm_a, bar(FULL + slot),
                    ch * C::CHUNK, b.h, b.s0 + kBN * kt);
      ++c;
    }
  }
  if (!ok) {
    drain_copies(bar(FULL), C::P, c);
    if (KQ) drain_copies(bar(C::B_QFULL), C::QS, qc);
  }
}

// MMA issuers.  A thread's tcgen05.mma returns only when the tensor pipe
// takes it, so a thread that issues products cannot meanwhile wait on
// barriers or compute addresses; the QK and PV products therefore come from
// two threads, each with little work between its products, and every
// product's operands are pinned in registers before a burst starts.
//
// QK issuer (one thread, owns TMEM): S_j = Q K^T of step t into S buffer
// j = t mod P (P = 3), once K(t) has landed and PV(t-P), which read P from
// that buffer, has completed (QK-ready); the products of different
// accumulators are not ordered with respect to each other, so this wait is
// needed.  It runs up to P steps ahead of the PV issuer.
template <int D, int VAR>
__device__ void role_mma_qk(const FwdArgs& a, uint32_t base, uint32_t tmem, const WaitCtx& w) {
  using C = Cfg<D>;
  constexpr bool TGT = has_targets<VAR>;
  constexpr int P = C::P;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  constexpr uint32_t IDESC_QK = make_idesc(kBM, kBN, 0);
  constexpr int QK_STEPS = D / 16;
  constexpr int STEPS_PER_CHUNK = C::CHUNK / 16;
  const uint64_t q_desc0 = smem_desc(base + C::Q_OFF, 16, C::ATOMB, C::LAYOUT);
  const uint64_t k_desc0 = smem_desc(base + C::K_OFF, 16, C::ATOMB, C::LAYOUT);
  bool ok = true;
  // Test hook: wait on a barrier that nothing arrives on, so that the
  // bounded wait runs out and the whole CTA takes its give-up path.
  if (a.debug_flags & kDebugUnsignalledWait) ok = wait_one(bar(C::B_DRAIN), 0u, w, kSiteUnsignalled);
  Cursor<VAR> qc;
  qc.start(a);
  uint32_t ph = 0;  // (qc.tc / P) & 1
  auto step = [&](auto jc) -> bool {
    constexpr int J = decltype(jc)::value;
    if (!ok || !qc.valid) return false;
    const int qs = C::QS == 1 ? 0 : (qc.it & 1);
    if (qc.ki == 0 &&
        !(ok = wait_one(bar(C::B_QFULL + qs), (uint32_t)(qc.it / C::QS) & 1u, w, kSiteQFull)))
      return false;
    if (!(ok = wait_one(bar(C::B_QKREADY + J), ph, w, kSiteKFull))) return false;
    tc_fence_after();
    trace(a, kEvQkIssue, qc.tc);
    const int cols = qc.b.cols(qc.kt);
    const uint32_t s_tmem = pin32(tmem + (uint32_t)(J * 128));
    const uint32_t idesc = pin32(cols == kBN ? IDESC_QK : make_idesc(kBM, cols, 0));
    // 16-wide K steps: within a swizzled 64-column chunk the start address
    // advances 32 bytes per step, across chunks by a whole chunk
    const uint64_t qd0 = q_desc0 + (uint64_t)((qs * C::TILEB) >> 4);
    uint64_t qd[QK_STEPS], kd[QK_STEPS];
#pragma unroll
    for (int kk = 0; kk < QK_STEPS; ++kk) {
      const uint32_t off = (kk / STEPS_PER_CHUNK) * C::CHUNKB + (kk % STEPS_PER_CHUNK) * 32;
      qd[kk] = pin64(qd0 + (uint64_t)(off >> 4));
      kd[kk] = pin64(k_desc0 + (uint64_t)((J * C::TILEB + off) >> 4));
    }
    mma_ss_c<0>(s_tmem, qd[0], kd[0], idesc);
#pragma unroll
    for (int kk = 1; kk < QK_STEPS; ++kk) mma_ss_c<1>(s_tmem, qd[kk], kd[kk], idesc);
    mma_commit(bar(C::B_SFULL + J));
    if (qc.kt == qc.b.qt) mma_commit(bar(C::B_QEMPTY + qs));
    qc.advance(a);
    if (J == P - 1) ph ^= 1u;
    return true;
  };
  run_unrolled<P>(step);
  if (!ok) {
    // Drain: a commit arrives once every MMA issued before it has finished.
    mma_commit(bar(C::B_DRAIN));
    wait_drain(bar(C::B_DRAIN), 0);
  }
}

// PV issuer (one thread).  Step s issues O += P_hi V + P_lo V once the SiLU
// warpgroup has written P (P-full) and V(s) has landed, into O buffer
// ob = item mod OB, and commits QK-ready (S buffer and V slot free).  The
// barriers of the next step are tested (without blocking) before the
// current step's products are issued, so that the tests' latency overlaps
// them.  16-key step k: P_hi in columns 32 (k/2) + 8 (k%2) + [0, 8), P_lo 16
// columns further; V rows 16 k.. (two 8-row atoms per step).
template <int D, int VAR>
__device__ void role_mma_pv(const FwdArgs& a, uint32_t base, uint32_t tmem, const WaitCtx& w) {
  using C = Cfg<D>;
  constexpr bool TGT = has_targets<VAR>;
  constexpr int P = C::P;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  constexpr uint32_t IDESC_PV = make_idesc(kBM, D, 1);
  const uint64_t v_desc0 = smem_desc(base + C::V_OFF, C::CHUNKB, C::ATOMB, C::LAYOUT);
  bool ok = true;
  Cursor<VAR> pc;
  pc.start(a);
  uint32_t ph = 0;  // (pc.tc / P) & 1

  auto issue_pv = [&](auto jc, auto hc, int ob) {
    constexpr int J = decltype(jc)::value;
    constexpr int H = decltype(hc)::value;
    const uint32_t o_tmem = pin32(tmem + C::O_COL + (uint32_t)(ob * D));
    uint32_t pa[8];
    uint64_t vb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int kk = 4 * H + i;
      // P_hi and P_lo of 16-key step kk (the SiLU stage's layout)
      const int hi_col = kWideSilu<D, VAR> ? 16 * kk : 32 * (kk >> 1) + 8 * (kk & 1);
      constexpr int lo_off = kWideSilu<D, VAR> ? 8 : 16;
      pa[2 * i] = pin32(tmem + (uint32_t)(J * 128 + hi_col));
      pa[2 * i + 1] = pin32(tmem + (uint32_t)(J * 128 + hi_col + lo_off));
      vb[i] = pin64(v_desc0 + (uint64_t)((J * C::TILEB + kk * 2 * C::ATOMB) >> 4));
    }
    if (pc.kt != pc.b.qt && (H == 1 || pc.ki != 0)) {
      // full half continuing an accumulation
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        mma_ts_c<1>(o_tmem, pa[2 * i], vb[i], IDESC_PV);
        mma_ts_c<1>(o_tmem, pa[2 * i + 1], vb[i], IDESC_PV);
      }
    } else {
      // an item's first block (the first product overwrites O) or its last
      // (only the 16-key steps that hold keys < n)
      const int cols = pc.b.cols(pc.kt);
      const int n_steps = (cols - 64 * H) / 16;  // <= 0: none in this half
      const bool first = H == 0 && pc.ki == 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i < n_steps) {
          if (i == 0 && first)
            mma_ts_c<0>(o_tmem, pa[0], vb[0], IDESC_PV);
          else
            mma_ts_c<1>(o_tmem, pa[2 * i], vb[i], IDESC_PV);
          mma_ts_c<1>(o_tmem, pa[2 * i + 1], vb[i], IDESC_PV);
        }
      }
    }
  };

  bool pa_ready = false, v_ready = false;  // tests made for the coming PV_0
  auto step = [&](auto ic) -> bool {
    constexpr int J = decltype(ic)::value;
    constexpr int JN = (J + 1) % P;  // next step's buffer
    if (!ok || !pc.valid) return false;
    const int ob = C::OB == 1 ? 0 : (pc.it & 1);
    const bool last = pc.kt == pc.b.qt;
    if (!pa_ready && !(ok = wait_one(bar(C::B_PFULL + J), ph, w, kSitePFull))) return false;
    if (pc.ki == 0 &&
        !(ok = wait_one(bar(C::B_OEMPTY + ob), ((uint32_t)(pc.it / C::OB) & 1u) ^ 1u, w, kSiteOEmpty)))
      return false;
    if (!v_ready && !(ok = wait_one(bar(C::B_VFULL + J), ph, w, kSiteVFull))) return false;
    if (last) {
      // Keys in [n, cols) lie past the end of the sequence: zero their V
      // rows so that the zero P entries never meet non-finite values of the
      // next sequence.
      const int cols = pc.b.cols(pc.kt);
      const int r_end = pc.b.n - kBN * pc.kt;
      if (r_end < cols) {
        const uint32_t v_addr = base + C::V_OFF + J * C::TILEB;
#pragma unroll
        for (int ch = 0; ch < C::NCHUNK; ++ch) {
          const uint32_t z0 = v_addr + ch * C::CHUNKB + r_end * C::ROWB;
          const uint32_t z1 = v_addr + ch * C::CHUNKB + cols * C::ROWB;
          for (uint32_t z = z0; z < z1; z += 16)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(z), "r"(0) : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
    }
    tc_fence_after();
    trace(a, kEvPvIssue, pc.tc);
    const uint32_t npar = J + 1 == P ? ph ^ 1u : ph;
    pa_ready = mbar_test(bar(C::B_PFULL + JN), npar);
    v_ready = mbar_test(bar(C::B_VFULL + JN), npar);
    issue_pv(std::integral_constant<int, J>{}, std::integral_constant<int, 0>{}, ob);
    issue_pv(std::integral_constant<int, J>{}, std::integral_constant<int, 1>{}, ob);
    mma_commit(bar(C::B_QKREADY + J));  // PV(s) done: S buffer J and V slot J free
    if (last) mma_commit(bar(C::B_OFULL + ob));
    pc.advance(a);
    if (J == P - 1) ph ^= 1u;
    return true;
  };
  run_unrolled<P>(step);
  if (!ok) {
    mma_commit(bar(C::B_DRAIN + 1));
    wait_drain(bar(C::B_DRAIN + 1), 0);
  }
}

// silu of the 32 scores s of one row, written over their own TMEM columns
// at t: keys 16h..16h+15 go to P_hi columns t + 8h + [0, 8) and P_lo columns
// t + 16 + 8h + [0, 8).  Processed in 16-key halves to keep register
// pressure down.  MASK 0: no mask; 1: keep keys k <= lim (the diagonal
// block); 2: also drop keys k >= lim_hist other than k == lim (the candidate
// mask).
// The relative attention bias rab_{p,t} (HSTU paper section 3; section 3.4
// for candidates).  The construction is lost in extraction; the reading
// taken is a pair of bucketed tables added to the scaled score:
//   bias(i, j) = pos[min(floor(log2(dp + 1)), npos - 1)]
//              + time[min(floor(log2(dt + 1)), ntime - 1)],
//   dp = p(i) - p(j) (p(i) = i, or hist for a candidate), dt = max(ts_i - ts_j, 0).
// floor(log2(x)) = 31 - clz(x) for 1 <= x <= 2^31, so lane l holds half the
// entry of bucket 31 - l (clamped to the table), and a lookup is one shuffle
// from lane clz(x): no gather, no clamp.
struct RabRow {
  const int32_t* ts;  // timestamps of the item's sequence
  int last;           // its last token (sequence-local)
  int pe_i;           // the row's position (hist for a candidate)
  int ts_i;
  int hist;           // candidates: the history length
  float pos_l, time_l;  // this lane's table entries, halved
};

// A chunk of 32 keys j0 .. j0 + 31 for the warp's 32 rows.  Position buckets
// never grow with j (p is non-decreasing), and neither do time buckets
// when the chunk's timestamps are in order.  So a part whose buckets at the
// chunk's two ends agree on every lane of the warp is one value per row;
// only the other parts are looked up per key.
struct RabChunk {
  int ts_lane;       // timestamp of key j0 + lane
  float pos_c, time_c;  // the row's table entries (as the lanes hold them) at the chunk's first key
  int lp0, lt0;         // the lanes that hold them
  bool fix_p, fix_t;    // warp-uniform: the part is constant over the chunk
};

template <bool TGT>
__device__ __forceinline__ int rab_pe(const RabRow& r, int j) {
  return TGT ? (j < r.hist ? j : r.hist) : j;
}

__device__ __forceinline__ int rab_lane(int delta) {  // source lane of delta's bucket
  return __clz((int)((uint32_t)(delta > 0 ? delta : 0) + 1u));
}

// ts_lane: the timestamp of key j0 + lane (loaded ahead by the caller).
template <bool TGT>
__device__ __forceinline__ RabChunk rab_chunk(const RabRow& r, int j0, int ts_lane) {
  RabChunk c;
  const int lane = threadIdx.x & 31;
  c.ts_lane = ts_lane;
  const int nxt = __shfl_down_sync(0xffffffffu, c.ts_lane, 1);
  const bool in_order = __all_sync(0xffffffffu, lane == 31 || c.ts_lane <= nxt);
  const int ts_first = __shfl_sync(0xffffffffu, c.ts_lane, 0);
  const int ts_end = __shfl_sync(0xffffffffu, c.ts_lane, 31);
  const int lp0 = rab_lane(r.pe_i - rab_pe<TGT>(r, j0));
  const int lp1 = rab_lane(r.pe_i - rab_pe<TGT>(r, j0 + 31));
  const int lt0 = rab_lane(r.ts_i - ts_first);
  const int lt1 = rab_lane(r.ts_i - ts_end);
  c.fix_p = __all_sync(0xffffffffu, lp0 == lp1);
  c.fix_t = in_order && __all_sync(0xffffffffu, lt0 == lt1);
  c.pos_c = __shfl_sync(0xffffffffu, r.pos_l, lp0);
  c.time_c = __shfl_sync(0xffffffffu, r.time_l, lt0);
  c.lp0 = lp0;
  c.lt0 = lt0;
  return c;
}

// Halved bias of key j0 + k (k a compile-time constant after unrolling).
template <bool TGT, bool FP, bool FT>
__device__ __forceinline__ float rab_half(const RabRow& r, const RabChunk& c, int j0, int k) {
  float bp, bt;
  if constexpr (FP) {
    bp = c.pos_c;
  } else {
    bp = __shfl_sync(0xffffffffu, r.pos_l, rab_lane(r.pe_i - rab_pe<TGT>(r, j0 + k)));
  }
  if constexpr (FT) {
    bt = c.time_c;
  } else {
    const int ts_j = __shfl_sync(0xffffffffu, c.ts_lane, k);
    bt = __shfl_sync(0xffffffffu, r.time_l, rab_lane(r.ts_i - ts_j));
  }
  return bp + bt;
}

// MASK 0: none; 1: keep key k iff k <= lim; 2: the candidate mask.  RAB:
// add the relative attention bias of keys j0 .. j0 + 31 (sequence-local),
// FP / FT: its position / time part is constant over the chunk.
// WL: the wide P layout (16-key step k's P_hi at 16 k + [0, 8), P_lo at
// 16 k + [8, 16)), else P_hi of keys 16h.. at t + 8h + [0, 8) and P_lo at
// t + 16 + 8h + [0, 8).
template <int MASK, bool RAB = false, bool TGT = false, bool FP = false, bool FT = false,
          bool WL = false>
__device__ __forceinline__ void silu_store32_body(const uint32_t (&s)[32], float2 ha2, int lim,
                                                  int lim_hist, uint32_t t, const RabRow* rab,
                                                  const RabChunk* rc, int j0) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int k = 16 * h + 2 * m;
      float2 x;
      if constexpr (RAB) {
        const float2 bh = make_float2(rab_half<TGT, FP, FT>(*rab, *rc, j0, k),
                                      rab_half<TGT, FP, FT>(*rab, *rc, j0, k + 1));
        x = __ffma2_rn(make_float2(__uint_as_float(s[k]), __uint_as_float(s[k + 1])), ha2, bh);
      } else {
        x = __fmul2_rn(make_float2(__uint_as_float(s[k]), __uint_as_float(s[k + 1])), ha2);
      }
      float2 p = __ffma2_rn(x, make_float2(tanh_approx(x.x), tanh_approx(x.y)), x);
      if (MASK == 1) {  // keep key k iff k <= lim (causal)
        p.x = (k > lim) ? 0.0f : p.x;
        p.y = (k + 1 > lim) ? 0.0f : p.y;
      } else if (MASK == 2) {
        // and a key past the history (k >= lim_hist) is seen by its own row
        // (k == lim) only
        p.x = (k > lim || (k >= lim_hist && k != lim)) ? 0.0f : p.x;
        p.y = (k + 1 > lim || (k + 1 >= lim_hist && k + 1 != lim)) ? 0.0f : p.y;
      }
      const uint32_t ph = pack_bf16x2(p.x, p.y);
      const float2 r = __fadd2_rn(
          p, make_float2(-__uint_as_float(ph << 16), -__uint_as_float(ph & 0xFFFF0000u)));
      hi[m] = ph;
      lo[m] = pack_bf16x2(r.x, r.y);
    }
    tmem_st8(t + (WL ? 16u * h : 8u * h), hi);
    tmem_st8(t + (WL ? 16u * h + 8u : 16u + 8u * h), lo);
  }
}

// silu of 16 scores s of one row (the wide layout): P_hi of the 16 keys to
// columns t + [0, 8), P_lo to t + [8, 16), over the scores just read.
// MASK 0: none; 1: keep key k iff k <= lim; 2: the candidate mask.
template <int MASK>
__device__ __forceinline__ void silu_store16(const uint32_t (&s)[16], float2 ha2, int lim, int lim_hist,
                                             uint32_t t) {
  uint32_t hi[8], lo[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int k = 2 * m;
    const float2 x = __fmul2_rn(make_float2(__uint_as_float(s[k]), __uint_as_float(s[k + 1])), ha2);
    float2 p = __ffma2_rn(x, make_float2(tanh_approx(x.x), tanh_approx(x.y)), x);
    if (MASK == 1) {
      p.x = (k > lim) ? 0.0f : p.x;
      p.y = (k + 1 > lim) ? 0.0f : p.y;
    } else if (MASK == 2) {
      p.x = (k > lim || (k >= lim_hist && k != lim)) ? 0.0f : p.x;
      p.y = (k + 1 > lim || (k + 1 >= lim_hist && k + 1 != lim)) ? 0.0f : p.y;
    }
    const uint32_t ph = pack_bf16x2(p.x, p.y);
    const float2 r = __fadd2_rn(
        p, make_float2(-__uint_as_float(ph << 16), -__uint_as_float(ph & 0xFFFF0000u)));
    hi[m] = ph;
    lo[m] = pack_bf16x2(r.x, r.y);
  }
  tmem_st8(t, hi);
  tmem_st8(t + 8u, lo);
}

template <int MASK, bool RAB = false, bool TGT = false, bool WL = false>
__device__ __forceinline__ void silu_store32(const uint32_t (&s)[32], float2 ha2, int lim, int lim_hist,
                                             uint32_t t, const RabRow* rab = nullptr, int j0 = 0,
                                             int ts_lane = 0) {
  if constexpr (!RAB) {
    silu_store32_body<MASK, false, false, false, false, WL>(s, ha2, lim, lim_hist, t, nullptr,
                                                            nullptr, 0);
  } else {
    const RabChunk rc = rab_chunk<TGT>(*rab, j0, ts_lane);
    if (rc.fix_p && rc.fix_t)
      silu_store32_body<MASK, true, TGT, true, true, WL>(s, ha2, lim, lim_hist, t, rab, &rc, j0);
    else if (rc.fix_p)
      silu_store32_body<MASK, true, TGT, true, false, WL>(s, ha2, lim, lim_hist, t, rab, &rc, j0);
    else if (rc.fix_t)
      silu_store32_body<MASK, true, TGT, false, true, WL>(s, ha2, lim, lim_hist, t, rab, &rc, j0);
    else
      silu_store32_body<MASK, true, TGT, false, false, WL>(s, ha2, lim, lim_hist, t, rab, &rc, j0);
  }
}

// SiLU warpgroups (warps 8-11 and 12-15): warpgroup e takes the steps with
// tc % 2 == e, all 128 key columns of the block (whole blocks amortise the
// per-step waits and arrivals twice as well as half blocks do).  In the
// wide variant (warps 8-23) pair e = warpgroups 2e and 2e + 1 takes those
// steps, warpgroup 2e + h the key columns [64 h, 64 h + 64).  Thread r
// owns score row r.  Every lane waits on S-full and arrives on P-full
// itself (a vote keeps the warp's view uniform), so no lane-0 relay or warp
// barrier sits on the path.
template <int D, int VAR>
__device__ void role_silu(const FwdArgs& a, uint32_t base, uint32_t tmem, const WaitCtx& w, int warp,
                          int lane) {
  using C = Cfg<D>;
  constexpr bool TGT = has_targets<VAR>;
  constexpr int P = C::P;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  constexpr bool WIDE = kWideSilu<D, VAR>;
  const int wg = (warp - kEwWarp0) >> 2;
  const int e = WIDE ? wg >> 1 : wg;  // takes the steps with tc % 2 == e
  const int half = WIDE ? wg & 1 : 0;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
  const float2 ha2 = make_float2(a.half_alpha, a.half_alpha);
  constexpr bool RAB = has_rab<VAR>;
  RabRow rr{};
  if constexpr (RAB) {
    const int bp = 31 - lane, bt = 31 - lane;
    rr.pos_l = 0.5f * __ldg(a.rab_pos + (bp < a.rab_npos - 1 ? bp : a.rab_npos - 1));
    rr.time_l = 0.5f * __ldg(a.rab_time + (bt < a.rab_ntime - 1 ? bt : a.rab_ntime - 1));
  }
  Cursor<VAR> cur;
  cur.start(a);
  uint32_t s0[32], s1[32];
  while (cur.valid) {
    if ((int)(cur.tc & 1u) != e) {
      cur.advance(a);
      continue;
    }
    const int j = (int)(cur.tc % P);
    const int kbase = kBN * cur.kt;
    int tsk[4];  // the block's key timestamps, key kbase + 32 c + lane
    if constexpr (RAB) {
      // the row's position and timestamp (a row past the sequence reads its
      // last token; its results are never stored), loaded with the keys'
      // timestamps before the wait so that their latency hides behind it
      const int i = kBM * cur.b.qt + row;
      rr.ts = a.rab_ts + cur.b.s0;
      rr.last = cur.b.n - 1;
      if constexpr (TGT) {
        rr.hist = cur.b.hist;
        rr.pe_i = i < cur.b.hist ? i : cur.b.hist;
      } else {
        rr.pe_i = i;
      }
      rr.ts_i = __ldg(rr.ts + (i < rr.last ? i : rr.last));
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int jk = kbase + 32 * c + lane;
        tsk[c] = __ldg(rr.ts + (jk < rr.last ? jk : rr.last));
      }
    }
    {
      const bool ok = wait_one(bar(C::B_SFULL + j), (cur.tc / P) & 1u, w, kSiteSFull);
      if (!__all_sync(0xffffffffu, ok)) return;
    }
    tc_fence_after();
    trace(a, kEvSiluStart, cur.tc);
    const uint32_t t_s = lane_base + (uint32_t)(j * 128);
    bool plain = cur.kt != cur.b.qt;
    if constexpr (TGT) plain = cur.b.unmasked(cur.kt);
    // the 32-key chunks this warp takes: its half of the block when wide
    const int c0 = WIDE ? 2 * half : 0, c1 = WIDE ? 2 * half + 2 : 4;
    if constexpr (WIDE && !RAB) {
      // this warpgroup's four 16-key steps k = 4 half + u of the block
      if (quarter * 32 < cur.b.rows()) {
        uint32_t w0[16], w1[16];
        if (plain) {
          const uint32_t t_h = t_s + 64u * (uint32_t)half;
          tmem_ld16_async(t_h, w0);
          tmem_wait_ld16(w0);
#pragma unroll 1
          for (int u = 0; u < 4; u += 2) {
            tmem_ld16_async(t_h + 16u * (u + 1), w1);
            silu_store16<0>(w0, ha2, 0, 0, t_h + 16u * u);
            tmem_wait_ld16(w1);
            if (u + 2 < 4) tmem_ld16_async(t_h + 16u * (u + 2), w0);
            silu_store16<0>(w1, ha2, 0, 0, t_h + 16u * (u + 1));
            if (u + 2 < 4) tmem_wait_ld16(w0);
          }
        } else {
          // a masked block, as in the two-warpgroup path below, in 16-key
          // steps: steps wholly above the diagonal for this warp are zeros,
          // steps at or past cols are not read by the PV products
          const int cols = cur.b.cols(cur.kt);
          const bool diag = cur.kt == cur.b.qt;
          const int lim0 = kBM * cur.b.qt + row - kBN * cur.kt;
          int hist0 = 0;
          if constexpr (TGT) hist0 = cur.b.hist - kBN * cur.kt;
#pragma unroll 1
          for (int u = 0; u < 4; ++u) {
            const int k = 4 * half + u;
            if (16 * k >= cols) break;
            const uint32_t t_k = t_s + 16u * (uint32_t)k;
            if (diag && (k >> 1) > quarter) {
#pragma unroll
              for (int m = 0; m < 16; ++m) w0[m] = 0u;
              tmem_st16(t_k, w0);
            } else {
              tmem_ld16_async(t_k, w0);
              tmem_wait_ld16(w0);
              silu_store16<TGT ? 2 : 1>(w0, ha2, lim0 - 16 * k, hist0 - 16 * k, t_k);
            }
          }
        }
        tmem_wait_st();
      }
    } else if (RAB && plain && quarter * 32 < cur.b.rows()) {
      // one score buffer: the bias computation needs the registers
#pragma unroll 1
      for (int c = c0; c < c1; ++c) {
        tmem_ld32(t_s + 32u * c, s1);
        const int tsl = c == 0 ? tsk[0] : c == 1 ? tsk[1] : c == 2 ? tsk[2] : tsk[3];
        silu_store32<0, RAB, TGT, WIDE>(s1, ha2, 0, 0, t_s + 32u * c, &rr, kbase + 32 * c, tsl);
      }
      tmem_wait_st();
    } else if (plain && quarter * 32 < cur.b.rows()) {  // (without the bias)
      tmem_ld32_async(t_s, s0);
      tmem_wait_ld(s0);
#pragma unroll 1
      for (int c = 0; c < 4; c += 2) {
        tmem_ld32_async(t_s + 32u * (c + 1), s1);
        silu_store32<0>(s0, ha2, 0, 0, t_s + 32u * c);
        tmem_wait_ld(s1);
        if (c + 2 < 4) tmem_ld32_async(t_s + 32u * (c + 2), s0);
        silu_store32<0>(s1, ha2, 0, 0, t_s + 32u * (c + 1));
        if (c + 2 < 4) tmem_wait_ld(s0);
      }
      tmem_wait_st();
    } else if (quarter * 32 < cur.b.rows()) {
      // masked block: the diagonal one (keep keys j <= row), or one that
      // reaches past the history (keys of candidates are seen by their own
      // row only).  On the diagonal block, chunks c > quarter lie wholly
      // above the diagonal for this warp (zeros); columns >= cols are not
      // read by the PV products.
      const int cols = cur.b.cols(cur.kt);
      const bool diag = cur.kt == cur.b.qt;
      // row and history end relative to the block's first key
      const int lim0 = kBM * cur.b.qt + row - kBN * cur.kt;
      int hist0 = 0;
      if constexpr (TGT) hist0 = cur.b.hist - kBN * cur.kt;
#pragma unroll 1
      for (int c = c0; c < c1 && 32 * c < cols; ++c) {
        if (diag && c > quarter) {
          uint32_t z[16];
#pragma unroll
          for (int m = 0; m < 16; ++m) z[m] = 0u;
          tmem_st16(t_s + 32u * c, z);
          tmem_st16(t_s + 32u * c + 16u, z);
        } else {
          tmem_ld32(t_s + 32u * c, s1);
          const int tsl = c == 0 ? tsk[0] : c == 1 ? tsk[1] : c == 2 ? tsk[2] : tsk[3];
          silu_store32<TGT ? 2 : 1, RAB, TGT, WIDE>(s1, ha2, lim0 - 32 * c, hist0 - 32 * c,
                                                    t_s + 32u * c, &rr, kbase + 32 * c, tsl);
        }
      }
      tmem_wait_st();
    }
    tc_fence_before();
    trace(a, kEvSiluEnd, cur.tc);
    mbar_arrive(bar(C::B_PFULL + j));
    cur.advance(a);
  }
}

// Epilogue warpgroup (warps 0-3): O -> x inv_n -> bf16 -> out.  Thread r
// owns output row r of the item; rows past the sequence end are not stored.
// ------------------------------------------------ output stage Norm(O) (.) U
// HSTU paper section 3: the layer's pointwise transformation takes
// Norm(A(X) V(X)) (.) U(X), where Norm is a layer norm (section 3.1 requires
// it right after the pointwise pooling) over the token's outputs of all
// heads, with affine gamma and beta, and U already went through the SiLU
// of the first sub-layer.
//
// The heads of a token are separate items, on any CTAs, so the norm is
// split in two.  Here, in the attention epilogue, each row of each head
// leaves its fp32 values x = O inv_n in xs (total, heads * d) and their
// mean and M2 in stats (total, heads).  A second, bandwidth-bound kernel on
// the same stream (norm_gate_kernel below) merges the heads' moments and
// writes y.  Nothing waits on another CTA.
struct RowStats {
  float n, mean, m2;
};

// Fold 32 values of a row into (n, mean, m2): Chan, Golub and LeVeque's
// pairwise update with the chunk's own mean and M2.
__device__ __forceinline__ void stats_add32(RowStats& st, const float (&x)[32]) {
  float sum = 0.f;
#pragma unroll
  for (int m = 0; m < 32; ++m) sum += x[m];
  const float cmean = sum * (1.f / 32.f);
  float cm2 = 0.f;
#pragma unroll
  for (int m = 0; m < 32; ++m) {
    const float e = x[m] - cmean;
    cm2 = fmaf(e, e, cm2);
  }
  const float n1 = st.n + 32.f;
  const float delta = cmean - st.mean;
  const float wgt = 32.f / n1;
  st.mean = fmaf(delta, wgt, st.mean);
  st.m2 += cm2 + delta * delta * st.n * wgt;
  st.n = n1;
}

// One head of one item for the warp's 32 rows (lane = row): x and the
// row's moments out, then the O buffer released.
template <int D, int VAR>
__device__ __forceinline__ void norm_item(const FwdArgs& a, const BlockOf<has_targets<VAR>>& b,
                                          uint32_t o_t, uint32_t oempty, int quarter, int lane) {
  const int live = b.rows() - 32 * quarter;  // rows of the warp's quarter that exist (may be <= 0)
  const size_t t = (size_t)b.s0 + kBM * b.qt + 32 * quarter + lane;
  float* xrow = a.xs + t * (size_t)(a.heads * D) + (size_t)b.h * D;
  RowStats st{0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(o_t + 32u * c, o);
    float x[32];
#pragma unroll
    for (int m = 0; m < 32; ++m) x[m] = __uint_as_float(o[m]) * a.inv_n;
    stats_add32(st, x);
    if (lane < live) {
      float4* dst = reinterpret_cast<float4*>(xrow + 32 * c);
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(oempty);
  if (lane < live) a.stats[t * (size_t)a.heads + b.h] = make_float2(st.mean, st.m2);
}

template <int D, int VAR>
__device__ void role_epilogue(const FwdArgs& a, uint32_t base, uint32_t tmem, const WaitCtx& w,
                              int warp, int lane) {
  using C = Cfg<D>;
  constexpr bool TGT = has_targets<VAR>;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
  const float inv_n = a.inv_n;
  uint16_t* out = static_cast<uint16_t*>(a.out);
  constexpr bool norm = has_norm<VAR>;
  BlockOf<TGT> b;
  for (int it = 0; load_block<VAR>(a, it, b); ++it) {
    const int ob = it % C::OB;
    if (!wait_warp(bar(C::B_OFULL + ob), (uint32_t)(it / C::OB) & 1u, w, kSiteOFull)) return;
    tc_fence_after();
    trace(a, kEvEpiStart, (unsigned)it);
    const uint32_t o_t = tmem + lane_off + C::O_COL + (uint32_t)(ob * D);
    if constexpr (norm) {
      norm_item<D, VAR>(a, b, o_t, bar(C::B_OEMPTY + ob), quarter, lane);
      trace(a, kEvEpiEnd, (unsigned)it);
      continue;
    }
    uint4* dst = reinterpret_cast<uint4*>(
        out + ((size_t)(b.s0 + kBM * b.qt + row) * (size_t)a.heads + (size_t)b.h) * D);
    const bool live = row < b.rows();
    // The whole row is read, scaled and packed first, so that the O buffer
    // is released before the stores (the PV issuer waits on it at the next
    // item but one).
    uint32_t packed[D / 2];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(o_t + 32u * c, o);
#pragma unroll
      for (int m = 0; m < 16; ++m)
        packed[16 * c + m] =
            pack_bf16x2(__uint_as_float(o[2 * m]) * inv_n, __uint_as_float(o[2 * m + 1]) * inv_n);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(C::B_OEMPTY + ob));
    if (live) {
#pragma unroll
      for (int u = 0; u < D / 8; ++u)
        dst[u] = make_uint4(packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
    }
    trace(a, kEvEpiEnd, (unsigned)it);
  }
}

template <int D, int VAR>
__global__ void __launch_bounds__(kFwdThreadsOf<D, VAR>, 1)
    hstu_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars = base + C::BAR_OFF;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBARS; ++i) mbar_init(bars + 8u * i, C::arrivals(i, kWideSilu<D, VAR>));
    // QK-ready phase 0 has no PV before it: arrive for it now
    for (int j = 0; j < C::P; ++j) mbar_arrive(bars + 8u * (C::B_QKREADY + j));
    *abort_flag = 0;
    for (int i = 0; i < kTraceWarps; ++i) trace_counters()[i] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (lane == 0 && (warp == kTmaWarpK || warp == kTmaWarpV)) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(warp == kTmaWarpK ? &tm_k : &tm_v))
                 : "memory");
    if (warp == kTmaWarpK)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
  }
  if (warp == kMmaWarpQK) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx w{a.timeout_ns, abort_flag};

  if (warp == kTmaWarpK) {
    if (lane == 0) role_producer<D, true, VAR>(&tm_k, &tm_q, a, base, w);
    __syncwarp();
  } else if (warp == kTmaWarpV) {
    if (lane == 0) role_producer<D, false, VAR>(&tm_v, &tm_q, a, base, w);
    __syncwarp();
  } else if (warp == kMmaWarpQK) {
    if (lane == 0) role_mma_qk<D, VAR>(a, base, tmem, w);
    __syncwarp();
  } else if (warp == kMmaWarpPV) {
    if (lane == 0) role_mma_pv<D, VAR>(a, base, tmem, w);
    __syncwarp();
  } else if (warp >= kEwWarp0 && warp < kEwWarp0 + (kWideSilu<D, VAR> ? 16 : 8)) {
    role_silu<D, VAR>(a, base, tmem, w, warp, lane);
  } else if (warp < kEpiWarp0 + 4) {
    role_epilogue<D, VAR>(a, base, tmem, w, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if ((a.debug_flags & kDebugTrace) && blockIdx.x == 0 && threadIdx.x < kTraceWarps)
    g_trace_n[threadIdx.x] = trace_counters()[threadIdx.x];
  if (warp == kMmaWarpQK) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// y = Norm(x) (.) u over all tokens, grid-stride over tiles of R
// consecutive tokens per warp, R = 128 / n4 when a row has n4 <= 128
// 4-column chunks (so that every lane issues kLoads loads per round), else 1.
// The heads' moments merge with equal counts d: mean = mean of the means,
// M2 = sum of (M2_h + d (mean_h - mean)^2); lane r < R merges token r's and
// hands them out by shuffle.  Consecutive lanes take consecutive chunks of
// the tile's contiguous rows, so every access coalesces.
constexpr int kNormThreads = 256;
constexpr int kLoads = 4;
__global__ void __launch_bounds__(kNormThreads) norm_gate_kernel(const FwdArgs a, int d,
                                                                 long long total) {
  const int lane = threadIdx.x & 31;
  const int heads = a.heads;
  const int n4 = heads * d / 4;  // chunks of a row: a multiple of 8
  const int rows = n4 <= 32 * kLoads ? 32 * kLoads / n4 : 1;  // tokens per tile
  const int span = rows * n4;    // chunks of a tile
  const long long tiles = (total + rows - 1) / rows;
  const long long nwarps = (long long)gridDim.x * (kNormThreads / 32);
  const float4* g4 = reinterpret_cast<const float4*>(a.gamma);
  const float4* b4 = reinterpret_cast<const float4*>(a.beta);
  for (long long tile = (long long)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5);
       tile < tiles; tile += nwarps) {
    const long long t0 = tile * rows;
    const int live = (int)(total - t0 < rows ? total - t0 : rows);  // tokens of the tile
    const int lim = live * n4;
    const float4* xs = reinterpret_cast<const float4*>(a.xs) + t0 * n4;
    const uint2* u = reinterpret_cast<const uint2*>(a.u) + t0 * n4;
    uint2* y = reinterpret_cast<uint2*>(a.out) + t0 * n4;
    // the moments of token t0 + lane (lanes < live)
    float mean = 0.f, rstd = 0.f;
    if (lane < live) {
      const float2* st = a.stats + (t0 + lane) * heads;
      float msum = 0.f;
      for (int h = 0; h < heads; ++h) msum += __ldg(st + h).x;
      mean = msum / (float)heads;
      float m2 = 0.f;
      for (int h = 0; h < heads; ++h) {
        const float2 v = __ldg(st + h);
        const float dm = v.x - mean;
        m2 += v.y + (float)d * dm * dm;
      }
      rstd = rsqrtf(m2 / (float)(heads * d) + a.eps);
    }
    for (int e0 = 0; e0 < span; e0 += 32 * kLoads) {
      float4 x[kLoads];
      uint2 uu[kLoads];
#pragma unroll
      for (int k = 0; k < kLoads; ++k) {
        const int e = e0 + 32 * k + lane;
        if (e < lim) {
          x[k] = __ldcs(xs + e);
          uu[k] = __ldcs(u + e);
        }
      }
#pragma unroll
      for (int k = 0; k < kLoads; ++k) {
        const int e = e0 + 32 * k + lane;
        const int r = e / n4;  // token of the tile (< rows <= 32)
        const int c = e - r * n4;
        const float mr = __shfl_sync(0xffffffffu, mean, r & 31);
        const float rr = __shfl_sync(0xffffffffu, rstd, r & 31);
        if (e < lim) {
          const float4 g = __ldg(g4 + c), bb = __ldg(b4 + c);
          const float y0 = fmaf((x[k].x - mr) * rr, g.x, bb.x) * bf16_lo(uu[k].x);
          const float y1 = fmaf((x[k].y - mr) * rr, g.y, bb.y) * bf16_hi(uu[k].x);
          const float y2 = fmaf((x[k].z - mr) * rr, g.z, bb.z) * bf16_lo(uu[k].y);
          const float y3 = fmaf((x[k].w - mr) * rr, g.w, bb.w) * bf16_hi(uu[k].y);
          y[e] = make_uint2(pack_bf16x2(y0, y1), pack_bf16x2(y2, y3));
        }
      }
    }
  }
}

template <int D, int VAR>
cudaError_t launch_dt(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const FwdArgs& a, int grid, cudaStream_t stream) {
  using C = Cfg<D>;
  cudaError_t e = cudaFuncSetAttribute(hstu_fwd_kernel<D, VAR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_LAUNCH);
  if (e != cudaSuccess) return e;
  hstu_fwd_kernel<D, VAR><<<grid, kFwdThreadsOf<D, VAR>, C::SMEM_LAUNCH, stream>>>(tq, tk, tv, a);
  if ((e = cudaGetLastError()) != cudaSuccess || !has_norm<VAR>) return e;
  norm_gate_kernel<<<a.norm_grid, kNormThreads, 0, stream>>>(a, D, a.total);
  return cudaGetLastError();
}

// The variant follows the arguments: a history array selects the candidate
// mask, a U pointer the output stage, a timestamp array the bias.
template <int D>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const FwdArgs& a, int grid, cudaStream_t stream) {
  switch ((a.item_hist ? kVarTargets : 0) | (a.u ? kVarNorm : 0) | (a.rab_ts ? kVarRab : 0)) {
    case 0: return launch_dt<D, 0>(tq, tk, tv, a, grid, stream);
    case 1: return launch_dt<D, 1>(tq, tk, tv, a, grid, stream);
    case 2: return launch_dt<D, 2>(tq, tk, tv, a, grid, stream);
    case 3: return launch_dt<D, 3>(tq, tk, tv, a, grid, stream);
    case 4: return launch_dt<D, 4>(tq, tk, tv, a, grid, stream);
    case 5: return launch_dt<D, 5>(tq, tk, tv, a, grid, stream);
    case 6: return launch_dt<D, 6>(tq, tk, tv, a, grid, stream);
    default: return launch_dt<D, 7>(tq, tk, tv, a, grid, stream);
  }
}

#include "hstu_bwd.cuh"
#include "hstu_bwd_t.cuh"
#include "hstu_fwd_pair.cuh"

}  // namespace

int fwd_pair_smem_bytes(int d) {
  switch (d) {
    case 64: return PCfg<64>::SMEM_LAUNCH;
    case 128: return PCfg<128>::SMEM_LAUNCH;
    default: return -1;
  }
}

cudaError_t launch_fwd_pairs(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdArgs& a, int grid, cudaStream_t stream) {
  switch (d) {
    case 64: return launch_pair_d<64>(tq, tk, tv, a, grid, stream);
    case 128: return launch_pair_d<128>(tq, tk, tv, a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int fwd_smem_bytes(int d) {
  switch (d) {
    case 32: return Cfg<32>::SMEM_LAUNCH;
    case 64: return Cfg<64>::SMEM_LAUNCH;
    case 128: return Cfg<128>::SMEM_LAUNCH;
    default: return -1;
  }
}

int fwd_swizzle_bytes(int d) { return d >= 64 ? 128 : 64; }

int fwd_block_threads(int d, bool rab) {
  switch (d) {
    case 32: return rab ? kFwdThreadsOf<32, kVarRab> : kFwdThreadsOf<32, 0>;
    case 64: return rab ? kFwdThreadsOf<64, kVarRab> : kFwdThreadsOf<64, 0>;
    case 128: return rab ? kFwdThreadsOf<128, kVarRab> : kFwdThreadsOf<128, 0>;
    default: return -1;
  }
}

cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                       cudaStream_t stream) {
  switch (d) {
    case 32: return launch_bwd_d<32>(tq, tk, tv, tdo, tdq, a, grid, stream);
    case 64: return launch_bwd_d<64>(tq, tk, tv, tdo, tdq, a, grid, stream);
    case 128: return launch_bwd_d<128>(tq, tk, tv, tdo, tdq, a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, int grid, cudaStream_t stream) {
  switch (d) {
    case 32: return launch_d<32>(tq, tk, tv, a, grid, stream);
    case 64: return launch_d<64>(tq, tk, tv, a, grid, stream);
    case 128: return launch_d<128>(tq, tk, tv, a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t read_and_clear_trace(unsigned long long* dst, int capacity, int* n) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  unsigned cnt[kTraceWarps];
  if ((e = cudaMemcpyFromSymbol(cnt, g_trace_n, sizeof(cnt))) != cudaSuccess) return e;
  static unsigned long long buf[kTraceWarps * kTracePerWarp * 2];
  if ((e = cudaMemcpyFromSymbol(buf, g_trace, sizeof(buf))) != cudaSuccess) return e;
  int k = 0;
  for (int wp = 0; wp < kTraceWarps; ++wp)
    for (unsigned i = 0; i < cnt[wp] && i < (unsigned)kTracePerWarp; ++i) {
      if (k < capacity && dst) {
        dst[2 * k] = buf[2 * ((size_t)wp * kTracePerWarp + i)];
        dst[2 * k + 1] = buf[2 * ((size_t)wp * kTracePerWarp + i) + 1];
      }
      ++k;
    }
  *n = k < capacity ? k : capacity;
  const unsigned zero[kTraceWarps] = {};
  return cudaMemcpyToSymbol(g_trace_n, zero, sizeof(zero));
}

cudaError_t read_and_clear_device_status(unsigned* status, unsigned* site) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(status, g_dev_status, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(site, g_dev_site, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_dev_status, &zero, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_dev_site, &zero, sizeof(unsigned));
}

}  // namespace hstu
