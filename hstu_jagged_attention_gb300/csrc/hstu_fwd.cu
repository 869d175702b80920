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
// Design (one persistent CTA per SM, 16 warps, warp-specialised):
//   warp 4        TMA producer: Q block of the work item, then K and V blocks
//                 kt = 0..qt into shared-memory rings (128B-swizzled tiles).
//   warp 5        MMA issuer (one thread): S = Q K^T into a TMEM buffer
//                 (tcgen05.mma kind::f16, fp32 accumulate), then
//                 O += P_hi V + P_lo V with P read from TMEM.  Owns TMEM.
//   warps 8-15    two "SiLU" warpgroups; warpgroup e handles the blocks whose
//                 running index is e mod 2, i.e. S buffer e.  Thread r owns
//                 score row r: tcgen05.ld S, p = h + h tanh(h) with
//                 h = alpha s / 2 (= alpha s sigmoid(alpha s)), tril select on
//                 the diagonal block, split p = bf16(p) + bf16(p - bf16(p)),
//                 tcgen05.st both halves over the S columns just read.
//   warps 0-3     epilogue: reads the finished O buffer (double-buffered in
//                 TMEM), scales by inv_n, rounds to bf16 and stores the valid
//                 rows with 16-byte stores.
// The three roles overlap the way the post's three-stage pipeline does
// (section 5.2): QK of block t+1 runs on the tensor cores while the SiLU
// warps work on block t and PV of block t-1 drains.
//
// TMEM columns (512 allocated): S0 [0,128), S1 [128,256), O0 [256,256+d),
// O1 [256+d, 256+2d).  P of a block overwrites its own S buffer: for the
// 32-key chunk c, P_hi keys pairs go to columns 32c+[0,16) and P_lo to
// 32c+[16,32) (two bf16 per 32-bit column).
//
// Every mbarrier wait is bounded by a %globaltimer limit.  A wait that runs
// out records a status word, raises a CTA-wide abort flag that every other
// wait checks, and the CTA drains its own TMA copies and MMAs, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hstu_internal.h"

namespace hstu {

__device__ unsigned int g_dev_status;
__device__ unsigned int g_dev_site;

namespace {

constexpr int kBM = 128;  // query rows per item == TMEM lanes
constexpr int kBN = 128;  // keys per K/V block
constexpr int kEpiWarp0 = 0;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kEwWarp0 = 8;
constexpr uint32_t kTmemCols = 512;

// wait-site codes reported through g_dev_site
enum : int {
  kSiteQEmpty = 1, kSiteKEmpty, kSiteVEmpty, kSiteQFull, kSiteKFull, kSitePFull, kSiteOEmpty,
  kSiteVFull, kSiteSFull, kSiteOFull, kSiteUnsignalled
};

template <int D>
struct Cfg {
  static constexpr int CHUNK = D < 64 ? D : 64;  // elements per swizzled row
  static constexpr int NCHUNK = D / CHUNK;
  static constexpr int ROWB = CHUNK * 2;          // bytes per swizzled row: 128 or 64
  static constexpr int ATOMB = 8 * ROWB;          // 8-row swizzle atom
  static constexpr int CHUNKB = kBM * ROWB;       // 128 rows of one chunk
  static constexpr int TILEB = kBM * D * 2;       // one 128 x D bf16 block
  static constexpr int QS = 2;
  static constexpr int KS = D == 128 ? 2 : 4;
  static constexpr int VS = D == 128 ? 3 : 4;
  static constexpr uint64_t LAYOUT = ROWB == 128 ? 2 : 4;  // descriptor layout: 128B / 64B swizzle
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + QS * TILEB;
  static constexpr int V_OFF = K_OFF + KS * TILEB;
  static constexpr int BAR_OFF = V_OFF + VS * TILEB;
  static constexpr int B_QFULL = 0;
  static constexpr int B_QEMPTY = B_QFULL + QS;
  static constexpr int B_KFULL = B_QEMPTY + QS;
  static constexpr int B_KEMPTY = B_KFULL + KS;
  static constexpr int B_VFULL = B_KEMPTY + KS;
  static constexpr int B_VEMPTY = B_VFULL + VS;
  static constexpr int B_SFULL = B_VEMPTY + VS;
  static constexpr int B_PFULL = B_SFULL + 2;
  static constexpr int B_OFULL = B_PFULL + 2;
  static constexpr int B_OEMPTY = B_OFULL + 2;
  static constexpr int B_DRAIN = B_OEMPTY + 2;
  static constexpr int NBARS = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag
  static constexpr int USED = MISC_OFF + 16;
  static constexpr int SMEM = ((USED + 1023) / 1024) * 1024 + 1024;  // + realignment slack
  // Ask for more than half an SM's shared memory so that exactly one CTA
  // (and one 512-column TMEM allocation) lives on each SM.
  static constexpr int SMEM_LAUNCH = SMEM < 120 * 1024 ? 120 * 1024 : SMEM;
  static constexpr uint32_t O_COL = 256;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(256 + 2 * D <= (int)kTmemCols, "TMEM budget");
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
__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort_flag) return false;
    if (globaltimer() - t0 > w.limit_ns) {
      signal_timeout(w, site);
      return false;
    }
  }
}

// Whole-warp bounded wait with a warp-uniform result.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
  const bool ok = wait_one(bar, parity, w, site);
  return __all_sync(0xffffffffu, ok);
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

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
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

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
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

__device__ __forceinline__ int item_index(int it, int cta, int grid) {
  // serpentine over the longest-first list: even rounds left to right, odd
  // rounds right to left, so that CTAs even out the cost of their items.
  const int base = it * grid;
  return (it & 1) ? base + (grid - 1 - cta) : base + cta;
}

// ------------------------------------------------------------------ roles
template <int D>
__device__ void role_producer(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              const FwdArgs& a, uint32_t base, const WaitCtx& w, int lane) {
  using C = Cfg<D>;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  uint32_t qc = 0, kc = 0, vc = 0;
  bool ok = true;
  for (int it = 0; ok; ++it) {
    const int idx = item_index(it, blockIdx.x, gridDim.x);
    if (idx >= a.n_items) break;
    const Item item = __ldg(&a.items[idx]);
    const int s0 = item.x, h = item.z, qt = item.w;
    const int qs = (int)(qc % C::QS);
    if (!(ok = wait_warp(bar(C::B_QEMPTY + qs), ((qc / C::QS) & 1u) ^ 1u, w, kSiteQEmpty))) break;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(C::B_QFULL + qs), C::TILEB);
#pragma unroll
      for (int ch = 0; ch < C::NCHUNK; ++ch)
        tma_load_3d(base + C::Q_OFF + qs * C::TILEB + ch * C::CHUNKB, tq, bar(C::B_QFULL + qs),
                    ch * C::CHUNK, h, s0 + kBM * qt);
    }
    __syncwarp();
    ++qc;
    for (int kt = 0; kt <= qt; ++kt) {
      const int ks = (int)(kc % C::KS);
      if (!(ok = wait_warp(bar(C::B_KEMPTY + ks), ((kc / C::KS) & 1u) ^ 1u, w, kSiteKEmpty))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::B_KFULL + ks), C::TILEB);
#pragma unroll
        for (int ch = 0; ch < C::NCHUNK; ++ch)
          tma_load_3d(base + C::K_OFF + ks * C::TILEB + ch * C::CHUNKB, tk, bar(C::B_KFULL + ks),
                      ch * C::CHUNK, h, s0 + kBN * kt);
      }
      __syncwarp();
      ++kc;
      const int vs = (int)(vc % C::VS);
      if (!(ok = wait_warp(bar(C::B_VEMPTY + vs), ((vc / C::VS) & 1u) ^ 1u, w, kSiteVEmpty))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(C::B_VFULL + vs), C::TILEB);
#pragma unroll
        for (int ch = 0; ch < C::NCHUNK; ++ch)
          tma_load_3d(base + C::V_OFF + vs * C::TILEB + ch * C::CHUNKB, tv, bar(C::B_VFULL + vs),
                      ch * C::CHUNK, h, s0 + kBN * kt);
      }
      __syncwarp();
      ++vc;
    }
  }
  if (!ok && lane == 0) {
    // Drain: wait for the last phase armed on every full barrier, so no
    // copy is still landing in shared memory when the CTA exits.
    auto drain = [&](int first, int slots, uint32_t count) {
      for (int s = 0; s < slots; ++s) {
        if (count > (uint32_t)s) {
          const uint32_t uses = (count - 1u - (uint32_t)s) / (uint32_t)slots + 1u;
          wait_drain(bar(first + s), (uses - 1u) & 1u);
        }
      }
    };
    drain(C::B_QFULL, C::QS, qc);
    drain(C::B_KFULL, C::KS, kc);
    drain(C::B_VFULL, C::VS, vc);
  }
}

template <int D>
__device__ void role_mma(const FwdArgs& a, uint32_t base, uint32_t tmem, const WaitCtx& w, int lane) {
  using C = Cfg<D>;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  constexpr uint32_t IDESC_QK = make_idesc(kBM, kBN, 0);
  constexpr uint32_t IDESC_PV = make_idesc(kBM, D, 1);
  uint32_t qc = 0, kc = 0, vc = 0, tc = 0;
  bool ok = true;
  // Test hook: wait on a barrier that nothing arrives on, so that the
  // bounded wait runs out and the whole CTA takes its give-up path.
  if (a.debug_flags & kDebugUnsignalledWait)
    ok = wait_warp(bar(C::B_DRAIN), 0u, w, kSiteUnsignalled);

  for (int it = 0; ok; ++it) {
    const int idx = item_index(it, blockIdx.x, gridDim.x);
    if (idx >= a.n_items) break;
    const Item item = __ldg(&a.items[idx]);
    const int n = item.y, qt = item.w;
    const int qs = (int)(qc % C::QS);
    const int ob = it & 1;
    const uint32_t o_tmem = tmem + C::O_COL + (uint32_t)(ob * D);
    if (!(ok = wait_warp(bar(C::B_QFULL + qs), (qc / C::QS) & 1u, w, kSiteQFull))) break;
    const uint32_t q_addr = base + C::Q_OFF + qs * C::TILEB;

    // PV of one block: waits for its P, for the O buffer (first block), for V.
    auto issue_pv = [&](uint32_t ptc, int pkt, uint32_t pvc) -> bool {
      const int pb = (int)(ptc & 1u);
      if (!wait_warp(bar(C::B_PFULL + pb), (ptc >> 1) & 1u, w, kSitePFull)) return false;
      if (pkt == 0 &&
          !wait_warp(bar(C::B_OEMPTY + ob), ((uint32_t)(it >> 1) & 1u) ^ 1u, w, kSiteOEmpty))
        return false;
      const int vs = (int)(pvc % C::VS);
      if (!wait_warp(bar(C::B_VFULL + vs), (pvc / C::VS) & 1u, w, kSiteVFull)) return false;
      const uint32_t v_addr = base + C::V_OFF + vs * C::TILEB;
      const int r_end = n - kBM * qt;
      if (pkt == qt && r_end < kBN) {
        // Keys past the end of the sequence: zero their V rows so that the
        // zero P entries never meet non-finite values of the next sequence.
        const int n16 = (kBN - r_end) * C::ROWB / 16;
#pragma unroll
        for (int ch = 0; ch < C::NCHUNK; ++ch) {
          const uint32_t z0 = v_addr + ch * C::CHUNKB + r_end * C::ROWB;
          for (int i = lane; i < n16; i += 32)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(z0 + 16 * i), "r"(0)
                         : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t p_tmem = tmem + (uint32_t)(pb * 128);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t bdesc =
              smem_desc(v_addr + kk * 2 * C::ATOMB, C::CHUNKB, C::ATOMB, C::LAYOUT);
          const uint32_t col = 32u * (kk >> 1) + 8u * (kk & 1);
          mma_ts(o_tmem, p_tmem + col, bdesc, IDESC_PV, (pkt > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t bdesc =
              smem_desc(v_addr + kk * 2 * C::ATOMB, C::CHUNKB, C::ATOMB, C::LAYOUT);
          const uint32_t col = 32u * (kk >> 1) + 16u + 8u * (kk & 1);
          mma_ts(o_tmem, p_tmem + col, bdesc, IDESC_PV, 1u);
        }
        mma_commit(bar(C::B_VEMPTY + vs));
      }
      __syncwarp();
      return true;
    };

    uint32_t prev_tc = 0, prev_vc = 0;
    int prev_kt = -1;
    for (int kt = 0; kt <= qt; ++kt) {
      const int ks = (int)(kc % C::KS);
      const int b = (int)(tc & 1u);
      if (!(ok = wait_warp(bar(C::B_KFULL + ks), (kc / C::KS) & 1u, w, kSiteKFull))) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t k_addr = base + C::K_OFF + ks * C::TILEB;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / (C::CHUNK / 16)) * C::CHUNKB + (kk % (C::CHUNK / 16)) * 32;
          const uint64_t adesc = smem_desc(q_addr + off, 16, C::ATOMB, C::LAYOUT);
          const uint64_t bdesc = smem_desc(k_addr + off, 16, C::ATOMB, C::LAYOUT);
          mma_ss(tmem + (uint32_t)(b * 128), adesc, bdesc, IDESC_QK, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::B_SFULL + b));
        mma_commit(bar(C::B_KEMPTY + ks));
        if (kt == qt) mma_commit(bar(C::B_QEMPTY + qs));
      }
      __syncwarp();
      ++kc;
      if (prev_kt >= 0 && !(ok = issue_pv(prev_tc, prev_kt, prev_vc))) break;
      prev_tc = tc;
      prev_kt = kt;
      prev_vc = vc;
      ++tc;
      ++vc;
    }
    if (!ok) break;
    ++qc;
    if (!(ok = issue_pv(prev_tc, prev_kt, prev_vc))) break;
    if (lane == 0) mma_commit(bar(C::B_OFULL + ob));
    __syncwarp();
  }
  if (!ok) {
    // Drain: a commit arrives once every MMA issued before it has finished.
    if (lane == 0) mma_commit(bar(C::B_DRAIN));
    __syncwarp();
    if (lane == 0) wait_drain(bar(C::B_DRAIN), 0);
    __syncwarp();
  }
}

template <int D>
__device__ void role_silu(const FwdArgs& a, uint32_t base, uint32_t tmem, const WaitCtx& w, int warp,
                          int lane) {
  using C = Cfg<D>;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  const int e = (warp - kEwWarp0) >> 2;  // which S buffer this warpgroup owns
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t t_s = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(e * 128);
  const float ha = a.half_alpha;
  uint32_t tc = 0, mine = 0;
  for (int it = 0;; ++it) {
    const int idx = item_index(it, blockIdx.x, gridDim.x);
    if (idx >= a.n_items) break;
    const int qt = __ldg(&a.items[idx].w);
    for (int kt = 0; kt <= qt; ++kt, ++tc) {
      if ((int)(tc & 1u) != e) continue;
      if (!wait_warp(bar(C::B_SFULL + e), mine & 1u, w, kSiteSFull)) return;
      tc_fence_after();
      const bool diag = kt == qt;
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t s[32];
        tmem_ld32(t_s + 32u * c, s);
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float h0 = __uint_as_float(s[2 * m]) * ha;
          const float h1 = __uint_as_float(s[2 * m + 1]) * ha;
          float p0 = fmaf(h0, tanh_approx(h0), h0);
          float p1 = fmaf(h1, tanh_approx(h1), h1);
          if (diag) {
            const int j = 32 * c + 2 * m;
            p0 = (j > row) ? 0.0f : p0;
            p1 = (j + 1 > row) ? 0.0f : p1;
          }
          const uint32_t ph = pack_bf16x2(p0, p1);
          const float r0 = p0 - __uint_as_float(ph << 16);
          const float r1 = p1 - __uint_as_float(ph & 0xFFFF0000u);
          hi[m] = ph;
          lo[m] = pack_bf16x2(r0, r1);
        }
        tmem_st16(t_s + 32u * c, hi);
        tmem_st16(t_s + 32u * c + 16u, lo);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::B_PFULL + e));
      ++mine;
    }
  }
}

template <int D>
__device__ void role_epilogue(const FwdArgs& a, uint32_t base, uint32_t tmem, const WaitCtx& w,
                              int warp, int lane) {
  using C = Cfg<D>;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
  const float inv_n = a.inv_n;
  uint16_t* out = static_cast<uint16_t*>(a.out);
  for (int it = 0;; ++it) {
    const int idx = item_index(it, blockIdx.x, gridDim.x);
    if (idx >= a.n_items) break;
    const Item item = __ldg(&a.items[idx]);
    const int s0 = item.x, n = item.y, h = item.z, qt = item.w;
    const int ob = it & 1;
    if (!wait_warp(bar(C::B_OFULL + ob), (uint32_t)(it >> 1) & 1u, w, kSiteOFull)) return;
    tc_fence_after();
    uint32_t packed[D / 2];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tmem + lane_off + C::O_COL + (uint32_t)(ob * D + 32 * c), o);
#pragma unroll
      for (int m = 0; m < 16; ++m)
        packed[16 * c + m] = pack_bf16x2(__uint_as_float(o[2 * m]) * inv_n,
                                         __uint_as_float(o[2 * m + 1]) * inv_n);
    }
    tc_fence_before();
    mbar_arrive(bar(C::B_OEMPTY + ob));
    const int r_valid = n - kBM * qt;
    if (row < r_valid) {
      uint4* dst = reinterpret_cast<uint4*>(
          out + ((size_t)(s0 + kBM * qt + row) * (size_t)a.heads + (size_t)h) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
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
    for (int i = 0; i < C::NBARS; ++i) {
      const bool many = (i == C::B_PFULL || i == C::B_PFULL + 1 || i == C::B_OEMPTY ||
                         i == C::B_OEMPTY + 1);
      mbar_init(bars + 8u * i, many ? 128u : 1u);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == kTmaWarp && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
  }
  if (warp == kMmaWarp) {
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

  if (warp == kTmaWarp) {
    role_producer<D>(&tm_q, &tm_k, &tm_v, a, base, w, lane);
  } else if (warp == kMmaWarp) {
    role_mma<D>(a, base, tmem, w, lane);
  } else if (warp >= kEwWarp0) {
    role_silu<D>(a, base, tmem, w, warp, lane);
  } else if (warp < kEpiWarp0 + 4) {
    role_epilogue<D>(a, base, tmem, w, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

template <int D>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const FwdArgs& a, int grid, cudaStream_t stream) {
  using C = Cfg<D>;
  static bool configured = false;  // per process; the attribute is per function
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(hstu_fwd_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_LAUNCH);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  hstu_fwd_kernel<D><<<grid, kFwdThreads, C::SMEM_LAUNCH, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

int fwd_smem_bytes(int d) {
  switch (d) {
    case 32: return Cfg<32>::SMEM_LAUNCH;
    case 64: return Cfg<64>::SMEM_LAUNCH;
    case 128: return Cfg<128>::SMEM_LAUNCH;
    default: return -1;
  }
}

int fwd_swizzle_bytes(int d) { return d >= 64 ? 128 : 64; }

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, int grid, cudaStream_t stream) {
  switch (d) {
    case 32: return launch_d<32>(tq, tk, tv, a, grid, stream);
    case 64: return launch_d<64>(tq, tk, tv, a, grid, stream);
    case 128: return launch_d<128>(tq, tk, tv, a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
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
