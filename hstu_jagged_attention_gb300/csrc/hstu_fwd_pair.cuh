// HSTU jagged causal attention forward on CTA pairs (sm_103a, 2-CTA clusters).
// Included by hstu_fwd.cu inside its anonymous namespace: it uses that
// file's PTX helpers, barrier waits, trace and work-item types.
//
// The plain causal forward at d = 64 and 128 spends most of its time
// issuing tensor products: a 128 x 128 block takes 4 QK and 16 PV (P_hi,
// P_lo) products, and one thread issuing them with their barrier tests and
// commits leaves the tensor pipe idle much of the time.  A tcgen05.mma with
// cta_group::2 runs M = 256 rows over the two SMs of a cluster in the same
// cycles per instruction as an M = 128 product on one SM (measured on
// GB300: 44.6 cycles for N = 64 from TMEM, 64 for N = 128), so one issuing
// thread covers both SMs' blocks and the issue overhead per block halves.
//
// A pair item is 256 query rows of one (sequence, head): CTA r of the
// cluster owns query block qt_r = 2 qp + r.  The pair walks key blocks
// 0 .. kmax together (kmax = the last block holding keys of the pair's last
// valid row); CTA 0 sees key block 2 qp + 1 above its diagonal (all masked,
// P = 0).  Operands of a product are split between the two CTAs' shared
// memory and TMEM (checked element by element on GB300):
//   QK  S (256 x 128) = Q (256 x d) K^T: each CTA holds its own 128 query
//       rows of Q and 64 of the block's 128 keys (CTA r: keys 64 r ..); S
//       rows land in each CTA's own TMEM.
//   PV  O (256 x d) += P (256 x 128) V: P from each CTA's own TMEM, V split
//       by columns (CTA r: columns r d/2 .. of every key row).
// Roles (16 warps per CTA):
//   warp 4      K producer (both CTAs): the CTA's Q rows and its half of
//               each K block, with .cta_group::2 bulk copies whose bytes
//               count on CTA 0's barriers.
//   warp 6      V producer (both CTAs): the CTA's half of each V block.
//   warp 5      QK issuer (CTA 0 only; both CTAs' warp 5 allocate TMEM).
//   warp 7      PV issuer (CTA 0 only).
//   warps 8-15  SiLU warpgroups (both CTAs, alternate steps), as the
//               one-CTA kernel, each on its own 128 rows; they arrive on
//               CTA 0's P-full barrier (CTA 1 remotely).
//   warps 0-3   epilogue (both CTAs): the CTA's own O rows.
// Commits multicast to both CTAs' barriers (S-full, Q-empty, QK-ready,
// O-full); CTA 1's arrivals reach CTA 0 through cluster addresses.

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address in the cluster window of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Waits of CTA 0's issuers on barriers that CTA 1 also signals (its SiLU's
// and epilogue's arrivals, its copies' bytes): acquire at cluster scope, so
// that CTA 1's writes before its release are visible to the products.
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool wait_one_cl(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if ((it & 3u) == 0) {
      if (*w.abort_flag) return false;
      if (globaltimer() - t0 > w.limit_ns) {
        signal_timeout(w, site);
        return false;
      }
    }
  }
}

// Arrive on an mbarrier given by its cluster address (CTA 0's, from CTA 1).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}

// Bulk tensor copy into this CTA's shared memory whose completion counts on
// the barrier at cluster address `cbar` (CTA 0's).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t cbar, int x,
                                                 int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(cbar)
      : "memory");
}

template <int ACC>
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc) {
  if (ACC)
    asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, 1;" ::"r"(d_tmem), "l"(a), "l"(b),
                 "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, 0;" ::"r"(d_tmem), "l"(a), "l"(b),
                 "r"(idesc)
                 : "memory");
}

template <int ACC>
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc) {
  if (ACC)
    asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem), "r"(a_tmem),
                 "l"(b), "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, 0;" ::"r"(d_tmem), "r"(a_tmem),
                 "l"(b), "r"(idesc)
                 : "memory");
}

// Arrives on the barrier at the same offset in both CTAs once every product
// issued before it has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"((uint16_t)3)
      : "memory");
}

template <int D>
struct PCfg {
  static_assert(D == 64 || D == 128, "pair kernel: d = 64 or 128");
  static constexpr int NCHUNK = D / 64;       // 64-element (128-byte) swizzled chunks of a row
  static constexpr int QTILEB = kBM * D * 2;  // the CTA's 128 query rows
  static constexpr int QCHUNKB = kBM * 128;
  static constexpr int KHALF = kBN / 2;       // keys of a K block held by each CTA
  static constexpr int KTILEB = KHALF * D * 2;
  static constexpr int KCHUNKB = KHALF * 128;
  static constexpr int VCOLS = D / 2;         // value columns held by each CTA
  static constexpr int VROWB = VCOLS * 2;     // bytes of one key row of the CTA's V half: 64 or 128
  static constexpr int VTILEB = kBN * VROWB;
  static constexpr int VATOMB = 8 * VROWB;
  static constexpr uint64_t VLAYOUT = VROWB == 128 ? 2 : 4;  // 128B / 64B swizzle
  static constexpr uint64_t LAYOUT = 2;                      // Q and K: 128B swizzle
  static constexpr int P = 3;   // S buffers, K and V slots
  static constexpr int QS = 2;  // Q slots
  static constexpr int OB = 128 * P + 2 * D <= (int)kTmemCols ? 2 : 1;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + QS * QTILEB;
  static constexpr int V_OFF = K_OFF + P * KTILEB;
  static constexpr int BAR_OFF = V_OFF + P * VTILEB;
  static constexpr int B_QFULL = 0;               // CTA 0: both CTAs' Q rows landed
  static constexpr int B_QEMPTY = B_QFULL + QS;    // an item's last QK done (both CTAs)
  // QK-ready j: CTA 0: both K halves of step t landed and PV(t - P) done;
  // CTA 1: PV(t - P) done (its V slot j is free)
  static constexpr int B_QKREADY = B_QEMPTY + QS;
  static constexpr int B_VFULL = B_QKREADY + P;    // CTA 0: both V halves landed
  static constexpr int B_SFULL = B_VFULL + P;      // QK done (both CTAs)
  static constexpr int B_PFULL = B_SFULL + P;      // CTA 0: both CTAs' SiLU wrote P
  static constexpr int B_OFULL = B_PFULL + P;      // an item's last PV done (both CTAs)
  static constexpr int B_OEMPTY = B_OFULL + OB;    // CTA 0: both CTAs' epilogues released O
  static constexpr int B_DRAIN = B_OEMPTY + OB;    // [2]: CTA 0's issuers' drains
  static constexpr int NBARS = B_DRAIN + 2;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
  static constexpr int USED = MISC_OFF + 16;
  static constexpr int SMEM = ((USED + 1023) / 1024) * 1024 + 1024;
  static constexpr int SMEM_LAUNCH = SMEM < 120 * 1024 ? 120 * 1024 : SMEM;
  static constexpr uint32_t O_COL = 128u * P;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(128 * P + OB * D <= (int)kTmemCols, "TMEM budget");
  __host__ __device__ static constexpr uint32_t arrivals(int i, uint32_t rank) {
    return (i >= B_PFULL && i < B_PFULL + P)     ? 256u
           : (i >= B_OEMPTY && i < B_OEMPTY + OB) ? 8u
           : (i >= B_QKREADY && i < B_QKREADY + P) ? (rank == 0 ? 2u : 1u)
                                                  : 1u;
  }
};

// A pair item decoded: query blocks 2 qp and 2 qp + 1 of one (sequence, head).
struct PairBlock {
  int s0, n, h, qp;
  int kmax;  // the last key block the pair walks
  __device__ __forceinline__ int qt(uint32_t rank) const { return 2 * qp + (int)rank; }
  __device__ __forceinline__ int rows(uint32_t rank) const {  // valid query rows of CTA rank (0..128)
    const int r = n - kBM * qt(rank);
    return r < 0 ? 0 : (r < kBM ? r : kBM);
  }
  // Keys of key block kt that a valid row can see: 128, except the last
  // block when the sequence ends inside it (rounded up to the 16-key step).
  __device__ __forceinline__ int cols(int kt) const {
    if (kt != kmax) return kBN;
    const int r = n - kBN * kt;
    return r >= kBN ? kBN : ((r + 15) & ~15);
  }
};

__device__ __forceinline__ bool load_pair(const FwdArgs& a, int it, PairBlock& b) {
  const int clusters = (int)(gridDim.x >> 1);
  const int idx = item_index(it, (int)(blockIdx.x >> 1), clusters);
  if (idx >= a.n_items) return false;
  const Item x = __ldg(&a.items[idx]);
  b.s0 = x.x;
  b.n = x.y;
  b.h = x.z;
  b.qp = x.w;
  const int last = (b.n - 1) / kBN;
  b.kmax = 2 * b.qp + 1 < last ? 2 * b.qp + 1 : last;
  return true;
}

// A cursor over the pair's key-block steps (the next item fetched one item ahead).
struct PairCursor {
  int it, kt;
  uint32_t tc;
  PairBlock b, nb;
  bool valid, nvalid;
  __device__ __forceinline__ void start(const FwdArgs& a) {
    it = 0;
    kt = 0;
    tc = 0;
    valid = load_pair(a, 0, b);
    nvalid = valid && load_pair(a, 1, nb);
  }
  __device__ __forceinline__ void advance(const FwdArgs& a) {
    ++tc;
    if (++kt > b.kmax) {
      kt = 0;
      ++it;
      valid = nvalid;
      b = nb;
      nvalid = valid && load_pair(a, it + 1, nb);
    }
  }
};

// K producer (both CTAs): the CTA's Q rows of each item, then its half of
// each K block.  K slot t mod P is free once QK(t - P) has completed
// (S-full, multicast to both CTAs).  Byte counts land on CTA 0's barriers,
// whose expected totals CTA 0 sets for both halves.
template <int D>
__device__ void pair_producer_k(const CUtensorMap* tm_q, const CUtensorMap* tm_k, const FwdArgs& a,
                                uint32_t base, uint32_t rank, const WaitCtx& w) {
  using C = PCfg<D>;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  auto bar0 = [&](int i) { return cluster_addr(bar(i), 0); };
  uint32_t c = 0, qc = 0;
  bool ok = true;
  PairBlock b;
  for (int it = 0; ok && load_pair(a, it, b); ++it) {
    const int qs = (int)(qc % C::QS);
    if (!(ok = wait_one(bar(C::B_QEMPTY + qs), ((qc / C::QS) & 1u) ^ 1u, w, kSiteQEmpty))) break;
    if (rank == 0) mbar_arrive_expect_tx(bar(C::B_QFULL + qs), 2u * C::QTILEB);
#pragma unroll
    for (int ch = 0; ch < C::NCHUNK; ++ch)
      tma_load_3d_pair(base + C::Q_OFF + qs * C::QTILEB + ch * C::QCHUNKB, tm_q, bar0(C::B_QFULL + qs), 64 * ch,
                       b.h, b.s0 + kBM * b.qt(rank));
    ++qc;
    for (int kt = 0; kt <= b.kmax; ++kt) {
      const int slot = (int)(c % C::P);
      if (!(ok = wait_one(bar(C::B_SFULL + slot), ((c / C::P) & 1u) ^ 1u, w, kSiteKEmpty))) break;
      if (rank == 0) mbar_arrive_expect_tx(bar(C::B_QKREADY + slot), 2u * C::KTILEB);
#pragma unroll
      for (int ch = 0; ch < C::NCHUNK; ++ch)
        tma_load_3d_pair(base + C::K_OFF + slot * C::KTILEB + ch * C::KCHUNKB, tm_k, bar0(C::B_QKREADY + slot),
                         64 * ch, b.h, b.s0 + kBN * kt + C::KHALF * (int)rank);
      ++c;
    }
  }
}

// V producer (both CTAs): the CTA's half (columns rank d/2 ..) of each V
// block.  V slot t mod P is free once PV(t - P) has completed, which both
// CTAs' QK-ready barriers include (CTA 0's also counts K(t), which lands
// before PV(t) anyway).
template <int D>
__device__ void pair_producer_v(const CUtensorMap* tm_v, const FwdArgs& a, uint32_t base, uint32_t rank,
                                const WaitCtx& w) {
  using C = PCfg<D>;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  uint32_t c = 0;
  bool ok = true;
  PairBlock b;
  for (int it = 0; ok && load_pair(a, it, b); ++it) {
    for (int kt = 0; kt <= b.kmax; ++kt) {
      const int slot = (int)(c % C::P);
      if (!(ok = wait_one(bar(C::B_QKREADY + slot), (c / C::P) & 1u, w, kSiteVEmpty))) break;
      if (rank == 0) mbar_arrive_expect_tx(bar(C::B_VFULL + slot), 2u * C::VTILEB);
      tma_load_3d_pair(base + C::V_OFF + slot * C::VTILEB, tm_v, cluster_addr(bar(C::B_VFULL + slot), 0),
                       C::VCOLS * (int)rank, b.h, b.s0 + kBN * kt);
      ++c;
    }
  }
}

// QK issuer (CTA 0): S_j (256 x 128) = Q K^T of step t into S buffer
// j = t mod P of both CTAs, once both K halves have landed and PV(t - P)
// has completed (QK-ready).  Always N = 128: keys past the sequence are
// masked by the SiLU stage's select.
template <int D>
__device__ void pair_mma_qk(const FwdArgs& a, uint32_t base, uint32_t tmem, const WaitCtx& w) {
  using C = PCfg<D>;
  constexpr int P = C::P;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  constexpr uint32_t IDESC_QK = make_idesc(2 * kBM, kBN, 0);
  constexpr int QK_STEPS = D / 16;
  const uint64_t q_desc0 = smem_desc(base + C::Q_OFF, 16, 1024, C::LAYOUT);
  const uint64_t k_desc0 = smem_desc(base + C::K_OFF, 16, 1024, C::LAYOUT);
  bool ok = true;
  if (a.debug_flags & kDebugUnsignalledWait) ok = wait_one_cl(bar(C::B_DRAIN), 0u, w, kSiteUnsignalled);
  PairCursor qc;
  qc.start(a);
  uint32_t ph = 0;
  auto step = [&](auto jc) -> bool {
    constexpr int J = decltype(jc)::value;
    if (!ok || !qc.valid) return false;
    const int qs = qc.it & 1;
    if (qc.kt == 0 &&
        !(ok = wait_one_cl(bar(C::B_QFULL + qs), (uint32_t)(qc.it / C::QS) & 1u, w, kSiteQFull)))
      return false;
    if (!(ok = wait_one_cl(bar(C::B_QKREADY + J), ph, w, kSiteKFull))) return false;
    tc_fence_after();
    trace(a, kEvQkIssue, qc.tc);
    const uint32_t s_tmem = pin32(tmem + (uint32_t)(J * 128));
    const uint64_t qd0 = q_desc0 + (uint64_t)((qs * C::QTILEB) >> 4);
    uint64_t qd[QK_STEPS], kd[QK_STEPS];
#pragma unroll
    for (int kk = 0; kk < QK_STEPS; ++kk) {
      qd[kk] = pin64(qd0 + (uint64_t)(((kk / 4) * C::QCHUNKB + (kk % 4) * 32) >> 4));
      kd[kk] = pin64(k_desc0 + (uint64_t)((J * C::KTILEB + (kk / 4) * C::KCHUNKB + (kk % 4) * 32) >> 4));
    }
    mma_ss_pair<0>(s_tmem, qd[0], kd[0], IDESC_QK);
#pragma unroll
    for (int kk = 1; kk < QK_STEPS; ++kk) mma_ss_pair<1>(s_tmem, qd[kk], kd[kk], IDESC_QK);
    mma_commit_pair(bar(C::B_SFULL + J));
    if (qc.kt == qc.b.kmax) mma_commit_pair(bar(C::B_QEMPTY + qs));
    qc.advance(a);
    if (J == P - 1) ph ^= 1u;
    return true;
  };
  run_unrolled<P>(step);
  if (!ok) {
    mma_commit_pair(bar(C::B_DRAIN));
    wait_drain(bar(C::B_DRAIN), 0);
  }
}

// PV issuer (CTA 0): O += P_hi V + P_lo V (M = 256) into O buffer
// ob = item mod OB of both CTAs once both CTAs' SiLU warpgroups have written
// P (P-full) and both V halves have landed; then commits QK-ready (S buffer
// and V slot free) to both CTAs, and O-full after an item's last block.
// The barriers of the next step are tested (without blocking) before the
// current products are issued, so that the tests' latency overlaps them.
template <int D>
__device__ void pair_mma_pv(const FwdArgs& a, uint32_t base, uint32_t tmem, const WaitCtx& w) {
  using C = PCfg<D>;
  constexpr int P = C::P;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  constexpr uint32_t IDESC_PV = make_idesc(2 * kBM, D, 1);
  const uint64_t v_desc0 = smem_desc(base + C::V_OFF, C::VTILEB, C::VATOMB, C::VLAYOUT);
  bool ok = true;
  PairCursor pc;
  pc.start(a);
  uint32_t ph = 0;
  bool pa_ready = false, v_ready = false;  // tests made for the coming step
  auto step = [&](auto ic) -> bool {
    constexpr int J = decltype(ic)::value;
    constexpr int JN = (J + 1) % P;
    if (!ok || !pc.valid) return false;
    const int ob = C::OB == 1 ? 0 : (pc.it & 1);
    const bool last = pc.kt == pc.b.kmax;
    if (!pa_ready && !(ok = wait_one_cl(bar(C::B_PFULL + J), ph, w, kSitePFull))) return false;
    if (pc.kt == 0 &&
        !(ok = wait_one_cl(bar(C::B_OEMPTY + ob), ((uint32_t)(pc.it / C::OB) & 1u) ^ 1u, w, kSiteOEmpty)))
      return false;
    if (!v_ready && !(ok = wait_one_cl(bar(C::B_VFULL + J), ph, w, kSiteVFull))) return false;
    const int cols = pc.b.cols(pc.kt);
    if (last) {
      // Keys in [n, cols) lie past the end of the sequence: zero their V
      // rows in both CTAs' halves so that the zero P entries never meet
      // non-finite values of the next sequence.
      const int r_end = pc.b.n - kBN * pc.kt;
      if (r_end < cols) {
        const uint32_t z0 = base + C::V_OFF + J * C::VTILEB + r_end * C::VROWB;
        const uint32_t z1 = base + C::V_OFF + J * C::VTILEB + cols * C::VROWB;
        const uint32_t peer = cluster_addr(z0, 1) - z0;
        for (uint32_t z = z0; z < z1; z += 16) {
          asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(z), "r"(0) : "memory");
          asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(z + peer), "r"(0) : "memory");
        }
        asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
      }
    }
    tc_fence_after();
    trace(a, kEvPvIssue, pc.tc);
    const uint32_t npar = J + 1 == P ? ph ^ 1u : ph;
    pa_ready = mbar_test_cl(bar(C::B_PFULL + JN), npar);
    v_ready = mbar_test_cl(bar(C::B_VFULL + JN), npar);
    const uint32_t o_tmem = pin32(tmem + C::O_COL + (uint32_t)(ob * D));
    uint32_t pa[16];
    uint64_t vb[8];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      pa[2 * kk] = pin32(tmem + (uint32_t)(J * 128 + 32 * (kk >> 1) + 8 * (kk & 1)));
      pa[2 * kk + 1] = pin32(tmem + (uint32_t)(J * 128 + 32 * (kk >> 1) + 8 * (kk & 1) + 16));
      vb[kk] = pin64(v_desc0 + (uint64_t)((J * C::VTILEB + kk * 2 * C::VATOMB) >> 4));
    }
    if (cols == kBN && pc.kt != 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        mma_ts_pair<1>(o_tmem, pa[2 * kk], vb[kk], IDESC_PV);
        mma_ts_pair<1>(o_tmem, pa[2 * kk + 1], vb[kk], IDESC_PV);
      }
    } else {
      // an item's first block (its first product overwrites O) or the
      // sequence's last block (only the 16-key steps holding keys < n)
      const int n_steps = cols / 16;
      const bool first = pc.kt == 0;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        if (kk < n_steps) {
          if (kk == 0 && first)
            mma_ts_pair<0>(o_tmem, pa[0], vb[0], IDESC_PV);
          else
            mma_ts_pair<1>(o_tmem, pa[2 * kk], vb[kk], IDESC_PV);
          mma_ts_pair<1>(o_tmem, pa[2 * kk + 1], vb[kk], IDESC_PV);
        }
      }
    }
    mma_commit_pair(bar(C::B_QKREADY + J));  // PV(t) done: S buffer J and V slot J free
    if (last) mma_commit_pair(bar(C::B_OFULL + ob));
    pc.advance(a);
    if (J == P - 1) ph ^= 1u;
    return true;
  };
  run_unrolled<P>(step);
  if (!ok) {
    mma_commit_pair(bar(C::B_DRAIN + 1));
    wait_drain(bar(C::B_DRAIN + 1), 0);
  }
}

// SiLU warpgroups (both CTAs, warps 8-11 and 12-15, alternate steps): the
// CTA's 128 rows of S; then an arrival on CTA 0's P-full.  The CTA's rows
// belong to query block qt = 2 qp + rank: key blocks below it are
// unmasked, its diagonal block is triangular, and a block above it (CTA 0
// at kt = 2 qp + 1) is all masked (P = 0).  Rows past the sequence are not
// written (their outputs are never stored).
template <int D>
__device__ void pair_silu(const FwdArgs& a, uint32_t base, uint32_t tmem, uint32_t rank, const WaitCtx& w,
                          int warp, int lane) {
  using C = PCfg<D>;
  constexpr int P = C::P;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  const int e = (warp - kEwWarp0) >> 2;
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
  const float2 ha2 = make_float2(a.half_alpha, a.half_alpha);
  PairCursor cur;
  cur.start(a);
  uint32_t s0[32], s1[32];
  while (cur.valid) {
    if ((int)(cur.tc & 1u) != e) {
      cur.advance(a);
      continue;
    }
    const int j = (int)(cur.tc % P);
    {
      const bool ok = wait_one(bar(C::B_SFULL + j), (cur.tc / P) & 1u, w, kSiteSFull);
      if (!__all_sync(0xffffffffu, ok)) return;
    }
    tc_fence_after();
    trace(a, kEvSiluStart, cur.tc);
    const uint32_t t_s = lane_base + (uint32_t)(j * 128);
    const int qt = cur.b.qt(rank);
    const bool live = quarter * 32 < cur.b.rows(rank);
    if (live && cur.kt < qt) {
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
    } else if (live) {
      // the diagonal block (keep keys j <= row; chunks c > quarter lie wholly
      // above the diagonal for this warp), or a block above it (all zero);
      // columns >= cols are not read by the PV products
      const int cols = cur.b.cols(cur.kt);
      const int lim0 = kBM * qt + row - kBN * cur.kt;
      const bool above = cur.kt > qt;
#pragma unroll 1
      for (int c = 0; c < 4 && 32 * c < cols; ++c) {
        if (above || c > quarter) {
          uint32_t z[16];
#pragma unroll
          for (int m = 0; m < 16; ++m) z[m] = 0u;
          tmem_st16(t_s + 32u * c, z);
          tmem_st16(t_s + 32u * c + 16u, z);
        } else {
          tmem_ld32(t_s + 32u * c, s1);
          silu_store32<1>(s1, ha2, lim0 - 32 * c, 0, t_s + 32u * c);
        }
      }
      tmem_wait_st();
    }
    tc_fence_before();
    trace(a, kEvSiluEnd, cur.tc);
    if (rank == 0)
      mbar_arrive(bar(C::B_PFULL + j));
    else
      mbar_arrive_cluster(cluster_addr(bar(C::B_PFULL + j), 0));
    cur.advance(a);
  }
}

// Epilogue (both CTAs, warps 0-3): the CTA's O rows -> x inv_n -> bf16 ->
// out; then an arrival on CTA 0's O-empty.  The whole row is read and
// packed first, so that the O buffer is released before the stores.
template <int D>
__device__ void pair_epilogue(const FwdArgs& a, uint32_t base, uint32_t tmem, uint32_t rank, const WaitCtx& w,
                              int warp, int lane) {
  using C = PCfg<D>;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  const int quarter = warp & 3;
  const int row = quarter * 32 + lane;
  const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
  const float inv_n = a.inv_n;
  uint16_t* out = static_cast<uint16_t*>(a.out);
  PairBlock b;
  for (int it = 0; load_pair(a, it, b); ++it) {
    const int ob = it % C::OB;
    if (!wait_warp(bar(C::B_OFULL + ob), (uint32_t)(it / C::OB) & 1u, w, kSiteOFull)) return;
    tc_fence_after();
    trace(a, kEvEpiStart, (unsigned)it);
    const uint32_t o_t = tmem + lane_off + C::O_COL + (uint32_t)(ob * D);
    uint32_t packed[D / 2];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(o_t + 32u * c, o);
#pragma unroll
      for (int m = 0; m < 16; ++m)
        packed[16 * c + m] = pack_bf16x2(__uint_as_float(o[2 * m]) * inv_n, __uint_as_float(o[2 * m + 1]) * inv_n);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (rank == 0)
        mbar_arrive(bar(C::B_OEMPTY + ob));
      else
        mbar_arrive_cluster(cluster_addr(bar(C::B_OEMPTY + ob), 0));
    }
    if (row < b.rows(rank)) {
      uint4* dst = reinterpret_cast<uint4*>(
          out + ((size_t)(b.s0 + kBM * b.qt(rank) + row) * (size_t)a.heads + (size_t)b.h) * D);
#pragma unroll
      for (int u = 0; u < D / 8; ++u)
        dst[u] = make_uint4(packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
    }
    trace(a, kEvEpiEnd, (unsigned)it);
  }
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    hstu_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using C = PCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars = base + C::BAR_OFF;
  const uint32_t rank = cluster_rank();

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBARS; ++i) mbar_init(bars + 8u * i, C::arrivals(i, rank));
    // QK-ready phase 0 has no PV before it: its PV arrival now (CTA 1's only one)
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
    // one allocation of 512 columns at the same address in both CTAs
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx w{a.timeout_ns, abort_flag};

  if (warp == kTmaWarpK) {
    if (lane == 0) pair_producer_k<D>(&tm_q, &tm_k, a, base, rank, w);
    __syncwarp();
  } else if (warp == kTmaWarpV) {
    if (lane == 0) pair_producer_v<D>(&tm_v, a, base, rank, w);
    __syncwarp();
  } else if (warp == kMmaWarpQK) {
    if (rank == 0 && lane == 0) pair_mma_qk<D>(a, base, tmem, w);
    __syncwarp();
  } else if (warp == kMmaWarpPV) {
    if (rank == 0 && lane == 0) pair_mma_pv<D>(a, base, tmem, w);
    __syncwarp();
  } else if (warp >= kEwWarp0 && warp < kEwWarp0 + 8) {
    pair_silu<D>(a, base, tmem, rank, w, warp, lane);
  } else if (warp < kEpiWarp0 + 4) {
    pair_epilogue<D>(a, base, tmem, rank, w, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while the other's products may read its memory
  if ((a.debug_flags & kDebugTrace) && blockIdx.x == 0 && threadIdx.x < kTraceWarps)
    g_trace_n[threadIdx.x] = trace_counters()[threadIdx.x];
  if (warp == kMmaWarpQK) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}

template <int D>
cudaError_t launch_pair_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdArgs& a, int grid, cudaStream_t stream) {
  using C = PCfg<D>;
  cudaError_t e =
      cudaFuncSetAttribute(hstu_fwd_pair_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_LAUNCH);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kFwdThreads);
  cfg.dynamicSmemBytes = C::SMEM_LAUNCH;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, hstu_fwd_pair_kernel<D>, tq, tk, tv, a);
}
