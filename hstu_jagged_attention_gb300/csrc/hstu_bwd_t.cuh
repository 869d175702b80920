// Backward pass in transposed form, for d <= 64 without the bias (HSTU
// paper Appendix G: the backward recomputes the attention and accumulates
// the gradients on chip).  The gradients are those of hstu_bwd.cuh; only
// the orientation of the recomputed scores differs.
//
// Work item, as in hstu_bwd.cuh: one 128-key block kt of one (sequence,
// head), walking the query blocks qt that see it.  Per query block:
//   1. S^T = K Q^T and dP^T = V dO^T into TMEM, so that the TMEM lanes are
//      the block's keys and the columns its queries.
//   2. Thread r (and r + 128, each taking half of the queries) owns key r:
//      P^T = inv_n silu(alpha S^T) and dS^T = inv_n silu'(alpha S^T) (.) dP^T,
//      each split into bf16 hi + lo, overwrite S^T and dP^T in TMEM (16
//      columns of hi and 16 of lo per 32 queries, the A-operand layout of
//      a product read from TMEM).  dS^T also goes to shared memory, rows =
//      keys, queries contiguous (128-byte swizzle).
//   3. dV += P^T dO and dK += dS^T Q read their A operand from TMEM; no
//      shared tile is written for them.
//   4. dQ_part = dS K reads the shared dS^T tile as an MN-major A operand
//      (M = queries); it runs while the threads work on the next block, and
//      alpha dQ_part goes into the fp32 accumulator by bulk tensor
//      reductions from a staging tile, as in hstu_bwd.cuh.
// Warp 8 (one thread) issues the copies and the products; warps 0-7 do the
// elementwise work, the dQ staging and the item's dV / dK stores.  Once a
// block's elementwise pass is done, its dV and dK products run, then the
// next block's S^T and dP^T (they overwrite the columns the products read,
// so they wait for them), then this block's dQ.
//
// The last key block of a sequence reaches into the next sequence (or past
// the tensor, read as zeros).  Its key rows past the end carry P = dS = 0,
// and the K tile's rows past the end are zeroed before dQ reads them, so
// that 0 x (an infinite key of the next sequence) cannot reach dQ; the
// last query block's Q and dO rows past the end are zeroed before dK and
// dV read them.

template <int D>
struct TCfg {
  static_assert(D == 32 || D == 64, "transposed backward: d = 32 or 64");
  static constexpr int CHUNK = D < 64 ? D : 64;  // elements per swizzled row of a d-wide tile
  static constexpr int NCHUNK = D / CHUNK;
  static constexpr int ROWB = CHUNK * 2;
  static constexpr int ATOMB = 8 * ROWB;
  static constexpr int CHUNKB = kBM * ROWB;
  static constexpr int TILEB = kBM * D * 2;
  static constexpr uint64_t LAYOUT = ROWB == 128 ? 2 : 4;  // 128B / 64B swizzle
  // dS^T: 128 keys x 128 queries bf16 as two 64-query chunks, 128B swizzle
  static constexpr int PCHUNKB = kBM * 128;
  static constexpr int PTILEB = 2 * PCHUNKB;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILEB;
  static constexpr int Q_OFF = V_OFF + TILEB;        // two buffers
  static constexpr int DO_OFF = Q_OFF + 2 * TILEB;   // two buffers
  static constexpr int DHI_OFF = DO_OFF + 2 * TILEB;
  static constexpr int DLO_OFF = DHI_OFF + PTILEB;
  // alpha dQ_part staging: D / 32 boxes of 128 rows x 32 fp32 (128B swizzle)
  static constexpr int STG_OFF = DLO_OFF + PTILEB;
  static constexpr int STGB = D / 32 * kBM * 128;
  static constexpr int BAR_OFF = STG_OFF + STGB;
  // K and V landed; Q and dO landed [2]; S^T and dP^T done; dV and dK
  // products done; dQ product done; a block's elementwise pass done (256
  // arrivals); the staging tile read by its reduction; drain
  static constexpr int B_KV = 0, B_QD = 1, B_SDP = 3, B_PROD = 4, B_DQ = 5, B_PASS = 6, B_STG = 7,
                       B_DRAIN = 8, NBARS = 9;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag
  static constexpr int USED = MISC_OFF + 16;
  static constexpr int SMEM = ((USED + 1023) / 1024) * 1024 + 1024;  // + realignment slack
  static constexpr int SMEM_LAUNCH = SMEM < 120 * 1024 ? 120 * 1024 : SMEM;
  static_assert(SMEM <= 232448, "shared memory budget");
  // TMEM columns: S^T (then P^T) at 0, dP^T (then dS^T) at 128, dV, dK,
  // dQ_part (lanes = queries)
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 256 + D,
                            DQ_COL = 256 + 2 * D;
  static_assert(256 + 3 * D <= (int)kTmemCols, "TMEM budget");
};

constexpr int kBwdTThreads = 288;  // 8 elementwise warps + the issuing warp
constexpr int kBwdTIssueWarp = 8;

template <int D>
__global__ void __launch_bounds__(kBwdTThreads, 1)
    hstu_bwd_t_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
  using C = TCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };

  if (tid == 0) {
    for (int i = 0; i < C::NBARS; ++i) mbar_init(bar(i), i == C::B_PASS ? 256u : 1u);
    // the staging tile starts free
    mbar_arrive(bar(C::B_STG));
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
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
  const float alpha = a.alpha;

  // the CTA's items: a host-built schedule's range, else every grid-th item
  const int idx0 = a.cta_first ? __ldg(&a.cta_first[blockIdx.x]) : (int)blockIdx.x;
  const int idx_end = a.cta_first ? __ldg(&a.cta_first[blockIdx.x + 1]) : a.n_items;
  const int idx_step = a.cta_first ? 1 : (int)gridDim.x;
  auto nq_of = [&](const BwdBlock& b, int hist) {
    // a key block of candidates only is seen by its own rows: the diagonal
    // query block alone
    return kBN * b.kt >= hist ? b.kt + 1 : (b.n + kBM - 1) / kBM;
  };

  if (warp == kBwdTIssueWarp) {
    // ------------------------------------------------------------ issuer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_do)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_dq)) : "memory");
      constexpr uint32_t IDESC_S = make_idesc(kBM, kBN, 0);
      constexpr uint32_t IDESC_TS = make_idesc(kBM, D, 1);          // A from TMEM, B MN-major
      constexpr uint32_t IDESC_DQ = make_idesc_ab(kBM, D, 1, 1);    // A and B MN-major
      constexpr int DSTEPS = D / 16, SPC = C::CHUNK / 16;
      const uint64_t k_kmaj = smem_desc(base + C::K_OFF, 16, C::ATOMB, C::LAYOUT);
      const uint64_t v_kmaj = smem_desc(base + C::V_OFF, 16, C::ATOMB, C::LAYOUT);
      const uint64_t q_kmaj0 = smem_desc(base + C::Q_OFF, 16, C::ATOMB, C::LAYOUT);
      const uint64_t do_kmaj0 = smem_desc(base + C::DO_OFF, 16, C::ATOMB, C::LAYOUT);
      const uint64_t k_mn = smem_desc(base + C::K_OFF, C::CHUNKB, C::ATOMB, C::LAYOUT);
      const uint64_t q_mn0 = smem_desc(base + C::Q_OFF, C::CHUNKB, C::ATOMB, C::LAYOUT);
      const uint64_t do_mn0 = smem_desc(base + C::DO_OFF, C::CHUNKB, C::ATOMB, C::LAYOUT);
      const uint64_t dhi_mn = smem_desc(base + C::DHI_OFF, C::PCHUNKB, 1024, 2);
      const uint64_t dlo_mn = smem_desc(base + C::DLO_OFF, C::PCHUNKB, 1024, 2);
      auto buf_desc = [&](uint64_t d0, int qb) { return d0 + (uint64_t)((qb * C::TILEB) >> 4); };
      auto load_tile = [&](const CUtensorMap* map, int off, int b, int h, int row0) {
#pragma unroll
        for (int ch = 0; ch < C::NCHUNK; ++ch)
          tma_load_3d(base + off + ch * C::CHUNKB, map, bar(b), ch * C::CHUNK, h, row0);
      };
      // S^T or dP^T = X Y^T over d: both K-major
      auto mma_xyt = [&](uint32_t d_col, uint64_t xd, uint64_t yd) {
#pragma unroll
        for (int kk = 0; kk < DSTEPS; ++kk) {
          const uint32_t off = (kk / SPC) * C::CHUNKB + (kk % SPC) * 32;
          if (kk == 0)
            mma_ss_c<0>(tmem + d_col, xd + (off >> 4), yd + (off >> 4), IDESC_S);
          else
            mma_ss_c<1>(tmem + d_col, xd + (off >> 4), yd + (off >> 4), IDESC_S);
        }
      };
      // T (+)= (hi + lo from TMEM at a_col, lanes = keys) B over the 128
      // queries: 16 queries a step, B MN-major.  Operands pinned first.
      auto mma_t = [&](uint32_t d_col, uint32_t a_col, uint64_t bd, bool first) {
        uint32_t ah[8];
        uint64_t bb[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          ah[kk] = pin32(tmem + a_col + (uint32_t)(32 * (kk >> 1) + 8 * (kk & 1)));
          bb[kk] = pin64(bd + (uint64_t)((kk * 2 * C::ATOMB) >> 4));
        }
        const uint32_t dt = pin32(tmem + d_col);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          if (first && kk == 0)
            mma_ts_c<0>(dt, ah[kk], bb[kk], IDESC_TS);
          else
            mma_ts_c<1>(dt, ah[kk], bb[kk], IDESC_TS);
          mma_ts_c<1>(dt, ah[kk] + 16u, bb[kk], IDESC_TS);
        }
      };
      // dQ_part = dS K over the 128 keys: dS^T tile read MN-major (M =
      // queries), K MN-major
      auto mma_dq = [&]() {
        uint64_t ah[8], al[8], bb[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          ah[kk] = pin64(dhi_mn + (uint64_t)((kk * 2048) >> 4));
          al[kk] = pin64(dlo_mn + (uint64_t)((kk * 2048) >> 4));
          bb[kk] = pin64(k_mn + (uint64_t)((kk * 2 * C::ATOMB) >> 4));
        }
        const uint32_t dt = pin32(tmem + C::DQ_COL);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          if (kk == 0)
            mma_ss_c<0>(dt, ah[kk], bb[kk], IDESC_DQ);
          else
            mma_ss_c<1>(dt, ah[kk], bb[kk], IDESC_DQ);
          mma_ss_c<1>(dt, al[kk], bb[kk], IDESC_DQ);
        }
      };
      auto reduce_dq = [&](int h, int row0) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
          asm volatile(
              "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
              " [%0, {%1, %2, %3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(&tm_dq)),
              "r"(32 * c), "r"(h), "r"(row0), "r"(base + C::STG_OFF + c * (kBM * 128))
              : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      };

      uint32_t n_kv = 0, n_qd[2] = {0, 0}, w_qd[2] = {0, 0};  // loads issued / waited per barrier
      uint32_t n_prod = 0, n_dq = 0, ph_pass = 0;
      uint32_t qiter = 0;
      bool ok = true, pending = false;
      int pend_h = 0, pend_row = 0;
      // test hook: a wait on a barrier that nothing signals runs out
      if (a.debug_flags & kDebugUnsignalledWait) ok = wait_one(bar(C::B_DRAIN), 0u, w, kSiteUnsignalled);
      auto load_qd = [&](int qb, const BwdBlock& b, int qt) {
        mbar_arrive_expect_tx(bar(C::B_QD + qb), 2 * C::TILEB);
        load_tile(&tm_q, C::Q_OFF + qb * C::TILEB, C::B_QD + qb, b.h, b.s0 + kBM * qt);
        load_tile(&tm_do, C::DO_OFF + qb * C::TILEB, C::B_QD + qb, b.h, b.s0 + kBM * qt);
        ++n_qd[qb];
      };
      auto wait_qd = [&](int qb) -> bool {
        const bool r = wait_one(bar(C::B_QD + qb), w_qd[qb] & 1u, w, kSiteQFull);
        ++w_qd[qb];
        return r;
      };
      for (int idx = idx0; ok && idx < idx_end; idx += idx_step) {
        const Item it = __ldg(&a.items[idx]);
        const BwdBlock b{it.x, it.y, it.z, it.w};
        const int hist = a.item_hist ? __ldg(a.item_hist + idx) : b.n;
        const int nq = nq_of(b, hist);
        // the previous item's products have finished reading K, V, Q, dO
        if (n_prod && !(ok = wait_one(bar(C::B_PROD), (n_prod - 1) & 1u, w, kSiteVFull))) break;
        if (n_dq && !(ok = wait_one(bar(C::B_DQ), (n_dq - 1) & 1u, w, kSiteOFull))) break;
        mbar_arrive_expect_tx(bar(C::B_KV), 2 * C::TILEB);
        load_tile(&tm_k, C::K_OFF, C::B_KV, b.h, b.s0 + kBN * b.kt);
        load_tile(&tm_v, C::V_OFF, C::B_KV, b.h, b.s0 + kBN * b.kt);
        ++n_kv;
        const int qb0 = (int)(qiter & 1u);
        load_qd(qb0, b, b.kt);
        if (b.kt + 1 < nq) load_qd(qb0 ^ 1, b, b.kt + 1);
        if (!(ok = wait_one(bar(C::B_KV), (n_kv - 1) & 1u, w, kSiteKFull))) break;
        if (!(ok = wait_qd(qb0))) break;
        tc_fence_after();
        mma_xyt(C::S_COL, k_kmaj, buf_desc(q_kmaj0, qb0));
        mma_xyt(C::DP_COL, v_kmaj, buf_desc(do_kmaj0, qb0));
        mma_commit(bar(C::B_SDP));
        if (pending) {
          // the previous item's last dQ, staged at that item's end
          if (!(ok = wait_one(bar(C::B_PASS), ph_pass, w, kSitePFull))) break;
          ph_pass ^= 1u;
          reduce_dq(pend_h, pend_row);
          asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          mbar_arrive(bar(C::B_STG));
          pending = false;
        }
        for (int qt = b.kt; qt < nq; ++qt, ++qiter) {
          const int qb = (int)(qiter & 1u);
          if (!(ok = wait_one(bar(C::B_PASS), ph_pass, w, kSitePFull))) break;
          ph_pass ^= 1u;
          tc_fence_after();
          // the pass staged the previous block's dQ
          if (qt > b.kt) reduce_dq(b.h, b.s0 + kBM * (qt - 1));
          mma_t(C::DV_COL, C::S_COL, buf_desc(do_mn0, qb), qt == b.kt);
          mma_t(C::DK_COL, C::DP_COL, buf_desc(q_mn0, qb), qt == b.kt);
          mma_commit(bar(C::B_PROD));
          ++n_prod;
          if (qt + 1 < nq) {
            // the next block's S^T and dP^T overwrite what dV and dK read
            if (!(ok = wait_one(bar(C::B_PROD), (n_prod - 1) & 1u, w, kSiteVFull))) break;
            if (qt + 2 < nq) load_qd(qb, b, qt + 2);  // buffer qb is free
            if (!(ok = wait_qd(qb ^ 1))) break;
            tc_fence_after();
            mma_xyt(C::S_COL, k_kmaj, buf_desc(q_kmaj0, qb ^ 1));
            mma_xyt(C::DP_COL, v_kmaj, buf_desc(do_kmaj0, qb ^ 1));
            mma_commit(bar(C::B_SDP));
          }
          mma_dq();
          mma_commit(bar(C::B_DQ));
          ++n_dq;
          if (qt > b.kt) {
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            mbar_arrive(bar(C::B_STG));
          }
        }
        if (!ok) break;
        pending = true;
        pend_h = b.h;
        pend_row = b.s0 + kBM * (nq - 1);
      }
      if (ok && pending) {
        // the last item's end phase: its last dQ is staged
        if ((ok = wait_one(bar(C::B_PASS), ph_pass, w, kSitePFull))) {
          reduce_dq(pend_h, pend_row);
        }
      }
      if (!ok) {
        // drain: every product issued, then every copy issued, has landed
        mma_commit(bar(C::B_DRAIN));
        wait_drain(bar(C::B_DRAIN), 0);
        if (n_kv) wait_drain(bar(C::B_KV), (n_kv - 1) & 1u);
        for (int qb = 0; qb < 2; ++qb)
          if (n_qd[qb] > w_qd[qb]) wait_drain(bar(C::B_QD + qb), (n_qd[qb] - 1) & 1u);
      }
      // the reductions have finished before the CTA (and its shared memory) goes
      asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- elementwise warps
    const int row = tid & 127;  // TMEM lane: the key (the query when staging dQ)
    const int wg = tid >> 7;    // half of the queries (of the dQ columns)
    const uint32_t lane_tm = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float ha = 0.5f * alpha, inv_n = a.inv_n;
    uint32_t ph_kv = 0, ph_sdp = 0, ph_dq = 0, ph_stg = 0, n_prod = 0;
    bool ok = true;
    // alpha dQ_part from TMEM into the staging tile (128B-swizzled fp32
    // boxes of 32 columns); the staging tile is free once B_STG says so
    auto stage_dq = [&]() -> bool {
      if (!wait_warp(bar(C::B_STG), ph_stg, w, kSiteOEmpty)) return false;
      ph_stg ^= 1u;
      tc_fence_after();
#pragma unroll 1
      for (int c = wg; c < D / 32; c += 2) {
        uint32_t r[32];
        tmem_ld32(lane_tm + C::DQ_COL + 32u * c, r);
        uint8_t* box = smem + C::STG_OFF + c * (kBM * 128);
#pragma unroll
        for (int g = 0; g < 8; ++g)
          *reinterpret_cast<float4*>(box + row * 128 + ((g ^ (row & 7)) << 4)) =
              make_float4(alpha * __uint_as_float(r[4 * g]), alpha * __uint_as_float(r[4 * g + 1]),
                          alpha * __uint_as_float(r[4 * g + 2]), alpha * __uint_as_float(r[4 * g + 3]));
      }
      return true;
    };
    // zero rows r0 .. 127 of a d-wide tile (every chunk)
    auto zero_rows = [&](int off, int r0) {
      for (int i = tid; i < (kBM - r0) * C::NCHUNK * (C::ROWB / 16); i += 256) {
        const int per_row = C::NCHUNK * (C::ROWB / 16);
        const int r = r0 + i / per_row, rest = i % per_row;
        const int ch = rest / (C::ROWB / 16), g = rest % (C::ROWB / 16);
        *reinterpret_cast<uint4*>(smem + off + ch * C::CHUNKB + r * C::ROWB + g * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    };
    uint32_t qiter = 0;
    for (int idx = idx0; ok && idx < idx_end; idx += idx_step) {
      const Item it = __ldg(&a.items[idx]);
      const BwdBlock b{it.x, it.y, it.z, it.w};
      const int hist = a.item_hist ? __ldg(a.item_hist + idx) : b.n;
      const int nq = nq_of(b, hist);
      const int key_rows = b.n - kBN * b.kt;  // keys of the block that exist (>= 1)
      const int j = kBN * b.kt + row;         // this thread's key, sequence-local
      if (!(ok = wait_warp(bar(C::B_KV), ph_kv, w, kSiteKFull))) break;
      ph_kv ^= 1u;
      // K rows past the sequence: zero before dQ reads them
      if (key_rows < kBN) zero_rows(C::K_OFF, key_rows);
      for (int qt = b.kt; qt < nq; ++qt, ++qiter) {
        const int qb = (int)(qiter & 1u);
        if (!(ok = wait_warp(bar(C::B_SDP), ph_sdp, w, kSiteSFull))) break;
        ph_sdp ^= 1u;
        tc_fence_after();
        // kept queries of this key: q in [qlo, qhi) of the block (causal:
        // from the key on, up to the sequence end; a candidate key: itself)
        const int i0 = kBM * qt;
        const int qlo = j - i0;
        int qhi = b.n - i0;
        if (j >= hist) qhi = qhi < qlo + 1 ? qhi : qlo + 1;
        uint32_t dsh[2][16], dsl[2][16];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * wg + cc;
          uint32_t sr[32], pr[32];
          tmem_ld32_async(lane_tm + C::S_COL + 32u * c, sr);
          tmem_ld32_async(lane_tm + C::DP_COL + 32u * c, pr);
          tmem_wait_ld(sr);
          tmem_wait_ld(pr);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t ph[8], pl[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              float pv[2], dv[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int k = 16 * h + 2 * m + e;
                const int q = 32 * c + k;
                const bool keep = q >= qlo && q < qhi;
                const float s = __uint_as_float(sr[k]);
                const float x = alpha * s;
                const float sg = fmaf(0.5f, tanh_approx(ha * s), 0.5f);
                const float isg = inv_n * sg;
                pv[e] = keep ? isg * x : 0.0f;
                dv[e] = keep ? isg * fmaf(x, 1.0f - sg, 1.0f) * __uint_as_float(pr[k]) : 0.0f;
              }
              const uint32_t p_hi = pack_bf16x2(pv[0], pv[1]);
              ph[m] = p_hi;
              pl[m] = pack_bf16x2(pv[0] - __uint_as_float(p_hi << 16),
                                  pv[1] - __uint_as_float(p_hi & 0xFFFF0000u));
              const uint32_t d_hi = pack_bf16x2(dv[0], dv[1]);
              dsh[cc][8 * h + m] = d_hi;
              dsl[cc][8 * h + m] = pack_bf16x2(dv[0] - __uint_as_float(d_hi << 16),
                                               dv[1] - __uint_as_float(d_hi & 0xFFFF0000u));
            }
            tmem_st8(lane_tm + C::S_COL + 32u * c + 8u * h, ph);
            tmem_st8(lane_tm + C::S_COL + 32u * c + 16u + 8u * h, pl);
          }
          uint32_t t8[8];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int m = 0; m < 8; ++m) t8[m] = dsh[cc][8 * h + m];
            tmem_st8(lane_tm + C::DP_COL + 32u * c + 8u * h, t8);
#pragma unroll
            for (int m = 0; m < 8; ++m) t8[m] = dsl[cc][8 * h + m];
            tmem_st8(lane_tm + C::DP_COL + 32u * c + 16u + 8u * h, t8);
          }
        }
        // the last query block's Q and dO rows past the sequence: zero
        // before dK and dV read them
        if (b.n - i0 < kBM) {
          zero_rows(C::Q_OFF + qb * C::TILEB, b.n - i0);
          zero_rows(C::DO_OFF + qb * C::TILEB, b.n - i0);
        }
        if (qt > b.kt) {
          // the previous block's dQ product is done: its dS^T tile is free
          // and its dQ_part final
          if (!(ok = wait_warp(bar(C::B_DQ), ph_dq, w, kSiteOFull))) break;
          ph_dq ^= 1u;
        }
        // dS^T into the shared tiles: row = key, 32 queries per chunk
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * wg + cc;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint32_t o = ptile_off(row, 32 * c + 8 * g);
            *reinterpret_cast<uint4*>(smem + C::DHI_OFF + o) =
                make_uint4(dsh[cc][4 * g], dsh[cc][4 * g + 1], dsh[cc][4 * g + 2], dsh[cc][4 * g + 3]);
            *reinterpret_cast<uint4*>(smem + C::DLO_OFF + o) =
                make_uint4(dsl[cc][4 * g], dsl[cc][4 * g + 1], dsl[cc][4 * g + 2], dsl[cc][4 * g + 3]);
          }
        }
        if (qt > b.kt && !(ok = stage_dq())) break;
        tmem_wait_st();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        mbar_arrive(bar(C::B_PASS));
        ++n_prod;
      }
      if (!ok) break;
      // the item's end: its last dV / dK and dQ products are done
      if (!(ok = wait_warp(bar(C::B_PROD), (n_prod - 1) & 1u, w, kSiteVFull))) break;
      if (!(ok = wait_warp(bar(C::B_DQ), ph_dq, w, kSiteOFull))) break;
      ph_dq ^= 1u;
      if (!(ok = stage_dq())) break;
      // dV and alpha dK of the item's keys (key row = TMEM lane)
      tc_fence_after();
      {
        const bool key_ok = row < key_rows;
        const size_t trow = ((size_t)(b.s0 + kBN * b.kt + row) * a.heads + b.h) * D;
#pragma unroll 1
        for (int c = wg; c < D / 32; c += 2) {
          uint32_t rv[32], rk[32];
          tmem_ld32(lane_tm + C::DV_COL + 32u * c, rv);
          tmem_ld32(lane_tm + C::DK_COL + 32u * c, rk);
          if (key_ok) {
            uint4* dv = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dv) + trow + 32 * c);
            uint4* dk = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dk) + trow + 32 * c);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              uint32_t pv[4], pk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int q = 8 * m + 2 * e;
                pv[e] = pack_bf16x2(__uint_as_float(rv[q]), __uint_as_float(rv[q + 1]));
                pk[e] = pack_bf16x2(alpha * __uint_as_float(rk[q]), alpha * __uint_as_float(rk[q + 1]));
              }
              dv[m] = make_uint4(pv[0], pv[1], pv[2], pv[3]);
              dk[m] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(bar(C::B_PASS));  // the item's end phase: dQ staged, dV and dK read
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

template <int D>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                         cudaStream_t stream) {
  using C = TCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(hstu_bwd_t_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_LAUNCH);
  if (e != cudaSuccess) return e;
  hstu_bwd_t_kernel<D><<<grid, kBwdTThreads, C::SMEM_LAUNCH, stream>>>(tq, tk, tv, tdo, tdq, a);
  return cudaGetLastError();
}
