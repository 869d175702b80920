// Backward pass in transposed form, for d <= 64 without the bias (HSTU
// paper Appendix G: the backward recomputes the attention and accumulates
// the gradients on chip).  The gradients are those of hstu_bwd.cuh; only
// the orientation of the recomputed scores differs.
//
// Work item, as in hstu_bwd.cuh: one 128-key block kt of one (sequence,
// head), walking the query blocks qt that see it.  A query block is taken
// in two halves of 64 queries.  Per half h of block qt:
//   1. S^T = K Q_h^T and dP^T = V dO_h^T into TMEM (M = 128 keys, N = 64
//      queries): the TMEM lanes are the block's keys, the columns queries.
//   2. Thread r (and r + 128, each taking 32 of the half's queries) owns
//      key r: P^T = inv_n silu(alpha S^T) and dS^T = inv_n silu'(alpha S^T)
//      (.) dP^T, each split into bf16 hi + lo, overwrite S^T and dP^T in
//      TMEM (16 columns of hi and 16 of lo per 32 queries: the A-operand
//      layout of a product read from TMEM).
//   3. dV += P_h^T dO_h and dK += dS_h^T Q_h read their A operand from
//      TMEM: no shared tile is written for them.
// Each half's dS^T also goes to shared memory (rows = keys, 64 queries
// contiguous, 128-byte swizzle; half 0 into one of two buffers by block
// parity, since the previous block's dQ may still be reading the other).
// Once both halves are there, dQ_part = dS K reads them as one MN-major A
// operand (M = queries; the descriptor's leading offset spans the two
// halves); alpha dQ_part goes into the fp32 accumulator by bulk tensor
// reductions from a staging tile, as in hstu_bwd.cuh.
//
// Warp 8 (one thread) issues the copies and the S^T, dP^T, dV and dK
// products; warp 9 (one thread) issues dQ and its reductions, so that
// neither stream waits behind the other's barriers; warps 0-7 do the
// elementwise work, the dQ staging and the item's dV / dK stores.  The
// halves pipeline: while the threads work on half 1, half 0's dV and dK
// products run and then the next block's half-0 S^T and dP^T (which
// overwrite the columns those products read, so they wait for them); while
// the threads work on the next block's half 0, half 1's products, its next
// S^T and dP^T, and the block's dQ run.  Q and dO load half a block at a
// time, two blocks ahead.
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
  static constexpr int HALFB = TILEB / 2;           // a half block's bytes (64 rows)
  static constexpr uint64_t LAYOUT = ROWB == 128 ? 2 : 4;  // 128B / 64B swizzle
  // dS^T halves: 128 keys x 64 queries bf16 (128B swizzle), hi and lo;
  // half 0 in two buffers (buffer b: hi at D0_OFF + 2 b PCHUNKB, lo after
  // it), half 1 in one
  static constexpr int PCHUNKB = kBM * 128;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILEB;
  static constexpr int Q_OFF = V_OFF + TILEB;        // two buffers
  static constexpr int DO_OFF = Q_OFF + 2 * TILEB;   // two buffers
  static constexpr int D0_OFF = DO_OFF + 2 * TILEB;
  static constexpr int HI1_OFF = D0_OFF + 4 * PCHUNKB;
  static constexpr int LO1_OFF = HI1_OFF + PCHUNKB;
  __host__ __device__ static constexpr int hi0_off(int b) { return D0_OFF + 2 * b * PCHUNKB; }
  // alpha dQ_part staging: D / 32 boxes of 128 rows x 32 fp32 (128B swizzle)
  static constexpr int STG_OFF = LO1_OFF + PCHUNKB;
  static constexpr int STGB = D / 32 * kBM * 128;
  static constexpr int BAR_OFF = STG_OFF + STGB;
  // K and V landed; Q and dO landed [buffer][half]; S^T and dP^T done
  // [half]; dV and dK products done [half]; dQ product done; a half's
  // elementwise pass done [half] (256 arrivals); the staging tile read by
  // its reduction; the two issuing threads' drains
  static constexpr int B_KV = 0, B_QD = 1 /* [4] */, B_SDP = 5 /* [2] */, B_PROD = 7 /* [2] */,
                       B_DQ = 9, B_PASS = 10 /* [2] */, B_STG = 12, B_DRAIN = 13 /* [2] */,
                       NBARS = 15;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag
  static constexpr int USED = MISC_OFF + 16;
  static constexpr int SMEM = ((USED + 1023) / 1024) * 1024 + 1024;  // + realignment slack
  static constexpr int SMEM_LAUNCH = SMEM < 120 * 1024 ? 120 * 1024 : SMEM;
  static_assert(SMEM <= 232448, "shared memory budget");
  // TMEM columns: S^T (then P^T) at 0, dP^T (then dS^T) at 128 (half h at
  // + 64 h), dV, dK, dQ_part (lanes = queries)
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 256 + D,
                            DQ_COL = 256 + 2 * D;
  static_assert(256 + 3 * D <= (int)kTmemCols, "TMEM budget");
  static __host__ __device__ constexpr uint32_t arrivals(int i) {
    return (i == B_PASS || i == B_PASS + 1) ? 256u : 1u;
  }
};

// 8 elementwise warps, the warp that issues the copies and the S^T, dP^T,
// dV and dK products, and the warp that issues dQ and its reductions
constexpr int kBwdTThreads = 320;
constexpr int kBwdTIssueWarp = 8;
constexpr int kBwdTDqWarp = 9;

// One 32-query chunk of a key row: P and dS from the recomputed scores s
// and dP (fp32 TMEM words), split into bf16 hi + lo words (word m holds
// queries 2m, 2m + 1).  P goes into TMEM at t_p (hi: 16 columns, then lo:
// 16) as each 16 queries are done; dS stays in dh / dl.  MASK: keep query q
// (0..31) iff qlo <= q < qhi.
template <bool MASK>
__device__ __forceinline__ void bwd_t_chunk(const uint32_t (&sr)[32], const uint32_t (&pr)[32],
                                            float2 a2, float2 ha2, float2 in2, int qlo, int qhi,
                                            uint32_t t_p, uint32_t (&dh)[16], uint32_t (&dl)[16]) {
  const float2 one = make_float2(1.0f, 1.0f), half = make_float2(0.5f, 0.5f);
  const float2 mone = make_float2(-1.0f, -1.0f);
  uint32_t ph[8], pl[8];
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    const float2 s = make_float2(__uint_as_float(sr[2 * m]), __uint_as_float(sr[2 * m + 1]));
    const float2 dp = make_float2(__uint_as_float(pr[2 * m]), __uint_as_float(pr[2 * m + 1]));
    const float2 x = __fmul2_rn(s, a2);
    const float2 h = __fmul2_rn(s, ha2);
    const float2 sg = __ffma2_rn(make_float2(tanh_approx(h.x), tanh_approx(h.y)), half, half);
    const float2 isg = __fmul2_rn(sg, in2);
    float2 p = __fmul2_rn(isg, x);
    // silu'(x) = sg (1 + x (1 - sg))
    const float2 om = __ffma2_rn(sg, mone, one);
    float2 d = __fmul2_rn(__fmul2_rn(__ffma2_rn(x, om, one), isg), dp);
    if constexpr (MASK) {
      const int q = 2 * m;
      const bool k0 = q >= qlo && q < qhi, k1 = q + 1 >= qlo && q + 1 < qhi;
      p.x = k0 ? p.x : 0.0f;
      p.y = k1 ? p.y : 0.0f;
      d.x = k0 ? d.x : 0.0f;
      d.y = k1 ? d.y : 0.0f;
    }
    const uint32_t p_hi = pack_bf16x2(p.x, p.y);
    const float2 pr2 = __fadd2_rn(
        p, make_float2(-__uint_as_float(p_hi << 16), -__uint_as_float(p_hi & 0xFFFF0000u)));
    ph[m & 7] = p_hi;
    pl[m & 7] = pack_bf16x2(pr2.x, pr2.y);
    const uint32_t d_hi = pack_bf16x2(d.x, d.y);
    const float2 dr2 = __fadd2_rn(
        d, make_float2(-__uint_as_float(d_hi << 16), -__uint_as_float(d_hi & 0xFFFF0000u)));
    dh[m] = d_hi;
    dl[m] = pack_bf16x2(dr2.x, dr2.y);
    if ((m & 7) == 7) {
      tmem_st8(t_p + (uint32_t)(m & 8), ph);
      tmem_st8(t_p + 16u + (uint32_t)(m & 8), pl);
    }
  }
}

// 16 words into TMEM as two groups of 8 columns (the A-operand layout:
// queries 0-15 in the first 8 columns, 16-31 in the next 8).
__device__ __forceinline__ void bwd_t_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  uint32_t t8[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) t8[m] = r[m];
  tmem_st8(taddr, t8);
#pragma unroll
  for (int m = 0; m < 8; ++m) t8[m] = r[8 + m];
  tmem_st8(taddr + 8u, t8);
}

// Bounded wait for the issuing thread: a non-blocking test first (a
// try_wait on a phase that is already complete still holds the thread for
// a few hundred cycles, and with it the stream of products it feeds).
__device__ __forceinline__ bool wait_issuer(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
  if (mbar_test(bar, parity)) return true;
  return wait_one(bar, parity, w, site);
}

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
    for (int i = 0; i < C::NBARS; ++i) mbar_init(bar(i), C::arrivals(i));
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

  if (warp == kBwdTIssueWarp || warp == kBwdTDqWarp) {
    // ------------------------------------------------------- issuers
    if (lane == 0) {
      if (warp == kBwdTIssueWarp) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_do)) : "memory");
      } else {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_dq)) : "memory");
      }
      constexpr uint32_t IDESC_S = make_idesc(kBM, kBN / 2, 0);     // N = 64 queries
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
      // dS^T as the MN-major A operand of dQ: half 0 of buffer b, then half 1
      // at the leading byte offset; lo PCHUNKB after hi in both
      auto ds_desc = [&](int b) {
        return smem_desc(base + C::hi0_off(b), C::HI1_OFF - C::hi0_off(b), 1024, 2);
      };
      // descriptor of buffer qb's half h (64 rows: 64 * ROWB bytes into each chunk)
      auto half_desc = [&](uint64_t d0, int qb, int h) {
        return d0 + (uint64_t)((qb * C::TILEB + h * 64 * C::ROWB) >> 4);
      };
      // S^T or dP^T of half h = X Y_h^T over d: both K-major; operands pinned
      auto mma_xyt = [&](uint32_t d_col, uint64_t xd, uint64_t yd) {
        uint64_t xa[DSTEPS], ya[DSTEPS];
#pragma unroll
        for (int kk = 0; kk < DSTEPS; ++kk) {
          const uint32_t off = (kk / SPC) * C::CHUNKB + (kk % SPC) * 32;
          xa[kk] = pin64(xd + (off >> 4));
          ya[kk] = pin64(yd + (off >> 4));
        }
        const uint32_t dt = pin32(tmem + d_col);
        mma_ss_c<0>(dt, xa[0], ya[0], IDESC_S);
#pragma unroll
        for (int kk = 1; kk < DSTEPS; ++kk) mma_ss_c<1>(dt, xa[kk], ya[kk], IDESC_S);
      };
      // T (+)= (hi + lo from TMEM at a_col, lanes = keys) B over half h's
      // 64 queries: 16 queries a step, B MN-major.  Operands pinned first;
      // the first product overwrites where `first` says so.
      auto mma_t = [&](uint32_t d_col, uint32_t a_col, uint64_t bd, int h, bool first) {
        uint32_t ah[4], al[4];
        uint64_t bb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kk = 4 * h + i;
          ah[i] = pin32(tmem + a_col + (uint32_t)(32 * (kk >> 1) + 8 * (kk & 1)));
          al[i] = pin32(tmem + a_col + (uint32_t)(32 * (kk >> 1) + 8 * (kk & 1) + 16));
          bb[i] = pin64(bd + (uint64_t)((kk * 2 * C::ATOMB) >> 4));
        }
        const uint32_t dt = pin32(tmem + d_col);
        if (first)
          mma_ts_c<0>(dt, ah[0], bb[0], IDESC_TS);
        else
          mma_ts_c<1>(dt, ah[0], bb[0], IDESC_TS);
        mma_ts_c<1>(dt, al[0], bb[0], IDESC_TS);
#pragma unroll
        for (int i = 1; i < 4; ++i) {
          mma_ts_c<1>(dt, ah[i], bb[i], IDESC_TS);
          mma_ts_c<1>(dt, al[i], bb[i], IDESC_TS);
        }
      };
      // dQ_part = dS K over the 128 keys: the dS^T halves of buffer b read
      // MN-major (M = queries), K MN-major
      auto mma_dq = [&](int buf) {
        const uint64_t dhi_mn = ds_desc(buf), dlo_mn = dhi_mn + (uint64_t)(C::PCHUNKB >> 4);
        uint64_t ah[8], al[8], bb[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          ah[kk] = pin64(dhi_mn + (uint64_t)((kk * 2048) >> 4));
          al[kk] = pin64(dlo_mn + (uint64_t)((kk * 2048) >> 4));
          bb[kk] = pin64(k_mn + (uint64_t)((kk * 2 * C::ATOMB) >> 4));
        }
        const uint32_t dt = pin32(tmem + C::DQ_COL);
        mma_ss_c<0>(dt, ah[0], bb[0], IDESC_DQ);
        mma_ss_c<1>(dt, al[0], bb[0], IDESC_DQ);
#pragma unroll
        for (int kk = 1; kk < 8; ++kk) {
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

      bool ok = true;
      uint32_t ph_pass[2] = {0, 0};
      auto wait_pass = [&](int h) -> bool {
        const bool r = wait_issuer(bar(C::B_PASS + h), ph_pass[h], w, kSitePFull);
        ph_pass[h] ^= 1u;
        return r;
      };
      if (warp == kBwdTIssueWarp) {
        // copies issued / waited per Q-dO barrier ([buffer][half]); blocks
        // whose products were issued (one dV/dK commit per half and one dQ
        // commit each)
        uint32_t n_kv = 0, n_qd[4] = {0, 0, 0, 0}, w_qd[4] = {0, 0, 0, 0};
        uint32_t n_prod = 0, qiter = 0;
        // test hook: a wait on a barrier that nothing signals runs out
        if (a.debug_flags & kDebugUnsignalledWait) ok = wait_issuer(bar(C::B_DRAIN), 0u, w, kSiteUnsignalled);
        auto load_half = [&](int qb, int h, const BwdBlock& b, int qt) {
          const int i = 2 * qb + h;
          const int row0 = b.s0 + kBM * qt + 64 * h;
          mbar_arrive_expect_tx(bar(C::B_QD + i), 2 * C::HALFB);
#pragma unroll
          for (int ch = 0; ch < C::NCHUNK; ++ch) {
            tma_load_3d(base + C::Q_OFF + qb * C::TILEB + ch * C::CHUNKB + h * 64 * C::ROWB, &tm_q,
                        bar(C::B_QD + i), ch * C::CHUNK, b.h, row0);
            tma_load_3d(base + C::DO_OFF + qb * C::TILEB + ch * C::CHUNKB + h * 64 * C::ROWB, &tm_do,
                        bar(C::B_QD + i), ch * C::CHUNK, b.h, row0);
          }
          ++n_qd[i];
        };
        auto wait_half = [&](int qb, int h) -> bool {
          const int i = 2 * qb + h;
          const bool r = wait_issuer(bar(C::B_QD + i), w_qd[i] & 1u, w, kSiteQFull);
          ++w_qd[i];
          return r;
        };
        auto issue_sdp = [&](int qb, int h) {
          tc_fence_after();
          mma_xyt(C::S_COL + 64u * h, k_kmaj, half_desc(q_kmaj0, qb, h));
          mma_xyt(C::DP_COL + 64u * h, v_kmaj, half_desc(do_kmaj0, qb, h));
          mma_commit(bar(C::B_SDP + h));
        };
        for (int idx = idx0; ok && idx < idx_end; idx += idx_step) {
          const Item it = __ldg(&a.items[idx]);
          const BwdBlock b{it.x, it.y, it.z, it.w};
          const int hist = a.item_hist ? __ldg(a.item_hist + idx) : b.n;
          const int nq = nq_of(b, hist);
          // the previous item's products have finished reading K, V, Q, dO
          // (its last dQ, issued by the other thread, reads K)
          if (n_prod) {
            if (!(ok = wait_issuer(bar(C::B_PROD), (n_prod - 1) & 1u, w, kSiteVFull))) break;
            if (!(ok = wait_issuer(bar(C::B_PROD + 1), (n_prod - 1) & 1u, w, kSiteVFull))) break;
            if (!(ok = wait_issuer(bar(C::B_DQ), (n_prod - 1) & 1u, w, kSiteOFull))) break;
          }
          mbar_arrive_expect_tx(bar(C::B_KV), 2 * C::TILEB);
#pragma unroll
          for (int ch = 0; ch < C::NCHUNK; ++ch) {
            tma_load_3d(base + C::K_OFF + ch * C::CHUNKB, &tm_k, bar(C::B_KV), ch * C::CHUNK, b.h,
                        b.s0 + kBN * b.kt);
            tma_load_3d(base + C::V_OFF + ch * C::CHUNKB, &tm_v, bar(C::B_KV), ch * C::CHUNK, b.h,
                        b.s0 + kBN * b.kt);
          }
          ++n_kv;
          const int qb0 = (int)(qiter & 1u);
          load_half(qb0, 0, b, b.kt);
          load_half(qb0, 1, b, b.kt);
          if (b.kt + 1 < nq) {
            load_half(qb0 ^ 1, 0, b, b.kt + 1);
            load_half(qb0 ^ 1, 1, b, b.kt + 1);
          }
          if (!(ok = wait_issuer(bar(C::B_KV), (n_kv - 1) & 1u, w, kSiteKFull))) break;
          if (!(ok = wait_half(qb0, 0))) break;
          issue_sdp(qb0, 0);
          // The previous item's end phase of the half-1 pass barrier: its dV
          // and dK have left TMEM before this item's first products
          // overwrite them.  It is waited for before this item's first
          // half-1 S^T and dP^T are issued: no elementwise warp can then
          // arrive for this item's first half-1 pass while another has yet
          // to arrive for the end phase (the barrier counts arrivals, not
          // who makes them), and the phase cannot be overtaken.
          if (n_prod && !(ok = wait_pass(1))) break;
          if (!(ok = wait_half(qb0, 1))) break;
          issue_sdp(qb0, 1);
          for (int qt = b.kt; qt < nq; ++qt, ++qiter) {
            const int qb = (int)(qiter & 1u);
            const bool first = qt == b.kt;
            for (int h = 0; h < 2; ++h) {
              if (!(ok = wait_pass(h))) break;
              tc_fence_after();
              mma_t(C::DV_COL, C::S_COL, half_desc(do_mn0, qb, 0), h, first && h == 0);
              mma_t(C::DK_COL, C::DP_COL, half_desc(q_mn0, qb, 0), h, first && h == 0);
              mma_commit(bar(C::B_PROD + h));
              if (qt + 1 < nq) {
                // the next block's half-h S^T and dP^T overwrite what these
                // products read; half h of buffer qb is then free for block qt + 2
                if (!(ok = wait_issuer(bar(C::B_PROD + h), n_prod & 1u, w, kSiteVFull))) break;
                if (qt + 2 < nq) load_half(qb, h, b, qt + 2);
                if (!(ok = wait_half(qb ^ 1, h))) break;
                issue_sdp(qb ^ 1, h);
              }
            }
            if (!ok) break;
            ++n_prod;
          }
        }
        if (!ok) {
          // drain: every product issued, then every copy issued, has landed
          mma_commit(bar(C::B_DRAIN));
          wait_drain(bar(C::B_DRAIN), 0);
          if (n_kv) wait_drain(bar(C::B_KV), (n_kv - 1) & 1u);
          for (int i = 0; i < 4; ++i)
            if (n_qd[i] > w_qd[i]) wait_drain(bar(C::B_QD + i), (n_qd[i] - 1) & 1u);
        }
      } else {
        // dQ: per block, once the elementwise pass has written dS^T (and
        // staged the previous block's dQ_part), the reduction of that part,
        // then the block's dQ product; at an item's end, the reduction of
        // its last part.  The staging tile goes back to the elementwise
        // warps once a reduction has read it.
        uint32_t qiter = 0;
        auto release_stg = [&]() {
          asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          mbar_arrive(bar(C::B_STG));
        };
        for (int idx = idx0; ok && idx < idx_end; idx += idx_step) {
          const Item it = __ldg(&a.items[idx]);
          const BwdBlock b{it.x, it.y, it.z, it.w};
          const int hist = a.item_hist ? __ldg(a.item_hist + idx) : b.n;
          const int nq = nq_of(b, hist);
          for (int qt = b.kt; qt < nq; ++qt, ++qiter) {
            if (!(ok = wait_pass(1))) break;
            tc_fence_after();
            if (qt > b.kt) reduce_dq(b.h, b.s0 + kBM * (qt - 1));
            mma_dq((int)(qiter & 1u));
            mma_commit(bar(C::B_DQ));
            if (qt > b.kt) release_stg();
          }
          if (!ok) break;
          // the item's end phase: its last dQ_part is staged
          if (!(ok = wait_pass(1))) break;
          reduce_dq(b.h, b.s0 + kBM * (nq - 1));
          release_stg();
        }
        if (!ok) {
          mma_commit(bar(C::B_DRAIN + 1));
          wait_drain(bar(C::B_DRAIN + 1), 0);
        }
        // the reductions have finished before the CTA (and its shared memory) goes
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- elementwise warps
    const int row = tid & 127;  // TMEM lane: the key (the query when staging dQ)
    const int wg = tid >> 7;    // which 32 queries of a half (which dQ columns)
    const uint32_t lane_tm = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float2 a2 = make_float2(alpha, alpha), ha2 = make_float2(0.5f * alpha, 0.5f * alpha);
    const float2 in2 = make_float2(a.inv_n, a.inv_n);
    uint32_t ph_kv = 0, ph_sdp[2] = {0, 0}, ph_dq = 0, ph_stg = 0, n_prod = 0;
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
    // zero rows r0 .. r1 - 1 of a d-wide tile (every chunk)
    auto zero_rows = [&](int off, int r0, int r1) {
      constexpr int per_row = C::NCHUNK * (C::ROWB / 16);
      for (int i = tid; i < (r1 - r0) * per_row; i += 256) {
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
      if (key_rows < kBN) zero_rows(C::K_OFF, key_rows, kBN);
      for (int qt = b.kt; qt < nq; ++qt, ++qiter) {
        const int qb = (int)(qiter & 1u);
        const int i0 = kBM * qt;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t dh[16], dl[16];  // this chunk's dS hi / lo
          if (!(ok = wait_warp(bar(C::B_SDP + h), ph_sdp[h], w, kSiteSFull))) break;
          ph_sdp[h] ^= 1u;
          tc_fence_after();
          const int c = 2 * h + wg;  // this thread's 32 queries: 32 c .. 32 c + 31
          // kept queries of this key in the chunk: q in [qlo, qhi) (causal:
          // from the key on, up to the sequence end; a candidate key: itself)
          const int qlo = j - i0 - 32 * c;
          int qhi = b.n - i0 - 32 * c;
          if (j >= hist) qhi = qhi < qlo + 1 ? qhi : qlo + 1;
          uint32_t sr[32], pr[32];
          tmem_ld32_async(lane_tm + C::S_COL + 32u * c, sr);
          tmem_ld32_async(lane_tm + C::DP_COL + 32u * c, pr);
          tmem_wait_ld(sr);
          tmem_wait_ld(pr);
          const uint32_t t_p = lane_tm + C::S_COL + 32u * c;
          if (__all_sync(0xffffffffu, qlo <= 0 && qhi >= 32))
            bwd_t_chunk<false>(sr, pr, a2, ha2, in2, qlo, qhi, t_p, dh, dl);
          else
            bwd_t_chunk<true>(sr, pr, a2, ha2, in2, qlo, qhi, t_p, dh, dl);
          bwd_t_st16(lane_tm + C::DP_COL + 32u * c, dh);
          bwd_t_st16(lane_tm + C::DP_COL + 32u * c + 16u, dl);
          // the last query block's Q and dO rows past the sequence, in this
          // half: zero before dK and dV read them
          const int live = b.n - i0 - 64 * h;  // rows of the half that exist
          if (live < 64) {
            const int r0 = 64 * h + (live > 0 ? live : 0);
            zero_rows(C::Q_OFF + qb * C::TILEB, r0, 64 * h + 64);
            zero_rows(C::DO_OFF + qb * C::TILEB, r0, 64 * h + 64);
          }
          // half 1's shared tile (and the staging tile) are free once the
          // previous block's dQ product is done; half 0 writes the buffer
          // that the block before that read
          if (h == 1 && qt > b.kt) {
            if (!(ok = wait_warp(bar(C::B_DQ), ph_dq, w, kSiteOFull))) break;
            ph_dq ^= 1u;
          }
          // dS^T into this half's shared tile: row = key, 32 queries
          {
            const int hi_off = h == 0 ? C::hi0_off((int)(qiter & 1u)) : C::HI1_OFF;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint32_t o =
                  (uint32_t)(row * 128 + ((((32 * wg + 8 * g) >> 3) ^ (row & 7)) << 4));
              *reinterpret_cast<uint4*>(smem + hi_off + o) =
                  make_uint4(dh[4 * g], dh[4 * g + 1], dh[4 * g + 2], dh[4 * g + 3]);
              *reinterpret_cast<uint4*>(smem + hi_off + C::PCHUNKB + o) =
                  make_uint4(dl[4 * g], dl[4 * g + 1], dl[4 * g + 2], dl[4 * g + 3]);
            }
          }
          if (h == 1 && qt > b.kt && !(ok = stage_dq())) break;
          tmem_wait_st();
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_before();
          mbar_arrive(bar(C::B_PASS + h));
        }
        if (!ok) break;
        ++n_prod;
      }
      if (!ok) break;
      // the item's end: its last dV / dK and dQ products are done
      if (!(ok = wait_warp(bar(C::B_PROD), (n_prod - 1) & 1u, w, kSiteVFull))) break;
      if (!(ok = wait_warp(bar(C::B_PROD + 1), (n_prod - 1) & 1u, w, kSiteVFull))) break;
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
      mbar_arrive(bar(C::B_PASS + 1));  // the item's end phase: dQ staged, dV and dK read
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
