// Backward pass of the HSTU jagged attention (HSTU paper Appendix G: the
// backward recomputes the attention; its gradients follow the forward
// definition).  With s_ij = alpha q_i.k_j, P_ij = inv_n silu(s_ij) on kept
// pairs (causal, same sequence; with candidates, the candidate mask) and
// out_i = sum_j P_ij v_j:
//
//   dV = P^T dO,   dP = dO V^T,   dS = inv_n silu'(s) (.) dP (kept pairs),
//   dQ = alpha dS K,   dK = alpha dS^T Q,   silu'(x) = sig(x) (1 + x (1 - sig(x))).
//
// Included into hstu_fwd.cu's anonymous namespace: it shares that file's
// PTX helpers, bounded waits and device status word.
//
// Work item: one 128-key block kt of one (sequence, head); the CTA walks the
// query blocks qt = kt .. last that see it.  K and V load once per item,
// Q and dO once per query block (double-buffered where shared memory has
// room).  One thread issues the copies and the products; two warpgroups
// (thread r and r + 128 share TMEM lane r, each taking half of the key
// columns) turn S and dP into P and dS.  Per query block:
//   1. S = Q K^T and dP = dO V^T into TMEM (fp32).
//   2. P = inv_n silu(alpha S), split into bf16 hi + lo, written to two
//      128B-swizzled shared tiles (rows = queries, 64-key chunks).
//   3. dV += P_hi^T dO + P_lo^T dO: the tile read as an MN-major A operand
//      (M = keys), dO as an MN-major B operand, accumulated in TMEM.
//   4. dS, split the same way into the same tiles (P's products are done).
//   5. dK += dS^T Q (as step 3) and dQ_part = dS K (the tile read as a
//      K-major A operand, K as an MN-major B), dQ_part over S in TMEM.
//   6. dQ_part * alpha is added into an fp32 accumulator in global memory
//      by bulk tensor reductions from a shared staging tile: query block qt
//      gets one part per key block.
// At the item's end dV and alpha dK leave TMEM as bf16.  The P and dS
// splits keep the products' error at the bf16 output rounding, as in the
// forward.  Where shared memory has room (d <= 64) P and dS have tiles of
// their own: one pass computes both, and steps 3 and 5 issue together, and
// the next block's S and dP are issued behind the current products.
//
// Candidates (HSTU paper section 3.4, Appendix H): each item carries its
// history length hist.  A candidate sees the history and itself, so a key
// block of candidates only is walked for its own query block alone, and a
// chunk holding candidate keys selects with the candidate mask.
//
// The bias rab_{p,t} (variant RAB): s_ij gains pos[bucket] + time[bucket],
// recomputed as in the forward.  The tables' gradients are the sums of dS
// over each bucket's kept pairs.  Each thread keeps running sums, added into
// a CTA-wide histogram where its bucket changes, and into dpos / dtime at
// exit.

template <int D, bool RAB = false>
struct BCfg {
  static constexpr int CHUNK = D < 64 ? D : 64;  // elements per swizzled row of a d-wide tile
  static constexpr int NCHUNK = D / CHUNK;
  static constexpr int ROWB = CHUNK * 2;
  static constexpr int ATOMB = 8 * ROWB;
  static constexpr int CHUNKB = kBM * ROWB;
  static constexpr int TILEB = kBM * D * 2;
  static constexpr uint64_t LAYOUT = ROWB == 128 ? 2 : 4;  // 128B / 64B swizzle
  // P / dS tiles: 128 rows x 128 keys bf16 as two 64-key chunks, 128B swizzle
  static constexpr int PCHUNKB = kBM * 128;
  static constexpr int PTILEB = 2 * PCHUNKB;
  // Q and dO blocks: double-buffered (the next query block loads during
  // the current one) where shared memory has room
  static constexpr int QB = 6 * TILEB + 2 * PTILEB + 4096 <= 232448 - 1024 ? 2 : 1;
  // P and dS in tiles of their own (one pass computes both, and all the
  // products of a block issue together) where shared memory has room; else
  // dS reuses P's tiles after the dV products
  static constexpr bool MERGED = 2 * TILEB + 2 * QB * TILEB + 4 * PTILEB + 2048 <= 232448 - 1024;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILEB;
  static constexpr int Q_OFF = V_OFF + TILEB;        // QB buffers
  static constexpr int DO_OFF = Q_OFF + QB * TILEB;  // QB buffers
  static constexpr int HI_OFF = DO_OFF + QB * TILEB;
  static constexpr int LO_OFF = HI_OFF + PTILEB;
  static constexpr int DHI_OFF = MERGED ? LO_OFF + PTILEB : HI_OFF;  // dS tiles
  static constexpr int DLO_OFF = MERGED ? DHI_OFF + PTILEB : LO_OFF;
  // bias variant: the CTA's 32 position and 32 time gradient sums, by the
  // lane that holds the bucket's table entry
  static constexpr int HIST_OFF = (MERGED ? DLO_OFF : LO_OFF) + PTILEB;
  static constexpr int HISTB = RAB ? 64 * 4 : 0;
  static constexpr int BAR_OFF = HIST_OFF + HISTB;
  // S / dP done; the other products done; drain
  static constexpr int B_KV = 0, B_QD = 1 /* [QB] */, B_SDP = 1 + QB, B_PROD = 2 + QB,
                       B_DRAIN = 3 + QB, NBARS = 4 + QB;
  static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // tmem base, abort flag
  static constexpr int USED = MISC_OFF + 16;
  static constexpr int SMEM = ((USED + 1023) / 1024) * 1024 + 1024;  // + realignment slack
  // more than half an SM's shared memory: one CTA (and one TMEM allocation) per SM
  static constexpr int SMEM_LAUNCH = SMEM < 120 * 1024 ? 120 * 1024 : SMEM;
  static_assert(SMEM <= 232448, "shared memory budget");
  // TMEM columns: S at 0, dP at 128, dV at 256, dK at 256 + D, dQ_part at
  // 256 + 2 D where TMEM has room (d <= 64; the next block's S and dP then
  // run under the dQ staging), else over S
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 256 + D;
  static constexpr uint32_t DQ_COL = 256 + 3 * D <= (int)kTmemCols ? 256 + 2 * D : 0;
  static_assert(256 + 2 * D <= (int)kTmemCols, "TMEM budget");
  static_assert(!MERGED || DQ_COL != 0, "the pipelined path keeps dQ_part apart from S");
};

// Two warpgroups: warps w and w + 4 share TMEM lanes 32 (w % 4) ..; each
// takes half of a block's key columns (and half of the d columns).
constexpr int kBwdThreads = 256;

// Instruction descriptor with both operand majors: A MN-major at bit 15.
__host__ __device__ constexpr uint32_t make_idesc_ab(int M, int N, int a_mn_major, int b_mn_major) {
  return make_idesc(M, N, b_mn_major) | ((uint32_t)a_mn_major << 15);
}

// Byte offset of element (row r, key c) in a 128 x 128 bf16 tile stored as
// two 64-key chunks with the 128-byte swizzle: within a chunk row r is 128
// bytes at r * 128, and its 16-byte granule g sits at granule g ^ (r % 8).
__device__ __forceinline__ uint32_t ptile_off(int r, int c) {
  return (uint32_t)((c >> 6) * (kBM * 128) + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) +
                    ((c & 7) << 1));
}

struct BwdBlock {
  int s0, n, h, kt;
};

template <int D, bool RAB>
__global__ void __launch_bounds__(kBwdThreads, 1)
    hstu_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
  using C = BCfg<D, RAB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127;  // TMEM lane: the query row (or key row at the item's end)
  const int wg = tid >> 7;    // column half
  const uint32_t bars = base + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };

  if constexpr (RAB) {
    float* hist = reinterpret_cast<float*>(smem + C::HIST_OFF);
    for (int i = tid; i < 64; i += kBwdThreads) hist[i] = 0.f;
  }
  if (tid == 0) {
    for (int i = 0; i < C::NBARS; ++i) mbar_init(bar(i), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_do)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_dq)) : "memory");
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
  const uint32_t lane_tm = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's TMEM lanes
  const WaitCtx w{a.timeout_ns, abort_flag};

  constexpr uint32_t IDESC_S = make_idesc(kBM, kBN, 0);
  constexpr uint32_t IDESC_T = make_idesc_ab(kBM, D, 1, 1);   // dV, dK: A and B MN-major
  constexpr uint32_t IDESC_DQ = make_idesc_ab(kBM, D, 0, 1);  // dQ: A K-major, B MN-major
  constexpr int DSTEPS = D / 16, SPC = C::CHUNK / 16;
  const uint64_t q_kmaj0 = smem_desc(base + C::Q_OFF, 16, C::ATOMB, C::LAYOUT);
  const uint64_t k_kmaj = smem_desc(base + C::K_OFF, 16, C::ATOMB, C::LAYOUT);
  const uint64_t v_kmaj = smem_desc(base + C::V_OFF, 16, C::ATOMB, C::LAYOUT);
  const uint64_t do_kmaj0 = smem_desc(base + C::DO_OFF, 16, C::ATOMB, C::LAYOUT);
  const uint64_t q_mn0 = smem_desc(base + C::Q_OFF, C::CHUNKB, C::ATOMB, C::LAYOUT);
  const uint64_t k_mn = smem_desc(base + C::K_OFF, C::CHUNKB, C::ATOMB, C::LAYOUT);
  const uint64_t do_mn0 = smem_desc(base + C::DO_OFF, C::CHUNKB, C::ATOMB, C::LAYOUT);
  auto buf_desc = [&](uint64_t d0, int qb) { return d0 + (uint64_t)((qb * C::TILEB) >> 4); };
  const uint64_t hi_mn = smem_desc(base + C::HI_OFF, C::PCHUNKB, 1024, 2);
  const uint64_t lo_mn = smem_desc(base + C::LO_OFF, C::PCHUNKB, 1024, 2);
  const uint64_t dhi_mn = smem_desc(base + C::DHI_OFF, C::PCHUNKB, 1024, 2);
  const uint64_t dlo_mn = smem_desc(base + C::DLO_OFF, C::PCHUNKB, 1024, 2);
  const uint64_t dhi_kmaj = smem_desc(base + C::DHI_OFF, 16, 1024, 2);
  const uint64_t dlo_kmaj = smem_desc(base + C::DLO_OFF, 16, 1024, 2);

  uint32_t ph_kv = 0, ph_qd[2] = {0, 0}, ph_sdp = 0, ph_prod = 0;
  uint32_t qiter = 0;  // query blocks done by this CTA: buffer qiter % QB
  bool ok = true;
  // every thread waits (bounded); the CTA continues only if all succeeded
  auto wait_all = [&](int b, uint32_t& ph, int site) -> bool {
    const bool mine = wait_one(bar(b), ph, w, site);
    ph ^= 1u;
    return !__syncthreads_or(mine ? 0 : 1);
  };
  auto load_tile = [&](const CUtensorMap* map, int off, int b, int h, int row0) {
#pragma unroll
    for (int ch = 0; ch < C::NCHUNK; ++ch)
      tma_load_3d(base + off + ch * C::CHUNKB, map, bar(b), ch * C::CHUNK, h, row0);
  };
  // S or dP = X Y^T over d: both K-major
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
  // T += tile^T B over the 128 query rows: tile MN-major (M = keys), B MN-major
  auto mma_tt = [&](uint32_t d_col, uint64_t tile_mn, uint64_t bd, bool first) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t ad = tile_mn + (uint64_t)((kk * 2048) >> 4);
      const uint64_t b2 = bd + (uint64_t)((kk * 2 * C::ATOMB) >> 4);
      if (first && kk == 0)
        mma_ss_c<0>(tmem + d_col, ad, b2, IDESC_T);
      else
        mma_ss_c<1>(tmem + d_col, ad, b2, IDESC_T);
    }
  };
  // dQ_part (+)= tile K over the 128 keys: tile K-major, K MN-major
  auto mma_dq = [&](uint64_t tile_k, bool first) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t ad = tile_k + (uint64_t)(((kk >> 2) * C::PCHUNKB + (kk & 3) * 32) >> 4);
      const uint64_t b2 = k_mn + (uint64_t)((kk * 2 * C::ATOMB) >> 4);
      if (first && kk == 0)
        mma_ss_c<0>(tmem + C::DQ_COL, ad, b2, IDESC_DQ);
      else
        mma_ss_c<1>(tmem + C::DQ_COL, ad, b2, IDESC_DQ);
    }
  };
  // Element (row r = tid, key c) of the current block pair is kept.
  const float alpha = a.alpha, inv_n = a.inv_n;
  // write 8 keys (c8 .. c8 + 7) of this thread's row, split into hi and lo
  auto put8 = [&](uint8_t* hi_tile, uint8_t* lo_tile, int c8, const float (&v)[8]) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t ph = pack_bf16x2(v[2 * m], v[2 * m + 1]);
      const float r0 = v[2 * m] - __uint_as_float(ph << 16);
      const float r1 = v[2 * m + 1] - __uint_as_float(ph & 0xFFFF0000u);
      hw[m] = ph;
      lw[m] = pack_bf16x2(r0, r1);
    }
    const uint32_t o = ptile_off(row, c8);
    *reinterpret_cast<uint4*>(hi_tile + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(lo_tile + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  };

  // The bias (variant RAB): lane l holds the tables' entries of bucket
  // 31 - l (clamped), so a lookup is one shuffle from lane rab_lane(delta).
  // The current item's history length (its length, without candidates)
  // and length.  A row's kept keys in the item's block: c < cmax (causal);
  // with candidates, c < cm or c == dg (dg = -1 for a history row).
  int item_hist = 0, item_n = 0;
  struct RowMask {
    int cmax, cm, dg;
    bool ok;
  };
  RabRow rr{};
  if constexpr (RAB) {
    const int bl = 31 - lane;
    rr.pos_l = __ldg(a.rab_pos + (bl < a.rab_npos - 1 ? bl : a.rab_npos - 1));
    rr.time_l = __ldg(a.rab_time + (bl < a.rab_ntime - 1 ? bl : a.rab_ntime - 1));
  }
  float* hp = reinterpret_cast<float*>(smem + C::HIST_OFF);  // the CTA's sums
  float* ht = hp + 32;
  // each thread's running sums of dS and the buckets (as lanes) they belong
  // to, carried over chunks and blocks: added into the CTA's sums when the
  // bucket changes, and at the end
  float run_p = 0.f, run_t = 0.f;
  int cur_p = 0, cur_t = 0;
  // a running sum leaves bucket cur for nxt: where the whole warp leaves one
  // bucket together (a bucket edge between chunks, a jump in time), its 32
  // sums add as one; else each lane that leaves adds its own.  The warp is
  // converged here.
  auto flush_warp = [&](float* h, int& cur, float& sum, int nxt) {
    const bool mine = nxt != cur;
    const unsigned m = __ballot_sync(0xffffffffu, mine);
    if (m) {  // m is the same in every lane: the warp stays converged
      const int c0 = __shfl_sync(0xffffffffu, cur, 0);
      const bool one = __all_sync(0xffffffffu, cur == c0);
      if (m == 0xffffffffu && one) {
        float v = sum;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) atomicAdd(h + c0, v);
      } else if (mine) {
        atomicAdd(h + cur, sum);
      }
      if (mine) {
        sum = 0.f;
        cur = nxt;
      }
    }
  };
  // A 32-key chunk of this warp's 32 rows, for the bias.  Along the keys a
  // row's position bucket never grows, nor does its time bucket when the
  // chunk's timestamps are in order.  So a part is one of:
  //   0  constant over the chunk for every row: one value per row;
  //   1  at most two adjacent buckets per row: the row's first key of the
  //      lower bucket (kbp, kbt; 32 if none) decides between two values;
  //   2  anything else (a diagonal chunk, out-of-order times): a lookup per
  //      key.
  // Modes are warp-uniform; a chunk with a part in mode 2 takes mode 2 for
  // both.
  struct BRab {
    float p0, p1, t0, t1;  // the row's entries of its first and second buckets
    uint32_t pk;           // lp0 | lt0 << 5 | kbp << 10 | kbt << 16 | pm << 22 | tm << 24
  };
  // the chunk of keys j0 .. j0 + 31, key j0 + lane's timestamp ts_key,
  // ord: those are in order; rr holds the row's position and timestamp
  auto prep_chunk = [&](int j0, int ts_key, bool ord) -> BRab {
    const int d0 = rr.pe_i - j0;
    const int lp0 = rab_lane(d0), lp1 = rab_lane(d0 - 31);
    const int ts_first = __shfl_sync(0xffffffffu, ts_key, 0);
    const int ts_last = __shfl_sync(0xffffffffu, ts_key, 31);
    const int lt0 = rab_lane(rr.ts_i - ts_first), lt1 = rab_lane(rr.ts_i - ts_last);
    const int dp = lp1 - lp0, dt = lt1 - lt0;
    const bool p_fix = __all_sync(0xffffffffu, dp == 0);
    const bool p_two = __all_sync(0xffffffffu, dp <= 1);
    const bool t_fix = __all_sync(0xffffffffu, dt == 0);
    const bool t_two = __all_sync(0xffffffffu, dt >= 0 && dt <= 1);
    int pm = p_fix ? 0 : (p_two ? 1 : 2);
    int tm = !ord ? 2 : (t_fix ? 0 : (t_two ? 1 : 2));
    if (pm == 2 || tm == 2) pm = tm = 2;
    // position: bucket 31 - lp0 holds deltas >= 2^(31 - lp0) - 1, so the
    // first key below it is d0 + 2 - 2^(31 - lp0)
    const int kbp = pm == 1 && dp == 1 ? d0 + 2 - (1 << (31 - lp0)) : 32;
    // time: keys in order; the first bucket (>= 1 when it changes) holds
    // the keys with ts <= ts_i + 1 - 2^(31 - lt0): count them by bisection
    int kbt = 32;
    if (tm == 1) {  // warp-uniform
      const long long thr = (long long)rr.ts_i + 1 - (1LL << (31 - lt0));
      int cnt = 0;
#pragma unroll
      for (int st = 16; st > 0; st >>= 1) {
        const int probe = __shfl_sync(0xffffffffu, ts_key, cnt + st - 1);
        cnt += (long long)probe <= thr ? st : 0;
      }
      const int probe = __shfl_sync(0xffffffffu, ts_key, cnt);
      cnt += (long long)probe <= thr ? 1 : 0;
      if (dt == 1) kbt = cnt;
    }
    BRab q;
    q.p0 = __shfl_sync(0xffffffffu, rr.pos_l, lp0);
    q.p1 = __shfl_sync(0xffffffffu, rr.pos_l, lp0 < 31 ? lp0 + 1 : 31);
    q.t0 = __shfl_sync(0xffffffffu, rr.time_l, lt0);
    q.t1 = __shfl_sync(0xffffffffu, rr.time_l, lt0 < 31 ? lt0 + 1 : 31);
    q.pk = (uint32_t)lp0 | ((uint32_t)lt0 << 5) | ((uint32_t)kbp << 10) | ((uint32_t)kbt << 16) |
           ((uint32_t)pm << 22) | ((uint32_t)tm << 24);
    return q;
  };
  // One 32-key chunk c of this thread's row: MODE 0 writes P and dS, 1 P,
  // 2 dS; PM and TM are the bias parts' modes.  The dS goes into the running
  // sums: in modes 0 and 1 as at most two sums per part at the chunk's end;
  // in mode 2 a running sum moves on where the row's bucket changes.
  auto chunk = [&](auto pm_t, auto tm_t, auto mode_t, auto cm_t, int c, const uint32_t (&sr)[32],
                   const uint32_t (&pr)[32], const BRab& q, int ts_key, int j0,
                   const RowMask& rm) {
    constexpr int PM = decltype(pm_t)::value;
    constexpr int TM = decltype(tm_t)::value;
    constexpr int MODE = decltype(mode_t)::value;
    constexpr bool CM = decltype(cm_t)::value;  // the chunk holds candidate keys
    constexpr bool GEN = PM == 2;
    [[maybe_unused]] const int lp0 = q.pk & 31, lt0 = (q.pk >> 5) & 31;
    [[maybe_unused]] const int kbp = (q.pk >> 10) & 63, kbt = (q.pk >> 16) & 63;
    float& sp = run_p;
    float& st = run_t;
    int& cp = cur_p;
    int& ct = cur_t;
    if constexpr (RAB && MODE != 1 && !GEN) {
      // the running sums move to the chunk's first buckets
      flush_warp(hp, cp, sp, lp0);
      flush_warp(ht, ct, st, lt0);
    }
    [[maybe_unused]] float tot = 0.f, ap1 = 0.f, at1 = 0.f;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      // eight keys without a branch (their lookups and SiLUs overlap), then
      // their dS into the sums
      float vp[8], vs[8];
      [[maybe_unused]] int lpv[8], ltv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int k = 8 * g + e;
        const int col = 32 * c + k;
        const bool keep = CM ? rm.ok && (col < rm.cm || col == rm.dg) : rm.ok && col < rm.cmax;
        float x = alpha * __uint_as_float(sr[k]);
        if constexpr (RAB) {
          if constexpr (GEN) {
            const int jk = j0 + k;  // every candidate sits at position hist
            lpv[e] = rab_lane(rr.pe_i - (jk < item_hist ? jk : item_hist));
            ltv[e] = rab_lane(rr.ts_i - __shfl_sync(0xffffffffu, ts_key, k));
            x += __shfl_sync(0xffffffffu, rr.pos_l, lpv[e]) +
                 __shfl_sync(0xffffffffu, rr.time_l, ltv[e]);
          } else {
            const float bp = (PM == 1 && k >= kbp) ? q.p1 : q.p0;
            const float bt = (TM == 1 && k >= kbt) ? q.t1 : q.t0;
            x += bp + bt;
          }
        }
        const float sg = fmaf(0.5f, tanh_approx(0.5f * x), 0.5f);
        const float isg = inv_n * sg;
        if constexpr (MODE != 2) vp[e] = keep ? isg * x : 0.0f;
        if constexpr (MODE != 1)
          vs[e] = keep ? isg * fmaf(x, 1.0f - sg, 1.0f) * __uint_as_float(pr[k]) : 0.0f;
      }
      if constexpr (MODE != 2) put8(smem + C::HI_OFF, smem + C::LO_OFF, 32 * c + 8 * g, vp);
      if constexpr (MODE != 1) put8(smem + C::DHI_OFF, smem + C::DLO_OFF, 32 * c + 8 * g, vs);
      if constexpr (RAB && MODE != 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int k = 8 * g + e;
          if constexpr (GEN) {
            if (lpv[e] != cp) {  // rows cross a position edge at different keys
              atomicAdd(hp + cp, sp);
              sp = 0.f;
              cp = lpv[e];
            }
            sp += vs[e];
            flush_warp(ht, ct, st, ltv[e]);
            st += vs[e];
          } else {
            tot += vs[e];
            if constexpr (PM == 1) ap1 += k >= kbp ? vs[e] : 0.0f;
            if constexpr (TM == 1) at1 += k >= kbt ? vs[e] : 0.0f;
          }
        }
      }
    }
    if constexpr (RAB && MODE != 1 && !GEN) {
      if constexpr (PM == 0) {
        sp += tot;
      } else {
        sp += tot - ap1;
        flush_warp(hp, cp, sp, kbp < 32 ? lp0 + 1 : lp0);
        sp += ap1;
      }
      if constexpr (TM == 0) {
        st += tot;
      } else {
        st += tot - at1;
        flush_warp(ht, ct, st, kbt < 32 ? lt0 + 1 : lt0);
        st += at1;
      }
    }
  };
  using I0 = std::integral_constant<int, 0>;
  using I1 = std::integral_constant<int, 1>;
  using I2 = std::integral_constant<int, 2>;
  using CM0 = std::false_type;
  using CM1 = std::true_type;
  // the bias's view of this warp's two key chunks of the current item:
  // the timestamps (lane = key) and whether they are in order; and of the
  // current query block, each chunk's modes and values
  int ts_key0 = 0, ts_key1 = 0;
  bool ord0 = true, ord1 = true;
  BRab q0{}, q1{};
  // the timestamp of this thread's row of query block qt (a row past the
  // sequence reads the last token; its results are never kept)
  auto row_ts = [&](int qt) -> int {
    if constexpr (RAB) {
      const int i = kBM * qt + row;
      return __ldg(rr.ts + (i < rr.last ? i : rr.last));
    } else {
      return 0;
    }
  };
  // the two chunks' modes and values for query block qt, whose row
  // timestamp ts_i was loaded ahead
  auto prep = [&](int qt, int ts_i, int kbase) {
    if constexpr (RAB) {
      const int i = kBM * qt + row;
      rr.pe_i = i < item_hist ? i : item_hist;
      rr.ts_i = ts_i;
      q0 = prep_chunk(kbase + 64 * wg, ts_key0, ord0);
      q1 = prep_chunk(kbase + 64 * wg + 32, ts_key1, ord1);
    }
  };
  // the pass of MODE over this warpgroup's two chunks of query block qt
  auto pass = [&](auto mode_t, int kbase, const RowMask& rm) {
#pragma unroll 1
    for (int c = 2 * wg; c < 2 * wg + 2; ++c) {
      uint32_t sr[32], pr[32];
      tmem_ld32(lane_tm + C::S_COL + 32u * c, sr);
      if constexpr (decltype(mode_t)::value != 1) tmem_ld32(lane_tm + C::DP_COL + 32u * c, pr);
      const int j0 = kbase + 32 * c;
      // a chunk holding candidate keys (warp-uniform) takes the candidate
      // mask and, with the bias, the per-key lookups
      const bool cand = item_hist < item_n && j0 + 31 >= item_hist;
      if constexpr (RAB) {
        const BRab q = (c & 1) ? q1 : q0;
        const int tsk = (c & 1) ? ts_key1 : ts_key0;
        const uint32_t modes = (q.pk >> 22) & 15u;  // pm | tm << 2, warp-uniform
        if (cand)
          chunk(I2{}, I2{}, mode_t, CM1{}, c, sr, pr, q, tsk, j0, rm);
        else if (modes == 0u)
          chunk(I0{}, I0{}, mode_t, CM0{}, c, sr, pr, q, tsk, j0, rm);
        else if (modes == 1u)
          chunk(I1{}, I0{}, mode_t, CM0{}, c, sr, pr, q, tsk, j0, rm);
        else if (modes == 4u)
          chunk(I0{}, I1{}, mode_t, CM0{}, c, sr, pr, q, tsk, j0, rm);
        else if (modes == 5u)
          chunk(I1{}, I1{}, mode_t, CM0{}, c, sr, pr, q, tsk, j0, rm);
        else
          chunk(I2{}, I2{}, mode_t, CM0{}, c, sr, pr, q, tsk, j0, rm);
      } else {
        const BRab q{};
        if (cand)
          chunk(I0{}, I0{}, mode_t, CM1{}, c, sr, pr, q, 0, j0, rm);
        else
          chunk(I0{}, I0{}, mode_t, CM0{}, c, sr, pr, q, 0, j0, rm);
      }
    }
  };

  // the CTA's items: a host-built schedule's range, else every grid-th item
  const int idx0 = a.cta_first ? __ldg(&a.cta_first[blockIdx.x]) : (int)blockIdx.x;
  const int idx_end = a.cta_first ? __ldg(&a.cta_first[blockIdx.x + 1]) : a.n_items;
  const int idx_step = a.cta_first ? 1 : (int)gridDim.x;
  for (int idx = idx0; ok && idx < idx_end; idx += idx_step) {
    const Item it = __ldg(&a.items[idx]);
    const BwdBlock b{it.x, it.y, it.z, it.w};
    item_hist = a.item_hist ? __ldg(a.item_hist + idx) : b.n;
    item_n = b.n;
    // a key block of candidates only is seen by its own rows: the diagonal
    // query block alone
    const int nq = kBN * b.kt >= item_hist ? b.kt + 1 : (b.n + kBM - 1) / kBM;
    const int key_rows = b.n - kBN * b.kt;  // keys of the block that exist (>= 1)
    if (tid == 0) {
      mbar_arrive_expect_tx(bar(C::B_KV), 2 * C::TILEB);
      load_tile(&tm_k, C::K_OFF, C::B_KV, b.h, b.s0 + kBN * b.kt);
      load_tile(&tm_v, C::V_OFF, C::B_KV, b.h, b.s0 + kBN * b.kt);
    }
    auto load_qd = [&](int qb, int qt) {
      mbar_arrive_expect_tx(bar(C::B_QD + qb), 2 * C::TILEB);
      load_tile(&tm_q, C::Q_OFF + qb * C::TILEB, C::B_QD + qb, b.h, b.s0 + kBM * qt);
      load_tile(&tm_do, C::DO_OFF + qb * C::TILEB, C::B_QD + qb, b.h, b.s0 + kBM * qt);
    };
    // row tid of query block qt sees key c of block kt iff both exist and
    // the key is not after the row; with candidates, iff also the key is in
    // the history or is the row's own
    auto mask_of = [&](int qt) -> RowMask {
      const int row_i = kBM * qt + row;    // sequence-local query
      const int lim = row_i - kBN * b.kt;  // keys c <= lim are not after the row
      RowMask m;
      m.cmax = key_rows < lim + 1 ? key_rows : lim + 1;  // causal: kept keys c < cmax
      m.ok = row_i < b.n;
      const int hl = item_hist - kBN * b.kt;  // keys c < hl are history
      m.cm = m.cmax < hl ? m.cmax : hl;
      m.dg = row_i >= item_hist ? lim : -1;
      return m;
    };
    // alpha dQ_part of block qt (TMEM columns DQ_COL) staged over the P
    // tiles as 128B-swizzled fp32 boxes of 32 columns, then added into the
    // accumulator by bulk tensor reductions.  Rows past the sequence carry
    // dS = 0, so their parts are exactly zero; rows past the tensor are
    // clipped by the copy.
    auto put_dq = [&](int qt) {
#pragma unroll 1
      for (int c = wg; c < D / 32; c += 2) {
        uint32_t r[32];
        tmem_ld32(lane_tm + C::DQ_COL + 32u * c, r);
        uint8_t* box = smem + C::HI_OFF + c * (kBM * 128);
#pragma unroll
        for (int g = 0; g < 8; ++g)
          *reinterpret_cast<float4*>(box + row * 128 + ((g ^ (row & 7)) << 4)) =
              make_float4(alpha * __uint_as_float(r[4 * g]), alpha * __uint_as_float(r[4 * g + 1]),
                          alpha * __uint_as_float(r[4 * g + 2]), alpha * __uint_as_float(r[4 * g + 3]));
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
          asm volatile(
              "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
              " [%0, {%1, %2, %3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(&tm_dq)),
              "r"(32 * c), "r"(b.h), "r"(b.s0 + kBM * qt), "r"(base + C::HI_OFF + c * (kBM * 128))
              : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    };
    auto issue_sdp = [&](int qb) {
      tc_fence_after();
      mma_xyt(C::S_COL, buf_desc(q_kmaj0, qb), k_kmaj);
      mma_xyt(C::DP_COL, buf_desc(do_kmaj0, qb), v_kmaj);
      mma_commit(bar(C::B_SDP));
    };
    if constexpr (RAB) {
      rr.ts = a.rab_ts + b.s0;
      rr.last = b.n - 1;
      const int j0 = kBN * b.kt + 64 * wg + lane;
      ts_key0 = __ldg(rr.ts + (j0 < rr.last ? j0 : rr.last));
      ts_key1 = __ldg(rr.ts + (j0 + 32 < rr.last ? j0 + 32 : rr.last));
      // every lane takes part in the shuffles (none inside a condition)
      const int nx0 = __shfl_down_sync(0xffffffffu, ts_key0, 1);
      const int nx1 = __shfl_down_sync(0xffffffffu, ts_key1, 1);
      ord0 = __all_sync(0xffffffffu, lane == 31 || ts_key0 <= nx0);
      ord1 = __all_sync(0xffffffffu, lane == 31 || ts_key1 <= nx1);
      prep(b.kt, row_ts(b.kt), kBN * b.kt);
    }
    if constexpr (C::MERGED && C::QB == 2) {
      // Pipelined: while block qt's products run, block qt + 1's S and dP
      // follow them on the tensor cores, and the threads stage qt's dQ.
      const int qb0 = (int)(qiter % C::QB);
      if (tid == 0) {
        load_qd(qb0, b.kt);
        if (b.kt + 1 < nq) load_qd(qb0 ^ 1, b.kt + 1);
      }
      if (!(ok = wait_all(C::B_KV, ph_kv, kSiteKFull))) break;
      if (tid == 0 && (ok = wait_one(bar(C::B_QD + qb0), ph_qd[qb0], w, kSiteQFull))) {
        ph_qd[qb0] ^= 1u;
        issue_sdp(qb0);
      }
      for (int qt = b.kt; qt < nq; ++qt, ++qiter) {
        const bool first = qt == b.kt;
        const int qb = (int)(qiter % C::QB);
        // the previous block's dQ reductions have read their staging (the P
        // tiles, rewritten below)
        if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        if (!(ok = wait_all(C::B_SDP, ph_sdp, kSiteSFull))) break;
        tc_fence_after();
        const RowMask rm = mask_of(qt);
        // P and dS in one pass over this warpgroup's two 32-key chunks
        pass(std::integral_constant<int, 0>{}, kBN * b.kt, rm);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncthreads();  // S and dP read, the tiles written
        const int ts_next = row_ts(qt + 1);  // loads under the product issue
        if (tid == 0) {
          tc_fence_after();
          const uint64_t q_mn = buf_desc(q_mn0, qb), do_mn = buf_desc(do_mn0, qb);
          mma_tt(C::DV_COL, hi_mn, do_mn, first);
          mma_tt(C::DV_COL, lo_mn, do_mn, false);
          mma_tt(C::DK_COL, dhi_mn, q_mn, first);
          mma_tt(C::DK_COL, dlo_mn, q_mn, false);
          mma_dq(dhi_kmaj, true);
          mma_dq(dlo_kmaj, false);
          mma_commit(bar(C::B_PROD));
          // the next block's S and dP, once its Q and dO have landed
          if (qt + 1 < nq && (ok = wait_one(bar(C::B_QD + (qb ^ 1)), ph_qd[qb ^ 1], w, kSiteQFull))) {
            ph_qd[qb ^ 1] ^= 1u;
            issue_sdp(qb ^ 1);
          }
        }
        // the next block's bias parts while the products run
        if (qt + 1 < nq) prep(qt + 1, ts_next, kBN * b.kt);
        if (!(ok = wait_all(C::B_PROD, ph_prod, kSiteVFull))) break;
        tc_fence_after();
        // buffer qb is free (its last readers were these products): the
        // block after next loads into it
        if (tid == 0 && qt + 2 < nq) load_qd(qb, qt + 2);
        put_dq(qt);
      }
    } else {
      // One block at a time: P and dS in one pass where they have tiles of
      // their own, else P, dV, then dS in P's tiles.
      if (tid == 0) load_qd(0, b.kt);
      if (!(ok = wait_all(C::B_KV, ph_kv, kSiteKFull))) break;
      for (int qt = b.kt; qt < nq; ++qt, ++qiter) {
        const bool first = qt == b.kt;
        if (!first) prep(qt, row_ts(qt), kBN * b.kt);  // under the waits below
        if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        if (!(ok = wait_all(C::B_QD, ph_qd[0], kSiteQFull))) break;
        const uint64_t q_mn = buf_desc(q_mn0, 0), do_mn = buf_desc(do_mn0, 0);
        if (tid == 0) issue_sdp(0);
        if (!(ok = wait_all(C::B_SDP, ph_sdp, kSiteSFull))) break;
        tc_fence_after();
        const RowMask rm = mask_of(qt);
        if constexpr (C::MERGED) {
          pass(std::integral_constant<int, 0>{}, kBN * b.kt, rm);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_before();
          __syncthreads();
          if (tid == 0) {
            tc_fence_after();
            mma_tt(C::DV_COL, hi_mn, do_mn, first);
            mma_tt(C::DV_COL, lo_mn, do_mn, false);
            mma_tt(C::DK_COL, dhi_mn, q_mn, first);
            mma_tt(C::DK_COL, dlo_mn, q_mn, false);
            mma_dq(dhi_kmaj, true);
            mma_dq(dlo_kmaj, false);
            mma_commit(bar(C::B_PROD));
          }
        } else {
          // 2. P
          pass(std::integral_constant<int, 1>{}, kBN * b.kt, rm);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_before();
          __syncthreads();
          // 3. dV += P^T dO
          if (tid == 0) {
            tc_fence_after();
            mma_tt(C::DV_COL, hi_mn, do_mn, first);
            mma_tt(C::DV_COL, lo_mn, do_mn, false);
            mma_commit(bar(C::B_PROD));
          }
          if (!(ok = wait_all(C::B_PROD, ph_prod, kSiteOFull))) break;
          tc_fence_after();
          // 4. dS, into the same tiles (the dV products are done)
          pass(std::integral_constant<int, 2>{}, kBN * b.kt, rm);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_before();
          __syncthreads();
          // 5. dK += dS^T Q, dQ_part = dS K
          if (tid == 0) {
            tc_fence_after();
            mma_tt(C::DK_COL, dhi_mn, q_mn, first);
            mma_tt(C::DK_COL, dlo_mn, q_mn, false);
            mma_dq(dhi_kmaj, true);
            mma_dq(dlo_kmaj, false);
            mma_commit(bar(C::B_PROD));
          }
        }
        if (!(ok = wait_all(C::B_PROD, ph_prod, kSiteVFull))) break;
        tc_fence_after();
        // 6. the single Q / dO buffer is free: the next block loads under the staging
        if (tid == 0 && qt + 1 < nq) load_qd(0, qt + 1);
        put_dq(qt);
      }
    }
    if (!ok) break;
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
    tc_fence_before();
    __syncthreads();  // dV and dK read before the next item overwrites them
  }
  if (!ok && tid == 0) {
    // drain: a commit arrives once every product issued before it is done
    mma_commit(bar(C::B_DRAIN));
    wait_drain(bar(C::B_DRAIN), 0);
  }
  // the last reductions have finished before the CTA (and its shared memory) goes
  if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  if constexpr (RAB) {
    // the running sums into the CTA's, those into the tables' gradients:
    // lane sum L holds bucket min(31 - L, entries - 1)
    atomicAdd(hp + cur_p, run_p);
    atomicAdd(ht + cur_t, run_t);
    __syncthreads();
    if (ok && tid < 64) {
      const float sum = hp[tid];
      const int L = tid & 31;
      if (sum != 0.f) {
        if (tid < 32)
          atomicAdd(a.dpos + (31 - L < a.rab_npos - 1 ? 31 - L : a.rab_npos - 1), sum);
        else
          atomicAdd(a.dtime + (31 - L < a.rab_ntime - 1 ? 31 - L : a.rab_ntime - 1), sum);
      }
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

// dQ = bf16(acc): the accumulated fp32 gradient, rounded once.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* acc, uint16_t* dq, long long n8) {
  for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < n8; i += (long long)gridDim.x * 256) {
    const float4 x0 = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 x1 = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    reinterpret_cast<uint4*>(dq)[i] = make_uint4(pack_bf16x2(x0.x, x0.y), pack_bf16x2(x0.z, x0.w),
                                                 pack_bf16x2(x1.x, x1.y), pack_bf16x2(x1.z, x1.w));
  }
}

template <int D, bool RAB>
cudaError_t launch_bwd_dr(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                          cudaStream_t stream) {
  using C = BCfg<D, RAB>;
  static_assert(D / 32 * kBM * 128 <= 2 * C::PTILEB, "dQ staging fits the P tiles");
  cudaError_t e = cudaFuncSetAttribute(hstu_bwd_kernel<D, RAB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_LAUNCH);
  if (e != cudaSuccess) return e;
  hstu_bwd_kernel<D, RAB><<<grid, kBwdThreads, C::SMEM_LAUNCH, stream>>>(tq, tk, tv, tdo, tdq, a);
  return cudaGetLastError();
}

// The transposed form (hstu_bwd_t.cuh), for d <= 64 without the bias.
template <int D>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                         cudaStream_t stream);

template <int D>
cudaError_t launch_bwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                         cudaStream_t stream) {
  cudaError_t e;
  if constexpr (D <= 64) {
    if (a.transposed)
      e = launch_bwd_t<D>(tq, tk, tv, tdo, tdq, a, grid, stream);
    else
      e = a.rab_ts ? launch_bwd_dr<D, true>(tq, tk, tv, tdo, tdq, a, grid, stream)
                   : launch_bwd_dr<D, false>(tq, tk, tv, tdo, tdq, a, grid, stream);
  } else {
    if (a.transposed) return cudaErrorInvalidValue;
    e = a.rab_ts ? launch_bwd_dr<D, true>(tq, tk, tv, tdo, tdq, a, grid, stream)
                 : launch_bwd_dr<D, false>(tq, tk, tv, tdo, tdq, a, grid, stream);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long n8 = a.total * a.heads * D / 8;
  const int cgrid = (int)std::min<long long>((n8 + 255) / 256, 4LL * 1024);
  dq_convert_kernel<<<cgrid, 256, 0, stream>>>(a.dq_acc, static_cast<uint16_t*>(a.dq), n8);
  return cudaGetLastError();
}
