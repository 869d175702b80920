// Host side of libhstu: argument validation, the longest-first work-list
// builder, launch plans, TMA tensor maps and the C ABI of include/hstu_attn.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <limits>
#include <mutex>
#include <new>
#include <vector>

#include "hstu_attn.h"
#include "hstu_internal.h"

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 4000000000ull;
unsigned long long g_timeout_ns = 0;  // 0 = not yet read from the environment
unsigned g_debug_flags = 0;
std::mutex g_mu;

unsigned long long wait_timeout_ns() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_timeout_ns == 0) {
    const char* env = std::getenv("HSTU_WAIT_TIMEOUT_NS");
    unsigned long long v = env ? std::strtoull(env, nullptr, 10) : 0ull;
    g_timeout_ns = v ? v : kDefaultTimeoutNs;
  }
  return g_timeout_ns;
}

bool supported_d(int d) { return d == 32 || d == 64 || d == 128; }

// Offsets: offsets[0] == 0, non-decreasing, every length <= max_len,
// total < 2^31.  max_len < 0 means unbounded.
int check_offsets(const int32_t* off, int batch, long long max_len) {
  if (batch < 0) return HSTU_ERR_INVALID_ARG;
  if (batch == 0) return HSTU_OK;
  if (!off || off[0] != 0) return HSTU_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b) {
    const long long len = (long long)off[b + 1] - (long long)off[b];
    if (len < 0) return HSTU_ERR_INVALID_ARG;
    if (max_len >= 0 && len > max_len) return HSTU_ERR_INVALID_ARG;
  }
  return HSTU_OK;
}

// 0 <= num_targets[b] <= n_b for every sequence.
int check_targets(const int32_t* off, const int32_t* nt, int batch) {
  for (int b = 0; b < batch; ++b)
    if (nt[b] < 0 || nt[b] > off[b + 1] - off[b]) return HSTU_ERR_INVALID_ARG;
  return HSTU_OK;
}

// Work list and (with candidates) the per-item history lengths.
int build_worklist(const int32_t* off, const int32_t* nt, int batch, int heads,
                   std::vector<hstu::Item>& items, std::vector<int32_t>& hist,
                   bool candidates_only = false) {
  try {
    items.resize((size_t)hstu::count_items(off, batch, heads));
    if (nt) {
      hist.resize(items.size());
      hstu::fill_items_targets(off, nt, batch, heads, items.data(), hist.data());
      if (candidates_only) {
        // keep the query blocks that hold a candidate row (rows hist .. n-1):
        // qt >= hist / 128, with at least one candidate; the order stays
        size_t m = 0;
        for (size_t i = 0; i < items.size(); ++i) {
          const int n = items[i].y, qt = items[i].w, hs = hist[i];
          if (hs < n && qt >= hs / HSTU_BLOCK_M) {
            items[m] = items[i];
            hist[m] = hist[i];
            ++m;
          }
        }
        items.resize(m);
        hist.resize(m);
      }
    } else {
      hstu::fill_items(off, batch, heads, items.data());
    }
  } catch (const std::bad_alloc&) {
    return HSTU_ERR_NO_MEMORY;
  }
  if (items.size() > (size_t)INT32_MAX) return HSTU_ERR_INVALID_ARG;
  return HSTU_OK;
}

std::vector<hstu::Item> build_items(const int32_t* off, int batch, int heads) {
  std::vector<hstu::Item> items((size_t)hstu::count_items(off, batch, heads));
  hstu::fill_items(off, batch, heads, items.data());
  return items;
}

int check_buffers(const void* q, const void* k, const void* v, const void* out) {
  const void* ptrs[4] = {q, k, v, out};
  for (const void* p : ptrs)
    if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) return HSTU_ERR_INVALID_ARG;
  return HSTU_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// (d, heads, total) bf16 view with box (min(d,64), 1, 128) and the kernel's swizzle.
int make_map(CUtensorMap* m, const void* ptr, long long total, int heads, int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return HSTU_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)total};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2u, (cuuint64_t)heads * (cuuint64_t)d * 2u};
  const cuuint32_t box[3] = {(cuuint32_t)std::min(d, 64), 1u, (cuuint32_t)HSTU_BLOCK_M};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUtensorMapSwizzle sw = hstu::fwd_swizzle_bytes(d) == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                                   : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? HSTU_OK : HSTU_ERR_CUDA;
}

// fp32 (d, heads, total) view with box (32, 1, 128) and the 128-byte
// swizzle: the backward's dQ accumulator, target of bulk reductions.
int make_map_f32(CUtensorMap* m, const void* ptr, long long total, int heads, int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return HSTU_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)total};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 4u, (cuuint64_t)heads * (cuuint64_t)d * 4u};
  const cuuint32_t box[3] = {32u, 1u, (cuuint32_t)HSTU_BLOCK_M};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? HSTU_OK : HSTU_ERR_CUDA;
}

int device_check(int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HSTU_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return HSTU_ERR_CUDA;
  if (major != 10 || minor != 3) return HSTU_ERR_UNSUPPORTED;
  return HSTU_OK;
}

// CTAs of a launch: one per SM at most, and no more than there are items.
int grid_for(int n_items, int sms) { return std::min(n_items, sms); }

// The backward's work list in its device form: the items (and, with
// candidates, each item's history length) in schedule order, then
// first[grid + 1]; one allocation, in that order.
struct ListLayout {
  std::vector<hstu::Item> items;
  std::vector<int32_t> hist, first;
  int grid = 0;
  size_t ibytes() const { return items.size() * sizeof(hstu::Item); }
  size_t hbytes() const { return hist.size() * sizeof(int32_t); }
  size_t bytes() const { return ibytes() + hbytes() + first.size() * sizeof(int32_t); }
};

// Lays out the backward's longest-first list (items, hist: empty or one
// per item) for `sms` SMs.  Item (.., kt) walks query blocks kt .. nq - 1,
// or kt alone for a block of candidate keys.
int layout_list_bwd(const std::vector<hstu::Item>& items, const std::vector<int32_t>& hist, int sms,
                    ListLayout* L) {
  const int n = (int)items.size();
  try {
    std::vector<int32_t> cost((size_t)n), order((size_t)n);
    for (int i = 0; i < n; ++i) {
      const hstu::Item& x = items[(size_t)i];
      const int nq = (x.y + HSTU_BLOCK_M - 1) / HSTU_BLOCK_M;
      const int h = hist.empty() ? x.y : hist[(size_t)i];
      cost[(size_t)i] = HSTU_BLOCK_M * x.w >= h ? 1 : nq - x.w;
    }
    L->grid = std::max(1, std::min(n, sms));
    L->first.resize((size_t)L->grid + 1);
    hstu::schedule_items(cost.data(), n, L->grid, order.data(), L->first.data());
    L->items.resize((size_t)n);
    L->hist.resize(hist.size());
    for (int r = 0; r < n; ++r) {
      L->items[(size_t)r] = items[(size_t)order[(size_t)r]];
      if (!hist.empty()) L->hist[(size_t)r] = hist[(size_t)order[(size_t)r]];
    }
  } catch (const std::bad_alloc&) {
    return HSTU_ERR_NO_MEMORY;
  }
  return HSTU_OK;
}

// Copies a layout to dst (device, L.bytes() bytes): on stream s (from
// pageable memory each copy returns once its bytes are staged), or, with
// sync, synchronously.
cudaError_t copy_list(const ListLayout& L, char* dst, cudaStream_t s, bool sync = false) {
  auto copy = [&](void* to, const void* from, size_t n) {
    return sync ? cudaMemcpy(to, from, n, cudaMemcpyHostToDevice)
                : cudaMemcpyAsync(to, from, n, cudaMemcpyHostToDevice, s);
  };
  cudaError_t e = copy(dst, L.items.data(), L.ibytes());
  if (e == cudaSuccess && L.hbytes()) e = copy(dst + L.ibytes(), L.hist.data(), L.hbytes());
  if (e == cudaSuccess)
    e = copy(dst + L.ibytes() + L.hbytes(), L.first.data(), L.first.size() * sizeof(int32_t));
  return e;
}

int sm_count_of_current_device(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return HSTU_ERR_CUDA;
  return HSTU_OK;
}

int launch(const hstu::Item* d_items, const int32_t* d_hist, int n_items, long long total,
           int heads, int d, const void* q, const void* k, const void* v, float alpha, float inv_n,
           void* out, const hstu::NormGate* ng, cudaStream_t stream, const hstu_rab* rab = nullptr) {
  if (n_items == 0) return HSTU_OK;
  int sms = 0;
  int rc = device_check(&sms);
  if (rc != HSTU_OK) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = make_map(&tq, q, total, heads, d)) != HSTU_OK) return rc;
  if ((rc = make_map(&tk, k, total, heads, d)) != HSTU_OK) return rc;
  if ((rc = make_map(&tv, v, total, heads, d)) != HSTU_OK) return rc;
  hstu::FwdArgs a{};
  a.items = d_items;
  a.item_hist = d_hist;
  a.n_items = n_items;
  a.out = out;
  a.u = ng ? ng->u : nullptr;
  a.gamma = ng ? ng->gamma : nullptr;
  a.beta = ng ? ng->beta : nullptr;
  a.eps = ng ? ng->eps : 0.f;
  a.xs = ng ? ng->xs : nullptr;
  a.stats = ng ? ng->stats : nullptr;
  a.total = total;
  // the output-stage kernel: one warp per token, up to 8 blocks of 8 warps per SM
  a.norm_grid = (int)std::min<long long>((total + 7) / 8, 8LL * sms);
  a.rab_ts = rab ? rab->timestamps : nullptr;
  a.rab_pos = rab ? rab->pos : nullptr;
  a.rab_time = rab ? rab->time : nullptr;
  a.rab_npos = rab ? rab->num_pos : 0;
  a.rab_ntime = rab ? rab->num_time : 0;
  a.heads = heads;
  a.half_alpha = 0.5f * alpha;
  a.inv_n = inv_n;
  a.timeout_ns = wait_timeout_ns();
  {
    std::lock_guard<std::mutex> lk(g_mu);
    a.debug_flags = g_debug_flags;
  }
  const int grid = grid_for(n_items, sms);
  const cudaError_t e = hstu::launch_fwd(d, tq, tk, tv, a, grid, stream);
  if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
    return HSTU_ERR_UNSUPPORTED;
  return e == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}

// Tensor maps of the pair kernel: k with box (64, 1, 64) (each CTA holds 64
// keys of a block), v with box (d/2, 1, 128) (each CTA holds half the
// columns) and the swizzle of a d-byte row.
int make_map_pair(CUtensorMap* m, const void* ptr, long long total, int heads, int d, int box_x,
                  int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return HSTU_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)total};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2u, (cuuint64_t)heads * (cuuint64_t)d * 2u};
  const cuuint32_t box[3] = {(cuuint32_t)box_x, 1u, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUtensorMapSwizzle sw = box_x * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? HSTU_OK : HSTU_ERR_CUDA;
}

// Clusters of a pair launch: one per two SMs at most, and no more than
// there are pair items; two CTAs each.
int pair_grid_for(int n_pairs, int sms) { return 2 * std::min(n_pairs, sms / 2); }

int launch_pairs(const hstu::Item* d_pairs, int n_pairs, long long total, int heads, int d, const void* q,
                 const void* k, const void* v, float alpha, float inv_n, void* out, cudaStream_t stream) {
  if (n_pairs == 0) return HSTU_OK;
  int sms = 0;
  int rc = device_check(&sms);
  if (rc != HSTU_OK) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = make_map(&tq, q, total, heads, d)) != HSTU_OK) return rc;
  if ((rc = make_map_pair(&tk, k, total, heads, d, 64, HSTU_BLOCK_M / 2)) != HSTU_OK) return rc;
  if ((rc = make_map_pair(&tv, v, total, heads, d, d / 2, HSTU_BLOCK_M)) != HSTU_OK) return rc;
  hstu::FwdArgs a{};
  a.items = d_pairs;
  a.n_items = n_pairs;
  a.out = out;
  a.total = total;
  a.heads = heads;
  a.half_alpha = 0.5f * alpha;
  a.inv_n = inv_n;
  a.timeout_ns = wait_timeout_ns();
  {
    std::lock_guard<std::mutex> lk(g_mu);
    a.debug_flags = g_debug_flags;
  }
  const cudaError_t e = hstu::launch_fwd_pairs(d, tq, tk, tv, a, pair_grid_for(n_pairs, sms), stream);
  if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
    return HSTU_ERR_UNSUPPORTED;
  return e == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}

bool pairs_disabled() {
  std::lock_guard<std::mutex> lk(g_mu);
  return (g_debug_flags & hstu::kDebugNoPairs) != 0;
}

// Whether a plan or call picks CTA pairs by itself: not at present.  A
// pair step still gives each SM one block of SiLU work, and its issuing
// thread's serial chain per step (barrier tests, products, commits) is as
// long as the one-CTA kernel's, so pairs measured no faster on any of the
// five workloads (dense 0.268 against 0.245 ms on GB300).  Plans made with
// HSTU_PLAN_PAIRS still use them.  The waste rule below (within 15% of the
// one-CTA work list's SM-blocks) is kept for when they are.
constexpr bool kPairsByDefault = false;
bool use_pairs(const int32_t* off, int batch, int d) {
  if (!kPairsByDefault || (d != 64 && d != 128)) return false;
  long long single = 0, pair = 0;
  for (int b = 0; b < batch; ++b) {
    const long long nq = (off[b + 1] - off[b] + HSTU_BLOCK_M - 1) / HSTU_BLOCK_M;
    single += nq * (nq + 1) / 2;
    for (long long qp = 0; 2 * qp < nq; ++qp) pair += 2 * std::min(2 * qp + 2, nq);
  }
  return single > 0 && pair * 100 <= single * 115;
}

// (The plan type is defined below; make_plan and oneshot are declared here
// and defined after it.)
int make_plan(const int32_t* off, const int32_t* nt, int batch, int heads, int d, int max_seqlen,
              unsigned flags, hstu_plan** plan);
int oneshot(const void* q, const void* k, const void* v, const int32_t* offsets,
            const int32_t* num_targets, int batch, int heads, int d, int max_seqlen, float alpha,
            float inv_n, void* out, const hstu::NormGate* ng, cudaStream_t s,
            const hstu_rab* rab = nullptr);

// The bias: timestamps 4-byte aligned, tables 4-byte aligned with 1..32 entries.
int check_rab(const hstu_rab* r) {
  if (!r->timestamps || !r->pos || !r->time) return HSTU_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(r->timestamps) | reinterpret_cast<uintptr_t>(r->pos) |
       reinterpret_cast<uintptr_t>(r->time)) & 3u)
    return HSTU_ERR_INVALID_ARG;
  if (r->num_pos < 1 || r->num_pos > 32 || r->num_time < 1 || r->num_time > 32)
    return HSTU_ERR_INVALID_ARG;
  return HSTU_OK;
}

// The output stage's buffers: u and y like q, gamma and beta 16-byte
// aligned, eps finite and >= 0.
int check_norm_gate(const void* u, const float* gamma, const float* beta, float eps) {
  const void* ptrs[3] = {u, gamma, beta};
  for (const void* p : ptrs)
    if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) return HSTU_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || eps > 3.0e38f) return HSTU_ERR_INVALID_ARG;
  return HSTU_OK;
}

}  // namespace

// Entry points into the helpers above for the other host translation units.
namespace hstu {
// The work list: one item per (sequence, head, 128-row query block qt); the
// block needs key blocks 0..qt and costs qt+1.  Ordered by cost descending,
// then sequence, head, qt ascending: generated level by level (qt from the
// largest down), which is that order without a comparison sort.
long long count_items(const int32_t* off, int batch, int heads) {
  long long n = 0;
  for (int b = 0; b < batch; ++b)
    n += (long long)((off[b + 1] - off[b] + HSTU_BLOCK_M - 1) / HSTU_BLOCK_M) * heads;
  return n;
}

void fill_items(const int32_t* off, int batch, int heads, Item* dst) {
  int max_tiles = 0;
  for (int b = 0; b < batch; ++b) {
    const int tiles = (off[b + 1] - off[b] + HSTU_BLOCK_M - 1) / HSTU_BLOCK_M;
    if (tiles > max_tiles) max_tiles = tiles;
  }
  long long i = 0;
  for (int qt = max_tiles - 1; qt >= 0; --qt)
    for (int b = 0; b < batch; ++b) {
      const int n = off[b + 1] - off[b];
      if ((n + HSTU_BLOCK_M - 1) / HSTU_BLOCK_M > qt)
        for (int h = 0; h < heads; ++h) dst[i++] = make_int4(off[b], n, h, qt);
    }
}

// Pair items: (first token, length, head, qp) for qp < ceil(nq / 2), each
// walking min(2 qp + 2, nq) key blocks; (cost, b, h, qp) generated in b, h,
// qp order, then a stable sort by cost descending.
long long count_pairs(const int32_t* off, int batch, int heads) {
  long long n = 0;
  for (int b = 0; b < batch; ++b) {
    const long long nq = (off[b + 1] - off[b] + HSTU_BLOCK_M - 1) / HSTU_BLOCK_M;
    n += (nq + 1) / 2 * heads;
  }
  return n;
}

void fill_pairs(const int32_t* off, int batch, int heads, Item* dst) {
  struct Entry {
    int cost;
    Item item;
  };
  std::vector<Entry> e;
  e.reserve((size_t)count_pairs(off, batch, heads));
  for (int b = 0; b < batch; ++b) {
    const int n = off[b + 1] - off[b];
    const int nq = (n + HSTU_BLOCK_M - 1) / HSTU_BLOCK_M;
    for (int h = 0; h < heads; ++h)
      for (int qp = 0; 2 * qp < nq; ++qp)
        e.push_back(Entry{std::min(2 * qp + 2, nq), make_int4(off[b], n, h, qp)});
  }
  std::stable_sort(e.begin(), e.end(), [](const Entry& x, const Entry& y) { return x.cost > y.cost; });
  for (size_t i = 0; i < e.size(); ++i) dst[i] = e[i].item;
}

void fill_items_targets(const int32_t* off, const int32_t* num_targets, int batch, int heads,
                        Item* dst, int32_t* hist_dst) {
  // (cost, b, h, qt) generated in b, h, qt order; a stable sort by cost
  // descending then gives cost descending, then b, h, qt ascending
  struct Entry {
    int cost, hist;
    Item item;
  };
  std::vector<Entry> e;
  e.reserve((size_t)count_items(off, batch, heads));
  for (int b = 0; b < batch; ++b) {
    const int n = off[b + 1] - off[b];
    const int hist = n - num_targets[b];
    const int kh = (hist + HSTU_BLOCK_M - 1) / HSTU_BLOCK_M;
    const int tiles = (n + HSTU_BLOCK_M - 1) / HSTU_BLOCK_M;
    for (int h = 0; h < heads; ++h)
      for (int qt = 0; qt < tiles; ++qt)
        e.push_back(Entry{(qt < kh ? qt : kh) + 1, hist, make_int4(off[b], n, h, qt)});
  }
  std::stable_sort(e.begin(), e.end(), [](const Entry& x, const Entry& y) { return x.cost > y.cost; });
  for (size_t i = 0; i < e.size(); ++i) {
    dst[i] = e[i].item;
    hist_dst[i] = e[i].hist;
  }
}

void fill_items_bwd(const int32_t* off, int batch, int heads, Item* dst, const int32_t* num_targets,
                    int32_t* hist_dst) {
  // (cost, b, h, kt) generated in b, h, kt order; a stable sort by cost
  // descending then gives cost descending, then b, h, kt ascending.  With
  // candidates, a key block without history keys is seen by its own rows
  // only: cost 1 (the diagonal query block).
  struct Entry {
    int cost, hist;
    Item item;
  };
  std::vector<Entry> e;
  e.reserve((size_t)count_items(off, batch, heads));
  for (int b = 0; b < batch; ++b) {
    const int n = off[b + 1] - off[b];
    const int hist = num_targets ? n - num_targets[b] : n;
    const int nq = (n + HSTU_BLOCK_M - 1) / HSTU_BLOCK_M;
    for (int h = 0; h < heads; ++h)
      for (int kt = 0; kt < nq; ++kt)
        e.push_back(Entry{HSTU_BLOCK_M * kt >= hist ? 1 : nq - kt, hist, make_int4(off[b], n, h, kt)});
  }
  std::stable_sort(e.begin(), e.end(), [](const Entry& x, const Entry& y) { return x.cost > y.cost; });
  for (size_t i = 0; i < e.size(); ++i) {
    dst[i] = e[i].item;
    if (hist_dst) hist_dst[i] = e[i].hist;
  }
}

// Static schedule of a longest-first work list over `grid` CTAs (list
// scheduling): an item takes cost + 1 units (its blocks, plus its loads and
// epilogue) and goes, in list order, to the CTA that is free first (ties:
// the lower CTA), so no CTA ends more than one item's units after the mean.
// Output: order[] (item indices, CTA 0's first) and first[grid + 1] (CTA c
// runs order[first[c] .. first[c + 1] - 1], in list order).
long long schedule_items(const int32_t* cost, int n, int grid, int32_t* order, int32_t* first) {
  std::vector<std::pair<long long, int>> heap;  // (free at, CTA): a min-heap
  heap.reserve((size_t)grid);
  for (int c = 0; c < grid; ++c) heap.emplace_back(0ll, c);
  std::vector<int> owner((size_t)n);
  long long span = 0;
  for (int i = 0; i < n; ++i) {
    std::pop_heap(heap.begin(), heap.end(), std::greater<>());
    auto& top = heap.back();
    owner[(size_t)i] = top.second;
    top.first += (long long)cost[i] + 1;
    span = std::max(span, top.first);
    std::push_heap(heap.begin(), heap.end(), std::greater<>());
  }
  std::fill(first, first + grid + 1, 0);
  for (int i = 0; i < n; ++i) ++first[owner[(size_t)i] + 1];
  for (int c = 0; c < grid; ++c) first[c + 1] += first[c];
  std::vector<int32_t> fill(first, first + grid);
  for (int i = 0; i < n; ++i) order[fill[(size_t)owner[(size_t)i]]++] = i;
  return span;
}

int host_check_offsets(const int32_t* off, int batch, long long max_len) {
  return check_offsets(off, batch, max_len);
}
int host_check_buffers(const void* q, const void* k, const void* v, const void* out) {
  return check_buffers(q, k, v, out);
}
int host_launch(const Item* d_items, const int32_t* d_hist, int n_items, long long total, int heads,
                int d, const void* q, const void* k, const void* v, float alpha, float inv_n,
                void* out, const NormGate* ng, cudaStream_t stream) {
  return launch(d_items, d_hist, n_items, total, heads, d, q, k, v, alpha, inv_n, out, ng, stream);
}
}  // namespace hstu

struct hstu_plan {
  int batch = 0, heads = 0, d = 0, max_seqlen = 0;
  long long total = 0;
  std::vector<hstu::Item> items;
  std::vector<int32_t> hist;        // history length per item; empty: no candidates
  unsigned flags = 0;               // HSTU_PLAN_* bits
  hstu::Item* d_items = nullptr;    // device copy of items, then hist (one allocation)
  int32_t* d_hist = nullptr;
  // output-stage scratch (HSTU_PLAN_NORM_GATE): xs, then stats
  char* d_norm = nullptr;
  // backward (HSTU_PLAN_BACKWARD): its work list and (with candidates) each
  // item's history length in schedule order, the schedule's first[grid + 1],
  // then the fp32 dQ accumulator; one allocation
  int n_bwd = 0;
  char* d_bwd = nullptr;
  int32_t* d_bwd_hist = nullptr;
  int32_t* d_bwd_first = nullptr;
  int bwd_grid = 0;
  float* d_bwd_acc = nullptr;
  // the plain forward on CTA pairs (where use_pairs holds): its work list
  int n_pairs = 0;
  hstu::Item* d_pairs = nullptr;
  int device = -1;
};

namespace {

hstu::NormGate norm_views(char* block, long long total, int heads, int d) {
  hstu::NormGate ng{};
  ng.xs = reinterpret_cast<float*>(block);
  ng.stats = reinterpret_cast<float2*>(block + hstu::norm_xs_bytes(total, heads, d));
  return ng;
}

int make_plan(const int32_t* off, const int32_t* nt, int batch, int heads, int d, int max_seqlen,
              unsigned flags, hstu_plan** plan) {
  if (!plan) return HSTU_ERR_INVALID_ARG;
  *plan = nullptr;
  if (heads < 1 || max_seqlen < 0 ||
      (flags & ~(unsigned)(HSTU_PLAN_NORM_GATE | HSTU_PLAN_BACKWARD | HSTU_PLAN_CANDIDATES_ONLY |
                           HSTU_PLAN_PAIRS)))
    return HSTU_ERR_INVALID_ARG;
  if ((flags & HSTU_PLAN_PAIRS) && nt) return HSTU_ERR_INVALID_ARG;
  // the candidates' rows only: needs candidates; the output stage normalises
  // every row and the backward every pair, so neither combines with it
  const bool cand_only = (flags & HSTU_PLAN_CANDIDATES_ONLY) != 0;
  if (cand_only && (!nt || (flags & (HSTU_PLAN_NORM_GATE | HSTU_PLAN_BACKWARD))))
    return HSTU_ERR_INVALID_ARG;
  const bool norm = (flags & HSTU_PLAN_NORM_GATE) != 0;
  if (!supported_d(d)) return HSTU_ERR_UNSUPPORTED;
  int rc = check_offsets(off, batch, max_seqlen);
  if (rc != HSTU_OK) return rc;
  if (nt && (rc = check_targets(off, nt, batch)) != HSTU_OK) return rc;
  hstu_plan* p = new (std::nothrow) hstu_plan;
  if (!p) return HSTU_ERR_NO_MEMORY;
  p->batch = batch;
  p->heads = heads;
  p->d = d;
  p->max_seqlen = max_seqlen;
  p->flags = flags;
  p->total = batch ? off[batch] : 0;
  if ((rc = build_worklist(off, nt, batch, heads, p->items, p->hist, cand_only)) != HSTU_OK) {
    delete p;
    return rc;
  }
  if (p->items.empty()) {
    *plan = p;
    return HSTU_OK;
  }
  auto fail = [&](int code) {
    if (p->d_items) cudaFree(p->d_items);
    if (p->d_norm) cudaFree(p->d_norm);
    if (p->d_bwd) cudaFree(p->d_bwd);
    if (p->d_pairs) cudaFree(p->d_pairs);
    delete p;
    return code;
  };
  auto mem_code = [](cudaError_t e) {
    return e == cudaErrorMemoryAllocation ? HSTU_ERR_NO_MEMORY : HSTU_ERR_CUDA;
  };
  if (cudaGetDevice(&p->device) != cudaSuccess) return fail(HSTU_ERR_CUDA);
  // one allocation: the items, then (with candidates) the history lengths
  const size_t ibytes = p->items.size() * sizeof(hstu::Item);
  const size_t hbytes = p->hist.size() * sizeof(int32_t);
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&p->d_items), ibytes + hbytes);
  if (e != cudaSuccess) return fail(mem_code(e));
  if (hbytes) p->d_hist = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(p->d_items) + ibytes);
  if (cudaMemcpy(p->d_items, p->items.data(), ibytes, cudaMemcpyHostToDevice) != cudaSuccess ||
      (hbytes &&
       cudaMemcpy(p->d_hist, p->hist.data(), hbytes, cudaMemcpyHostToDevice) != cudaSuccess))
    return fail(HSTU_ERR_CUDA);
  if (!nt && (d == 64 || d == 128) && ((flags & HSTU_PLAN_PAIRS) || use_pairs(off, batch, d))) {
    std::vector<hstu::Item> pairs;
    try {
      pairs.resize((size_t)hstu::count_pairs(off, batch, heads));
    } catch (const std::bad_alloc&) {
      return fail(HSTU_ERR_NO_MEMORY);
    }
    hstu::fill_pairs(off, batch, heads, pairs.data());
    p->n_pairs = (int)pairs.size();
    if ((e = cudaMalloc(reinterpret_cast<void**>(&p->d_pairs), pairs.size() * sizeof(hstu::Item))) !=
        cudaSuccess)
      return fail(mem_code(e));
    if (cudaMemcpy(p->d_pairs, pairs.data(), pairs.size() * sizeof(hstu::Item), cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return fail(HSTU_ERR_CUDA);
  }
  if (norm) {
    if ((e = cudaMalloc(reinterpret_cast<void**>(&p->d_norm),
                        hstu::norm_scratch_bytes(p->total, heads, d))) != cudaSuccess)
      return fail(mem_code(e));
  }
  if (flags & HSTU_PLAN_BACKWARD) {
    std::vector<hstu::Item> bw;
    try {
      bw.resize(p->items.size());
    } catch (const std::bad_alloc&) {
      return fail(HSTU_ERR_NO_MEMORY);
    }
    std::vector<int32_t> bh;
    try {
      if (nt) bh.resize(bw.size());
    } catch (const std::bad_alloc&) {
      return fail(HSTU_ERR_NO_MEMORY);
    }
    hstu::fill_items_bwd(off, batch, heads, bw.data(), nt, nt ? bh.data() : nullptr);
    p->n_bwd = (int)bw.size();
    int sms = 0;
    if ((rc = sm_count_of_current_device(&sms)) != HSTU_OK) return fail(rc);
    ListLayout L;
    if ((rc = layout_list_bwd(bw, bh, sms, &L)) != HSTU_OK) return fail(rc);
    const size_t lbytes = (L.bytes() + 15) / 16 * 16;  // keeps the accumulator 16-aligned
    if ((e = cudaMalloc(reinterpret_cast<void**>(&p->d_bwd),
                        lbytes + (size_t)p->total * heads * d * sizeof(float))) != cudaSuccess)
      return fail(mem_code(e));
    if (nt) p->d_bwd_hist = reinterpret_cast<int32_t*>(p->d_bwd + L.ibytes());
    p->d_bwd_first = reinterpret_cast<int32_t*>(p->d_bwd + L.ibytes() + L.hbytes());
    p->bwd_grid = L.grid;
    p->d_bwd_acc = reinterpret_cast<float*>(p->d_bwd + lbytes);
    if (copy_list(L, p->d_bwd, nullptr, true) != cudaSuccess) return fail(HSTU_ERR_CUDA);
  }
  *plan = p;
  return HSTU_OK;
}

int oneshot(const void* q, const void* k, const void* v, const int32_t* offsets,
            const int32_t* num_targets, int batch, int heads, int d, int max_seqlen, float alpha,
            float inv_n, void* out, const hstu::NormGate* ng, cudaStream_t s,
            const hstu_rab* rab) {
  if (heads < 1 || max_seqlen < 0 || batch < 0) return HSTU_ERR_INVALID_ARG;
  if (!supported_d(d)) return HSTU_ERR_UNSUPPORTED;
  if (batch == 0) return HSTU_OK;
  if (!offsets) return HSTU_ERR_INVALID_ARG;
  int rc = HSTU_OK;
  if (ng && (rc = check_norm_gate(ng->u, ng->gamma, ng->beta, ng->eps)) != HSTU_OK) return rc;
  if (rab && (rc = check_rab(rab)) != HSTU_OK) return rc;

  // Offsets may live on the host or on the device.
  std::vector<int32_t> host_off;
  const int32_t* off = offsets;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, offsets) != cudaSuccess) return HSTU_ERR_CUDA;
  if (attr.type == cudaMemoryTypeDevice) {
    try {
      host_off.resize((size_t)batch + 1);
    } catch (const std::bad_alloc&) {
      return HSTU_ERR_NO_MEMORY;
    }
    if (cudaMemcpyAsync(host_off.data(), offsets, host_off.size() * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return HSTU_ERR_CUDA;
    off = host_off.data();
  }
  if ((rc = check_offsets(off, batch, max_seqlen)) != HSTU_OK) return rc;
  if (num_targets && (rc = check_targets(off, num_targets, batch)) != HSTU_OK) return rc;
  const long long total = off[batch];
  if (total == 0) return HSTU_OK;
  if ((rc = check_buffers(q, k, v, out)) != HSTU_OK) return rc;

  if (!ng && !rab && !num_targets && !pairs_disabled() && use_pairs(off, batch, d)) {
    std::vector<hstu::Item> pairs;
    try {
      pairs.resize((size_t)hstu::count_pairs(off, batch, heads));
    } catch (const std::bad_alloc&) {
      return HSTU_ERR_NO_MEMORY;
    }
    hstu::fill_pairs(off, batch, heads, pairs.data());
    if (pairs.empty()) return HSTU_OK;
    const size_t pbytes = pairs.size() * sizeof(hstu::Item);
    hstu::Item* d_pairs = nullptr;
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&d_pairs), pbytes, s);
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? HSTU_ERR_NO_MEMORY : HSTU_ERR_CUDA;
    // pageable source: the copy returns once the bytes are staged
    if (cudaMemcpyAsync(d_pairs, pairs.data(), pbytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
      cudaFreeAsync(d_pairs, s);
      return HSTU_ERR_CUDA;
    }
    rc = launch_pairs(d_pairs, (int)pairs.size(), total, heads, d, q, k, v, alpha, inv_n, out, s);
    if (cudaFreeAsync(d_pairs, s) != cudaSuccess && rc == HSTU_OK) rc = HSTU_ERR_CUDA;
    return rc;
  }
  std::vector<hstu::Item> items;
  std::vector<int32_t> hist;
  if ((rc = build_worklist(off, num_targets, batch, heads, items, hist)) != HSTU_OK) return rc;
  if (items.empty()) return HSTU_OK;
  // one stream-ordered allocation: the output-stage scratch (if any), the
  // items, then (with candidates) the history lengths
  const size_t nbytes = ng ? hstu::norm_scratch_bytes(total, heads, d) : 0;
  const size_t ibytes = items.size() * sizeof(hstu::Item);
  const size_t hbytes = hist.size() * sizeof(int32_t);
  char* block = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&block), nbytes + ibytes + hbytes, s);
  if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? HSTU_ERR_NO_MEMORY : HSTU_ERR_CUDA;
  hstu::Item* d_items = reinterpret_cast<hstu::Item*>(block + nbytes);
  int32_t* d_hist = hbytes ? reinterpret_cast<int32_t*>(block + nbytes + ibytes) : nullptr;
  // Pageable sources: each copy returns once the bytes are staged, so the
  // host vectors may go out of scope afterwards.
  e = cudaMemcpyAsync(d_items, items.data(), ibytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && hbytes)
    e = cudaMemcpyAsync(d_hist, hist.data(), hbytes, cudaMemcpyHostToDevice, s);
  hstu::NormGate ngw{};
  if (ng && e == cudaSuccess) {
    ngw = norm_views(block, total, heads, d);
    ngw.u = ng->u;
    ngw.gamma = ng->gamma;
    ngw.beta = ng->beta;
    ngw.eps = ng->eps;
  }
  if (e != cudaSuccess) {
    cudaFreeAsync(block, s);
    return HSTU_ERR_CUDA;
  }
  rc = launch(d_items, d_hist, (int)items.size(), total, heads, d, q, k, v, alpha, inv_n, out,
              ng ? &ngw : nullptr, s, rab);
  if (cudaFreeAsync(block, s) != cudaSuccess && rc == HSTU_OK) rc = HSTU_ERR_CUDA;
  return rc;
}

// The bias's table gradients: non-null, 4-byte aligned.
int check_rab_grads(const float* dpos, const float* dtime) {
  if (!dpos || !dtime) return HSTU_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dpos) | reinterpret_cast<uintptr_t>(dtime)) & 3u)
    return HSTU_ERR_INVALID_ARG;
  return HSTU_OK;
}

// No token: the tables' gradients are zero.
int zero_rab_grads(const hstu_rab* rab, float* dpos, float* dtime, cudaStream_t s) {
  if (!rab) return HSTU_OK;
  if (cudaMemsetAsync(dpos, 0, (size_t)rab->num_pos * sizeof(float), s) != cudaSuccess ||
      cudaMemsetAsync(dtime, 0, (size_t)rab->num_time * sizeof(float), s) != cudaSuccess)
    return HSTU_ERR_CUDA;
  return HSTU_OK;
}

int launch_backward(const hstu::Item* d_items, int n_items, long long total, int heads, int d,
                    const void* q, const void* k, const void* v, const void* dout, float alpha,
                    float inv_n, float* dq_acc, void* dq, void* dk, void* dv, cudaStream_t stream,
                    const hstu_rab* rab = nullptr, float* dpos = nullptr, float* dtime = nullptr,
                    const int32_t* d_hist = nullptr, const int32_t* d_first = nullptr,
                    int sched_grid = 0) {
  int sms = 0;
  int rc = device_check(&sms);
  if (rc != HSTU_OK) return rc;
  unsigned dbg;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    dbg = g_debug_flags;
  }
  // the transposed form (d <= 64 without the bias) loads Q and dO half a
  // block at a time
  const bool transposed = d <= 64 && !rab && !(dbg & HSTU_DEBUG_BWD_ROWS);
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (transposed) {
    if ((rc = make_map_pair(&tq, q, total, heads, d, std::min(d, 64), HSTU_BLOCK_M / 2)) != HSTU_OK)
      return rc;
    if ((rc = make_map_pair(&tdo, dout, total, heads, d, std::min(d, 64), HSTU_BLOCK_M / 2)) != HSTU_OK)
      return rc;
  } else {
    if ((rc = make_map(&tq, q, total, heads, d)) != HSTU_OK) return rc;
    if ((rc = make_map(&tdo, dout, total, heads, d)) != HSTU_OK) return rc;
  }
  if ((rc = make_map(&tk, k, total, heads, d)) != HSTU_OK) return rc;
  if ((rc = make_map(&tv, v, total, heads, d)) != HSTU_OK) return rc;
  if ((rc = make_map_f32(&tdq, dq_acc, total, heads, d)) != HSTU_OK) return rc;
  hstu::BwdArgs a{};  // every field zero: no bias unless set below
  a.transposed = transposed;
  a.debug_flags = dbg;
  a.items = d_items;
  a.n_items = n_items;
  a.heads = heads;
  a.alpha = alpha;
  a.inv_n = inv_n;
  a.dq_acc = dq_acc;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.total = total;
  a.timeout_ns = wait_timeout_ns();
  a.item_hist = d_hist;
  if (rab) {
    a.rab_ts = rab->timestamps;
    a.rab_pos = rab->pos;
    a.rab_time = rab->time;
    a.rab_npos = rab->num_pos;
    a.rab_ntime = rab->num_time;
    a.dpos = dpos;
    a.dtime = dtime;
  }
  // the accumulators start at zero on the stream, before the kernel
  if (cudaMemsetAsync(dq_acc, 0, (size_t)total * heads * d * sizeof(float), stream) != cudaSuccess)
    return HSTU_ERR_CUDA;
  if (rab && (cudaMemsetAsync(dpos, 0, (size_t)rab->num_pos * sizeof(float), stream) != cudaSuccess ||
              cudaMemsetAsync(dtime, 0, (size_t)rab->num_time * sizeof(float), stream) != cudaSuccess))
    return HSTU_ERR_CUDA;
  a.cta_first = d_first;
  const int grid = d_first ? sched_grid : grid_for(n_items, sms);
  const cudaError_t e = hstu::launch_bwd(d, tq, tk, tv, tdo, tdq, a, grid, stream);
  if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
    return HSTU_ERR_UNSUPPORTED;
  return e == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}

// The host-buffer forward's copy streams of the current device: one for
// q, k, v (copies on more streams at once measured no faster: they share
// one host link), one for out.  Non-blocking, created on first use, kept
// until exit.
constexpr int kMaxDevices = 64;
constexpr int kCopyStreams = 2;
std::mutex g_copy_mu;
cudaStream_t g_copy_streams[kMaxDevices][kCopyStreams] = {};

int copy_streams(cudaStream_t (&st)[kCopyStreams]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HSTU_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_copy_mu);
  for (int i = 0; i < kCopyStreams; ++i) {
    cudaStream_t& c = g_copy_streams[dev][i];
    if (!c && cudaStreamCreateWithFlags(&c, cudaStreamNonBlocking) != cudaSuccess) {
      c = nullptr;
      return HSTU_ERR_CUDA;
    }
    st[i] = c;
  }
  return HSTU_OK;
}

// Runs of the host-buffer forward when the caller asks for none.
constexpr int kHostRuns = 4;
int host_run_count(int batch, int n_chunks) {
  return std::min(batch, n_chunks > 0 ? n_chunks : kHostRuns);
}

// Splits sequences 0 .. batch-1 into nc runs of whole sequences with about
// equal token counts: run c is sequences first[c] .. first[c+1]-1 (a run
// may be empty when one sequence holds most tokens).
std::vector<int> chunk_sequences(const int32_t* off, int batch, int nc) {
  std::vector<int> first((size_t)nc + 1, batch);
  first[0] = 0;
  const long long total = off[batch];
  int b = 0;
  for (int c = 1; c < nc; ++c) {
    const long long target = total * c / nc;
    while (b < batch && off[b] < target) ++b;
    first[(size_t)c] = std::max(b, first[(size_t)c - 1]);
  }
  return first;
}

// Events of one host-buffer call, destroyed on scope exit (a pending
// event's resources are released once it completes).
struct EventSet {
  std::vector<cudaEvent_t> ev;
  ~EventSet() {
    for (cudaEvent_t e : ev)
      if (e) cudaEventDestroy(e);
  }
  cudaEvent_t make() {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    ev.push_back(e);
    return e;
  }
};

int fwd_host(const void* q_host, const void* k_host, const void* v_host, const int32_t* off,
             int batch, int heads, int d, int max_seqlen, float alpha, float inv_n, void* out_host,
             void* q_dev, void* k_dev, void* v_dev, void* out_dev, int n_chunks, cudaStream_t s) {
  if (heads < 1 || max_seqlen < 0 || batch < 0 || n_chunks < 0) return HSTU_ERR_INVALID_ARG;
  if (!supported_d(d)) return HSTU_ERR_UNSUPPORTED;
  if (batch == 0) return HSTU_OK;
  if (!off) return HSTU_ERR_INVALID_ARG;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, off) != cudaSuccess) return HSTU_ERR_CUDA;
  if (attr.type == cudaMemoryTypeDevice) return HSTU_ERR_INVALID_ARG;
  int rc = check_offsets(off, batch, max_seqlen);
  if (rc != HSTU_OK) return rc;
  const long long total = off[batch];
  if (total == 0) return HSTU_OK;
  if (!q_host || !k_host || !v_host || !out_host) return HSTU_ERR_INVALID_ARG;
  if ((rc = check_buffers(q_dev, k_dev, v_dev, out_dev)) != HSTU_OK) return rc;
  cudaStream_t cs[kCopyStreams] = {};
  if ((rc = copy_streams(cs)) != HSTU_OK) return rc;
  cudaStream_t s_in = cs[0], s_out = cs[1];

  const int nc = host_run_count(batch, n_chunks);
  std::vector<hstu::Item> all, items;
  std::vector<int32_t> hist;
  std::vector<int> seq_first, item_first;
  try {
    if ((rc = build_worklist(off, nullptr, batch, heads, all, hist)) != HSTU_OK) return rc;
    seq_first = chunk_sequences(off, batch, nc);
    // each run's items, in the longest-first order of the whole list: a
    // counting sort by run, keyed on the item's first row
    std::vector<int32_t> run_row((size_t)nc);
    for (int c = 0; c < nc; ++c) run_row[(size_t)c] = off[seq_first[(size_t)c + 1]];
    auto run_of = [&](const hstu::Item& it) {
      return (int)(std::upper_bound(run_row.begin(), run_row.end(), it.x) - run_row.begin());
    };
    item_first.assign((size_t)nc + 1, 0);
    for (const hstu::Item& it : all) ++item_first[(size_t)run_of(it) + 1];
    for (int c = 0; c < nc; ++c) item_first[(size_t)c + 1] += item_first[(size_t)c];
    items.resize(all.size());
    std::vector<int> fill(item_first.begin(), item_first.end() - 1);
    for (const hstu::Item& it : all) items[(size_t)fill[(size_t)run_of(it)]++] = it;
  } catch (const std::bad_alloc&) {
    return HSTU_ERR_NO_MEMORY;
  }

  const size_t ibytes = items.size() * sizeof(hstu::Item);
  hstu::Item* d_items = nullptr;
  if (ibytes) {
    const cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&d_items), ibytes, s);
    if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? HSTU_ERR_NO_MEMORY : HSTU_ERR_CUDA;
    // pageable source: the copy returns once the bytes are staged
    if (cudaMemcpyAsync(d_items, items.data(), ibytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
      cudaFreeAsync(d_items, s);
      return HSTU_ERR_CUDA;
    }
  }
  EventSet evs;
  rc = [&]() -> int {
    cudaEvent_t start = evs.make(), done_out = evs.make();
    if (!start || !done_out) return HSTU_ERR_CUDA;
    // the copies in start after the caller's earlier work on s
    if (cudaEventRecord(start, s) != cudaSuccess || cudaStreamWaitEvent(s_in, start, 0) != cudaSuccess)
      return HSTU_ERR_CUDA;
    const size_t row = (size_t)heads * d * 2;
    const void* src[3] = {q_host, k_host, v_host};
    void* dst[3] = {q_dev, k_dev, v_dev};
    std::vector<cudaEvent_t> landed((size_t)nc);  // run c's q, k, v are on the device
    for (int c = 0; c < nc; ++c) {
      const size_t r0 = (size_t)off[seq_first[(size_t)c]], r1 = (size_t)off[seq_first[(size_t)c + 1]];
      for (int t = 0; t < 3 && r1 > r0; ++t)
        if (cudaMemcpyAsync(static_cast<char*>(dst[t]) + r0 * row,
                            static_cast<const char*>(src[t]) + r0 * row, (r1 - r0) * row,
                            cudaMemcpyHostToDevice, s_in) != cudaSuccess)
          return HSTU_ERR_CUDA;
      if (!(landed[(size_t)c] = evs.make()) || cudaEventRecord(landed[(size_t)c], s_in) != cudaSuccess)
        return HSTU_ERR_CUDA;
    }
    for (int c = 0; c < nc; ++c) {
      const size_t r0 = (size_t)off[seq_first[(size_t)c]], r1 = (size_t)off[seq_first[(size_t)c + 1]];
      if (cudaStreamWaitEvent(s, landed[(size_t)c], 0) != cudaSuccess) return HSTU_ERR_CUDA;
      const int n = item_first[(size_t)c + 1] - item_first[(size_t)c];
      const int lrc = launch(d_items + item_first[(size_t)c], nullptr, n, total, heads, d, q_dev,
                             k_dev, v_dev, alpha, inv_n, out_dev, nullptr, s);
      if (lrc != HSTU_OK) return lrc;
      cudaEvent_t computed = evs.make();
      if (!computed || cudaEventRecord(computed, s) != cudaSuccess ||
          cudaStreamWaitEvent(s_out, computed, 0) != cudaSuccess)
        return HSTU_ERR_CUDA;
      if (r1 > r0 && cudaMemcpyAsync(static_cast<char*>(out_host) + r0 * row,
                                     static_cast<const char*>(out_dev) + r0 * row, (r1 - r0) * row,
                                     cudaMemcpyDeviceToHost, s_out) != cudaSuccess)
        return HSTU_ERR_CUDA;
    }
    // later work on s sees out_host written
    if (cudaEventRecord(done_out, s_out) != cudaSuccess ||
        cudaStreamWaitEvent(s, done_out, 0) != cudaSuccess)
      return HSTU_ERR_CUDA;
    return HSTU_OK;
  }();
  if (d_items && cudaFreeAsync(d_items, s) != cudaSuccess && rc == HSTU_OK) rc = HSTU_ERR_CUDA;
  return rc;
}

}  // namespace

extern "C" {

const char* hstu_status_string(int status) {
  switch (status) {
    case HSTU_OK: return "ok";
    case HSTU_ERR_INVALID_ARG: return "invalid argument";
    case HSTU_ERR_UNSUPPORTED: return "unsupported head dimension or device (needs d in {32,64,128} on sm_103)";
    case HSTU_ERR_CUDA: return "CUDA runtime or driver error";
    case HSTU_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    case HSTU_ERR_NO_MEMORY: return "out of memory";
    case HSTU_ERR_CAPACITY:
      return "work list larger than the fixed capacity of hstu_attn_fwd_noalloc (HSTU_NOALLOC_MAX_ITEMS)";
    default: return "unknown status";
  }
}

int hstu_worklist_build(const int32_t* host_offsets, int batch, int heads, int32_t* host_dst,
                        int capacity, int* n_items) {
  if (!n_items || heads < 1 || capacity < 0) return HSTU_ERR_INVALID_ARG;
  int rc = check_offsets(host_offsets, batch, -1);
  if (rc != HSTU_OK) return rc;
  std::vector<hstu::Item> items;
  try {
    items = build_items(host_offsets, batch, heads);
  } catch (const std::bad_alloc&) {
    return HSTU_ERR_NO_MEMORY;
  }
  if (items.size() > (size_t)INT32_MAX) return HSTU_ERR_INVALID_ARG;
  *n_items = (int)items.size();
  if (host_dst) {
    const size_t n = std::min(items.size(), (size_t)capacity);
    std::memcpy(host_dst, items.data(), n * sizeof(hstu::Item));
  }
  return HSTU_OK;
}

int hstu_plan_create(const int32_t* host_offsets, int batch, int heads, int d, int max_seqlen,
                     hstu_plan** plan) {
  return make_plan(host_offsets, nullptr, batch, heads, d, max_seqlen, 0u, plan);
}

int hstu_plan_create_targets(const int32_t* host_offsets, const int32_t* host_num_targets, int batch,
                             int heads, int d, int max_seqlen, hstu_plan** plan) {
  if (!host_num_targets && batch > 0) return HSTU_ERR_INVALID_ARG;
  return make_plan(host_offsets, host_num_targets, batch, heads, d, max_seqlen, 0u, plan);
}

int hstu_plan_create_ex(const int32_t* host_offsets, const int32_t* host_num_targets, int batch,
                        int heads, int d, int max_seqlen, uint32_t flags, hstu_plan** plan) {
  return make_plan(host_offsets, host_num_targets, batch, heads, d, max_seqlen, flags, plan);
}

int hstu_plan_destroy(hstu_plan* plan) {
  if (!plan) return HSTU_OK;
  int rc = HSTU_OK;
  if (plan->d_items && cudaFree(plan->d_items) != cudaSuccess) rc = HSTU_ERR_CUDA;
  if (plan->d_norm && cudaFree(plan->d_norm) != cudaSuccess) rc = HSTU_ERR_CUDA;
  if (plan->d_bwd && cudaFree(plan->d_bwd) != cudaSuccess) rc = HSTU_ERR_CUDA;
  if (plan->d_pairs && cudaFree(plan->d_pairs) != cudaSuccess) rc = HSTU_ERR_CUDA;
  delete plan;
  return rc;
}

int hstu_plan_num_items(const hstu_plan* plan, int* n_items) {
  if (!plan || !n_items) return HSTU_ERR_INVALID_ARG;
  *n_items = (int)plan->items.size();
  return HSTU_OK;
}

int hstu_plan_num_pairs(const hstu_plan* plan, int* n_pairs) {
  if (!plan || !n_pairs) return HSTU_ERR_INVALID_ARG;
  *n_pairs = plan->n_pairs;
  return HSTU_OK;
}

int hstu_worklist_build_pairs(const int32_t* host_offsets, int batch, int heads, int32_t* host_dst,
                              int capacity, int* n_items) {
  if (!n_items || heads < 1 || capacity < 0) return HSTU_ERR_INVALID_ARG;
  int rc = check_offsets(host_offsets, batch, -1);
  if (rc != HSTU_OK) return rc;
  std::vector<hstu::Item> pairs;
  try {
    pairs.resize((size_t)hstu::count_pairs(host_offsets, batch, heads));
  } catch (const std::bad_alloc&) {
    return HSTU_ERR_NO_MEMORY;
  }
  if (pairs.size() > (size_t)INT32_MAX) return HSTU_ERR_INVALID_ARG;
  hstu::fill_pairs(host_offsets, batch, heads, pairs.data());
  *n_items = (int)pairs.size();
  if (host_dst) {
    const size_t n = std::min(pairs.size(), (size_t)capacity);
    std::memcpy(host_dst, pairs.data(), n * sizeof(hstu::Item));
  }
  return HSTU_OK;
}

int hstu_worklist_schedule(const int32_t* host_cost, int n_items, int grid, int32_t* host_order,
                           int32_t* host_first, long long* makespan) {
  if (!host_cost || !host_order || !host_first || n_items < 1 || grid < 1 || grid > n_items)
    return HSTU_ERR_INVALID_ARG;
  for (int i = 0; i < n_items; ++i)
    if (host_cost[i] < 1) return HSTU_ERR_INVALID_ARG;
  long long span = 0;
  try {
    span = hstu::schedule_items(host_cost, n_items, grid, host_order, host_first);
  } catch (const std::bad_alloc&) {
    return HSTU_ERR_NO_MEMORY;
  }
  if (makespan) *makespan = span;
  return HSTU_OK;
}

int hstu_host_runs(const int32_t* host_offsets, int batch, int n_chunks, int32_t* host_first,
                   int capacity, int* n_runs) {
  if (!host_offsets || !n_runs || batch < 0 || n_chunks < 0) return HSTU_ERR_INVALID_ARG;
  int rc = check_offsets(host_offsets, batch, std::numeric_limits<int32_t>::max());
  if (rc != HSTU_OK) return rc;
  const int nc = host_run_count(batch, n_chunks);
  *n_runs = nc;
  if (!host_first) return HSTU_OK;
  if (capacity < nc + 1) return HSTU_ERR_INVALID_ARG;
  try {
    const std::vector<int> first = chunk_sequences(host_offsets, batch, nc);
    for (int c = 0; c <= nc; ++c) host_first[c] = first[(size_t)c];
  } catch (const std::bad_alloc&) {
    return HSTU_ERR_NO_MEMORY;
  }
  return HSTU_OK;
}

int hstu_plan_worklist(const hstu_plan* plan, int32_t* host_dst, int capacity, int* n_items) {
  if (!plan || !n_items) return HSTU_ERR_INVALID_ARG;
  *n_items = (int)plan->items.size();
  if (!host_dst) return HSTU_OK;
  if (capacity < (int)plan->items.size()) return HSTU_ERR_INVALID_ARG;
  std::memcpy(host_dst, plan->items.data(), plan->items.size() * sizeof(hstu::Item));
  return HSTU_OK;
}

int hstu_plan_item_hist(const hstu_plan* plan, int32_t* host_dst, int capacity, int* n_items) {
  if (!plan || !n_items) return HSTU_ERR_INVALID_ARG;
  *n_items = (int)plan->items.size();
  if (!host_dst) return HSTU_OK;
  if (capacity < (int)plan->items.size()) return HSTU_ERR_INVALID_ARG;
  for (size_t i = 0; i < plan->items.size(); ++i)
    host_dst[i] = plan->hist.empty() ? plan->items[i].y : plan->hist[i];
  return HSTU_OK;
}

int hstu_worklist_build_targets(const int32_t* host_offsets, const int32_t* host_num_targets,
                                int batch, int heads, int32_t* host_items, int32_t* host_hist,
                                int capacity, int* n_items) {
  if (!n_items || heads < 1 || capacity < 0 || (!host_num_targets && batch > 0))
    return HSTU_ERR_INVALID_ARG;
  int rc = check_offsets(host_offsets, batch, -1);
  if (rc != HSTU_OK) return rc;
  if ((rc = check_targets(host_offsets, host_num_targets, batch)) != HSTU_OK) return rc;
  std::vector<hstu::Item> items;
  std::vector<int32_t> hist;
  if ((rc = build_worklist(host_offsets, host_num_targets, batch, heads, items, hist)) != HSTU_OK)
    return rc;
  *n_items = (int)items.size();
  const size_t n = std::min(items.size(), (size_t)capacity);
  if (host_items) std::memcpy(host_items, items.data(), n * sizeof(hstu::Item));
  if (host_hist) std::memcpy(host_hist, hist.data(), n * sizeof(int32_t));
  return HSTU_OK;
}

int hstu_worklist_build_candidates(const int32_t* host_offsets, const int32_t* host_num_targets,
                                   int batch, int heads, int32_t* host_items, int32_t* host_hist,
                                   int capacity, int* n_items) {
  if (!n_items || heads < 1 || capacity < 0 || (!host_num_targets && batch > 0))
    return HSTU_ERR_INVALID_ARG;
  int rc = check_offsets(host_offsets, batch, -1);
  if (rc != HSTU_OK) return rc;
  if ((rc = check_targets(host_offsets, host_num_targets, batch)) != HSTU_OK) return rc;
  std::vector<hstu::Item> items;
  std::vector<int32_t> hist;
  if ((rc = build_worklist(host_offsets, host_num_targets, batch, heads, items, hist, true)) !=
      HSTU_OK)
    return rc;
  *n_items = (int)items.size();
  const size_t n = std::min(items.size(), (size_t)capacity);
  if (host_items) std::memcpy(host_items, items.data(), n * sizeof(hstu::Item));
  if (host_hist) std::memcpy(host_hist, hist.data(), n * sizeof(int32_t));
  return HSTU_OK;
}

int hstu_launch_shape(const hstu_plan* plan, int* grid, int* block, int* smem_bytes) {
  if (!plan || !grid || !block || !smem_bytes) return HSTU_ERR_INVALID_ARG;
  int sms = 0;
  const int rc = device_check(&sms);
  if (rc != HSTU_OK) return rc;
  if (plan->d_pairs && !pairs_disabled()) {
    *grid = pair_grid_for(plan->n_pairs, sms);
    *block = hstu::kFwdThreads;
    *smem_bytes = hstu::fwd_pair_smem_bytes(plan->d);
    return HSTU_OK;
  }
  *grid = grid_for((int)plan->items.size(), sms);
  *block = hstu::fwd_block_threads(plan->d, false);
  *smem_bytes = hstu::fwd_smem_bytes(plan->d);
  return HSTU_OK;
}

int hstu_attn_fwd_plan(const hstu_plan* plan, const void* q, const void* k, const void* v,
                       float alpha, float inv_n, void* out, hstu_stream_t stream) {
  if (!plan) return HSTU_ERR_INVALID_ARG;
  if (plan->items.empty()) return HSTU_OK;
  int rc = check_buffers(q, k, v, out);
  if (rc != HSTU_OK) return rc;
  if (plan->d_pairs && !pairs_disabled())
    return launch_pairs(plan->d_pairs, plan->n_pairs, plan->total, plan->heads, plan->d, q, k, v, alpha,
                        inv_n, out, reinterpret_cast<cudaStream_t>(stream));
  return launch(plan->d_items, plan->d_hist, (int)plan->items.size(), plan->total, plan->heads,
                plan->d, q, k, v, alpha, inv_n, out, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int hstu_attn_fwd_norm_gate_plan(const hstu_plan* plan, const void* q, const void* k, const void* v,
                                 const void* u, const float* gamma, const float* beta, float eps,
                                 float alpha, float inv_n, void* y, hstu_stream_t stream) {
  if (!plan || !(plan->flags & HSTU_PLAN_NORM_GATE)) return HSTU_ERR_INVALID_ARG;
  if (plan->items.empty()) return HSTU_OK;
  int rc = check_buffers(q, k, v, y);
  if (rc != HSTU_OK) return rc;
  if ((rc = check_norm_gate(u, gamma, beta, eps)) != HSTU_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  hstu::NormGate ng = norm_views(plan->d_norm, plan->total, plan->heads, plan->d);
  ng.u = u;
  ng.gamma = gamma;
  ng.beta = beta;
  ng.eps = eps;
  return launch(plan->d_items, plan->d_hist, (int)plan->items.size(), plan->total, plan->heads,
                plan->d, q, k, v, alpha, inv_n, y, &ng, s);
}

int hstu_attn_fwd_plan_ex(const hstu_plan* plan, const void* q, const void* k, const void* v,
                          const hstu_rab* rab, const hstu_norm_gate* ng, float alpha, float inv_n,
                          void* out, hstu_stream_t stream) {
  if (!plan || (ng && !(plan->flags & HSTU_PLAN_NORM_GATE))) return HSTU_ERR_INVALID_ARG;
  if (plan->items.empty()) return HSTU_OK;
  int rc = check_buffers(q, k, v, out);
  if (rc != HSTU_OK) return rc;
  if (ng && (rc = check_norm_gate(ng->u, ng->gamma, ng->beta, ng->eps)) != HSTU_OK) return rc;
  if (rab && (rc = check_rab(rab)) != HSTU_OK) return rc;
  hstu::NormGate ngw{};
  if (ng) {
    ngw = norm_views(plan->d_norm, plan->total, plan->heads, plan->d);
    ngw.u = ng->u;
    ngw.gamma = ng->gamma;
    ngw.beta = ng->beta;
    ngw.eps = ng->eps;
  }
  if (!ng && !rab && plan->d_pairs && !pairs_disabled())
    return launch_pairs(plan->d_pairs, plan->n_pairs, plan->total, plan->heads, plan->d, q, k, v, alpha,
                        inv_n, out, reinterpret_cast<cudaStream_t>(stream));
  return launch(plan->d_items, plan->d_hist, (int)plan->items.size(), plan->total, plan->heads,
                plan->d, q, k, v, alpha, inv_n, out, ng ? &ngw : nullptr,
                reinterpret_cast<cudaStream_t>(stream), rab);
}

int hstu_attn_fwd_ex(const void* q, const void* k, const void* v, const int32_t* offsets,
                     const int32_t* host_num_targets, int batch, int heads, int d, int max_seqlen,
                     const hstu_rab* rab, const hstu_norm_gate* ng, float alpha, float inv_n,
                     void* out, hstu_stream_t stream) {
  hstu::NormGate ngw{};
  if (ng) {
    ngw.u = ng->u;
    ngw.gamma = ng->gamma;
    ngw.beta = ng->beta;
    ngw.eps = ng->eps;
  }
  return oneshot(q, k, v, offsets, host_num_targets, batch, heads, d, max_seqlen, alpha, inv_n, out,
                 ng ? &ngw : nullptr, reinterpret_cast<cudaStream_t>(stream), rab);
}

int hstu_attn_fwd_norm_gate(const void* q, const void* k, const void* v, const void* u,
                            const float* gamma, const float* beta, float eps, const int32_t* offsets,
                            const int32_t* host_num_targets, int batch, int heads, int d,
                            int max_seqlen, float alpha, float inv_n, void* y,
                            hstu_stream_t stream) {
  hstu::NormGate ng{};
  ng.u = u;
  ng.gamma = gamma;
  ng.beta = beta;
  ng.eps = eps;
  return oneshot(q, k, v, offsets, host_num_targets, batch, heads, d, max_seqlen, alpha, inv_n, y,
                 &ng, reinterpret_cast<cudaStream_t>(stream));
}

int hstu_attn_fwd(const void* q, const void* k, const void* v, const int32_t* offsets, int batch,
                  int heads, int d, int max_seqlen, float alpha, float inv_n, void* out,
                  hstu_stream_t stream) {
  return oneshot(q, k, v, offsets, nullptr, batch, heads, d, max_seqlen, alpha, inv_n, out,
                 nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int hstu_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                       const int32_t* offsets, int batch, int heads, int d, int max_seqlen,
                       float alpha, float inv_n, void* out_host, void* q_dev, void* k_dev,
                       void* v_dev, void* out_dev, int n_chunks, hstu_stream_t stream) {
  return fwd_host(q_host, k_host, v_host, offsets, batch, heads, d, max_seqlen, alpha, inv_n,
                  out_host, q_dev, k_dev, v_dev, out_dev, n_chunks,
                  reinterpret_cast<cudaStream_t>(stream));
}

int hstu_attn_fwd_targets(const void* q, const void* k, const void* v, const int32_t* offsets,
                          const int32_t* host_num_targets, int batch, int heads, int d,
                          int max_seqlen, float alpha, float inv_n, void* out,
                          hstu_stream_t stream) {
  if (!host_num_targets && batch > 0) return HSTU_ERR_INVALID_ARG;
  return oneshot(q, k, v, offsets, host_num_targets, batch, heads, d, max_seqlen, alpha, inv_n, out,
                 nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int hstu_worklist_build_bwd_targets(const int32_t* host_offsets, const int32_t* host_num_targets,
                                    int batch, int heads, int32_t* host_items, int32_t* host_hist,
                                    int capacity, int* n_items) {
  if (!n_items || heads < 1 || capacity < 0 || (!host_num_targets && batch > 0))
    return HSTU_ERR_INVALID_ARG;
  int rc = check_offsets(host_offsets, batch, -1);
  if (rc != HSTU_OK) return rc;
  if ((rc = check_targets(host_offsets, host_num_targets, batch)) != HSTU_OK) return rc;
  std::vector<hstu::Item> items;
  std::vector<int32_t> hist;
  try {
    items.resize((size_t)hstu::count_items(host_offsets, batch, heads));
    hist.resize(items.size());
    hstu::fill_items_bwd(host_offsets, batch, heads, items.data(), host_num_targets, hist.data());
  } catch (const std::bad_alloc&) {
    return HSTU_ERR_NO_MEMORY;
  }
  if (items.size() > (size_t)INT32_MAX) return HSTU_ERR_INVALID_ARG;
  *n_items = (int)items.size();
  const size_t n = std::min(items.size(), (size_t)capacity);
  if (host_items) std::memcpy(host_items, items.data(), n * sizeof(hstu::Item));
  if (host_hist) std::memcpy(host_hist, hist.data(), n * sizeof(int32_t));
  return HSTU_OK;
}

int hstu_worklist_build_bwd(const int32_t* host_offsets, int batch, int heads, int32_t* host_dst,
                            int capacity, int* n_items) {
  if (!n_items || heads < 1 || capacity < 0) return HSTU_ERR_INVALID_ARG;
  int rc = check_offsets(host_offsets, batch, -1);
  if (rc != HSTU_OK) return rc;
  std::vector<hstu::Item> items;
  try {
    items.resize((size_t)hstu::count_items(host_offsets, batch, heads));
    hstu::fill_items_bwd(host_offsets, batch, heads, items.data());
  } catch (const std::bad_alloc&) {
    return HSTU_ERR_NO_MEMORY;
  }
  if (items.size() > (size_t)INT32_MAX) return HSTU_ERR_INVALID_ARG;
  *n_items = (int)items.size();
  if (host_dst)
    std::memcpy(host_dst, items.data(), std::min(items.size(), (size_t)capacity) * sizeof(hstu::Item));
  return HSTU_OK;
}

int hstu_attn_bwd(const void* q, const void* k, const void* v, const void* dout,
                  const int32_t* offsets, int batch, int heads, int d, int max_seqlen, float alpha,
                  float inv_n, void* dq, void* dk, void* dv, hstu_stream_t stream) {
  return hstu_attn_bwd_ex(q, k, v, dout, offsets, nullptr, batch, heads, d, max_seqlen, nullptr,
                          alpha, inv_n, dq, dk, dv, nullptr, nullptr, stream);
}

int hstu_attn_bwd_ex(const void* q, const void* k, const void* v, const void* dout,
                     const int32_t* offsets, const int32_t* host_num_targets, int batch, int heads,
                     int d, int max_seqlen, const hstu_rab* rab, float alpha, float inv_n, void* dq,
                     void* dk, void* dv, float* dpos, float* dtime, hstu_stream_t stream) {
  if (heads < 1 || max_seqlen < 0 || batch < 0) return HSTU_ERR_INVALID_ARG;
  int rc;
  if (rab && ((rc = check_rab(rab)) != HSTU_OK || (rc = check_rab_grads(dpos, dtime)) != HSTU_OK))
    return rc;
  if (!supported_d(d)) return HSTU_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (batch == 0) return zero_rab_grads(rab, dpos, dtime, s);
  if (!offsets) return HSTU_ERR_INVALID_ARG;
  std::vector<int32_t> host_off;
  const int32_t* off = offsets;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, offsets) != cudaSuccess) return HSTU_ERR_CUDA;
  if (attr.type == cudaMemoryTypeDevice) {
    try {
      host_off.resize((size_t)batch + 1);
    } catch (const std::bad_alloc&) {
      return HSTU_ERR_NO_MEMORY;
    }
    if (cudaMemcpyAsync(host_off.data(), offsets, host_off.size() * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return HSTU_ERR_CUDA;
    off = host_off.data();
  }
  rc = check_offsets(off, batch, max_seqlen);
  if (rc != HSTU_OK) return rc;
  if (host_num_targets && (rc = check_targets(off, host_num_targets, batch)) != HSTU_OK) return rc;
  const long long total = off[batch];
  if (total == 0) return zero_rab_grads(rab, dpos, dtime, s);
  if ((rc = check_buffers(q, k, v, dout)) != HSTU_OK || (rc = check_buffers(dq, dk, dv, dv)) != HSTU_OK)
    return rc;
  std::vector<hstu::Item> items;
  std::vector<int32_t> hist;
  try {
    items.resize((size_t)hstu::count_items(off, batch, heads));
    if (host_num_targets) hist.resize(items.size());
    hstu::fill_items_bwd(off, batch, heads, items.data(), host_num_targets,
                         host_num_targets ? hist.data() : nullptr);
  } catch (const std::bad_alloc&) {
    return HSTU_ERR_NO_MEMORY;
  }
  if (items.empty()) return zero_rab_grads(rab, dpos, dtime, s);
  if (items.size() > (size_t)INT32_MAX) return HSTU_ERR_INVALID_ARG;
  int sms = 0;
  if ((rc = sm_count_of_current_device(&sms)) != HSTU_OK) return rc;
  ListLayout L;
  if ((rc = layout_list_bwd(items, hist, sms, &L)) != HSTU_OK) return rc;
  // one stream-ordered allocation: the fp32 dQ accumulator, then the list's
  // layout
  const size_t abytes = (size_t)total * heads * d * sizeof(float);
  char* block = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&block), abytes + L.bytes(), s);
  if (e != cudaSuccess) return e == cudaErrorMemoryAllocation ? HSTU_ERR_NO_MEMORY : HSTU_ERR_CUDA;
  hstu::Item* d_items = reinterpret_cast<hstu::Item*>(block + abytes);
  int32_t* d_hist = L.hbytes() ? reinterpret_cast<int32_t*>(block + abytes + L.ibytes()) : nullptr;
  const int32_t* d_first = reinterpret_cast<int32_t*>(block + abytes + L.ibytes() + L.hbytes());
  // pageable sources: each copy returns once its bytes are staged
  if (copy_list(L, block + abytes, s) != cudaSuccess) {
    cudaFreeAsync(block, s);
    return HSTU_ERR_CUDA;
  }
  rc = launch_backward(d_items, (int)items.size(), total, heads, d, q, k, v, dout, alpha, inv_n,
                       reinterpret_cast<float*>(block), dq, dk, dv, s, rab, dpos, dtime, d_hist,
                       d_first, L.grid);
  if (cudaFreeAsync(block, s) != cudaSuccess && rc == HSTU_OK) rc = HSTU_ERR_CUDA;
  return rc;
}

int hstu_attn_bwd_plan(const hstu_plan* plan, const void* q, const void* k, const void* v,
                       const void* dout, float alpha, float inv_n, void* dq, void* dk, void* dv,
                       hstu_stream_t stream) {
  return hstu_attn_bwd_plan_ex(plan, q, k, v, dout, nullptr, alpha, inv_n, dq, dk, dv, nullptr,
                               nullptr, stream);
}

int hstu_attn_bwd_plan_ex(const hstu_plan* plan, const void* q, const void* k, const void* v,
                          const void* dout, const hstu_rab* rab, float alpha, float inv_n, void* dq,
                          void* dk, void* dv, float* dpos, float* dtime, hstu_stream_t stream) {
  if (!plan || !(plan->flags & HSTU_PLAN_BACKWARD)) return HSTU_ERR_INVALID_ARG;
  int rc;
  if (rab && ((rc = check_rab(rab)) != HSTU_OK || (rc = check_rab_grads(dpos, dtime)) != HSTU_OK))
    return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (plan->items.empty()) return zero_rab_grads(rab, dpos, dtime, s);
  rc = check_buffers(q, k, v, dout);
  if (rc != HSTU_OK || (rc = check_buffers(dq, dk, dv, dv)) != HSTU_OK) return rc;
  return launch_backward(reinterpret_cast<const hstu::Item*>(plan->d_bwd), plan->n_bwd, plan->total,
                         plan->heads, plan->d, q, k, v, dout, alpha, inv_n, plan->d_bwd_acc, dq, dk,
                         dv, s, rab, dpos, dtime, plan->d_bwd_hist, plan->d_bwd_first, plan->bwd_grid);
}

int hstu_last_status(int* device_status, int* site) {
  if (!device_status) return HSTU_ERR_INVALID_ARG;
  unsigned st = 0, where = 0;
  if (hstu::read_and_clear_device_status(&st, &where) != cudaSuccess) return HSTU_ERR_CUDA;
  *device_status = (st & 1u) ? HSTU_ERR_TIMEOUT : HSTU_OK;
  if (site) *site = (int)where;
  return HSTU_OK;
}

int hstu_set_wait_timeout_ns(uint64_t ns) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timeout_ns = ns ? ns : 0;
  if (ns == 0) {
    const char* env = std::getenv("HSTU_WAIT_TIMEOUT_NS");
    unsigned long long v = env ? std::strtoull(env, nullptr, 10) : 0ull;
    g_timeout_ns = v ? v : kDefaultTimeoutNs;
  }
  return HSTU_OK;
}

int hstu_set_debug_flags(uint32_t flags) {
  if (flags & ~(uint32_t)(HSTU_DEBUG_UNSIGNALLED_WAIT | HSTU_DEBUG_TRACE | HSTU_DEBUG_NO_PAIRS |
                          HSTU_DEBUG_BWD_ROWS))
    return HSTU_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_debug_flags = flags;
  return HSTU_OK;
}

int hstu_trace_read(uint64_t* dst, int capacity, int* n_events) {
  if (!n_events || capacity < 0) return HSTU_ERR_INVALID_ARG;
  int n = 0;
  if (hstu::read_and_clear_trace(reinterpret_cast<unsigned long long*>(dst), dst ? capacity : 0,
                                 &n) != cudaSuccess)
    return HSTU_ERR_CUDA;
  *n_events = n;
  return HSTU_OK;
}

}  // extern "C"
