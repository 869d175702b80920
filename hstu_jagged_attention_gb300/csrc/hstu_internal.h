// Internal interface between the host library (hstu_api.cpp) and the
// sm_103a kernel translation unit (hstu_fwd.cu).  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hstu {

// One work item: 128 query rows of one (sequence, head).
//   x = first token of the sequence, y = sequence length, z = head,
//   w = query block index qt (rows x + 128*qt ...).  Key blocks 0..qt.
using Item = int4;

// Work list (host): number of items, and the items in scheduling order
// (qt descending, then sequence, head, qt ascending).
long long count_items(const int32_t* off, int batch, int heads);
// Static schedule of a longest-first work list over `grid` CTAs, an item
// costing cost[i] + 1 units: order[] (item indices, CTA 0's first) and
// first[grid + 1].  Returns the longest CTA's units.
long long schedule_items(const int32_t* cost, int n, int grid, int32_t* order, int32_t* first);
void fill_items(const int32_t* off, int batch, int heads, Item* dst);
// With candidates (the last num_targets[b] tokens of sequence b see the
// history and themselves only): the same items, each costing
// min(qt, ceil(hist/128)) + 1 key blocks, ordered by cost descending, then
// sequence, head, qt ascending; hist_dst[i] is item i's history length.
void fill_items_targets(const int32_t* off, const int32_t* num_targets, int batch, int heads,
                        Item* dst, int32_t* hist_dst);
// The output stage's arguments (null: plain attention output).
struct NormGate {
  const void* u;
  const float* gamma;
  const float* beta;
  float eps;
  float* xs;
  float2* stats;
};
// Scratch of the output stage in one allocation: xs, then stats (each part
// rounded up to 16 bytes, so that what follows stays aligned).
inline size_t norm_xs_bytes(long long total, int heads, int d) {
  return (size_t)total * (size_t)heads * (size_t)d * sizeof(float);
}
inline size_t norm_stats_bytes(long long total, int heads) {
  return ((size_t)total * (size_t)heads * 2u * sizeof(float) + 15u) & ~(size_t)15u;
}
inline size_t norm_scratch_bytes(long long total, int heads, int d) {
  return norm_xs_bytes(total, heads, d) + norm_stats_bytes(total, heads);
}

struct FwdArgs {
  const Item* items;   // device, n_items entries, longest first
  const int32_t* item_hist;  // device, history length per item; null: no candidates
  int n_items;
  void* out;           // bf16 (total, heads, d): the attention output, or y with the output stage
  // Output stage y = Norm(out) (.) u (null u: none).  u bf16 (total, heads, d);
  // gamma, beta fp32 (heads * d); xs fp32 (total, heads * d) and stats
  // (total, heads): the attention kernel's rows and per-head moments, read
  // by the output-stage kernel (norm_grid blocks) that follows it.
  const void* u;
  const float* gamma;
  const float* beta;
  float eps;
  float* xs;
  float2* stats;
  long long total;
  int norm_grid;
  // Relative attention bias (null rab_ts: none): int32 timestamp per token,
  // fp32 tables of rab_npos and rab_ntime (1..32) entries.
  const int32_t* rab_ts;
  const float* rab_pos;
  const float* rab_time;
  int rab_npos, rab_ntime;
  int heads;
  float half_alpha;    // alpha / 2 (silu(a s) = h + h tanh(h), h = a s / 2)
  float inv_n;
  unsigned long long timeout_ns;
  unsigned debug_flags;  // kDebug* bits; 0 in normal use
};

// Backward pass: items (first token, length, head, key block kt), each
// walking the query blocks kt .. last; dq_acc: fp32 (total, heads, d),
// zeroed before the launch; dq, dk, dv: bf16 (total, heads, d).
struct BwdArgs {
  const Item* items;
  int n_items;
  // device, grid + 1 entries: CTA c runs items cta_first[c] .. cta_first[c + 1] - 1
  // in order (a schedule built on the host); null: CTA c takes items c, c + grid, ...
  const int32_t* cta_first;
  int heads;
  float alpha, inv_n;
  float* dq_acc;
  void* dq;
  void* dk;
  void* dv;
  long long total;
  unsigned long long timeout_ns;
  // The relative attention bias (null rab_ts: none), as FwdArgs; dpos and
  // dtime (rab_npos, rab_ntime fp32, zeroed before the launch) receive the
  // tables' gradients.
  const int32_t* rab_ts = nullptr;
  const float* rab_pos = nullptr;
  const float* rab_time = nullptr;
  int rab_npos = 0, rab_ntime = 0;
  float* dpos = nullptr;
  float* dtime = nullptr;
  // candidates (null: none): each item's history length, parallel to items
  const int32_t* item_hist = nullptr;
  unsigned debug_flags = 0;  // kDebug* bits; 0 in normal use
  // the transposed form (hstu_bwd_t.cuh): d <= 64 without the bias; its Q
  // and dO tensor maps then have 64-row boxes (half a block)
  bool transposed = false;
};
// Work list of the backward: one item per (sequence, head, key block kt),
// costing nq - kt query blocks; ordered by cost descending, then sequence,
// head, kt ascending.
// With num_targets (else null), hist_dst receives each item's history
// length, and a key block of candidates only costs 1.
void fill_items_bwd(const int32_t* off, int batch, int heads, Item* dst,
                    const int32_t* num_targets = nullptr, int32_t* hist_dst = nullptr);
// The backward kernel for head dimension d on `grid` CTAs, then the dQ
// conversion; tdo describes dout like q, tdq the fp32 accumulator as
// (d, heads, total) with box (32, 1, 128) and the 128-byte swizzle.
cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, int grid,
                       cudaStream_t stream);

// Test hook: the MMA warp first waits on a barrier nothing signals.
constexpr unsigned kDebugUnsignalledWait = 1u;
// Tracing: CTA 0 records a clock64 stamp per pipeline event (see
// read_and_clear_trace).
constexpr unsigned kDebugTrace = 2u;
// The plain forward on one CTA per work item even where CTA pairs apply.
constexpr unsigned kDebugNoPairs = 4u;
// The backward in its row form (hstu_bwd.cuh) where the transposed form
// (hstu_bwd_t.cuh) would run: d <= 64 without the bias.
constexpr unsigned kDebugBwdRows = 8u;

// Trace records: {clock64, (event << 48) | (warp << 40) | index}.
cudaError_t read_and_clear_trace(unsigned long long* dst, int capacity, int* n);

// Shared-memory bytes and grid the d-specialised kernel needs.
int fwd_smem_bytes(int d);
constexpr int kFwdThreads = 512;
// Threads of the single-CTA forward kernel for head dimension d, with or
// without the bias, and without the output stage: 768 (four SiLU
// warpgroups) for d <= 64, else kFwdThreads.
int fwd_block_threads(int d, bool rab);

// Launch the persistent kernel for head dimension d on `grid` CTAs (and,
// with the output stage, the output-stage kernel after it).
// The three tensor maps describe q, k, v as (d, heads, total) bf16 with box
// (min(d,64), 1, 128) and the swizzle the kernel expects (fwd_swizzle_bytes).
cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, int grid, cudaStream_t stream);

// Swizzle span in bytes of one shared-memory row for head dimension d (128 or 64).
int fwd_swizzle_bytes(int d);

// The forward on CTA pairs (2-CTA clusters, d = 64 or 128, plain causal):
// items are pair items (first token, length, head, qp), each covering query
// blocks 2 qp and 2 qp + 1 of one (sequence, head); grid is even (two CTAs
// per cluster).  tq describes q as for launch_fwd (box (64, 1, 128)); tk
// describes k with box (64, 1, 64) and the 128-byte swizzle; tv describes v
// with box (d/2, 1, 128) and the swizzle of a d-byte row (64 or 128 bytes).
cudaError_t launch_fwd_pairs(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdArgs& a, int grid, cudaStream_t stream);
int fwd_pair_smem_bytes(int d);

// Pair work list (host): one item per two consecutive query blocks of a
// (sequence, head), (first token, length, head, qp), costing
// min(2 qp + 2, ceil(n / 128)) key blocks; ordered by cost descending, then
// sequence, head, qp ascending.
long long count_pairs(const int32_t* off, int batch, int heads);
void fill_pairs(const int32_t* off, int batch, int heads, Item* dst);

// Device status word (bit 0: a bounded wait gave up) and the code of the
// first wait that gave up; read and cleared together.
cudaError_t read_and_clear_device_status(unsigned* status, unsigned* site);

// Host helpers defined in hstu_api.cpp (argument checks and the launch),
// shared with hstu_noalloc.cu.
int host_check_offsets(const int32_t* off, int batch, long long max_len);
int host_check_buffers(const void* q, const void* k, const void* v, const void* out);
int host_launch(const Item* d_items, const int32_t* d_hist, int n_items, long long total, int heads,
                int d, const void* q, const void* k, const void* v, float alpha, float inv_n,
                void* out, const NormGate* ng, cudaStream_t stream);

}  // namespace hstu
