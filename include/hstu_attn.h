/*
 * hstu_attn.h -- C ABI of the GB300 (sm_103a) HSTU jagged causal attention
 * forward library (libhstu.so).
 *
 * The operation (ai6s.net "HSTU fused operator" post: section 1, the HSTU
 * formula and its PyTorch definition; section 3.2, the in-kernel block mask,
 * lower-triangular including the diagonal, blocks above the diagonal
 * skipped; section 4.2, jagged values + offsets; HSTU paper section 3.1,
 * pointwise aggregated attention without softmax normalisation):
 *
 *   for every sequence b in [0, batch), head h in [0, heads) and token t with
 *   offsets[b] <= t < offsets[b+1]:
 *
 *     out[t,h,:] = inv_n * sum_{j = offsets[b]..t} silu(alpha * <q[t,h,:], k[j,h,:]>) * v[j,h,:]
 *
 *   with silu(x) = x * sigmoid(x).  No (s x s) score or mask buffer is ever
 *   materialised.  A dense (batch, s, heads, d) token-major tensor is the
 *   case offsets[b] = b * s; a head-major (batch, heads, s, d) tensor must
 *   be permuted to token-major by the caller first.
 *
 * Layout.  q, k, v and out are contiguous row-major bf16 arrays of shape
 * (total, heads, d), total = offsets[batch]; the row stride is heads*d
 * elements.  Base addresses must be 16-byte aligned.  offsets is int32 with
 * batch+1 entries, offsets[0] == 0, non-decreasing; empty sequences are
 * allowed and produce no rows.  d must be 32, 64 or 128.
 *
 * Precision.  bf16 inputs; Q.K^T and P.V accumulate in fp32 on the tensor
 * cores; silu in fp32; P is passed to the P.V product as the exact split
 * P = P_hi + P_lo of two bf16 terms; the output is rounded to bf16
 * (round to nearest even).
 *
 * Ownership and synchronisation.  The caller owns every buffer.  Calls are
 * asynchronous on the given stream (a cudaStream_t; NULL = legacy default
 * stream) and return once the work is enqueued.  Outputs are complete when
 * the stream reaches that point.  Nothing here synchronises the device
 * except where a function says so (hstu_attn_fwd_noalloc waits for the
 * stream's earlier work; see there).
 *
 * Errors.  Every function returns HSTU_OK (0) or a negative hstu_status.
 * Argument checks happen before anything is enqueued; on an argument error
 * nothing is written.  Device-side waits inside the kernel are bounded: a
 * wait that runs out sets a device status word that hstu_last_status()
 * reports as HSTU_ERR_TIMEOUT, and the kernel returns instead of hanging.
 * No C++ exception crosses this interface.
 */
#ifndef HSTU_ATTN_H_
#define HSTU_ATTN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
typedef enum hstu_status {
  HSTU_OK = 0,
  HSTU_ERR_INVALID_ARG = -1, /* bad pointer, size, offsets or alignment */
  HSTU_ERR_UNSUPPORTED = -2, /* d not in {32, 64, 128}, or the device is not sm_103 */
  HSTU_ERR_CUDA = -3,        /* a CUDA runtime or driver call failed */
  HSTU_ERR_TIMEOUT = -4,     /* a bounded device-side wait ran out (see hstu_last_status) */
  HSTU_ERR_NO_MEMORY = -5,   /* host or device allocation failed */
  HSTU_ERR_CAPACITY = -6     /* work list exceeds HSTU_NOALLOC_MAX_ITEMS (hstu_attn_fwd_noalloc) */
} hstu_status;

/* Same type as cudaStream_t, declared here so this header needs no CUDA headers. */
typedef struct CUstream_st* hstu_stream_t;

/* Opaque, reusable launch plan for one offsets array (see hstu_plan_create). */
typedef struct hstu_plan hstu_plan;

/* Rows of queries per work item and keys per K/V block (both 128). */
#define HSTU_BLOCK_M 128
#define HSTU_BLOCK_N 128

/*
 * hstu_attn_fwd -- the forward operation above, in one call.
 *
 *   q, k, v      device pointers, bf16 (total, heads, d), read only.
 *   offsets      int32[batch+1]; a host pointer or a device pointer (told
 *                apart with cudaPointerGetAttributes).  A device pointer is
 *                copied to the host first, which synchronises `stream`.
 *   batch        number of sequences (>= 0; 0 is a no-op).
 *   heads        number of heads (>= 1).
 *   d            head dimension: 32, 64 or 128.
 *   max_seqlen   upper bound on every sequence length; used for validation
 *                only (it is not the 1/n normaliser).
 *   alpha        the score scale: silu(alpha * q.k).
 *   inv_n        the output scale 1/n.
 *   out          device pointer, bf16 (total, heads, d), written.  Every
 *                row of every sequence is written; no other byte is.
 *   stream       CUDA stream the work is enqueued on.
 *
 * Builds the work list on the host (as hstu_plan_create), copies it to a
 * stream-ordered device allocation that is released on the same stream
 * after the kernel, and launches.  Errors: HSTU_ERR_INVALID_ARG (offsets
 * not starting at 0, decreasing, a length above max_seqlen, null or
 * misaligned buffers), HSTU_ERR_UNSUPPORTED, HSTU_ERR_CUDA,
 * HSTU_ERR_NO_MEMORY.
 */
int hstu_attn_fwd(const void* q, const void* k, const void* v, const int32_t* offsets, int batch,
                  int heads, int d, int max_seqlen, float alpha, float inv_n, void* out,
                  hstu_stream_t stream);

/*
 * hstu_attn_fwd_noalloc -- hstu_attn_fwd for callers that cannot allocate.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that own every byte of device memory themselves -- a serving process with
 * a fixed memory budget, or a framework whose allocator must not be
 * bypassed -- and so cannot let the library call cudaMalloc or
 * cudaMallocAsync, which may also synchronise or fail under memory
 * pressure in the middle of a request.  It computes exactly what
 * hstu_attn_fwd computes and calls no allocating routine, on the host or
 * the device.
 *
 * Instead of a per-call device allocation, the work list goes into one
 * fixed array of HSTU_NOALLOC_MAX_ITEMS items (16 bytes each, 1 MiB) that
 * lives in the library's device memory on every GPU that loads it, until
 * the process exits.  Consequences:
 *   - A call whose work list would exceed HSTU_NOALLOC_MAX_ITEMS (one item
 *     per 128 query rows of each sequence and head) is rejected with
 *     HSTU_ERR_CAPACITY before anything is enqueued.
 *   - All calls on a device share the array.  Calls enqueued on one stream
 *     run one after the other and are safe; calls whose work overlaps on
 *     the GPU (other streams, other threads) overwrite each other's work
 *     list and give wrong results.  Each call writes every entry it reads,
 *     so nothing needs clearing between calls.
 *   - The list is built on the host in a fixed pageable array and copied
 *     in with cudaMemcpyAsync.  A copy from pageable memory first waits
 *     for the work already enqueued on `stream`, so unlike hstu_attn_fwd
 *     this call blocks the calling thread until that earlier work has
 *     finished (the attention kernel itself is still only enqueued).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, once per device, with that device current);
 *     make that first call before any stream capture.
 *
 *   offsets    host pointer only, int32[batch+1] (a device pointer is
 *              rejected with HSTU_ERR_INVALID_ARG, since copying it back
 *              would need host staging).
 * Other arguments, layout and errors as hstu_attn_fwd.
 */
#define HSTU_NOALLOC_MAX_ITEMS 65536
int hstu_attn_fwd_noalloc(const void* q, const void* k, const void* v, const int32_t* offsets,
                          int batch, int heads, int d, int max_seqlen, float alpha, float inv_n,
                          void* out, hstu_stream_t stream);

/*
 * hstu_attn_fwd_host -- hstu_attn_fwd from host buffers to host buffers,
 * with the copies overlapped with the kernel.
 *
 * No page defines this call; it serves callers whose q, k, v come from
 * and whose out goes to host memory (a serving process fed from the host).
 * The sequences are split into n_chunks runs of whole sequences with about
 * equal token counts (0: min(batch, 4)).  Chunk c's q, k, v rows are copied
 * in on an internal stream, its forward runs on `stream` once they have
 * landed, and its out rows are copied back on a second internal stream.
 * So chunk c + 1's copy in and chunk c - 1's copy out run under chunk c's
 * kernel.  Each output row is computed by the same kernel arithmetic as
 * hstu_attn_fwd's, so the two agree bit for bit.
 *
 *   q_host, k_host, v_host  host, (total, heads, d) bf16 row-major.
 *   out_host                host, (total, heads, d) bf16, written.
 *   q_dev, k_dev, v_dev,    device staging of the same shape, owned by the
 *   out_dev                 caller (16-byte aligned), overwritten; q_dev,
 *                           k_dev, v_dev and out_dev must not overlap.
 *   offsets                 host pointer only, int32[batch+1].
 *   n_chunks                >= 0; more chunks than sequences are capped.
 * The host buffers must stay valid, and out_host must not be read, until
 * `stream` reaches the end of the call.  Page-locked host memory
 * (cudaHostAlloc, cudaHostRegister) lets the copies run asynchronously and
 * overlap.  With pageable memory each copy waits for earlier work on its
 * stream and the call blocks the calling thread.
 * The two internal streams (non-blocking, one pair per device, created on
 * first use and kept until exit) are joined to `stream` by events: work
 * enqueued on `stream` before the call is done before the first copy, and
 * work enqueued after it sees out_host written.  The work list goes into a
 * stream-ordered allocation on `stream`, as in hstu_attn_fwd.
 * A chunk's kernel may read, through the last 128-row tile of its last
 * sequence, staged rows of the next chunk while they are being copied in.
 * Those rows only feed masked terms, so the results do not depend on them.
 * Errors: as hstu_attn_fwd, and HSTU_ERR_INVALID_ARG for a device offsets
 * pointer, a negative n_chunks or a null host buffer; those are found
 * before anything is enqueued.  A CUDA error while enqueuing (after the
 * first copy) returns HSTU_ERR_CUDA with part of the work enqueued and
 * `stream` not joined to the internal streams: synchronise the device
 * before reusing the buffers.
 */
int hstu_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                       const int32_t* offsets, int batch, int heads, int d, int max_seqlen,
                       float alpha, float inv_n, void* out_host, void* q_dev, void* k_dev,
                       void* v_dev, void* out_dev, int n_chunks, hstu_stream_t stream);

/*
 * hstu_host_runs -- the runs of whole sequences hstu_attn_fwd_host takes
 * for these offsets and n_chunks, on the host only (no CUDA call).
 *   host_offsets  int32[batch+1], validated as in hstu_attn_fwd.
 *   n_runs        out: min(batch, n_chunks), or min(batch, 4) for 0.
 *   host_first    int32[n_runs + 1], out (NULL: only *n_runs): run c is
 *                 sequences host_first[c] .. host_first[c + 1] - 1.
 *   capacity      entries host_first holds (>= n_runs + 1).
 * Run c (c < n_runs - 1) ends before the first sequence that starts at
 * or past token floor(total * (c + 1) / n_runs), and after run c - 1; the
 * last run ends at batch.  So every run holds at most about total / n_runs
 * tokens plus one sequence, and a run may be empty.
 * Errors: HSTU_ERR_INVALID_ARG for a NULL offsets or n_runs pointer,
 * negative batch or n_chunks, invalid offsets or a short capacity.
 */
int hstu_host_runs(const int32_t* host_offsets, int batch, int n_chunks, int32_t* host_first,
                   int capacity, int* n_runs);

/*
 * hstu_plan_create -- validate host offsets and build the device work list once.
 *
 * The work list holds one item per (sequence, head, 128-row query block);
 * query block qt needs key blocks 0..qt (the blocks above the diagonal are
 * skipped, ai6s.net post section 3.2), and items are ordered longest first
 * (qt descending, then sequence, head, qt ascending) for the persistent
 * kernel's scheduler.  The plan owns its device buffer (allocated with
 * cudaMalloc on the current device) and is immutable after creation, so
 * one plan may be used by several streams at once.
 *
 *   host_offsets  int32[batch+1], host memory, read during the call only.
 *   *plan         receives the new plan; set to NULL on error.
 *
 * Errors: as hstu_attn_fwd (argument checks), HSTU_ERR_NO_MEMORY.
 */
int hstu_plan_create(const int32_t* host_offsets, int batch, int heads, int d, int max_seqlen,
                     hstu_plan** plan);

/*
 * hstu_attn_fwd_plan -- the forward operation for a plan's offsets and shape.
 * Arguments as hstu_attn_fwd.  Enqueues exactly one kernel (none when the
 * plan has no work items) and allocates nothing.
 *
 * At d = 64 and 128 the plain operation can also run on CTA pairs (two-CTA
 * clusters whose tensor products cover 256 query rows over both SMs; see
 * hstu_worklist_build_pairs) in plans made with HSTU_PLAN_PAIRS; the
 * result is the same operation within the stated precision.
 */
int hstu_attn_fwd_plan(const hstu_plan* plan, const void* q, const void* k, const void* v,
                       float alpha, float inv_n, void* out, hstu_stream_t stream);

/* Release a plan (device memory freed with cudaFree).  NULL is accepted. */
int hstu_plan_destroy(hstu_plan* plan);

/* Number of work items in a plan. */
int hstu_plan_num_items(const hstu_plan* plan, int* n_items);

/* Number of pair items in a plan: 0 when the plan runs on one CTA per item. */
int hstu_plan_num_pairs(const hstu_plan* plan, int* n_pairs);

/*
 * hstu_plan_worklist -- copy a plan's host-side work list out.
 *
 *   host_dst   int32[4 * capacity] or NULL; item i is
 *              (first token of its sequence, sequence length, head, qt).
 *   capacity   entries host_dst can hold.
 *   *n_items   receives the item count (also when host_dst is NULL).
 * Errors: HSTU_ERR_INVALID_ARG if capacity is too small for a non-NULL host_dst.
 */
int hstu_plan_worklist(const hstu_plan* plan, int32_t* host_dst, int capacity, int* n_items);

/*
 * hstu_worklist_build -- the same work list, computed on the host only (no
 * CUDA call): validates offsets as hstu_plan_create does (with max_seqlen
 * taken as unbounded) and writes up to `capacity` items into host_dst.
 * *n_items receives the full count; host_dst may be NULL to query it.
 */
int hstu_worklist_build(const int32_t* host_offsets, int batch, int heads, int32_t* host_dst,
                        int capacity, int* n_items);

/*
 * hstu_worklist_schedule -- the static per-CTA schedule that the backward
 * (hstu_attn_bwd*, and plans made with HSTU_PLAN_BACKWARD) gives its work
 * list, on the host only (no CUDA call).  The forward keeps the
 * longest-first list, which its CTAs take serpentine.
 *
 *   host_cost   int32[n_items]: each item's blocks (>= 1), in the order of
 *               a longest-first list (the backward's: query blocks walked).
 *   grid        CTAs, 1 .. n_items (launches use min(items, SMs)).
 *   host_order  int32[n_items], out: item indices, CTA 0's items first,
 *               each CTA's in list order.
 *   host_first  int32[grid + 1], out: CTA c runs host_order[host_first[c]]
 *               .. host_order[host_first[c + 1] - 1].
 *   makespan    out (NULL: not wanted): the longest CTA's units.
 * List scheduling: an item takes cost + 1 units (its blocks, plus its
 * loads and stores) and goes, in list order, to the CTA that is free first
 * (ties: the lower CTA), so no CTA runs more than one item's units past the
 * mean.
 * Errors: HSTU_ERR_INVALID_ARG for a NULL array, n_items < 1, grid outside
 * 1 .. n_items or a cost < 1.
 */
int hstu_worklist_schedule(const int32_t* host_cost, int n_items, int grid, int32_t* host_order,
                           int32_t* host_first, long long* makespan);

/*
 * hstu_worklist_build_pairs -- the work list of CTA pairs, on the host only.
 *
 * A pair item covers two consecutive query blocks, 2 qp and 2 qp + 1 (256
 * rows), of one (sequence, head); the two CTAs of a cluster take one block
 * each and walk the key blocks 0 .. min(2 qp + 1, nq - 1) together
 * (nq = ceil(n / 128)), so an item costs min(2 qp + 2, nq) key blocks; a
 * sequence with an odd number of blocks ends in a pair whose second block
 * is empty.  Items (first token, length, head, qp), ordered by cost
 * descending, then sequence, head, qp ascending.  Arguments and errors as
 * hstu_worklist_build.
 */
int hstu_worklist_build_pairs(const int32_t* host_offsets, int batch, int heads, int32_t* host_dst,
                              int capacity, int* n_items);

/*
 * Candidates (M-FALCON): HSTU paper section 3.4 and Appendix H, Algorithm 1.
 *
 * For ranking, the last num_targets[b] tokens of sequence b are candidates
 * that must not see one another: with hist = n_b - num_targets[b] (the
 * history) the causal sum above is further restricted, for token t = the
 * i-th of its sequence, to
 *
 *     keys j (sequence-local) with  j <= i  and  (j < hist  or  j == i),
 *
 * so each candidate's output equals that of a separate causal pass over the
 * history followed by that candidate alone.  Query block qt then needs only
 * the key blocks that hold history keys, 0 .. min(qt, ceil(hist/128)) - 1,
 * and its diagonal block qt; its work item costs min(qt, ceil(hist/128)) + 1
 * key blocks.  num_targets[b] = 0 everywhere is the causal operation.
 *
 *   host_num_targets  int32[batch], host memory, 0 <= num_targets[b] <= n_b;
 *                     read during the call only.
 *
 * hstu_attn_fwd_targets    as hstu_attn_fwd, with the candidate mask.
 * hstu_plan_create_targets as hstu_plan_create; hstu_attn_fwd_plan then
 *                          applies the mask.  Items are ordered by cost
 *                          descending, then sequence, head, qt ascending.
 * hstu_plan_item_hist      copies each item's history length (the sequence
 *                          length for a plan without candidates).
 * hstu_worklist_build_targets  the host-only work list: items as
 *                          hstu_worklist_build, and each item's history length.
 * Errors: as the causal counterparts; HSTU_ERR_INVALID_ARG also for a NULL
 * host_num_targets with batch > 0 or a count outside [0, n_b].
 */
int hstu_attn_fwd_targets(const void* q, const void* k, const void* v, const int32_t* offsets,
                          const int32_t* host_num_targets, int batch, int heads, int d,
                          int max_seqlen, float alpha, float inv_n, void* out, hstu_stream_t stream);
int hstu_plan_create_targets(const int32_t* host_offsets, const int32_t* host_num_targets, int batch,
                             int heads, int d, int max_seqlen, hstu_plan** plan);
int hstu_plan_item_hist(const hstu_plan* plan, int32_t* host_dst, int capacity, int* n_items);
int hstu_worklist_build_targets(const int32_t* host_offsets, const int32_t* host_num_targets,
                                int batch, int heads, int32_t* host_items, int32_t* host_hist,
                                int capacity, int* n_items);

/*
 * Output stage Norm(A V) (.) U: HSTU paper section 3 (the layer's pointwise
 * transformation after the spatial aggregation), section 3.1 (a layer norm
 * must follow the pointwise pooling) and the feature-interaction paragraph,
 * which writes the term as Norm(A(X) V(X)) (.) U(X).  The paper's equations
 * are lost in extraction; the operation implemented is the plain reading:
 *
 *     x[t, :]  = the attention output of token t, all heads concatenated
 *                (heads * d values, fp32 inside the kernel, never rounded)
 *     y[t, c]  = ((x[t,c] - mean_t) / sqrt(var_t + eps) * gamma[c] + beta[c]) * u[t, c]
 *
 * with mean_t and var_t (biased, 1/(heads*d)) over the heads * d values of
 * token t.  U is taken as given: it already went through the SiLU of the
 * layer's first sub-layer.  Dropout is not applied.
 *
 *   u      bf16 device ptr, (total, heads, d) like q; 16-byte aligned.
 *   gamma, beta  fp32 device ptrs, heads * d entries each (index h * d + c);
 *          16-byte aligned.
 *   eps    finite, >= 0.
 *   y      bf16 device ptr, (total, heads, d); caller-allocated, written for
 *          every token (bf16, round to nearest even).  The attention output
 *          itself is not stored.
 *
 * The norm spans all heads of a token, while each work item is one head,
 * so the call enqueues two kernels on the stream.  The attention kernel's
 * epilogue writes every row's fp32 values and, per row and head, their mean
 * and M2 to a scratch; an output-stage kernel then merges the heads'
 * moments, normalises, applies gamma and beta and gates by U.  Scratch:
 * 4 * total * heads * d bytes (rows) and 8 * total * heads (moments).
 *
 * hstu_plan_create_ex       as hstu_plan_create_targets (host_num_targets
 *                           may be NULL: no candidates) with flags.
 *                           HSTU_PLAN_NORM_GATE makes the plan own the
 *                           output stage's scratch.  Such a plan also serves
 *                           hstu_attn_fwd_plan.
 * hstu_attn_fwd_norm_gate_plan  y for a HSTU_PLAN_NORM_GATE plan (else
 *                           HSTU_ERR_INVALID_ARG); asynchronous on stream.
 *                           Launches on one stream at a time per plan: the
 *                           scratch is shared by its launches.
 * hstu_attn_fwd_norm_gate   the one-shot form: offsets as hstu_attn_fwd,
 *                           host_num_targets may be NULL; the scratch is
 *                           allocated and freed stream-ordered.
 * Errors: as hstu_attn_fwd; HSTU_ERR_INVALID_ARG also for a NULL or
 * misaligned u, gamma, beta, a negative or non-finite eps, or unknown flags.
 */
#define HSTU_PLAN_NORM_GATE 1u
typedef struct hstu_norm_gate {
  const void* u;        /* bf16 (total, heads, d), 16-byte aligned */
  const float* gamma;   /* fp32 heads * d, 16-byte aligned */
  const float* beta;    /* fp32 heads * d, 16-byte aligned */
  float eps;            /* finite, >= 0 */
} hstu_norm_gate;
int hstu_plan_create_ex(const int32_t* host_offsets, const int32_t* host_num_targets, int batch,
                        int heads, int d, int max_seqlen, uint32_t flags, hstu_plan** plan);

/*
 * The candidates' rows only -- HSTU paper section 3.4 (M-FALCON): the
 * history's keys and values are computed once and serve every batch of
 * candidates.  A plan made by hstu_plan_create_ex with host_num_targets
 * and HSTU_PLAN_CANDIDATES_ONLY keeps only the work items of query blocks
 * that hold a candidate row (qt >= hist / 128, num_targets[b] > 0).  So
 * hstu_attn_fwd_plan and hstu_attn_fwd_plan_ex (rab allowed, ng not)
 * compute:
 *   - every candidate row, as with the full candidate mask;
 *   - the history rows that share a 128-row block with the first
 *     candidates, with the same values as the full pass;
 *   - no other history row: those rows of out are left as they were.
 * The keys and values of the history are read from k and v: these hold the
 * cached history followed by the candidates.
 *
 * HSTU_PLAN_CANDIDATES_ONLY needs host_num_targets; with
 * HSTU_PLAN_NORM_GATE or HSTU_PLAN_BACKWARD: HSTU_ERR_INVALID_ARG.
 * hstu_worklist_build_candidates  the host-only work list of such a plan
 * (items and their history lengths, as hstu_worklist_build_targets).
 */
#define HSTU_PLAN_CANDIDATES_ONLY 4u
/*
 * HSTU_PLAN_PAIRS: build the CTA-pair work list whenever the plain forward
 * can run on CTA pairs (d = 64 or 128, no host_num_targets), not only when
 * the pairs waste little work on these offsets; hstu_attn_fwd_plan and
 * hstu_attn_fwd_plan_ex without rab and ng then use it.  With
 * host_num_targets: HSTU_ERR_INVALID_ARG.  At d = 32 it has no effect.
 */
#define HSTU_PLAN_PAIRS 8u
int hstu_worklist_build_candidates(const int32_t* host_offsets, const int32_t* host_num_targets,
                                   int batch, int heads, int32_t* host_items, int32_t* host_hist,
                                   int capacity, int* n_items);

/*
 * Relative attention bias rab_{p,t}: HSTU paper section 3 (a bias that
 * merges relative position p and time t, added inside the attention's
 * nonlinearity), section 3.4 (M-FALCON modifies it for candidates) and
 * Appendix G (its construction fused into the attention operator).  The
 * construction is lost in extraction; the reading implemented is a pair of
 * bucketed tables added to the scaled score:
 *
 *   score(i, j) = alpha * <q_i, k_j> + pos[min(floor(log2(dp + 1)), num_pos - 1)]
 *                                    + time[min(floor(log2(dt + 1)), num_time - 1)]
 *   dp = p(i) - p(j),  dt = max(ts_i - ts_j, 0)
 *
 * with sequence-local positions p(i) = i, except that every candidate
 * (with host_num_targets) sits at p = hist, as in its own causal pass.
 *
 *   timestamps  device int32, one per token, in [0, 2^31); 4-byte aligned.
 *   pos, time   device fp32 tables of num_pos and num_time entries, 1..32
 *               each (log2 buckets of 32-bit differences never exceed 31).
 */
typedef struct hstu_rab {
  const int32_t* timestamps;
  const float* pos;
  int num_pos;
  const float* time;
  int num_time;
} hstu_rab;

/*
 * hstu_attn_fwd_plan_ex / hstu_attn_fwd_ex -- every option in one call:
 * rab (NULL: no bias) and ng (NULL: out is the attention output; else out
 * is y of the output stage, and a plan needs HSTU_PLAN_NORM_GATE).  The
 * one-shot form takes host_num_targets (NULL: none) as
 * hstu_attn_fwd_targets.  Errors: as the specific calls, and
 * HSTU_ERR_INVALID_ARG for NULL or misaligned rab pointers or table sizes
 * outside 1..32.
 */
int hstu_attn_fwd_plan_ex(const hstu_plan* plan, const void* q, const void* k, const void* v,
                          const hstu_rab* rab, const hstu_norm_gate* ng, float alpha, float inv_n,
                          void* out, hstu_stream_t stream);
int hstu_attn_fwd_ex(const void* q, const void* k, const void* v, const int32_t* offsets,
                     const int32_t* host_num_targets, int batch, int heads, int d, int max_seqlen,
                     const hstu_rab* rab, const hstu_norm_gate* ng, float alpha, float inv_n,
                     void* out, hstu_stream_t stream);
int hstu_attn_fwd_norm_gate_plan(const hstu_plan* plan, const void* q, const void* k, const void* v,
                                 const void* u, const float* gamma, const float* beta, float eps,
                                 float alpha, float inv_n, void* y, hstu_stream_t stream);
int hstu_attn_fwd_norm_gate(const void* q, const void* k, const void* v, const void* u,
                            const float* gamma, const float* beta, float eps, const int32_t* offsets,
                            const int32_t* host_num_targets, int batch, int heads, int d,
                            int max_seqlen, float alpha, float inv_n, void* y,
                            hstu_stream_t stream);

/*
 * Backward pass -- HSTU paper Appendix G: the backward recomputes the
 * attention (no (s x s) buffer is kept from the forward) and its gradients
 * are those of the forward definition.  For dout = d out:
 *
 *   dv[j] = sum_i P_ij dout[i],   P_ij = inv_n silu(alpha q_i.k_j)   (kept pairs)
 *   ds_ij = inv_n silu'(alpha q_i.k_j) <dout[i], v[j]>
 *   dq[i] = alpha sum_j ds_ij k[j],   dk[j] = alpha sum_i ds_ij q[i]
 *
 * over the causal pairs of each sequence, silu'(x) = sig(x) (1 + x (1 - sig(x))).
 *
 * hstu_attn_bwd  q, k, v, dout: bf16 device (total, heads, d); dq, dk, dv:
 *                bf16 device (total, heads, d), written for every token.
 *                offsets, batch, heads, d, max_seqlen, alpha, inv_n as
 *                hstu_attn_fwd.  Enqueues, on `stream`: a zeroing of an
 *                fp32 dQ accumulator (4 * total * heads * d bytes, allocated
 *                and freed stream-ordered with the work list), the backward
 *                kernel and the dQ conversion.  One work item per (sequence,
 *                head, 128-key block kt) walks the query blocks kt .. last.
 * hstu_worklist_build_bwd  the host-only work list: items (first token,
 *                length, head, kt), costing nq - kt query blocks, ordered by
 *                cost descending, then sequence, head, kt ascending.
 * Errors: as hstu_attn_fwd (all seven buffers non-null and 16-byte aligned).
 */
int hstu_attn_bwd(const void* q, const void* k, const void* v, const void* dout,
                  const int32_t* offsets, int batch, int heads, int d, int max_seqlen, float alpha,
                  float inv_n, void* dq, void* dk, void* dv, hstu_stream_t stream);
/* The backward on a plan made by hstu_plan_create_ex with HSTU_PLAN_BACKWARD
 * (host_num_targets given: with the candidate mask, as the forward's): the
 * plan owns the backward work list and the fp32 dQ accumulator; launches on
 * one stream at a time per plan.  A plan without the flag:
 * HSTU_ERR_INVALID_ARG. */
#define HSTU_PLAN_BACKWARD 2u
int hstu_attn_bwd_plan(const hstu_plan* plan, const void* q, const void* k, const void* v,
                       const void* dout, float alpha, float inv_n, void* dq, void* dk, void* dv,
                       hstu_stream_t stream);
int hstu_worklist_build_bwd(const int32_t* host_offsets, int batch, int heads, int32_t* host_dst,
                            int capacity, int* n_items);
/* The backward's work list with candidates: as hstu_worklist_build_bwd,
 * except that a key block without history keys (128 kt >= hist) is seen by
 * its own rows only and costs 1; host_hist receives each item's history
 * length.  Arguments as hstu_worklist_build_targets. */
int hstu_worklist_build_bwd_targets(const int32_t* host_offsets, const int32_t* host_num_targets,
                                    int batch, int heads, int32_t* host_items, int32_t* host_hist,
                                    int capacity, int* n_items);

/*
 * hstu_attn_bwd_ex / hstu_attn_bwd_plan_ex -- the backward with candidates
 * and the relative attention bias.  host_num_targets (NULL: none) as
 * hstu_attn_fwd_targets: the gradients are those of the forward with the
 * candidate mask, the kept pairs being the mask's.  rab NULL: no bias (as
 * hstu_attn_bwd / _plan).  The score
 * is that of hstu_rab, ds_ij = inv_n silu'(score_ij) <dout[i], v[j]>, dq, dk
 * and dv as above, and the tables' gradients (HSTU paper Appendix G: the
 * bias's construction and its backward fused into the attention):
 *
 *   dpos[b]  = sum of ds_ij over the kept pairs and heads whose position
 *              bucket is b (the clamped bucket: b = num_pos - 1 collects
 *              every larger one); dtime likewise over the time buckets.
 *
 *   dpos, dtime  device fp32 of num_pos and num_time entries, 4-byte
 *                aligned, overwritten (zeroed on `stream`, then added into
 *                by the kernel's float atomics, so their last bits may vary
 *                from run to run).  Ignored when rab is NULL.
 * Errors: as hstu_attn_bwd, and HSTU_ERR_INVALID_ARG for the rab checks of
 * hstu_attn_fwd_ex or NULL / misaligned dpos or dtime (with rab).
 */
int hstu_attn_bwd_ex(const void* q, const void* k, const void* v, const void* dout,
                     const int32_t* offsets, const int32_t* host_num_targets, int batch, int heads,
                     int d, int max_seqlen, const hstu_rab* rab, float alpha, float inv_n, void* dq,
                     void* dk, void* dv, float* dpos, float* dtime, hstu_stream_t stream);
int hstu_attn_bwd_plan_ex(const hstu_plan* plan, const void* q, const void* k, const void* v,
                          const void* dout, const hstu_rab* rab, float alpha, float inv_n, void* dq,
                          void* dk, void* dv, float* dpos, float* dtime, hstu_stream_t stream);

/*
 * hstu_launch_shape -- the grid the next launch for `plan` would use on the
 * current device: *grid persistent CTAs of *block threads with *smem_bytes
 * of dynamic shared memory.  Queries device attributes; launches nothing.
 * *block is that of a call without the output stage: 768 for d <= 64
 * (four SiLU warpgroups), 512 for d = 128 and for pair plans; a call with
 * the output stage runs 512.
 */
int hstu_launch_shape(const hstu_plan* plan, int* grid, int* block, int* smem_bytes);

/*
 * hstu_last_status -- read and clear the device-side status word of the
 * current device.  Synchronises the device.  *device_status receives
 * HSTU_OK, or HSTU_ERR_TIMEOUT if a kernel since the last call gave up on a
 * bounded wait; *site (may be NULL) receives an internal code of the first
 * wait that gave up (0 if none).  Kernels running concurrently share the
 * word.
 */
int hstu_last_status(int* device_status, int* site);

/*
 * hstu_set_wait_timeout_ns -- limit, in nanoseconds of %globaltimer, for
 * any single device-side wait in kernels launched after this call
 * (process-wide; default 4e9, or the HSTU_WAIT_TIMEOUT_NS environment
 * variable).  0 restores the default.  A tiny limit makes the kernel give up
 * at its first wait that is not already satisfied; tests use this to check
 * that the give-up path returns instead of hanging.
 */
int hstu_set_wait_timeout_ns(uint64_t ns);

/*
 * hstu_set_debug_flags -- test hooks for kernels launched after this call
 * (process-wide; 0 = none, the default).
 *   HSTU_DEBUG_UNSIGNALLED_WAIT  the kernel first waits on a barrier that
 *       nothing signals, so its bounded wait runs out after the limit of
 *       hstu_set_wait_timeout_ns; the kernel then drains its own copies,
 *       frees TMEM, returns, and hstu_last_status reports HSTU_ERR_TIMEOUT.
 *       The output is not written.  Used to test the give-up path without
 *       hanging or faulting the GPU.
 *   HSTU_DEBUG_TRACE  record the pipeline trace (see hstu_trace_read).
 *   HSTU_DEBUG_NO_PAIRS  run the plain forward on one CTA per work item even
 *       where a plan or call would use CTA pairs (for comparing the two).
 *   HSTU_DEBUG_BWD_ROWS  run the backward in its row form (query rows on
 *       the TMEM lanes) where it would run in its transposed form (key rows
 *       on the lanes: d <= 64 without the bias), for comparing the two.
 * The unsignalled wait applies to the forward and to the backward's
 * transposed form.
 * Errors: HSTU_ERR_INVALID_ARG for unknown bits.
 */
#define HSTU_DEBUG_UNSIGNALLED_WAIT 1u
#define HSTU_DEBUG_TRACE 2u
#define HSTU_DEBUG_NO_PAIRS 4u
#define HSTU_DEBUG_BWD_ROWS 8u
int hstu_set_debug_flags(uint32_t flags);

/*
 * hstu_trace_read -- the pipeline trace of the last kernels launched with
 * HSTU_DEBUG_TRACE set (read and cleared; synchronises the device).
 *
 * With the flag set, the first CTA of each launch records one event per
 * pipeline step from lane 0 of the warp taking it: TMA loads issued (Q, K,
 * V), QK and PV products issued, SiLU start/end of each block, epilogue
 * start/end of each item.  Event i occupies dst[2i] = clock64 of the SM and
 * dst[2i+1] = (event code << 48) | (warp << 40) | index, index being the
 * running block, ring or item counter of that role.  Event codes: 1 QK
 * issue starts, 2 PV issue starts, 3 SiLU start, 4 SiLU end, 5 epilogue
 * start, 6 epilogue end, 7 K load, 8 V load, 9 Q load, 10 K block present
 * at the MMA warp, 11 QK issued, 12 P present at the MMA warp, 13 PV
 * issued.  Up to 2048 events per warp are kept, grouped by warp;
 * `capacity` counts events (dst holds 2*capacity words).
 */
int hstu_trace_read(uint64_t* dst, int capacity, int* n_events);

/* Static description of a status code. */
const char* hstu_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* HSTU_ATTN_H_ */
