// hstu_attn_fwd_noalloc: the forward for callers that cannot allocate.
//
// The work list that hstu_attn_fwd places in a per-call stream-ordered
// allocation lives here in one fixed device array instead.  The host side
// builds the list in a fixed host staging array and copies it in with one
// cudaMemcpyAsync; neither side allocates.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "hstu_attn.h"
#include "hstu_internal.h"

namespace {

constexpr int kMaxItems = HSTU_NOALLOC_MAX_ITEMS;
constexpr int kMaxDevices = 64;

// The work-list array: 1 MiB on every GPU that loads the library, held
// until the process exits.  Shared by every call on that device.
static __device__ __align__(256) hstu::Item g_noalloc_items[kMaxItems];

// Host staging for the list.  A pageable-to-device cudaMemcpyAsync first
// waits for the work already on the stream, then returns once the source
// has been staged, so the array is free again when the call returns; the
// mutex keeps concurrent callers from interleaving.
hstu::Item g_host_items[kMaxItems];
std::mutex g_mu;
hstu::Item* g_dev_ptr[kMaxDevices] = {};

// Device address of g_noalloc_items on the current device (set-up once per
// device).  In host code the array's name only stands in for the symbol.
int items_address(hstu::Item** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HSTU_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return HSTU_ERR_UNSUPPORTED;
  if (!g_dev_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_items) != cudaSuccess || !p) return HSTU_ERR_CUDA;
    g_dev_ptr[dev] = static_cast<hstu::Item*>(p);
  }
  *out = g_dev_ptr[dev];
  return HSTU_OK;
}

}  // namespace

extern "C" int hstu_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                     const int32_t* offsets, int batch, int heads, int d,
                                     int max_seqlen, float alpha, float inv_n, void* out,
                                     hstu_stream_t stream) {
  if (heads < 1 || max_seqlen < 0 || batch < 0) return HSTU_ERR_INVALID_ARG;
  if (d != 32 && d != 64 && d != 128) return HSTU_ERR_UNSUPPORTED;
  if (batch == 0) return HSTU_OK;
  if (!offsets) return HSTU_ERR_INVALID_ARG;
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, offsets) != cudaSuccess) return HSTU_ERR_CUDA;
  if (attr.type == cudaMemoryTypeDevice) return HSTU_ERR_INVALID_ARG;
  int rc = hstu::host_check_offsets(offsets, batch, max_seqlen);
  if (rc != HSTU_OK) return rc;
  const long long total = offsets[batch];
  if (total == 0) return HSTU_OK;
  if ((rc = hstu::host_check_buffers(q, k, v, out)) != HSTU_OK) return rc;

  std::lock_guard<std::mutex> lk(g_mu);
  hstu::Item* d_items = nullptr;
  if ((rc = items_address(&d_items)) != HSTU_OK) return rc;
  const long long n = hstu::count_items(offsets, batch, heads);
  if (n > kMaxItems) return HSTU_ERR_CAPACITY;
  if (n == 0) return HSTU_OK;
  hstu::fill_items(offsets, batch, heads, g_host_items);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(d_items, g_host_items, (size_t)n * sizeof(hstu::Item), cudaMemcpyHostToDevice,
                      s) != cudaSuccess)
    return HSTU_ERR_CUDA;
  return hstu::host_launch(d_items, nullptr, (int)n, total, heads, d, q, k, v, alpha, inv_n, out,
                           nullptr, s);
}
