// Page selection without a caller-provided workspace.
//
// oomb_page_select needs a few MB of device scratch (per-block query partial sums,
// the mean query and one score per candidate page) that the caller normally
// allocates and passes in.  Some callers cannot allocate device memory at all:
// a host framework that owns every device allocation through its own pool and
// forbids any other, a steady-state training or serving loop in which a
// cudaMalloc (which can synchronize the device and can fail under memory
// pressure) is not allowed, or a plain C host that links only this library and
// has no allocator of its own.  For them this file keeps the scratch in a
// fixed-size static device array that every GPU loading the library holds until
// the process exits, and forwards to oomb_page_select with it.
#include <atomic>
#include <mutex>

#include "oomb_internal.h"

namespace {

// Largest scratch the static array provides: 4 MiB.  It covers, for example,
// 4 KV heads x head_dim 128 with up to 225,280 logical pages (28.8M tokens at 128
// tokens per page), or 8 KV heads x head_dim 128 with up to 94,208.
constexpr size_t kNoAllocSelectBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_select_scratch[kNoAllocSelectBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of g_select_scratch on the current device, looked up once per
// device (the first call on a device does this; it must not be inside a stream
// capture).  The host-side symbol g_select_scratch is not a device address.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
      e = cudaGetSymbolAddress(&p, g_select_scratch);
      if (e != cudaSuccess) return e;
      if (!p) return cudaErrorInvalidSymbol;
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" oomb_status oomb_page_select_noalloc(oomb_pool* pool, const void* q, int64_t q_start, int n_q,
                                                int top_k, int n_sink, int32_t* sel, int32_t* sel_count,
                                                int max_sel, void* stream) {
  if (!pool) return OOMB_ERR_ARG;
  const size_t need = oomb_workspace_size(pool, OOMB_OP_SELECT, n_q);
  if (need == 0) return OOMB_ERR_ARG;
  if (need > kNoAllocSelectBytes) return OOMB_ERR_WORKSPACE;  // pool geometry beyond the static maximum
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return OOMB_ERR_CUDA;
  return oomb_page_select(pool, q, q_start, n_q, top_k, n_sink, sel, sel_count, max_sel, scratch,
                          kNoAllocSelectBytes, stream);
}
