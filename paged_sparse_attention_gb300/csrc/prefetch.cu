// Offload mode: gather the selected (page, KV head) K/V blocks from the pinned
// host pools into an HBM staging buffer.
//
// "Out of the Memory Barrier" (gist.science explainer, 2.C "Asynchronous KV Cache
// CPU Offloading"): the KV cache lives in CPU memory and moves to the GPU in the
// background, hidden behind computation; with page-level sparse attention only the
// selected pages move (2.D).  On a Grace-Blackwell node the host pools are reached
// over NVLink-C2C; this kernel reads them directly (zero-copy) with 16-byte loads
// and writes the staging slots, so a whole chunk's gather is one launch on the side
// stream instead of one copy call per 32 KB block.
#include "oomb_internal.h"

namespace oomb {
namespace {

constexpr int kPrefetchThreads = 512;

// block (s, h, which): slot (stage_h0 + h) * stride + s  <-  pool block (phi(sel[h][s]), h)
__global__ void __launch_bounds__(kPrefetchThreads)
    gather_pages(Geometry g, const uint8_t* __restrict__ k_pool, const uint8_t* __restrict__ v_pool,
                 const int32_t* __restrict__ table, const int32_t* __restrict__ sel,
                 const int32_t* __restrict__ sel_count, int max_sel, uint8_t* __restrict__ stage_k,
                 uint8_t* __restrict__ stage_v, int stage_h0, int stride, uint32_t* err) {
  const int s = blockIdx.x, h = blockIdx.y;
  if (s >= sel_count[h]) return;
  const int p = sel[(size_t)h * max_sel + s];
  if (p < 0 || p >= g.max_logical) {
    if (threadIdx.x == 0) atomicOr(err, OOMB_DEVERR_SEL);
    return;
  }
  const int phys = table[p];
  if (phys < 0 || phys >= g.num_phys) {
    if (threadIdx.x == 0) atomicOr(err, OOMB_DEVERR_PAGE);
    return;
  }
  const size_t bytes = (size_t)g.P * g.d * dtype_size(g.dtype);
  const uint8_t* src = (blockIdx.z == 0 ? k_pool : v_pool) + ((size_t)phys * g.Hkv + h) * bytes;
  uint8_t* dst = (blockIdx.z == 0 ? stage_k : stage_v) + ((size_t)(stage_h0 + h) * stride + s) * bytes;
  const int n16 = (int)(bytes / 16);
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  int i = threadIdx.x;
  for (; i + 3 * kPrefetchThreads < n16; i += 4 * kPrefetchThreads) {
    uint4 a0 = s4[i], a1 = s4[i + kPrefetchThreads], a2 = s4[i + 2 * kPrefetchThreads],
          a3 = s4[i + 3 * kPrefetchThreads];
    d4[i] = a0;
    d4[i + kPrefetchThreads] = a1;
    d4[i + 2 * kPrefetchThreads] = a2;
    d4[i + 3 * kPrefetchThreads] = a3;
  }
  for (; i < n16; i += kPrefetchThreads) d4[i] = s4[i];
}

}  // namespace

cudaError_t launch_prefetch(const Geometry& g, const void* k_pool, const void* v_pool, const int32_t* table,
                            const int32_t* sel, const int32_t* sel_count, int max_sel, void* stage_k, void* stage_v,
                            int stage_h0, int stage_stride, uint32_t* err, cudaStream_t st) {
  dim3 grid(max_sel, g.Hkv, 2);
  gather_pages<<<grid, kPrefetchThreads, 0, st>>>(g, (const uint8_t*)k_pool, (const uint8_t*)v_pool, table, sel,
                                                  sel_count, max_sel, (uint8_t*)stage_k, (uint8_t*)stage_v,
                                                  stage_h0, stage_stride, err);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace oomb
