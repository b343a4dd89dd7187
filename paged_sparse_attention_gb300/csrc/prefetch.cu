// Offload mode: move the selected (page, KV head) blocks between the pinned host
// pools and the HBM staging buffers.
//
// "Out of the Memory Barrier" (gist.science explainer, 2.C "Asynchronous KV Cache
// CPU Offloading"): the KV cache and its gradients live in CPU memory and move to
// the GPU in the background, hidden behind computation; with page-level sparse
// attention only the selected pages move (2.D).  On a Grace-Blackwell node the host
// pools are reached over NVLink-C2C; these kernels read and write them directly
// (zero-copy, 16-byte accesses), so a chunk's transfer is one launch on the side
// stream instead of one copy call per block.
//
// Each launch is a small persistent grid (8 or 16 thread blocks of 256 threads,
// at most 32 registers each) that walks the chunk's blocks.  An attention CTA holds
// nearly all of its SM's shared memory, so a transfer block takes an SM of its own
// while it runs: issued on a high-priority stream (otherwise the block scheduler
// places it only after a long attention grid's last pending block) it starts on the
// next SM an attention CTA leaves, and a transfer takes only a few SMs from the
// attention kernels.
//
//   gather_pages  K/V: slot (buf, h, s) <- pool block (phi(sel[h][s]), h), or the
//                 reverse (to_host: a chunk's own pages appended into their slots only)
//   grad_copy     fp32 dK/dV, mode
//                   from host: slot (buf, h, s) <- pool block, for pages not in prev;
//                              a block that no write-back has reached since its page
//                              was appended (grad_state 0) is zero-filled instead
//                   carry:     slot (buf, h, s) <- slot (1 - buf, h, j) where
//                              prev[h][j] == sel[h][s] (the previous chunk's staged
//                              block, which holds that chunk's contribution)
//                   to host:   pool block <- slot (buf, h, s), every selected page;
//                              grad_state of the block becomes 1
#include "oomb_internal.h"

namespace oomb {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kInFlight = 4;  // 16-byte loads per thread before the stores
// Thread blocks of one transfer launch.  Measured on GB300 at 4M tokens (K/V and
// gradients offloaded, side stream at high priority): gradient copies with 16 blocks
// move ~59 GB/s beside the attention kernels with 74 ms of a 5.97 s step exposed; 32
// and 64 move more but slow the attention kernels on their SMs by more than they hide
// (step 5.99 / 6.27 s).  K/V gathers need less (a forward-sweep chunk's history pages
// in the ~2.3 ms of its forward): with 8 blocks instead of 16 the forward beside them
// keeps ~1065 instead of ~1040 TFLOP/s at the same exposed time.
constexpr int kCopyCtas = 16;
constexpr int kGatherCtas = 8;

// Copy `n16` 16-byte words from src to dst, kInFlight loads per thread in flight.
__device__ __forceinline__ void copy_block(uint4* __restrict__ dst, const uint4* __restrict__ src, int n16) {
  int i = threadIdx.x;
  for (; i + (kInFlight - 1) * kCopyThreads < n16; i += kInFlight * kCopyThreads) {
    uint4 v[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) v[u] = src[i + u * kCopyThreads];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) dst[i + u * kCopyThreads] = v[u];
  }
  for (; i < n16; i += kCopyThreads) dst[i] = src[i];
}

__device__ __forceinline__ void zero_block(uint4* __restrict__ dst, int n16) {
  for (int i = threadIdx.x; i < n16; i += kCopyThreads) dst[i] = make_uint4(0, 0, 0, 0);
}

// Checked entry count of a selection row (flagged and 0 when outside [0, max_sel]).
__device__ __forceinline__ int checked_count(const int32_t* count, int h, int max_sel, uint32_t* err) {
  const int c = count[h];
  if (c < 0 || c > max_sel) {
    if (threadIdx.x == 0) atomicOr(err, OOMB_DEVERR_SEL);
    return 0;
  }
  return c;
}

// Physical page of selected page s of KV head h, or -1 (flagged) when invalid.
__device__ __forceinline__ int selected_phys(const Geometry& g, const int32_t* table, const int32_t* sel, int max_sel,
                                             int h, int s, int* logical, uint32_t* err) {
  const int p = sel[(size_t)h * max_sel + s];
  *logical = p;
  if (p < 0 || p >= g.max_logical) {
    if (threadIdx.x == 0) atomicOr(err, OOMB_DEVERR_SEL);
    return -1;
  }
  const int phys = table[p];
  if (phys < 0 || phys >= g.num_phys) {
    if (threadIdx.x == 0) atomicOr(err, OOMB_DEVERR_PAGE);
    return -1;
  }
  return phys;
}

// item = (s, h, which) in s-major order: slot (stage_h0 + h) * stride + s  <-  pool block
// (phi(sel[h][s]), h), for every item of the chunk's selection whose logical page is in
// [first_page, end_page).
__global__ void __launch_bounds__(kCopyThreads, 8)
    gather_pages(Geometry g, uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
                 const int32_t* __restrict__ table, const int32_t* __restrict__ sel,
                 const int32_t* __restrict__ sel_count, int max_sel, uint8_t* __restrict__ stage_k,
                 uint8_t* __restrict__ stage_v, int stage_h0, int stride, int first_page, int end_page, int to_host,
                 uint32_t* err) {
  const size_t bytes = (size_t)g.P * g.d * dtype_size(g.dtype);
  const int n_items = max_sel * g.Hkv * 2;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int which = it & 1, h = (it >> 1) % g.Hkv, s = (it >> 1) / g.Hkv;
    if (s >= checked_count(sel_count, h, max_sel, err)) continue;
    const int pg = sel[(size_t)h * max_sel + s];
    if (pg >= 0 && (pg < first_page || pg >= end_page)) continue;  // outside the requested pages
    int p;
    const int phys = selected_phys(g, table, sel, max_sel, h, s, &p, err);
    if (phys < 0) continue;
    uint8_t* pool = (which == 0 ? k_pool : v_pool) + ((size_t)phys * g.Hkv + h) * bytes;
    uint8_t* slot = (which == 0 ? stage_k : stage_v) + ((size_t)(stage_h0 + h) * stride + s) * bytes;
    if (to_host) copy_block(reinterpret_cast<uint4*>(pool), reinterpret_cast<const uint4*>(slot), (int)(bytes / 16));
    else copy_block(reinterpret_cast<uint4*>(slot), reinterpret_cast<const uint4*>(pool), (int)(bytes / 16));
  }
}

// Index of page p in the ascending row prev[0..n), or -1.
__device__ __forceinline__ int find_sorted(const int32_t* prev, int n, int p) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int v = prev[mid];
    if (v == p) return mid;
    if (v < p) lo = mid + 1;
    else hi = mid;
  }
  return -1;
}

// item = (s, h, which = dK or dV) of the fp32 gradient pools; see the file comment.
__global__ void __launch_bounds__(kCopyThreads, 8)
    grad_copy(Geometry g, int mode, float* __restrict__ dk_pool, float* __restrict__ dv_pool,
              uint8_t* __restrict__ grad_state, const int32_t* __restrict__ table, const int32_t* __restrict__ sel,
              const int32_t* __restrict__ sel_count, const int32_t* __restrict__ prev_sel,
              const int32_t* __restrict__ prev_count, int max_sel, float* __restrict__ stage_dk,
              float* __restrict__ stage_dv, int buf, int stride, uint32_t* err) {
  const size_t elems = (size_t)g.P * g.d;
  const int n_items = max_sel * g.Hkv * 2;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int which = it & 1, h = (it >> 1) % g.Hkv, s = (it >> 1) / g.Hkv;
    if (s >= checked_count(sel_count, h, max_sel, err)) continue;
    int p;
    const int phys = selected_phys(g, table, sel, max_sel, h, s, &p, err);
    if (phys < 0) continue;
    int j = -1;  // slot of page p in the previous chunk's selection
    if (mode != kGradToHost && prev_sel != nullptr) {
      const int n_prev = checked_count(prev_count, h, max_sel, err);
      j = find_sorted(prev_sel + (size_t)h * max_sel, n_prev, p);
    }
    if ((mode == kGradFromHost && j >= 0) || (mode == kGradCarry && j < 0)) continue;
    float* pool = which == 0 ? dk_pool : dv_pool;
    float* stage = which == 0 ? stage_dk : stage_dv;
    float* slot = stage + ((size_t)(buf * g.Hkv + h) * stride + s) * elems;
    float* host = pool + ((size_t)phys * g.Hkv + h) * elems;
    uint8_t* state = grad_state + (size_t)phys * g.Hkv + h;
    const int n16 = (int)(elems / 4);
    if (mode == kGradFromHost) {
      if (*state) copy_block(reinterpret_cast<uint4*>(slot), reinterpret_cast<const uint4*>(host), n16);
      else zero_block(reinterpret_cast<uint4*>(slot), n16);  // nothing written back yet: zero
    } else if (mode == kGradCarry) {
      const float* src = stage + ((size_t)((1 - buf) * g.Hkv + h) * stride + j) * elems;
      copy_block(reinterpret_cast<uint4*>(slot), reinterpret_cast<const uint4*>(src), n16);
    } else {
      copy_block(reinterpret_cast<uint4*>(host), reinterpret_cast<const uint4*>(slot), n16);
      if (which == 1 && threadIdx.x == 0) *state = 1;  // the dV item follows the dK item of the block
    }
  }
}

}  // namespace

cudaError_t launch_prefetch(const Geometry& g, const void* k_pool, const void* v_pool, const int32_t* table,
                            const int32_t* sel, const int32_t* sel_count, int max_sel, void* stage_k, void* stage_v,
                            int stage_h0, int stage_stride, int first_page, int end_page, uint32_t* err,
                            cudaStream_t st, int to_host) {
  const int grid = std::min(max_sel * g.Hkv * 2, kGatherCtas);
  gather_pages<<<grid, kCopyThreads, 0, st>>>(g, (uint8_t*)const_cast<void*>(k_pool),
                                              (uint8_t*)const_cast<void*>(v_pool), table, sel, sel_count, max_sel,
                                              (uint8_t*)stage_k, (uint8_t*)stage_v, stage_h0, stage_stride,
                                              first_page, end_page, to_host, err);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_grad_copy(const Geometry& g, int mode, float* dk_pool, float* dv_pool, uint8_t* grad_state,
                             const int32_t* table, const int32_t* sel, const int32_t* sel_count,
                             const int32_t* prev_sel, const int32_t* prev_count, int max_sel, float* stage_dk,
                             float* stage_dv, int buf, int stage_stride, uint32_t* err, cudaStream_t st) {
  const int grid = std::min(max_sel * g.Hkv * 2, kCopyCtas);
  grad_copy<<<grid, kCopyThreads, 0, st>>>(g, mode, dk_pool, dv_pool, grad_state, table, sel, sel_count, prev_sel,
                                           prev_count, max_sel, stage_dk, stage_dv, buf, stage_stride, err);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace oomb
