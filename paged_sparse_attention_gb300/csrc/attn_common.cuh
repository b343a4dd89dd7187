// Device helpers shared by the attention kernels: page addressing through the
// page table (or the offload staging slots) and element conversion.
#pragma once
#include <cuda_bf16.h>
#include "oomb_internal.h"

namespace oomb {

template <typename T>
__device__ __forceinline__ float to_float(T x);
template <>
__device__ __forceinline__ float to_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_float<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Entries of KV head h's selection: sel_count[h], flagged and clamped to [0, max_sel]
// when out of range (a longer count would read past the row).
__device__ __forceinline__ int sel_count_checked(const AttnArgs& a, int h) {
  const int c = a.sel_count[h];
  if (c < 0 || c > a.max_sel) {
    atomicOr(a.err, OOMB_DEVERR_SEL);
    return c < 0 ? 0 : a.max_sel;
  }
  return c;
}

// Selected logical page s of KV head h, checked against the chunk's page range and
// against the previous entry (a selection is strictly ascending).
__device__ __forceinline__ int sel_page(const AttnArgs& a, int h, int s, int n_pages_visible, bool& ok) {
  const int32_t* row = a.sel + (size_t)h * a.max_sel;
  const int p = row[s];
  if (p < 0 || p >= n_pages_visible || (s > 0 && row[s - 1] >= p)) {
    ok = false;
    atomicOr(a.err, OOMB_DEVERR_SEL);
  }
  return p;
}

// Physical page of logical page p, checked.
__device__ __forceinline__ int phys_page(const AttnArgs& a, int p, bool& ok) {
  const int phys = a.kv.table[p];
  if (phys < 0 || phys >= a.g.num_phys) {
    ok = false;
    atomicOr(a.err, OOMB_DEVERR_PAGE);
  }
  return phys;
}

// Index of the (P x d) fp32 gradient block of selected page s (physical page phys) of
// KV head h: its slot in the gradient staging buffers, or its block in the pool.
__device__ __forceinline__ size_t grad_block(const AttnArgs& a, int h, int s, int phys) {
  if (a.grad_staged) return (size_t)(a.kv.stage_h0 + h) * a.kv.stage_stride + s;
  return (size_t)phys * a.g.Hkv + h;
}

// Index of the (P x d) K/V block holding selected page s (logical p) of KV head h.
__device__ __forceinline__ size_t kv_block(const AttnArgs& a, int h, int s, int p, bool& ok) {
  if (a.kv.staged) return (size_t)(a.kv.stage_h0 + h) * a.kv.stage_stride + s;
  const int phys = phys_page(a, p, ok);
  return (size_t)phys * a.g.Hkv + h;
}

}  // namespace oomb
