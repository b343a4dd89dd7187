// The append of one (new page, KV head) block by 256 threads: the body shared by the
// append kernel (one block per unit) and the fused selection-and-append kernel (two
// units at a time in its 512-thread blocks).
//
// "Out of the Memory Barrier" (gist.science explainer, 2.B "Paged KV Cache and
// Gradient Management", and the lay summary's "Trick A"): a chunk's K/V go onto
// the next free fixed-size pages through the page table, without copying earlier
// pages; the KV gradients live in pages that share the same table.  The page
// summary is the representative vector of 2.D, fixed as the mean key per page.
//
// The 256 threads load the page's K and V rows with several 16-byte loads in flight
// per thread, zero both gradient pages while those loads are in flight (or, with the
// gradient pools in host memory, mark the block empty), sum the K rows for the
// summary from the same registers (K is read once), write the pool pages and/or the
// staging slot, and reduce the summary in a fixed order (deterministic).
#pragma once
#include "oomb_internal.h"
#include "sm103_ptx.cuh"

namespace oomb {

constexpr int kAppendThreads = 256;
constexpr int kAppendRowsInFlight = 8;  // K and V rows loaded per thread before any store

// Optional second destination of the new pages (offload mode): the staging slots of
// the chunk's own pages, which are the last n_own entries of each KV head's selection.
struct StageTarget {
  void* k;                   // staging buffers [2, Hkv, stride, P, d], or nullptr
  void* v;
  const int32_t* sel_count;  // [Hkv] (read when slot0 < 0)
  int stage_h0, stride, max_sel, n_own, first_own;  // first_own: own page index of new page 0
  int skip_pool;             // 1: write the staging slots only; the host pool blocks are written later
  int slot0;                 // >= 0: own page 0's slot, the same for every KV head (known on the host)
};

// One chunk's append, as the device sees it.
struct AppendJob {
  Geometry g;
  void* k_pool;
  void* v_pool;
  float* dk_pool;
  float* dv_pool;
  float* summary;
  int32_t* table;
  const void* k;  // [n_tokens, Hkv, d], tokens from first_token
  const void* v;
  int64_t first_token, end_token;
  int first_new_logical;
  uint8_t* grad_state;  // gradient pools in host memory: state bytes instead of zeroing
  StageTarget stg;
  uint32_t* err;
};

// Host: the job of one append (stage: optional staging target, slot0 from it).
AppendJob append_job(const Geometry& g, void* k_pool, void* v_pool, float* dk_pool, float* dv_pool, float* summary,
                     int32_t* table, const void* k, const void* v, int64_t first_token, int64_t total_tokens,
                     int n_new, int first_new_logical, uint8_t* grad_state, const StageArgs* stage, uint32_t* err);

template <typename T>
__device__ __forceinline__ float append_to_f(T x);
template <>
__device__ __forceinline__ float append_to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float append_to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// New page i (physical page `phys`) for KV head h.  tid in [0, 256); `part` is
// 256 * (16 / sizeof(T)) floats of shared memory owned by these 256 threads; they
// synchronise on named barrier `bar_id` (the whole block when it has 256 threads).
// ROWS: K and V rows in flight per thread; every thread still adds its rows in
// ascending order, so the summary's bits do not depend on it.
template <typename T, int ROWS = kAppendRowsInFlight>
__device__ void append_unit(const AppendJob& a, int phys, int i, int h, int tid, float* part, int bar_id) {
  const Geometry& g = a.g;
  const int P = g.P, d = g.d, Hkv = g.Hkv;
  if (phys < 0 || phys >= g.num_phys) {
    if (tid == 0) atomicOr(a.err, OOMB_DEVERR_PAGE);
    return;
  }
  const int64_t logical = (int64_t)a.first_new_logical + i;
  if (h == 0 && tid == 0) a.table[logical] = phys;
  const int64_t t0 = logical * P;
  const int m = (int)(a.end_token - t0 < P ? a.end_token - t0 : P);  // tokens present in this page

  constexpr int VEC = 16 / sizeof(T);
  const int nvec = d / VEC;                 // 16-byte vectors per row
  const int n_rg = kAppendThreads / nvec;   // rows per pass
  const int c = tid % nvec, rg = tid / nvec;
  const size_t blk = ((size_t)phys * Hkv + h) * (size_t)P * d;
  const int64_t tok0 = t0 - a.first_token;  // row 0 of the page in the chunk's K/V
  T* k_pool = reinterpret_cast<T*>(a.k_pool);
  T* v_pool = reinterpret_cast<T*>(a.v_pool);
  const T* k = reinterpret_cast<const T*>(a.k);
  const T* v = reinterpret_cast<const T*>(a.v);
  // the page's staging slot: own page j of the chunk is entry count - n_own + j
  T* sk = nullptr;
  T* sv = nullptr;
  const StageTarget& stg = a.stg;
  if (stg.k) {
    int s;
    bool ok;
    if (stg.slot0 >= 0) {
      s = stg.slot0 + stg.first_own + i;
      ok = s < stg.max_sel;
    } else {
      const int count = stg.sel_count[h];
      s = count - stg.n_own + stg.first_own + i;
      ok = !(count < stg.n_own || count > stg.max_sel || s < 0 || s >= count);
    }
    if (!ok) {
      if (tid == 0) atomicOr(a.err, OOMB_DEVERR_SEL);
    } else {
      const size_t sblk = ((size_t)(stg.stage_h0 + h) * stg.stride + s) * (size_t)P * d;
      sk = reinterpret_cast<T*>(stg.k) + sblk;
      sv = reinterpret_cast<T*>(stg.v) + sblk;
    }
  }
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  if (a.grad_state) {
    // gradient pools in host memory: the block counts as zero until its first write-back
    if (tid == 0) a.grad_state[(size_t)phys * Hkv + h] = 0;
  }
  // zero both gradient pages (streaming stores: they are next read by a later backward);
  // a thread does its share once, right after its first loads are issued
  bool zeroed = a.grad_state != nullptr;
  auto zero_grads = [&]() {
    const int nvec4 = P * d / 4;
    float4* gk = reinterpret_cast<float4*>(a.dk_pool + blk);
    float4* gv = reinterpret_cast<float4*>(a.dv_pool + blk);
    for (int idx = tid; idx < nvec4; idx += kAppendThreads) {
      __stcs(gk + idx, make_float4(0.f, 0.f, 0.f, 0.f));
      __stcs(gv + idx, make_float4(0.f, 0.f, 0.f, 0.f));
    }
    zeroed = true;
  };
  if (rg < n_rg) {
    for (int rb = rg; rb < P; rb += n_rg * ROWS) {
      uint4 kr[ROWS], vr[ROWS];
#pragma unroll
      for (int u = 0; u < ROWS; ++u) {
        const int r = rb + u * n_rg;
        kr[u] = vr[u] = make_uint4(0, 0, 0, 0);  // absent tail rows of a partial page are zero
        if (r < m) {
          const size_t off = ((size_t)(tok0 + r) * Hkv + h) * d + (size_t)c * VEC;
          kr[u] = __ldcs(reinterpret_cast<const uint4*>(k + off));
          vr[u] = __ldcs(reinterpret_cast<const uint4*>(v + off));
        }
      }
      if (!zeroed) zero_grads();  // independent of the loads in flight
#pragma unroll
      for (int u = 0; u < ROWS; ++u) {
        const int r = rb + u * n_rg;
        if (r < P) {
          if (!stg.skip_pool) {
            const size_t off = blk + (size_t)r * d + (size_t)c * VEC;
            *reinterpret_cast<uint4*>(k_pool + off) = kr[u];
            *reinterpret_cast<uint4*>(v_pool + off) = vr[u];
          }
          if (sk) {
            const size_t so = (size_t)r * d + (size_t)c * VEC;
            *reinterpret_cast<uint4*>(sk + so) = kr[u];
            *reinterpret_cast<uint4*>(sv + so) = vr[u];
          }
          const T* x = reinterpret_cast<const T*>(&kr[u]);
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[e] += append_to_f<T>(x[e]);  // rows in ascending order per thread
        }
      }
    }
  }
  if (!zeroed) zero_grads();  // threads that had no row to load
  // mean key over the m tokens present: fixed-order reduction, deterministic
#pragma unroll
  for (int e = 0; e < VEC; ++e) part[tid * VEC + e] = acc[e];
  named_bar_sync(bar_id, kAppendThreads);
  for (int col = tid; col < d; col += kAppendThreads) {
    const int cc = col / VEC, e = col % VEC;
    float s = 0.f;
    for (int r = 0; r < n_rg; ++r) s += part[(r * nvec + cc) * VEC + e];
    a.summary[((size_t)phys * Hkv + h) * d + col] = s / (float)m;
  }
  named_bar_sync(bar_id, kAppendThreads);  // `part` is reused by the next unit
}

}  // namespace oomb
