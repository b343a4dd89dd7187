// Paged KV append with fused page summary and gradient-page zeroing.
//
// "Out of the Memory Barrier" (gist.science explainer, 2.B "Paged KV Cache and
// Gradient Management", and the lay summary's "Trick A"): a chunk's K/V go onto
// the next free fixed-size pages through the page table, without copying earlier
// pages; the KV gradients live in pages that share the same table.  The page
// summary is the representative vector of 2.D, fixed as the mean key per page.
//
// One thread block per (new page, KV head): it loads the page's K and V rows with
// several 16-byte loads in flight per thread, zeroes both gradient pages while those
// loads are in flight, sums the K rows for the summary from the same registers (K is
// read once) and writes both pages.  (Splitting a page over more blocks, by rows with
// a cluster reduction of the summary or by columns, measured slower on GB300: a
// chunk's append moves 34-67 MB, and its time is the loads' latency plus the stores'
// drain, not the number of blocks.)  HBM traffic per token and KV head: read K,V
// (2 d esize), write K,V (2 d esize), zero dK,dV (2 d 4 bytes); plus one fp32 summary
// row per page and head.
#include "oomb_internal.h"

namespace oomb {
namespace {

constexpr int kAppendThreads = 256;
constexpr int kMaxNewPerLaunch = 1024;
constexpr int kRowsInFlight = 8;  // K and V rows loaded per thread before any store

struct NewPages {
  int32_t phys[kMaxNewPerLaunch];
};

// Optional second destination of the new pages (offload mode): the staging slots of
// the chunk's own pages, which are the last n_own entries of each KV head's selection.
struct StageTarget {
  void* k;                   // staging buffers [2, Hkv, stride, P, d], or nullptr
  void* v;
  const int32_t* sel_count;  // [Hkv]
  int stage_h0, stride, max_sel, n_own, first_own;  // first_own: own page index of new page 0
  int skip_pool;  // 1: write the staging slots only; the host pool blocks are written later
};

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__global__ void __launch_bounds__(kAppendThreads)
    kv_append_kernel(Geometry g, T* __restrict__ k_pool, T* __restrict__ v_pool, float* __restrict__ dk_pool,
                     float* __restrict__ dv_pool, float* __restrict__ summary, int32_t* __restrict__ table,
                     const T* __restrict__ k, const T* __restrict__ v, int64_t first_token, int64_t end_token,
                     int first_new_logical, const __grid_constant__ NewPages np, int n_new, uint8_t* grad_state,
                     StageTarget stg, uint32_t* err) {
  const int i = blockIdx.x, h = blockIdx.y;
  const int P = g.P, d = g.d, Hkv = g.Hkv;
  const int phys = np.phys[i];
  if (phys < 0 || phys >= g.num_phys) {
    if (threadIdx.x == 0) atomicOr(err, OOMB_DEVERR_PAGE);
    return;
  }
  const int64_t logical = (int64_t)first_new_logical + i;
  if (h == 0 && threadIdx.x == 0) table[logical] = phys;
  const int64_t t0 = logical * P;
  const int m = (int)(end_token - t0 < P ? end_token - t0 : P);  // tokens present in this page

  constexpr int VEC = 16 / sizeof(T);
  const int nvec = d / VEC;                 // 16-byte vectors per row
  const int n_rg = kAppendThreads / nvec;   // rows per pass of the block
  const int c = threadIdx.x % nvec, rg = threadIdx.x / nvec;
  const size_t blk = ((size_t)phys * Hkv + h) * (size_t)P * d;
  const int64_t tok0 = t0 - first_token;    // row 0 of the page in the chunk's K/V
  // the page's staging slot: own page j of the chunk is entry count - n_own + j
  T* sk = nullptr;
  T* sv = nullptr;
  if (stg.k) {
    const int count = stg.sel_count[h];
    const int s = count - stg.n_own + stg.first_own + i;
    if (count < stg.n_own || count > stg.max_sel || s < 0 || s >= count) {
      if (threadIdx.x == 0) atomicOr(err, OOMB_DEVERR_SEL);
    } else {
      const size_t sblk = ((size_t)(stg.stage_h0 + h) * stg.stride + s) * (size_t)P * d;
      sk = reinterpret_cast<T*>(stg.k) + sblk;
      sv = reinterpret_cast<T*>(stg.v) + sblk;
    }
  }
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  if (grad_state) {
    // gradient pools in host memory: the block counts as zero until its first write-back
    if (threadIdx.x == 0) grad_state[(size_t)phys * Hkv + h] = 0;
  }
  // zero both gradient pages (streaming stores: they are next read by a later backward);
  // a thread does its share once, right after its first loads are issued
  bool zeroed = grad_state != nullptr;
  auto zero_grads = [&]() {
    const int nvec4 = P * d / 4;
    float4* gk = reinterpret_cast<float4*>(dk_pool + blk);
    float4* gv = reinterpret_cast<float4*>(dv_pool + blk);
    for (int idx = threadIdx.x; idx < nvec4; idx += kAppendThreads) {
      __stcs(gk + idx, make_float4(0.f, 0.f, 0.f, 0.f));
      __stcs(gv + idx, make_float4(0.f, 0.f, 0.f, 0.f));
    }
    zeroed = true;
  };
  if (rg < n_rg) {
    for (int rb = rg; rb < P; rb += n_rg * kRowsInFlight) {
      uint4 kr[kRowsInFlight], vr[kRowsInFlight];
#pragma unroll
      for (int u = 0; u < kRowsInFlight; ++u) {
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
      for (int u = 0; u < kRowsInFlight; ++u) {
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
          for (int e = 0; e < VEC; ++e) acc[e] += to_f<T>(x[e]);  // rows in ascending order per thread
        }
      }
    }
  }
  if (!zeroed) zero_grads();  // threads that had no row to load
  // mean key over the m tokens present: fixed-order reduction, deterministic
  __shared__ float part[kAppendThreads * VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) part[threadIdx.x * VEC + e] = acc[e];
  __syncthreads();
  for (int col = threadIdx.x; col < d; col += kAppendThreads) {
    const int cc = col / VEC, e = col % VEC;
    float s = 0.f;
    for (int r = 0; r < n_rg; ++r) s += part[(r * nvec + cc) * VEC + e];
    summary[((size_t)phys * Hkv + h) * d + col] = s / (float)m;
  }
}

}  // namespace

cudaError_t launch_kv_append(const Geometry& g, void* k_pool, void* v_pool, float* dk_pool, float* dv_pool,
                             float* summary, int32_t* table, const void* k, const void* v, int64_t first_token,
                             int n_tokens, int64_t total_tokens, const int32_t* new_phys, int n_new,
                             int first_new_logical, uint8_t* grad_state, const StageArgs* stage, uint32_t* err,
                             cudaStream_t st) {
  (void)n_tokens;
  for (int base = 0; base < n_new; base += kMaxNewPerLaunch) {
    const int cnt = n_new - base < kMaxNewPerLaunch ? n_new - base : kMaxNewPerLaunch;
    NewPages np;
    for (int i = 0; i < cnt; ++i) np.phys[i] = new_phys[base + i];
    StageTarget stg = {};
    if (stage) {
      stg.k = stage->k;
      stg.v = stage->v;
      stg.sel_count = stage->sel_count;
      stg.stage_h0 = stage->stage_h0;
      stg.stride = stage->stride;
      stg.max_sel = stage->max_sel;
      stg.n_own = n_new;
      stg.first_own = base;
      stg.skip_pool = stage->skip_pool;
    }
    dim3 grid(cnt, g.Hkv);
    if (g.dtype == OOMB_FP32) {
      kv_append_kernel<float><<<grid, kAppendThreads, 0, st>>>(
          g, (float*)k_pool, (float*)v_pool, dk_pool, dv_pool, summary, table, (const float*)k, (const float*)v,
          first_token, total_tokens, first_new_logical + base, np, cnt, grad_state, stg, err);
    } else {
      kv_append_kernel<__nv_bfloat16><<<grid, kAppendThreads, 0, st>>>(
          g, (__nv_bfloat16*)k_pool, (__nv_bfloat16*)v_pool, dk_pool, dv_pool, summary, table,
          (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, first_token, total_tokens, first_new_logical + base,
          np, cnt, grad_state, stg, err);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
  }
  return cudaSuccess;
}

}  // namespace oomb
