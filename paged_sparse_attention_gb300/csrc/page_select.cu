// Page-level top-K selection for one query chunk.
//
// "Out of the Memory Barrier" (gist.science explainer, 2.D "Page-Level Sparse
// Attention"): only the top-K most relevant key pages are retrieved, ranked by a
// representative (averaged) vector.  The scoring rule is the mean key of each
// page against the mean query of the chunk's KV group; ties go to the lower
// logical page.  The sink pages and the chunk's own pages are always kept.
//
// One cooperative kernel, one CTA per SM, four phases separated by grid barriers
// whose waits are bounded (a barrier that runs out sets OOMB_DEVERR_TIMEOUT and
// the CTA returns):
//   1. query sum     every CTA sums a contiguous slice of the chunk's query rows
//                    per KV group (Q is read exactly once, 16-byte loads, several
//                    rows in flight per thread) -> partial[cta][Hkv*d]
//   2. mean query    fixed-order sum of the partials -> qbar[Hkv*d]
//   3. page scores   qbar[h] . summary[phi(p)][h] for every candidate page and KV
//                    head, written as order-preserving 32-bit keys
//   4. top-k         one CTA per KV head: 8-bit radix select over the keys staged
//                    in shared memory (warp-aggregated histograms, parallel bin
//                    search), ties resolved by page index, ordered compaction.
// Every sum runs in a fixed order, so the selection is deterministic.
// The barrier counters live in the pool's control words (one call at a time per pool).
#include "oomb_internal.h"

namespace oomb {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxBlocks = 256;       // upper bound of the grid (one CTA per SM)
constexpr int kRowUnroll = 8;         // query rows in flight per thread in phase 1
constexpr int kMaxSmemKeys = 40960;   // candidates per KV head staged in shared memory
constexpr long long kSpinLimit = 1ll << 31;

// control words (after the error word): barrier counters and release flags
constexpr int kCtrlCount = 4;
constexpr int kCtrlFlag = 8;

struct SelParams {
  Geometry g;
  const void* q;
  int n_q;
  int rows_per_block;
  const float* summary;
  const int32_t* table;
  int n_sinks, cand0, n_cand, own0, n_own, top_k, max_sel;
  int lanes_per_item;  // phase 3: lanes that share one (page, head) dot product
  float inv_count;
  float* partial;      // [gridDim.x][Hkv*d]
  float* qbar;         // [Hkv*d]
  uint32_t* keys;      // [Hkv][key_stride]
  int key_stride;
  int keys_in_smem;
  int need_scores;
  int32_t* sel;
  int32_t* sel_count;
  uint32_t* err;
  uint32_t* ctrl;
  uint32_t epoch;
};

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f + 0.0f);  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid barrier i.  Every CTA arrives; the last one to arrive resets the counter and
// publishes this call's epoch in the flag.  With wait == false the CTA only arrives.
// Returns false when the wait ran out (~1 s), after setting the timeout bit.
__device__ bool grid_sync(const SelParams& p, int i, bool wait) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t* cnt = p.ctrl + kCtrlCount + i;
    uint32_t* flag = p.ctrl + kCtrlFlag + i;
    __threadfence();
    const uint32_t arrived = atomicAdd(cnt, 1u) + 1u;
    int ok = 1;
    if (arrived == gridDim.x) {
      atomicExch(cnt, 0u);
      __threadfence();
      st_release(flag, p.epoch);
    } else if (wait) {
      const long long t0 = clock64();
      while (ld_acquire(flag) != p.epoch) {
        if (clock64() - t0 > kSpinLimit) {
          atomicOr(p.err, OOMB_DEVERR_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Phase 1: this CTA's rows of the chunk, summed per KV group -> partial[blockIdx.x].
template <typename T>
__device__ void query_sum(const SelParams& p, float* sh) {
  constexpr int VEC = 16 / sizeof(T);
  const Geometry& g = p.g;
  const int tid = threadIdx.x;
  const int row_vecs = g.Hq * g.d / VEC;
  const bool narrow = row_vecs <= kThreads;
  const int spp = narrow ? kThreads / row_vecs : 1;  // rows per pass of the CTA
  const int n_slots = narrow ? 1 : (row_vecs + kThreads - 1) / kThreads;
  const int phase = narrow ? tid / row_vecs : 0;
  const int r0 = blockIdx.x * p.rows_per_block;
  const int r1 = min(p.n_q, r0 + p.rows_per_block);
  const uint4* q4 = reinterpret_cast<const uint4*>(p.q);
  const int HqD = g.Hq * g.d;
  for (int s = 0; s < n_slots; ++s) {
    const int col = narrow ? tid % row_vecs : tid + s * kThreads;
    const bool active = narrow ? (tid < spp * row_vecs) : (col < row_vecs);
    if (!active) continue;
    float acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
    for (int rb = r0 + phase; rb < r1; rb += spp * kRowUnroll) {
      uint4 buf[kRowUnroll];
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const int r = rb + u * spp;
        buf[u] = r < r1 ? __ldg(q4 + (size_t)r * row_vecs + col) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kRowUnroll; ++u) {
        const T* x = reinterpret_cast<const T*>(&buf[u]);
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] += to_f<T>(x[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) sh[phase * HqD + col * VEC + e] = acc[e];
  }
  __syncthreads();
  const int HD = g.Hkv * g.d;
  for (int idx = tid; idx < HD; idx += kThreads) {
    const int h = idx / g.d, c = idx % g.d;
    float s = 0.f;
    for (int ph = 0; ph < spp; ++ph)
      for (int gg = 0; gg < g.G; ++gg) s += sh[ph * HqD + (h * g.G + gg) * g.d + c];
    p.partial[(size_t)blockIdx.x * HD + idx] = s;
  }
}

// Phase 2: qbar = (sum of the partials) / (rows x group size); one warp per output.
__device__ void mean_query(const SelParams& p) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int HD = p.g.Hkv * p.g.d;
  const int nb = gridDim.x;
  for (int o = blockIdx.x * kWarps + warp; o < HD; o += nb * kWarps) {
    float s = 0.f;
    for (int b = lane; b < nb; b += 32) s += __ldcg(p.partial + (size_t)b * HD + o);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) p.qbar[o] = s * p.inv_count;
  }
}

// Phase 3: one key per (candidate page, KV head); lanes_per_item lanes share a dot product.
__device__ void page_scores(const SelParams& p, float* sh) {
  const Geometry& g = p.g;
  const int tid = threadIdx.x, lane = tid % 32;
  const int qs = g.d + 4;  // padded qbar rows in shared memory
  for (int i = tid; i < g.Hkv * g.d; i += kThreads) sh[(i / g.d) * qs + i % g.d] = __ldcg(p.qbar + i);
  __syncthreads();
  const int L = p.lanes_per_item;
  const int nv = g.d / 4 / L;  // float4 per lane
  const int sub = lane % L;
  const int per_warp = 32 / L;
  const int n_items = p.n_cand * g.Hkv;
  const int n_wi = (n_items + per_warp - 1) / per_warp;
  const int total_warps = gridDim.x * kWarps;
  for (int wi = blockIdx.x * kWarps + tid / 32; wi < n_wi; wi += total_warps) {
    const int it = wi * per_warp + lane / L;
    const bool valid = it < n_items;
    const int i = valid ? it / g.Hkv : 0, h = valid ? it % g.Hkv : 0;
    float s = 0.f;
    if (valid) {
      const int phys = __ldg(p.table + p.cand0 + i);
      if (phys < 0 || phys >= g.num_phys) {
        if (sub == 0) atomicOr(p.err, OOMB_DEVERR_PAGE);
      } else {
        const float4* kb = reinterpret_cast<const float4*>(p.summary + ((size_t)phys * g.Hkv + h) * g.d) + sub * nv;
        const float* qb = sh + h * qs + sub * nv * 4;
        for (int v0 = 0; v0 < nv; v0 += 8) {
          float4 buf[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (v0 + u < nv) buf[u] = __ldg(kb + v0 + u);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (v0 + u < nv) {
              const float4 a = *reinterpret_cast<const float4*>(qb + (v0 + u) * 4);
              s += a.x * buf[u].x + a.y * buf[u].y + a.z * buf[u].z + a.w * buf[u].w;
            }
        }
      }
    }
    for (int off = L >> 1; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (valid && sub == 0) p.keys[(size_t)h * p.key_stride + i] = order_key(s);
  }
}

// Block-wide exclusive scan of one int per thread.  Returns the total.
__device__ int block_exclusive_scan(int v, int* out, int* sh_warp) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? sh_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh_warp[lane] = w;  // inclusive prefix over warps
  }
  __syncthreads();
  *out = (warp > 0 ? sh_warp[warp - 1] : 0) + x - v;
  const int total = sh_warp[kWarps - 1];
  __syncthreads();
  return total;
}

__device__ __forceinline__ uint32_t key_at(const uint32_t* keys, bool smem, int i) {
  return smem ? keys[i] : __ldcg(keys + i);
}

// Phase 4 for KV head h: sinks, the kept candidates in ascending page order, own pages.
__device__ void top_k_head(const SelParams& p, int h, uint32_t* sh_keys) {
  __shared__ int hist[256];
  __shared__ int sh_warp[32];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_need;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int n_cand = p.n_cand, top_k = p.top_k;
  int32_t* out = p.sel + (size_t)h * p.max_sel;
  const bool take_all = (top_k < 0) || (n_cand <= top_k);
  const bool scored = !take_all && top_k > 0;
  const bool smem = scored && p.keys_in_smem;
  const uint32_t* keys = p.keys + (size_t)h * p.key_stride;
  if (smem) {
    for (int i = tid; i < n_cand; i += kThreads) sh_keys[i] = __ldcg(keys + i);
    keys = sh_keys;
  }
  __syncthreads();

  uint32_t T = 0;
  int need_eq = 0;  // keys equal to T that are kept (lowest pages first)
  if (scored) {
    uint32_t prefix = 0, mask = 0;
    int k_rem = top_k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      for (int base = warp * 32; base < n_cand; base += kThreads) {
        const int i = base + lane;
        const uint32_t u = i < n_cand ? key_at(keys, smem, i) : 0u;
        const bool want = i < n_cand && (u & mask) == prefix;
        const uint32_t m = __ballot_sync(0xffffffffu, want);
        if (want) {
          const uint32_t bin = (u >> shift) & 0xFFu;
          const uint32_t peers = __match_any_sync(m, bin);
          if (lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
        }
      }
      __syncthreads();
      if (warp == 0) {
        int c8[8], t = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          c8[e] = hist[lane * 8 + e];
          t += c8[e];
        }
        int suf = t;  // sum over lanes >= this lane
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_down_sync(0xffffffffu, suf, off);
          if (lane + off < 32) suf += y;
        }
        const uint32_t bal = __ballot_sync(0xffffffffu, suf >= k_rem);
        const int top_lane = 31 - __clz((int)bal);
        if (lane == top_lane) {
          int cum = suf - t;  // keys in higher bins
          int b = 7;
          for (; b > 0; --b) {
            if (cum + c8[b] >= k_rem) break;
            cum += c8[b];
          }
          sh_prefix = prefix | ((uint32_t)(lane * 8 + b) << shift);
          sh_need = k_rem - cum;
        }
      }
      __syncthreads();
      prefix = sh_prefix;
      k_rem = sh_need;
      mask |= 0xFFu << shift;
      __syncthreads();
    }
    T = prefix;
    need_eq = k_rem;
  }
  // ordered compaction; thread t owns a contiguous segment of the candidates
  const int seg = (n_cand + kThreads - 1) / kThreads;
  const int i0 = min(n_cand, tid * seg), i1 = min(n_cand, i0 + seg);
  int n_eq = 0;
  if (scored)
    for (int i = i0; i < i1; ++i) n_eq += (key_at(keys, smem, i) == T);
  int eq_before;
  block_exclusive_scan(n_eq, &eq_before, sh_warp);
  int n_keep = 0;
  if (take_all) {
    n_keep = i1 - i0;
  } else if (scored) {
    int eq_seen = eq_before;
    for (int i = i0; i < i1; ++i) {
      const uint32_t u = key_at(keys, smem, i);
      if (u > T || (u == T && eq_seen++ < need_eq)) ++n_keep;
    }
  }
  int keep_before;
  const int kept = block_exclusive_scan(n_keep, &keep_before, sh_warp);
  if (n_keep > 0) {
    int o = p.n_sinks + keep_before;
    int eq_seen = eq_before;
    for (int i = i0; i < i1; ++i) {
      bool take = true;
      if (!take_all) {
        const uint32_t u = key_at(keys, smem, i);
        take = u > T || (u == T && eq_seen++ < need_eq);
      }
      if (take) out[o++] = p.cand0 + i;
    }
  }
  for (int s = tid; s < p.n_sinks; s += kThreads) out[s] = s;
  for (int s = tid; s < p.n_own; s += kThreads) out[p.n_sinks + kept + s] = p.own0 + s;
  if (tid == 0) p.sel_count[h] = p.n_sinks + kept + p.n_own;
  __syncthreads();  // shared memory is reused by the next head
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) page_select_kernel(const SelParams p) {
  extern __shared__ __align__(16) float sh[];
  if (p.need_scores) {
    query_sum<T>(p, sh);
    if (!grid_sync(p, 0, true)) return;
    mean_query(p);
    if (!grid_sync(p, 1, true)) return;
    page_scores(p, sh);
    const bool selects = (int)blockIdx.x < p.g.Hkv;
    if (!grid_sync(p, 2, selects) || !selects) return;
  }
  for (int h = blockIdx.x; h < p.g.Hkv; h += gridDim.x) top_k_head(p, h, reinterpret_cast<uint32_t*>(sh));
}

size_t query_sum_smem(const Geometry& g) {
  const int VEC = (int)(16 / dtype_size(g.dtype));
  const int row_vecs = g.Hq * g.d / VEC;
  const int spp = row_vecs <= kThreads ? kThreads / row_vecs : 1;
  return (size_t)spp * g.Hq * g.d * sizeof(float);
}

}  // namespace

size_t select_workspace_bytes(const Geometry& g, int n_q) {
  (void)n_q;
  const size_t HD = (size_t)g.Hkv * g.d;
  return align_up((size_t)kMaxBlocks * HD * 4, 256) + align_up(HD * 4, 256) +
         align_up((size_t)g.Hkv * align_up(g.max_logical, 64) * 4, 256);
}

cudaError_t launch_page_select(const Geometry& g, const float* summary, const int32_t* table, const void* q,
                               int64_t q_start, int n_q, int top_k, int n_sink, int32_t* sel, int32_t* sel_count,
                               int max_sel, void* ws, uint32_t* err, uint32_t* ctrl, uint32_t epoch,
                               cudaStream_t st) {
  const size_t HD = (size_t)g.Hkv * g.d;
  char* w = (char*)ws;
  SelParams p;
  p.g = g;
  p.q = q;
  p.n_q = n_q;
  p.summary = summary;
  p.table = table;
  p.partial = (float*)w;
  w += align_up((size_t)kMaxBlocks * HD * 4, 256);
  p.qbar = (float*)w;
  w += align_up(HD * 4, 256);
  p.keys = (uint32_t*)w;
  p.key_stride = (int)align_up(g.max_logical, 64);
  const int P = g.P;
  const int n_hist = (int)(q_start / P);
  p.n_sinks = n_sink < n_hist ? n_sink : n_hist;
  p.cand0 = p.n_sinks;
  p.n_cand = n_hist - p.n_sinks;
  p.own0 = n_hist;
  p.n_own = (int)((q_start + n_q + P - 1) / P) - n_hist;
  p.top_k = top_k;
  p.max_sel = max_sel;
  p.sel = sel;
  p.sel_count = sel_count;
  p.err = err;
  p.ctrl = ctrl;
  p.epoch = epoch;
  p.inv_count = 1.0f / ((float)n_q * g.G);
  p.need_scores = p.n_cand > 0 && top_k > 0 && p.n_cand > top_k;
  p.keys_in_smem = p.n_cand <= kMaxSmemKeys;

  const bool bf16 = g.dtype != OOMB_FP32;
  const void* fn = bf16 ? (const void*)page_select_kernel<__nv_bfloat16> : (const void*)page_select_kernel<float>;
  size_t smem = 0;
  int grid = g.Hkv;
  if (p.need_scores) {
    smem = query_sum_smem(g);
    smem = std::max(smem, (size_t)g.Hkv * (g.d + 4) * sizeof(float));
    if (p.keys_in_smem) smem = std::max(smem, (size_t)p.n_cand * sizeof(uint32_t));
  }
  static size_t configured[2] = {0, 0};
  if (smem > 48 * 1024 && smem > configured[bf16]) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[bf16] = smem;
  }
  if (!p.need_scores) {
    p.rows_per_block = 0;
    p.lanes_per_item = 1;
    void* args[] = {&p};
    cudaError_t e = cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, smem, st);
    count_launches(1);
    return e;
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  grid = std::min(num_sms(), kMaxBlocks);
  p.rows_per_block = (n_q + grid - 1) / grid;
  // lanes per (page, head) item: enough items to give every thread work, at most a warp
  const long long n_items = (long long)p.n_cand * g.Hkv;
  int L = 32;
  while (L > 1 && (n_items * L > (long long)grid * kThreads || (g.d / 4) % L != 0)) L >>= 1;
  p.lanes_per_item = L;
  void* args[] = {&p};
  e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), args, smem, st);
  count_launches(1);
  return e;
}

}  // namespace oomb
