// Page-level top-K selection for one query chunk.
//
// "Out of the Memory Barrier" (gist.science explainer, 2.D "Page-Level Sparse
// Attention"): only the top-K most relevant key pages are retrieved, ranked by a
// representative (averaged) vector.  The scoring rule is the mean key of each
// page against the mean query of the chunk's KV group; ties go to the lower
// logical page.  The sink pages and the chunk's own pages are always kept.
//
// Four small kernels, all bandwidth- or latency-bound:
//   qsum_partial  sum of the chunk's queries per block and KV group (reads Q once)
//   qbar_reduce   fixed-order sum of the partials -> mean query per KV head
//   page_score    one warp per candidate page: qbar . summary[phi(p)]
//   topk_select   one block per KV head: 4-pass radix select on order-preserving
//                 32-bit keys, ties resolved by page index, ordered compaction.
#include "oomb_internal.h"

namespace oomb {
namespace {

constexpr int kQsumThreads = 512;
constexpr int kMaxQsumBlocks = 512;
constexpr int kScoreWarps = 8;
constexpr int kTopkThreads = 1024;

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

// partial[b][h][col] = sum over rows of block b and heads g of group h of q[row, h*G+g, col]
template <typename T>
__global__ void __launch_bounds__(kQsumThreads)
    qsum_partial(Geometry g, const T* __restrict__ q, int n_q, int rows_per_block, float* __restrict__ partial) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int kMaxPerThread = 4;
  const int nvec = g.d / VEC;
  const int row_vecs = g.Hq * nvec;
  const int r0 = blockIdx.x * rows_per_block;
  const int r1 = min(n_q, r0 + rows_per_block);
  float acc[kMaxPerThread][VEC];
#pragma unroll
  for (int j = 0; j < kMaxPerThread; ++j)
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[j][e] = 0.f;
  for (int r = r0; r < r1; ++r) {
    const T* row = q + (size_t)r * row_vecs * VEC;
#pragma unroll
    for (int j = 0; j < kMaxPerThread; ++j) {
      const int vi = threadIdx.x + j * kQsumThreads;
      if (vi < row_vecs) {
        uint4 raw = __ldg(reinterpret_cast<const uint4*>(row) + vi);
        const T* x = reinterpret_cast<const T*>(&raw);
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[j][e] += to_f<T>(x[e]);
      }
    }
  }
  extern __shared__ float sh[];  // [row_vecs][VEC]
#pragma unroll
  for (int j = 0; j < kMaxPerThread; ++j) {
    const int vi = threadIdx.x + j * kQsumThreads;
    if (vi < row_vecs)
#pragma unroll
      for (int e = 0; e < VEC; ++e) sh[vi * VEC + e] = acc[j][e];
  }
  __syncthreads();
  const int HD = g.Hkv * g.d;
  for (int idx = threadIdx.x; idx < HD; idx += kQsumThreads) {
    const int h = idx / g.d, col = idx % g.d;
    float s = 0.f;
    for (int gg = 0; gg < g.G; ++gg) s += sh[(h * g.G + gg) * g.d + col];
    partial[(size_t)blockIdx.x * HD + idx] = s;
  }
}

__global__ void qbar_reduce(Geometry g, const float* __restrict__ partial, int nb, float inv_count,
                            float* __restrict__ qbar) {
  const int HD = g.Hkv * g.d;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < HD; idx += gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int b = 0; b < nb; ++b) s += partial[(size_t)b * HD + idx];
    qbar[idx] = s * inv_count;
  }
}

// scores[h][i] = qbar[h] . summary[phi(cand0 + i)][h]
__global__ void __launch_bounds__(kScoreWarps * 32)
    page_score(Geometry g, const float* __restrict__ qbar, const float* __restrict__ summary,
               const int32_t* __restrict__ table, int cand0, int n_cand, int score_stride,
               float* __restrict__ scores, uint32_t* err) {
  const int h = blockIdx.y;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int i = blockIdx.x * kScoreWarps + warp;
  if (i >= n_cand) return;
  const int p = cand0 + i;
  const int phys = table[p];
  float s = 0.f;
  if (phys < 0 || phys >= g.num_phys) {
    if (lane == 0) atomicOr(err, OOMB_DEVERR_PAGE);
  } else {
    const float* kb = summary + ((size_t)phys * g.Hkv + h) * g.d;
    const float* qb = qbar + (size_t)h * g.d;
    for (int c = lane * 4; c < g.d; c += 128) {
      float4 a = *reinterpret_cast<const float4*>(qb + c);
      float4 b = __ldg(reinterpret_cast<const float4*>(kb + c));
      s += a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  }
  if (lane == 0) scores[(size_t)h * score_stride + i] = s;
}

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f + 0.0f);  // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread (blockDim = kTopkThreads). Returns the total.
__device__ int block_exclusive_scan(int v, int* out, int* sh_warp) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < kTopkThreads / 32) ? sh_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh_warp[lane] = w;  // inclusive prefix over warps
  }
  __syncthreads();
  const int warp_base = warp > 0 ? sh_warp[warp - 1] : 0;
  *out = warp_base + x - v;
  const int total = sh_warp[kTopkThreads / 32 - 1];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kTopkThreads)
    topk_select(Geometry g, const float* __restrict__ scores, int score_stride, int n_sinks, int cand0, int n_cand,
                int top_k, int own0, int n_own, int32_t* __restrict__ sel, int32_t* __restrict__ sel_count,
                int max_sel) {
  const int h = blockIdx.x;
  const float* sc = scores + (size_t)h * score_stride;
  int32_t* out = sel + (size_t)h * max_sel;
  __shared__ int hist[256];
  __shared__ int sh_warp[32];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_need;

  const bool take_all = (top_k < 0) || (n_cand <= top_k);
  uint32_t T = 0;
  int need_eq = 0;  // keys equal to T that are taken (lowest pages first)
  if (!take_all && top_k > 0) {
    uint32_t prefix = 0, mask = 0;
    int k_rem = top_k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int b = threadIdx.x; b < 256; b += kTopkThreads) hist[b] = 0;
      __syncthreads();
      for (int i = threadIdx.x; i < n_cand; i += kTopkThreads) {
        const uint32_t u = order_key(sc[i]);
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 0xFF], 1);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int cum = 0, b = 255;
        for (; b > 0; --b) {
          if (cum + hist[b] >= k_rem) break;
          cum += hist[b];
        }
        sh_prefix = prefix | ((uint32_t)b << shift);
        sh_need = k_rem - cum;
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
  // ordered compaction of the kept candidates; thread t owns a contiguous segment
  const int seg = (n_cand + kTopkThreads - 1) / kTopkThreads;
  const int i0 = min(n_cand, threadIdx.x * seg), i1 = min(n_cand, i0 + seg);
  int n_eq = 0;
  if (!take_all)
    for (int i = i0; i < i1; ++i) n_eq += (order_key(sc[i]) == T);
  int eq_before;
  block_exclusive_scan(n_eq, &eq_before, sh_warp);
  int n_keep = 0;
  if (take_all) {
    n_keep = i1 - i0;
  } else if (top_k > 0) {
    int eq_seen = eq_before;
    for (int i = i0; i < i1; ++i) {
      const uint32_t u = order_key(sc[i]);
      if (u > T || (u == T && eq_seen++ < need_eq)) ++n_keep;
    }
  }
  int keep_before;
  const int kept = block_exclusive_scan(n_keep, &keep_before, sh_warp);
  {
    int o = n_sinks + keep_before;
    int eq_seen = eq_before;
    for (int i = i0; i < i1; ++i) {
      bool take;
      if (take_all) {
        take = true;
      } else if (top_k > 0) {
        const uint32_t u = order_key(sc[i]);
        take = u > T || (u == T && eq_seen++ < need_eq);
      } else {
        take = false;
      }
      if (take) out[o++] = cand0 + i;
    }
  }
  for (int s = threadIdx.x; s < n_sinks; s += kTopkThreads) out[s] = s;
  for (int s = threadIdx.x; s < n_own; s += kTopkThreads) out[n_sinks + kept + s] = own0 + s;
  if (threadIdx.x == 0) sel_count[h] = n_sinks + kept + n_own;
}

}  // namespace

size_t select_workspace_bytes(const Geometry& g, int n_q) {
  (void)n_q;
  const size_t HD = (size_t)g.Hkv * g.d;
  return align_up((size_t)kMaxQsumBlocks * HD * 4, 256) + align_up(HD * 4, 256) +
         align_up((size_t)g.Hkv * align_up(g.max_logical, 64) * 4, 256);
}

cudaError_t launch_page_select(const Geometry& g, const float* summary, const int32_t* table, const void* q,
                               int64_t q_start, int n_q, int top_k, int n_sink, int32_t* sel, int32_t* sel_count,
                               int max_sel, void* ws, uint32_t* err, cudaStream_t st) {
  const size_t HD = (size_t)g.Hkv * g.d;
  char* w = (char*)ws;
  float* partial = (float*)w;
  w += align_up((size_t)kMaxQsumBlocks * HD * 4, 256);
  float* qbar = (float*)w;
  w += align_up(HD * 4, 256);
  float* scores = (float*)w;
  const int score_stride = (int)align_up(g.max_logical, 64);

  const int P = g.P;
  const int n_hist = (int)(q_start / P);
  const int n_sinks = n_sink < n_hist ? n_sink : n_hist;
  const int cand0 = n_sinks, n_cand = n_hist - n_sinks;
  const int own0 = n_hist;
  const int n_own = (int)((q_start + n_q + P - 1) / P) - n_hist;

  const bool need_scores = n_cand > 0 && top_k >= 0 && n_cand > top_k && top_k > 0;
  if (need_scores) {
    int nb = 2 * num_sms();
    if (nb > kMaxQsumBlocks) nb = kMaxQsumBlocks;
    if (nb > n_q) nb = n_q;
    const int rows = (n_q + nb - 1) / nb;
    nb = (n_q + rows - 1) / rows;
    const size_t esz = dtype_size(g.dtype);
    const int VEC = (int)(16 / esz);
    if (g.Hq * (g.d / VEC) > 4 * kQsumThreads) return cudaErrorInvalidValue;
    const size_t shb = (size_t)g.Hq * g.d * sizeof(float);
    if (g.dtype == OOMB_FP32)
      qsum_partial<float><<<nb, kQsumThreads, shb, st>>>(g, (const float*)q, n_q, rows, partial);
    else
      qsum_partial<__nv_bfloat16><<<nb, kQsumThreads, shb, st>>>(g, (const __nv_bfloat16*)q, n_q, rows, partial);
    qbar_reduce<<<(int)((HD + 255) / 256), 256, 0, st>>>(g, partial, nb, 1.0f / ((float)n_q * g.G), qbar);
    dim3 sg((n_cand + kScoreWarps - 1) / kScoreWarps, g.Hkv);
    page_score<<<sg, kScoreWarps * 32, 0, st>>>(g, qbar, summary, table, cand0, n_cand, score_stride, scores, err);
    count_launches(3);
  }
  topk_select<<<g.Hkv, kTopkThreads, 0, st>>>(g, scores, score_stride, n_sinks, cand0, n_cand, top_k, own0, n_own,
                                               sel, sel_count, max_sel);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace oomb
