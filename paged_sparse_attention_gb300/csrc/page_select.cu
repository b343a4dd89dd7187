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
// the CTA returns).  Every CTA owns a contiguous slice of the query rows and a
// contiguous slice of the candidate pages.
//   0. prefetch      at launch, warp 0 bulk-copies the summary rows of the CTA's
//                    pages (all KV heads of a page are contiguous) into shared
//                    memory; the copies land while phase 1 runs
//   1. query sum     work unit u = (row slice u / Hkv, KV head u % Hkv): the G
//                    query heads of the head over the slice's rows, 16-byte loads,
//                    several rows in flight per thread -> partial[u][d]
//                    (Q is read exactly once)
//   2. mean query    every CTA sums the partials of each head itself, slices in
//                    one fixed order, into shared memory (no second barrier;
//                    every CTA gets the same bits)
//   3. page scores   qbar[h] . summary row, from shared memory; each score is
//                    stored as an order-preserving 32-bit key and counted in a
//                    per-head histogram of its top 12 bits (global atomics)
//   (with an append fused in: before phase 1, the CTA's two 256-thread halves append
//    (new page, KV head) units of the chunk's own K/V, append_unit.cuh, the same
//    arithmetic as the append kernel; the selection reads only history pages, the
//    append writes only the own pages, so the two share nothing)
//   4. top-k         one CTA per KV head: the histogram gives the 12-bit prefix of
//                    the k-th largest key; the keys in that bin are gathered and a
//                    bitwise search over the remaining 20 bits finds the exact
//                    threshold; an ordered, warp-contiguous compaction keeps every
//                    key above it and, among keys equal to it, the lowest pages.
// Every sum runs in a fixed order and the histogram is integer, so the selection
// is deterministic.  The barrier counters live in the pool's control block and
// are sense-reversing (see grid_sync): the host keeps no state between calls.
#include "append_unit.cuh"
#include "oomb_internal.h"
#include "sm103_ptx.cuh"

namespace oomb {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxBlocks = 256;        // upper bound of the grid (one CTA per SM)
constexpr int kRowUnroll = 8;          // query rows in flight per thread in phase 1
constexpr int kMaxSlots = 4;           // 16-byte query columns per thread (G*d <= 2048 vectors)
constexpr int kHistBits = 12;          // top bits of a key counted in phase 3
constexpr int kHistBins = 1 << kHistBits;
constexpr int kListCap = 2048;         // keys of the threshold bin gathered for the exact search
constexpr int kMaxSmemKeys = 40960;    // candidates per KV head staged in shared memory
constexpr size_t kSumBytesCap = 128 * 1024;  // summary rows staged per CTA (two halves)
constexpr long long kSpinLimit = 1ll << 31;
constexpr int kCtrlCount = 4;          // control-block words 4..5: barrier counters
constexpr int kBarriers = 2;
static_assert(kCtrlCount + kBarriers <= OOMB_CTRL_WORDS, "barrier counters must fit the control block");
static_assert(kThreads * 8 == kHistBins, "phase 4 gives every thread eight histogram bins");

struct SelParams {
  Geometry g;
  const void* q;
  int n_q;
  int rows_per_block;   // query rows of one slice
  int n_slices;         // row slices; work units = n_slices * Hkv
  const float* summary;
  const int32_t* table;
  int n_sinks, cand0, n_cand, own0, n_own, top_k, max_sel;
  int n_mapped_cand;    // candidates whose page is mapped (freed pages are not candidates)
  int any_unmapped;     // some sink or candidate page is unmapped
  int pages_per_block;  // candidate pages scored by one CTA
  int half_pages;       // pages per shared-memory summary buffer (two buffers)
  uint32_t sum_off;     // byte offset of the summary buffers in dynamic shared memory
  float inv_count;
  float* partial;       // [gridDim.x][Hkv*d]
  uint32_t* keys;       // [Hkv][key_stride]
  uint32_t* hist;       // [Hkv][kHistBins]
  int key_stride;
  int keys_in_smem;
  int need_scores;
  int32_t* sel;
  int32_t* sel_count;
  uint32_t* err;
  uint32_t* ctrl;
};

// The append fused into a selection: the chunk's own pages, new_phys[i] for own page i.
struct FusedAppend {
  int n_new;
  AppendJob job;
  int32_t new_phys[kMaxFusedAppendPages];
};


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
__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}
__device__ __forceinline__ uint32_t atom_release_add(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Grid barrier i, sense-reversing: CTA 0 adds 2^31 - (gridDim.x - 1) to counter i
// and every other CTA adds 1, so one barrier's arrivals sum to exactly 2^31.  The
// counter's low 31 bits are zero between barriers, so its top bit flips when, and
// only when, the last CTA arrives (before that, CTA 0's share borrows from it);
// a waiting CTA spins until the top bit differs from the one its own arrival saw.
// The counter needs no reset and the host keeps no state, so the launch can be
// replayed from a CUDA graph.  Returns false when the wait ran out (~1 s), after
// setting the timeout bit (oomb_check then clears the whole control block).
__device__ bool grid_sync(const SelParams& p, int i, bool wait) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t* cnt = p.ctrl + kCtrlCount + i;
    const uint32_t add = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1u) : 1u;
    const uint32_t sense = atom_release_add(cnt, add) & 0x80000000u;
    int ok = 1;
    if (wait) {
      const long long t0 = clock64();
      while ((ld_acquire(cnt) & 0x80000000u) == sense) {
        if (clock64() - t0 > kSpinLimit) {
          atomicOr(p.err, OOMB_DEVERR_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// ------------------------------------------------------------------ phase 0
// Bulk-copy the summary rows (Hkv * d fp32, contiguous per page) of pages
// [first, first + n) of the candidates into buffer `buf`.  Called by warp 0.
// An unmapped (freed) page's row is zero-filled; it gets the lowest key in phase 3.
__device__ void prefetch_summaries(const SelParams& p, uint8_t* smem, uint64_t* bar, int buf, int first, int n) {
  const int lane = threadIdx.x % 32;
  const uint32_t row_bytes = (uint32_t)(p.g.Hkv * p.g.d * 4);
  uint8_t* dst0 = smem + p.sum_off + (size_t)buf * p.half_pages * row_bytes;
  int n_valid = 0;
  for (int j = lane; j < n; j += 32) {
    const int phys = __ldg(p.table + p.cand0 + first + j);
    n_valid += (phys >= 0 && phys < p.g.num_phys);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n_valid += __shfl_xor_sync(0xffffffffu, n_valid, o);
  if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)n_valid * row_bytes);
  __syncwarp();
  for (int j = lane; j < n; j += 32) {
    const int phys = __ldg(p.table + p.cand0 + first + j);
    uint8_t* dst = dst0 + (size_t)j * row_bytes;
    if (phys >= 0 && phys < p.g.num_phys) {
      bulk_load(dst, p.summary + (size_t)phys * p.g.Hkv * p.g.d, row_bytes, bar);
    } else {
      if (phys >= p.g.num_phys) atomicOr(p.err, OOMB_DEVERR_PAGE);  // corrupt entry (-1 = freed)
      for (uint32_t b = 0; b < row_bytes; b += 16) *reinterpret_cast<uint4*>(dst + b) = make_uint4(0, 0, 0, 0);
    }
  }
}

// ------------------------------------------------------------------ phase 1
// Work units u = slice * Hkv + h for u = blockIdx.x, blockIdx.x + gridDim.x, ...
template <typename T>
__device__ void query_sum(const SelParams& p, float* sh) {
  constexpr int VEC = 16 / sizeof(T);
  const Geometry& g = p.g;
  const int tid = threadIdx.x;
  const int row_vecs = g.G * g.d / VEC;  // one KV group of one row
  const int stride = g.Hq * g.d / VEC;   // one row
  const bool narrow = row_vecs <= kThreads;
  const int spp = narrow ? kThreads / row_vecs : 1;  // rows per pass of the CTA
  const int n_slots = narrow ? 1 : (row_vecs + kThreads - 1) / kThreads;
  const int phase = narrow ? tid / row_vecs : 0;
  const int GD = g.G * g.d;
  const uint4* q4 = reinterpret_cast<const uint4*>(p.q);
  for (int u = blockIdx.x; u < p.n_slices * g.Hkv; u += gridDim.x) {
    const int h = u % g.Hkv, slice = u / g.Hkv;
    const int r0 = slice * p.rows_per_block;
    const int r1 = min(p.n_q, r0 + p.rows_per_block);
    const uint4* base = q4 + (size_t)h * row_vecs;
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
        for (int k = 0; k < kRowUnroll; ++k) {
          const int r = rb + k * spp;
          buf[k] = r < r1 ? __ldg(base + (size_t)r * stride + col) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < kRowUnroll; ++k) {
          const T* x = reinterpret_cast<const T*>(&buf[k]);
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[e] += to_f<T>(x[e]);
        }
      }
#pragma unroll
      for (int e = 0; e < VEC; ++e) sh[phase * GD + col * VEC + e] = acc[e];
    }
    __syncthreads();
    for (int c = tid; c < g.d; c += kThreads) {
      float t = 0.f;
      for (int ph = 0; ph < spp; ++ph)
        for (int gg = 0; gg < g.G; ++gg) t += sh[ph * GD + gg * g.d + c];
      p.partial[(size_t)u * g.d + c] = t;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ phase 2
// qbar[h] = (sum over slices of partial[slice * Hkv + h]) / (rows x group size),
// computed by every CTA into shared memory: thread t sums float4 column t % n4 of
// qbar over the slices gi, gi + groups, ... (gi = t / n4), then the groups are
// added in order.
__device__ void mean_query(const SelParams& p, float* sh) {
  const int tid = threadIdx.x;
  const int d4 = p.g.d / 4, n4 = p.g.Hkv * d4;
  const int ns = p.n_slices;
  const int width = min(n4, kThreads);
  const int groups = max(1, kThreads / n4);
  float4* part = reinterpret_cast<float4*>(sh + 4 * n4);  // [groups][width]
  const float4* src = reinterpret_cast<const float4*>(p.partial);
  const int stride = p.g.Hkv * d4;  // float4 per slice
  for (int c0 = 0; c0 < n4; c0 += width) {
    const int col = c0 + tid % width, gi = tid / width;
    if (gi < groups && col < n4) {
      const int h = col / d4, c4 = col % d4;
      const float4* s0 = src + (size_t)h * d4 + c4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      int sl = gi;
      for (; sl + 7 * groups < ns; sl += 8 * groups) {
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __ldcg(s0 + (size_t)(sl + k * groups) * stride);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          acc.x += v[k].x;
          acc.y += v[k].y;
          acc.z += v[k].z;
          acc.w += v[k].w;
        }
      }
      for (; sl < ns; sl += groups) {
        const float4 v = __ldcg(s0 + (size_t)sl * stride);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      part[gi * width + (col - c0)] = acc;
    }
    __syncthreads();
    for (int c = tid; c < min(width, n4 - c0); c += kThreads) {
      float4 t = part[c];
      for (int gi2 = 1; gi2 < groups; ++gi2) {
        const float4 v = part[gi2 * width + c];
        t.x += v.x;
        t.y += v.y;
        t.z += v.z;
        t.w += v.w;
      }
      const float inv = p.inv_count;
      reinterpret_cast<float4*>(sh)[c0 + c] = make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ phase 3
// Scores of this CTA's pages from the staged summary rows, one warp per (page,
// head) item: lane l reads float4 l of the row and of qbar (conflict-free), two
// items per iteration.  Rounds of half_pages pages alternate between the two
// buffers; round r + 2 is fetched once round r is done.
__device__ __forceinline__ float warp_dot(const float4* a, const float4* b, int d4, int lane) {
  float s = 0.f;
  for (int c = lane; c < d4; c += 32) {
    const float4 x = a[c], y = b[c];
    s += x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
  }
  return s;
}

__device__ bool page_scores(const SelParams& p, float* sh, uint64_t* sum_full, volatile int* abort) {
  const Geometry& g = p.g;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int d4 = g.d / 4;
  const float4* qbar4 = reinterpret_cast<const float4*>(sh);
  const int j0 = blockIdx.x * p.pages_per_block;
  const int n_pages = max(0, min(p.n_cand, j0 + p.pages_per_block) - j0);
  const int n_rounds = (n_pages + p.half_pages - 1) / p.half_pages;
  const uint8_t* smem = reinterpret_cast<const uint8_t*>(sh);
  bool ok = true;
  int waited = 0, issued = min(2, n_rounds);  // rounds whose copies landed / were issued
  __syncthreads();
  for (int r = 0; r < n_rounds; ++r) {
    const int buf = r & 1;
    const int first = r * p.half_pages, n = min(p.half_pages, n_pages - first);
    ok = ok && mbar_wait(&sum_full[buf], (r >> 1) & 1, p.err, abort);
    if (ok) {
      waited = r + 1;
      // item it = page jj * Hkv + head h is row it of the buffer (rows are [page][head][d])
      const float4* rows = reinterpret_cast<const float4*>(smem + p.sum_off) + (size_t)buf * p.half_pages * g.Hkv * d4;
      const int n_items = n * g.Hkv;
      for (int it = warp; it < n_items; it += 2 * kWarps) {  // warp-uniform
        const int it2 = it + kWarps;
        float s0 = warp_dot(qbar4 + (it % g.Hkv) * d4, rows + (size_t)it * d4, d4, lane);
        float s1 = it2 < n_items ? warp_dot(qbar4 + (it2 % g.Hkv) * d4, rows + (size_t)it2 * d4, d4, lane) : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          s0 += __shfl_xor_sync(0xffffffffu, s0, off);
          s1 += __shfl_xor_sync(0xffffffffu, s1, off);
        }
        if (lane < 2 && (lane == 0 || it2 < n_items)) {
          const int i2 = lane == 0 ? it : it2;
          const int h = i2 % g.Hkv, j = j0 + first + i2 / g.Hkv;
          // a mapped page's key is at least 1; an unmapped (freed) page's is 0, below all
          uint32_t key = max(order_key(lane == 0 ? s0 : s1), 1u);
          if (p.any_unmapped && __ldg(p.table + p.cand0 + j) < 0) key = 0u;
          p.keys[(size_t)h * p.key_stride + j] = key;
          atomicAdd(&p.hist[h * kHistBins + (key >> (32 - kHistBits))], 1u);
        }
      }
    }
    __syncthreads();  // this buffer is free again
    if (ok && !*abort && r + 2 < n_rounds) {
      if (tid < 32) {
        const int f2 = (r + 2) * p.half_pages;
        prefetch_summaries(p, reinterpret_cast<uint8_t*>(sh), &sum_full[buf], buf, j0 + f2,
                           min(p.half_pages, n_pages - f2));
      }
      issued = r + 3;
    }
  }
  if (!ok && tid == 0)  // copies still in flight land (bounded wait) before the CTA leaves
    for (int r = waited; r < issued; ++r) mbar_wait(&sum_full[r & 1], (r >> 1) & 1, p.err, nullptr);
  __syncthreads();
  return ok;
}

// ------------------------------------------------------------------ phase 4
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
// Keys i .. i+3 (i a multiple of 4; key rows are padded to 64 keys and 16-byte aligned).
__device__ __forceinline__ uint4 keys4_at(const uint32_t* keys, bool smem, int i) {
  return smem ? *reinterpret_cast<const uint4*>(keys + i) : __ldcg(reinterpret_cast<const uint4*>(keys + i));
}

// Sinks, the kept candidates in ascending page order, own pages, for KV head h.
// Candidates are split into warp-contiguous segments; lanes stride by one key.
__device__ void top_k_head(const SelParams& p, int h, uint32_t* sh_keys) {
  __shared__ int sh_warp[32];
  __shared__ int w_gt[kWarps], w_eq[kWarps], w_eq_before[kWarps], w_keep_before[kWarps];
  __shared__ uint32_t list_key[kListCap];
  __shared__ int list_idx[kListCap];
  __shared__ int list_n, sh_bin, sh_krem, sh_kept, sh_need;
  __shared__ uint32_t sh_T;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  __shared__ int sh_ns;
  const int n_cand = p.n_cand, top_k = p.top_k;
  int32_t* out = p.sel + (size_t)h * p.max_sel;
  const bool take_all = (top_k < 0) || (p.n_mapped_cand <= top_k);
  const bool scored = !take_all && top_k > 0;
  // the sink pages that are mapped (a freed page is no longer kept), in order
  int ns = p.n_sinks;
  if (p.any_unmapped) {
    if (tid == 0) {
      int c = 0;
      for (int s = 0; s < p.n_sinks; ++s)
        if (__ldg(p.table + s) >= 0) out[c++] = s;
      sh_ns = c;
    }
    __syncthreads();
    ns = sh_ns;
  } else {
    for (int s = tid; s < p.n_sinks; s += kThreads) out[s] = s;
  }
  int kept = 0;
  if (take_all && !p.any_unmapped) {
    for (int i = tid; i < n_cand; i += kThreads) out[ns + i] = p.cand0 + i;
    kept = n_cand;
  } else if (take_all) {  // every mapped candidate, in page order
    for (int base = 0; base < n_cand; base += kThreads) {
      const int i = base + tid;
      const int mapped = (i < n_cand && __ldg(p.table + p.cand0 + i) >= 0) ? 1 : 0;
      int before;
      const int total = block_exclusive_scan(mapped, &before, sh_warp);
      if (mapped) out[ns + kept + before] = p.cand0 + i;
      kept += total;
    }
  } else if (scored) {
    const bool smem = p.keys_in_smem;
    const uint32_t* keys = p.keys + (size_t)h * p.key_stride;
    // (1) 12-bit prefix of the top_k-th largest key.  Thread t holds bins 4095-8t .. 4088-8t.
    const uint32_t* hist = p.hist + (size_t)h * kHistBins;
    int c8[8], s8 = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) c8[e] = (int)__ldcg(hist + (kHistBins - 1 - (tid * 8 + e)));
    if (smem) {  // 16-byte loads; key rows are 16-byte aligned and padded to 64 keys
      const int n4 = (n_cand + 3) / 4;
      for (int i = tid; i < n4; i += kThreads)
        reinterpret_cast<uint4*>(sh_keys)[i] = __ldcg(reinterpret_cast<const uint4*>(keys) + i);
      keys = sh_keys;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) s8 += c8[e];
    if (tid == 0) list_n = 0;
    if (tid < kWarps) w_gt[tid] = w_eq[tid] = 0;
    int above;
    block_exclusive_scan(s8, &above, sh_warp);  // keys in higher bins than this thread's
    if (above < top_k && above + s8 >= top_k) {
      int cum = above, pick = 7;
      bool found = false;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (!found && cum + c8[e] >= top_k) {
          pick = e;
          found = true;
        }
        if (!found) cum += c8[e];
      }
      sh_bin = kHistBins - 1 - (tid * 8 + pick);
      sh_krem = top_k - cum;  // keys of that bin still to take
    }
    __syncthreads();
    const uint32_t bin = (uint32_t)sh_bin;
    const int k_rem = sh_krem;
    const bool listed = (int)__ldcg(hist + bin) <= kListCap;
    // warp w owns keys [w*wseg, (w+1)*wseg); a round gives every lane four consecutive keys
    const int wseg = ((n_cand + kWarps * 128 - 1) / (kWarps * 128)) * 128;
    const int i0 = min(n_cand, warp * wseg), i1 = min(n_cand, i0 + wseg);
    // (2) one pass: keys in higher bins per warp; the bin's keys (with their index) to the list
    int n_above = 0;
    for (int base = i0; base < i1; base += 128) {
      const int i = base + 4 * lane;
      uint32_t u[4] = {0u, 0u, 0u, 0u};
      if (i < i1) {
        const uint4 v = keys4_at(keys, smem, i);
        u[0] = v.x; u[1] = v.y; u[2] = v.z; u[3] = v.w;
      }
      bool in[4];
      uint32_t m[4];
      int total = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t pre = u[e] >> (32 - kHistBits);
        n_above += (i + e < i1 && pre > bin);
        in[e] = listed && i + e < i1 && pre == bin;
        m[e] = __ballot_sync(0xffffffffu, in[e]);
        total += __popc(m[e]);
      }
      if (total) {  // warp-uniform; the list's order does not matter
        int slot0 = 0;
        if (lane == 0) slot0 = atomicAdd(&list_n, total);
        slot0 = __shfl_sync(0xffffffffu, slot0, 0);
        const uint32_t lt = lanemask_lt();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (in[e]) {
            const int sidx = slot0 + __popc(m[e] & lt);
            list_key[sidx] = u[e];
            list_idx[sidx] = i + e;
          }
          slot0 += __popc(m[e]);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n_above += __shfl_xor_sync(0xffffffffu, n_above, o);
    __syncthreads();
    // (3) exact threshold T: the k_rem-th largest key of the bin
    if (listed) {
      const int n = list_n;
      if (n <= kThreads) {  // rank of every listed key by counting (broadcast reads)
        if (tid < n) {
          const uint32_t x = list_key[tid];
          int greater = 0, equal = 0;
          for (int i = 0; i < n; ++i) {
            const uint32_t y = list_key[i];
            greater += y > x;
            equal += y == x;
          }
          if (greater < k_rem && greater + equal >= k_rem) sh_T = x;  // every writer writes x
        }
      } else {  // bitwise search over the low 20 bits, counted with one barrier per slot
        uint32_t t = bin << (32 - kHistBits);
        for (int b = 31 - kHistBits; b >= 0; --b) {
          const uint32_t trial = t | (1u << b);
          int c = 0;
          for (int s0 = 0; s0 < n; s0 += kThreads) c += __syncthreads_count(s0 + tid < n && list_key[s0 + tid] >= trial);
          if (c >= k_rem) t = trial;
        }
        if (tid == 0) sh_T = t;
      }
    } else {
      // more tied-bin keys than the list holds: the whole block searches over every key
      uint32_t t = bin << (32 - kHistBits);
      for (int b = 31 - kHistBits; b >= 0; --b) {
        const uint32_t trial = t | (1u << b);
        int c = 0;
        for (int i = tid; i < n_cand; i += kThreads) {
          const uint32_t u = key_at(keys, smem, i);
          c += ((u >> (32 - kHistBits)) == bin && u >= trial);
        }
        int dummy;
        const int total = block_exclusive_scan(c, &dummy, sh_warp);
        if (total >= k_rem) t = trial;
      }
      if (tid == 0) sh_T = t;
    }
    __syncthreads();
    const uint32_t T = sh_T;
    // (4) per-warp counts of keys > T and == T
    if (listed) {
      for (int s = tid; s < list_n; s += kThreads) {
        const uint32_t u = list_key[s];
        const int w = list_idx[s] / wseg;
        if (u > T) atomicAdd(&w_gt[w], 1);
        if (u == T) atomicAdd(&w_eq[w], 1);
      }
      if (lane == 0) atomicAdd(&w_gt[warp], n_above);
    } else {
      int gt = 0, eq = 0;
      for (int base = i0; base < i1; base += 128) {
        const int i = base + 4 * lane;
        if (i < i1) {
          const uint4 v = keys4_at(keys, smem, i);
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            gt += (i + e < i1 && u[e] > T);
            eq += (i + e < i1 && u[e] == T);
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        gt += __shfl_xor_sync(0xffffffffu, gt, o);
        eq += __shfl_xor_sync(0xffffffffu, eq, o);
      }
      if (lane == 0) {
        w_gt[warp] = gt;
        w_eq[warp] = eq;
      }
    }
    __syncthreads();
    if (warp == 0) {
      // every key > T is kept; among keys == T the first need_eq (lowest pages)
      int g_all = lane < kWarps ? w_gt[lane] : 0;
      const int e_w = lane < kWarps ? w_eq[lane] : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) g_all += __shfl_xor_sync(0xffffffffu, g_all, o);
      const int need_eq = top_k - g_all;
      int e_inc = e_w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, e_inc, o);
        if (lane >= o) e_inc += y;
      }
      const int e_before = e_inc - e_w;
      const int keep = (lane < kWarps ? w_gt[lane] : 0) + max(0, min(need_eq - e_before, e_w));
      int k_inc = keep;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, k_inc, o);
        if (lane >= o) k_inc += y;
      }
      if (lane < kWarps) {
        w_eq_before[lane] = e_before;
        w_keep_before[lane] = k_inc - keep;
      }
      if (lane == 31) sh_kept = k_inc;
      if (lane == 0) sh_need = need_eq;
    }
    __syncthreads();
    // (5) ordered compaction
    const int need_eq = sh_need;
    int pos = ns + w_keep_before[warp], eq_rank = w_eq_before[warp];
    for (int base = i0; base < i1; base += 128) {
      const int i = base + 4 * lane;
      uint32_t u[4] = {0u, 0u, 0u, 0u};
      if (i < i1) {
        const uint4 v = keys4_at(keys, smem, i);
        u[0] = v.x; u[1] = v.y; u[2] = v.z; u[3] = v.w;
      }
      // key (lane l, element e) comes before (l', e') iff l < l', or l == l' and e < e'
      const uint32_t lt = lanemask_lt();
      bool is_eq[4], take[4];
      int eq_lower = 0, eq_total = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        is_eq[e] = i + e < i1 && u[e] == T;
        const uint32_t m = __ballot_sync(0xffffffffu, is_eq[e]);
        eq_lower += __popc(m & lt);
        eq_total += __popc(m);
      }
      int r = eq_rank + eq_lower;  // tie rank of this lane's first key
      int t_lower = 0, t_total = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        take[e] = (i + e < i1 && u[e] > T) || (is_eq[e] && r < need_eq);
        r += is_eq[e];
        const uint32_t m = __ballot_sync(0xffffffffu, take[e]);
        t_lower += __popc(m & lt);
        t_total += __popc(m);
      }
      int o = pos + t_lower;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (take[e]) out[o++] = p.cand0 + i + e;
      pos += t_total;
      eq_rank += eq_total;
    }
    kept = sh_kept;
  }
  for (int s = tid; s < p.n_own; s += kThreads) out[ns + kept + s] = p.own0 + s;
  if (tid == 0) p.sel_count[h] = ns + kept + p.n_own;
  __syncthreads();  // shared memory is reused by the next head
}

// The selection, with (FUSED) or without the chunk's append before its query sum.
template <typename T, bool FUSED>
__device__ __forceinline__ void select_main(const SelParams& p, const FusedAppend* fa) {
  extern __shared__ __align__(128) float sh[];
  __shared__ uint64_t sum_full[2];
  __shared__ int abort_flag;
  if (p.need_scores) {
    const int j0 = blockIdx.x * p.pages_per_block;
    const int n_pages = max(0, min(p.n_cand, j0 + p.pages_per_block) - j0);
    if (threadIdx.x == 0) {
      abort_flag = 0;
      mbar_init(&sum_full[0], 1);
      mbar_init(&sum_full[1], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      for (int r = 0; r < 2; ++r) {
        const int first = r * p.half_pages;
        if (first < n_pages)
          prefetch_summaries(p, reinterpret_cast<uint8_t*>(sh), &sum_full[r], r, j0 + first,
                             min(p.half_pages, n_pages - first));
      }
    }
    // this CTA's slice of the histogram is zeroed here; it is first counted after two barriers
    const int hn = p.g.Hkv * kHistBins, hs = (hn + gridDim.x - 1) / gridDim.x;
    const int h0 = blockIdx.x * hs, h1 = min(hn, h0 + hs);
    for (int i = h0 + threadIdx.x; i < h1; i += kThreads) p.hist[i] = 0u;
    if (FUSED) {
      // the fused append: unit u = (own page u / Hkv, KV head u % Hkv), two at a time per
      // CTA, each half of the CTA on its own named barrier; `sh` is free until phase 1
      const int half = threadIdx.x / kAppendThreads;
      float* part = sh + half * kAppendThreads * 8;
      const int units = fa->n_new * p.g.Hkv;
      for (int u = 2 * blockIdx.x + half; u < units; u += 2 * gridDim.x)
        append_unit<T, 2>(fa->job, fa->new_phys[u / p.g.Hkv], u / p.g.Hkv, u % p.g.Hkv,
                          threadIdx.x % kAppendThreads, part, 1 + half);
      __syncthreads();
    }
    query_sum<T>(p, sh);
    if (!grid_sync(p, 0, true)) return;
    mean_query(p, sh);
    const bool ok = page_scores(p, sh, sum_full, &abort_flag);
    const bool selects = (int)blockIdx.x < p.g.Hkv;
    if (!grid_sync(p, 1, selects) || !selects || !ok) return;
  }
  for (int h = blockIdx.x; h < p.g.Hkv; h += gridDim.x) top_k_head(p, h, reinterpret_cast<uint32_t*>(sh));
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) page_select_kernel(const SelParams p) {
  select_main<T, false>(p, nullptr);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    page_select_append_kernel(const SelParams p, const __grid_constant__ FusedAppend fa) {
  select_main<T, true>(p, &fa);
}

size_t query_sum_smem(const Geometry& g) {
  const int VEC = (int)(16 / dtype_size(g.dtype));
  const int row_vecs = g.G * g.d / VEC;
  const int spp = row_vecs <= kThreads ? kThreads / row_vecs : 1;
  return (size_t)spp * g.G * g.d * sizeof(float);
}

}  // namespace

bool select_scores(int64_t q_start, int n_sink, int top_k, int n_mapped_cand, const Geometry& g) {
  const int n_hist = (int)(q_start / g.P);
  const int n_cand = n_hist - (n_sink < n_hist ? n_sink : n_hist);
  return n_cand > 0 && top_k > 0 && n_mapped_cand > top_k;
}

size_t select_workspace_bytes(const Geometry& g, int n_q) {
  (void)n_q;
  const size_t HD = (size_t)g.Hkv * g.d;
  return align_up((size_t)kMaxBlocks * HD * 4, 256) + align_up((size_t)g.Hkv * kHistBins * 4, 256) + align_up((size_t)g.Hkv * align_up(g.max_logical, 64) * 4, 256);
}

cudaError_t launch_page_select(const Geometry& g, const float* summary, const int32_t* table, const void* q,
                               int64_t q_start, int n_q, int top_k, int n_sink, int n_mapped_cand, int any_unmapped,
                               int32_t* sel, int32_t* sel_count, int max_sel, void* ws, uint32_t* err, uint32_t* ctrl,
                               cudaStream_t st, const AppendJob* job, const int32_t* new_phys, int n_new) {
  const size_t HD = (size_t)g.Hkv * g.d;
  char* w = (char*)ws;
  SelParams p;
  FusedAppend fa;
  fa.n_new = 0;
  if (job) {  // the caller has checked select_scores
    if (n_new <= 0 || n_new > kMaxFusedAppendPages) return cudaErrorInvalidValue;
    fa.n_new = n_new;
    fa.job = *job;
    for (int i = 0; i < n_new; ++i) fa.new_phys[i] = new_phys[i];
  }
  p.g = g;
  p.q = q;
  p.n_q = n_q;
  p.summary = summary;
  p.table = table;
  p.partial = (float*)w;
  w += align_up((size_t)kMaxBlocks * HD * 4, 256);
  p.hist = (uint32_t*)w;
  w += align_up((size_t)g.Hkv * kHistBins * 4, 256);
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
  p.inv_count = 1.0f / ((float)n_q * g.G);
  p.n_mapped_cand = n_mapped_cand;
  p.any_unmapped = any_unmapped;
  p.need_scores = p.n_cand > 0 && top_k > 0 && n_mapped_cand > top_k;
  p.keys_in_smem = p.n_cand <= kMaxSmemKeys;
  p.rows_per_block = 0;
  p.n_slices = 1;
  p.pages_per_block = p.half_pages = 0;
  p.sum_off = 0;

  const bool bf16 = g.dtype != OOMB_FP32;
  const void* fn = job ? (bf16 ? (const void*)page_select_append_kernel<__nv_bfloat16>
                               : (const void*)page_select_append_kernel<float>)
                       : (bf16 ? (const void*)page_select_kernel<__nv_bfloat16> : (const void*)page_select_kernel<float>);
  if (!p.need_scores) {
    if (job) return cudaErrorInvalidValue;  // a fused append needs the cooperative grid
    void* args[] = {&p};
    cudaError_t e = cudaLaunchKernel(fn, dim3(g.Hkv), dim3(kThreads), args, 0, st);
    count_launches(1);
    return e;
  }
  const int VEC = (int)(16 / dtype_size(g.dtype));
  if (g.G * g.d / VEC > kMaxSlots * kThreads) return cudaErrorInvalidValue;
  const int grid = std::min(device_sm_count(), kMaxBlocks);
  p.n_slices = std::max(1, grid / g.Hkv);
  p.rows_per_block = (n_q + p.n_slices - 1) / p.n_slices;
  p.pages_per_block = (p.n_cand + grid - 1) / grid;
  const size_t row_bytes = HD * 4;
  p.half_pages = (int)std::max<size_t>(1, std::min<size_t>((size_t)p.pages_per_block,
                                                            kSumBytesCap / 2 / row_bytes));
  const int n4 = (int)(HD / 4), groups = std::max(1, kThreads / n4);
  const size_t qbar_bytes = HD * sizeof(float) + (size_t)groups * std::min(n4, kThreads) * 16;
  size_t front = align_up(std::max(query_sum_smem(g), qbar_bytes), 128);
  if (job) front = std::max(front, (size_t)2 * kAppendThreads * 8 * sizeof(float));  // the append halves' `part`
  p.sum_off = (uint32_t)front;
  size_t smem = front + 2 * (size_t)p.half_pages * row_bytes;
  if (p.keys_in_smem) smem = std::max(smem, align_up((size_t)p.n_cand, 4) * sizeof(uint32_t));
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  // the default dynamic limit is 48 KB minus the static shared memory: always opt in
  static size_t smem_set[2][2][kMaxDevices] = {};
  {
    cudaError_t e = set_smem_limit(fn, smem, smem_set[job ? 1 : 0][bf16]);
    if (e != cudaSuccess) return e;
  }
  // one CTA per SM always fits (<= 200 KB of shared memory, 512 threads); a grid that
  // could not be co-resident is refused by the cooperative launch itself
  void* args[] = {&p, &fa};
  cudaError_t e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), args, smem, st);
  count_launches(1);
  return e;
}

}  // namespace oomb
