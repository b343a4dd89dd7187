// tcgen05 chunk-attention forward (bf16 in, fp32 accumulate; head_dim 128, page 128).
//
// Paged sparse attention of one query chunk ("Out of the Memory Barrier",
// gist.science explainer 2.D): query head hq attends to every key of the pages
// selected for its KV head hq/G that precede it causally; O and the natural-log
// LSE are written.
//
// One CTA per (query head, 128-row query tile t).  The tile's rows are exactly the
// tokens of the chunk's own page t, so the selected pages split into full pages
// (history and own pages before t), the diagonal page t (causal mask j <= r) and
// pages after t (skipped).
//
// Warp roles (192 threads):
//   warp 0    TMA producer: Q tile once, then each selected page's K and V tile,
//             gathered through the page table (row = (phys * Hkv + h) * 128).
//   warp 1    TMEM owner + MMA issuer: S_j = Q K_j^T into one of two TMEM S buffers,
//             then O += P_j V_j with P_j read from TMEM (bf16 written over S_j).
//   warps 2-5 softmax, thread == query row (TMEM lane): online softmax in base 2
//             with lazy rescaling of O (only when the row max grows by > 2^8),
//             then the epilogue O / l, LSE = (m + log2 l) ln 2.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384).
#include "tc_common.cuh"

namespace oomb {
namespace {

using namespace tc;

constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct FwdParams {
  const int32_t* sel;
  const int32_t* sel_count;
  const int32_t* table;
  void* o;
  float* lse;
  uint32_t* err;
  int max_sel, n_q, Hq, G, Hkv, num_phys, max_logical, n_tiles;
  int64_t q_start;
  float scale_log2;
  int staged, stage_h0, stage_stride;
};

struct __align__(8) FwdBarriers {
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kSmemBytes = 1024 + kTileBytes * (1 + 2 * kStages) + sizeof(FwdBarriers);

__device__ __forceinline__ int next_tile_page(const FwdParams& p, int h, int& s, int count, int diag) {
  // advance s to the next selected page <= diag; returns the page or -1 when done
  while (s < count) {
    const int pg = p.sel[(size_t)h * p.max_sel + s];
    if (pg > diag) return -1;
    if (pg >= 0) return pg;
    ++s;  // negative entries are skipped (flagged by the producer)
  }
  return -1;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm;
  uint8_t* sK = sm + kTileBytes;                       // kStages tiles
  uint8_t* sV = sm + kTileBytes * (1 + kStages);       // kStages tiles
  FwdBarriers* bar = reinterpret_cast<FwdBarriers*>(sm + kTileBytes * (1 + 2 * kStages));

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int hq = blockIdx.x;
  const int t = p.n_tiles - 1 - (int)blockIdx.y;  // heaviest tiles first
  const int h = hq / p.G;
  const int diag = (int)(p.q_start / kTile) + t;
  const int count = p.sel_count[h];
  volatile int* abort = &bar->abort;

  if (threadIdx.x == 0) {
    mbar_init(&bar->q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar->k_full[i], 1);
      mbar_init(&bar->v_full[i], 1);
      mbar_init(&bar->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_full[i], 128);
    }
    mbar_init(&bar->o_done, 1);
    bar->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bar->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      // every selection entry must name an existing page of this chunk's view
      const int nvis = (int)((p.q_start + p.n_q + kTile - 1) / kTile);
      for (int e = 0; e < count; ++e) {
        const int pe = p.sel[(size_t)h * p.max_sel + e];
        if (pe < 0 || pe >= nvis) {
          atomicOr(p.err, OOMB_DEVERR_SEL);
          break;
        }
      }
      mbar_arrive_expect_tx(&bar->q_full, kTileBytes);
      tma_load_3d(sQ, &tq, &bar->q_full, 0, hq, t * kTile);
      tma_load_3d(sQ + kHalfBytes, &tq, &bar->q_full, 64, hq, t * kTile);
      int s = 0, j = 0;
      for (int pg; (pg = next_tile_page(p, h, s, count, diag)) >= 0; ++s, ++j) {
        const int st = j % kStages;
        if (j >= kStages && !mbar_wait(&bar->kv_empty[st], ((j / kStages) - 1) & 1, p.err, abort)) break;
        int64_t blk;
        if (p.staged) {
          blk = (int64_t)(p.stage_h0 + h) * p.stage_stride + s;
        } else {
          int phys = (pg < p.max_logical) ? p.table[pg] : -1;
          if (phys < 0 || phys >= p.num_phys) {
            atomicOr(p.err, OOMB_DEVERR_PAGE);
            phys = 0;  // keep the pipeline consistent; the result is flagged as invalid
          }
          blk = (int64_t)phys * p.Hkv + h;
        }
        const int row = (int)(blk * kTile);
        mbar_arrive_expect_tx(&bar->k_full[st], kTileBytes);
        tma_load_2d(sK + st * kTileBytes, &tk, &bar->k_full[st], 0, row);
        tma_load_2d(sK + st * kTileBytes + kHalfBytes, &tk, &bar->k_full[st], 64, row);
        mbar_arrive_expect_tx(&bar->v_full[st], kTileBytes);
        tma_load_2d(sV + st * kTileBytes, &tv, &bar->v_full[st], 0, row);
        tma_load_2d(sV + st * kTileBytes + kHalfBytes, &tv, &bar->v_full[st], 64, row);
      }
      // drain: every armed stage must have landed before the CTA may exit
      const int n = j;
      for (int jj = (n > kStages ? n - kStages : 0); jj < n; ++jj) {
        const int st = jj % kStages;
        mbar_wait(&bar->k_full[st], (jj / kStages) & 1, p.err, nullptr);
        mbar_wait(&bar->v_full[st], (jj / kStages) & 1, p.err, nullptr);
      }
      mbar_wait(&bar->q_full, 0, p.err, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      const uint32_t idesc_o = idesc_bf16_f32(128, 128, false, true);
      const uint32_t tS[2] = {tmem, tmem + 128};
      const uint32_t tO = tmem + 256;
      const uint32_t aQ = smem_u32(sQ);
      bool ok = mbar_wait(&bar->q_full, 0, p.err, abort);
      int s = 0, j = 0;
      while (ok && next_tile_page(p, h, s, count, diag) >= 0) {
        const int st = j % kStages;
        if (!mbar_wait(&bar->k_full[st], (j / kStages) & 1, p.err, abort)) { ok = false; break; }
        tc_fence_after();
        const uint32_t aK = smem_u32(sK + st * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tS[j & 1], desc_kmajor(aQ, kk), desc_kmajor(aK, kk), idesc_s, kk > 0);
        mma_commit(&bar->s_full[j & 1]);
        if (j > 0) {
          const int jp = j - 1, stp = jp % kStages;
          if (!mbar_wait(&bar->p_full[jp & 1], (jp >> 1) & 1, p.err, abort)) { ok = false; break; }
          if (!mbar_wait(&bar->v_full[stp], (jp / kStages) & 1, p.err, abort)) { ok = false; break; }
          tc_fence_after();
          const uint32_t aV = smem_u32(sV + stp * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tO, tS[jp & 1] + kk * 8, desc_mnmajor(aV, kk), idesc_o, (jp > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar->kv_empty[stp]);
          mma_commit(&bar->o_done);
        }
        ++s;
        ++j;
      }
      if (ok && j > 0) {
        const int jp = j - 1, stp = jp % kStages;
        if (mbar_wait(&bar->p_full[jp & 1], (jp >> 1) & 1, p.err, abort) &&
            mbar_wait(&bar->v_full[stp], (jp / kStages) & 1, p.err, abort)) {
          tc_fence_after();
          const uint32_t aV = smem_u32(sV + stp * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tO, tS[jp & 1] + kk * 8, desc_mnmajor(aV, kk), idesc_o, (jp > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar->kv_empty[stp]);
          mma_commit(&bar->o_done);
        }
      }
      // all issued MMAs must finish before TMEM is released: wait for the last commit
      if (j > 0) mbar_wait(&bar->o_done, (j - 1) & 1, p.err, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int r = (warp & 3) * 32 + lane;  // TMEM lane == query row in the tile
    const uint32_t lane_off = tmem_lane_base(warp);
    const int qrow = t * kTile + r;
    float m = -INFINITY, l = 0.f;
    int s = 0, j = 0;
    bool ok = true;
    for (int pg; (pg = next_tile_page(p, h, s, count, diag)) >= 0; ++s, ++j) {
      const int b = j & 1;
      if (!mbar_wait(&bar->s_full[b], (j >> 1) & 1, p.err, abort)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[128];
      {
        uint32_t (&c0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
        uint32_t (&c1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
        uint32_t (&c2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[64]);
        uint32_t (&c3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[96]);
        tmem_ld32(tmem + lane_off + b * 128 + 0, c0);
        tmem_ld32(tmem + lane_off + b * 128 + 32, c1);
        tmem_ld32(tmem + lane_off + b * 128 + 64, c2);
        tmem_ld32(tmem + lane_off + b * 128 + 96, c3);
        tmem_wait_ld();
      }
      const bool diag_tile = (pg == diag);
      float x[128];
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        float v = __uint_as_float(sr[c]) * p.scale_log2;
        if (diag_tile && c > r) v = -INFINITY;
        x[c] = v;
        tmax = fmaxf(tmax, v);
      }
      bool rescale_o = false;
      float alpha = 1.f;
      if (tmax > m + kRescaleThreshold || (m == -INFINITY && tmax > -INFINITY)) {
        const float m_new = fmaxf(m, tmax);
        alpha = exp2f(m - m_new);  // 0 when m == -inf
        rescale_o = (j > 0) && (m > -INFINITY);
        l *= alpha;
        m = m_new;
      }
      float rowsum = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = exp2f(x[2 * c] - m), p1 = exp2f(x[2 * c + 1] - m);
        rowsum += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l += rowsum;
      if (j > 0) {
        if (!mbar_wait(&bar->o_done, (j - 1) & 1, p.err, abort)) { ok = false; break; }
        tc_fence_after();
      }
      if (rescale_o) {
        const uint32_t tO = tmem + lane_off + 256;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + cc * 32, o);
        }
      }
      {
        uint32_t (&p0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[0]);
        uint32_t (&p1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[32]);
        tmem_st32(tmem + lane_off + b * 128 + 0, p0);
        tmem_st32(tmem + lane_off + b * 128 + 32, p1);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar->p_full[b]);
    }
    // epilogue
    const int n = j;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.o);
    if (ok && n > 0 && mbar_wait(&bar->o_done, (n - 1) & 1, p.err, abort)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const uint32_t tO = tmem + lane_off + 256;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_wait_ld();
        if (qrow < p.n_q) {
          uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)qrow * p.Hq + hq) * kD + cc * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
            dst[v] = w;
          }
        }
      }
      if (qrow < p.n_q) p.lse[(size_t)hq * p.n_q + qrow] = (m + log2f(l)) * kLn2;
    } else if (qrow < p.n_q) {
      uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)qrow * p.Hq + hq) * kD);
      for (int v = 0; v < 16; ++v) dst[v] = make_uint4(0, 0, 0, 0);
      p.lse[(size_t)hq * p.n_q + qrow] = -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool tc_supported(const Geometry& g) { return g.dtype == OOMB_BF16 && g.d == kD && g.P == kTile; }

cudaError_t launch_attn_fwd_tc(const AttnArgs& a, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap tq, tk, tv;
  if (!make_tmap_heads(&tq, a.q, a.n_q, a.g.Hq) || !make_tmap_rows(&tk, a.kv.k, kv_rows(a)) ||
      !make_tmap_rows(&tv, a.kv.v, kv_rows(a)))
    return cudaErrorInvalidValue;
  FwdParams p;
  p.sel = a.sel;
  p.sel_count = a.sel_count;
  p.table = a.kv.table;
  p.o = a.o_out;
  p.lse = a.lse_out;
  p.err = a.err;
  p.max_sel = a.max_sel;
  p.n_q = a.n_q;
  p.Hq = a.g.Hq;
  p.G = a.g.G;
  p.Hkv = a.g.Hkv;
  p.num_phys = a.g.num_phys;
  p.max_logical = a.g.max_logical;
  p.n_tiles = (a.n_q + kTile - 1) / kTile;
  p.q_start = a.q_start;
  p.scale_log2 = a.scale * kLog2e;
  p.staged = a.kv.staged;
  p.stage_h0 = a.kv.stage_h0;
  p.stage_stride = a.kv.stage_stride;
  dim3 grid(a.g.Hq, p.n_tiles);
  attn_fwd_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace oomb
