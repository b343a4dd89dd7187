// tcgen05 chunk-attention forward (bf16 in, fp32 accumulate; head_dim 128, page 128).
//
// Paged sparse attention of one query chunk ("Out of the Memory Barrier",
// gist.science explainer 2.D): query head hq attends to every key of the pages
// selected for its KV head hq/G that precede it causally; O and the natural-log
// LSE are written.
//
// A 128-row query tile t holds exactly the tokens of the chunk's own page t, so its
// selected pages are: full pages (history and own pages before t), the diagonal
// page t (causal mask key <= row) and pages after t (skipped).
//
// One CTA per (query head, tile pair {t, n-1-t}): the earlier tile A and the later
// tile B share every page A sees, so each shared K/V page is loaded once for both,
// and the pair's causal work is the same for every t.  With an odd tile count the
// middle tile runs alone as B.
//
// Warp roles (320 threads):
//   warp 0     TMA producer: both Q tiles once, then each page's K (3-stage ring)
//              and V (2-stage ring), gathered through the page table.
//   warp 1     TMEM owner + MMA issuer, ping-pong between the tiles,
//                S_A(0) S_B(0) | PV_A(0) S_A(1) | PV_B(0) S_B(1) | PV_A(1) S_A(2) ...
//              so one tile's MMAs run while the other tile's softmax does.  P is
//              written back over S as bf16 and read from TMEM as the A operand.
//              On the pages only B sees, B double-buffers S in both S regions.
//   warps 2-5  softmax of tile A, warps 6-9 softmax of tile B; thread == query row
//              (TMEM lane): base-2 online softmax with lazy rescaling of O (only when
//              the row max grows by more than 2^8); epilogue O / l and
//              LSE = (m + log2 l) ln 2.
// TMEM columns: S region 0 [0,128) (A), S region 1 [128,256) (B), O_A [256,384),
// O_B [384,512).
#include "tc_common.cuh"

namespace oomb {
namespace {

using namespace tc;

constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kThreads = 320;
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
  uint64_t k_full[kKStages];
  uint64_t k_empty[kKStages];
  uint64_t v_full[kVStages];
  uint64_t v_empty[kVStages];
  uint64_t s_full[2];  // per S region
  uint64_t p_full[2];  // per tile
  uint64_t o_done[2];  // per tile
  uint32_t tmem_base;
  int abort;
};

constexpr uint32_t kOffQ = 0;  // Q_A, Q_B
constexpr uint32_t kOffK = 2 * kTileBytes;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffBar = kOffV + kVStages * kTileBytes;
constexpr size_t kSmemBytes = 1024 + kOffBar + sizeof(FwdBarriers);

// Leading selection entries (ascending pages) that are <= diag.  A negative entry
// is invalid (flagged by the producer) and ends the list.
__device__ __forceinline__ int pages_upto(const FwdParams& p, int h, int count, int diag) {
  int n = 0;
  while (n < count) {
    const int pg = p.sel[(size_t)h * p.max_sel + n];
    if (pg < 0 || pg > diag) break;
    ++n;
  }
  return n;
}

// S region used by `tile` at page step j, and how many earlier S results that region
// has received (its mbarrier phase): A always uses region 0; B uses region 1 while A
// is active and alternates regions 1, 0, 1, ... on the pages only B sees.
__device__ __forceinline__ int s_region(int tile, int j, int nA) {
  if (tile == 0 || j < nA) return tile;
  return ((j - nA) & 1) ? 0 : 1;
}
__device__ __forceinline__ int s_use(int tile, int j, int nA) {
  if (tile == 0 || j < nA) return j;
  return nA + ((j - nA) >> 1);  // region 1 had nA uses by B, region 0 nA uses by A
}

__device__ void softmax_tile(const FwdParams& p, FwdBarriers* bar, uint32_t tmem, int tile, int n, int nA,
                             int t, int diag, int hq, int h, int warp, int lane, volatile int* abort) {
  const int r = (warp & 3) * 32 + lane;  // TMEM lane == query row in the tile
  const uint32_t lane_off = tmem_lane_base(warp);
  const uint32_t tO = tmem + lane_off + 256 + tile * 128;
  const int qrow = t * kTile + r;
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int j = 0; j < n; ++j) {
    const int pg = p.sel[(size_t)h * p.max_sel + j];
    const int reg = s_region(tile, j, nA);
    if (!mbar_wait(&bar->s_full[reg], s_use(tile, j, nA) & 1, p.err, abort)) { ok = false; break; }
    tc_fence_after();
    const uint32_t tS = tmem + lane_off + reg * 128;
    uint32_t sr[128];
    tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
    tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
    tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
    tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
    tmem_wait_ld();
    if (pg == diag) {  // causal mask on the diagonal page: key c visible to row r iff c <= r
#pragma unroll
      for (int c = 0; c < 128; ++c)
        if (c > r) sr[c] = 0xff800000u;  // -inf
    }
    // row max of the raw logits (scale > 0 commutes with max); 8 independent chains
    float mx[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) mx[k] = __uint_as_float(sr[k]);
#pragma unroll
    for (int c = 8; c < 128; c += 8)
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], __uint_as_float(sr[c + k]));
    const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * p.scale_log2;
    bool rescale_o = false;
    float alpha = 1.f;
    if (tmax > m + kRescaleThreshold || (m == -INFINITY && tmax > -INFINITY)) {
      const float m_new = fmaxf(m, tmax);
      alpha = exp2f(m - m_new);  // 0 when m == -inf
      rescale_o = (j > 0) && (m > -INFINITY);
      l *= alpha;
      m = m_new;
    }
    // p = 2^(s * scale * log2e - m), one FFMA + one ex2 per element; 8 partial sums
    const float neg_m = (m == -INFINITY) ? 0.f : -m;
    float sum[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) sum[k] = 0.f;
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      const float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * c]), p.scale_log2, neg_m));
      const float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * c + 1]), p.scale_log2, neg_m));
      sum[c & 7] += p0 + p1;
      sr[c] = pack_bf16x2(p0, p1);  // packed P overwrites the consumed front of the row
    }
    l += ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
    if (j > 0) {  // PV of the previous page is done: O may be rescaled
      if (!mbar_wait(&bar->o_done[tile], (j - 1) & 1, p.err, abort)) { ok = false; break; }
      tc_fence_after();
    }
    if (rescale_o) {
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st32(tO + cc * 32, o);
      }
    }
    tmem_st32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
    tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bar->p_full[tile]);
  }
  // epilogue
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.o);
  if (ok && n > 0 && mbar_wait(&bar->o_done[tile], (n - 1) & 1, p.err, abort)) {
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
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

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBarriers* bar = reinterpret_cast<FwdBarriers*>(sm + kOffBar);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int hq = blockIdx.x;
  const int pair = blockIdx.y;
  const int tA = pair, tB = p.n_tiles - 1 - pair;  // tA <= tB; equal: a single tile (B)
  const bool hasA = tA < tB;
  const int h = hq / p.G;
  const int first_own = (int)(p.q_start / kTile);
  const int diagA = first_own + tA, diagB = first_own + tB;
  const int count = p.sel_count[h];
  const int nB = pages_upto(p, h, count, diagB);
  const int nA = hasA ? pages_upto(p, h, nB, diagA) : 0;
  volatile int* abort = &bar->abort;

  if (threadIdx.x == 0) {
    mbar_init(&bar->q_full, 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bar->k_full[i], 1);
      mbar_init(&bar->k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bar->v_full[i], 1);
      mbar_init(&bar->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_full[i], 128);
      mbar_init(&bar->o_done[i], 1);
    }
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
      mbar_arrive_expect_tx(&bar->q_full, (hasA ? 2 : 1) * kTileBytes);
      if (hasA) {
        tma_load_3d(sm + kOffQ, &tq, &bar->q_full, 0, hq, tA * kTile);
        tma_load_3d(sm + kOffQ + kHalfBytes, &tq, &bar->q_full, 64, hq, tA * kTile);
      }
      tma_load_3d(sm + kOffQ + kTileBytes, &tq, &bar->q_full, 0, hq, tB * kTile);
      tma_load_3d(sm + kOffQ + kTileBytes + kHalfBytes, &tq, &bar->q_full, 64, hq, tB * kTile);
      int jk = 0, jv = 0;
      bool ok = true;
      for (int j = 0; ok && j < nB; ++j) {
        const int pg = p.sel[(size_t)h * p.max_sel + j];
        int64_t blk;
        if (p.staged) {
          blk = (int64_t)(p.stage_h0 + h) * p.stage_stride + j;
        } else {
          int phys = (pg < p.max_logical) ? p.table[pg] : -1;
          if (phys < 0 || phys >= p.num_phys) {
            atomicOr(p.err, OOMB_DEVERR_PAGE);
            phys = 0;  // keep the pipeline consistent; the result is flagged as invalid
          }
          blk = (int64_t)phys * p.Hkv + h;
        }
        const int row = (int)(blk * kTile);
        const int ks = j % kKStages, vs = j % kVStages;
        if (j >= kKStages && !(ok = mbar_wait(&bar->k_empty[ks], ((j / kKStages) - 1) & 1, p.err, abort))) break;
        mbar_arrive_expect_tx(&bar->k_full[ks], kTileBytes);
        tma_load_2d(sm + kOffK + ks * kTileBytes, &tk, &bar->k_full[ks], 0, row);
        tma_load_2d(sm + kOffK + ks * kTileBytes + kHalfBytes, &tk, &bar->k_full[ks], 64, row);
        jk = j + 1;
        if (j >= kVStages && !(ok = mbar_wait(&bar->v_empty[vs], ((j / kVStages) - 1) & 1, p.err, abort))) break;
        mbar_arrive_expect_tx(&bar->v_full[vs], kTileBytes);
        tma_load_2d(sm + kOffV + vs * kTileBytes, &tv, &bar->v_full[vs], 0, row);
        tma_load_2d(sm + kOffV + vs * kTileBytes + kHalfBytes, &tv, &bar->v_full[vs], 64, row);
        jv = j + 1;
      }
      // drain: every armed stage must have landed before the CTA may exit
      for (int jj = (jk > kKStages ? jk - kKStages : 0); jj < jk; ++jj)
        mbar_wait(&bar->k_full[jj % kKStages], (jj / kKStages) & 1, p.err, nullptr);
      for (int jj = (jv > kVStages ? jv - kVStages : 0); jj < jv; ++jj)
        mbar_wait(&bar->v_full[jj % kVStages], (jj / kVStages) & 1, p.err, nullptr);
      mbar_wait(&bar->q_full, 0, p.err, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nB > 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      const uint32_t idesc_o = idesc_bf16_f32(128, 128, false, true);
      const uint32_t aQ0 = smem_u32(sm + kOffQ), aQ1 = smem_u32(sm + kOffQ + kTileBytes);
      bool ok = mbar_wait(&bar->q_full, 0, p.err, abort);
      // S = Q_tile K_j^T into the tile's S region for step j
      auto issue_s = [&](int tile, int j) -> bool {
        const int ks = j % kKStages;
        if (!mbar_wait(&bar->k_full[ks], (j / kKStages) & 1, p.err, abort)) return false;
        tc_fence_after();
        const uint32_t aK = smem_u32(sm + kOffK + ks * kTileBytes);
        const int reg = s_region(tile, j, nA);
        const uint32_t aQ = tile == 0 ? aQ0 : aQ1;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tmem + reg * 128, desc_kmajor(aQ, kk), desc_kmajor(aK, kk), idesc_s, kk > 0);
        mma_commit(&bar->s_full[reg]);
        if (tile == 1) mma_commit(&bar->k_empty[ks]);  // B is the last reader of K_j
        return true;
      };
      // O_tile += P_tile(j) V_j once the tile's softmax of step j is done
      auto issue_pv = [&](int tile, int j) -> bool {
        const int vs = j % kVStages;
        if (!mbar_wait(&bar->p_full[tile], j & 1, p.err, abort)) return false;
        if (!mbar_wait(&bar->v_full[vs], (j / kVStages) & 1, p.err, abort)) return false;
        tc_fence_after();
        const uint32_t aV = smem_u32(sm + kOffV + vs * kTileBytes);
        const uint32_t a = tmem + s_region(tile, j, nA) * 128;
        const uint32_t d = tmem + 256 + tile * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ts(d, a + kk * 8, desc_mnmajor(aV, kk), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar->o_done[tile]);
        if (tile == 1) mma_commit(&bar->v_empty[vs]);  // B is the last reader of V_j
        return true;
      };
      int nextB = 0;  // next B step whose S is still to be issued
      if (ok && nA > 0) ok = issue_s(0, 0);
      if (ok) ok = issue_s(1, nextB++);
      if (ok && nA == 0 && nB > 1) ok = issue_s(1, nextB++);  // B alone: run one page ahead
      for (int j = 0; ok && j < nB; ++j) {
        if (j < nA) {
          ok = issue_pv(0, j);
          if (ok && j + 1 < nA) ok = issue_s(0, j + 1);
          if (!ok) break;
        }
        ok = issue_pv(1, j);
        if (!ok) break;
        // B's S results that may now be issued: the next one while A shares the
        // pipeline, up to two ahead once only B is left (double buffering)
        const int limit = (j + 1 < nA) ? j + 1 : j + 2;
        while (ok && nextB <= limit && nextB < nB) ok = issue_s(1, nextB++);
      }
      // every issued MMA must finish before TMEM is released
      if (nA > 0) mbar_wait(&bar->o_done[0], (nA - 1) & 1, p.err, nullptr);
      mbar_wait(&bar->o_done[1], (nB - 1) & 1, p.err, nullptr);
    }
  } else if (warp < 6) {
    if (hasA) softmax_tile(p, bar, tmem, 0, nA, nA, tA, diagA, hq, h, warp, lane, abort);
  } else {
    softmax_tile(p, bar, tmem, 1, nB, nA, tB, diagB, hq, h, warp, lane, abort);
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
  dim3 grid(a.g.Hq, (p.n_tiles + 1) / 2);
  attn_fwd_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace oomb
