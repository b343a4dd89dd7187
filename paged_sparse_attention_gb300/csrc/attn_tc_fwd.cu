// tcgen05 chunk-attention forward (bf16 in, fp32 accumulate; head_dim 128, page 128).
//
// Paged sparse attention of one query chunk ("Out of the Memory Barrier",
// gist.science explainer 2.D): query head hq attends to every key of the pages
// selected for its KV head hq/G that precede it causally; O and the natural-log
// LSE are written.
//
// One CTA per (query head, 128-row query tile t).  The tile's rows are exactly the
// tokens of the chunk's own page t, so its selected pages split into full pages
// (history and own pages before t), the diagonal page t (causal mask key <= row)
// and pages after t (skipped).  CTAs are ordered heaviest tile first.
//
// Warp roles (320 threads):
//   warp 0     TMA producer: Q once, then each selected page's K tile (4-stage
//              ring, freed as soon as S has read it) and V tile (2-stage ring,
//              freed after PV), gathered through the page table.
//   warp 1     TMEM owner + MMA issuer: S_j = Q K_j^T into one of two TMEM S
//              buffers -- S_{j+1} is computed while the softmax works on S_j --
//              then O += P_j V_j with P_j (bf16, written over S_j) read from TMEM.
//   warps 2-9  softmax: two warps per TMEM lane quarter, each owning 64 of the 128
//              key columns of its 32 query rows; the pair exchanges its partial row
//              max through shared memory.  Base-2 online softmax with lazy
//              rescaling of O (only when the row max grows by more than 2^8); each
//              thread rescales and finally normalises its 64 columns of O.
// TMEM columns: S0 [0,128), S1 [128,256), O [256,384).
#include "tc_common.cuh"

namespace oomb {
namespace {

using namespace tc;

constexpr int kKStages = 4;
constexpr int kVStages = 2;
constexpr int kThreads = 320;
constexpr int kSoftmaxThreads = 256;
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
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done;
  uint32_t tmem_base;
  int abort;
  float xchg[2][128];  // [column half][row]: partial row maxima, then (epilogue) partial row sums
};

constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kTileBytes;
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

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdBarriers* bar = reinterpret_cast<FwdBarriers*>(sm + kOffBar);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int hq = blockIdx.x;
  const int t = p.n_tiles - 1 - (int)blockIdx.y;  // heaviest tiles first
  const int h = hq / p.G;
  const int diag = (int)(p.q_start / kTile) + t;
  const int count = p.sel_count[h];
  const int n = pages_upto(p, h, count, diag);  // pages this tile attends to
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
      mbar_init(&bar->p_full[i], kSoftmaxThreads);
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
      tma_load_3d(sm + kOffQ, &tq, &bar->q_full, 0, hq, t * kTile);
      tma_load_3d(sm + kOffQ + kHalfBytes, &tq, &bar->q_full, 64, hq, t * kTile);
      // K and V are issued independently, each as soon as its ring has a free slot
      // (K runs up to kKStages pages ahead, V up to kVStages); the loop gives up after
      // ~2^31 cycles without progress.
      auto block_of = [&](int j) -> int64_t {
        if (p.staged) return (int64_t)(p.stage_h0 + h) * p.stage_stride + j;
        const int pg = p.sel[(size_t)h * p.max_sel + j];
        int phys = (pg >= 0 && pg < p.max_logical) ? p.table[pg] : -1;
        if (phys < 0 || phys >= p.num_phys) {
          atomicOr(p.err, OOMB_DEVERR_PAGE);
          phys = 0;  // keep the pipeline consistent; the result is flagged as invalid
        }
        return (int64_t)phys * p.Hkv + h;
      };
      int jk = 0, jv = 0;
      long long last = clock64();
      while (jk < n || jv < n) {
        bool progressed = false;
        if (jk < n) {
          const int ks = jk % kKStages;
          if (jk < kKStages || mbar_try_wait(&bar->k_empty[ks], ((jk / kKStages) - 1) & 1)) {
            const int row = (int)(block_of(jk) * kTile);
            mbar_arrive_expect_tx(&bar->k_full[ks], kTileBytes);
            tma_load_2d(sm + kOffK + ks * kTileBytes, &tk, &bar->k_full[ks], 0, row);
            tma_load_2d(sm + kOffK + ks * kTileBytes + kHalfBytes, &tk, &bar->k_full[ks], 64, row);
            ++jk;
            progressed = true;
          }
        }
        if (jv < jk) {
          const int vs = jv % kVStages;
          if (jv < kVStages || mbar_try_wait(&bar->v_empty[vs], ((jv / kVStages) - 1) & 1)) {
            const int row = (int)(block_of(jv) * kTile);
            mbar_arrive_expect_tx(&bar->v_full[vs], kTileBytes);
            tma_load_2d(sm + kOffV + vs * kTileBytes, &tv, &bar->v_full[vs], 0, row);
            tma_load_2d(sm + kOffV + vs * kTileBytes + kHalfBytes, &tv, &bar->v_full[vs], 64, row);
            ++jv;
            progressed = true;
          }
        }
        if (progressed) {
          last = clock64();
        } else if (*abort) {
          break;
        } else if (clock64() - last > (1ll << 31)) {
          atomicOr(p.err, kErrMbarTimeout);
          *abort = 1;
          break;
        }
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
    if (lane == 0 && n > 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      const uint32_t idesc_o = idesc_bf16_f32(128, 128, false, true);
      const uint32_t aQ = smem_u32(sm + kOffQ);
      const uint32_t tO = tmem + 256;
      auto issue_s = [&](int j) -> bool {
        const int ks = j % kKStages;
        if (!mbar_wait(&bar->k_full[ks], (j / kKStages) & 1, p.err, abort)) return false;
        tc_fence_after();
        const uint32_t aK = smem_u32(sm + kOffK + ks * kTileBytes);
        const uint32_t d = tmem + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(d, desc_kmajor(aQ, kk), desc_kmajor(aK, kk), idesc_s, kk > 0);
        mma_commit(&bar->s_full[j & 1]);
        mma_commit(&bar->k_empty[ks]);
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int vs = j % kVStages;
        if (!mbar_wait(&bar->p_full[j & 1], (j >> 1) & 1, p.err, abort)) return false;
        if (!mbar_wait(&bar->v_full[vs], (j / kVStages) & 1, p.err, abort)) return false;
        tc_fence_after();
        const uint32_t aV = smem_u32(sm + kOffV + vs * kTileBytes);
        const uint32_t a = tmem + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tO, a + kk * 8, desc_mnmajor(aV, kk), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar->v_empty[vs]);
        mma_commit(&bar->o_done);
        return true;
      };
      bool ok = mbar_wait(&bar->q_full, 0, p.err, abort) && issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) ok = issue_s(j + 1);  // S_{j+1} while the softmax works on S_j
        if (ok) ok = issue_pv(j);
      }
      // every issued MMA must finish before TMEM is released
      mbar_wait(&bar->o_done, (n - 1) & 1, p.err, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int q4 = warp & 3;               // TMEM lane quarter
    const int hc = (warp - 2) >> 2;        // which 64 key columns (and O columns) this warp owns
    const int r = q4 * 32 + lane;          // query row in the tile
    const uint32_t lane_off = tmem_lane_base(warp);
    const uint32_t tO = tmem + lane_off + 256 + hc * 64;
    const int qrow = t * kTile + r;
    const int bar_id = 1 + q4;             // named barrier of the two warps sharing this quarter
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // On an abort every thread still runs all named barriers (only the work is skipped),
    // so the two warps of a pair can never wait on each other forever.
    for (int j = 0; j < n; ++j) {
      const int pg = p.sel[(size_t)h * p.max_sel + j];
      const int b = j & 1;
      const uint32_t tS = tmem + lane_off + b * 128;
      uint32_t sr[64];
      float my_max = -INFINITY;
      if (ok) ok = mbar_wait(&bar->s_full[b], (j >> 1) & 1, p.err, abort);
      ok = __all_sync(0xffffffffu, ok);  // TMEM loads and stores below are warp-collective
      if (ok) {
        tc_fence_after();
        tmem_ld32(tS + hc * 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tS + hc * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_wait_ld();
        if (pg == diag) {  // causal mask: key column c visible to row r iff c <= r
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (hc * 64 + c > r) sr[c] = 0xff800000u;  // -inf
        }
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = __uint_as_float(sr[k]);
#pragma unroll
        for (int c = 8; c < 64; c += 8)
#pragma unroll
          for (int k = 0; k < 8; ++k) mx[k] = fmaxf(mx[k], __uint_as_float(sr[c + k]));
        my_max = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      }
      // exchange the partial maxima; both threads of a row then take the same decisions.
      // The barrier also orders this pair's S reads before either writes P over S.
      bar->xchg[hc][r] = my_max;
      named_bar_sync(bar_id, 64);
      const float tmax = fmaxf(my_max, bar->xchg[hc ^ 1][r]) * p.scale_log2;
      named_bar_sync(bar_id, 64);  // both have read before the slot is reused
      if (!ok) continue;
      bool rescale_o = false;
      float alpha = 1.f;
      if (tmax > m + kRescaleThreshold || (m == -INFINITY && tmax > -INFINITY)) {
        const float m_new = fmaxf(m, tmax);
        alpha = exp2f(m - m_new);  // 0 when m == -inf
        rescale_o = (j > 0) && (m > -INFINITY);
        l *= alpha;
        m = m_new;
      }
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * c]), p.scale_log2, neg_m));
        const float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * c + 1]), p.scale_log2, neg_m));
        sum[c & 3] += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l += (sum[0] + sum[1]) + (sum[2] + sum[3]);
      if (j > 0) {  // PV of the previous page is done: O may be rescaled
        ok = __all_sync(0xffffffffu, mbar_wait(&bar->o_done, (j - 1) & 1, p.err, abort));
        if (!ok) continue;
        tc_fence_after();
      }
      // The rescale is decided per row but the TMEM accesses are warp-collective: the warp
      // rescales when any of its rows needs it, the other rows scale by alpha = 1 (exact).
      if (__any_sync(0xffffffffu, rescale_o)) {
        if (!rescale_o) alpha = 1.f;
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + cc * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + cc * 32, o);
        }
      }
      tmem_st32(tS + hc * 32, pk);  // packed P: key columns 2c, 2c+1 of this half -> column 32 hc + c
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar->p_full[b]);
    }
    // epilogue: combine the pair's partial row sums, normalise this thread's 64 columns of O
    bar->xchg[hc][r] = l;
    named_bar_sync(bar_id, 64);
    const float l_row = l + bar->xchg[hc ^ 1][r];
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.o);
    if (__all_sync(0xffffffffu, ok && n > 0 && mbar_wait(&bar->o_done, (n - 1) & 1, p.err, abort))) {
      tc_fence_after();
      const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_wait_ld();
        if (qrow < p.n_q) {
          uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)qrow * p.Hq + hq) * kD + hc * 64 + cc * 32);
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
      if (qrow < p.n_q && hc == 0) p.lse[(size_t)hq * p.n_q + qrow] = (m + log2f(l_row)) * kLn2;
    } else if (qrow < p.n_q) {
      uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)qrow * p.Hq + hq) * kD + hc * 64);
      for (int v = 0; v < 8; ++v) dst[v] = make_uint4(0, 0, 0, 0);
      if (hc == 0) p.lse[(size_t)hq * p.n_q + qrow] = -INFINITY;
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
