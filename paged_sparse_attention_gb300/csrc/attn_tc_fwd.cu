// tcgen05 chunk-attention forward (bf16 in, fp32 accumulate; head_dim 128, page 128).
//
// Paged sparse attention of one query chunk ("Out of the Memory Barrier",
// gist.science explainer 2.D): query head hq attends to every key of the pages
// selected for its KV head hq/G that precede it causally; O and the natural-log
// LSE are written.
//
// One CTA per (query head, pair of 128-row query tiles A = 2u, B = 2u + 1).  A
// tile's rows are exactly the tokens of the chunk's own page t, so its selected
// pages are a prefix of the ascending selection: every entry <= t's page, the last
// one being the diagonal page (causal mask key <= row).  Tile B's pages are A's
// plus B's own diagonal page.  Both tiles share every K and V tile loaded.  CTAs
// are ordered heaviest pair first.
//
// Warp roles (320 threads):
//   warp 0     TMA producer: both Q tiles once, then each selected page's K tile
//              (3-stage ring, freed once both S tiles have read it) and V tile
//              (2-stage ring, freed after both PV), gathered through the page table.
//   warp 1     TMEM owner + MMA issuer.  Per page j the tensor core runs
//              PV_A(j-1), S_A(j), PV_B(j-1), S_B(j): while the softmax of one tile
//              works, the tensor core computes the other tile's products, so each
//              softmax has the time of two MMAs before its PV is due.
//              S = Q K^T into the tile's S columns; O += P V with P (bf16, written
//              over S by the softmax) read from TMEM.
//   warps 2-5  softmax of tile A, warps 6-9 softmax of tile B: one thread per query
//              row holding all 128 key columns.  Base-2 online softmax with lazy
//              rescaling of O (only when the row max grows by more than 2^8).
// The MMA issuer commits only "S_X(j) ready" per page (its tensor-pipe queue is a few
// instructions deep, so every extra commit or wait between groups idles the pipe).
// MMAs complete in issue order, so a softmax warp that has seen S_X(j) also knows
// that PV_X(j-1) has finished (O may be rescaled) and, when its tile is the last
// user of page j, that K_j and V_{j-1} are free: it releases those ring slots.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
#include "tc_common.cuh"

namespace oomb {
namespace {

using namespace tc;

constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kThreads = 320;
constexpr int kGroupThreads = 128;         // softmax threads of one tile
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct FwdParams {
  const int32_t* sel;
  const int32_t* sel_count;
  const int32_t* table;
  void* o;
  float* lse;
  uint32_t* err;
  int max_sel, n_q, Hq, G, Hkv, num_phys, max_logical, n_tiles, n_pairs;
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
  uint64_t s_full[2];  // per tile: S_j in TMEM
  uint64_t p_full[2];  // per tile: P_j written over S_j (and O rescaled)
  uint64_t o_done[2];  // per tile: its last PV finished
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

constexpr uint32_t kOffQ = 0;                              // tiles A and B
constexpr uint32_t kOffK = 2 * kTileBytes;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffBar = kOffV + kVStages * kTileBytes;
constexpr size_t kSmemBytes = 1024 + kOffBar + sizeof(FwdBarriers);
static_assert(kSmemBytes <= 232448, "shared memory budget");

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
  const int pair = p.n_pairs - 1 - (int)blockIdx.y;  // heaviest pairs first
  const int tA = 2 * pair, tB = 2 * pair + 1;
  const bool hasB = tB < p.n_tiles;
  const int h = hq / p.G;
  const int diagA = (int)(p.q_start / kTile) + tA;
  int count = p.sel_count[h];
  if (count < 0 || count > p.max_sel) {  // flagged by the producer below; never read past the row
    count = count < 0 ? 0 : p.max_sel;
  }
  const int nA = pages_upto(p, h, count, diagA);
  const int nB = hasB ? pages_upto(p, h, count, diagA + 1) : 0;
  const int n = max(nA, nB);  // pages loaded
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
      mbar_init(&bar->p_full[i], kGroupThreads / 32);  // one arrival per softmax warp
      mbar_init(&bar->o_done[i], 1);
    }
    mbar_init(&bar->mma_done, 1);
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
      // the selection must be strictly ascending pages of this chunk's view (the tiles
      // take its prefixes); a count outside [0, max_sel] is flagged too
      const int nvis = (int)((p.q_start + p.n_q + kTile - 1) / kTile);
      const int raw_count = p.sel_count[h];
      if (raw_count < 0 || raw_count > p.max_sel) atomicOr(p.err, OOMB_DEVERR_SEL);
      int prev = -1;
      for (int e = 0; e < count; ++e) {
        const int pe = p.sel[(size_t)h * p.max_sel + e];
        if (pe <= prev || pe >= nvis) {
          atomicOr(p.err, OOMB_DEVERR_SEL);
          break;
        }
        prev = pe;
      }
      mbar_arrive_expect_tx(&bar->q_full, (hasB ? 2u : 1u) * kTileBytes);
      tma_load_3d(sm + kOffQ, &tq, &bar->q_full, 0, hq, tA * kTile);
      tma_load_3d(sm + kOffQ + kHalfBytes, &tq, &bar->q_full, 64, hq, tA * kTile);
      if (hasB) {
        tma_load_3d(sm + kOffQ + kTileBytes, &tq, &bar->q_full, 0, hq, tB * kTile);
        tma_load_3d(sm + kOffQ + kTileBytes + kHalfBytes, &tq, &bar->q_full, 64, hq, tB * kTile);
      }
      // K and V are issued independently, each as soon as its ring has a free slot;
      // the loop gives up after ~2^31 cycles without progress.
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
          if (jk < kKStages || mbar_test_wait(&bar->k_empty[ks], ((jk / kKStages) - 1) & 1)) {
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
          if (jv < kVStages || mbar_test_wait(&bar->v_empty[vs], ((jv / kVStages) - 1) & 1)) {
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
      const int nt[2] = {nA, nB};
      bool ok = mbar_wait(&bar->q_full, 0, p.err, abort);
      // S_X(j) = Q_X K_j^T into the S columns of tile X (the K tile has landed)
      auto issue_s = [&](int x, int j) {
        const uint32_t aQ = smem_u32(sm + kOffQ + x * kTileBytes);
        const uint32_t aK = smem_u32(sm + kOffK + (j % kKStages) * kTileBytes);
        const uint32_t d = tmem + x * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(d, desc_kmajor(aQ, kk), desc_kmajor(aK, kk), idesc_s, kk > 0);
        mma_commit(&bar->s_full[x]);
      };
      // O_X += P_X(j) V_j once the softmax has written P_X(j) (the V tile has landed)
      auto issue_pv = [&](int x, int j) -> bool {
        if (!mbar_wait(&bar->p_full[x], j & 1, p.err, abort)) return false;
        tc_fence_after();
        const uint32_t aV = smem_u32(sm + kOffV + (j % kVStages) * kTileBytes);
        const uint32_t a = tmem + x * 128, o = tmem + 256 + x * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ts(o, a + kk * 8, desc_mnmajor(aV, kk), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        if (j == nt[x] - 1) mma_commit(&bar->o_done[x]);  // the tile's last PV
        return true;
      };
      // page 0: both S
      if (ok) ok = mbar_wait(&bar->k_full[0], 0, p.err, abort);
      if (ok) {
        tc_fence_after();
        for (int x = 0; x < 2; ++x)
          if (0 < nt[x]) issue_s(x, 0);
      }
      for (int j = 0; ok && j < n; ++j) {
        const int j1 = j + 1;
        bool v_waited = false, k_waited = false;
        for (int x = 0; ok && x < 2; ++x) {
          if (j < nt[x]) {  // PV_X(j)
            if (!v_waited) {
              ok = mbar_wait(&bar->v_full[j % kVStages], (j / kVStages) & 1, p.err, abort);
              v_waited = true;
            }
            ok = ok && issue_pv(x, j);
          }
          if (ok && j1 < nt[x]) {  // S_X(j+1)
            if (!k_waited) {
              ok = mbar_wait(&bar->k_full[j1 % kKStages], (j1 / kKStages) & 1, p.err, abort);
              k_waited = true;
              if (ok) tc_fence_after();
            }
            if (ok) issue_s(x, j1);
          }
        }
      }
      // every issued MMA must finish before TMEM is released
      mma_commit(&bar->mma_done);
      mbar_wait(&bar->mma_done, 0, p.err, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int x = (warp - 2) >> 2;  // tile of this warp group (0: A, 1: B)
    const int nx = x == 0 ? nA : nB;
    const int t = x == 0 ? tA : tB;
    const int diag = diagA + x;
    const int q4 = warp & 3;  // TMEM lane quarter
    const int r = q4 * 32 + lane;  // query row in the tile
    const uint32_t lane_off = tmem_lane_base(warp);
    const uint32_t tS = tmem + lane_off + x * 128;
    const uint32_t tO = tmem + lane_off + 256 + x * 128;
    const int qrow = t * kTile + r;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nx; ++j) {
      const int pg = p.sel[(size_t)h * p.max_sel + j];
      if (ok) ok = mbar_wait(&bar->s_full[x], j & 1, p.err, abort);
      ok = __all_sync(0xffffffffu, ok);  // TMEM loads and stores below are warp-collective
      if (!ok) break;
      tc_fence_after();
      // the last user of page j frees K_j and V_{j-1} (their MMAs precede S_X(j))
      if ((warp & 3) == 2 && lane == 0 && (x == 1 || j >= nB)) {
        mbar_arrive(&bar->k_empty[j % kKStages]);
        if (j > 0) mbar_arrive(&bar->v_empty[(j - 1) % kVStages]);
      }
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
      tmem_wait_ld();
      if (pg == diag) {  // causal mask: key column c visible to row r iff c <= r
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > r) sr[c] = 0xff800000u;  // -inf
      }
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = fmaxf(__uint_as_float(sr[k]), __uint_as_float(sr[8 + k]));
#pragma unroll
      for (int c = 16; c < 128; c += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mx[k] = fmax3(mx[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 8 + k]));
      const float tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) *
                         p.scale_log2;
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
      // p = 2^(s * scale_log2 - m) two columns per packed FMA; two packed sum chains
      const uint64_t scale2 = f32x2(p.scale_log2, p.scale_log2), negm2 = f32x2(neg_m, neg_m);
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float t0, t1;
        f32x2_split(ffma2(f32x2(sr[2 * c], sr[2 * c + 1]), scale2, negm2), t0, t1);
        const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
        sum[c & 3] += p0 + p1;
        sr[c] = pack_bf16x2(p0, p1);  // packed P: key columns 2c, 2c+1 -> column c
      }
      l += (sum[0] + sum[1]) + (sum[2] + sum[3]);
      // The rescale is decided per row but the TMEM accesses are warp-collective: the warp
      // rescales when any of its rows needs it, the other rows scale by alpha = 1 (exact).
      if (__any_sync(0xffffffffu, rescale_o)) {  // PV_{j-1} finished before S_j
        if (!rescale_o) alpha = 1.f;
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
      tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar->p_full[x]);
    }
    // epilogue: normalise this thread's row of O
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.o);
    const bool have = x == 0 || hasB;
    if (__all_sync(0xffffffffu, ok && nx > 0 && mbar_wait(&bar->o_done[x], 0, p.err, abort))) {
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
    } else if (have && qrow < p.n_q) {
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
  static size_t smem_set[kMaxDevices] = {};
  cudaError_t e = set_smem_limit((const void*)attn_fwd_tc_kernel, kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
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
  p.n_pairs = (p.n_tiles + 1) / 2;
  p.q_start = a.q_start;
  p.scale_log2 = a.scale * kLog2e;
  p.staged = a.kv.staged;
  p.stage_h0 = a.kv.stage_h0;
  p.stage_stride = a.kv.stage_stride;
  dim3 grid(a.g.Hq, p.n_pairs);
  attn_fwd_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace oomb
