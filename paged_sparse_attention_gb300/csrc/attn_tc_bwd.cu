// tcgen05 chunk-attention backward (bf16 in, fp32 accumulate; head_dim 128, page 128).
//
// "Out of the Memory Barrier" (gist.science explainer): the backward recomputes the
// attention probabilities on the fly (2.A) and accumulates the key/value gradients
// in place in the paged gradient pool that shares the KV page table (2.B).
//
// Kernels of one backward call:
//   bwd_prep     D_i = dO_i . O_i (fp32) and zero the fp32 dQ accumulator
//   bwd_main     one thread-block cluster of n_split CTAs per (selected page, KV
//                head), launched page-major (all KV heads of a page, then the next
//                page; the chunk's own pages, which see fewer query tiles, last): K
//                and V of the page stay in shared memory; the page's steps (every
//                128-row query tile that can see the page, for each of the G query
//                heads of the group) are cut into n_split contiguous ranges, one per
//                CTA, chosen on the host from a model of how the clusters fill the
//                SMs.  A CTA walks its steps in two 64-row halves:
//                  S^T  = K Q_h^T       dP^T = V dO_h^T          (TMEM, fp32)
//                  P^T  = exp2(S^T scale log2e - LSE log2e)     (masked on the diagonal)
//                  dS^T = P^T (dP^T - D)
//                  dV  += P^T dO_h      dK  += dS^T Q_h          (A operands from TMEM)
//                  dQ^T = K^T dS^T      (dS^T also written to shared memory as the B
//                                        operand; dQ^T read out of TMEM and added
//                                        to the fp32 accumulator with global reductions)
//                Epilogue: every CTA stages its partial dV | scale*dK in its own shared
//                memory; CTA r of the cluster then owns key rows [128r/n, 128(r+1)/n):
//                it sums the n partials of those rows in rank order, reading its
//                peers' staging through distributed shared memory, and adds the sum
//                into the page's rows of the fp32 gradient pool.  Every pool row has
//                one writer and a fixed summation order: no atomics on the pool, and
//                dK/dV are the same bits on every run.
//   bwd_convert  dq = bf16(scale * dQ accumulator), token-major.
//
// Warp roles of bwd_main (448 threads):
//   warp 0      TMA producer (K, V once; then a ring of Q/dO half tiles + LSE/D)
//   warp 1      TMEM owner and MMA issuer
//   warps 2-9   softmax: two warps per TMEM lane quarter (thread == key row), each
//               owning 32 of the half tile's 64 query columns; the dK/dV epilogue
//   warps 10-13 dQ read-out: thread == head-dim column (TMEM lane of dQ^T)
// TMEM columns: half a [0,128), half b [128,256): S^T [0,64) dP^T [64,128); after the
// softmax, query columns [32c, 32c+32) hold P^T packed in [32c, 32c+16) and dS^T
// packed in [32c+16, 32c+32), and dQ^T overwrites [64,128); dV [256,384); dK [384,512).
#include <array>
#include <map>
#include <mutex>
#include <queue>
#include <vector>

#include "tc_common.cuh"

namespace oomb {
namespace {

using namespace tc;

constexpr int kRing = 4;  // Q/dO half tiles in flight: the loads come from L2 and need the depth
constexpr int kHalf = 64;
constexpr uint32_t kHalfTile = kHalf * kD * 2;  // 16 KB: one 64-row half tile (two 8 KB boxes)
constexpr uint32_t kHalfBox = kHalfTile / 2;
constexpr int kThreads = 448;
constexpr int kSoftmaxThreads = 256;
constexpr int kMaxCluster = 4;  // CTAs sharing one (page, KV head)
constexpr int kBatch = 4;       // epilogue: pool rows in flight per thread

struct BwdParams {
  const int32_t* sel;
  const int32_t* sel_count;
  const int32_t* table;
  const float* lse2;  // [Hq, n_pad] LSE * log2(e), +inf on padded rows
  const float* Dbuf;  // [Hq, n_pad] rowsum(dO * O), 0 on padded rows
  float* dq_acc;
  float* dk_pool;     // gradient pool, or the gradient staging buffers (grad_staged)
  float* dv_pool;
  uint32_t* err;
  int max_sel, n_q, n_pad, Hq, G, Hkv, num_phys, max_logical, n_tiles;
  int n_split;  // CTAs (one cluster) sharing one (page, KV head): each takes a contiguous range of its steps
  int64_t q_start;
  float scale, scale_log2;
  int staged, stage_h0, stage_stride, grad_staged;
};

struct __align__(8) BwdBarriers {
  uint64_t kv_full;
  uint64_t hs_full[kRing];
  uint64_t hs_empty[kRing];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t dq_full[2];
  uint64_t dq_free[2];
  uint64_t acc_full;
  uint64_t staged;   // one arrival per CTA of the cluster: its partial dK/dV is staged
  uint64_t reduced;  // one arrival per CTA of the cluster: it has read every staging
  uint32_t tmem_base;
  int abort;
};

// shared memory map (offsets from the 1024-aligned base)
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kTileBytes;
constexpr uint32_t kOffRing = kOffV + kTileBytes;                 // kRing x (Q half, dO half)
constexpr uint32_t kOffDS = kOffRing + kRing * 2 * kHalfTile;     // 2 x dS^T half [128 keys][64 q]
constexpr uint32_t kOffVec = kOffDS + 2 * kHalfTile;              // kRing x (lse2[64], D[64])
constexpr uint32_t kOffBar = kOffVec + kRing * 2 * kHalf * 4;
// No alignment slack: the kernel has no static shared memory, and its dynamic window
// starts on a 1 KB boundary (checked at entry; the swizzled tiles need it).
constexpr size_t kSmemBytes = kOffBar + sizeof(BwdBarriers);
static_assert(kSmemBytes <= 232448, "shared memory budget");
// Epilogue staging of a CTA's partial gradients, over the K/V tiles and the ring (all
// MMAs have completed by then): [128 key rows][64 float4] = dV columns (float4 0..31)
// then scale*dK (32..63), float4 c of row j stored at position c ^ (j & 7).
constexpr uint32_t kOffStage = 0;
constexpr uint32_t kStageRow = 2 * kD * 4;  // 1 KB
static_assert(kOffStage + kTile * kStageRow <= kOffDS, "staging must not reach the dS tiles");

__device__ __forceinline__ uint32_t stage_off(int j, int c) {
  return (uint32_t)j * kStageRow + (uint32_t)((c ^ (j & 7)) * 16);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                       const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                       const BwdParams p) {
  // cluster = the n_split CTAs of one (page s, KV head h); page-major order: every KV
  // head of selected page s before page s + 1, so that the lighter own pages run last.
  // Every early return below depends on (s, h) alone, so a cluster leaves as a whole.
  const int part = (int)(blockIdx.x % (unsigned)p.n_split);
  const int r = (int)(blockIdx.x / (unsigned)p.n_split);
  const int h = r % p.Hkv, s = r / p.Hkv;
  const int32_t* row = p.sel + (size_t)h * p.max_sel;
  int count = p.sel_count[h];
  if (count < 0 || count > p.max_sel) {
    if (threadIdx.x == 0 && part == 0 && s == 0) atomicOr(p.err, OOMB_DEVERR_SEL);
    count = count < 0 ? 0 : p.max_sel;
  }
  if (s >= count) return;
  const int first_own = (int)(p.q_start / kTile);
  const int nvis = (int)((p.q_start + p.n_q + kTile - 1) / kTile);
  const int pg = row[s];
  // in range, and strictly above the previous entry and below the next one (so the
  // whole selection is strictly ascending, the order the forward relies on)
  if (pg < 0 || pg >= nvis || pg >= p.max_logical || (s > 0 && row[s - 1] >= pg) ||
      (s + 1 < count && row[s + 1] <= pg)) {
    if (threadIdx.x == 0 && part == 0) atomicOr(p.err, OOMB_DEVERR_SEL);
    return;
  }
  const int phys = p.table[pg];
  if (phys < 0 || phys >= p.num_phys) {
    if (threadIdx.x == 0 && part == 0) atomicOr(p.err, OOMB_DEVERR_PAGE);
    return;
  }
  const int own = pg - first_own;           // >= 0 for the chunk's own pages
  const int t0 = own > 0 ? own : 0;
  // steps (query tile t0 + su / G, query head su % G) for su in [u0, u0 + n_steps); a CTA
  // with no step (fewer steps than CTAs) still stages a zero partial for the reduction
  const int all_steps = (p.n_tiles - t0) * p.G;
  const int u0 = (int)((int64_t)all_steps * part / p.n_split);
  const int n_steps = (int)((int64_t)all_steps * (part + 1) / p.n_split) - u0;

  extern __shared__ uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // uniform over the grid: every CTA leaves here
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.err, OOMB_DEVERR_SMEM);
    return;
  }
  uint8_t* sm = smem_raw;
  BwdBarriers* bar = reinterpret_cast<BwdBarriers*>(sm + kOffBar);
  float* vec = reinterpret_cast<float*>(sm + kOffVec);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  volatile int* abort = &bar->abort;

  if (threadIdx.x == 0) {
    mbar_init(&bar->kv_full, 1);
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bar->hs_full[i], 1);
      mbar_init(&bar->hs_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_full[i], kSoftmaxThreads / 32);  // one arrival per softmax warp
      mbar_init(&bar->dq_full[i], 1);
      mbar_init(&bar->dq_free[i], 4);                    // one arrival per read-out warp
    }
    mbar_init(&bar->acc_full, 1);
    mbar_init(&bar->staged, (uint32_t)p.n_split);
    mbar_init(&bar->reduced, (uint32_t)p.n_split);
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
  // every CTA of the cluster has initialised its barriers once all have arrived here;
  // the epilogue waits for that before its first arrival on a peer's barrier
  cluster_arrive();
  const uint32_t tmem = bar->tmem_base;
  bool ok_acc = n_steps > 0;  // softmax warps: this CTA's dK/dV accumulators are complete

  if (n_steps <= 0) {
    // no step: nothing to load or compute
  } else if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tdo);
      const int64_t blk = p.staged ? (int64_t)(p.stage_h0 + h) * p.stage_stride + s : (int64_t)phys * p.Hkv + h;
      const int row = (int)(blk * kTile);
      mbar_arrive_expect_tx(&bar->kv_full, 2 * kTileBytes);
      tma_load_2d(sm + kOffK, &tk, &bar->kv_full, 0, row);
      tma_load_2d(sm + kOffK + kHalfBytes, &tk, &bar->kv_full, 64, row);
      tma_load_2d(sm + kOffV, &tv, &bar->kv_full, 0, row);
      tma_load_2d(sm + kOffV + kHalfBytes, &tv, &bar->kv_full, 64, row);
    }
    int v = 0;
    if (lane == 0) {
      for (; v < 2 * n_steps; ++v) {
        const int slot = v % kRing;
        if (v >= kRing && !mbar_wait(&bar->hs_empty[slot], ((v / kRing) - 1) & 1, p.err, abort)) break;
        const int su = u0 + (v >> 1), hh = v & 1;
        const int t = t0 + su / p.G, g = su % p.G;
        const int hq = h * p.G + g;
        const int q0 = t * kTile + hh * kHalf;
        uint8_t* dst = sm + kOffRing + slot * 2 * kHalfTile;
        float* vs = vec + slot * 2 * kHalf;
        mbar_arrive_expect_tx(&bar->hs_full[slot], 2 * kHalfTile + 2 * kHalf * 4);
        tma_load_3d(dst, &tq, &bar->hs_full[slot], 0, hq, q0);
        tma_load_3d(dst + kHalfBox, &tq, &bar->hs_full[slot], 64, hq, q0);
        tma_load_3d(dst + kHalfTile, &tdo, &bar->hs_full[slot], 0, hq, q0);
        tma_load_3d(dst + kHalfTile + kHalfBox, &tdo, &bar->hs_full[slot], 64, hq, q0);
        // LSE * log2(e) and D of the 64 rows (padded rows hold +inf and 0)
        bulk_load(vs, p.lse2 + (size_t)hq * p.n_pad + q0, kHalf * 4, &bar->hs_full[slot]);
        bulk_load(vs + kHalf, p.Dbuf + (size_t)hq * p.n_pad + q0, kHalf * 4, &bar->hs_full[slot]);
      }
    }
    if (lane == 0) {  // drain the copies still in flight before the CTA may exit
      for (int vv = (v > kRing ? v - kRing : 0); vv < v; ++vv)
        mbar_wait(&bar->hs_full[vv % kRing], (vv / kRing) & 1, p.err, nullptr);
      mbar_wait(&bar->kv_full, 0, p.err, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 64, false, false);   // S^T, dP^T
      const uint32_t id_acc = idesc_bf16_f32(128, 128, false, true);  // dV, dK (A from TMEM)
      const uint32_t id_dq = idesc_bf16_f32(128, 64, true, true);     // dQ^T
      const uint32_t aK = smem_u32(sm + kOffK), aV = smem_u32(sm + kOffV);
      bool ok = mbar_wait(&bar->kv_full, 0, p.err, abort);
      bool first_acc = true;
      // S^T, dP^T of half-step v = 2u + hh into the half's TMEM region
      auto issue_sdp = [&](int u, int hh) -> bool {
        const int v = 2 * u + hh, slot = v % kRing;
        if (!mbar_wait(&bar->hs_full[slot], (v / kRing) & 1, p.err, abort)) return false;
        if (u > 0 && !mbar_wait(&bar->dq_free[hh], (u - 1) & 1, p.err, abort)) return false;  // dQ^T read out
        tc_fence_after();
        const uint32_t aQ = smem_u32(sm + kOffRing + slot * 2 * kHalfTile);
        const uint32_t adO = aQ + kHalfTile;
        const uint32_t tS = tmem + hh * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss(tS, desc_kmajor(aK, kk), desc_kmajor(aQ, kk, kHalfBox), id_s, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tS + 64, desc_kmajor(aV, kk), desc_kmajor(adO, kk, kHalfBox), id_s, kk > 0);
        mma_commit(&bar->s_full[hh]);
        return true;
      };
      // dQ^T = K^T dS^T, then dV += P^T dO and dK += dS^T Q once the half's softmax is
      // done (dQ^T first, so that its read-out overlaps dV and dK)
      auto issue_acc = [&](int u, int hh) -> bool {
        const int v = 2 * u + hh, slot = v % kRing;
        if (!mbar_wait(&bar->p_full[hh], u & 1, p.err, abort)) return false;
        tc_fence_after();
        const uint32_t aQ = smem_u32(sm + kOffRing + slot * 2 * kHalfTile);
        const uint32_t adO = aQ + kHalfTile;
        const uint32_t tS = tmem + hh * 128;
        const uint32_t adS = smem_u32(sm + kOffDS + hh * kHalfTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tS + 64, desc_mnmajor(aK, kk), desc_mnmajor(adS, kk, kHalfBox), id_dq, kk > 0);
        mma_commit(&bar->dq_full[hh]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // query columns [16 kk, 16 kk + 16): packed P^T / dS^T of column group kk / 2
          const uint32_t a = tS + 32 * (kk >> 1) + 8 * (kk & 1);
          mma_ts(tmem + 256, a, desc_mnmajor(adO, kk, kHalfBox), id_acc, first_acc ? 0u : 1u);
          mma_ts(tmem + 384, a + 16, desc_mnmajor(aQ, kk, kHalfBox), id_acc, first_acc ? 0u : 1u);
          first_acc = false;
        }
        mma_commit(&bar->hs_empty[slot]);
        return true;
      };
      // half b's softmax overlaps the next step's S/dP of half a, and vice versa
      if (ok) ok = issue_sdp(0, 0) && issue_sdp(0, 1);
      for (int u = 0; ok && u < n_steps; ++u) {
        ok = issue_acc(u, 0);
        if (ok && u + 1 < n_steps) ok = issue_sdp(u + 1, 0);
        if (ok) ok = issue_acc(u, 1);
        if (ok && u + 1 < n_steps) ok = issue_sdp(u + 1, 1);
      }
      mma_commit(&bar->acc_full);
      mbar_wait(&bar->acc_full, 0, p.err, nullptr);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------------ softmax
    const int j = (warp & 3) * 32 + lane;  // key row of the page
    const int hc = (warp - 2) >> 2;        // query columns [32 hc, 32 hc + 32) of each half
    const uint32_t lane_off = tmem_lane_base(warp);
    bool ok = true;
    for (int u = 0; ok && u < n_steps; ++u) {
      const int t = t0 + (u0 + u) / p.G;
      const bool diag = (own >= 0) && (t == own);
      for (int hh = 0; hh < 2; ++hh) {
        const int v = 2 * u + hh, slot = v % kRing;
        ok = mbar_wait(&bar->s_full[hh], u & 1, p.err, abort) &&
             mbar_wait(&bar->hs_full[slot], (v / kRing) & 1, p.err, abort);
        ok = __all_sync(0xffffffffu, ok);  // TMEM loads and stores below are warp-collective
        if (!ok) break;
        tc_fence_after();
        const uint32_t base = tmem + lane_off + hh * 128 + 32 * hc;
        uint32_t sr[32], dr[32];
        tmem_ld32(base, sr);
        tmem_ld32(base + 64, dr);
        tmem_wait_ld();
        const float4* vs4 = reinterpret_cast<const float4*>(vec + slot * 2 * kHalf) + 8 * hc;  // lse2, D
        const int qbase = hh * kHalf + 32 * hc;  // query row (within the tile) of this thread's column 0
        const bool masked = diag && (j > qbase);  // some column is in the key's future
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 L = vs4[c4], Dv = vs4[16 + c4];
          const float l4[4] = {L.x, L.y, L.z, L.w}, d4[4] = {Dv.x, Dv.y, Dv.z, Dv.w};
          float pr[4], dsr[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = 4 * c4 + e;
            float pv = ex2_approx(fmaf(__uint_as_float(sr[i]), p.scale_log2, -l4[e]));
            if (masked && j > qbase + i) pv = 0.f;
            pr[e] = pv;
            dsr[e] = pv * (__uint_as_float(dr[i]) - d4[e]);
          }
          pk[2 * c4] = pack_bf16x2(pr[0], pr[1]);
          pk[2 * c4 + 1] = pack_bf16x2(pr[2], pr[3]);
          dk[2 * c4] = pack_bf16x2(dsr[0], dsr[1]);
          dk[2 * c4 + 1] = pack_bf16x2(dsr[2], dsr[3]);
        }
        // P^T and dS^T go over this thread's own (already loaded) S^T columns
        tmem_st16(base, pk);
        tmem_st16(base + 16, dk);
        // dS^T row j, query columns [32 hc, 32 hc + 32): four 16-byte chunks of the swizzled tile
        uint8_t* drow = sm + kOffDS + hh * kHalfTile + j * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int chunk = hc * 4 + c;
          uint4 w = make_uint4(dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
          *reinterpret_cast<uint4*>(drow + ((chunk ^ (j & 7)) * 16)) = w;
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->p_full[hh]);
      }
    }
    ok_acc = ok;
  } else {
    // ------------------------------------------------------------------ dQ read-out
    // Each thread holds one head-dim column of dQ^T for the half's 64 query rows and adds
    // it into the fp32 accumulator with global reductions: for a given row the warp's 32
    // lanes cover 32 consecutive columns (one 128-byte line), and no shared memory is used.
    const int col = (warp & 3) * 32 + lane;  // head-dim column == TMEM lane of dQ^T
    const uint32_t lane_off = tmem_lane_base(warp);
    bool ok = true;
    for (int u = 0; ok && u < n_steps; ++u) {
      const int t = t0 + (u0 + u) / p.G, g = (u0 + u) % p.G;
      const int hq = h * p.G + g;
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t r[64];
        ok = __all_sync(0xffffffffu, mbar_wait(&bar->dq_full[hh], u & 1, p.err, abort));
        if (!ok) break;
        tc_fence_after();
        tmem_ld32(tmem + lane_off + hh * 128 + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld32(tmem + lane_off + hh * 128 + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->dq_free[hh]);  // dQ^T is in registers: its columns are free
        const int q0 = t * kTile + hh * kHalf;
        const int nrows = min(kHalf, p.n_q - q0);
        float* dst = p.dq_acc + ((size_t)hq * p.n_q + q0) * kD + col;
#pragma unroll
        for (int rr = 0; rr < kHalf; ++rr)
          if (rr < nrows) atomicAdd(dst + (size_t)rr * kD, __uint_as_float(r[rr]));
      }
    }
  }

  // ------------------------------------------------------------------ dK/dV epilogue
  if (warp >= 2 && warp < 10) {
    const int et = threadIdx.x - 64;  // 0..255
    const int j = (warp & 3) * 32 + lane;  // key row == TMEM lane
    const int hc = (warp - 2) >> 2;        // dV / dK columns [64 hc, 64 hc + 64)
    const uint32_t lane_off = tmem_lane_base(warp);
    // the pool rows this CTA will own: key rows [r0, r1) of the block's dV and dK, pulled
    // into L2 while the partials are staged
    const uint32_t n = (uint32_t)p.n_split;
    const int rank = (int)cluster_ctarank();
    const int r0 = kTile * rank / (int)n, r1 = kTile * (rank + 1) / (int)n;
    const size_t blk = p.grad_staged ? (size_t)(p.stage_h0 + h) * p.stage_stride + s : (size_t)phys * p.Hkv + h;
    float4* gdv = reinterpret_cast<float4*>(p.dv_pool + blk * kTile * kD);
    float4* gdk = reinterpret_cast<float4*>(p.dk_pool + blk * kTile * kD);
    if (et == 0) {
      prefetch_l2(gdv + (size_t)r0 * (kD / 4), (uint32_t)(r1 - r0) * kD * 4);
      prefetch_l2(gdk + (size_t)r0 * (kD / 4), (uint32_t)(r1 - r0) * kD * 4);
    }
    // (1) stage this CTA's partial (zero when it had no step or its pipeline gave up)
    const bool have = __all_sync(0xffffffffu, ok_acc && mbar_wait(&bar->acc_full, 0, p.err, abort));
    if (have) tc_fence_after();
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t a[32], b[32];
      if (have) {
        tmem_ld32(tmem + lane_off + 256 + 64 * hc + cc * 32, a);
        tmem_ld32(tmem + lane_off + 384 + 64 * hc + cc * 32, b);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) a[e] = b[e] = 0u;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = 16 * hc + 8 * cc + e;  // float4 column of dV; 32 + c of dK
        *reinterpret_cast<float4*>(sm + kOffStage + stage_off(j, c)) =
            make_float4(__uint_as_float(a[4 * e]), __uint_as_float(a[4 * e + 1]), __uint_as_float(a[4 * e + 2]),
                        __uint_as_float(a[4 * e + 3]));
        *reinterpret_cast<float4*>(sm + kOffStage + stage_off(j, 32 + c)) =
            make_float4(p.scale * __uint_as_float(b[4 * e]), p.scale * __uint_as_float(b[4 * e + 1]),
                        p.scale * __uint_as_float(b[4 * e + 2]), p.scale * __uint_as_float(b[4 * e + 3]));
      }
    }
    fence_acq_rel_cluster();
    named_bar_sync(1, kSoftmaxThreads);
    cluster_wait();  // every peer's barriers are initialised
    if (et == 0)
      for (uint32_t q = 0; q < n; ++q) mbar_arrive_cluster(mapa_shared(smem_u32(&bar->staged), q));
    // (2) reduce key rows [r0, r1) over the cluster's partials, in rank order, into the pool
    if (__all_sync(0xffffffffu, mbar_wait_cluster(&bar->staged, 0, p.err))) {
      const uint32_t base = smem_u32(sm + kOffStage);
      const int n_items = (r1 - r0) * 64;  // (row, float4 column); a warp: one row, 32 consecutive float4
      // kBatch items per thread in flight: pool loads (from L2, prefetched above) and the
      // partials of every rank are all issued before the first add
      for (int i0 = et; i0 < n_items; i0 += kBatch * kSoftmaxThreads) {
        float4 x[kBatch], t[kBatch];
        float4* g[kBatch];
        uint32_t off[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int idx = min(i0 + u * kSoftmaxThreads, n_items - 1);  // clamped duplicates are not stored
          const int jj = r0 + idx / 64, c = idx % 64;
          off[u] = stage_off(jj, c);
          g[u] = (c < 32 ? gdv : gdk) + (size_t)jj * (kD / 4) + (c & 31);
          x[u] = *g[u];
          t[u] = ld_dsmem_f4(mapa_shared(base + off[u], 0));
        }
        for (uint32_t q = 1; q < n; ++q) {
#pragma unroll
          for (int u = 0; u < kBatch; ++u) {
            const float4 v = ld_dsmem_f4(mapa_shared(base + off[u], q));
            t[u].x += v.x;
            t[u].y += v.y;
            t[u].z += v.z;
            t[u].w += v.w;
          }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          if (i0 + u * kSoftmaxThreads < n_items) {
            x[u].x += t[u].x;
            x[u].y += t[u].y;
            x[u].z += t[u].z;
            x[u].w += t[u].w;
            *g[u] = x[u];
          }
        }
      }
    }
    // (3) this CTA has read every peer's staging; wait until its own was read by all
    fence_acq_rel_cluster();
    named_bar_sync(1, kSoftmaxThreads);
    if (et == 0)
      for (uint32_t q = 0; q < n; ++q) mbar_arrive_cluster(mapa_shared(smem_u32(&bar->reduced), q));
    mbar_wait_cluster(&bar->reduced, 0, p.err);
  } else {
    cluster_wait();  // every thread that arrived also waits once (long complete by now)
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Per (row, head) of the padded range: D = rowsum(dO * O) and LSE * log2(e) into
// [Hq, n_pad] buffers (rows past n_q: D = 0, LSE = +inf so that P = 0), and the
// row of the fp32 dQ accumulator zeroed.  One warp per (row, head).
__global__ void bwd_prep(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                         const float* __restrict__ lse, int n_q, int n_pad, int Hq, float* __restrict__ Dbuf,
                         float* __restrict__ lse2, float* __restrict__ dq_acc) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
  if (w >= n_pad * Hq) return;
  const int i = w / Hq, hq = w % Hq;
  if (i >= n_q) {
    if (lane == 0) {
      Dbuf[(size_t)hq * n_pad + i] = 0.f;
      lse2[(size_t)hq * n_pad + i] = INFINITY;
    }
    return;
  }
  const size_t off = ((size_t)i * Hq + hq) * kD + lane * 4;
  const uint2 a = *reinterpret_cast<const uint2*>(o + off);
  const uint2 b = *reinterpret_cast<const uint2*>(dout + off);
  const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const float2 x = __bfloat1622float2(a2[e]), y = __bfloat1622float2(b2[e]);
    s += x.x * y.x + x.y * y.y;
  }
#pragma unroll
  for (int off2 = 16; off2 > 0; off2 >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off2);
  if (lane == 0) {
    Dbuf[(size_t)hq * n_pad + i] = s;
    lse2[(size_t)hq * n_pad + i] = lse[(size_t)hq * n_q + i] * kLog2e;
  }
  reinterpret_cast<float4*>(dq_acc + ((size_t)hq * n_q + i) * kD)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dq[i][hq][:] = bf16(scale * dq_acc[hq][i][:]).  One warp per (row, head).
__global__ void bwd_convert(const float* __restrict__ dq_acc, int n_q, int Hq, float scale,
                            __nv_bfloat16* __restrict__ dq) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
  if (w >= n_q * Hq) return;
  const int i = w / Hq, hq = w % Hq;
  const float4 x = reinterpret_cast<const float4*>(dq_acc + ((size_t)hq * n_q + i) * kD)[lane];
  uint2 out;
  out.x = pack_bf16x2(x.x * scale, x.y * scale);
  out.y = pack_bf16x2(x.z * scale, x.w * scale);
  *reinterpret_cast<uint2*>(dq + ((size_t)i * Hq + hq) * kD + lane * 4) = out;
}

// How many CTAs (one cluster) share one (page, KV head).  A CTA's work is its number of
// steps (query tile x query head); history pages have n_tiles * G of them and the
// chunk's own page k has (n_tiles - k) * G.  A cluster of ns CTAs splits a page's steps
// into ns ranges and starts as a whole once ns SMs are free: with cluster_slots[ns]
// clusters resident at once (the device's cluster occupancy, which leaves SMs idle
// where a GPC's SM count is not a multiple of ns), the clusters start in launch order
// on the first free slot, each taking its longest part plus a fixed cost (K/V load,
// pipeline fill and drain, the dK/dV reduction) of about one step.  That greedy
// schedule is replayed for kMinSplit..kMaxSplit CTAs, and the fewest within 1% of the
// shortest schedule win.  Measured on GB300 (backward calls of whole sweeps), two CTAs
// beat one on every workload, also where this model sees no tail (1M tokens, chunks
// of 8192: 923 against 906 TFLOP/s), so two is the floor; more win where the grid is
// small (a 4K-token window over 4K chunks).  The selection counts live on the device,
// so every one of the max_sel slots is assumed filled; empty slots exit at once.
// Cached per shape.
constexpr int kMinSplit = 2;
constexpr int kMaxSplit = kMaxCluster;
constexpr double kCtaOverheadSteps = 1.0;

}  // namespace

int bwd_split(int max_sel, int n_own, int n_tiles, int G, int Hkv, const int* cluster_slots) {
  static std::mutex mu;
  static std::map<std::array<int, 9>, int> cache;
  const std::array<int, 9> key = {max_sel, n_own, n_tiles, G, Hkv, cluster_slots[1], cluster_slots[2],
                                  cluster_slots[3], cluster_slots[4]};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const int n_hist = std::max(0, max_sel - n_own);
  int best = kMinSplit;
  double best_t = -1.0;
  for (int ns = kMinSplit; ns <= kMaxSplit; ++ns) {
    const int slots = cluster_slots[ns];
    if (slots <= 0) continue;
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < slots; ++i) free_at.push(0.0);
    double end = 0.0;
    for (int sl = 0; sl < max_sel; ++sl) {
      const int k = sl - n_hist;  // own page index (< 0: history page)
      const int steps = (n_tiles - (k > 0 ? k : 0)) * G;
      const int w = (steps + ns - 1) / ns;  // longest part
      for (int hk = 0; hk < Hkv; ++hk) {
        const double t = free_at.top() + kCtaOverheadSteps + w;
        free_at.pop();
        free_at.push(t);
        end = std::max(end, t);
      }
    }
    if (best_t < 0.0 || end < 0.99 * best_t) {
      best = ns;
      best_t = end;
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = best;
  return best;
}

namespace {

// Clusters of ns CTAs of the backward kernel that can be resident at once on the
// current device (cudaOccupancyMaxActiveClusters), per device and ns.
cudaError_t cluster_slots(int* out /* [kMaxSplit + 1] */) {
  static int slots[kMaxDevices][kMaxSplit + 1] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!slots[dev][1]) {
    int tmp[kMaxSplit + 1] = {};
    for (int ns = 1; ns <= kMaxSplit; ++ns) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(ns * 64);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kSmemBytes;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = ns;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&tmp[ns], (const void*)attn_bwd_tc_kernel, &cfg);
      if (e != cudaSuccess) return e;
    }
    for (int ns = 1; ns <= kMaxSplit; ++ns) slots[dev][ns] = tmp[ns];
  }
  for (int ns = 0; ns <= kMaxSplit; ++ns) out[ns] = slots[dev][ns];
  return cudaSuccess;
}

}  // namespace

size_t bwd_tc_workspace_bytes(const Geometry& g, int n_q) {
  const size_t n_pad = (size_t)(n_q + kTile - 1) / kTile * kTile;
  return 2 * align_up((size_t)g.Hq * n_pad * 4, 256) + align_up((size_t)g.Hq * n_q * kD * 4, 256);
}

cudaError_t launch_attn_bwd_tc(const AttnArgs& a, cudaStream_t st) {
  static size_t smem_set[kMaxDevices] = {};
  cudaError_t e = set_smem_limit((const void*)attn_bwd_tc_kernel, kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  const int n_pad = (a.n_q + kTile - 1) / kTile * kTile;
  char* ws = reinterpret_cast<char*>(a.ws);
  float* Dbuf = reinterpret_cast<float*>(ws);
  float* lse2 = reinterpret_cast<float*>(ws + align_up((size_t)a.g.Hq * n_pad * 4, 256));
  float* dq_acc = reinterpret_cast<float*>(ws + 2 * align_up((size_t)a.g.Hq * n_pad * 4, 256));
  const int warps = a.n_q * a.g.Hq;
  const int warps_pad = n_pad * a.g.Hq;
  bwd_prep<<<(warps_pad + 7) / 8, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(a.o),
                                                reinterpret_cast<const __nv_bfloat16*>(a.dout), a.lse_in, a.n_q,
                                                n_pad, a.g.Hq, Dbuf, lse2, dq_acc);
  CUtensorMap tq, tdo, tk, tv;
  if (!make_tmap_heads(&tq, a.q, a.n_q, a.g.Hq, kHalf) || !make_tmap_heads(&tdo, a.dout, a.n_q, a.g.Hq, kHalf) ||
      !make_tmap_rows(&tk, a.kv.k, kv_rows(a)) || !make_tmap_rows(&tv, a.kv.v, kv_rows(a)))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.sel = a.sel;
  p.sel_count = a.sel_count;
  p.table = a.kv.table;
  p.lse2 = lse2;
  p.Dbuf = Dbuf;
  p.dq_acc = dq_acc;
  p.dk_pool = a.dk_pool;
  p.dv_pool = a.dv_pool;
  p.err = a.err;
  p.max_sel = a.max_sel;
  p.n_q = a.n_q;
  p.n_pad = n_pad;
  p.Hq = a.g.Hq;
  p.G = a.g.G;
  p.Hkv = a.g.Hkv;
  p.num_phys = a.g.num_phys;
  p.max_logical = a.g.max_logical;
  p.n_tiles = (a.n_q + kTile - 1) / kTile;
  p.q_start = a.q_start;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.staged = a.kv.staged;
  p.stage_h0 = a.kv.stage_h0;
  p.stage_stride = a.kv.stage_stride;
  p.grad_staged = a.grad_staged;
  const int first_own = (int)(a.q_start / kTile);
  const int n_own = (int)((a.q_start + a.n_q + kTile - 1) / kTile) - first_own;
  int slots[kMaxSplit + 1];
  e = cluster_slots(slots);
  if (e != cudaSuccess) return e;
  p.n_split = bwd_split(a.max_sel, n_own, p.n_tiles, p.G, p.Hkv, slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.max_sel * (unsigned)p.n_split * (unsigned)p.Hkv);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = (unsigned)p.n_split;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_bwd_tc_kernel, tq, tdo, tk, tv, p);
  if (e != cudaSuccess) return e;
  bwd_convert<<<(warps + 7) / 8, 256, 0, st>>>(dq_acc, a.n_q, a.g.Hq, a.scale,
                                               reinterpret_cast<__nv_bfloat16*>(a.dq));
  count_launches(3);
  return cudaGetLastError();
}

}  // namespace oomb
