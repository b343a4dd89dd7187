// SIMT (CUDA-core, fp32 arithmetic) chunk attention, forward and backward.
//
// Used for fp32 pools (full fp32 accuracy, no TF32) and for bf16 shapes the
// tensor-core kernels do not cover.  Same semantics as the tcgen05 kernels:
// causal GQA softmax attention of one query chunk over the keys of its selected
// pages ("Out of the Memory Barrier", gist.science explainer 2.D), backward with
// the probabilities recomputed from the saved LSE (2.A) and dK/dV added in place
// into the paged fp32 gradient pool (2.B), one thread block per (page, KV head,
// key sub-tile) so that no two blocks touch the same gradient rows.
//
// Kernels:
//   fwd_rows      one warp per query row, online softmax over 32-key sub-tiles
//   bwd_dot       D_i = dO_i . O_i
//   bwd_dq_rows   one warp per query row: dq = scale * sum_j dS_ij k_j
//   bwd_dkdv      one block per (selected page, KV head, 32-key sub-tile)
#include <cmath>

#include "attn_common.cuh"

namespace oomb {
namespace {

constexpr int kRowsPerBlock = 8;  // warps per block in the row kernels
constexpr int kKT = 32;           // keys per sub-tile
constexpr int kMaxD = 128;
constexpr int kDPerLane = kMaxD / 32;

// Visible-page bound for the chunk: pages at or after this index do not exist yet.
__device__ __forceinline__ int pages_visible(const AttnArgs& a) {
  return (int)((a.q_start + a.n_q + a.g.P - 1) / a.g.P);
}

template <typename T>
__global__ void __launch_bounds__(kRowsPerBlock * 32) fwd_rows(AttnArgs a) {
  const int d = a.g.d, P = a.g.P;
  const int hq = blockIdx.y, h = hq / a.g.G;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row0 = blockIdx.x * kRowsPerBlock;
  const int i = row0 + warp;
  const bool active = i < a.n_q;
  const int64_t qpos = a.q_start + i;
  const int64_t max_pos = a.q_start + min(a.n_q, row0 + kRowsPerBlock) - 1;

  __shared__ float sq[kRowsPerBlock][kMaxD];
  __shared__ float sk[kKT][kMaxD + 1];
  __shared__ float sv[kKT][kMaxD];
  const T* q = reinterpret_cast<const T*>(a.q);
  if (active)
    for (int e = lane; e < d; e += 32) sq[warp][e] = to_float<T>(q[((size_t)i * a.g.Hq + hq) * d + e]) * a.scale;

  float m = -INFINITY, l = 0.f;
  float o[kDPerLane];
#pragma unroll
  for (int r = 0; r < kDPerLane; ++r) o[r] = 0.f;

  const T* kp = reinterpret_cast<const T*>(a.kv.k);
  const T* vp = reinterpret_cast<const T*>(a.kv.v);
  const int count = sel_count_checked(a, h);
  const int nvis = pages_visible(a);
  for (int s = 0; s < count; ++s) {
    bool ok = true;
    const int p = sel_page(a, h, s, nvis, ok);
    if (!ok) continue;
    if ((int64_t)p * P > max_pos) continue;  // page entirely in the future of every row here
    const size_t blk = kv_block(a, h, s, p, ok);
    if (!ok) continue;
    for (int t0 = 0; t0 < P; t0 += kKT) {
      const int kt = min(kKT, P - t0);
      if ((int64_t)p * P + t0 > max_pos) break;
      __syncthreads();
      for (int idx = threadIdx.x; idx < kt * d; idx += blockDim.x) {
        const int r = idx / d, e = idx % d;
        const size_t off = (blk * P + t0 + r) * d + e;
        sk[r][e] = to_float<T>(kp[off]);
        sv[r][e] = to_float<T>(vp[off]);
      }
      __syncthreads();
      if (!active) continue;
      const int64_t kpos = (int64_t)p * P + t0 + lane;
      float sc = -INFINITY;
      if (lane < kt && kpos <= qpos) {
        float acc = 0.f;
        for (int e = 0; e < d; ++e) acc += sq[warp][e] * sk[lane][e];
        sc = acc;
      }
      float tmax = sc;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      if (tmax == -INFINITY) continue;
      const float m_new = fmaxf(m, tmax);
      const float alpha = expf(m - m_new);  // m = -inf -> 0
      const float pj = (sc == -INFINITY) ? 0.f : expf(sc - m_new);
      float psum = pj;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
      l = l * alpha + psum;
#pragma unroll
      for (int r = 0; r < kDPerLane; ++r) o[r] *= alpha;
      for (int j = 0; j < kt; ++j) {
        const float pjj = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
        for (int r = 0; r < kDPerLane; ++r) {
          const int e = lane + 32 * r;
          if (e < d) o[r] += pjj * sv[j][e];
        }
      }
      m = m_new;
    }
  }
  if (!active) return;
  T* out = reinterpret_cast<T*>(a.o_out);
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int r = 0; r < kDPerLane; ++r) {
    const int e = lane + 32 * r;
    if (e < d) out[((size_t)i * a.g.Hq + hq) * d + e] = from_float<T>(o[r] * inv);
  }
  if (lane == 0) a.lse_out[(size_t)hq * a.n_q + i] = m + logf(l);
}

template <typename T>
__global__ void bwd_dot(AttnArgs a, float* __restrict__ Dbuf) {
  // one warp per (row, head)
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
  if (w >= a.n_q * a.g.Hq) return;
  const int i = w / a.g.Hq, hq = w % a.g.Hq;
  const T* o = reinterpret_cast<const T*>(a.o) + ((size_t)i * a.g.Hq + hq) * a.g.d;
  const T* dout = reinterpret_cast<const T*>(a.dout) + ((size_t)i * a.g.Hq + hq) * a.g.d;
  float s = 0.f;
  for (int e = lane; e < a.g.d; e += 32) s += to_float<T>(o[e]) * to_float<T>(dout[e]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) Dbuf[(size_t)hq * a.n_q + i] = s;
}

template <typename T>
__global__ void __launch_bounds__(kRowsPerBlock * 32) bwd_dq_rows(AttnArgs a, const float* __restrict__ Dbuf) {
  const int d = a.g.d, P = a.g.P;
  const int hq = blockIdx.y, h = hq / a.g.G;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row0 = blockIdx.x * kRowsPerBlock;
  const int i = row0 + warp;
  const bool active = i < a.n_q;
  const int64_t qpos = a.q_start + i;
  const int64_t max_pos = a.q_start + min(a.n_q, row0 + kRowsPerBlock) - 1;

  __shared__ float sq[kRowsPerBlock][kMaxD];
  __shared__ float sdo[kRowsPerBlock][kMaxD];
  __shared__ float sk[kKT][kMaxD + 1];
  __shared__ float sv[kKT][kMaxD + 1];
  const T* q = reinterpret_cast<const T*>(a.q);
  const T* dout = reinterpret_cast<const T*>(a.dout);
  float lse = 0.f, Di = 0.f;
  if (active) {
    for (int e = lane; e < d; e += 32) {
      sq[warp][e] = to_float<T>(q[((size_t)i * a.g.Hq + hq) * d + e]);
      sdo[warp][e] = to_float<T>(dout[((size_t)i * a.g.Hq + hq) * d + e]);
    }
    lse = a.lse_in[(size_t)hq * a.n_q + i];
    Di = Dbuf[(size_t)hq * a.n_q + i];
  }
  float dq[kDPerLane];
#pragma unroll
  for (int r = 0; r < kDPerLane; ++r) dq[r] = 0.f;

  const T* kp = reinterpret_cast<const T*>(a.kv.k);
  const T* vp = reinterpret_cast<const T*>(a.kv.v);
  const int count = sel_count_checked(a, h);
  const int nvis = pages_visible(a);
  for (int s = 0; s < count; ++s) {
    bool ok = true;
    const int p = sel_page(a, h, s, nvis, ok);
    if (!ok) continue;
    if ((int64_t)p * P > max_pos) continue;
    const size_t blk = kv_block(a, h, s, p, ok);
    if (!ok) continue;
    for (int t0 = 0; t0 < P; t0 += kKT) {
      const int kt = min(kKT, P - t0);
      if ((int64_t)p * P + t0 > max_pos) break;
      __syncthreads();
      for (int idx = threadIdx.x; idx < kt * d; idx += blockDim.x) {
        const int r = idx / d, e = idx % d;
        const size_t off = (blk * P + t0 + r) * d + e;
        sk[r][e] = to_float<T>(kp[off]);
        sv[r][e] = to_float<T>(vp[off]);
      }
      __syncthreads();
      if (!active) continue;
      const int64_t kpos = (int64_t)p * P + t0 + lane;
      float ds = 0.f;
      if (lane < kt && kpos <= qpos) {
        float sacc = 0.f, dpacc = 0.f;
        for (int e = 0; e < d; ++e) {
          sacc += sq[warp][e] * sk[lane][e];
          dpacc += sdo[warp][e] * sv[lane][e];
        }
        const float pj = expf(sacc * a.scale - lse);
        ds = pj * (dpacc - Di);
      }
      for (int j = 0; j < kt; ++j) {
        const float dsj = __shfl_sync(0xffffffffu, ds, j);
#pragma unroll
        for (int r = 0; r < kDPerLane; ++r) {
          const int e = lane + 32 * r;
          if (e < d) dq[r] += dsj * sk[j][e];
        }
      }
    }
  }
  if (!active) return;
  T* out = reinterpret_cast<T*>(a.dq);
#pragma unroll
  for (int r = 0; r < kDPerLane; ++r) {
    const int e = lane + 32 * r;
    if (e < d) out[((size_t)i * a.g.Hq + hq) * d + e] = from_float<T>(dq[r] * a.scale);
  }
}

// Block (s, h, kt): keys [kt*32, kt*32+32) of selected page s of KV head h.
// Threads: 256.  Per (query head g, 32-row query tile): S and dP (32x32) into
// shared memory, then dV += P^T dO and dK += dS^T Q with thread (key j, column
// group cg) accumulating columns cg, cg+8, ... of key j.
constexpr int kDkdvThreads = 256;
constexpr int kColGroups = kDkdvThreads / kKT;  // 8
constexpr int kColsPerThread = kMaxD / kColGroups;  // 16

template <typename T>
__global__ void __launch_bounds__(kDkdvThreads) bwd_dkdv(AttnArgs a, const float* __restrict__ Dbuf) {
  const int d = a.g.d, P = a.g.P, G = a.g.G;
  const int s = blockIdx.x, h = blockIdx.y, kt0 = blockIdx.z * kKT;
  if (kt0 >= P) return;
  if (s >= sel_count_checked(a, h)) return;
  bool ok = true;
  const int nvis = pages_visible(a);
  const int p = sel_page(a, h, s, nvis, ok);
  if (!ok) return;
  const size_t blk = kv_block(a, h, s, p, ok);
  if (!ok) return;
  const int phys = a.kv.table[p];
  if (phys < 0 || phys >= a.g.num_phys) {
    if (threadIdx.x == 0) atomicOr(a.err, OOMB_DEVERR_PAGE);
    return;
  }
  const int kt = min(kKT, P - kt0);
  const int64_t key_pos0 = (int64_t)p * P + kt0;

  // dynamic shared memory: K, V, Q, dO tiles [32][d+1], P and dS [32][33], LSE and D
  extern __shared__ float dyn[];
  const int ld = d + 1;
  float* sk_ = dyn;
  float* sv_ = sk_ + kKT * ld;
  float* sq_ = sv_ + kKT * ld;
  float* sdo_ = sq_ + kKT * ld;
  float(*sp)[kKT + 1] = reinterpret_cast<float(*)[kKT + 1]>(sdo_ + kKT * ld);  // [row][key]
  float(*sds)[kKT + 1] = sp + kKT;                                             // [row][key]
  float* slse = reinterpret_cast<float*>(sds + kKT);
  float* sD = slse + kKT;
#define SK(r, c) sk_[(r) * ld + (c)]
#define SV(r, c) sv_[(r) * ld + (c)]
#define SQ(r, c) sq_[(r) * ld + (c)]
#define SDO(r, c) sdo_[(r) * ld + (c)]

  const T* kp = reinterpret_cast<const T*>(a.kv.k);
  const T* vp = reinterpret_cast<const T*>(a.kv.v);
  for (int idx = threadIdx.x; idx < kKT * d; idx += kDkdvThreads) {
    const int r = idx / d, e = idx % d;
    float kx = 0.f, vx = 0.f;
    if (r < kt) {
      const size_t off = (blk * P + kt0 + r) * d + e;
      kx = to_float<T>(kp[off]);
      vx = to_float<T>(vp[off]);
    }
    SK(r, e) = kx;
    SV(r, e) = vx;
  }
  const int j = threadIdx.x % kKT, cg = threadIdx.x / kKT;
  float dk[kColsPerThread], dv[kColsPerThread];
#pragma unroll
  for (int c = 0; c < kColsPerThread; ++c) dk[c] = dv[c] = 0.f;

  const T* q = reinterpret_cast<const T*>(a.q);
  const T* dout = reinterpret_cast<const T*>(a.dout);
  // first query row that can see the first key of this sub-tile
  const int64_t first_row = key_pos0 > a.q_start ? key_pos0 - a.q_start : 0;
  for (int gq = 0; gq < G; ++gq) {
    const int hq = h * G + gq;
    for (int r0 = (int)(first_row / kKT) * kKT; r0 < a.n_q; r0 += kKT) {
      __syncthreads();
      for (int idx = threadIdx.x; idx < kKT * d; idx += kDkdvThreads) {
        const int r = idx / d, e = idx % d;
        const int i = r0 + r;
        float qx = 0.f, dx = 0.f;
        if (i < a.n_q) {
          const size_t off = ((size_t)i * a.g.Hq + hq) * d + e;
          qx = to_float<T>(q[off]);
          dx = to_float<T>(dout[off]);
        }
        SQ(r, e) = qx;
        SDO(r, e) = dx;
      }
      if (threadIdx.x < kKT) {
        const int i = r0 + threadIdx.x;
        slse[threadIdx.x] = i < a.n_q ? a.lse_in[(size_t)hq * a.n_q + i] : 0.f;
        sD[threadIdx.x] = i < a.n_q ? Dbuf[(size_t)hq * a.n_q + i] : 0.f;
      }
      __syncthreads();
      // S, dP for 32 rows x 32 keys: entry e = threadIdx.x + 256 u
      for (int u = 0; u < (kKT * kKT) / kDkdvThreads; ++u) {
        const int e = threadIdx.x + kDkdvThreads * u;
        const int r = e / kKT, jj = e % kKT;
        const int i = r0 + r;
        const int64_t qpos = a.q_start + i;
        const int64_t kpos = key_pos0 + jj;
        float pv = 0.f, dsv = 0.f;
        if (i < a.n_q && jj < kt && kpos <= qpos) {
          float sacc = 0.f, dpacc = 0.f;
          for (int c = 0; c < d; ++c) {
            sacc += SQ(r, c) * SK(jj, c);
            dpacc += SDO(r, c) * SV(jj, c);
          }
          pv = expf(sacc * a.scale - slse[r]);
          dsv = pv * (dpacc - sD[r]);
        }
        sp[r][jj] = pv;
        sds[r][jj] = dsv;
      }
      __syncthreads();
      for (int r = 0; r < kKT; ++r) {
        const float pr = sp[r][j], dsr = sds[r][j];
#pragma unroll
        for (int c = 0; c < kColsPerThread; ++c) {
          const int col = cg + kColGroups * c;
          if (col < d) {
            dv[c] += pr * SDO(r, col);
            dk[c] += dsr * SQ(r, col);
          }
        }
      }
    }
  }
  if (j >= kt) return;
  const size_t gbase = (grad_block(a, h, s, phys) * P + kt0 + j) * d;
#pragma unroll
  for (int c = 0; c < kColsPerThread; ++c) {
    const int col = cg + kColGroups * c;
    if (col < d) {
      a.dk_pool[gbase + col] += a.scale * dk[c];
      a.dv_pool[gbase + col] += dv[c];
    }
  }
}
#undef SK
#undef SV
#undef SQ
#undef SDO

template <typename T>
cudaError_t fwd_simt(const AttnArgs& a, cudaStream_t st) {
  dim3 grid((a.n_q + kRowsPerBlock - 1) / kRowsPerBlock, a.g.Hq);
  fwd_rows<T><<<grid, kRowsPerBlock * 32, 0, st>>>(a);
  count_launches(1);
  return cudaGetLastError();
}

template <typename T>
cudaError_t bwd_simt(const AttnArgs& a, cudaStream_t st) {
  float* Dbuf = reinterpret_cast<float*>(a.ws);
  const int warps = a.n_q * a.g.Hq;
  bwd_dot<T><<<(warps * 32 + 255) / 256, 256, 0, st>>>(a, Dbuf);
  dim3 gq((a.n_q + kRowsPerBlock - 1) / kRowsPerBlock, a.g.Hq);
  bwd_dq_rows<T><<<gq, kRowsPerBlock * 32, 0, st>>>(a, Dbuf);
  dim3 gk(a.max_sel, a.g.Hkv, (a.g.P + kKT - 1) / kKT);
  const size_t shb = (size_t)(4 * kKT * (a.g.d + 1) + 2 * kKT * (kKT + 1) + 2 * kKT) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(bwd_dkdv<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shb);
  if (e != cudaSuccess) return e;
  bwd_dkdv<T><<<gk, kDkdvThreads, shb, st>>>(a, Dbuf);
  count_launches(3);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(const Geometry& g, int n_q) {
  const size_t simt = align_up((size_t)g.Hq * n_q * 4, 256);  // D
  return tc_supported(g) ? bwd_tc_workspace_bytes(g, n_q) : simt;
}

cudaError_t launch_attn_fwd_simt(const AttnArgs& a, cudaStream_t st) {
  return a.g.dtype == OOMB_FP32 ? fwd_simt<float>(a, st) : fwd_simt<__nv_bfloat16>(a, st);
}

cudaError_t launch_attn_bwd_simt(const AttnArgs& a, cudaStream_t st) {
  return a.g.dtype == OOMB_FP32 ? bwd_simt<float>(a, st) : bwd_simt<__nv_bfloat16>(a, st);
}

}  // namespace oomb
