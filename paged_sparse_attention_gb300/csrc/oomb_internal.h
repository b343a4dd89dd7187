// Internal declarations shared by the C-ABI layer and the kernel translation units.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <algorithm>
#include <cstdint>
#include <vector>

#include "../../include/oomb.h"

namespace oomb {

// Where a chunk's K/V blocks are read from.
//  resident: block(p, h) = table[p] * Hkv + h          in k/v
//  staged:   block(s, h) = (stage_base + h) * stride + s  in k/v (= staging buffers)
struct KvSource {
  const void* k;
  const void* v;
  const int32_t* table;  // logical -> physical page (resident mode and dK/dV addressing)
  int staged;            // 1: read K/V from staging slots
  int stage_h0;          // buffer index * Hkv
  int stage_stride;      // stage_max_sel
};

struct Geometry {
  int Hq, Hkv, G, d, P;
  int num_phys;
  int max_logical;
  int dtype;  // oomb_dtype
};

struct AttnArgs {
  Geometry g;
  KvSource kv;
  const void* q;
  const void* o;
  const void* dout;
  const float* lse_in;
  float* lse_out;
  void* o_out;
  void* dq;
  float* dk_pool;      // gradient pool, or the gradient staging buffers when grad_staged
  float* dv_pool;
  int grad_staged;     // 1: dK/dV blocks live in staging slots indexed like the staged K/V
  const int32_t* sel;
  const int32_t* sel_count;
  int max_sel;
  int64_t q_start;
  int n_q;
  float scale;
  uint32_t* err;
  void* ws;  // backward workspace
  size_t ws_bytes;
};

// Offload mode: the new pages of an append also go to the staging slots of the
// chunk's own pages (the last entries of each KV head's selection).
struct StageArgs {
  void* k;
  void* v;
  const int32_t* sel_count;
  int stage_h0, stride, max_sel;
  int skip_pool;  // 1: the new pages go to the staging slots only (the host pools later)
  int slot0 = -1; // >= 0: staging slot of own page 0 for every KV head (else read from sel_count)
};

// ---- launchers (return cudaGetLastError of the launch) ----
cudaError_t launch_kv_append(const Geometry& g, void* k_pool, void* v_pool, float* dk_pool, float* dv_pool,
                             float* summary, int32_t* table, const void* k, const void* v, int64_t first_token,
                             int n_tokens, int64_t total_tokens, const int32_t* new_phys, int n_new,
                             int first_new_logical, uint8_t* grad_state, const StageArgs* stage, uint32_t* err,
                             cudaStream_t st);

size_t select_workspace_bytes(const Geometry& g, int n_q);
// n_mapped_cand: candidate pages [n_sink', q_start/P) whose table entry is mapped;
// any_unmapped: some sink or candidate page is unmapped (freed) and must be skipped.
// job/new_phys/n_new: an append fused into the launch (only where select_scores holds and
// n_new <= kMaxFusedAppendPages; the append's staging slot must then be known, slot0 >= 0).
struct AppendJob;
constexpr int kMaxFusedAppendPages = 256;
cudaError_t launch_page_select(const Geometry& g, const float* summary, const int32_t* table, const void* q,
                               int64_t q_start, int n_q, int top_k, int n_sink, int n_mapped_cand, int any_unmapped,
                               int32_t* sel, int32_t* sel_count, int max_sel, void* ws, uint32_t* err, uint32_t* ctrl,
                               cudaStream_t st, const AppendJob* job = nullptr, const int32_t* new_phys = nullptr,
                               int n_new = 0);
// The selection scores pages (the cooperative grid runs), given the mapped candidates.
bool select_scores(int64_t q_start, int n_sink, int top_k, int n_mapped_cand, const Geometry& g);

// sel[h] = [0, sinks) U [lo, own_end) for every KV head h (host-validated bounds)
cudaError_t launch_window_select(const Geometry& g, int sinks, int lo, int own_end, int32_t* sel,
                                 int32_t* sel_count, int max_sel, cudaStream_t st);

size_t bwd_workspace_bytes(const Geometry& g, int n_q);
cudaError_t launch_attn_fwd_simt(const AttnArgs& a, cudaStream_t st);
cudaError_t launch_attn_bwd_simt(const AttnArgs& a, cudaStream_t st);
bool tc_supported(const Geometry& g);
cudaError_t launch_attn_fwd_tc(const AttnArgs& a, cudaStream_t st);
cudaError_t launch_attn_bwd_tc(const AttnArgs& a, cudaStream_t st);
size_t bwd_tc_workspace_bytes(const Geometry& g, int n_q);

cudaError_t launch_prefetch(const Geometry& g, const void* k_pool, const void* v_pool, const int32_t* table,
                            const int32_t* sel, const int32_t* sel_count, int max_sel, void* stage_k, void* stage_v,
                            int stage_h0, int stage_stride, int first_page, int end_page, uint32_t* err,
                            cudaStream_t st, int to_host = 0);

// Gradient staging (offload mode with host-resident dK/dV pools).  mode 0: stage the
// blocks of `sel` whose page is not in `prev` from the host pools; mode 1: copy the
// blocks whose page is in `prev` from the other staging buffer (slot of that page in
// prev); mode 2: write every block of `sel` back to the host pools.
enum GradCopyMode { kGradFromHost = 0, kGradCarry = 1, kGradToHost = 2 };
cudaError_t launch_grad_copy(const Geometry& g, int mode, float* dk_pool, float* dv_pool, uint8_t* grad_state,
                             const int32_t* table, const int32_t* sel, const int32_t* sel_count,
                             const int32_t* prev_sel, const int32_t* prev_count, int max_sel, float* stage_dk,
                             float* stage_dv, int buf, int stage_stride, uint32_t* err, cudaStream_t st);

cudaError_t launch_grad_gather(const Geometry& g, const float* dk_pool, const float* dv_pool, const int32_t* table,
                               int64_t first_token, int n_tokens, float* dk, float* dv, uint32_t* err,
                               cudaStream_t st);

__host__ __device__ inline size_t dtype_size(int dt) { return dt == OOMB_FP32 ? 4 : 2; }
// Count of kernel launches issued by the library (reported by oomb_launch_count).
void count_launches(int n);

// Per-device host caches (CUDA function attributes and device properties are per device).
constexpr int kMaxDevices = 64;
// Raises `fn`'s dynamic shared-memory limit to `bytes` on the current device, once per
// device and size; `done` is the caller's [kMaxDevices] record of sizes already set.
cudaError_t set_smem_limit(const void* fn, size_t bytes, size_t* done);
// Number of SMs of the current device.
int device_sm_count();

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace oomb
