// Paged KV append with fused page summary and gradient-page zeroing.
//
// "Out of the Memory Barrier" (gist.science explainer, 2.B "Paged KV Cache and
// Gradient Management", and the lay summary's "Trick A"): a chunk's K/V go onto
// the next free fixed-size pages through the page table, without copying earlier
// pages; the KV gradients live in pages that share the same table.  The page
// summary is the representative vector of 2.D, fixed as the mean key per page.
//
// One thread block per (new page, KV head) runs append_unit (append_unit.cuh): it
// loads the page's K and V rows with several 16-byte loads in flight per thread,
// zeroes both gradient pages while those loads are in flight, sums the K rows for the
// summary from the same registers (K is read once) and writes both pages; the fused
// selection-and-append kernel runs the same body.  (Splitting a page over more blocks, by rows with
// a cluster reduction of the summary or by columns, measured slower on GB300: a
// chunk's append moves 34-67 MB, and its time is the loads' latency plus the stores'
// drain, not the number of blocks.)  HBM traffic per token and KV head: read K,V
// (2 d esize), write K,V (2 d esize), zero dK,dV (2 d 4 bytes); plus one fp32 summary
// row per page and head.
#include "append_unit.cuh"

namespace oomb {
namespace {

constexpr int kMaxNewPerLaunch = 1024;

struct NewPages {
  int32_t phys[kMaxNewPerLaunch];
};

template <typename T>
__global__ void __launch_bounds__(kAppendThreads)
    kv_append_kernel(const __grid_constant__ AppendJob job, const __grid_constant__ NewPages np) {
  __shared__ float part[kAppendThreads * 8];
  const int i = blockIdx.x, h = blockIdx.y;
  append_unit<T>(job, np.phys[i], i, h, threadIdx.x, part, 1);
}

}  // namespace

AppendJob append_job(const Geometry& g, void* k_pool, void* v_pool, float* dk_pool, float* dv_pool, float* summary,
                     int32_t* table, const void* k, const void* v, int64_t first_token, int64_t total_tokens,
                     int n_new, int first_new_logical, uint8_t* grad_state, const StageArgs* stage, uint32_t* err) {
  AppendJob j = {};
  j.g = g;
  j.k_pool = k_pool;
  j.v_pool = v_pool;
  j.dk_pool = dk_pool;
  j.dv_pool = dv_pool;
  j.summary = summary;
  j.table = table;
  j.k = k;
  j.v = v;
  j.first_token = first_token;
  j.end_token = total_tokens;
  j.first_new_logical = first_new_logical;
  j.grad_state = grad_state;
  j.err = err;
  j.stg.slot0 = -1;
  if (stage) {
    j.stg.k = stage->k;
    j.stg.v = stage->v;
    j.stg.sel_count = stage->sel_count;
    j.stg.stage_h0 = stage->stage_h0;
    j.stg.stride = stage->stride;
    j.stg.max_sel = stage->max_sel;
    j.stg.n_own = n_new;
    j.stg.first_own = 0;
    j.stg.skip_pool = stage->skip_pool;
    j.stg.slot0 = stage->slot0;
  }
  return j;
}

cudaError_t launch_kv_append(const Geometry& g, void* k_pool, void* v_pool, float* dk_pool, float* dv_pool,
                             float* summary, int32_t* table, const void* k, const void* v, int64_t first_token,
                             int n_tokens, int64_t total_tokens, const int32_t* new_phys, int n_new,
                             int first_new_logical, uint8_t* grad_state, const StageArgs* stage, uint32_t* err,
                             cudaStream_t st) {
  (void)n_tokens;
  AppendJob job = append_job(g, k_pool, v_pool, dk_pool, dv_pool, summary, table, k, v, first_token, total_tokens,
                             n_new, first_new_logical, grad_state, stage, err);
  for (int base = 0; base < n_new; base += kMaxNewPerLaunch) {
    const int cnt = n_new - base < kMaxNewPerLaunch ? n_new - base : kMaxNewPerLaunch;
    NewPages np;
    for (int i = 0; i < cnt; ++i) np.phys[i] = new_phys[base + i];
    AppendJob jb = job;
    jb.first_new_logical = first_new_logical + base;
    jb.stg.first_own = base;
    dim3 grid(cnt, g.Hkv);
    if (g.dtype == OOMB_FP32) {
      kv_append_kernel<float><<<grid, kAppendThreads, 0, st>>>(jb, np);
    } else {
      kv_append_kernel<__nv_bfloat16><<<grid, kAppendThreads, 0, st>>>(jb, np);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
  }
  return cudaSuccess;
}

}  // namespace oomb
