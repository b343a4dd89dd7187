// C-ABI layer: pool object, host-side page allocator, argument checks and
// dispatch to the kernels.  No call here allocates device memory.
#include <atomic>
#include <climits>
#include <cstring>
#include <new>

#include "append_unit.cuh"
#include "oomb_internal.h"

using namespace oomb;

struct oomb_pool {
  oomb_pool_desc d;
  Geometry g;
  std::vector<int32_t> order;      // creation order of physical pages
  std::vector<int32_t> free_list;  // stack: back() is handed out next
  std::vector<int32_t> table;      // host copy of the page table
  std::vector<int64_t> freed;      // logical pages freed since the last reset, ascending
  int64_t n_tokens = 0;
  int stage_buf = 0;
  bool table_dirty = true;  // device page table still needs its -1 fill
};

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

void oomb::count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

cudaError_t oomb::set_smem_limit(const void* fn, size_t bytes, size_t* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done[dev] = bytes;
  return e;
}

int oomb::device_sm_count() {
  static int count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  if (!count[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    count[dev] = n > 0 ? n : 148;
  }
  return count[dev];
}

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

thread_local const char* t_last_cuda_error = "";

oomb_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return OOMB_OK;
  t_last_cuda_error = cudaGetErrorString(e);
  return OOMB_ERR_CUDA;
}

Geometry geometry_of(const oomb_pool_desc& d) {
  Geometry g;
  g.Hq = d.n_q_heads;
  g.Hkv = d.n_kv_heads;
  g.G = d.n_kv_heads > 0 ? d.n_q_heads / d.n_kv_heads : 0;
  g.d = d.head_dim;
  g.P = d.page_size;
  g.num_phys = d.num_phys_pages;
  g.max_logical = d.max_logical_pages;
  g.dtype = d.dtype;
  return g;
}

void rebuild_free_list(oomb_pool* p) {
  p->free_list.assign(p->order.rbegin(), p->order.rend());
  std::fill(p->table.begin(), p->table.end(), -1);
  p->freed.clear();
  p->n_tokens = 0;
  p->table_dirty = true;
}

// Fill the device page table with -1 (all-ones bytes) before its first use.
cudaError_t clear_table_if_dirty(oomb_pool* p, cudaStream_t st) {
  if (!p->table_dirty) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(p->d.page_table, 0xFF, sizeof(int32_t) * (size_t)p->g.max_logical, st);
  if (e == cudaSuccess) p->table_dirty = false;
  return e;
}

KvSource kv_source(const oomb_pool* p) {
  KvSource s;
  s.table = p->d.page_table;
  if (p->d.offload) {
    s.k = p->d.stage_k;
    s.v = p->d.stage_v;
    s.staged = 1;
    s.stage_h0 = p->stage_buf * p->g.Hkv;
    s.stage_stride = p->d.stage_max_sel;
  } else {
    s.k = p->d.k_pool;
    s.v = p->d.v_pool;
    s.staged = 0;
    s.stage_h0 = 0;
    s.stage_stride = 0;
  }
  return s;
}

// Checks shared by the chunk-level calls.  `own_appended`: the chunk's own K/V must
// already be in the pool (attention); a selection reads history pages only, so it
// needs just the history.
oomb_status check_chunk(const oomb_pool* p, const void* q, int64_t q_start, int n_q, const int32_t* sel,
                        const int32_t* sel_count, int max_sel, bool own_appended = true) {
  if (!p || !q || !sel || !sel_count) return OOMB_ERR_ARG;
  if (n_q <= 0 || q_start < 0 || max_sel <= 0) return OOMB_ERR_ARG;
  if (q_start % p->g.P != 0) return OOMB_ERR_ALIGN;
  if (q_start > p->n_tokens) return OOMB_ERR_ARG;                       // the history
  if (own_appended && q_start + n_q > p->n_tokens) return OOMB_ERR_ARG;  // own K/V
  if (q_start + n_q > (int64_t)p->g.max_logical * p->g.P) return OOMB_ERR_ARG;
  if (!aligned(q, 16) || !aligned(sel, 4) || !aligned(sel_count, 4)) return OOMB_ERR_ALIGN;
  return OOMB_OK;
}

}  // namespace

extern "C" {

const char* oomb_status_str(oomb_status s) {
  switch (s) {
    case OOMB_OK: return "ok";
    case OOMB_ERR_ARG: return "bad argument";
    case OOMB_ERR_OUT_OF_PAGES: return "out of pages";
    case OOMB_ERR_ALIGN: return "misaligned pointer or offset";
    case OOMB_ERR_DTYPE: return "unknown dtype";
    case OOMB_ERR_KERNEL: return "kernel raised the device error word";
    case OOMB_ERR_TIMEOUT: return "device wait timed out";
    case OOMB_ERR_CUDA: return "CUDA runtime error";
    case OOMB_ERR_UNSUPPORTED: return "unsupported shape, dtype or mode";
    case OOMB_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

oomb_status oomb_pool_create(const oomb_pool_desc* desc, oomb_pool** out) {
  if (!desc || !out) return OOMB_ERR_ARG;
  *out = nullptr;
  const oomb_pool_desc& d = *desc;
  if (d.dtype != OOMB_BF16 && d.dtype != OOMB_FP32) return OOMB_ERR_DTYPE;
  if (d.n_q_heads <= 0 || d.n_kv_heads <= 0 || d.n_q_heads % d.n_kv_heads) return OOMB_ERR_ARG;
  if (d.head_dim <= 0 || d.head_dim > 128) return OOMB_ERR_UNSUPPORTED;
  if (d.head_dim % (d.dtype == OOMB_FP32 ? 4 : 8)) return OOMB_ERR_UNSUPPORTED;
  if (d.page_size <= 0 || d.page_size > 256) return OOMB_ERR_UNSUPPORTED;
  if (d.num_phys_pages <= 0 || d.max_logical_pages <= 0) return OOMB_ERR_ARG;
  if (!d.k_pool || !d.v_pool || !d.dk_pool || !d.dv_pool || !d.summary || !d.page_table || !d.error_word)
    return OOMB_ERR_ARG;
  const void* ptrs[] = {d.k_pool, d.v_pool, d.dk_pool, d.dv_pool, d.summary, d.error_word};
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return OOMB_ERR_ALIGN;
  if (!aligned(d.page_table, 4)) return OOMB_ERR_ALIGN;
  if (d.offload) {
    if (!d.stage_k || !d.stage_v || d.stage_max_sel <= 0) return OOMB_ERR_ARG;
    if (!aligned(d.stage_k, 16) || !aligned(d.stage_v, 16)) return OOMB_ERR_ALIGN;
  }
  if (d.offload_grads) {
    if (!d.offload || !d.stage_dk || !d.stage_dv || !d.grad_state) return OOMB_ERR_ARG;
    if (!aligned(d.stage_dk, 16) || !aligned(d.stage_dv, 16)) return OOMB_ERR_ALIGN;
  }
  oomb_pool* p = new (std::nothrow) oomb_pool;
  if (!p) return OOMB_ERR_ARG;
  p->d = d;
  p->d.page_order = nullptr;
  p->g = geometry_of(d);
  p->order.resize(d.num_phys_pages);
  if (d.page_order) {
    std::vector<char> seen(d.num_phys_pages, 0);
    for (int i = 0; i < d.num_phys_pages; ++i) {
      int32_t v = d.page_order[i];
      if (v < 0 || v >= d.num_phys_pages || seen[v]) {
        delete p;
        return OOMB_ERR_ARG;
      }
      seen[v] = 1;
      p->order[i] = v;
    }
  } else {
    for (int i = 0; i < d.num_phys_pages; ++i) p->order[i] = i;
  }
  p->table.assign(d.max_logical_pages, -1);
  rebuild_free_list(p);
  *out = p;
  return OOMB_OK;
}

void oomb_pool_destroy(oomb_pool* pool) { delete pool; }

oomb_status oomb_pool_reset(oomb_pool* p, void* stream) {
  if (!p) return OOMB_ERR_ARG;
  rebuild_free_list(p);
  return cuda_status(clear_table_if_dirty(p, (cudaStream_t)stream));
}

int64_t oomb_pool_tokens(const oomb_pool* p) { return p ? p->n_tokens : -1; }
int oomb_pool_free_pages(const oomb_pool* p) { return p ? (int)p->free_list.size() : -1; }

int oomb_page_table_host(const oomb_pool* p, int32_t* out, int n) {
  if (!p || !out || n < 0) return 0;
  int m = n < p->g.max_logical ? n : p->g.max_logical;
  std::memcpy(out, p->table.data(), sizeof(int32_t) * (size_t)m);
  return m;
}

const char* oomb_last_cuda_error(void) { return t_last_cuda_error; }

uint64_t oomb_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int oomb_uses_tensor_cores(const oomb_pool* p) { return p && tc_supported(p->g) ? 1 : 0; }

// An append about to be launched: its new pages are taken from the free list and
// entered in the host table; undone by release() if the launch fails.
struct PendingAppend {
  std::vector<int32_t> newp;
  int64_t first_page = 0, end = 0;
  int n_new = 0;
  void release(oomb_pool* p) {
    for (int i = n_new - 1; i >= 0; --i) {
      p->free_list.push_back(newp[i]);
      p->table[first_page + i] = -1;
    }
  }
};

static oomb_status prepare_append(oomb_pool* p, const void* k, const void* v, int64_t first_token, int n_tokens,
                                  void* stream, PendingAppend* pa) {
  if (!p || !k || !v || n_tokens <= 0 || first_token < 0) return OOMB_ERR_ARG;
  if (first_token != p->n_tokens) return OOMB_ERR_ARG;
  if (first_token % p->g.P != 0) return OOMB_ERR_ALIGN;
  if (!aligned(k, 16) || !aligned(v, 16)) return OOMB_ERR_ALIGN;
  const int P = p->g.P;
  const int64_t end = first_token + n_tokens;
  const int64_t first_page = first_token / P;
  const int64_t end_page = (end + P - 1) / P;
  if (end_page > p->g.max_logical) return OOMB_ERR_ARG;
  const int n_new = (int)(end_page - first_page);
  if (n_new > (int)p->free_list.size()) return OOMB_ERR_OUT_OF_PAGES;
  cudaError_t e = clear_table_if_dirty(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e);
  pa->newp.resize(n_new);
  for (int i = 0; i < n_new; ++i) {
    pa->newp[i] = p->free_list.back();
    p->free_list.pop_back();
    p->table[first_page + i] = pa->newp[i];
  }
  pa->first_page = first_page;
  pa->end = end;
  pa->n_new = n_new;
  return OOMB_OK;
}

// Shared body of oomb_kv_append, oomb_kv_append_staged and oomb_kv_append_deferred.
static oomb_status kv_append_impl(oomb_pool* p, const void* k, const void* v, int64_t first_token, int n_tokens,
                                  const StageArgs* stage, void* stream) {
  PendingAppend pa;
  oomb_status s = prepare_append(p, k, v, first_token, n_tokens, stream, &pa);
  if (s != OOMB_OK) return s;
  cudaError_t e = launch_kv_append(p->g, p->d.k_pool, p->d.v_pool, p->d.dk_pool, p->d.dv_pool, p->d.summary,
                                   p->d.page_table, k, v, first_token, n_tokens, pa.end, pa.newp.data(), pa.n_new,
                                   (int)pa.first_page, p->d.offload_grads ? p->d.grad_state : nullptr, stage,
                                   p->d.error_word, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    pa.release(p);
    return cuda_status(e);
  }
  p->n_tokens = pa.end;
  return OOMB_OK;
}

oomb_status oomb_kv_append(oomb_pool* p, const void* k, const void* v, int64_t first_token, int n_tokens,
                           void* stream) {
  return kv_append_impl(p, k, v, first_token, n_tokens, nullptr, stream);
}

// Shared body of oomb_kv_append_staged and oomb_kv_append_deferred.
static oomb_status kv_append_stage_impl(oomb_pool* p, const void* k, const void* v, int64_t first_token,
                                        int n_tokens, const int32_t* sel_count, int max_sel, int stage_buf,
                                        int skip_pool, void* stream) {
  if (!p || !sel_count || max_sel <= 0) return OOMB_ERR_ARG;
  if (!p->d.offload) return OOMB_ERR_UNSUPPORTED;
  if (stage_buf < 0 || stage_buf > 1 || max_sel > p->d.stage_max_sel) return OOMB_ERR_ARG;
  if (!aligned(sel_count, 4)) return OOMB_ERR_ALIGN;
  StageArgs sa;
  sa.k = p->d.stage_k;
  sa.v = p->d.stage_v;
  sa.sel_count = sel_count;
  sa.stage_h0 = stage_buf * p->g.Hkv;
  sa.stride = p->d.stage_max_sel;
  sa.max_sel = max_sel;
  sa.skip_pool = skip_pool;
  return kv_append_impl(p, k, v, first_token, n_tokens, &sa, stream);
}

oomb_status oomb_kv_append_staged(oomb_pool* p, const void* k, const void* v, int64_t first_token, int n_tokens,
                                  const int32_t* sel_count, int max_sel, int stage_buf, void* stream) {
  return kv_append_stage_impl(p, k, v, first_token, n_tokens, sel_count, max_sel, stage_buf, 0, stream);
}

oomb_status oomb_kv_append_deferred(oomb_pool* p, const void* k, const void* v, int64_t first_token, int n_tokens,
                                    const int32_t* sel_count, int max_sel, int stage_buf, void* stream) {
  return kv_append_stage_impl(p, k, v, first_token, n_tokens, sel_count, max_sel, stage_buf, 1, stream);
}

oomb_status oomb_page_free(oomb_pool* p, int64_t first_logical_page, int n_pages, void* stream) {
  if (!p || first_logical_page < 0 || n_pages <= 0) return OOMB_ERR_ARG;
  const int P = p->g.P;
  const int64_t end = first_logical_page + n_pages;
  if (end > (p->n_tokens + P - 1) / P) return OOMB_ERR_ARG;  // only appended pages
  for (int64_t i = first_logical_page; i < end; ++i)
    if (p->table[i] < 0) return OOMB_ERR_ARG;  // freed already
  cudaError_t e = cudaMemsetAsync(p->d.page_table + first_logical_page, 0xFF, sizeof(int32_t) * (size_t)n_pages,
                                  (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e);
  // the free list hands out from its back: push the highest page first
  for (int64_t i = end - 1; i >= first_logical_page; --i) {
    p->free_list.push_back(p->table[i]);
    p->table[i] = -1;
  }
  // appends map only new logical pages, so a freed logical page stays unmapped
  std::vector<int64_t> add;
  for (int64_t i = first_logical_page; i < end; ++i) add.push_back(i);
  std::vector<int64_t> merged(p->freed.size() + add.size());
  std::merge(p->freed.begin(), p->freed.end(), add.begin(), add.end(), merged.begin());
  p->freed.swap(merged);
  return OOMB_OK;
}

size_t oomb_workspace_size(const oomb_pool* p, int op, int n_q) {
  if (!p || n_q <= 0) return 0;
  if (op == OOMB_OP_SELECT) return select_workspace_bytes(p->g, n_q);
  if (op == OOMB_OP_BWD) return bwd_workspace_bytes(p->g, n_q);
  return 0;
}

// What a top-K selection of one chunk will hold, known on the host: the mapped
// candidates, whether any sink or candidate is freed, and the entry count per KV head
// (the same for every head: mapped sinks + kept candidates + own pages).
struct SelectPlan {
  int64_t mapped = 0, count = 0, n_own = 0;
  int any_unmapped = 0;
};

static oomb_status plan_select(oomb_pool* p, const void* q, int64_t q_start, int n_q, int top_k, int n_sink,
                               int32_t* sel, int32_t* sel_count, int max_sel, void* ws, size_t ws_bytes,
                               SelectPlan* plan) {
  oomb_status s = check_chunk(p, q, q_start, n_q, sel, sel_count, max_sel, false);
  if (s != OOMB_OK) return s;
  if (top_k < -1 || n_sink < 0) return OOMB_ERR_ARG;
  const int P = p->g.P;
  const int64_t n_hist = q_start / P;
  const int64_t n_own = (q_start + n_q + P - 1) / P - n_hist;
  const int64_t sinks = n_sink < n_hist ? n_sink : n_hist;
  const int64_t cand = n_hist - sinks;
  // freed pages are neither sinks nor candidates
  auto n_freed = [p](int64_t lo, int64_t hi) {
    return (int64_t)(std::lower_bound(p->freed.begin(), p->freed.end(), hi) -
                     std::lower_bound(p->freed.begin(), p->freed.end(), lo));
  };
  const int64_t freed_sinks = n_freed(0, sinks), freed_cand = n_freed(sinks, n_hist);
  const int64_t mapped = cand - freed_cand;
  const int64_t kept = (top_k < 0 || mapped <= top_k) ? mapped : top_k;
  if (sinks - freed_sinks + kept + n_own > max_sel) return OOMB_ERR_ARG;
  size_t need = select_workspace_bytes(p->g, n_q);
  if (!ws || ws_bytes < need) return OOMB_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return OOMB_ERR_ALIGN;
  plan->mapped = mapped;
  plan->count = sinks - freed_sinks + kept + n_own;
  plan->n_own = n_own;
  plan->any_unmapped = (freed_sinks + freed_cand) > 0 ? 1 : 0;
  return OOMB_OK;
}

oomb_status oomb_page_select(oomb_pool* p, const void* q, int64_t q_start, int n_q, int top_k, int n_sink,
                             int32_t* sel, int32_t* sel_count, int max_sel, void* ws, size_t ws_bytes,
                             void* stream) {
  SelectPlan plan;
  oomb_status s = plan_select(p, q, q_start, n_q, top_k, n_sink, sel, sel_count, max_sel, ws, ws_bytes, &plan);
  if (s != OOMB_OK) return s;
  return cuda_status(launch_page_select(p->g, p->d.summary, p->d.page_table, q, q_start, n_q, top_k, n_sink,
                                        (int)plan.mapped, plan.any_unmapped, sel, sel_count, max_sel, ws,
                                        p->d.error_word, p->d.error_word, (cudaStream_t)stream));
}

oomb_status oomb_page_select_append(oomb_pool* p, const void* q, const void* k, const void* v, int64_t q_start,
                                    int n_q, int top_k, int n_sink, int32_t* sel, int32_t* sel_count, int max_sel,
                                    void* ws, size_t ws_bytes, int append_mode, int stage_buf, void* stream) {
  if (!p) return OOMB_ERR_ARG;
  if (append_mode < OOMB_APPEND_POOL || append_mode > OOMB_APPEND_DEFERRED) return OOMB_ERR_ARG;
  if (append_mode != OOMB_APPEND_POOL) {
    if (!p->d.offload) return OOMB_ERR_UNSUPPORTED;
    if (stage_buf < 0 || stage_buf > 1 || max_sel > p->d.stage_max_sel) return OOMB_ERR_ARG;
  }
  if (q_start != p->n_tokens) return OOMB_ERR_ARG;  // the chunk's K/V are appended now
  SelectPlan plan;
  oomb_status s = plan_select(p, q, q_start, n_q, top_k, n_sink, sel, sel_count, max_sel, ws, ws_bytes, &plan);
  if (s != OOMB_OK) return s;
  PendingAppend pa;
  s = prepare_append(p, k, v, q_start, n_q, stream, &pa);
  if (s != OOMB_OK) return s;
  StageArgs sa;
  const StageArgs* stage = nullptr;
  if (append_mode != OOMB_APPEND_POOL) {
    sa.k = p->d.stage_k;
    sa.v = p->d.stage_v;
    sa.sel_count = sel_count;
    sa.stage_h0 = stage_buf * p->g.Hkv;
    sa.stride = p->d.stage_max_sel;
    sa.max_sel = max_sel;
    sa.skip_pool = append_mode == OOMB_APPEND_DEFERRED ? 1 : 0;
    sa.slot0 = (int)(plan.count - plan.n_own);  // own page 0's entry, the same for every KV head
    stage = &sa;
  }
  uint8_t* gs = p->d.offload_grads ? p->d.grad_state : nullptr;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e;
  if (select_scores(q_start, n_sink, top_k, (int)plan.mapped, p->g) && pa.n_new <= kMaxFusedAppendPages) {
    // one launch: the selection's grid appends the chunk's pages before its query sum
    const AppendJob job = append_job(p->g, p->d.k_pool, p->d.v_pool, p->d.dk_pool, p->d.dv_pool, p->d.summary,
                                     p->d.page_table, k, v, q_start, pa.end, pa.n_new, (int)pa.first_page, gs,
                                     stage, p->d.error_word);
    e = launch_page_select(p->g, p->d.summary, p->d.page_table, q, q_start, n_q, top_k, n_sink, (int)plan.mapped,
                           plan.any_unmapped, sel, sel_count, max_sel, ws, p->d.error_word, p->d.error_word, st,
                           &job, pa.newp.data(), pa.n_new);
  } else {  // a selection that scores nothing (or a very long chunk): two launches
    e = launch_page_select(p->g, p->d.summary, p->d.page_table, q, q_start, n_q, top_k, n_sink, (int)plan.mapped,
                           plan.any_unmapped, sel, sel_count, max_sel, ws, p->d.error_word, p->d.error_word, st);
    if (e == cudaSuccess)
      e = launch_kv_append(p->g, p->d.k_pool, p->d.v_pool, p->d.dk_pool, p->d.dv_pool, p->d.summary,
                           p->d.page_table, k, v, q_start, n_q, pa.end, pa.newp.data(), pa.n_new, (int)pa.first_page,
                           gs, stage, p->d.error_word, st);
  }
  if (e != cudaSuccess) {
    pa.release(p);
    return cuda_status(e);
  }
  p->n_tokens = pa.end;
  return OOMB_OK;
}

oomb_status oomb_window_select(oomb_pool* p, int64_t q_start, int n_q, int window, int n_sink, int32_t* sel,
                               int32_t* sel_count, int max_sel, void* stream) {
  if (!p || !sel || !sel_count) return OOMB_ERR_ARG;
  if (n_q <= 0 || q_start < 0 || max_sel <= 0 || window < 0 || n_sink < 0) return OOMB_ERR_ARG;
  if (q_start % p->g.P != 0) return OOMB_ERR_ALIGN;
  if (q_start > p->n_tokens) return OOMB_ERR_ARG;  // the history must be appended
  if (!aligned(sel, 4) || !aligned(sel_count, 4)) return OOMB_ERR_ALIGN;
  const int P = p->g.P;
  const int64_t n_hist = q_start / P;
  const int64_t own_end = (q_start + n_q + P - 1) / P;
  const int64_t sinks = n_sink < n_hist ? n_sink : n_hist;
  const int64_t lo = std::max<int64_t>(sinks, n_hist - window);
  if (own_end > p->g.max_logical) return OOMB_ERR_ARG;
  if (sinks + (own_end - lo) > max_sel) return OOMB_ERR_ARG;
  return cuda_status(launch_window_select(p->g, (int)sinks, (int)lo, (int)own_end, sel, sel_count, max_sel,
                                          (cudaStream_t)stream));
}

static AttnArgs make_args(oomb_pool* p, const void* q, int64_t q_start, int n_q, const int32_t* sel,
                          const int32_t* sel_count, int max_sel, float scale) {
  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.g = p->g;
  a.kv = kv_source(p);
  a.q = q;
  a.q_start = q_start;
  a.n_q = n_q;
  a.sel = sel;
  a.sel_count = sel_count;
  a.max_sel = max_sel;
  a.scale = scale;
  a.err = p->d.error_word;
  if (p->d.offload_grads) {  // the backward adds into the staged gradient blocks
    a.dk_pool = p->d.stage_dk;
    a.dv_pool = p->d.stage_dv;
    a.grad_staged = 1;
  } else {
    a.dk_pool = p->d.dk_pool;
    a.dv_pool = p->d.dv_pool;
    a.grad_staged = 0;
  }
  return a;
}

oomb_status oomb_chunk_attn_fwd(oomb_pool* p, const void* q, int64_t q_start, int n_q, const int32_t* sel,
                                const int32_t* sel_count, int max_sel, float scale, void* o, float* lse,
                                void* stream) {
  oomb_status s = check_chunk(p, q, q_start, n_q, sel, sel_count, max_sel);
  if (s != OOMB_OK) return s;
  if (!o || !lse) return OOMB_ERR_ARG;
  if (!aligned(o, 16) || !aligned(lse, 4)) return OOMB_ERR_ALIGN;
  if (p->d.offload && max_sel > p->d.stage_max_sel) return OOMB_ERR_ARG;
  AttnArgs a = make_args(p, q, q_start, n_q, sel, sel_count, max_sel, scale);
  a.o_out = o;
  a.lse_out = lse;
  cudaError_t e = tc_supported(p->g) ? launch_attn_fwd_tc(a, (cudaStream_t)stream)
                                     : launch_attn_fwd_simt(a, (cudaStream_t)stream);
  return cuda_status(e);
}

oomb_status oomb_chunk_attn_bwd(oomb_pool* p, const void* q, const void* o, const void* d_o, const float* lse,
                                int64_t q_start, int n_q, const int32_t* sel, const int32_t* sel_count, int max_sel,
                                float scale, void* dq, void* ws, size_t ws_bytes, void* stream) {
  oomb_status s = check_chunk(p, q, q_start, n_q, sel, sel_count, max_sel);
  if (s != OOMB_OK) return s;
  if (!o || !d_o || !lse || !dq) return OOMB_ERR_ARG;
  if (!aligned(o, 16) || !aligned(d_o, 16) || !aligned(dq, 16) || !aligned(lse, 4)) return OOMB_ERR_ALIGN;
  if (p->d.offload && max_sel > p->d.stage_max_sel) return OOMB_ERR_ARG;
  size_t need = bwd_workspace_bytes(p->g, n_q);
  if (need > 0 && (!ws || ws_bytes < need)) return OOMB_ERR_WORKSPACE;
  if (ws && !aligned(ws, 16)) return OOMB_ERR_ALIGN;
  AttnArgs a = make_args(p, q, q_start, n_q, sel, sel_count, max_sel, scale);
  a.o = o;
  a.dout = d_o;
  a.lse_in = lse;
  a.dq = dq;
  a.ws = ws;
  a.ws_bytes = ws_bytes;
  cudaError_t e = tc_supported(p->g) ? launch_attn_bwd_tc(a, (cudaStream_t)stream)
                                     : launch_attn_bwd_simt(a, (cudaStream_t)stream);
  return cuda_status(e);
}

oomb_status oomb_prefetch_pages(oomb_pool* p, const int32_t* sel, const int32_t* sel_count, int max_sel,
                                int stage_buf, int64_t first_page, int64_t end_page, void* stream) {
  if (!p || !sel || !sel_count || max_sel <= 0 || first_page < 0 || end_page < first_page) return OOMB_ERR_ARG;
  if (!p->d.offload) return OOMB_ERR_UNSUPPORTED;
  if (stage_buf < 0 || stage_buf > 1 || max_sel > p->d.stage_max_sel) return OOMB_ERR_ARG;
  if (!aligned(sel, 4) || !aligned(sel_count, 4)) return OOMB_ERR_ALIGN;
  const int lo = (int)std::min<int64_t>(first_page, INT32_MAX), hi = (int)std::min<int64_t>(end_page, INT32_MAX);
  return cuda_status(launch_prefetch(p->g, p->d.k_pool, p->d.v_pool, p->d.page_table, sel, sel_count, max_sel,
                                     p->d.stage_k, p->d.stage_v, stage_buf * p->g.Hkv, p->d.stage_max_sel, lo, hi,
                                     p->d.error_word, (cudaStream_t)stream));
}

oomb_status oomb_kv_writeback(oomb_pool* p, const int32_t* sel, const int32_t* sel_count, int max_sel,
                              int stage_buf, int64_t first_page, int64_t end_page, void* stream) {
  if (!p || !sel || !sel_count || max_sel <= 0 || first_page < 0 || end_page < first_page) return OOMB_ERR_ARG;
  if (!p->d.offload) return OOMB_ERR_UNSUPPORTED;
  if (stage_buf < 0 || stage_buf > 1 || max_sel > p->d.stage_max_sel) return OOMB_ERR_ARG;
  if (!aligned(sel, 4) || !aligned(sel_count, 4)) return OOMB_ERR_ALIGN;
  const int lo = (int)std::min<int64_t>(first_page, INT32_MAX), hi = (int)std::min<int64_t>(end_page, INT32_MAX);
  return cuda_status(launch_prefetch(p->g, p->d.k_pool, p->d.v_pool, p->d.page_table, sel, sel_count, max_sel,
                                     p->d.stage_k, p->d.stage_v, stage_buf * p->g.Hkv, p->d.stage_max_sel, lo, hi,
                                     p->d.error_word, (cudaStream_t)stream, 1));
}

oomb_status oomb_prefetch(oomb_pool* p, const int32_t* sel, const int32_t* sel_count, int max_sel, int stage_buf,
                          void* stream) {
  return oomb_prefetch_pages(p, sel, sel_count, max_sel, stage_buf, 0, INT32_MAX, stream);
}

// Shared checks of the gradient staging calls.
static oomb_status check_grad_call(const oomb_pool* p, const int32_t* sel, const int32_t* sel_count, int max_sel,
                                   int stage_buf) {
  if (!p || !sel || !sel_count || max_sel <= 0) return OOMB_ERR_ARG;
  if (!p->d.offload_grads) return OOMB_ERR_UNSUPPORTED;
  if (stage_buf < 0 || stage_buf > 1 || max_sel > p->d.stage_max_sel) return OOMB_ERR_ARG;
  if (!aligned(sel, 4) || !aligned(sel_count, 4)) return OOMB_ERR_ALIGN;
  return OOMB_OK;
}

oomb_status oomb_grad_prefetch(oomb_pool* p, const int32_t* sel, const int32_t* sel_count, int max_sel,
                               const int32_t* prev_sel, const int32_t* prev_count, int stage_buf, void* stream) {
  oomb_status s = check_grad_call(p, sel, sel_count, max_sel, stage_buf);
  if (s != OOMB_OK) return s;
  if ((prev_sel == nullptr) != (prev_count == nullptr)) return OOMB_ERR_ARG;
  if (!aligned(prev_sel, 4) || !aligned(prev_count, 4)) return OOMB_ERR_ALIGN;
  return cuda_status(launch_grad_copy(p->g, kGradFromHost, p->d.dk_pool, p->d.dv_pool, p->d.grad_state, p->d.page_table, sel,
                                      sel_count, prev_sel, prev_count, max_sel, p->d.stage_dk, p->d.stage_dv,
                                      stage_buf, p->d.stage_max_sel, p->d.error_word, (cudaStream_t)stream));
}

oomb_status oomb_grad_carry(oomb_pool* p, const int32_t* sel, const int32_t* sel_count, int max_sel,
                            const int32_t* prev_sel, const int32_t* prev_count, int stage_buf, void* stream) {
  oomb_status s = check_grad_call(p, sel, sel_count, max_sel, stage_buf);
  if (s != OOMB_OK) return s;
  if (!prev_sel || !prev_count) return OOMB_ERR_ARG;
  if (!aligned(prev_sel, 4) || !aligned(prev_count, 4)) return OOMB_ERR_ALIGN;
  return cuda_status(launch_grad_copy(p->g, kGradCarry, p->d.dk_pool, p->d.dv_pool, p->d.grad_state, p->d.page_table, sel,
                                      sel_count, prev_sel, prev_count, max_sel, p->d.stage_dk, p->d.stage_dv,
                                      stage_buf, p->d.stage_max_sel, p->d.error_word, (cudaStream_t)stream));
}

oomb_status oomb_grad_writeback(oomb_pool* p, const int32_t* sel, const int32_t* sel_count, int max_sel,
                                int stage_buf, void* stream) {
  oomb_status s = check_grad_call(p, sel, sel_count, max_sel, stage_buf);
  if (s != OOMB_OK) return s;
  return cuda_status(launch_grad_copy(p->g, kGradToHost, p->d.dk_pool, p->d.dv_pool, p->d.grad_state, p->d.page_table, sel,
                                      sel_count, nullptr, nullptr, max_sel, p->d.stage_dk, p->d.stage_dv, stage_buf,
                                      p->d.stage_max_sel, p->d.error_word, (cudaStream_t)stream));
}

oomb_status oomb_grad_gather(oomb_pool* p, int64_t first_token, int n_tokens, float* dk, float* dv, void* stream) {
  if (!p || !dk || !dv || n_tokens <= 0 || first_token < 0) return OOMB_ERR_ARG;
  if (first_token + n_tokens > p->n_tokens) return OOMB_ERR_ARG;
  if (!aligned(dk, 16) || !aligned(dv, 16)) return OOMB_ERR_ALIGN;
  return cuda_status(launch_grad_gather(p->g, p->d.dk_pool, p->d.dv_pool, p->d.page_table, first_token, n_tokens,
                                        dk, dv, p->d.error_word, (cudaStream_t)stream));
}

oomb_status oomb_pool_set_stage(oomb_pool* p, int stage_buf) {
  if (!p || stage_buf < 0 || stage_buf > 1) return OOMB_ERR_ARG;
  if (!p->d.offload) return OOMB_ERR_UNSUPPORTED;
  p->stage_buf = stage_buf;
  return OOMB_OK;
}

oomb_status oomb_check(oomb_pool* p, void* stream, uint32_t* bits_out) {
  if (!p) return OOMB_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t bits = 0;
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpy(&bits, p->d.error_word, sizeof(bits), cudaMemcpyDeviceToHost);
  // after an error the whole control block is cleared: a selection that gave up
  // at a grid barrier may have left a counter behind
  if (e == cudaSuccess && bits) {
    e = cudaMemset(p->d.error_word, 0, OOMB_CTRL_WORDS * sizeof(uint32_t));
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (bits_out) *bits_out = bits;
  if (e != cudaSuccess) return cuda_status(e);
  if (bits & OOMB_DEVERR_TIMEOUT) return OOMB_ERR_TIMEOUT;
  return bits ? OOMB_ERR_KERNEL : OOMB_OK;
}

}  // extern "C"
