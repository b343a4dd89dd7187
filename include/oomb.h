/*
 * oomb.h -- C ABI of the paged sparse chunk-attention library (liboomb.so).
 *
 * The operations are those of OOMB's chunk-recurrent long-context training
 * ("Out of the Memory Barrier: A Highly Memory Efficient Training System for LLMs
 * with Million-Token Contexts"; gist.science explainer, section 2 "Methodology"):
 * one query chunk attends, causally and with grouped KV heads, to the keys of a
 * paged KV cache that holds every earlier chunk, restricted to the top-K pages
 * chosen by a mean-key page summary plus the sink page and the chunk's own pages;
 * the backward pass recomputes the attention probabilities, writes dQ and adds
 * dK/dV in place into a paged fp32 gradient pool that shares the KV page table.
 *
 * Conventions shared by every call
 *  - Ownership: the caller allocates and owns every buffer named in
 *    oomb_pool_desc and every argument pointer.  The library owns only the opaque
 *    oomb_pool object (host memory: free list and a host copy of the page table).
 *    No call allocates device memory.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call is stream-ordered and asynchronous unless stated.
 *  - Errors: every call checks its arguments on the host and returns a status;
 *    nothing aborts, throws across the ABI or traps on the device.  Kernels that
 *    meet a bad page-table entry or selection index, or whose bounded waits run
 *    out, set bits in the caller's device error word and skip the access;
 *    oomb_check() reads and clears that word.
 *  - Layouts (row-major, innermost last):
 *      K/V of a chunk      [n_tokens, Hkv, d]        (token-major, dtype)
 *      Q, O, dO, dQ        [n_q, Hq, d]              (token-major, dtype)
 *      LSE                 [Hq, n_q] fp32            (natural log)
 *      K/V pools           [num_phys, Hkv, P, d]     (dtype)
 *      dK/dV pools         [num_phys, Hkv, P, d]     fp32
 *      page summary        [num_phys, Hkv, d]        fp32 (mean key)
 *      page table          [max_logical_pages] int32 (logical -> physical, -1 unmapped)
 *      selection           sel [Hkv, max_sel] int32 (logical pages, ascending),
 *                          sel_count [Hkv] int32
 *    Query head hq uses KV head hq / (Hq / Hkv).
 *  - Alignment: every pointer 16-byte aligned; pools 1024-byte aligned for the
 *    bf16 tensor-core path.  Appends start on a page boundary.
 *  - Supported shapes: fp32 with head_dim <= 128 (multiple of 4), any page size
 *    up to 256; bf16 with head_dim <= 128 (multiple of 8).  bf16 with head_dim 128
 *    and page size 128 runs on the tcgen05 tensor-core kernels; other bf16 shapes
 *    on the SIMT kernels.
 *  - Thread safety: one pool must not be used from two host threads at once.
 */
#ifndef OOMB_H
#define OOMB_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define OOMB_API __attribute__((visibility("default")))
#else
#define OOMB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OOMB_OK = 0,
  OOMB_ERR_ARG = 1,          /* bad argument (null pointer, size, shape) */
  OOMB_ERR_OUT_OF_PAGES = 2, /* the free list cannot cover the append */
  OOMB_ERR_ALIGN = 3,        /* pointer or token offset misaligned */
  OOMB_ERR_DTYPE = 4,        /* unknown dtype */
  OOMB_ERR_KERNEL = 5,       /* a kernel raised the device error word */
  OOMB_ERR_TIMEOUT = 6,      /* a bounded device wait gave up */
  OOMB_ERR_CUDA = 7,         /* a CUDA runtime call failed */
  OOMB_ERR_UNSUPPORTED = 8,  /* valid but not implemented (shape/dtype/device) */
  OOMB_ERR_WORKSPACE = 9     /* workspace missing or too small */
} oomb_status;

typedef enum { OOMB_BF16 = 0, OOMB_FP32 = 1 } oomb_dtype;

/* Operation selector for oomb_workspace_size. */
typedef enum { OOMB_OP_SELECT = 0, OOMB_OP_BWD = 1 } oomb_op;

/* Device error-word bits (see oomb_check). */
#define OOMB_DEVERR_TIMEOUT 0x1u  /* an mbarrier wait ran out */
#define OOMB_DEVERR_PAGE 0x2u     /* page table entry unmapped / out of range */
#define OOMB_DEVERR_SEL 0x4u      /* selection index out of range */
#define OOMB_DEVERR_TMEM 0x8u     /* tensor-memory allocation failed */
#define OOMB_DEVERR_SMEM 0x10u    /* a kernel's shared-memory window is not 1 KB aligned (nothing computed) */

/* Length of the pool's control block (oomb_pool_desc.error_word), in uint32.
 * Word 0 holds the error bits above; words 4..5 are the grid-barrier counters of
 * oomb_page_select.  Each barrier's arrivals add exactly 2^31 to its counter
 * (sense reversal), so the counters return to a state with zero low 31 bits
 * after every selection and the host keeps no barrier state: a selection can be
 * captured in a CUDA graph and replayed.  The counters are per pool, so page
 * selections on one pool must not run concurrently (issue them on one stream,
 * or order them with events). */
#define OOMB_CTRL_WORDS 16

typedef struct {
  int n_q_heads;         /* Hq */
  int n_kv_heads;        /* Hkv; Hq % Hkv == 0 */
  int head_dim;          /* d */
  int page_size;         /* P, tokens per page */
  int num_phys_pages;    /* pages in each pool */
  int max_logical_pages; /* entries of page_table */
  int dtype;             /* oomb_dtype of K/V pools, Q, O, dO, dQ */
  void* k_pool;          /* [num_phys, Hkv, P, d]; device, or pinned+mapped host if offload */
  void* v_pool;          /* same */
  float* dk_pool;        /* [num_phys, Hkv, P, d] fp32; device, or pinned+mapped host
                            if offload_grads */
  float* dv_pool;        /* same */
  float* summary;        /* [num_phys, Hkv, d] fp32 device */
  int32_t* page_table;   /* [max_logical_pages] device; written by the library */
  uint32_t* error_word;  /* control block: OOMB_CTRL_WORDS device uint32, all zero
                            at creation; 16-byte aligned */
  const int32_t* page_order; /* optional host [num_phys]: order in which physical
                                pages are handed out (copied at creation); NULL = 0..n-1 */
  int offload;           /* 1: k_pool/v_pool live in pinned host memory and the
                            attention kernels read selected pages from staging */
  void* stage_k;         /* offload only: [2, Hkv, stage_max_sel, P, d] device */
  void* stage_v;         /* same */
  int stage_max_sel;     /* offload only: selection capacity per KV head */
  int offload_grads;     /* 1 (needs offload = 1): dk_pool/dv_pool live in pinned host
                            memory too; the backward adds into the staged blocks
                            stage_dk/stage_dv, which oomb_grad_prefetch/carry fill and
                            oomb_grad_writeback returns to the host pools */
  float* stage_dk;       /* offload_grads only: [2, Hkv, stage_max_sel, P, d] fp32 device */
  float* stage_dv;       /* same */
  uint8_t* grad_state;   /* offload_grads only: [num_phys, Hkv] device bytes, owned by the
                            library: 0 = the host gradient block holds nothing yet (its
                            page was appended and no write-back has reached it; it counts
                            as zero and the append does not write the host block), 1 = the
                            host block holds the gradient written back last */
} oomb_pool_desc;

typedef struct oomb_pool oomb_pool;

/* Validate `desc`, copy it and build the free list.  Touches no device memory:
 * the page table is filled with -1 on the stream of the first append (or
 * reset).  On success *out owns a host object that oomb_pool_destroy frees. */
OOMB_API oomb_status oomb_pool_create(const oomb_pool_desc* desc, oomb_pool** out);
OOMB_API void oomb_pool_destroy(oomb_pool* pool);

/* Return every page to the free list, in the creation order, and set every
 * page-table entry to -1 (stream-ordered).  The pools' contents are kept. */
OOMB_API oomb_status oomb_pool_reset(oomb_pool* pool, void* stream);

/* Offload mode: oomb_kv_append, and the new pages also written into staging buffer
 * stage_buf at the slots of the chunk's own pages, so that the chunk's attention
 * needs only its history pages from host memory (oomb_prefetch_pages up to the
 * chunk's first page).  The chunk's selection (top-K or window, computed before the
 * append: a selection needs only the history) lists the own pages last: own page j
 * of n_own goes to slot sel_count[h] - n_own + j of KV head h.  The append must
 * cover exactly the chunk's tokens.  max_sel: the selection's row length (<=
 * stage_max_sel).  A count smaller than n_own or above max_sel sets OOMB_DEVERR_SEL
 * and that head's pages are not staged.
 * Errors: those of oomb_kv_append, UNSUPPORTED (pool not in offload mode). */
OOMB_API oomb_status oomb_kv_append_staged(oomb_pool* pool, const void* k, const void* v, int64_t first_token,
                                           int n_tokens, const int32_t* sel_count, int max_sel, int stage_buf,
                                           void* stream);

/* oomb_kv_append_staged without the host write: the new pages go to their staging
 * slots only (plus the page table, summaries and grad_state, all in device memory),
 * so the append on the critical path touches no host memory; the host pool blocks
 * are written afterwards by oomb_kv_writeback, e.g. on the side stream while the
 * chunk's forward runs (explainer 2.C: transfers hidden behind computation).  Until
 * that write-back has run, the host pools do not hold the chunk's pages: order it
 * before any oomb_prefetch / oomb_prefetch_pages that reads them, and before the
 * staging slots are written again.  Errors: those of oomb_kv_append_staged. */
OOMB_API oomb_status oomb_kv_append_deferred(oomb_pool* pool, const void* k, const void* v, int64_t first_token,
                                             int n_tokens, const int32_t* sel_count, int max_sel, int stage_buf,
                                             void* stream);

/* The reverse of oomb_prefetch_pages: every selected block of a page in
 * [first_page, end_page) is copied from staging buffer stage_buf to its block of
 * the host K/V pools.  Used after oomb_kv_append_deferred with the chunk's own pages
 * as the range.  Errors: ARG, ALIGN, UNSUPPORTED (not an offload pool), CUDA. */
OOMB_API oomb_status oomb_kv_writeback(oomb_pool* pool, const int32_t* sel, const int32_t* sel_count, int max_sel,
                                       int stage_buf, int64_t first_page, int64_t end_page, void* stream);

/* Return logical pages [first_logical_page, first_logical_page + n_pages) to the
 * free list (explainer 2.B: fixed-size pages; "3. Key Contributions": paged
 * memory without fragmentation).  Every page of the range must be mapped (already
 * appended and not yet freed).  Their page-table entries become -1 on `stream`
 * and their physical pages are handed out first by the next appends (lowest
 * logical page first); the pool's token count is unchanged, so later appends
 * continue at the end.  oomb_page_select leaves freed pages out (they are neither
 * sinks nor candidates).  The attention kernels flag an unmapped page in a caller's
 * selection (OOMB_DEVERR_PAGE) and skip it, and oomb_window_select does not look at
 * the table, so with a local window free only the pages behind it.
 * Errors: ARG (range outside the appended pages, or a page not mapped), CUDA
 * (nothing changes on the host). */
OOMB_API oomb_status oomb_page_free(oomb_pool* pool, int64_t first_logical_page, int n_pages, void* stream);

/* Paged KV append (explainer 2.B "Paged KV Cache and Gradient Management"; the
 * lay summary's "Trick A": each chunk's KV drops onto the next free page, no
 * copying of earlier pages).  Opens ceil((first_token+n)/P) - first_token/P new
 * logical pages, taking physical pages from the free list and writing their
 * page-table entries; copies k, v ([n_tokens, Hkv, d], dtype, device) into the
 * pools; zeroes the dK/dV rows of the written tokens (with offload_grads: marks
 * the pages' host gradient blocks as holding nothing yet, see grad_state); writes
 * the page summary
 * (fp32 mean key over the tokens present) of every touched page.
 * first_token must equal the tokens already appended and be a multiple of P.
 * Errors: ARG, ALIGN, OUT_OF_PAGES (nothing is written), CUDA. */
OOMB_API oomb_status oomb_kv_append(oomb_pool* pool, const void* k, const void* v, int64_t first_token, int n_tokens,
                           void* stream);

/* Page selection for one query chunk (explainer 2.D "Page-Level Sparse
 * Attention": top-K pages by a representative, averaged key).  With
 * qbar_h = mean of q over the chunk's n_q tokens and the G query heads of KV
 * head h, every complete history page p in [n_sink, q_start/P) is scored as
 * qbar_h . summary[phi(p), h]; the top_k highest scores are kept (ties to the
 * lower logical page), plus pages [0, n_sink) and the chunk's own pages
 * [q_start/P, ceil((q_start+n_q)/P)).  top_k < 0 keeps every page.  Pages freed
 * by oomb_page_free are skipped: a freed sink is dropped and the top_k is taken
 * over the mapped candidates (all of them when there are no more than top_k).
 * Output per KV head: ascending logical pages in sel[h*max_sel ...], count in
 * sel_count[h].  q: [n_q, Hq, d] device.  q_start must be a multiple of P and
 * every page before the chunk appended; the chunk's own K/V may come later (the
 * selection reads history pages only), so it can run before the chunk's K/V
 * projection.  Workspace: oomb_workspace_size(
 * OOMB_OP_SELECT, n_q) bytes of device memory, contents scratch.
 * Launch: one cooperative kernel (one CTA per SM) whose phases meet at grid
 * barriers kept in the pool's control block, so selections on one pool must be
 * ordered (one stream, or events).  No host state changes between calls, so the
 * call may be captured in a CUDA graph.  A barrier wait that runs out (~1 s) sets
 * OOMB_DEVERR_TIMEOUT; oomb_check reports it and clears the control block.
 * Errors: ARG (incl. max_sel below the mapped sinks + kept candidates + own
 * pages), ALIGN, WORKSPACE, CUDA. */
OOMB_API oomb_status oomb_page_select(oomb_pool* pool, const void* q, int64_t q_start, int n_q, int top_k, int n_sink,
                             int32_t* sel, int32_t* sel_count, int max_sel, void* workspace, size_t ws_bytes,
                             void* stream);

/* Where oomb_page_select_append writes the chunk's pages. */
typedef enum {
  OOMB_APPEND_POOL = 0,     /* the pools, as oomb_kv_append */
  OOMB_APPEND_STAGED = 1,   /* the pools and the staging slots, as oomb_kv_append_staged */
  OOMB_APPEND_DEFERRED = 2  /* the staging slots only, as oomb_kv_append_deferred */
} oomb_append_mode;

/* The selection of one chunk and the append of that chunk's own K/V in one launch
 * (explainer 2.D: pages are selected by their summaries; 2.B: the chunk's K/V go to
 * free pages).  Same results as oomb_page_select followed by the append named by
 * append_mode with k, v ([n_q, Hkv, d], first token q_start): the selection reads
 * only history pages and the append writes only the chunk's own pages, so when the
 * selection scores pages (more mapped candidates than top_k > 0) the selection's grid
 * also appends, before its query sum, with the append kernel's arithmetic (bit-
 * identical pools, summaries and slots); otherwise the two run as two launches.  The
 * own pages' staging slots need no selection result: the count of a top-K selection
 * is known beforehand (mapped sinks + min(top_k, mapped candidates) + own pages).
 * q_start must equal the tokens appended so far.  stage_buf: the staging buffer for
 * the STAGED and DEFERRED modes (offload pools only).  Errors: those of both calls;
 * nothing is appended when an error is returned. */
OOMB_API oomb_status oomb_page_select_append(oomb_pool* pool, const void* q, const void* k, const void* v,
                                            int64_t q_start, int n_q, int top_k, int n_sink, int32_t* sel,
                                            int32_t* sel_count, int max_sel, void* workspace, size_t ws_bytes,
                                            int append_mode, int stage_buf, void* stream);

/* oomb_page_select for callers that cannot allocate device memory.  The pages
 * describe no counterpart: this is a property of the library, not of the method.
 * Identical selection to oomb_page_select, but the scratch it needs comes from a
 * static device array of 4 MiB inside the library (held by every GPU that loads
 * the library until the process exits) instead of a caller workspace.  Meant for
 * callers that cannot call cudaMalloc: a framework that owns all device memory
 * through its own pool, a steady-state loop where allocation (which can
 * synchronize the device or fail under memory pressure) is forbidden, or a C host
 * with no allocator of its own.  The caller still passes q, sel and sel_count.
 *  - Limit: returns OOMB_ERR_WORKSPACE when oomb_workspace_size(pool,
 *    OOMB_OP_SELECT, n_q) exceeds 4 MiB (e.g. more than 225,280 logical pages at
 *    4 KV heads x head_dim 128).
 *  - Set-up: the first call on a device looks up the array's device address with
 *    cudaGetSymbolAddress while that device is current; make that first call
 *    before any stream capture.  The address is kept for the life of the process:
 *    after cudaDeviceReset (which destroys the context and the array with it) do
 *    not call this entry point again in that process.
 *  - Sharing: every call on a device uses the same array and leaves its contents
 *    behind; nothing in it needs to start at zero.  Calls that overlap on the GPU
 *    (different streams, or different host threads) race on the array: order
 *    them on one stream.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 * Errors: those of oomb_page_select, plus WORKSPACE (above the limit) and CUDA
 * (set-up failed). */
OOMB_API oomb_status oomb_page_select_noalloc(oomb_pool* pool, const void* q, int64_t q_start, int n_q, int top_k,
                                              int n_sink, int32_t* sel, int32_t* sel_count, int max_sel,
                                              void* stream);

/* Local sliding-window selection, the "local attention" that the explainer (2.D
 * "Page-Level Sparse Attention", native support for sparse-native models) pairs
 * with top-K retrieval: the sparse layers of such a model attend only to the
 * most recent context.  Page granularity, no scoring: with n_hist = q_start/P,
 * every KV head gets
 *     [0, min(n_sink, n_hist))                      sink pages (n_sink >= 0)
 *   U [max(n_sink', n_hist - window), n_hist)       the window history pages
 *                                                   right before the chunk
 *   U [n_hist, ceil((q_start + n_q)/P))             the chunk's own pages
 * ascending, in sel[h*max_sel ...] with the count in sel_count[h] (device,
 * int32; entries past the count are left as they were).  Feed the result to
 * oomb_chunk_attn_fwd/bwd (and oomb_prefetch) like a top-K selection.  Reads no
 * K/V and no workspace; one small kernel on the stream.  q_start must be a
 * multiple of P and every page before the chunk appended (the chunk's own K/V may
 * come later: the set is known before the chunk's K/V are).
 * Errors: ARG (window < 0, n_sink < 0, max_sel smaller than the set), ALIGN,
 * CUDA. */
OOMB_API oomb_status oomb_window_select(oomb_pool* pool, int64_t q_start, int n_q, int window, int n_sink,
                                        int32_t* sel, int32_t* sel_count, int max_sel, void* stream);

/* Chunk attention forward.  For query head hq and row i (absolute position
 * q_start+i): keys = every token of the selected pages of KV head hq/G with
 * position <= q_start+i; O_i = softmax(scale * q_i . k_j) V and
 * LSE_i = log sum_j exp(scale * q_i . k_j).  q/o: [n_q, Hq, d] device,
 * lse: [Hq, n_q] fp32 device.  sel/sel_count as written by oomb_page_select
 * (device).  In offload mode K/V are read from staging buffer
 * oomb_pool_set_stage(); the selection must equal the one prefetched.
 * Errors: ARG, ALIGN, UNSUPPORTED, CUDA. */
OOMB_API oomb_status oomb_chunk_attn_fwd(oomb_pool* pool, const void* q, int64_t q_start, int n_q, const int32_t* sel,
                                const int32_t* sel_count, int max_sel, float softmax_scale, void* o, float* lse,
                                void* stream);

/* Chunk attention backward with on-the-fly recomputation (explainer 2.A) and
 * in-place paged gradient accumulation (explainer 2.B).  With
 * P_ij = exp(scale q_i.k_j - LSE_i) over the forward's key set,
 * dP = dO V^T, D_i = dO_i . O_i, dS = P (dP - D):
 *   dq = scale dS K (written, dtype),
 *   dK_pool[phi(p), h] += scale dS^T Q,  dV_pool[phi(p), h] += P^T dO
 * summed over the G query heads of KV head h and every row of the chunk (with
 * offload_grads, into the staged blocks of buffer oomb_pool_set_stage()).
 * Summation order: dK/dV are partitioned by (page, KV head).  On the tensor-core
 * path (bf16, head_dim = page = 128) the work of a block is split over the 2-4
 * thread blocks of one cluster, whose partials are summed in a fixed order in
 * distributed shared memory and added once into the pool rows: no atomics on the
 * gradient pool, and dK/dV are bit-identical from run to run.  dq is accumulated
 * in fp32 across thread blocks with float reductions, so repeated runs agree to
 * rounding, not bit for bit.  The SIMT path (other shapes, fp32) gives each
 * gradient row one owner and is deterministic.  Backward calls on one pool must
 * be stream-ordered.  The selection is checked on the device (count within
 * [0, max_sel], entries strictly ascending and inside the chunk's view); a bad one
 * sets OOMB_DEVERR_SEL and the affected pages are skipped, as in the forward.
 * Workspace: oomb_workspace_size(OOMB_OP_BWD, n_q) bytes, contents scratch.
 * Errors: ARG, ALIGN, WORKSPACE, UNSUPPORTED, CUDA. */
OOMB_API oomb_status oomb_chunk_attn_bwd(oomb_pool* pool, const void* q, const void* o, const void* d_o, const float* lse,
                                int64_t q_start, int n_q, const int32_t* sel, const int32_t* sel_count, int max_sel,
                                float softmax_scale, void* dq, void* workspace, size_t ws_bytes, void* stream);

/* Offload mode (explainer 2.C "Asynchronous KV Cache CPU Offloading"): copy the
 * selected (page, KV head) blocks of K and V from the pinned host pools into
 * staging buffer `stage_buf` (0 or 1) on `stream` (normally a side stream;
 * order it against the attention calls with CUDA events).  Block s of KV head h
 * lands in slot (stage_buf, h, s).  Errors: ARG, ALIGN (selection not 4-byte
 * aligned), UNSUPPORTED (pool not in offload mode), CUDA. */
OOMB_API oomb_status oomb_prefetch(oomb_pool* pool, const int32_t* sel, const int32_t* sel_count, int max_sel,
                          int stage_buf, void* stream);

/* Gradient offload (explainer 2.C: the KV cache and its gradients are moved
 * between CPU and GPU memory; 2.B: gradient pages share the KV page table).  Needs offload_grads.
 * In the reverse sweep the backward of chunk c adds into the staged dK/dV blocks
 * of its selection (staging buffer c % 2, slot (h, s) as for K/V).  The three
 * calls below fill and drain those slots; `prev_sel/prev_count` is the selection
 * of the chunk whose backward ran just before (chunk c + 1, staged in buffer
 * 1 - stage_buf), NULL for the first chunk of the sweep.  max_sel is the row
 * length of sel and of prev_sel.
 *
 * oomb_grad_prefetch: stage the blocks of `sel` whose page is not in prev_sel
 * from the host pools into buffer stage_buf (zero-filled where grad_state is 0).  Those host blocks are final with
 * respect to the previous chunk, so this may run while the previous chunk's
 * backward runs (order it after the previous write-backs: same stream).
 * Errors: ARG, ALIGN, UNSUPPORTED (no offload_grads), CUDA. */
OOMB_API oomb_status oomb_grad_prefetch(oomb_pool* pool, const int32_t* sel, const int32_t* sel_count, int max_sel,
                                        const int32_t* prev_sel, const int32_t* prev_count, int stage_buf,
                                        void* stream);

/* oomb_grad_carry: copy the blocks of `sel` whose page is also in prev_sel from
 * the previous chunk's staging buffer (1 - stage_buf) into buffer stage_buf, so
 * that they carry the previous chunk's contribution without a round trip through
 * host memory.  Must run after the previous chunk's backward and before this
 * chunk's.  Errors: those of oomb_grad_prefetch (prev_sel is required). */
OOMB_API oomb_status oomb_grad_carry(oomb_pool* pool, const int32_t* sel, const int32_t* sel_count, int max_sel,
                                     const int32_t* prev_sel, const int32_t* prev_count, int stage_buf,
                                     void* stream);

/* oomb_grad_writeback: write every staged dK/dV block of `sel` (buffer stage_buf)
 * back to its block of the host pools and set its grad_state to 1.  Must run after this chunk's backward and
 * before any later oomb_grad_prefetch that reads those pages (one side stream
 * keeps that order) and before buffer stage_buf is filled again.
 * Errors: those of oomb_grad_prefetch. */
OOMB_API oomb_status oomb_grad_writeback(oomb_pool* pool, const int32_t* sel, const int32_t* sel_count, int max_sel,
                                         int stage_buf, void* stream);

/* oomb_prefetch restricted to the selected pages in [first_page, end_page): e.g.
 * the history pages of a chunk while its K/V projection runs (explainer 2.C: the
 * sparse transfers overlap the K/V projection; for local layers, one layer ahead),
 * then its own pages once they are appended.  Errors: those of oomb_prefetch. */
OOMB_API oomb_status oomb_prefetch_pages(oomb_pool* pool, const int32_t* sel, const int32_t* sel_count, int max_sel,
                                         int stage_buf, int64_t first_page, int64_t end_page, void* stream);

/* Offload mode: staging buffer that following attention calls read (K/V, and
 * with offload_grads the dK/dV blocks the backward adds into). */
OOMB_API oomb_status oomb_pool_set_stage(oomb_pool* pool, int stage_buf);

/* ---------------------------------------------------------------- layer step
 * The chunk-recurrent layer step around the attention path (explainer 2.A: the
 * chunk's activations are recomputed in the reverse sweep; its K/V gradients, final
 * once every later chunk has run its backward, flow back through the rotary
 * embedding and the projections Q = X Wq + bq, K = X Wk + bk, V = X Wv + bv). */

/* C[m, n] = alpha op(A) op(B) + beta C, row-major: op(A) is A stored [m, k]
 * (trans_a = 0) or the transpose of A stored [k, m]; op(B) is B stored [k, n] or the
 * transpose of B stored [n, k]; C is [m, n].  A and B are dtype_ab (OOMB_BF16 or
 * OOMB_FP32, both alike), C is dtype_c; fp32 accumulation, and fp32 operands are
 * multiplied in full fp32 (no TF32).  A plain library GEMM (cuBLASLt) on `stream`,
 * with the caller's device workspace (ws_bytes may be 0; 32 MiB lets every
 * algorithm run); the first call on a device creates a cuBLASLt handle (a host
 * object kept until exit).  Pointers 16-byte aligned.
 * Errors: ARG, DTYPE, ALIGN, UNSUPPORTED (no algorithm for the shape), CUDA. */
OOMB_API oomb_status oomb_gemm(int m, int n, int k, int trans_a, int trans_b, const void* a, const void* b, void* c,
                               int dtype_ab, int dtype_c, float alpha, float beta, void* workspace, size_t ws_bytes,
                               void* stream);

/* out[i, h, :] = R(pos0 + i) (in[i, h, :] + bias[h, :]) for token rows i < n and heads
 * h < H of a token-major [n, H, d] tensor (in may be a [n, H*d] GEMM output: the same
 * memory).  R(t) is the rotate-half rotary embedding: each pair (j, j + d/2) turned by
 * the angle t * theta^(-2j/d) (mode 1), by minus that angle (mode 2: the transpose,
 * which carries gradients back), or not at all (mode 0: bias and cast only).  bias:
 * fp32 [H*d] or NULL; in_dtype/out_dtype OOMB_BF16 or OOMB_FP32; in == out is allowed
 * for equal dtypes.  The angles' cos/sin are computed in double precision.
 * Errors: ARG (odd d, d > 128, theta <= 1 with a rotation), DTYPE, ALIGN (in, out or
 * bias not on a multiple of its element size), CUDA. */
OOMB_API oomb_status oomb_bias_rope(const void* in, int in_dtype, const float* bias, void* out, int out_dtype, int n,
                                    int H, int d, int64_t pos0, float theta, int mode, void* stream);

/* dK, dV of tokens [first_token, first_token + n_tokens) read from the paged fp32
 * gradient pool through the page table into token-major [n_tokens, Hkv, d] fp32
 * (device).  With offload_grads the pools are in host memory and are read there: the
 * blocks must have been written back (order the call after oomb_grad_writeback).
 * An unmapped page sets OOMB_DEVERR_PAGE and its rows read as zero.
 * Errors: ARG (range beyond the appended tokens), ALIGN, CUDA. */
OOMB_API oomb_status oomb_grad_gather(oomb_pool* pool, int64_t first_token, int n_tokens, float* dk, float* dv,
                                      void* stream);

/* Bytes of device workspace `op` needs for a chunk of n_q queries (0 on error). */
OOMB_API size_t oomb_workspace_size(const oomb_pool* pool, int op, int n_q);

/* Synchronize `stream`, read and clear the device error word.  Returns OK,
 * KERNEL (bits in *bits_out if non-NULL) or CUDA. */
OOMB_API oomb_status oomb_check(oomb_pool* pool, void* stream, uint32_t* bits_out);

/* Host copy of the page table (n entries from logical page 0). Returns entries copied. */
OOMB_API int oomb_page_table_host(const oomb_pool* pool, int32_t* out, int n);

/* Tokens appended so far and free pages left. */
OOMB_API int64_t oomb_pool_tokens(const oomb_pool* pool);
OOMB_API int oomb_pool_free_pages(const oomb_pool* pool);

OOMB_API const char* oomb_status_str(oomb_status s);

/* Text of the last CUDA runtime error a call of this library returned
 * OOMB_ERR_CUDA for on the calling host thread ("" if none). */
OOMB_API const char* oomb_last_cuda_error(void);

/* Kernels this library has launched since it was loaded (all pools, all devices). */
OOMB_API uint64_t oomb_launch_count(void);

/* Which attention kernels a call with this pool would use: 1 = tcgen05, 0 = SIMT. */
OOMB_API int oomb_uses_tensor_cores(const oomb_pool* pool);

#ifdef __cplusplus
}
#endif
#endif /* OOMB_H */
