"""CPU-only checks of the C ABI: the library builds, loads, exports every symbol
include/oomb.h declares, and its host-side argument checks and page allocator
answer without touching a GPU (pointers below are never dereferenced)."""
import ctypes as C

import pytest

import paged_sparse_attention_gb300 as L
from paged_sparse_attention_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return L.load()


def test_exports_every_declared_symbol(lib):
    names = L.header_symbols()
    assert len(names) >= 16
    for n in ["oomb_kv_append", "oomb_page_select", "oomb_chunk_attn_fwd", "oomb_chunk_attn_bwd",
              "oomb_prefetch"]:
        assert n in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for s in range(10):
        assert lib.oomb_status_str(s)
    assert lib.oomb_status_str(2) == b"out of pages"


def _desc(**kw):
    d = _lib.PoolDesc()
    d.n_q_heads, d.n_kv_heads, d.head_dim, d.page_size = 28, 4, 128, 128
    d.num_phys_pages, d.max_logical_pages, d.dtype = 4, 8, _lib.OOMB_BF16
    fake = 1 << 20
    for i, f in enumerate(["k_pool", "v_pool", "dk_pool", "dv_pool", "summary", "page_table", "error_word"]):
        setattr(d, f, fake * (i + 1))
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_pool_create_validation(lib):
    h = C.c_void_p()
    assert lib.oomb_pool_create(C.byref(_desc(dtype=7)), C.byref(h)) == 4
    assert lib.oomb_pool_create(C.byref(_desc(n_kv_heads=3)), C.byref(h)) == 1
    assert lib.oomb_pool_create(C.byref(_desc(head_dim=256)), C.byref(h)) == 8
    assert lib.oomb_pool_create(C.byref(_desc(k_pool=(1 << 20) + 4)), C.byref(h)) == 3
    assert lib.oomb_pool_create(C.byref(_desc(summary=None)), C.byref(h)) == 1
    assert lib.oomb_pool_create(C.byref(_desc(page_table=(6 << 20) + 2)), C.byref(h)) == 3
    bad_order = (C.c_int32 * 4)(0, 1, 1, 2)
    assert lib.oomb_pool_create(C.byref(_desc(page_order=C.addressof(bad_order))), C.byref(h)) == 1
    assert lib.oomb_pool_create(C.byref(_desc(offload=1)), C.byref(h)) == 1  # no staging buffers


def test_offload_pool_host_checks(lib):
    """An offload pool (staging buffers given): the stage buffer index and max_sel
    against the staging capacity are checked before any device work."""
    h = C.c_void_p()
    d = _desc(offload=1, stage_max_sel=8, stage_k=1 << 26, stage_v=1 << 27)
    assert lib.oomb_pool_create(C.byref(d), C.byref(h)) == 0
    pool = h.value
    fake = 1 << 24
    for fn in (lib.oomb_kv_append_staged, lib.oomb_kv_append_deferred):
        assert fn(pool, fake, fake, 0, 128, fake, 8, 2, None) == 1  # stage buffer 2
        assert fn(pool, fake, fake, 0, 128, fake, 9, 0, None) == 1  # max_sel above the staging capacity
        assert fn(pool, fake, fake, 0, 128, fake + 2, 8, 0, None) == 3  # misaligned counts
    assert lib.oomb_kv_writeback(pool, fake, fake, 8, 2, 0, 1, None) == 1
    assert lib.oomb_kv_writeback(pool, fake, fake, 9, 0, 0, 1, None) == 1
    assert lib.oomb_prefetch_pages(pool, fake, fake, 8, 0, 3, 2, None) == 1
    assert lib.oomb_prefetch(pool, fake + 2, fake, 8, 0, None) == 3  # misaligned selection
    assert lib.oomb_kv_writeback(pool, fake, fake + 1, 8, 0, 0, 1, None) == 3
    sa = lib.oomb_page_select_append
    for mode in (1, 2):  # staged and deferred: the stage buffer and max_sel against the capacity
        assert sa(pool, fake, fake, fake, 0, 128, 4, 1, fake, fake, 8, fake, 1 << 30, mode, 2, None) == 1
        assert sa(pool, fake, fake, fake, 0, 128, 4, 1, fake, fake, 9, fake, 1 << 30, mode, 0, None) == 1
    assert lib.oomb_pool_free_pages(pool) == 4  # nothing was taken
    lib.oomb_pool_destroy(pool)


def test_allocator_host_logic(lib):
    order = (C.c_int32 * 4)(2, 0, 3, 1)
    h = C.c_void_p()
    assert lib.oomb_pool_create(C.byref(_desc(page_order=C.addressof(order))), C.byref(h)) == 0
    pool = h.value
    assert lib.oomb_pool_free_pages(pool) == 4 and lib.oomb_pool_tokens(pool) == 0
    fake = 1 << 24
    # misaligned start, non-contiguous start, too many pages: refused before any device work
    assert lib.oomb_kv_append(pool, fake, fake, 64, 128, None) == 1
    assert lib.oomb_kv_append(pool, fake, fake, 0, 5 * 128, None) == 2
    assert lib.oomb_kv_append(pool, fake + 8, fake, 0, 128, None) == 3
    assert lib.oomb_pool_free_pages(pool) == 4
    # chunk-level calls before the chunk's K/V exist
    assert lib.oomb_chunk_attn_fwd(pool, fake, 0, 128, fake, fake, 8, 0.1, fake, fake, None) == 1
    # a selection needs the history only (its chunk's own K/V may come later): a chunk
    # that starts after the appended tokens is refused
    assert lib.oomb_page_select(pool, fake, 128, 128, 4, 1, fake, fake, 8, fake, 1 << 30, None) == 1
    assert lib.oomb_window_select(pool, 128, 128, 2, 1, fake, fake, 8, None) == 1  # history not appended
    assert lib.oomb_page_select(pool, fake, 0, 256, 4, 1, fake, fake, 1, fake, 1 << 30, None) == 1  # max_sel < own
    assert lib.oomb_page_free(pool, 0, 1, None) == 1  # nothing appended yet
    assert lib.oomb_page_free(pool, -1, 1, None) == 1 and lib.oomb_page_free(pool, 0, 0, None) == 1
    assert lib.oomb_window_select(pool, 0, 128, -1, 1, fake, fake, 8, None) == 1  # negative window
    assert lib.oomb_window_select(pool, 64, 128, 2, 1, fake, fake, 8, None) == 3  # start not on a page
    assert lib.oomb_prefetch(pool, fake, fake, 8, 0, None) == 8  # not an offload pool
    # the staged and deferred appends and the K/V write-back need an offload pool
    assert lib.oomb_kv_append_staged(pool, fake, fake, 0, 128, fake, 8, 0, None) == 8
    assert lib.oomb_kv_append_deferred(pool, fake, fake, 0, 128, fake, 8, 0, None) == 8
    assert lib.oomb_kv_writeback(pool, fake, fake, 8, 0, 0, 1, None) == 8
    assert lib.oomb_kv_writeback(pool, fake, fake, 8, 0, 2, 1, None) == 1  # end before start
    assert lib.oomb_kv_writeback(pool, None, fake, 8, 0, 0, 1, None) == 1
    assert lib.oomb_pool_set_stage(pool, 0) == 8
    # the selection fused with the chunk's append: the append mode, the pool kind and
    # the chunk's start (its K/V are appended by this call) are checked first
    sa = lib.oomb_page_select_append
    assert sa(pool, fake, fake, fake, 0, 128, 4, 1, fake, fake, 8, fake, 1 << 30, 3, 0, None) == 1
    assert sa(pool, fake, fake, fake, 0, 128, 4, 1, fake, fake, 8, fake, 1 << 30, -1, 0, None) == 1
    assert sa(pool, fake, fake, fake, 0, 128, 4, 1, fake, fake, 8, fake, 1 << 30, 1, 0, None) == 8
    assert sa(pool, fake, fake, fake, 0, 128, 4, 1, fake, fake, 8, fake, 1 << 30, 2, 0, None) == 8
    assert sa(pool, fake, fake, fake, 128, 128, 4, 1, fake, fake, 8, fake, 1 << 30, 0, 0, None) == 1
    assert sa(None, fake, fake, fake, 0, 128, 4, 1, fake, fake, 8, fake, 1 << 30, 0, 0, None) == 1
    assert lib.oomb_pool_free_pages(pool) == 4  # nothing was taken
    assert lib.oomb_workspace_size(pool, 0, 4096) > 0
    assert lib.oomb_workspace_size(pool, 1, 4096) >= 28 * 4096 * 4
    assert lib.oomb_workspace_size(pool, 9, 4096) == 0
    tab = (C.c_int32 * 8)()
    assert lib.oomb_page_table_host(pool, tab, 8) == 8 and list(tab) == [-1] * 8
    lib.oomb_pool_destroy(pool)


def test_gradient_transfer_host_checks(lib):
    """An offload pool with host-resident gradient pools: the gradient stage-in, carry
    and write-back check the stage buffer, the staging capacity and the alignment of
    both selections (this chunk's and the previous chunk's) before any device work."""
    h = C.c_void_p()
    d = _desc(offload=1, offload_grads=1, stage_max_sel=8, stage_k=1 << 26, stage_v=1 << 27,
              stage_dk=1 << 28, stage_dv=1 << 29, grad_state=1 << 30)
    assert lib.oomb_pool_create(C.byref(d), C.byref(h)) == 0
    pool = h.value
    fake = 1 << 24
    for fn in (lib.oomb_grad_prefetch, lib.oomb_grad_carry):
        assert fn(pool, fake, fake, 8, fake, fake, 2, None) == 1        # stage buffer 2
        assert fn(pool, fake, fake, 9, fake, fake, 0, None) == 1        # above the staging capacity
        assert fn(pool, fake + 2, fake, 8, fake, fake, 0, None) == 3    # misaligned selection
        assert fn(pool, fake, fake, 8, fake + 2, fake, 0, None) == 3    # misaligned previous selection
        assert fn(pool, fake, fake, 8, fake, fake + 1, 0, None) == 3    # misaligned previous counts
    assert lib.oomb_grad_prefetch(pool, fake, fake, 8, fake, None, 0, None) == 1  # one of the pair
    assert lib.oomb_grad_carry(pool, fake, fake, 8, None, None, 0, None) == 1     # carry needs prev
    assert lib.oomb_grad_writeback(pool, fake, fake, 8, 2, None) == 1
    assert lib.oomb_grad_writeback(pool, fake, fake + 2, 8, 0, None) == 3
    lib.oomb_pool_destroy(pool)
    # without host-resident gradients the calls are unsupported
    assert lib.oomb_pool_create(C.byref(_desc()), C.byref(h)) == 0
    assert lib.oomb_grad_writeback(h.value, fake, fake, 8, 0, None) == 8
    lib.oomb_pool_destroy(h.value)


def test_rope_host_checks(lib):
    """oomb_bias_rope refuses shapes it cannot run and pointers off their element size
    before launching anything."""
    fake = 1 << 24
    bf16, fp32 = _lib.OOMB_BF16, _lib.OOMB_FP32
    rope = lib.oomb_bias_rope
    assert rope(fake, bf16, None, fake, bf16, 4, 2, 7, 0, 1e6, 1, None) == 1       # odd head dim
    assert rope(fake, bf16, None, fake, bf16, 4, 2, 8, 0, 1.0, 1, None) == 1       # theta <= 1
    assert rope(fake, 5, None, fake, bf16, 4, 2, 8, 0, 1e6, 1, None) == 4          # dtype
    assert rope(fake, bf16, None, fake, fp32, 4, 2, 8, 0, 1e6, 1, None) == 1       # in place, two dtypes
    assert rope(fake + 1, bf16, None, fake + 64, bf16, 4, 2, 8, 0, 1e6, 1, None) == 3
    assert rope(fake + 2, fp32, None, fake + 64, fp32, 4, 2, 8, 0, 1e6, 1, None) == 3
    assert rope(fake, bf16, fake + 2, fake + 64, bf16, 4, 2, 8, 0, 1e6, 1, None) == 3  # bias
    assert rope(fake, bf16, None, fake + 65, bf16, 4, 2, 8, 0, 1e6, 1, None) == 3
