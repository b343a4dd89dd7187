"""oomb_page_select_noalloc: page selection for callers that cannot allocate
device memory (a framework owning all device memory, an allocation-free steady
state loop, a C host without an allocator).  Its scratch is a static device array
inside the library; this file checks it against oomb_page_select with a caller
workspace, on two calls in a row, and that pools needing more scratch than the
array holds are refused.  Collected last on purpose."""
import ctypes as C

import pytest
import torch

import paged_sparse_attention_gb300 as L
from paged_sparse_attention_gb300 import _lib, build, synth
from paged_sparse_attention_gb300.pool import PagedKVPool


def test_noalloc_rejects_pools_beyond_its_scratch():
    build.build()
    lib = L.load()
    d = _lib.PoolDesc()
    d.n_q_heads, d.n_kv_heads, d.head_dim, d.page_size = 28, 4, 128, 128
    d.num_phys_pages, d.max_logical_pages, d.dtype = 8, 400_000, _lib.OOMB_BF16
    fake = 1 << 20
    for i, f in enumerate(["k_pool", "v_pool", "dk_pool", "dv_pool", "summary", "page_table", "error_word"]):
        setattr(d, f, fake * (i + 1))
    h = C.c_void_p()
    assert lib.oomb_pool_create(C.byref(d), C.byref(h)) == 0
    assert lib.oomb_workspace_size(h.value, 0, 4096) > (4 << 20)
    # refused on the host before any device work (status ERR_WORKSPACE)
    assert lib.oomb_page_select_noalloc(h.value, fake, 0, 4096, 64, 1, fake, fake, 256, None) == 9
    lib.oomb_pool_destroy(h.value)


@pytest.mark.gpu
def test_noalloc_matches_workspace_select_twice():
    build.build()
    L.load()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    w = synth.scaled(synth.WORKLOADS["sparse128k"], "noalloc", seq=128 * 40, chunk=128 * 8, top_k=6, plants=2)
    plants = synth.PlantTable(w)
    pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages, w.torch_dtype, dev,
                       page_order=synth.page_order(w))
    ws = pool.workspace(L.OOMB_OP_SELECT, w.chunk)
    calls = 0
    for c in range(w.n_chunks):
        start, n = w.chunk_bounds(c)
        ch = {k: v.to(dev) for k, v in synth.make_chunk(w, c, plants=plants, need_do=False).items()}
        L.oomb_kv_append(pool.handle, ch["k"], ch["v"], start)
        if c < 3:
            continue
        ref = torch.full((w.n_kv_heads, w.max_sel), -7, dtype=torch.int32, device=dev)
        ref_cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
        L.oomb_page_select(pool.handle, ch["q"], start, w.top_k, w.n_sink, ref, ref_cnt, ws)
        got = torch.full((w.n_kv_heads, w.max_sel), -7, dtype=torch.int32, device=dev)
        got_cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
        L.oomb_page_select_noalloc(pool.handle, ch["q"], start, w.top_k, w.n_sink, got, got_cnt)
        torch.cuda.synchronize()
        assert torch.equal(got_cnt, ref_cnt)
        assert torch.equal(got, ref)  # integer output: exact
        calls += 1
    assert calls >= 2
    assert L.oomb_check(pool.handle) == 0
    pool.close()
