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
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_noalloc_matches_workspace_select_twice(dtype):
    """Two calls in a row (and more) give the workspace variant's selection exactly;
    one call is also checked against the oracle (up to near-ties); after a first call,
    further calls leave the device's free memory and torch's pool unchanged."""
    build.build()
    L.load()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import numpy as np

    import oracle.oomb_oracle as O
    dev = torch.device("cuda")
    w = synth.scaled(synth.WORKLOADS["sparse128k"], f"noalloc_{dtype}", seq=128 * 40, chunk=128 * 8, top_k=6,
                     plants=2, dtype=dtype)
    plants = synth.PlantTable(w)
    order = synth.page_order(w)
    opool = O.OraclePool(w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages)
    used = 0
    pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages, w.torch_dtype, dev,
                       page_order=order)
    ws = pool.workspace(L.OOMB_OP_SELECT, w.chunk)
    calls = 0
    mem = None
    for c in range(w.n_chunks):
        start, n = w.chunk_bounds(c)
        host = synth.make_chunk(w, c, plants=plants, need_do=False)
        ch = {k: v.to(dev) for k, v in host.items()}
        L.oomb_kv_append(pool.handle, ch["k"], ch["v"], start)
        npg = -(-n // w.page)
        opool.append(host["k"].double().numpy(), host["v"].double().numpy(), start, order[used:used + npg].tolist())
        used += npg
        if c < 3:
            continue
        ref = torch.full((w.n_kv_heads, w.max_sel), -7, dtype=torch.int32, device=dev)
        ref_cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
        L.oomb_page_select(pool.handle, ch["q"], start, w.top_k, w.n_sink, ref, ref_cnt, ws)
        got = torch.full((w.n_kv_heads, w.max_sel), -7, dtype=torch.int32, device=dev)
        got_cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()
        if mem is not None:
            mem = (torch.cuda.mem_get_info(dev)[0], torch.cuda.memory_reserved(dev))
        for _ in range(3):
            L.oomb_page_select_noalloc(pool.handle, ch["q"], start, w.top_k, w.n_sink, got, got_cnt)
        torch.cuda.synchronize()
        if mem is None:  # the first calls have done the set-up; from now on nothing may grow
            mem = (torch.cuda.mem_get_info(dev)[0], torch.cuda.memory_reserved(dev))
        else:
            assert (torch.cuda.mem_get_info(dev)[0], torch.cuda.memory_reserved(dev)) == mem
        assert torch.equal(got_cnt, ref_cnt)
        assert torch.equal(got, ref)  # integer output: exact
        if c == w.n_chunks - 1:  # and the oracle's selection, up to near-ties
            q64 = host["q"].double().numpy()
            ora = O.select_pages(opool, q64, start, w.top_k, w.n_sink)
            cand, scores = O.page_scores(opool, q64, start, w.n_sink)
            for hh in range(w.n_kv_heads):
                sel_h = got[hh, : int(got_cnt[hh])].cpu().numpy()
                assert O.near_tie_ok(sel_h, np.asarray(ora[hh]), cand, scores[hh], w.top_k)[0]
        calls += 1
    assert calls >= 2
    assert L.oomb_check(pool.handle) == 0
    pool.close()
