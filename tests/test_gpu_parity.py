"""GPU parity: every step of the hot path through the C ABI against the fp64 oracle.

Sizes span several pages and query tiles, with a ragged last chunk (partial last
page).  Tolerances: relative L2 <= 1e-5 in fp32, <= 1e-2 in bf16 (O, LSE, dQ, dK,
dV); page selection exact up to documented near-ties (relative score gap < 1e-4);
pool copies bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle.oomb_oracle as O
import paged_sparse_attention_gb300 as L
from paged_sparse_attention_gb300 import synth
from paged_sparse_attention_gb300.pool import PagedKVPool

from harness import TOL, GpuSweep, f64, make_chunks, oracle_sweep, pad_sel

pytestmark = pytest.mark.gpu

QWEN = synth.WORKLOADS["sparse128k"]
CASES = {
    # fp32, tiny geometry (d 64, page 64, 2/1 heads), dense, ragged last chunk
    "fp32_dense": synth.scaled(synth.WORKLOADS["tiny"], "fp32_dense", seq=1000, chunk=256),
    # fp32 sparse, GQA 4:2, odd page size, partial page inside the last chunk
    "fp32_sparse": synth.scaled(synth.WORKLOADS["tiny"], "fp32_sparse", n_q_heads=4, n_kv_heads=2, head_dim=32,
                                seq=1111, chunk=240, page=48, top_k=3, plants=2),
    # Qwen geometry bf16, dense, 4 chunks of 512 + ragged 200
    "bf16_dense": synth.scaled(QWEN, "bf16_dense", seq=2248, chunk=512, top_k=-1, plants=0),
    # Qwen geometry bf16, sparse top-4 with planted pages
    "bf16_sparse": synth.scaled(QWEN, "bf16_sparse", seq=3000, chunk=512, top_k=4, plants=2),
    # bf16 on a shape the tensor-core kernels do not take (d 64, page 64)
    "bf16_small_d": synth.scaled(QWEN, "bf16_small_d", n_q_heads=6, n_kv_heads=2, head_dim=64, page=64,
                                 seq=1300, chunk=320, top_k=3, plants=2),
    # tensor-core shape, plain multi-head attention (G = 1): one step per query tile and page
    "bf16_mha": synth.scaled(QWEN, "bf16_mha", n_q_heads=3, n_kv_heads=3, seq=2900, chunk=640, top_k=5,
                             plants=2),
    # tensor-core shape, chunks of one page and a last chunk of a single token
    "bf16_one_page_chunks": synth.scaled(QWEN, "bf16_one_page_chunks", n_q_heads=8, n_kv_heads=2, seq=5 * 128 + 1,
                                         chunk=128, top_k=2, plants=0),
    # tensor-core shape, a wide group (G = 8) over two KV heads
    "bf16_g8": synth.scaled(QWEN, "bf16_g8", n_q_heads=16, n_kv_heads=2, seq=2500, chunk=768, top_k=4,
                            plants=2),
}


# -- local sliding-window selection ------------------------------------------------
WINDOW_CASES = {
    # Qwen geometry bf16: 3-page window and one sink page, ragged last chunk
    "bf16_window": synth.scaled(QWEN, "bf16_window", seq=3000, chunk=512, top_k=-1, plants=0, window=3,
                                n_sink=1),
    # fp32 tiny geometry: chunk-local attention (no window, no sink)
    "fp32_local": synth.scaled(synth.WORKLOADS["tiny"], "fp32_local", seq=1000, chunk=256, window=0, n_sink=0),
    # fp32 GQA 4:2, odd page size, window 2 and two sinks
    "fp32_window": synth.scaled(synth.WORKLOADS["tiny"], "fp32_window", n_q_heads=4, n_kv_heads=2, head_dim=32,
                                seq=1111, chunk=240, page=48, window=2, n_sink=2),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_sparse_attention_gb300 import build
    build.build()
    L.load()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name", list(CASES))
def test_sweep_parity(name):
    w = CASES[name]
    chunks, plants = make_chunks(w)
    order = synth.page_order(w).tolist()
    ref = oracle_sweep(w, chunks, order)
    run = GpuSweep(w, chunks, order, sel_override=ref["sel"])
    assert run.err_bits == 0
    tol = TOL[w.dtype]
    for c in range(w.n_chunks):
        assert O.rel_l2(f64(run.O[c]), ref["O"][c]) < tol, ("O", c)
        assert O.rel_l2(f64(run.LSE[c]), ref["LSE"][c]) < tol, ("LSE", c)
        assert O.rel_l2(f64(run.dQ[c]), ref["dQ"][c]) < tol, ("dQ", c)
        # the reverse sweep's recomputed forward is bit-identical to the forward sweep
        assert torch.equal(run.O[c], run.O2[c]) and torch.equal(run.LSE[c], run.LSE2[c])
    rdk, rdv = ref["pool"].logical_grads()
    assert O.rel_l2(f64(run.dK), rdk) < tol
    assert O.rel_l2(f64(run.dV), rdv) < tol
    # selection (GPU's own) against the oracle, up to near-ties
    final = ref["pool"]
    swaps = 0
    for c in range(w.n_chunks):
        start, n = w.chunk_bounds(c)
        cand, scores = O.page_scores(final, chunks[c]["q"].double().numpy(), start, w.n_sink)
        for h in range(w.n_kv_heads):
            ok, k = O.near_tie_ok(run.gpu_sel[c][h], ref["sel"][c][h], cand, scores[h], w.top_k)
            assert ok, (c, h, run.gpu_sel[c][h], ref["sel"][c][h])
            swaps += k
        if plants is not None and n == w.chunk:  # a short ragged chunk's mean query is too noisy
            for h in range(w.n_kv_heads):
                for p in plants.planted.get((c, h), []):
                    assert p in set(run.gpu_sel[c][h].tolist())
    run.pool.close()


@pytest.mark.parametrize("name", ["fp32_dense", "bf16_sparse"])
def test_append_pools_bit_exact(name):
    w = CASES[name]
    chunks, _ = make_chunks(w)
    order = synth.page_order(w)
    dev = torch.device("cuda")
    pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages, w.torch_dtype,
                       dev, page_order=order)
    pool.dk_pool.fill_(7.0)
    pool.dv_pool.fill_(7.0)
    for c, ch in enumerate(chunks):
        start, _ = w.chunk_bounds(c)
        L.oomb_kv_append(pool.handle, ch["k"].to(dev), ch["v"].to(dev), start)
    assert L.oomb_check(pool.handle) == 0
    # page table = creation order, host copy == device table
    tab = pool.table_host(w.n_pages)
    assert tab == order[: w.n_pages].tolist()
    assert pool.page_table[: w.n_pages].cpu().tolist() == tab
    assert (pool.page_table[w.n_pages:].cpu() == -1).all()
    k, v = pool.logical_kv(w.seq)
    K = torch.cat([ch["k"] for ch in chunks])
    V = torch.cat([ch["v"] for ch in chunks])
    assert torch.equal(k.cpu(), K) and torch.equal(v.cpu(), V)
    dk, dv = pool.logical_grads(w.seq)
    assert (dk == 0).all() and (dv == 0).all()
    # summaries: mean key over the tokens present (partial last page included)
    Kd = K.double().numpy()
    for p in range(w.n_pages):
        m = min(w.page, w.seq - p * w.page)
        ref = Kd[p * w.page: p * w.page + m].mean(axis=0)  # [Hkv, d]
        got = f64(pool.summary[tab[p]])
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)
    assert L.oomb_pool_free_pages(pool.handle) == w.num_phys - w.n_pages
    pool.close()


def test_select_edge_cases():
    """top_k 0, top_k >= candidates, no sink, several sinks, first chunk."""
    w = synth.scaled(QWEN, "edge", seq=128 * 12, chunk=128 * 3, top_k=2, plants=0)
    chunks, _ = make_chunks(w)
    order = synth.page_order(w)
    dev = torch.device("cuda")
    pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages, w.torch_dtype,
                       dev, page_order=order)
    opool = O.OraclePool(w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages)
    ws = pool.workspace(L.OOMB_OP_SELECT, w.chunk)
    used = 0
    for c, ch in enumerate(chunks):
        start, n = w.chunk_bounds(c)
        L.oomb_kv_append(pool.handle, ch["k"].to(dev), ch["v"].to(dev), start)
        npg = -(-n // w.page)
        opool.append(ch["k"].double().numpy(), ch["v"].double().numpy(), start, order[used:used + npg].tolist())
        used += npg
        q = ch["q"].to(dev)
        for top_k, n_sink in [(0, 1), (2, 0), (2, 3), (100, 1), (-1, 1), (1, 1)]:
            max_sel = w.n_pages + 4
            sel = torch.full((w.n_kv_heads, max_sel), -1, dtype=torch.int32, device=dev)
            cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
            L.oomb_page_select(pool.handle, q, start, top_k, n_sink, sel, cnt, ws)
            ref = O.select_pages(opool, ch["q"].double().numpy(), start, top_k, n_sink)
            cand, scores = O.page_scores(opool, ch["q"].double().numpy(), start, n_sink)
            for h in range(w.n_kv_heads):
                got = sel[h, : int(cnt[h])].cpu().numpy()
                assert np.all(np.diff(got) > 0), "ascending"
                ok, _ = O.near_tie_ok(got, ref[h], cand, scores[h], top_k)
                assert ok, (c, top_k, n_sink, h, got, ref[h])
    assert L.oomb_check(pool.handle) == 0
    pool.close()


def test_host_errors_on_gpu():
    w = synth.scaled(QWEN, "err", seq=512, chunk=256, top_k=1, plants=0)
    dev = torch.device("cuda")
    pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, 3, 8, w.torch_dtype, dev)
    ch = synth.make_chunk(w, 0)
    k, v = ch["k"].to(dev), ch["v"].to(dev)
    with pytest.raises(L.OombError) as e:
        L.oomb_kv_append(pool.handle, k, v, 128)  # not contiguous with what is stored
    assert e.value.status == 1
    L.oomb_kv_append(pool.handle, k, v, 0)
    with pytest.raises(L.OombError) as e:  # 2 more pages needed, 1 free
        L.oomb_kv_append(pool.handle, k, v, 256)
    assert e.value.status == 2
    assert pool.n_tokens == 256
    sel = torch.zeros((w.n_kv_heads, 1), dtype=torch.int32, device=dev)
    cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
    ws = pool.workspace(L.OOMB_OP_SELECT, 256)
    with pytest.raises(L.OombError):  # max_sel 1 < 2 own pages
        L.oomb_page_select(pool.handle, ch["q"].to(dev), 0, 1, 1, sel, cnt, ws)
    # a selection index beyond the chunk raises the device error word, not a fault
    bad = torch.tensor([[0, 5]] * w.n_kv_heads, dtype=torch.int32, device=dev)
    bcnt = torch.full((w.n_kv_heads,), 2, dtype=torch.int32, device=dev)
    o = torch.empty_like(ch["q"].to(dev))
    lse = torch.empty(w.n_q_heads, 256, dtype=torch.float32, device=dev)
    L.oomb_chunk_attn_fwd(pool.handle, ch["q"].to(dev), 0, bad, bcnt, 0.1, o, lse)
    with pytest.raises(L.OombError) as e:
        L.oomb_check(pool.handle)
    assert e.value.status == 5
    assert L.oomb_check(pool.handle) == 0  # cleared
    pool.close()


@pytest.mark.parametrize("grads,staged", [(False, False), (True, False), (True, True), (True, "deferred")],
                         ids=["kv", "kv+grads", "kv+grads+staged-append", "kv+grads+deferred-append"])
@pytest.mark.parametrize("name", ["bf16_sparse", "fp32_sparse", "bf16_window"])
def test_offload_matches_resident(name, grads, staged):
    """K/V pools (and with grads the fp32 dK/dV pools) in pinned host memory, the
    selected blocks staged in HBM on a side stream (gradients staged in from the host
    or carried over from the previous chunk, and written back after each backward):
    the same outputs as the HBM-resident run -- bitwise for O, LSE, dK and dV (each
    gradient row is summed in a fixed order), dQ to rounding (fp32 reductions across
    thread blocks in a run-dependent order) -- and within tolerance of the oracle.
    With the staged append the selection comes first (it needs the history only), the
    append writes the chunk's own pages into their staging slots, and only the history
    pages are gathered from the host; with the deferred append the append writes the
    slots only and the own pages reach the host pools by the side stream's write-back
    (the reverse sweep gathers them from there, and the host pools must equal the
    resident pools)."""
    w = {**CASES, **WINDOW_CASES}[name]
    chunks, _ = make_chunks(w)
    order = synth.page_order(w).tolist()
    ref = oracle_sweep(w, chunks, order)
    res = GpuSweep(w, chunks, order, sel_override=ref["sel"])
    off = GpuSweep(w, chunks, order, sel_override=ref["sel"], offload=True, offload_grads=grads,
                   staged_append=staged)
    assert off.err_bits == 0
    for c in range(w.n_chunks):
        assert torch.equal(off.O[c], res.O[c]) and torch.equal(off.LSE[c], res.LSE[c])
        assert O.rel_l2(f64(off.dQ[c]), f64(res.dQ[c])) < 1e-3
        assert O.rel_l2(f64(off.dQ[c]), ref["dQ"][c]) < TOL[w.dtype]
    assert torch.equal(off.dK.cpu(), res.dK.cpu()) and torch.equal(off.dV.cpu(), res.dV.cpu())
    rdk, rdv = ref["pool"].logical_grads()
    assert O.rel_l2(f64(off.dK), rdk) < TOL[w.dtype] and O.rel_l2(f64(off.dV), rdv) < TOL[w.dtype]
    for a, b in zip(off.gpu_sel, res.gpu_sel):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)
    ok, ov = off.pool.logical_kv(w.seq)
    rk, rv = res.pool.logical_kv(w.seq)
    assert torch.equal(ok, rk) and torch.equal(ov, rv)
    res.pool.close()
    off.pool.close()


@pytest.mark.parametrize("name", ["bf16_sparse", "bf16_dense"])
def test_backward_gradients_deterministic(name):
    """dK/dV are partitioned by (page, KV head): the thread blocks that share a block
    sum their partials in a fixed order and add them once, so two runs of the same
    sweep give bit-identical gradient pools (no float atomics on the pool)."""
    w = CASES[name]
    chunks, _ = make_chunks(w)
    order = synth.page_order(w).tolist()
    a = GpuSweep(w, chunks, order)
    b = GpuSweep(w, chunks, order)
    assert a.err_bits == 0 and b.err_bits == 0
    assert torch.equal(a.dK, b.dK) and torch.equal(a.dV, b.dV)
    for c in range(w.n_chunks):
        assert torch.equal(a.O[c], b.O[c]) and torch.equal(a.LSE[c], b.LSE[c])
    a.pool.close()
    b.pool.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("bad", ["unsorted", "duplicate", "count_too_large", "negative_count"])
def test_malformed_selection_is_flagged(dtype, bad):
    """A selection that is not strictly ascending, repeats a page, or has a count
    outside [0, max_sel] raises OOMB_DEVERR_SEL (status KERNEL from oomb_check) in the
    forward and in the backward; the kernels read only inside the selection row, and
    the context stays usable (a valid call afterwards is clean)."""
    w = synth.scaled(QWEN, f"badsel_{dtype}", seq=1024, chunk=512, top_k=-1, plants=0, dtype=dtype)
    if dtype == "fp32":
        w = synth.scaled(synth.WORKLOADS["tiny"], "badsel_fp32", seq=512, chunk=256)
    chunks, _ = make_chunks(w, plants=False)
    dev = torch.device("cuda")
    pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages, w.torch_dtype,
                       dev, page_order=synth.page_order(w))
    for c, ch in enumerate(chunks):
        L.oomb_kv_append(pool.handle, ch["k"].to(dev), ch["v"].to(dev), w.chunk_bounds(c)[0])
    c = w.n_chunks - 1
    start, n = w.chunk_bounds(c)
    q, do = chunks[c]["q"].to(dev), chunks[c]["do"].to(dev)
    n_vis = -(-(start + n) // w.page)
    good = list(range(n_vis))
    max_sel = n_vis + 2
    rows = {"unsorted": [good[1], good[0]] + good[2:], "duplicate": good[:2] + [good[1]] + good[2:],
            "count_too_large": good, "negative_count": good}[bad]
    sel = torch.full((w.n_kv_heads, max_sel), -1, dtype=torch.int32)
    sel[:, : len(rows)] = torch.tensor(rows, dtype=torch.int32)
    count = {"count_too_large": max_sel + 5, "negative_count": -3}.get(bad, len(rows))
    cnt = torch.full((w.n_kv_heads,), count, dtype=torch.int32)
    sel, cnt = sel.to(dev), cnt.to(dev)
    scale = 1.0 / math.sqrt(w.head_dim)
    o = torch.empty_like(q)
    lse = torch.empty(w.n_q_heads, n, dtype=torch.float32, device=dev)
    L.oomb_chunk_attn_fwd(pool.handle, q, start, sel, cnt, scale, o, lse)
    with pytest.raises(L.OombError) as e:
        L.oomb_check(pool.handle)
    assert e.value.status == 5
    ws = pool.workspace(L.OOMB_OP_BWD, n)
    dq = torch.empty_like(q)
    L.oomb_chunk_attn_bwd(pool.handle, q, o, do, lse, start, sel, cnt, scale, dq, ws)
    with pytest.raises(L.OombError) as e:
        L.oomb_check(pool.handle)
    assert e.value.status == 5
    # a valid selection afterwards: no error
    gsel, gcnt = pad_sel([np.array(good)] * w.n_kv_heads, max_sel, dev)
    L.oomb_chunk_attn_fwd(pool.handle, q, start, gsel, gcnt, scale, o, lse)
    L.oomb_chunk_attn_bwd(pool.handle, q, o, do, lse, start, gsel, gcnt, scale, dq, ws)
    assert L.oomb_check(pool.handle) == 0
    pool.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_single_row_rescale(dtype):
    """One query row meets a key whose score jumps far above its running maximum on
    a later page, while the other rows of its warp see ordinary scores: the online
    softmax must rescale O for that row alone (and the warp must not diverge)."""
    w = synth.scaled(QWEN, f"rescale_{dtype}", seq=1024, chunk=512, top_k=-1, plants=0, dtype=dtype)
    chunks, _ = make_chunks(w, plants=False)
    q_tok, k_tok = 512 + 37, 200  # query in chunk 1 (tile 0), key on page 1 (second page visited)
    for g in range(w.group):      # every query head of KV head 0 gets its own spike key
        kt = k_tok + 3 * g
        qv = chunks[1]["q"][q_tok - 512 + g, g].float()
        # scaled score q.k / sqrt(d) = 14: ~16 in log2 units above the row's earlier maximum
        chunks[0]["k"][kt, 0] = (14.0 * math.sqrt(w.head_dim) * qv / qv.dot(qv)).to(w.torch_dtype)
    order = synth.page_order(w).tolist()
    ref = oracle_sweep(w, chunks, order)
    run = GpuSweep(w, chunks, order, sel_override=ref["sel"])
    assert run.err_bits == 0
    tol = TOL[w.dtype]
    for c in range(w.n_chunks):
        assert O.rel_l2(f64(run.O[c]), ref["O"][c]) < tol, ("O", c)
        assert O.rel_l2(f64(run.LSE[c]), ref["LSE"][c]) < tol, ("LSE", c)
        assert O.rel_l2(f64(run.dQ[c]), ref["dQ"][c]) < tol, ("dQ", c)
    # the spiked rows: LSE within rounding of the spike's own score
    for g in range(w.group):
        r = q_tok - 512 + g
        assert abs(float(run.LSE[1][g, r]) - ref["LSE"][1][g, r]) < 1e-2 * abs(ref["LSE"][1][g, r])
    rdk, rdv = ref["pool"].logical_grads()
    assert O.rel_l2(f64(run.dK), rdk) < tol
    assert O.rel_l2(f64(run.dV), rdv) < tol


@pytest.mark.parametrize("pattern", ["all_equal", "alternating"])
def test_select_exact_ties(pattern):
    """Exactly tied page scores go to the lowest logical pages.  'all_equal' gives
    every candidate the same summary (more tied keys than the threshold bin's
    gather list holds); 'alternating' ties half of the candidates at the top."""
    w = synth.scaled(QWEN, f"ties_{pattern}", seq=16 * 4224, chunk=16 * 2112, page=16, top_k=100, plants=0)
    dev = torch.device("cuda")
    order = synth.page_order(w)
    pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages, w.torch_dtype,
                       dev, page_order=order)
    opool = O.OraclePool(w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages)
    ws = pool.workspace(L.OOMB_OP_SELECT, w.chunk)
    g = torch.Generator().manual_seed(7)
    a = torch.randn(w.n_kv_heads, w.head_dim, generator=g)
    b = torch.randn(w.n_kv_heads, w.head_dim, generator=g)
    used = 0
    for c in range(w.n_chunks):
        start, n = w.chunk_bounds(c)
        tok = torch.arange(start, start + n)
        if pattern == "all_equal":
            k = a.expand(n, -1, -1)
        else:
            k = torch.where(((tok // w.page) % 2 == 0)[:, None, None], a, b)
        k = k.to(w.torch_dtype).contiguous()
        v = torch.randn(n, w.n_kv_heads, w.head_dim, generator=g).to(w.torch_dtype)
        L.oomb_kv_append(pool.handle, k.to(dev), v.to(dev), start)
        npg = -(-n // w.page)
        opool.append(k.double().numpy(), v.double().numpy(), start, order[used:used + npg].tolist())
        used += npg
    c = w.n_chunks - 1
    start, n = w.chunk_bounds(c)
    q = torch.randn(n, w.n_q_heads, w.head_dim, generator=g).to(w.torch_dtype)
    sel = torch.full((w.n_kv_heads, w.max_sel), -1, dtype=torch.int32, device=dev)
    cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
    L.oomb_page_select(pool.handle, q.to(dev), start, w.top_k, w.n_sink, sel, cnt, ws)
    ref = O.select_pages(opool, q.double().numpy(), start, w.top_k, w.n_sink)
    n_cand = start // w.page - w.n_sink
    assert n_cand > 2048
    for h in range(w.n_kv_heads):
        got = sel[h, : int(cnt[h])].cpu().numpy()
        assert np.array_equal(got, np.asarray(ref[h])), (h, got[:8], ref[h][:8])
    assert L.oomb_check(pool.handle) == 0
    pool.close()


@pytest.mark.parametrize("name", list(WINDOW_CASES))
def test_window_sweep_parity(name):
    """The whole sweep on the GPU's own window selection against the oracle's."""
    w = WINDOW_CASES[name]
    chunks, _ = make_chunks(w)
    order = synth.page_order(w).tolist()
    ref = oracle_sweep(w, chunks, order)
    run = GpuSweep(w, chunks, order)
    assert run.err_bits == 0
    tol = TOL[w.dtype]
    for c in range(w.n_chunks):
        for h in range(w.n_kv_heads):  # integer output: bit-exact
            assert run.gpu_sel[c][h].tolist() == ref["sel"][c][h].tolist(), (c, h)
        assert O.rel_l2(f64(run.O[c]), ref["O"][c]) < tol, ("O", c)
        assert O.rel_l2(f64(run.LSE[c]), ref["LSE"][c]) < tol, ("LSE", c)
        assert O.rel_l2(f64(run.dQ[c]), ref["dQ"][c]) < tol, ("dQ", c)
    rdk, rdv = ref["pool"].logical_grads()
    assert O.rel_l2(f64(run.dK), rdk) < tol
    assert O.rel_l2(f64(run.dV), rdv) < tol
    run.pool.close()


def test_window_select_edge_cases():
    """Bit-exact window sets: first chunk, ragged chunk, window longer than the
    history, sinks beyond the history, window 0; max_sel exactly the set size
    passes and one less is refused before any device work."""
    w = synth.scaled(QWEN, "wedge", seq=128 * 12, chunk=128 * 3, top_k=-1, plants=0)
    chunks, _ = make_chunks(w)
    dev = torch.device("cuda")
    pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages, w.torch_dtype,
                       dev, page_order=synth.page_order(w))
    for c, ch in enumerate(chunks):
        L.oomb_kv_append(pool.handle, ch["k"].to(dev), ch["v"].to(dev), w.chunk_bounds(c)[0])
    for q_start, n_q, window, n_sink in [(0, 384, 3, 1), (384, 384, 0, 0), (768, 384, 1, 1), (1152, 200, 2, 3),
                                         (1152, 384, 100, 1), (384, 128, 5, 9), (1152, 1, 0, 2)]:
        ref = O.window_pages(q_start, n_q, w.page, window, n_sink)
        for max_sel in (len(ref), len(ref) + 5):
            sel = torch.full((w.n_kv_heads, max_sel), -7, dtype=torch.int32, device=dev)
            cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
            L.oomb_window_select(pool.handle, q_start, n_q, window, n_sink, sel, cnt)
            torch.cuda.synchronize()
            for h in range(w.n_kv_heads):
                assert int(cnt[h]) == len(ref)
                assert sel[h, : len(ref)].cpu().tolist() == ref.tolist(), (q_start, n_q, window, n_sink, h)
                assert (sel[h, len(ref):].cpu() == -7).all()  # entries past the count untouched
        if len(ref) > 1:
            small = torch.zeros((w.n_kv_heads, len(ref) - 1), dtype=torch.int32, device=dev)
            with pytest.raises(L.OombError):
                L.oomb_window_select(pool.handle, q_start, n_q, window, n_sink, small, cnt)
    assert L.oomb_check(pool.handle) == 0
    pool.close()


def test_page_free_and_reuse():
    """Pages behind a local window are freed: their table entries become -1 (host
    and device), the window forward is unchanged bit for bit, a second free or a
    range past the appended pages is refused, and the next append takes the freed
    physical pages, lowest logical page first, with its K/V copied exactly."""
    w = synth.scaled(QWEN, "pfree", seq=128 * 12, chunk=128 * 3, top_k=-1, plants=0, window=2, n_sink=1)
    chunks, _ = make_chunks(w)
    dev = torch.device("cuda")
    order = synth.page_order(w)
    pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages + 3, w.torch_dtype,
                       dev, page_order=order)
    for c, ch in enumerate(chunks):
        L.oomb_kv_append(pool.handle, ch["k"].to(dev), ch["v"].to(dev), w.chunk_bounds(c)[0])
    c = w.n_chunks - 1
    start, n = w.chunk_bounds(c)
    q = chunks[c]["q"].to(dev)
    sel = torch.full((w.n_kv_heads, 8), -1, dtype=torch.int32, device=dev)
    cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
    L.oomb_window_select(pool.handle, start, n, w.window, w.n_sink, sel, cnt)
    scale = 1.0 / math.sqrt(w.head_dim)
    o1, l1 = torch.empty_like(q), torch.empty(w.n_q_heads, n, dtype=torch.float32, device=dev)
    L.oomb_chunk_attn_fwd(pool.handle, q, start, sel, cnt, scale, o1, l1)
    before = pool.table_host(w.n_pages)
    freed = before[1:7]  # logical pages 1..6: behind the window {0, 7, 8} + own {9, 10, 11}
    L.oomb_page_free(pool.handle, 1, 6)
    after = pool.table_host(w.n_pages)
    assert after[1:7] == [-1] * 6 and after[:1] == before[:1] and after[7:] == before[7:]
    assert pool.page_table[: w.n_pages].cpu().tolist() == after
    assert L.oomb_pool_free_pages(pool.handle) == w.num_phys - w.n_pages + 6
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    L.oomb_chunk_attn_fwd(pool.handle, q, start, sel, cnt, scale, o2, l2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for bad in [(3, 1), (11, 2), (12, 1)]:  # freed already; past the appended pages
        with pytest.raises(L.OombError):
            L.oomb_page_free(pool.handle, *bad)
    # the next append (3 pages) reuses the freed physical pages of logical pages 1, 2, 3
    k, v = chunks[0]["k"].to(dev), chunks[0]["v"].to(dev)
    L.oomb_kv_append(pool.handle, k, v, w.seq)
    tab = pool.table_host(w.n_pages + 3)
    assert tab[w.n_pages:] == freed[:3]
    kk, vv = pool.logical_kv(w.seq + k.shape[0])
    assert torch.equal(kk[w.seq:].cpu(), chunks[0]["k"]) and torch.equal(vv[w.seq:].cpu(), chunks[0]["v"])
    assert L.oomb_check(pool.handle) == 0
    pool.close()


def test_select_skips_freed_pages():
    """Freed pages (a sink and pages in the middle of the history) are never
    selected: the top-K is taken over the mapped candidates only, a freed sink is
    dropped, and "keep every candidate" keeps the mapped ones.  Expected: the
    oracle's scores restricted to the mapped pages; the forward on the selection
    then matches the oracle and raises no device error."""
    w = synth.scaled(QWEN, "freed", seq=128 * 20, chunk=128 * 4, top_k=4, plants=2)
    chunks, _ = make_chunks(w)
    order = synth.page_order(w)
    dev = torch.device("cuda")
    pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages, w.torch_dtype,
                       dev, page_order=order)
    opool = O.OraclePool(w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages)
    used = 0
    for c, ch in enumerate(chunks):
        start, n = w.chunk_bounds(c)
        L.oomb_kv_append(pool.handle, ch["k"].to(dev), ch["v"].to(dev), start)
        npg = -(-n // w.page)
        opool.append(ch["k"].double().numpy(), ch["v"].double().numpy(), start, order[used:used + npg].tolist())
        used += npg
    c = w.n_chunks - 1
    start, n = w.chunk_bounds(c)
    qn = chunks[c]["q"].double().numpy()
    q = chunks[c]["q"].to(dev)
    freed = [0, 3, 4, 9]  # logical pages: one sink, three candidates
    L.oomb_page_free(pool.handle, 0, 1)
    L.oomb_page_free(pool.handle, 3, 2)
    L.oomb_page_free(pool.handle, 9, 1)
    n_hist = start // w.page
    own = np.arange(n_hist, -(-(start + n) // w.page))
    ws = pool.workspace(L.OOMB_OP_SELECT, w.chunk)
    scale = 1.0 / math.sqrt(w.head_dim)
    # 16 history pages; with two sinks 14 candidates, 11 of them mapped
    for top_k, n_sink in [(4, 2), (10, 2), (11, 2), (12, 2), (-1, 2), (0, 1), (4, 0), (1, 3)]:
        max_sel = w.n_pages + 4
        sel = torch.full((w.n_kv_heads, max_sel), -1, dtype=torch.int32, device=dev)
        cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
        L.oomb_page_select(pool.handle, q, start, top_k, n_sink, sel, cnt, ws)
        cand, scores = O.page_scores(opool, qn, start, n_sink)
        keep = np.array([p not in freed for p in cand])
        mcand, mscores = cand[keep], scores[:, keep]
        sinks = np.array([p for p in range(min(n_sink, n_hist)) if p not in freed], dtype=np.int64)
        exp = []
        for h in range(w.n_kv_heads):
            if top_k < 0 or mcand.size <= top_k:
                chosen = mcand
            else:
                chosen = mcand[np.lexsort((mcand, -mscores[h]))[:top_k]]
            exp.append(np.sort(np.concatenate([sinks, chosen, own]).astype(np.int64)))
        got = [sel[h, : int(cnt[h])].cpu().numpy() for h in range(w.n_kv_heads)]
        for h in range(w.n_kv_heads):
            assert not set(got[h].tolist()) & set(freed), (top_k, n_sink, h, got[h])
            assert np.all(np.diff(got[h]) > 0), "ascending"
            ok, _ = O.near_tie_ok(got[h], exp[h], mcand, mscores[h], top_k)
            assert ok, (top_k, n_sink, h, got[h], exp[h])
        o = torch.empty_like(q)
        lse = torch.empty(w.n_q_heads, n, dtype=torch.float32, device=dev)
        L.oomb_chunk_attn_fwd(pool.handle, q, start, sel, cnt, scale, o, lse)
        ro, rl = O.chunk_attn_fwd(opool, qn, start, got, scale)
        assert O.rel_l2(f64(o), ro) < TOL[w.dtype] and O.rel_l2(f64(lse), rl) < TOL[w.dtype]
        assert L.oomb_check(pool.handle) == 0, (top_k, n_sink)
    # max_sel is checked against the mapped pages: 1 sink + 11 candidates + own fits exactly
    fit = 1 + 11 + own.size
    for slots, ok in [(fit, True), (fit - 1, False)]:
        sel = torch.full((w.n_kv_heads, slots), -1, dtype=torch.int32, device=dev)
        cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
        if ok:
            L.oomb_page_select(pool.handle, q, start, -1, 2, sel, cnt, ws)
            assert cnt.cpu().tolist() == [fit] * w.n_kv_heads
        else:
            with pytest.raises(L.OombError):
                L.oomb_page_select(pool.handle, q, start, -1, 2, sel, cnt, ws)
    assert L.oomb_check(pool.handle) == 0
    pool.close()


@pytest.mark.parametrize("mode", ["pool", "staged", "deferred"])
def test_select_append_fused_matches_separate(mode):
    """oomb_page_select_append against oomb_page_select followed by the append of the
    same mode, chunk by chunk over a sweep whose early chunks keep every candidate (two
    launches) and whose later chunks score pages (one launch): the same selections,
    page table, K/V pools, summaries, zeroed gradient pages and staging slots, bit for
    bit.  The staged modes run on offload pools with the gradients in host memory."""
    w = synth.scaled(QWEN, f"fused_{mode}", seq=11 * 512 + 200, chunk=512, top_k=3, plants=2)
    chunks, _ = make_chunks(w)
    order = synth.page_order(w)
    dev = torch.device("cuda")
    off = mode != "pool"

    def new_pool():
        return PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages, w.torch_dtype,
                           dev, page_order=order, offload=off, stage_max_sel=w.max_sel if off else 0,
                           offload_grads=off)

    sep, fus = new_pool(), new_pool()
    if off:  # slots the appends do not write must compare equal too
        for pl in (sep, fus):
            pl.stage_k.zero_()
            pl.stage_v.zero_()
    ws_s, ws_f = sep.workspace(L.OOMB_OP_SELECT, w.chunk), fus.workspace(L.OOMB_OP_SELECT, w.chunk)
    am = {"pool": L.OOMB_APPEND_POOL, "staged": L.OOMB_APPEND_STAGED, "deferred": L.OOMB_APPEND_DEFERRED}[mode]
    scored = 0
    for c, ch in enumerate(chunks):
        start, n = w.chunk_bounds(c)
        q, k, v = (ch[x].to(dev) for x in ("q", "k", "v"))
        outs = []
        for pl, ws, fused in ((sep, ws_s, False), (fus, ws_f, True)):
            sel = torch.full((w.n_kv_heads, w.max_sel), -1, dtype=torch.int32, device=dev)
            cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=dev)
            if fused:
                L.oomb_page_select_append(pl.handle, q, k, v, start, w.top_k, w.n_sink, sel, cnt, ws, am, c % 2)
            else:
                L.oomb_page_select(pl.handle, q, start, w.top_k, w.n_sink, sel, cnt, ws)
                if mode == "pool":
                    L.oomb_kv_append(pl.handle, k, v, start)
                elif mode == "staged":
                    L.oomb_kv_append_staged(pl.handle, k, v, start, cnt, w.max_sel, c % 2)
                else:
                    L.oomb_kv_append_deferred(pl.handle, k, v, start, cnt, w.max_sel, c % 2)
            outs.append((sel, cnt))
        torch.cuda.synchronize()
        assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][0], outs[1][0]), c
        n_hist = start // w.page
        scored += int(max(0, n_hist - w.n_sink) > w.top_k)
        if off:  # this chunk's staging buffer (its own slots were written by the append)
            assert torch.equal(sep.stage_k[c % 2], fus.stage_k[c % 2]) and torch.equal(sep.stage_v[c % 2],
                                                                                          fus.stage_v[c % 2]), c
    assert scored >= 5  # the fused single launch was exercised
    assert L.oomb_check(sep.handle) == 0 and L.oomb_check(fus.handle) == 0
    assert sep.table_host(w.n_pages) == fus.table_host(w.n_pages)
    assert torch.equal(sep.summary, fus.summary)
    if mode != "deferred":
        ks, vs = sep.logical_kv(w.seq)
        kf, vf = fus.logical_kv(w.seq)
        assert torch.equal(ks, kf) and torch.equal(vs, vf)
        assert torch.equal(ks.cpu(), torch.cat([ch["k"] for ch in chunks]))
    if off:
        assert torch.equal(sep.grad_state, fus.grad_state)
    else:
        assert torch.equal(sep.dk_pool, fus.dk_pool) and torch.equal(sep.dv_pool, fus.dv_pool)
    sep.close()
    fus.close()
