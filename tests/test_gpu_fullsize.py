"""Parity at every configuration's full size, in the launch configuration bench.py times.

The GPU runs the whole forward + reverse sweep of the 32K dense workload (and the
forward sweep of the 128K sparse workload) exactly as bench.Step does; the fp64
oracle recomputes sampled outputs for KV group 0:
  * dense32k, last chunk: O and LSE of the 7 query heads for every row; dQ for a
    block of 256 rows; dK/dV of the chunk's own pages, which no other chunk
    touches (exact from the full-chunk O and LSE and the own-page keys alone);
  * sparse128k: the page selection of sampled chunks (exact up to near-ties) and
    the forward of the last chunk on the oracle's own selection;
  * sparse1m (inputs generated on the device, as the benchmark does): the last
    chunk's selection over all 8063 candidates and the forward of its first and
    last 128 rows on the oracle's selection.
Per-call checks (``_check_calls``) replay sampled chunks of a finished step on the
oracle's selection for KV group 0 (every KV head gets that selection): O and LSE
and dQ on sampled rows (each row is a pure function of the chunk's inputs), and
the chunk's dK/dV contribution (gradient pool zeroed before the replay) on its
last own pages, which only the chunk's tail rows can see, so the oracle needs
those rows alone; optionally the whole chunk, which also covers history pages.
The final gradient pool of the step itself is checked on the last own pages of
the last chunk, which no other chunk touches.
"""
import math
import os
import sys

import numpy as np
import pytest
import torch

import oracle.oomb_oracle as O
import paged_sparse_attention_gb300 as L
from paged_sparse_attention_gb300 import synth

from harness import f64, pad_sel

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


def _oracle_pool(w, step, upto_chunk, h=0):
    """Oracle pool holding KV head h of chunks 0..upto_chunk, pages in the allocator's order."""
    order = synth.page_order(w).tolist()
    pool = O.OraclePool(1, w.head_dim, w.page, w.num_phys, w.n_pages)
    used = 0
    for c in range(upto_chunk + 1):
        start, n = w.chunk_bounds(c)
        hc = step.host_chunks[c]
        npg = -(-n // w.page)
        pool.append(hc["k"][:, h:h + 1].double().numpy(), hc["v"][:, h:h + 1].double().numpy(), start,
                    order[used:used + npg])
        used += npg
    return pool


def test_dense32k_last_chunk_fullsize():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_sparse_attention_gb300 import build
    build.build()
    w = synth.WORKLOADS["dense32k"]
    dev = torch.device("cuda")
    step = bench.Step(w, dev, host_inputs=True)
    step.run()
    torch.cuda.synchronize()
    assert L.oomb_check(step.pool.handle) == 0
    c = w.n_chunks - 1
    start, n = w.chunk_bounds(c)
    G = w.group
    step._fwd(c, step.chunks[c], start, n, False)  # O, LSE of chunk c (the forward has no side effects)
    torch.cuda.synchronize()
    o_gpu = f64(step.o[:n, :G])
    lse_gpu = f64(step.lse[:G])
    dq_gpu = f64(step.dq[c][:, :G])
    pool = _oracle_pool(w, step, c)
    hc = step.host_chunks[c]
    q = hc["q"][:, :G].double().numpy()
    do = hc["do"][:, :G].double().numpy()
    scale = 1.0 / math.sqrt(w.head_dim)
    all_pages = [np.arange(-(-(start + n) // w.page))]
    Oo, Lo = O.chunk_attn_fwd(pool, q, start, all_pages, scale)
    assert O.rel_l2(o_gpu, Oo) < 1e-2 and O.rel_l2(lse_gpu, Lo) < 1e-2
    # dQ for the last 256 rows (exact: a row's dQ needs only its own row)
    r0 = n - 256
    dq_o = O.chunk_attn_bwd(pool, q[r0:], Oo[r0:], do[r0:], Lo[:, r0:], start + r0, all_pages, scale)
    assert O.rel_l2(dq_gpu[r0:], dq_o) < 1e-2
    # dK/dV of the chunk's own pages: fresh oracle gradients from this chunk alone
    pool.dK[:] = 0
    pool.dV[:] = 0
    own = [np.arange(start // w.page, -(-(start + n) // w.page))]
    O.chunk_attn_bwd(pool, q, Oo, do, Lo, start, own, scale)
    dk_gpu, dv_gpu = step.pool.logical_grads(w.seq)
    dk_o, dv_o = pool.logical_grads()
    sl = slice(start, start + n)
    assert O.rel_l2(f64(dk_gpu[sl, :1]), dk_o[sl]) < 1e-2
    assert O.rel_l2(f64(dv_gpu[sl, :1]), dv_o[sl]) < 1e-2
    step.pool.close()


def test_sparse128k_selection_and_forward_fullsize():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_sparse_attention_gb300 import build
    build.build()
    w = synth.WORKLOADS["sparse128k"]
    dev = torch.device("cuda")
    step = bench.Step(w, dev, host_inputs=True)
    step.run()
    torch.cuda.synchronize()
    assert L.oomb_check(step.pool.handle) == 0
    S = w.n_chunks
    pool = _oracle_pool(w, step, S - 1)
    G = w.group
    plants = synth.PlantTable(w)
    for c in sorted({0, 1, 2, 3, S // 2, S - 1}):
        start, n = w.chunk_bounds(c)
        q = step.host_chunks[c]["q"][:, :G].double().numpy()
        ref = O.select_pages(pool, q, start, w.top_k, w.n_sink)
        cand, scores = O.page_scores(pool, q, start, w.n_sink)
        got = step.sel[c, 0, : int(step.cnt[c, 0])].cpu().numpy()
        ok, _ = O.near_tie_ok(got, ref[0], cand, scores[0], w.top_k)
        assert ok, (c, got, ref[0])
        for p in plants.planted.get((c, 0), []):
            assert p in set(got.tolist())
    # forward of the last chunk on the oracle's selection, KV group 0
    c = S - 1
    start, n = w.chunk_bounds(c)
    hc = step.host_chunks[c]
    q = hc["q"][:, :G].double().numpy()
    ref = O.select_pages(pool, q, start, w.top_k, w.n_sink)
    sel, cnt = pad_sel([ref[0]] * w.n_kv_heads, w.max_sel, dev)
    o = torch.empty_like(step.chunks[c]["q"])
    lse = torch.empty(w.n_q_heads, n, dtype=torch.float32, device=dev)
    L.oomb_chunk_attn_fwd(step.pool.handle, step.chunks[c]["q"], start, sel, cnt, step.scale, o, lse)
    Oo, Lo = O.chunk_attn_fwd(pool, q, start, ref, 1.0 / math.sqrt(w.head_dim))
    assert O.rel_l2(f64(o[:, :G]), Oo) < 1e-2 and O.rel_l2(f64(lse[:G]), Lo) < 1e-2
    step.pool.close()


@pytest.mark.slow
def test_sparse1m_last_chunk_fullsize():
    """1M tokens in chunks of 8192, top-128: the full step as bench.Step runs it (inputs
    generated on the device), then KV group 0 of the last chunk against the oracle:
    the page selection over all 8063 candidates (exact up to near-ties; planted pages
    kept) and the forward on the oracle's selection for the chunk's first and last
    128 rows (the rows with the fewest and the most visible keys)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_sparse_attention_gb300 import build
    build.build()
    w = synth.WORKLOADS["sparse1m"]
    dev = torch.device("cuda")
    step = bench.Step(w, dev)
    step.run()
    torch.cuda.synchronize()
    assert L.oomb_check(step.pool.handle) == 0
    S, G = w.n_chunks, w.group
    order = synth.page_order(w).tolist()
    pool = O.OraclePool(1, w.head_dim, w.page, w.num_phys, w.n_pages)
    used = 0
    for c in range(S):
        start, n = w.chunk_bounds(c)
        ch = step.chunks[c]
        npg = -(-n // w.page)
        pool.append(ch["k"][:, 0:1].double().cpu().numpy(), ch["v"][:, 0:1].double().cpu().numpy(), start,
                    order[used:used + npg])
        used += npg
    c = S - 1
    start, n = w.chunk_bounds(c)
    q = step.chunks[c]["q"][:, :G].double().cpu().numpy()
    ref = O.select_pages(pool, q, start, w.top_k, w.n_sink)
    cand, scores = O.page_scores(pool, q, start, w.n_sink)
    got = step.sel[c, 0, : int(step.cnt[c, 0])].cpu().numpy()
    ok, swaps = O.near_tie_ok(got, ref[0], cand, scores[0], w.top_k)
    assert ok, (got[:8], ref[0][:8])
    plants = synth.PlantTable(w)
    for p in plants.planted.get((c, 0), []):
        assert p in set(got.tolist())
    sel, cnt = pad_sel([ref[0]] * w.n_kv_heads, w.max_sel, dev)
    o = torch.empty_like(step.chunks[c]["q"])
    lse = torch.empty(w.n_q_heads, n, dtype=torch.float32, device=dev)
    L.oomb_chunk_attn_fwd(step.pool.handle, step.chunks[c]["q"], start, sel, cnt, step.scale, o, lse)
    torch.cuda.synchronize()
    for r0 in (0, n - 128):
        Oo, Lo = O.chunk_attn_fwd(pool, q[r0:r0 + 128], start + r0, ref, 1.0 / math.sqrt(w.head_dim))
        assert O.rel_l2(f64(o[r0:r0 + 128, :G]), Oo) < 1e-2, r0
        assert O.rel_l2(f64(lse[:G, r0:r0 + 128]), Lo) < 1e-2, r0
    step.pool.close()


def test_window128k_fullsize():
    """128K tokens, local window of 32 pages before each 4K chunk (no sink), as
    bench.Step runs it: every chunk's selection for every KV head bit-exact against
    the oracle's window set, then KV group 0 of the last chunk against the oracle:
    the forward for its first and last 128 rows and dQ for its last 128 rows."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_sparse_attention_gb300 import build
    build.build()
    w = synth.WORKLOADS["window128k"]
    dev = torch.device("cuda")
    step = bench.Step(w, dev)
    step.run()
    torch.cuda.synchronize()
    assert L.oomb_check(step.pool.handle) == 0
    S, G = w.n_chunks, w.group
    sel_all, cnt_all = step.sel.cpu().numpy(), step.cnt.cpu().numpy()
    for c in range(S):
        start, n = w.chunk_bounds(c)
        ref = O.window_pages(start, n, w.page, w.window, w.n_sink)
        for h in range(w.n_kv_heads):
            assert sel_all[c, h, : cnt_all[c, h]].tolist() == ref.tolist(), (c, h)
    order = synth.page_order(w).tolist()
    pool = O.OraclePool(1, w.head_dim, w.page, w.num_phys, w.n_pages)
    used = 0
    for c in range(S):
        start, n = w.chunk_bounds(c)
        ch = step.chunks[c]
        npg = -(-n // w.page)
        pool.append(ch["k"][:, 0:1].double().cpu().numpy(), ch["v"][:, 0:1].double().cpu().numpy(), start,
                    order[used:used + npg])
        used += npg
    c = S - 1
    start, n = w.chunk_bounds(c)
    sel = [O.window_pages(start, n, w.page, w.window, w.n_sink)]
    q = step.chunks[c]["q"][:, :G].double().cpu().numpy()
    do = step.chunks[c]["do"][:, :G].double().cpu().numpy()
    scale = 1.0 / math.sqrt(w.head_dim)
    step._fwd(c, step.chunks[c], start, n, False)  # O, LSE of chunk c (no side effects)
    torch.cuda.synchronize()
    for r0 in (0, n - 128):
        Oo, Lo = O.chunk_attn_fwd(pool, q[r0:r0 + 128], start + r0, sel, scale)
        assert O.rel_l2(f64(step.o[r0:r0 + 128, :G]), Oo) < 1e-2, r0
        assert O.rel_l2(f64(step.lse[:G, r0:r0 + 128]), Lo) < 1e-2, r0
    r0 = n - 128
    Oo, Lo = O.chunk_attn_fwd(pool, q[r0:], start + r0, sel, scale)
    dq_ref = O.chunk_attn_bwd(pool, q[r0:], Oo, do[r0:], Lo, start + r0, sel, scale)
    assert O.rel_l2(f64(step.dq[c][r0:, :G]), dq_ref) < 1e-2
    step.pool.close()



# ---------------------------------------------------------------------------------
# per-call replays at full size
def _oracle_pool_dev(w, chunks, upto_chunk, h=0):
    """Oracle pool holding KV head h of chunks 0..upto_chunk (device or host tensors),
    pages in the allocator's order."""
    order = synth.page_order(w).tolist()
    pool = O.OraclePool(1, w.head_dim, w.page, w.num_phys, w.n_pages)
    used = 0
    for c in range(upto_chunk + 1):
        start, n = w.chunk_bounds(c)
        npg = -(-n // w.page)
        k = chunks[c]["k"][:, h:h + 1].double().cpu().numpy()
        v = chunks[c]["v"][:, h:h + 1].double().cpu().numpy()
        pool.append(k, v, start, order[used:used + npg])
        used += npg
    return pool


def _gpu_page_grads(step, pages, h=0, buf=None, slots=None):
    """dK, dV of the given logical pages of KV head h, [len(pages), P, d] fp64: from the
    gradient pool through the page table, or from staging slots (buf, h, slot)."""
    if buf is not None:
        dk = step.pool.stage_dk[buf, h][slots]
        dv = step.pool.stage_dv[buf, h][slots]
    else:
        tab = step.pool.table_host(max(pages) + 1)
        phys = torch.tensor([tab[p] for p in pages], dtype=torch.long, device=step.pool.dk_pool.device)
        dk = step.pool.dk_pool[phys, h]
        dv = step.pool.dv_pool[phys, h]
    return f64(dk), f64(dv)


def _oracle_page_grads(pool, pages):
    ph = [pool.phi[p] for p in pages]
    return pool.dK[ph, 0].copy(), pool.dV[ph, 0].copy()


def _check_calls(w, step, chunks, pool, chunk_ids, fwd_rows=256, tail_pages=2, full_chunks=()):
    """Replay each sampled chunk's forward and backward through the C ABI on the
    oracle's selection (KV group 0) and compare with the oracle on sampled rows and
    on the dK/dV contribution of the chunk's last own pages (all pages for the chunks
    in ``full_chunks``).  ``pool``: oracle pool holding KV head 0 of at least the
    sampled chunks.  Returns the number of values compared."""
    dev = step.dev
    G, S, P = w.group, w.n_chunks, w.page
    scale = 1.0 / math.sqrt(w.head_dim)
    h = step.pool.handle
    compared = 0
    for c in sorted(set(chunk_ids)):
        start, n = w.chunk_bounds(c)
        ch = step.chunks[c]
        q = chunks[c]["q"][:, :G].double().cpu().numpy()
        do = chunks[c]["do"][:, :G].double().cpu().numpy()
        ref = O.select_pages(pool, q, start, w.top_k, w.n_sink)
        sel, cnt = pad_sel([ref[0]] * w.n_kv_heads, w.max_sel, dev)
        buf = c % 2
        if step.offload:
            L.oomb_prefetch(h, sel, cnt, buf)
            L.oomb_pool_set_stage(h, buf)
        if step.offload_grads:
            step.pool.stage_dk[buf].zero_()
            step.pool.stage_dv[buf].zero_()
        else:
            step.pool.dk_pool.zero_()
            step.pool.dv_pool.zero_()
        o = torch.empty_like(ch["q"])
        lse = torch.empty(w.n_q_heads, n, dtype=torch.float32, device=dev)
        L.oomb_chunk_attn_fwd(h, ch["q"], start, sel, cnt, scale, o, lse)
        dq = torch.empty_like(ch["q"])
        L.oomb_chunk_attn_bwd(h, ch["q"], o, ch["do"], lse, start, sel, cnt, scale, dq, step.ws_bwd)
        torch.cuda.synchronize()
        assert L.oomb_check(h) == 0
        own0 = start // P
        n_own = -(-n // P)
        full = c in full_chunks
        r_tail = 0 if full else max(0, (n_own - tail_pages) * P)
        rows = sorted(set(range(min(fwd_rows, n))) | set(range(max(0, n - fwd_rows), n)) | set(range(r_tail, n)))
        rows = np.arange(n) if full else np.array(rows)
        # O, LSE, dQ on the sampled rows: contiguous runs, each a pure function of its rows
        runs = np.split(rows, np.where(np.diff(rows) != 1)[0] + 1)
        tail_o = tail_l = None
        for run in runs:
            r0, r1 = int(run[0]), int(run[-1]) + 1
            Oo, Lo = O.chunk_attn_fwd(pool, q[r0:r1], start + r0, ref, scale)
            assert O.rel_l2(f64(o[r0:r1, :G]), Oo) < 1e-2, (c, r0, "O")
            assert O.rel_l2(f64(lse[:G, r0:r1]), Lo) < 1e-2, (c, r0, "LSE")
            pages = ref[0] if full else np.arange(own0 + n_own - tail_pages, own0 + n_own)
            for p in pages:  # fresh oracle gradients for the compared pages
                pool.dK[pool.phi[p]] = 0.0
                pool.dV[pool.phi[p]] = 0.0
            dq_o = O.chunk_attn_bwd(pool, q[r0:r1], Oo, do[r0:r1], Lo, start + r0, ref, scale)
            assert O.rel_l2(f64(dq[r0:r1, :G]), dq_o) < 1e-2, (c, r0, "dQ")
            compared += Oo.size + Lo.size + dq_o.size
            if r1 == n and r0 <= r_tail:  # this run holds every row that sees the compared pages
                pages = [int(x) for x in pages]
                dk_o, dv_o = _oracle_page_grads(pool, pages)
                if step.offload_grads:
                    slots = [int(np.searchsorted(ref[0], p)) for p in pages]
                    dk_g, dv_g = _gpu_page_grads(step, pages, buf=buf, slots=slots)
                else:
                    dk_g, dv_g = _gpu_page_grads(step, pages)
                assert O.rel_l2(dk_g, dk_o) < 1e-2, (c, "dK")
                assert O.rel_l2(dv_g, dv_o) < 1e-2, (c, "dV")
                compared += dk_o.size + dv_o.size
    return compared


def _check_final_pool_tail(w, step, chunks, pool, tail_pages=2):
    """The step's own gradient pool (before any replay): the last own pages of the last
    chunk receive contributions from that chunk's tail rows alone.  The GPU's own
    selection of the last chunk is used (checked against the oracle elsewhere).
    ``pool``: oracle pool holding KV head 0 of every chunk."""
    G, S, P = w.group, w.n_chunks, w.page
    c = S - 1
    start, n = w.chunk_bounds(c)
    n_own = -(-n // P)
    pages = list(range(start // P + n_own - tail_pages, start // P + n_own))
    dk_g, dv_g = _gpu_page_grads(step, pages)
    for p in pages:
        pool.dK[pool.phi[p]] = 0.0
        pool.dV[pool.phi[p]] = 0.0
    sel = [step.sel[c, 0, : int(step.cnt[c, 0])].cpu().numpy().astype(np.int64)]
    scale = 1.0 / math.sqrt(w.head_dim)
    r0 = (n_own - tail_pages) * P
    q = chunks[c]["q"][r0:, :G].double().cpu().numpy()
    do = chunks[c]["do"][r0:, :G].double().cpu().numpy()
    Oo, Lo = O.chunk_attn_fwd(pool, q, start + r0, sel, scale)
    O.chunk_attn_bwd(pool, q, Oo, do, Lo, start + r0, sel, scale)
    dk_o, dv_o = _oracle_page_grads(pool, pages)
    assert O.rel_l2(dk_g, dk_o) < 1e-2 and O.rel_l2(dv_g, dv_o) < 1e-2


def test_tiny_config_exact_shape():
    """The tiny configuration at its own shape: 4096 tokens in 4 chunks of 1024, page
    64, 64 physical pages handed out in a seeded shuffled order, 2 query heads / 1 KV
    head, head_dim 64, fp32, every page selected -- the whole sweep (O, LSE, dQ, dK,
    dV) against the oracle's chunked sweep at 1e-5, the selection bit-exact."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_sparse_attention_gb300 import build
    build.build()
    from harness import GpuSweep, make_chunks, oracle_sweep
    w = synth.WORKLOADS["tiny"]
    assert (w.seq, w.chunk, w.page, w.num_phys, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype) == \
        (4096, 1024, 64, 64, 2, 1, 64, "fp32")
    chunks, _ = make_chunks(w)
    order = synth.page_order(w).tolist()
    ref = oracle_sweep(w, chunks, order)
    run = GpuSweep(w, chunks, order)
    assert run.err_bits == 0
    for c in range(w.n_chunks):
        assert run.gpu_sel[c][0].tolist() == ref["sel"][c][0].tolist()
        assert O.rel_l2(f64(run.O[c]), ref["O"][c]) < 1e-5
        assert O.rel_l2(f64(run.LSE[c]), ref["LSE"][c]) < 1e-5
        assert O.rel_l2(f64(run.dQ[c]), ref["dQ"][c]) < 1e-5
    rdk, rdv = ref["pool"].logical_grads()
    assert O.rel_l2(f64(run.dK), rdk) < 1e-5 and O.rel_l2(f64(run.dV), rdv) < 1e-5
    run.pool.close()


def test_sparse128k_backward_calls_fullsize():
    """128K tokens, top-64: after the whole step, chunks {0, 1, S/2, S-1} replayed on
    the oracle's selection; chunk S-1 over every row (its dK/dV on every selected page,
    sink and retrieved history pages included)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_sparse_attention_gb300 import build
    build.build()
    w = synth.WORKLOADS["sparse128k"]
    dev = torch.device("cuda")
    step = bench.Step(w, dev, host_inputs=True)
    step.run()
    torch.cuda.synchronize()
    assert L.oomb_check(step.pool.handle) == 0
    S = w.n_chunks
    pool = _oracle_pool_dev(w, step.host_chunks, S - 1)
    _check_final_pool_tail(w, step, step.host_chunks, pool)
    n = _check_calls(w, step, step.host_chunks, pool, [0, 1, S // 2, S - 1], full_chunks=(S - 1,))
    assert n > 0
    step.pool.close()


@pytest.mark.slow
def test_sparse1m_calls_fullsize():
    """1M tokens in chunks of 8192, top-128, inputs generated on the device as the
    benchmark does: the step's final gradient pool on the last chunk's last own pages,
    then per-call replays of chunks {0, 1, 2, 3, S/2, S-1} on the oracle's selection."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_sparse_attention_gb300 import build
    build.build()
    w = synth.WORKLOADS["sparse1m"]
    dev = torch.device("cuda")
    step = bench.Step(w, dev)
    step.run()
    torch.cuda.synchronize()
    assert L.oomb_check(step.pool.handle) == 0
    S = w.n_chunks
    pool = _oracle_pool_dev(w, step.chunks, S - 1)
    _check_final_pool_tail(w, step, step.chunks, pool)
    n = _check_calls(w, step, step.chunks, pool, [0, 1, 2, 3, S // 2, S - 1], fwd_rows=128)
    assert n > 0
    step.pool.close()


@pytest.mark.slow
def test_offload4m_calls_fullsize():
    """4M tokens, K/V and fp32 gradient pools in pinned host memory (the benchmark's
    default workload), run as bench.Step runs it: the last chunk's selection against
    the oracle (near-ties), the step's final host gradient pool on the last chunk's
    last own pages, O and LSE of sampled chunks bit-identical to an HBM-resident pool
    holding the same pages, and per-call replays of chunks {0, 1, 2, 3, S/2, S-1} on
    the oracle's selection (gradients into the staging slots)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_sparse_attention_gb300 import build
    build.build()
    from paged_sparse_attention_gb300.pool import PagedKVPool
    w = synth.WORKLOADS["offload4m"]
    assert w.offload and w.offload_grads
    dev = torch.device("cuda")
    step = bench.Step(w, dev)
    step.run()
    torch.cuda.synchronize()
    assert L.oomb_check(step.pool.handle) == 0
    S, G = w.n_chunks, w.group
    # selection of the last chunk over all 32767 candidates
    c = S - 1
    start, n = w.chunk_bounds(c)
    pool = _oracle_pool_dev(w, step.chunks, c)
    q = step.chunks[c]["q"][:, :G].double().cpu().numpy()
    ref = O.select_pages(pool, q, start, w.top_k, w.n_sink)
    cand, scores = O.page_scores(pool, q, start, w.n_sink)
    got = step.sel[c, 0, : int(step.cnt[c, 0])].cpu().numpy()
    ok, _ = O.near_tie_ok(got, ref[0], cand, scores[0], w.top_k)
    assert ok
    _check_final_pool_tail(w, step, step.chunks, pool)
    # a resident pool with the same pages: forward bit-identical
    res = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages, w.torch_dtype, dev,
                      page_order=synth.page_order(w))
    for cc in range(S):
        L.oomb_kv_append(res.handle, step.chunks[cc]["k"], step.chunks[cc]["v"], w.chunk_bounds(cc)[0])
    h = step.pool.handle
    for cc in sorted({0, 1, S // 2, S - 1}):
        start, n = w.chunk_bounds(cc)
        ch = step.chunks[cc]
        sel, cnt = step.sel[cc], step.cnt[cc]
        outs = []
        for pl, off in ((step.pool, True), (res, False)):
            if off:
                L.oomb_prefetch(pl.handle, sel, cnt, cc % 2)
                L.oomb_pool_set_stage(pl.handle, cc % 2)
            o = torch.empty_like(ch["q"])
            lse = torch.empty(w.n_q_heads, n, dtype=torch.float32, device=dev)
            L.oomb_chunk_attn_fwd(pl.handle, ch["q"], start, sel, cnt, step.scale, o, lse)
            outs.append((o, lse))
        torch.cuda.synchronize()
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1]), cc
    assert L.oomb_check(h) == 0 and L.oomb_check(res.handle) == 0
    res.close()
    nvals = _check_calls(w, step, step.chunks, pool, [0, 1, 2, 3, S // 2, S - 1], fwd_rows=128)
    assert nvals > 0
    step.pool.close()
