"""Parity at the benchmark's full sizes, in the launch configuration bench.py times.

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
