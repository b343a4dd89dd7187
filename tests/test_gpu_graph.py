"""A whole step captured in one CUDA graph and replayed gives the eager step's
results: the same selections (bit-exact; the selection's grid barriers keep no
host state, so replays reuse the captured launch), and the same dQ, dK, dV up to
the order of their fp32 reductions across thread blocks.  Also checked
against the oracle on the window workload's last chunk."""
import math
import os
import sys

import pytest
import torch

import oracle.oomb_oracle as O
import paged_sparse_attention_gb300 as L
from paged_sparse_attention_gb300 import synth

from harness import f64

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu

QWEN = synth.WORKLOADS["sparse128k"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_sparse_attention_gb300 import build
    build.build()
    L.load()


@pytest.mark.parametrize("kind", ["topk", "window"])
def test_graph_replay_matches_eager(kind):
    if kind == "topk":  # 5 chunks of 8 pages, top-8: chunks 2..4 run the cooperative scoring path
        w = synth.scaled(QWEN, "graph_topk", seq=128 * 40, chunk=1024, top_k=8, plants=2)
    else:
        w = synth.scaled(QWEN, "graph_window", seq=128 * 40 + 100, chunk=1024, top_k=-1, plants=0, window=5,
                         n_sink=1)
    dev = torch.device("cuda")
    step = bench.Step(w, dev, host_inputs=True)
    step.run()
    torch.cuda.synchronize()
    assert L.oomb_check(step.pool.handle) == 0
    sel0, cnt0 = step.sel.clone(), step.cnt.clone()
    dq0 = [d.clone() for d in step.dq]
    dk0, dv0 = step.pool.dk_pool.clone(), step.pool.dv_pool.clone()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.run()
    # wipe every output so that only the replays can have written them
    step.sel.fill_(-5)
    step.cnt.zero_()
    for d in step.dq:
        d.zero_()
    step.pool.dk_pool.fill_(3.0)
    step.pool.dv_pool.fill_(3.0)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert L.oomb_check(step.pool.handle) == 0
    assert torch.equal(step.cnt, cnt0)
    for c in range(w.n_chunks):  # entries past a count are not written by a selection
        for h in range(w.n_kv_heads):
            k = int(cnt0[c, h])
            assert torch.equal(step.sel[c, h, :k], sel0[c, h, :k]), (c, h)
    # fp32 sums reduced across thread blocks in a run-dependent order: equal to rounding
    # (dQ is then rounded to bf16, where such differences can flip the last bit)
    for d, d0 in zip(step.dq, dq0):
        assert O.rel_l2(f64(d), f64(d0)) < 1e-4
    assert O.rel_l2(f64(step.pool.dk_pool), f64(dk0)) < 1e-6
    assert O.rel_l2(f64(step.pool.dv_pool), f64(dv0)) < 1e-6

    # the replayed last chunk's forward against the oracle (KV group 0)
    c = w.n_chunks - 1
    start, n = w.chunk_bounds(c)
    G = w.group
    step._fwd(c, step.chunks[c], start, n, False)
    torch.cuda.synchronize()
    lse = step.lse[:G] if n == w.chunk else step.lse_tail(n)[:G]
    order = synth.page_order(w).tolist()
    pool = O.OraclePool(1, w.head_dim, w.page, w.num_phys, w.n_pages)
    used = 0
    for i in range(c + 1):
        s0, m = w.chunk_bounds(i)
        hc = step.host_chunks[i]
        npg = -(-m // w.page)
        pool.append(hc["k"][:, :1].double().numpy(), hc["v"][:, :1].double().numpy(), s0, order[used:used + npg])
        used += npg
    sel = [step.sel[c, 0, : int(step.cnt[c, 0])].cpu().numpy()]
    q = step.host_chunks[c]["q"][:, :G].double().numpy()
    o_ref, lse_ref = O.chunk_attn_fwd(pool, q, start, sel, 1.0 / math.sqrt(w.head_dim))
    assert O.rel_l2(f64(step.o[:n, :G]), o_ref) < 1e-2
    assert O.rel_l2(f64(lse), lse_ref) < 1e-2
    if kind == "window":
        assert sel[0].tolist() == O.window_pages(start, n, w.page, w.window, w.n_sink).tolist()
    step.pool.close()
