"""The benchmark's credited work, checked by brute force on the CPU: the number of
selected, causally visible (query, key) pairs per chunk (summed over query heads)
that bench.py multiplies by 14 d FLOPs, for dense, top-K-like and window
selections, including a ragged last chunk and a partial last page."""
import os
import sys
import types

import numpy as np
import torch

from paged_sparse_attention_gb300 import synth

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _brute(w, sel, cnt):
    out = []
    for c in range(w.n_chunks):
        start, n = w.chunk_bounds(c)
        tot = 0
        for h in range(w.n_kv_heads):
            keys = [p * w.page + t for p in sel[c, h, : cnt[c, h]] for t in range(w.page)
                    if p * w.page + t < start + n]
            for i in range(start, start + n):
                tot += sum(1 for j in keys if j <= i)
        out.append(tot * w.group)
    return out


def _count(w, sel, cnt):
    ns = types.SimpleNamespace(w=w, sel=torch.from_numpy(sel), cnt=torch.from_numpy(cnt))
    return bench.Step.pairs_per_chunk(ns)


def _selections(w, kind, rng):
    sel = np.full((w.n_chunks, w.n_kv_heads, w.n_pages), -1, dtype=np.int32)
    cnt = np.zeros((w.n_chunks, w.n_kv_heads), dtype=np.int32)
    for c in range(w.n_chunks):
        start, n = w.chunk_bounds(c)
        n_hist = start // w.page
        own = list(range(n_hist, (start + n - 1) // w.page + 1))
        for h in range(w.n_kv_heads):
            if kind == "dense":
                pages = list(range(n_hist)) + own
            elif kind == "window":
                pages = [int(p) for p in range(max(0, n_hist - 2), n_hist)] + own
            else:  # a random subset of the history (different per head) plus the own pages
                k = min(n_hist, 3)
                pages = sorted(rng.choice(n_hist, size=k, replace=False).tolist()) + own if n_hist else own
            sel[c, h, : len(pages)] = pages
            cnt[c, h] = len(pages)
    return sel, cnt


def test_credited_pairs_match_brute_force():
    rng = np.random.default_rng(3)
    base = synth.WORKLOADS["tiny"]
    for kind in ("dense", "topk", "window"):
        # 4 query heads / 2 KV heads, pages of 8, chunks of 24 with a ragged last chunk of 13
        w = synth.scaled(base, f"acct_{kind}", n_q_heads=4, n_kv_heads=2, seq=85, chunk=24, page=8)
        sel, cnt = _selections(w, kind, rng)
        assert _count(w, sel, cnt) == _brute(w, sel, cnt), kind


def test_dense_credit_closed_form():
    """All pages selected: chunk c credits sum over its rows of (start + i + 1) keys."""
    w = synth.scaled(synth.WORKLOADS["tiny"], "acct_closed", n_q_heads=6, n_kv_heads=3, seq=100, chunk=32, page=8)
    sel, cnt = _selections(w, "dense", np.random.default_rng(0))
    got = _count(w, sel, cnt)
    for c in range(w.n_chunks):
        start, n = w.chunk_bounds(c)
        assert got[c] == sum(start + i + 1 for i in range(n)) * w.n_q_heads


def test_algorithmic_bytes_per_call():
    """Append: 2 KB per token and KV head at d = 128 (K, V read and written in bf16,
    both fp32 gradient rows zeroed) plus the 512-byte summary row of each page and
    head; selection: the chunk's Q once, each candidate's summary row once, plus the
    written set; state per 10K tokens: K/V bf16 + dK/dV fp32 + summaries (K/V on
    the host with offload)."""
    w = synth.WORKLOADS["sparse128k"]
    ns = types.SimpleNamespace(w=w, offload_grads=False)
    app, sel = bench.Step.hbm_bytes(ns)
    C, Hkv, Hq, d, P = w.chunk, w.n_kv_heads, w.n_q_heads, w.head_dim, w.page
    assert app[5] == C * Hkv * 2048 + (C // P) * Hkv * d * 4
    # gradient pools in host memory: no zeroing, one state byte per (page, KV head)
    app_off, _ = bench.Step.hbm_bytes(types.SimpleNamespace(w=w, offload_grads=True))
    assert app_off[5] == C * Hkv * 1024 + (C // P) * Hkv + (C // P) * Hkv * d * 4
    c = w.n_chunks - 1
    n_cand = c * C // P - w.n_sink
    assert sel[c] == C * Hq * d * 2 + n_cand * Hkv * d * 4 + 2 * n_cand * Hkv * 4 + Hkv * w.max_sel * 4
    assert sel[0] == Hkv * w.max_sel * 4  # nothing to score in the first chunk
    st = bench.state_bytes_per_10k(w)
    # the summary row of a page is shared by its P tokens: d * 4 / P bytes per token and head
    assert st["device"] == 10_000 * Hkv * d * (2 * 2 + 2 * 4) + 10_000 * Hkv * d * 4 // P
    assert st["host"] == 0
    w4 = synth.WORKLOADS["offload4m"]
    # K/V (bf16) and dK/dV (fp32) move to pinned host memory: only the summaries grow on the device
    off = bench.state_bytes_per_10k(synth.WORKLOADS["offload4m"])
    assert off["host"] == 10_000 * Hkv * d * (2 * 2 + 2 * 4) and off["device"] == st["device"] - off["host"]
    assert off["device"] == 10_000 * Hkv * d * 4 // P
    # fixed staging: two buffers of max_sel blocks per KV head, K/V bf16 and dK/dV fp32
    assert off["fixed_staging_device"] == 2 * Hkv * w4.max_sel * P * d * (2 * 2 + 2 * 4)
    kv_only = bench.state_bytes_per_10k(synth.scaled(w4, "kv_only", offload_grads=False))
    assert kv_only["host"] == 10_000 * Hkv * d * 2 * 2 and kv_only["device"] == st["device"] - kv_only["host"]


def test_host_link_bytes_hand_example():
    """The offload step's host-link bytes on a 3-chunk, 1-head example worked by hand:
    chunk 0 selects pages {0, 1} (own), chunk 1 {0 | 2, 3}, chunk 2 {1, 3 | 4, 5}.
    K/V: forward gathers 0 + 1 + 2 history blocks, reverse gathers 2 + 3 + 4, own pages
    written back 2 + 2 + 2.  Gradients, reverse order: chunk 2 zero-fills all four and
    writes them back; chunk 1 carries page 3, zero-fills 0 and 2 (never written back);
    chunk 0 carries page 0 and reads page 1 from the host (written back by chunk 2)."""
    w = synth.scaled(synth.WORKLOADS["tiny"], "link", n_q_heads=1, n_kv_heads=1, head_dim=64, page=128, seq=768,
                     chunk=256, top_k=-1, plants=0)
    sel = np.full((3, 1, 4), -1, dtype=np.int32)
    cnt = np.zeros((3, 1), dtype=np.int32)
    for c, pages in enumerate([[0, 1], [0, 2, 3], [1, 3, 4, 5]]):
        sel[c, 0, : len(pages)] = pages
        cnt[c, 0] = len(pages)
    esz = 2 if w.dtype == "bf16" else 4
    kv_blk, g_blk = 2 * 128 * 64 * esz, 2 * 128 * 64 * 4
    got = bench.host_link_bytes(w, sel, cnt, True)
    assert got == {"kv_in": 12 * kv_blk, "kv_out": 6 * kv_blk, "grad_in": 1 * g_blk, "grad_out": 9 * g_blk,
                   "grad_carried_on_device": 2 * g_blk}
    no_grads = bench.host_link_bytes(w, sel, cnt, False)
    assert no_grads["grad_in"] == no_grads["grad_out"] == no_grads["grad_carried_on_device"] == 0
    assert no_grads["kv_in"] == 12 * kv_blk and no_grads["kv_out"] == 6 * kv_blk
