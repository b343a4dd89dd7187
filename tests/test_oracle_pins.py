"""Pins of the fp64 oracle against things other than itself (CPU only).

* dense equivalence: with every page selected the chunked, paged result equals
  unchunked causal attention, which in turn equals torch's fp64
  scaled_dot_product_attention and its autograd gradients (a library routine);
* central finite differences of the implied loss sum(dO * O) on tiny inputs,
  with a sparse selection held fixed;
* closed forms: zero queries give uniform attention (O = mean of visible V,
  LSE = log of the visible count); constant V gives O = V (rows of P sum to 1);
* page-table permutations leave every output bit-identical;
* the page score equals the brute-force mean of the group's query-key logit block,
  and the top-K equals a full sort;
* a hand-worked selection fixture (tests/golden/);
* planted pages are selected;
* planted mistakes in the oracle are caught by these pins.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.oomb_oracle as O
from paged_sparse_attention_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_seq(rng, N, Hq, Hkv, d):
    return (rng.standard_normal((N, Hq, d)), rng.standard_normal((N, Hkv, d)),
            rng.standard_normal((N, Hkv, d)), rng.standard_normal((N, Hq, d)))


def _split(Q, K, V, dO, C):
    out = []
    for s in range(0, Q.shape[0], C):
        out.append({"q": Q[s:s + C], "k": K[s:s + C], "v": V[s:s + C], "do": dO[s:s + C]})
    return out


def _sweep(Q, K, V, dO, C, P, scale, order, top_k=-1, n_sink=1, sel=None):
    chunks = _split(Q, K, V, dO, C)
    Hkv = K.shape[1]
    num_phys = len(order)
    return O.chunked_sweep(chunks, order, Hkv, P, num_phys, scale, top_k, n_sink, sel)


def _cat(res, key):
    return np.concatenate(res[key], axis=0 if key != "LSE" else 1)


@pytest.mark.parametrize("N,C,P,Hq,Hkv,d", [(96, 32, 8, 4, 2, 8), (100, 40, 8, 3, 1, 16),
                                              (64, 64, 16, 2, 2, 4)])
def test_dense_equivalence_and_sdpa(N, C, P, Hq, Hkv, d):
    rng = np.random.default_rng(N * 31 + C)
    Q, K, V, dO = _rand_seq(rng, N, Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    n_pages = -(-N // P)
    order = rng.permutation(n_pages + 3)
    res = _sweep(Q, K, V, dO, C, P, scale, order)
    Od, Ld = O.dense_causal_attention(Q, K, V, scale)
    dQd, dKd, dVd = O.dense_causal_attention_grad(Q, K, V, dO, scale)
    dK, dV = res["pool"].logical_grads()
    assert O.rel_l2(_cat(res, "O"), Od) < 1e-12
    assert O.rel_l2(_cat(res, "LSE"), Ld) < 1e-12
    assert O.rel_l2(np.concatenate(res["dQ"]), dQd) < 1e-12
    assert O.rel_l2(dK, dKd) < 1e-12
    assert O.rel_l2(dV, dVd) < 1e-12

    # library pin: torch fp64 SDPA + autograd (GQA by repeat_interleave = consecutive groups)
    G = Hq // Hkv
    tq = torch.tensor(Q.transpose(1, 0, 2), dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(K.transpose(1, 0, 2), dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(V.transpose(1, 0, 2), dtype=torch.float64, requires_grad=True)
    to = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk.repeat_interleave(G, 0)[None], tv.repeat_interleave(G, 0)[None],
        is_causal=True, scale=scale)[0]
    (to * torch.tensor(dO.transpose(1, 0, 2))).sum().backward()
    assert O.rel_l2(Od, to.detach().numpy().transpose(1, 0, 2)) < 1e-12
    assert O.rel_l2(dQd, tq.grad.numpy().transpose(1, 0, 2)) < 1e-12
    assert O.rel_l2(dKd, tk.grad.numpy().transpose(1, 0, 2)) < 1e-12
    assert O.rel_l2(dVd, tv.grad.numpy().transpose(1, 0, 2)) < 1e-12
    # LSE pin: log-sum-exp by scipy on the explicit causal logits
    from scipy.special import logsumexp
    for hq in range(Hq):
        s = scale * Q[:, hq] @ K[:, hq // G].T
        for i in (0, N // 2, N - 1):
            assert abs(Ld[hq, i] - logsumexp(s[i, :i + 1])) < 1e-12


def _loss(Q, K, V, dO, C, P, scale, order, sel):
    res = _sweep(Q, K, V, dO, C, P, scale, order, sel=sel)
    return float((np.concatenate(res["O"]) * dO).sum())


@pytest.mark.parametrize("top_k", [-1, 1])
def test_finite_differences(top_k):
    N, C, P, Hq, Hkv, d = 16, 8, 2, 2, 1, 4
    rng = np.random.default_rng(7 + top_k)
    Q, K, V, dO = _rand_seq(rng, N, Hq, Hkv, d)
    scale = 0.5
    order = rng.permutation(N // P)
    res = _sweep(Q, K, V, dO, C, P, scale, order, top_k=top_k, n_sink=1)
    sel = res["sel"]
    if top_k == 1:  # selection of the last chunk really is sparse
        assert len(sel[1][0]) < N // P
    dQ = np.concatenate(res["dQ"])
    dK, dV = res["pool"].logical_grads()
    h = 1e-6
    for name, X, G in (("q", Q, dQ), ("k", K, dK), ("v", V, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(*X.shape):
            Xp = X.copy(); Xp[idx] += h
            Xm = X.copy(); Xm[idx] -= h
            args = {"q": Q, "k": K, "v": V}
            args[name] = Xp
            lp = _loss(args["q"], args["k"], args["v"], dO, C, P, scale, order, sel)
            args[name] = Xm
            lm = _loss(args["q"], args["k"], args["v"], dO, C, P, scale, order, sel)
            num[idx] = (lp - lm) / (2 * h)
        assert O.rel_l2(G, num) < 1e-6, name


def test_closed_forms_uniform_and_rowsum():
    N, C, P, Hq, Hkv, d = 48, 16, 8, 2, 1, 8
    rng = np.random.default_rng(3)
    _, K, V, dO = _rand_seq(rng, N, Hq, Hkv, d)
    Q = np.zeros((N, Hq, d))
    order = rng.permutation(N // P)
    res = _sweep(Q, K, V, dO, C, P, 0.3, order)
    Ocat = np.concatenate(res["O"])
    L = np.concatenate(res["LSE"], axis=1)
    for i in range(N):
        for hq in range(Hq):
            np.testing.assert_allclose(Ocat[i, hq], V[: i + 1, 0].mean(axis=0), rtol=1e-13, atol=1e-14)
            assert abs(L[hq, i] - math.log(i + 1)) < 1e-13
    # constant values: O == that constant for any logits (rows of P sum to 1)
    Q2 = rng.standard_normal((N, Hq, d)) * 3
    Vc = np.broadcast_to(np.arange(d, dtype=float), (N, Hkv, d)).copy()
    res2 = _sweep(Q2, K, Vc, dO, C, P, 1.0, order, top_k=2)
    for Oc in res2["O"]:
        np.testing.assert_allclose(Oc, np.broadcast_to(np.arange(d, dtype=float), Oc.shape), rtol=0, atol=1e-12)
    # LSE >= max visible logit (dense run: every earlier key visible)
    res3 = _sweep(Q2, K, V, dO, C, P, 1.0, order)
    L2 = np.concatenate(res3["LSE"], axis=1)
    for i in (0, 17, 47):
        s = Q2[i, 0] @ K[: i + 1, 0].T
        assert L2[0, i] >= s.max() - 1e-12


def test_permutation_invariance_bitwise():
    N, C, P, Hq, Hkv, d = 80, 32, 8, 4, 2, 8
    rng = np.random.default_rng(11)
    Q, K, V, dO = _rand_seq(rng, N, Hq, Hkv, d)
    n_pages = N // P
    a = _sweep(Q, K, V, dO, C, P, 0.35, list(range(n_pages)), top_k=2)
    b = _sweep(Q, K, V, dO, C, P, 0.35, list(rng.permutation(n_pages + 5)), top_k=2)
    for key in ("O", "LSE", "dQ"):
        for x, y in zip(a[key], b[key]):
            assert np.array_equal(x, y), key
    for x, y in zip(a["sel"], b["sel"]):
        for u, v in zip(x, y):
            assert np.array_equal(u, v)
    ga, gb = a["pool"].logical_grads(), b["pool"].logical_grads()
    assert np.array_equal(ga[0], gb[0]) and np.array_equal(ga[1], gb[1])


def test_score_identity_and_topk_sort():
    N, P, Hq, Hkv, d = 64 * 8, 8, 6, 2, 16
    rng = np.random.default_rng(5)
    K = rng.standard_normal((N, Hkv, d))
    V = rng.standard_normal((N, Hkv, d))
    n_pages = N // P
    pool = O.OraclePool(Hkv, d, P, n_pages, n_pages)
    pool.append(K, V, 0, list(rng.permutation(n_pages)))
    q_start = N  # a query chunk right after the history (its own pages not stored)
    q = rng.standard_normal((40, Hq, d))
    cand, scores = O.page_scores(pool, q, q_start, n_sink=2)
    G = Hq // Hkv
    for h in range(Hkv):
        for i, p in enumerate(cand):
            block = np.einsum("nge,te->ngt", q[:, h * G:(h + 1) * G], K[p * P:(p + 1) * P, h])
            assert abs(block.mean() - scores[h, i]) < 1e-12
    # top-k == full python sort on (-score, page)
    pool.n_tokens = N  # history only
    for k in (1, 5, 17):
        for h in range(Hkv):
            ref = sorted(range(cand.size), key=lambda i: (-scores[h, i], int(cand[i])))[:k]
            order = np.lexsort((cand, -scores[h]))[:k]
            assert sorted(int(cand[i]) for i in ref) == sorted(int(cand[i]) for i in order)


def test_select_ties_and_structure():
    # all pages of equal score: ties must go to the lowest logical pages
    N, P, Hkv, d = 32, 4, 1, 4
    K = np.ones((N, Hkv, d))
    pool = O.OraclePool(Hkv, d, P, 16, 16)
    pool.append(K, K, 0, list(range(8)))
    q = np.ones((6, 2, d))
    pool.append(np.ones((6, Hkv, d)), np.ones((6, Hkv, d)), N, [9, 8])
    sel = O.select_pages(pool, q, N, top_k=3, n_sink=1)
    assert sel[0].tolist() == [0, 1, 2, 3, 8, 9]
    # top_k < 0 keeps everything; first chunk has no sink
    assert O.select_pages(pool, q, N, -1, 1)[0].tolist() == list(range(10))
    assert O.select_pages(pool, np.ones((4, 2, d)), 0, 3, 1)[0].tolist() == [0]


def test_golden_handworked_selection():
    with open(os.path.join(GOLDEN, "select_handworked.json")) as f:
        g = json.load(f)
    K = np.array(g["keys"], dtype=float)[:, None, :]
    pool = O.OraclePool(1, K.shape[2], g["page_size"], g["num_phys"], g["num_phys"])
    pool.append(K, K, 0, g["phys_order"][: len(K) // g["page_size"]])
    q = np.array(g["queries"], dtype=float)[:, None, :]
    q_start = len(K)
    n_own = -(-len(q) // g["page_size"])
    pool.append(np.zeros((len(q), 1, K.shape[2])), np.zeros((len(q), 1, K.shape[2])), q_start,
                g["phys_order"][len(K) // g["page_size"]: len(K) // g["page_size"] + n_own])
    cand, scores = O.page_scores(pool, q, q_start, g["n_sink"])
    np.testing.assert_allclose(scores[0], g["expected_scores"], rtol=0, atol=1e-15)
    sel = O.select_pages(pool, q, q_start, g["top_k"], g["n_sink"])
    assert sel[0].tolist() == g["expected_selection"]


def test_planted_pages_selected():
    w = synth.scaled(synth.WORKLOADS["sparse128k"], "plant_mini", n_q_heads=4, n_kv_heads=2,
                     seq=4096, chunk=512, page=64, top_k=8, plants=4, head_dim=64)
    plants = synth.PlantTable(w)
    order = synth.page_order(w).tolist()
    chunks = [{k: v.double().numpy() for k, v in synth.make_chunk(w, c, plants=plants).items()}
              for c in range(w.n_chunks)]
    pool = O.OraclePool(w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages)
    used = 0
    for c, ch in enumerate(chunks):
        start, n = w.chunk_bounds(c)
        npg = -(-n // w.page)
        pool.append(ch["k"], ch["v"], start, order[used:used + npg])
        used += npg
        sel = O.select_pages(pool, ch["q"], start, w.top_k, w.n_sink)
        for h in range(w.n_kv_heads):
            for p in plants.planted.get((c, h), []):
                assert p in set(sel[h].tolist()), (c, h, p)


def test_planted_mistakes_are_caught(monkeypatch):
    """A dropped term in the backward (D = rowsum(dO * O) left out) must fail the
    dense-equivalence pin."""
    N, C, P, Hq, Hkv, d = 16, 8, 4, 2, 1, 4
    rng = np.random.default_rng(9)
    Q, K, V, dO = _rand_seq(rng, N, Hq, Hkv, d)
    order = list(range(N // P))
    good = O.chunk_attn_bwd

    def bad_bwd(pool, q, o, do, lse, q_start, sel, scale):  # drops the D term
        return good(pool, q, np.zeros_like(o), do, lse, q_start, sel, scale)

    monkeypatch.setattr(O, "chunk_attn_bwd", bad_bwd)
    res = _sweep(Q, K, V, dO, C, P, 0.5, order)
    monkeypatch.setattr(O, "chunk_attn_bwd", good)
    dQd, _, _ = O.dense_causal_attention_grad(Q, K, V, dO, 0.5)
    assert O.rel_l2(np.concatenate(res["dQ"]), dQd) > 1e-3

    res_ok = _sweep(Q, K, V, dO, C, P, 0.5, order)
    assert O.rel_l2(np.concatenate(res_ok["dQ"]), dQd) < 1e-12


def _select_ties_to_higher_page(pool, q, q_start, top_k, n_sink):
    """A planted mistake: the oracle's selection with the tie-break reversed (ties go
    to the higher logical page), everything else as in the oracle."""
    n_hist = q_start // pool.P
    own = np.arange(n_hist, (q_start + q.shape[0] - 1) // pool.P + 1)
    sinks = np.arange(0, min(n_sink, n_hist))
    cand, scores = O.page_scores(pool, q, q_start, n_sink)
    out = []
    for h in range(pool.Hkv):
        order = np.lexsort((-cand, -scores[h]))
        chosen = cand if cand.size <= top_k else cand[order[:top_k]]
        out.append(np.sort(np.concatenate([sinks, chosen, own]).astype(np.int64)))
    return out


def test_planted_flipped_tie_break_fails_fixture():
    """The hand-worked fixture has an exact tie at the K-th place: a selection that
    gives ties to the higher page must disagree with it (and the oracle agrees)."""
    with open(os.path.join(GOLDEN, "select_handworked.json")) as f:
        g = json.load(f)
    K = np.array(g["keys"], dtype=float)[:, None, :]
    pool = O.OraclePool(1, K.shape[2], g["page_size"], g["num_phys"], g["num_phys"])
    pool.append(K, K, 0, g["phys_order"][: len(K) // g["page_size"]])
    q = np.array(g["queries"], dtype=float)[:, None, :]
    n_own = -(-len(q) // g["page_size"])
    pool.append(np.zeros((len(q), 1, K.shape[2])), np.zeros((len(q), 1, K.shape[2])), len(K),
                g["phys_order"][len(K) // g["page_size"]: len(K) // g["page_size"] + n_own])
    bad = _select_ties_to_higher_page(pool, q, len(K), g["top_k"], g["n_sink"])
    assert bad[0].tolist() != g["expected_selection"]
    assert O.select_pages(pool, q, len(K), g["top_k"], g["n_sink"])[0].tolist() == g["expected_selection"]


def test_near_tie_rule():
    cand = np.arange(1, 6)
    scores = np.array([1.0, 0.5, 0.50000001, 0.2, 0.1])
    # the swap of pages 2 and 3, tied to 1e-8 of max|score| at the K-th place: allowed
    assert O.near_tie_ok(np.array([0, 1, 2]), np.array([0, 1, 3]), cand, scores, 2)[0]
    # page 4 (0.2) instead of page 3 (the K-th, 0.50000001): far from the boundary
    assert not O.near_tie_ok(np.array([0, 1, 4]), np.array([0, 1, 3]), cand, scores, 2)[0]


def test_near_tie_rule_rejects_other_differences():
    """Differences that no near-tie explains: a page more or fewer than the oracle
    (even a near-tied one), a page outside the candidates, and a swap whose gap to the
    K-th score is just above 1e-4 of max|score| (just below passes)."""
    cand = np.arange(1, 7)
    scores = np.array([1.0, 0.8, 0.6, 0.6 - 0.5e-4, 0.6 - 2e-4, 0.1])
    ora = np.array([0, 1, 2, 3, 7])  # sink 0, top-3 {1, 2, 3}, own page 7
    kth_swap = np.array([0, 1, 2, 4, 7])  # page 4 (gap 0.5e-4) for the K-th page 3
    assert O.near_tie_ok(kth_swap, ora, cand, scores, 3)[0]
    assert not O.near_tie_ok(np.array([0, 1, 2, 5, 7]), ora, cand, scores, 3)[0]  # gap 2e-4
    assert not O.near_tie_ok(np.array([0, 1, 2, 3, 4, 7]), ora, cand, scores, 3)[0]  # one page more
    assert not O.near_tie_ok(np.array([0, 1, 2, 7]), ora, cand, scores, 3)[0]  # one page fewer
    assert not O.near_tie_ok(np.array([1, 2, 3, 4, 7]), ora, cand, scores, 3)[0]  # sink dropped for a near-tie
    assert not O.near_tie_ok(np.array([0, 1, 2, 8, 7]), ora, cand, scores, 3)[0]  # not a candidate


# -- local sliding-window selection ------------------------------------------------
def test_golden_handworked_window():
    with open(os.path.join(GOLDEN, "window_handworked.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        got = O.window_pages(case["q_start"], case["n_q"], g["page_size"], case["window"], case["n_sink"])
        assert got.tolist() == case["expected"], case


def _sdpa_masked(Q, K, V, dO, scale, mask):
    """torch fp64 SDPA with an explicit boolean visibility mask [N, N] (library
    routine), GQA by repeat_interleave; returns O and the gradients of sum(dO*O)."""
    G = Q.shape[1] // K.shape[1]
    tq = torch.tensor(Q.transpose(1, 0, 2), dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(K.transpose(1, 0, 2), dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(V.transpose(1, 0, 2), dtype=torch.float64, requires_grad=True)
    to = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk.repeat_interleave(G, 0)[None], tv.repeat_interleave(G, 0)[None],
        attn_mask=torch.tensor(mask)[None, None], scale=scale)[0]
    (to * torch.tensor(dO.transpose(1, 0, 2))).sum().backward()
    t = lambda x: x.numpy().transpose(1, 0, 2)  # noqa: E731
    return t(to.detach()), t(tq.grad), t(tk.grad), t(tv.grad)


def _window_mask(N, C, P, window, n_sink):
    """Token-level visibility written from the definition in words: query i sees
    key j <= i when j lies in a sink page before i's chunk, in one of the `window`
    pages right before i's chunk, or in i's own chunk."""
    mask = np.zeros((N, N), dtype=bool)
    for i in range(N):
        first = (i // C) * C // P  # first page of i's chunk
        for j in range(i + 1):
            pj = j // P
            mask[i, j] = (pj >= first) or (first - window <= pj) or (pj < min(n_sink, first))
    return mask


@pytest.mark.parametrize("N,C,P,Hq,Hkv,d,window,n_sink", [
    (96, 32, 8, 4, 2, 8, 0, 0),     # chunk-local attention
    (96, 32, 8, 4, 2, 8, 2, 1),
    (100, 24, 4, 3, 1, 16, 3, 2),   # ragged last chunk
    (64, 16, 4, 2, 2, 4, 100, 1),   # window covers the history: dense
])
def test_window_sweep_equals_masked_sdpa(N, C, P, Hq, Hkv, d, window, n_sink):
    rng = np.random.default_rng(N + 7 * window + n_sink)
    Q, K, V, dO = _rand_seq(rng, N, Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    order = rng.permutation(-(-N // P) + 2)
    res = O.chunked_sweep(_split(Q, K, V, dO, C), order, Hkv, P, len(order), scale, n_sink=n_sink,
                          window=window)
    Ot, dQt, dKt, dVt = _sdpa_masked(Q, K, V, dO, scale, _window_mask(N, C, P, window, n_sink))
    dK, dV = res["pool"].logical_grads()
    assert O.rel_l2(_cat(res, "O"), Ot) < 1e-12
    assert O.rel_l2(np.concatenate(res["dQ"]), dQt) < 1e-12
    assert O.rel_l2(dK, dKt) < 1e-12
    assert O.rel_l2(dV, dVt) < 1e-12
    if window == 0 and n_sink == 0:  # block-diagonal: each chunk is plain causal attention on its own
        for s in range(0, N, C):
            Oc, _ = O.dense_causal_attention(Q[s:s + C], K[s:s + C], V[s:s + C], scale)
            assert O.rel_l2(Ot[s:s + C], Oc) < 1e-12


def test_window_off_by_one_is_caught(monkeypatch):
    """A window one page too short must fail the masked-SDPA pin."""
    N, C, P, Hq, Hkv, d = 64, 16, 4, 2, 1, 4
    rng = np.random.default_rng(5)
    Q, K, V, dO = _rand_seq(rng, N, Hq, Hkv, d)
    good = O.window_pages

    def short(q_start, n_q, page_size, window, n_sink):
        return good(q_start, n_q, page_size, max(0, window - 1), n_sink)

    monkeypatch.setattr(O, "window_pages", short)
    res = O.chunked_sweep(_split(Q, K, V, dO, C), list(range(N // P)), Hkv, P, N // P, 0.5, n_sink=1, window=2)
    monkeypatch.setattr(O, "window_pages", good)
    Ot, _, _, _ = _sdpa_masked(Q, K, V, dO, 0.5, _window_mask(N, C, P, 2, 1))
    assert O.rel_l2(_cat(res, "O"), Ot) > 1e-3


def test_degenerate_cases():
    """G = 1 is multi-head attention (no repeat needed): the paged sweep equals torch
    fp64 SDPA on the unrepeated heads; one chunk (C = N) is plain causal attention;
    a K at least the number of candidates selects everything, so the sweep equals
    the dense run bit for bit."""
    rng = np.random.default_rng(21)
    N, P, H, d = 48, 8, 3, 8
    Q, K, V, dO = _rand_seq(rng, N, H, H, d)
    scale = 1.0 / math.sqrt(d)
    order = rng.permutation(N // P)
    for C in (16, N):  # several chunks, and a single chunk
        res = _sweep(Q, K, V, dO, C, P, scale, order)
        tq = torch.tensor(Q.transpose(1, 0, 2), requires_grad=True)
        tk = torch.tensor(K.transpose(1, 0, 2), requires_grad=True)
        tv = torch.tensor(V.transpose(1, 0, 2), requires_grad=True)
        to = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None], is_causal=True,
                                                              scale=scale)[0]
        (to * torch.tensor(dO.transpose(1, 0, 2))).sum().backward()
        dK, dV = res["pool"].logical_grads()
        assert O.rel_l2(_cat(res, "O"), to.detach().numpy().transpose(1, 0, 2)) < 1e-12
        assert O.rel_l2(np.concatenate(res["dQ"]), tq.grad.numpy().transpose(1, 0, 2)) < 1e-12
        assert O.rel_l2(dK, tk.grad.numpy().transpose(1, 0, 2)) < 1e-12
        assert O.rel_l2(dV, tv.grad.numpy().transpose(1, 0, 2)) < 1e-12
    dense = _sweep(Q, K, V, dO, 16, P, scale, order, top_k=-1, n_sink=1)
    big_k = _sweep(Q, K, V, dO, 16, P, scale, order, top_k=N // P, n_sink=1)
    for key in ("O", "LSE"):
        for a, b in zip(dense[key], big_k[key]):
            assert np.array_equal(a, b)
    for a, b in zip(dense["sel"], big_k["sel"]):
        assert all(np.array_equal(x, y) for x, y in zip(a, b))
