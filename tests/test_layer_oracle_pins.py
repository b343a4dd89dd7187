"""Pins of the layer-step oracle (projections + rotary embedding + chunk-recurrent
paged attention) against things other than itself, on the CPU:

* the rotary embedding: its closed form for one pair, inverse = transpose,
  norms kept, and the relative-position property (the logit of a rotated query
  and key depends only on their distance);
* the chunked, paged layer step with the queries recomputed in the reverse sweep
  equals torch fp64 autograd of the unchunked layer (projections, rotation,
  scaled_dot_product_attention with an explicit visibility mask built from the
  selection) for dense, top-K and window selections: O and the gradients of X,
  Wq, Wk, Wv;
* central finite differences of the implied loss on tiny inputs;
* planted mistakes (a backward without the inverse rotation; K rotated the other
  way) fail these pins.
"""
import math

import numpy as np
import pytest
import torch

import oracle.layer_oracle as LO
import oracle.oomb_oracle as O


def test_rope_closed_form_and_properties():
    # one pair (d = 2): frequency theta^0 = 1, so (1, 0) at position p is (cos p, sin p)
    x = np.array([[[1.0, 0.0]]])
    for p in (0, 1, 5, 1000):
        np.testing.assert_allclose(LO.rope(x, p, 1e6)[0, 0], [math.cos(p), math.sin(p)], atol=1e-15)
    # d = 4, theta = 100: the second pair turns at 100^(-1/2) = 0.1 per position
    y = LO.rope(np.array([[[0.0, 2.0, 0.0, 0.0]]]), 3, 100.0)[0, 0]
    np.testing.assert_allclose(y, [0.0, 2 * math.cos(0.3), 0.0, 2 * math.sin(0.3)], atol=1e-15)
    rng = np.random.default_rng(0)
    a = rng.standard_normal((9, 3, 16))
    r = LO.rope(a, 17, 1e4)
    np.testing.assert_allclose(LO.rope(r, 17, 1e4, inverse=True), a, atol=1e-13)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(a, axis=-1), rtol=1e-13)
    q, k = rng.standard_normal((1, 1, 16)), rng.standard_normal((1, 1, 16))
    for m, n, shift in [(5, 2, 7), (40, 40, 123), (3, 11, 1000)]:
        d1 = float((LO.rope(q, m, 1e4) * LO.rope(k, n, 1e4)).sum())
        d2 = float((LO.rope(q, m + shift, 1e4) * LO.rope(k, n + shift, 1e4)).sum())
        assert abs(d1 - d2) < 1e-12 * max(1.0, abs(d1))


def _rope_t(x, theta):
    """Rotary embedding with torch ops (positions 0..N-1), for autograd."""
    n, _, d = x.shape
    half = d // 2
    freq = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / d)
    ang = torch.arange(n, dtype=torch.float64)[:, None] * freq[None, :]
    c, s = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return torch.cat([a * c - b * s, b * c + a * s], dim=-1)


def _autograd_layer(X, Wq, Wk, Wv, dO, Hq, Hkv, scale, theta, mask, bq=None, bk=None, bv=None):
    """Unchunked layer with torch autograd; mask [Hq, N, N] (True = visible)."""
    N = X.shape[0]
    d = Wq.shape[1] // Hq
    zq, zk = np.zeros(Hq * d), np.zeros(Hkv * d)
    src = dict(X=X, Wq=Wq, Wk=Wk, Wv=Wv, bq=zq if bq is None else bq, bk=zk if bk is None else bk,
               bv=zk if bv is None else bv)
    t = {k: torch.tensor(v, requires_grad=True) for k, v in src.items()}
    q = _rope_t((t["X"] @ t["Wq"] + t["bq"]).reshape(N, Hq, d), theta)
    k = _rope_t((t["X"] @ t["Wk"] + t["bk"]).reshape(N, Hkv, d), theta)
    v = (t["X"] @ t["Wv"] + t["bv"]).reshape(N, Hkv, d)
    G = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(0, 1)[None], k.transpose(0, 1).repeat_interleave(G, 0)[None],
        v.transpose(0, 1).repeat_interleave(G, 0)[None], attn_mask=torch.tensor(mask)[None], scale=scale)[0]
    o = o.transpose(0, 1)
    (o * torch.tensor(dO)).sum().backward()
    return o.detach().numpy(), {k: t[k].grad.numpy() for k in t}


def _mask_from_selection(sel, N, C, P, Hq, Hkv):
    """Query i (head hq) sees key j <= i when j's page is in the selection of i's
    chunk for KV head hq // G."""
    G = Hq // Hkv
    mask = np.zeros((Hq, N, N), dtype=bool)
    for ci, s in enumerate(range(0, N, C)):
        for hq in range(Hq):
            pages = set(int(p) for p in sel[ci][hq // G])
            for i in range(s, min(s + C, N)):
                for j in range(i + 1):
                    mask[hq, i, j] = (j // P) in pages
    return mask


def _problem(seed, N, Dm, Hq, Hkv, d):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((N, Dm))
    Wq = rng.standard_normal((Dm, Hq * d)) / math.sqrt(Dm)
    Wk = rng.standard_normal((Dm, Hkv * d)) / math.sqrt(Dm)
    Wv = rng.standard_normal((Dm, Hkv * d)) / math.sqrt(Dm)
    dO = rng.standard_normal((N, Hq, d))
    return rng, X, Wq, Wk, Wv, dO


@pytest.mark.parametrize("kind", ["dense", "topk", "window", "biased"])
def test_layer_step_equals_unchunked_autograd(kind):
    N, C, P, Hq, Hkv, d, Dm = 56, 16, 4, 4, 2, 8, 12
    theta = 1e4
    rng, X, Wq, Wk, Wv, dO = _problem(11, N, Dm, Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    order = rng.permutation(N // P + 2)
    kw = dict(top_k=-1) if kind == "dense" else dict(window=2) if kind == "window" else dict(top_k=3)
    bias = {}
    if kind == "biased":  # Qwen2.5-style projection biases, with a sparse selection
        bias = dict(bq=rng.standard_normal(Hq * d), bk=rng.standard_normal(Hkv * d),
                    bv=rng.standard_normal(Hkv * d))
    res = LO.layer_sweep(X, Wq, Wk, Wv, dO, Hq, Hkv, C, P, order, scale, theta, n_sink=1, **kw, **bias)
    if kind in ("topk", "biased"):  # the selection really drops pages
        assert len(res["sel"][-1][0]) < N // P
    mask = _mask_from_selection(res["sel"], N, C, P, Hq, Hkv)
    o_ref, g = _autograd_layer(X, Wq, Wk, Wv, dO, Hq, Hkv, scale, theta, mask, **bias)
    assert O.rel_l2(np.concatenate(res["O"]), o_ref) < 1e-12
    for name in ("X", "Wq", "Wk", "Wv"):
        assert O.rel_l2(res["d" + name], g[name]) < 1e-12, name
    if bias:
        for name in ("bq", "bk", "bv"):
            assert O.rel_l2(res["d" + name], g[name]) < 1e-12, name


def test_layer_step_finite_differences():
    N, C, P, Hq, Hkv, d, Dm = 24, 8, 4, 2, 1, 4, 3
    rng, X, Wq, Wk, Wv, dO = _problem(5, N, Dm, Hq, Hkv, d)
    order = list(range(N // P))
    base = LO.layer_sweep(X, Wq, Wk, Wv, dO, Hq, Hkv, C, P, order, 0.5, 1e4, top_k=1, n_sink=1)
    sel = base["sel"]
    assert len(sel[-1][0]) < N // P  # sparse: the last chunk drops history pages

    def loss(**kw):
        a = dict(X=X, Wq=Wq, Wk=Wk, Wv=Wv)
        a.update(kw)
        r = LO.layer_sweep(a["X"], a["Wq"], a["Wk"], a["Wv"], dO, Hq, Hkv, C, P, order, 0.5, 1e4,
                           sel_override=sel)
        return float((np.concatenate(r["O"]) * dO).sum())

    h = 1e-6
    for name, M in (("X", X), ("Wq", Wq), ("Wk", Wk), ("Wv", Wv)):
        num = np.zeros_like(M)
        for idx in np.ndindex(*M.shape):
            Mp, Mm = M.copy(), M.copy()
            Mp[idx] += h
            Mm[idx] -= h
            num[idx] = (loss(**{name: Mp}) - loss(**{name: Mm})) / (2 * h)
        assert O.rel_l2(base["d" + name], num) < 1e-6, name


def test_layer_planted_mistakes_are_caught(monkeypatch):
    """A backward that skips the inverse rotation, and a K rotated the other way,
    both fail the autograd pin."""
    N, C, P, Hq, Hkv, d, Dm = 32, 16, 4, 2, 1, 8, 6
    theta = 1e4
    rng, X, Wq, Wk, Wv, dO = _problem(2, N, Dm, Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    order = list(range(N // P))
    good = LO.rope
    mask = _mask_from_selection([[list(range(N // P))] * Hkv] * (N // C), N, C, P, Hq, Hkv)
    o_ref, g = _autograd_layer(X, Wq, Wk, Wv, dO, Hq, Hkv, scale, theta, mask)

    def no_inverse(x, pos0, th, inverse=False):
        return x if inverse else good(x, pos0, th)

    monkeypatch.setattr(LO, "rope", no_inverse)
    bad = LO.layer_sweep(X, Wq, Wk, Wv, dO, Hq, Hkv, C, P, order, scale, theta)
    assert O.rel_l2(bad["dWq"], g["Wq"]) > 1e-3
    calls = {"n": 0}

    def k_backwards(x, pos0, th, inverse=False):  # every second forward call is the K rotation
        if not inverse:
            calls["n"] += 1
            if x.shape[1] == Hkv and calls["n"] % 2 == 0:
                return good(x, pos0, th, inverse=True)
        return good(x, pos0, th, inverse)

    monkeypatch.setattr(LO, "rope", k_backwards)
    bad = LO.layer_sweep(X, Wq, Wk, Wv, dO, Hq, Hkv, C, P, order, scale, theta)
    assert O.rel_l2(np.concatenate(bad["O"]), o_ref) > 1e-3
    monkeypatch.setattr(LO, "rope", good)
    ok = LO.layer_sweep(X, Wq, Wk, Wv, dO, Hq, Hkv, C, P, order, scale, theta)
    assert O.rel_l2(ok["dWq"], g["Wq"]) < 1e-12
