"""GPU parity of the chunk-recurrent layer step (projections + rotary embedding +
paged sparse attention, queries recomputed in the reverse sweep) against the fp64
layer oracle: O of every chunk and the gradients of X, Wq, Wk, Wv and the biases.

The oracle computes Q, K, V in float64 from the same bf16- (or fp32-) valued X and
weights; the GPU rounds them to the layer's dtype before attention, so bf16 cases
are held to relative L2 1e-2 and fp32 cases to 1e-5.  The attention runs on the
oracle's selection (the GPU's own selection is checked against it separately).
"""
import math

import numpy as np
import pytest
import torch

import oracle.layer_oracle as LO
import oracle.oomb_oracle as O
import paged_sparse_attention_gb300 as L
from paged_sparse_attention_gb300 import synth
from paged_sparse_attention_gb300.layer import LayerStep
from paged_sparse_attention_gb300.pool import PagedKVPool

from harness import f64, pad_sel

pytestmark = pytest.mark.gpu

CASES = {
    # tensor-core geometry (head_dim = page = 128), GQA 2:1, top-2 + sink + own, biases
    "bf16_topk_bias": dict(dtype="bf16", N=1024, chunk=256, P=128, Hq=4, Hkv=2, d=128, Dm=256, top_k=2, n_sink=1,
                           window=-1, bias=True),
    # the same geometry with a local window of 2 pages (sparse-native layers), no biases
    "bf16_window": dict(dtype="bf16", N=1024, chunk=256, P=128, Hq=4, Hkv=2, d=128, Dm=128, top_k=-1, n_sink=1,
                        window=2, bias=False),
    # fp32 (SIMT attention, fp32 GEMMs): dense, ragged last chunk, biases
    "fp32_dense_bias": dict(dtype="fp32", N=600, chunk=128, P=64, Hq=2, Hkv=1, d=64, Dm=64, top_k=-1, n_sink=1,
                            window=-1, bias=True),
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_sparse_attention_gb300 import build
    build.build()
    L.load()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _inputs(cfg, seed=11):
    g = torch.Generator().manual_seed(seed)
    dt = torch.float32 if cfg["dtype"] == "fp32" else torch.bfloat16
    N, Dm, Hq, Hkv, d = cfg["N"], cfg["Dm"], cfg["Hq"], cfg["Hkv"], cfg["d"]
    X = torch.randn(N, Dm, generator=g).to(dt)
    Wq = (torch.randn(Dm, Hq * d, generator=g) / math.sqrt(Dm)).to(dt)
    Wk = (torch.randn(Dm, Hkv * d, generator=g) / math.sqrt(Dm)).to(dt)
    Wv = (torch.randn(Dm, Hkv * d, generator=g) / math.sqrt(Dm)).to(dt)
    dO = torch.randn(N, Hq, d, generator=g).to(dt)
    b = None
    if cfg["bias"]:
        b = [0.1 * torch.randn(H * d, generator=g) for H in (Hq, Hkv, Hkv)]
    return X, Wq, Wk, Wv, dO, b


@pytest.mark.parametrize("name", list(CASES))
def test_layer_step_matches_oracle(name):
    cfg = CASES[name]
    X, Wq, Wk, Wv, dO, b = _inputs(cfg)
    N, P, chunk = cfg["N"], cfg["P"], cfg["chunk"]
    Hq, Hkv, d = cfg["Hq"], cfg["Hkv"], cfg["d"]
    n_pages = -(-N // P)
    order = torch.randperm(n_pages, generator=torch.Generator().manual_seed(5)).to(torch.int32)
    scale = 1.0 / math.sqrt(d)
    theta = 1e6
    window = cfg["window"] if cfg["window"] >= 0 else None
    f = lambda t: None if t is None else t.double().numpy()  # noqa: E731
    ref = LO.layer_sweep(f(X), f(Wq), f(Wk), f(Wv), f(dO), Hq, Hkv, chunk, P, order.tolist(), scale, theta,
                         cfg["top_k"], cfg["n_sink"], window=window, bq=f(b[0]) if b else None,
                         bk=f(b[1]) if b else None, bv=f(b[2]) if b else None)
    dev = torch.device("cuda")
    dt = X.dtype
    pool = PagedKVPool(Hq, Hkv, d, P, n_pages, n_pages, dt, dev, page_order=order)
    step = LayerStep(pool, Wq.to(dev), Wk.to(dev), Wv.to(dev), *(t.to(dev) for t in b) if b else (None,) * 3,
                     chunk=chunk, theta=theta, top_k=cfg["top_k"], n_sink=cfg["n_sink"], window=cfg["window"])
    max_sel = step.max_sel()
    override = [pad_sel(s, max_sel, dev) for s in ref["sel"]]
    out = step.run(X.to(dev), dO.to(dev), sel_override=override)
    assert L.oomb_check(pool.handle) == 0
    tol = 1e-5 if cfg["dtype"] == "fp32" else 1e-2
    for c in range(len(ref["O"])):
        assert O.rel_l2(f64(out["O"][c]), ref["O"][c]) < tol, ("O", c)
        got = [out["sel"][c][0][h, : int(out["sel"][c][1][h])].cpu().tolist() for h in range(Hkv)]
        assert got == [s.tolist() for s in ref["sel"][c]], ("selection", c)
    for key in ("dX", "dWq", "dWk", "dWv"):
        assert O.rel_l2(f64(out[key]), ref[key]) < tol, key
    if b:
        for key in ("dbq", "dbk", "dbv"):
            assert O.rel_l2(f64(out[key]), ref[key]) < tol, key
    pool.close()


def test_bias_rope_matches_oracle_rotation():
    """The rotation alone at large absolute positions (4M tokens in): forward and
    inverse against the oracle's rotary embedding, fp32 in and out, and the inverse
    undoing the forward."""
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(3)
    n, H, d, pos0, theta = 64, 3, 128, 4_194_304 - 64, 1e6
    x = torch.randn(n, H, d, generator=g)
    bias = torch.randn(H * d, generator=g)
    y = torch.empty(n, H, d, device=dev)
    L.oomb_bias_rope(x.to(dev), bias.to(dev), y, H, pos0, theta, 1)
    ref = LO.rope(x.double().numpy() + bias.double().numpy().reshape(H, d)[None], pos0, theta)
    assert O.rel_l2(f64(y), ref) < 1e-6
    z = torch.empty_like(y)
    L.oomb_bias_rope(y, None, z, H, pos0, theta, 2)
    assert O.rel_l2(f64(z), LO.rope(ref, pos0, theta, inverse=True)) < 1e-6
    assert O.rel_l2(f64(z), x.double().numpy() + bias.double().numpy().reshape(H, d)[None]) < 1e-6


@pytest.mark.parametrize("ta,tb", [(False, False), (True, False), (False, True)])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_gemm_matches_numpy(dtype, ta, tb):
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(4)
    dt = torch.float32 if dtype == "fp32" else torch.bfloat16
    m, n, k = 96, 80, 112
    A = torch.randn(*((k, m) if ta else (m, k)), generator=g).to(dt)
    B = torch.randn(*((n, k) if tb else (k, n)), generator=g).to(dt)
    C0 = torch.randn(m, n, generator=g)
    C = C0.to(dev)
    ws = torch.empty(32 << 20, dtype=torch.uint8, device=dev)
    L.oomb_gemm(A.to(dev), B.to(dev), C, trans_a=ta, trans_b=tb, alpha=0.5, beta=2.0, workspace=ws)
    a = A.double().numpy()
    bb = B.double().numpy()
    ref = 0.5 * ((a.T if ta else a) @ (bb.T if tb else bb)) + 2.0 * C0.double().numpy()
    assert O.rel_l2(f64(C), ref) < 1e-6
