"""Plain float64 CPU oracle for one chunk-recurrent attention layer step: the Q/K/V
projections, the rotary position embedding and the paged sparse chunk attention,
forward in chunk order and backward replayed in reverse with the queries (and the
attention output) recomputed.

TEST INFRASTRUCTURE ONLY, like ``oomb_oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference arm of ``bench.py``
may import it; the CUDA library shares nothing with it.

It follows "Out of the Memory Barrier" (gist.science explainer): 2.A — the input
is processed chunk by chunk, activations are discarded after the forward and
recomputed on the fly just before the backward needs them; 2.B — K/V and their
gradients live in pages and are accumulated in place; 2.D — top-K page retrieval
(or, for the sparse layers of sparse-native models, a local window).

Readings where the pages are silent:
* the layer's trainable part on this path is the three projections
  Q = X Wq + bq, K = X Wk + bk, V = X Wv + bv (the biases are optional; Qwen2.5's
  projections carry them);
* the output projection and everything after it lie outside the attention path,
  so the gradient that arrives is dO, the gradient of the loss with respect to
  the attention output;
* the rotary embedding is the rotate-half form, pairs (i, i + d/2) turned by the
  angle position * theta^(-2i/d) at absolute positions (the form of the Qwen2.5
  models that the explainer's experiments use);
* K and V stay in the pool between the sweeps (the KV cache), so the reverse
  sweep recomputes only the queries and the attention output.

Matrix products via numpy are the only library steps.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .oomb_oracle import OraclePool, chunk_attn_bwd, chunk_attn_fwd, select_pages, window_pages

F64 = np.float64


def rope(x: np.ndarray, pos0: int, theta: float, inverse: bool = False) -> np.ndarray:
    """Rotary position embedding of x [n, H, d] at absolute positions pos0 ..
    pos0 + n - 1: the pair (x[i], x[i + d/2]) of every row is rotated by the angle
    position * theta^(-2i/d).  ``inverse`` rotates by minus that angle, which is
    the transpose of the rotation (the backward pass applies it to gradients)."""
    n, _, d = x.shape
    half = d // 2
    freq = theta ** (-2.0 * np.arange(half, dtype=F64) / d)
    ang = (pos0 + np.arange(n, dtype=F64))[:, None] * freq[None, :]
    if inverse:
        ang = -ang
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def layer_sweep(X: np.ndarray, Wq: np.ndarray, Wk: np.ndarray, Wv: np.ndarray, dO: np.ndarray,
                n_q_heads: int, n_kv_heads: int, chunk: int, page: int, phys_order: Sequence[int],
                scale: float, theta: float, top_k: int = -1, n_sink: int = 1,
                window: Optional[int] = None, sel_override=None, bq: Optional[np.ndarray] = None,
                bk: Optional[np.ndarray] = None, bv: Optional[np.ndarray] = None):
    """One layer step over the whole sequence.

    X [N, Dm] (the layer's input activations), Wq [Dm, Hq*d], Wk and Wv
    [Dm, Hkv*d], dO [N, Hq, d] (gradient of the loss with respect to the attention
    output).  Forward sweep, chunk c in order: Q, K, V of the chunk's tokens from X,
    the rotary embedding on Q and K, K/V appended to the paged pool, pages
    selected, attention forward.  Reverse sweep, chunk c from the last: Q recomputed
    from X, the attention forward recomputed, the attention backward (dK/dV added
    into the pool), and — the chunk's keys being seen only by queries of this and
    later chunks, all done by now — the chunk's dK/dV complete: the gradients go
    back through the rotary embedding (its inverse rotation) and the projections.

    bq [Hq*d], bk and bv [Hkv*d] are optional projection biases (None = none).

    Returns a dict: O (list per chunk), dX [N, Dm], dWq, dWk, dWv, dbq, dbk, dbv
    (zeros where there is no bias), sel.
    """
    N, Dm = X.shape
    Hq, Hkv = n_q_heads, n_kv_heads
    d = Wq.shape[1] // Hq
    n_pages = -(-N // page)
    pool = OraclePool(Hkv, d, page, len(phys_order), n_pages)
    order = list(phys_order)
    starts = list(range(0, N, chunk))
    used = 0
    out = {"O": [], "sel": []}

    zq, zk = np.zeros(Hq * d, F64), np.zeros(Hkv * d, F64)
    bq = zq if bq is None else bq
    bk = zk if bk is None else bk
    bv = zk if bv is None else bv

    def project_q(s, n):
        return rope((X[s:s + n] @ Wq + bq).reshape(n, Hq, d), s, theta)

    for s in starts:
        n = min(chunk, N - s)
        q = project_q(s, n)
        k = rope((X[s:s + n] @ Wk + bk).reshape(n, Hkv, d), s, theta)
        v = (X[s:s + n] @ Wv + bv).reshape(n, Hkv, d)
        npg = (s + n - 1) // page - s // page + 1
        pool.append(k, v, s, order[used:used + npg])
        used += npg
        ci = len(out["sel"])
        if sel_override is not None:
            sel = sel_override[ci]
        elif window is not None:
            sel = [window_pages(s, n, page, window, n_sink)] * Hkv
        else:
            sel = select_pages(pool, q, s, top_k, n_sink)
        o, _ = chunk_attn_fwd(pool, q, s, sel, scale)
        out["O"].append(o)
        out["sel"].append(sel)

    dX = np.zeros_like(X, dtype=F64)
    dWq, dWk, dWv = (np.zeros_like(W, dtype=F64) for W in (Wq, Wk, Wv))
    dbq, dbk, dbv = np.zeros_like(zq), np.zeros_like(zk), np.zeros_like(zk)
    for ci in range(len(starts) - 1, -1, -1):
        s = starts[ci]
        n = min(chunk, N - s)
        q = project_q(s, n)  # recomputed (explainer 2.A)
        o, lse = chunk_attn_fwd(pool, q, s, out["sel"][ci], scale)
        dq = chunk_attn_bwd(pool, q, o, dO[s:s + n], lse, s, out["sel"][ci], scale)
        dk_all, dv_all = pool.logical_grads()
        dk, dv = dk_all[s:s + n], dv_all[s:s + n]
        gq = rope(dq, s, theta, inverse=True).reshape(n, Hq * d)
        gk = rope(dk, s, theta, inverse=True).reshape(n, Hkv * d)
        gv = dv.reshape(n, Hkv * d)
        xc = X[s:s + n]
        dWq += xc.T @ gq
        dWk += xc.T @ gk
        dWv += xc.T @ gv
        dbq += gq.sum(axis=0)
        dbk += gk.sum(axis=0)
        dbv += gv.sum(axis=0)
        dX[s:s + n] = gq @ Wq.T + gk @ Wk.T + gv @ Wv.T
    out.update(dX=dX, dWq=dWq, dWk=dWk, dWv=dWv, dbq=dbq, dbk=dbk, dbv=dbv)
    return out
