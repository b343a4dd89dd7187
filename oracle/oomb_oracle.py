"""Plain float64 CPU oracle for paged sparse chunk attention (OOMB's hot path).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this module.  The CUDA
library never calls it and shares no code, table or helper with it; the two are
fed the same seeded inputs and compared.

It follows the method as "Out of the Memory Barrier" describes it (four web
pages: the arXiv abstract on mlsanity.com, the gist.science explainer, a
podcast summary and a Chinese digest):

* chunk-recurrent processing, forward in chunk order and backward replayed in
  reverse with the forward recomputed (gist.science explainer, 2.A
  "Chunk-Recurrent Training with Activation Recomputation");
* K/V and their gradients kept in fixed-size pages reached through a page table,
  gradients accumulated in place (explainer, 2.B "Paged KV Cache and Gradient
  Management"; abstract);
* top-K page retrieval by a representative (mean) key per page, with the sink
  page and the chunk's own pages always kept (explainer, 2.D "Page-Level Sparse
  Attention"; the scoring rule is fixed as mean key per page, ties to the lower
  page index);
* attention itself is textbook causal softmax attention with grouped KV heads,
  restricted to the keys of the selected pages.

Readings taken where the pages are silent: the query side of the page score is
the plain mean of the chunk's queries over all tokens and all query heads of the
KV group; the sink is logical
page 0 (``n_sink`` leading pages) and does not count toward K; the chunk's own
pages are "local"; ties go to the lower *logical* page index; the causal mask is
``key position <= query position`` on absolute positions; LSE is the natural log
of the sum of exp of the scaled logits; no gradient flows through selection.

Every function is written for clarity, not speed: matrix products via numpy are
the only library steps, with no blocking or reordering.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import numpy as np

F64 = np.float64


class OraclePool:
    """Paged K/V store and paged gradient pool sharing one page table.

    Layout mirrors the statement of the problem, not any kernel: pools are
    [num_phys, Hkv, P, d] float64, ``phi`` maps logical page -> physical page
    (-1 = unmapped).  (explainer, 2.B: fixed-size pages hold the KV cache and its
    gradients; abstract: paged memory manager for the KV cache and its
    gradients.)
    """

    def __init__(self, n_kv_heads: int, head_dim: int, page_size: int,
                 num_phys_pages: int, max_logical_pages: int):
        self.Hkv, self.d, self.P = n_kv_heads, head_dim, page_size
        shape = (num_phys_pages, n_kv_heads, page_size, head_dim)
        self.K = np.zeros(shape, F64)
        self.V = np.zeros(shape, F64)
        self.dK = np.zeros(shape, F64)
        self.dV = np.zeros(shape, F64)
        self.phi = np.full(max_logical_pages, -1, np.int64)
        self.n_tokens = 0

    # -- paged store ---------------------------------------------------------
    def append(self, k: np.ndarray, v: np.ndarray, first_token: int,
               new_phys: Sequence[int]) -> None:
        """Write a chunk's K/V ([n, Hkv, d]) into pages, next free page first.

        ``new_phys`` lists the physical pages handed out, in order, for the
        logical pages this append opens (explainer, lay summary "Trick A: the
        paged filing system": new KV goes onto the next blank page, no copying).
        Gradient rows of the written tokens start at zero.
        """
        n = k.shape[0]
        if first_token != self.n_tokens:
            raise ValueError("appends must be contiguous")
        if first_token % self.P != 0:
            raise ValueError("appends start on a page boundary")
        p_first = first_token // self.P
        p_last = (first_token + n - 1) // self.P if n > 0 else p_first - 1
        new_phys = list(new_phys)
        if len(new_phys) != p_last - p_first + 1:
            raise ValueError("one physical page per opened logical page")
        for i, p in enumerate(range(p_first, p_last + 1)):
            self.phi[p] = new_phys[i]
        for t in range(n):
            pos = first_token + t
            p, r = divmod(pos, self.P)
            ph = self.phi[p]
            self.K[ph, :, r, :] = k[t]
            self.V[ph, :, r, :] = v[t]
            self.dK[ph, :, r, :] = 0.0
            self.dV[ph, :, r, :] = 0.0
        self.n_tokens = first_token + n

    def tokens_in_page(self, p: int) -> int:
        return max(0, min(self.P, self.n_tokens - p * self.P))

    def page_keys(self, p: int, h: int) -> np.ndarray:
        return self.K[self.phi[p], h, : self.tokens_in_page(p), :]

    def page_values(self, p: int, h: int) -> np.ndarray:
        return self.V[self.phi[p], h, : self.tokens_in_page(p), :]

    def summary(self, p: int, h: int) -> np.ndarray:
        """Representative vector of a page: the mean key over the tokens present
        (explainer, 2.D: pages are ranked for top-K retrieval by an averaged
        representative vector; the mean key per page is the fixed scoring rule)."""
        return self.page_keys(p, h).mean(axis=0)

    def gather(self, pages: Sequence[int], h: int):
        """Keys, values and absolute positions of the tokens of ``pages``."""
        ks, vs, pos = [], [], []
        for p in pages:
            m = self.tokens_in_page(p)
            ks.append(self.page_keys(p, h))
            vs.append(self.page_values(p, h))
            pos.append(p * self.P + np.arange(m))
        if not ks:
            return (np.zeros((0, self.d)), np.zeros((0, self.d)), np.zeros(0, np.int64))
        return np.concatenate(ks), np.concatenate(vs), np.concatenate(pos)

    def scatter_grad(self, pages: Sequence[int], h: int, dk: np.ndarray, dv: np.ndarray):
        """Accumulate key/value gradients in place into the paged gradient pool
        (explainer, 2.B "In-place Gradient Accumulation")."""
        o = 0
        for p in pages:
            m = self.tokens_in_page(p)
            ph = self.phi[p]
            self.dK[ph, h, :m, :] += dk[o:o + m]
            self.dV[ph, h, :m, :] += dv[o:o + m]
            o += m

    def logical_grads(self, n_tokens: Optional[int] = None):
        """dK, dV as token-major [n, Hkv, d] arrays read through the table."""
        n = self.n_tokens if n_tokens is None else n_tokens
        dk = np.zeros((n, self.Hkv, self.d), F64)
        dv = np.zeros((n, self.Hkv, self.d), F64)
        for t in range(n):
            p, r = divmod(t, self.P)
            dk[t] = self.dK[self.phi[p], :, r, :]
            dv[t] = self.dV[self.phi[p], :, r, :]
        return dk, dv


# -- selection ------------------------------------------------------------------
def page_scores(pool: OraclePool, q: np.ndarray, q_start: int, n_sink: int):
    """Scores of the candidate history pages of one chunk, per KV head.

    q: [n_q, Hq, d].  Candidates are the complete pages before the chunk minus the
    sink pages.  score[h][p] = qbar_h . kbar_{p,h}, where qbar_h is the mean of
    the chunk's queries over all tokens and all query heads of group h.
    Returns (candidates, scores[Hkv, n_cand]).
    """
    n_q, Hq, d = q.shape
    G = Hq // pool.Hkv
    n_hist = q_start // pool.P
    cand = np.arange(min(n_sink, n_hist), n_hist)
    scores = np.zeros((pool.Hkv, cand.size), F64)
    for h in range(pool.Hkv):
        qbar = q[:, h * G:(h + 1) * G, :].reshape(-1, d).mean(axis=0)
        for i, p in enumerate(cand):
            scores[h, i] = float(qbar @ pool.summary(int(p), h))
    return cand, scores


def select_pages(pool: OraclePool, q: np.ndarray, q_start: int, top_k: int,
                 n_sink: int) -> List[np.ndarray]:
    """Selected logical pages per KV head, ascending (explainer, 2.D).

    S = sink pages  U  top-K candidates by score (ties: lower logical page)  U
    the chunk's own pages.  With ``top_k < 0`` or no more than K candidates, every
    candidate is kept.
    """
    n_q = q.shape[0]
    n_hist = q_start // pool.P
    own = np.arange(n_hist, (q_start + n_q - 1) // pool.P + 1) if n_q > 0 else np.arange(0)
    sinks = np.arange(0, min(n_sink, n_hist))
    cand, scores = page_scores(pool, q, q_start, n_sink)
    out = []
    for h in range(pool.Hkv):
        if top_k < 0 or cand.size <= top_k:
            chosen = cand
        else:
            order = np.lexsort((cand, -scores[h]))  # primary: score desc; then page asc
            chosen = cand[order[:top_k]]
        out.append(np.sort(np.concatenate([sinks, chosen, own]).astype(np.int64)))
    return out


def window_pages(q_start: int, n_q: int, page_size: int, window: int, n_sink: int) -> np.ndarray:
    """Local sliding-window selection, the same for every KV head (explainer, 2.D
    "Page-Level Sparse Attention": sparse-native models use local attention in
    their sparse layers).  Reading: page granularity and no scoring; the chunk
    keeps the sink pages, the ``window`` complete history pages right before it,
    and its own pages.  Written as a set union, ascending."""
    n_hist = q_start // page_size
    own = set(range(n_hist, (q_start + n_q - 1) // page_size + 1))
    sinks = set(range(0, min(n_sink, n_hist)))
    recent = set(p for p in range(n_hist) if n_hist - p <= window)
    return np.array(sorted(sinks | recent | own), dtype=np.int64)


# -- attention -------------------------------------------------------------------
def _row_softmax_stats(s: np.ndarray):
    """m, LSE and P of a masked logit matrix (masked entries are -inf)."""
    m = s.max(axis=1)
    lse = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
    p = np.exp(s - lse[:, None])
    return m, lse, p


def chunk_attn_fwd(pool: OraclePool, q: np.ndarray, q_start: int,
                   sel: Sequence[np.ndarray], scale: float):
    """Causal GQA attention of one query chunk over the selected pages.

    q: [n_q, Hq, d].  Query head hq reads KV head hq // G.  For row i (absolute
    position q_start+i) the keys are every token of the selected pages with
    position <= q_start+i.  Returns O [n_q, Hq, d] and LSE [Hq, n_q] (natural log
    of the scaled logits' exp-sum).
    """
    n_q, Hq, d = q.shape
    G = Hq // pool.Hkv
    O = np.zeros((n_q, Hq, d), F64)
    LSE = np.zeros((Hq, n_q), F64)
    qpos = q_start + np.arange(n_q)
    for hq in range(Hq):
        h = hq // G
        Kj, Vj, kpos = pool.gather(sel[h], h)
        s = scale * (q[:, hq, :] @ Kj.T)
        s = np.where(kpos[None, :] <= qpos[:, None], s, -np.inf)
        _, lse, p = _row_softmax_stats(s)
        O[:, hq, :] = p @ Vj
        LSE[hq] = lse
    return O, LSE


def chunk_attn_bwd(pool: OraclePool, q: np.ndarray, o: np.ndarray, do: np.ndarray,
                   lse: np.ndarray, q_start: int, sel: Sequence[np.ndarray], scale: float):
    """Analytic backward of ``chunk_attn_fwd`` for a fixed selection.

    P = exp(scale*q.k - LSE) (recomputed from the saved LSE, explainer 2.A),
    dP = dO V^T, D = rowsum(dO * O), dS = P * (dP - D),
    dQ = scale * dS K, dK += scale * dS^T Q, dV += P^T dO,
    with dK/dV added in place into the paged gradient pool (explainer 2.B).
    Returns dQ [n_q, Hq, d].
    """
    n_q, Hq, d = q.shape
    G = Hq // pool.Hkv
    dQ = np.zeros((n_q, Hq, d), F64)
    qpos = q_start + np.arange(n_q)
    for hq in range(Hq):
        h = hq // G
        Kj, Vj, kpos = pool.gather(sel[h], h)
        s = scale * (q[:, hq, :] @ Kj.T)
        mask = kpos[None, :] <= qpos[:, None]
        p = np.where(mask, np.exp(np.where(mask, s, 0.0) - lse[hq][:, None]), 0.0)
        dp = do[:, hq, :] @ Vj.T
        D = (do[:, hq, :] * o[:, hq, :]).sum(axis=1)
        ds = p * (dp - D[:, None])
        dQ[:, hq, :] = scale * (ds @ Kj)
        pool.scatter_grad(sel[h], h, scale * (ds.T @ q[:, hq, :]), p.T @ do[:, hq, :])
    return dQ


# -- whole sweep -----------------------------------------------------------------
def chunked_sweep(chunks, phys_order: Sequence[int], n_kv_heads: int, page_size: int,
                  num_phys: int, scale: float, top_k: int = -1, n_sink: int = 1,
                  sel_override=None, window: Optional[int] = None):
    """Chunk-recurrent forward (in order) then backward (reverse order).

    ``chunks`` is a list of dicts with float64 arrays q/k/v/do.  Physical pages are
    handed out in ``phys_order``.  Pages are chosen by top-K retrieval, or by the
    local window when ``window`` is given.  Returns per-chunk O, LSE, dQ,
    selections and the pool (whose dK/dV hold the accumulated key/value
    gradients).
    """
    d = chunks[0]["q"].shape[2]
    total = sum(c["q"].shape[0] for c in chunks)
    max_logical = -(-total // page_size)
    pool = OraclePool(n_kv_heads, d, page_size, num_phys, max_logical)
    order = list(phys_order)
    next_free = 0
    res = {"O": [], "LSE": [], "dQ": [None] * len(chunks), "sel": [], "starts": []}
    start = 0
    for ci, c in enumerate(chunks):
        n = c["q"].shape[0]
        p0 = start // page_size
        p1 = (start + n - 1) // page_size
        newp = order[next_free:next_free + (p1 - p0 + 1)]
        next_free += p1 - p0 + 1
        pool.append(c["k"], c["v"], start, newp)
        if sel_override is not None:
            sel = sel_override[ci]
        elif window is not None:
            sel = [window_pages(start, n, page_size, window, n_sink)] * n_kv_heads
        else:
            sel = select_pages(pool, c["q"], start, top_k, n_sink)
        O, L = chunk_attn_fwd(pool, c["q"], start, sel, scale)
        res["O"].append(O)
        res["LSE"].append(L)
        res["sel"].append(sel)
        res["starts"].append(start)
        start += n
    for ci in range(len(chunks) - 1, -1, -1):
        c = chunks[ci]
        st = res["starts"][ci]
        O, L = chunk_attn_fwd(pool, c["q"], st, res["sel"][ci], scale)  # recompute
        res["dQ"][ci] = chunk_attn_bwd(pool, c["q"], O, c["do"], L, st, res["sel"][ci], scale)
    res["pool"] = pool
    return res


# -- unchunked dense reference (self-check only) ---------------------------------
def dense_causal_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Plain causal softmax attention over the whole sequence, GQA by repeating
    each KV head for its G consecutive query heads.  Q: [N, Hq, d],
    K/V: [N, Hkv, d].  Returns O [N, Hq, d], LSE [Hq, N]."""
    N, Hq, d = Q.shape
    G = Hq // K.shape[1]
    O = np.zeros_like(Q, dtype=F64)
    LSE = np.zeros((Hq, N), F64)
    causal = np.tril(np.ones((N, N), dtype=bool))
    for hq in range(Hq):
        s = scale * (Q[:, hq] @ K[:, hq // G].T)
        s = np.where(causal, s, -np.inf)
        _, lse, p = _row_softmax_stats(s)
        O[:, hq] = p @ V[:, hq // G]
        LSE[hq] = lse
    return O, LSE


def dense_causal_attention_grad(Q, K, V, dO, scale: float):
    """Analytic gradients of sum(dO * O) for ``dense_causal_attention``."""
    N, Hq, d = Q.shape
    G = Hq // K.shape[1]
    O, LSE = dense_causal_attention(Q, K, V, scale)
    dQ = np.zeros_like(Q, dtype=F64)
    dK = np.zeros_like(K, dtype=F64)
    dV = np.zeros_like(V, dtype=F64)
    causal = np.tril(np.ones((N, N), dtype=bool))
    for hq in range(Hq):
        h = hq // G
        s = scale * (Q[:, hq] @ K[:, h].T)
        p = np.where(causal, np.exp(np.where(causal, s, 0.0) - LSE[hq][:, None]), 0.0)
        dp = dO[:, hq] @ V[:, h].T
        D = (dO[:, hq] * O[:, hq]).sum(axis=1)
        ds = p * (dp - D[:, None])
        dQ[:, hq] = scale * ds @ K[:, h]
        dK[:, h] += scale * ds.T @ Q[:, hq]
        dV[:, h] += p.T @ dO[:, hq]
    return dQ, dK, dV


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    """Relative L2 error ||a - b|| / ||b||."""
    a = np.asarray(a, F64)
    b = np.asarray(b, F64)
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (den if den > 0 else 1.0))


def near_tie_ok(gpu_sel: np.ndarray, ora_sel: np.ndarray, cand: np.ndarray,
                scores: np.ndarray, top_k: int, rel_gap: float = 1e-4) -> Tuple[bool, int]:
    """Selections agree up to swaps of near-tied pages across the K-th boundary.

    Two pages are near-tied when |s_a - s_b| / max|s| < rel_gap over the
    candidates.  Returns (ok, number of swapped pages).
    """
    g = set(int(x) for x in gpu_sel)
    o = set(int(x) for x in ora_sel)
    if g == o:
        return True, 0
    if top_k < 0 or cand.size <= top_k:
        return False, len(g ^ o)
    idx = {int(p): i for i, p in enumerate(cand)}
    extra = g - o
    missing = o - g
    if len(extra) != len(missing) or any(p not in idx for p in extra | missing):
        return False, len(extra) + len(missing)
    order = np.lexsort((cand, -scores))
    kth = scores[order[top_k - 1]]
    scale = np.abs(scores).max()
    scale = scale if scale > 0 else 1.0
    for p in extra | missing:
        if abs(scores[idx[p]] - kth) / scale >= rel_gap:
            return False, len(extra)
    return True, len(extra)
