"""One attention layer's chunk-recurrent training step through the C ABI.

"Out of the Memory Barrier" (gist.science explainer, 2.A "Chunk-Recurrent Training
with Activation Recomputation"): the layer input X is processed chunk by chunk.
Forward sweep, chunk c in order: Q, K, V projected from X (optional biases), the
rotary embedding on Q and K, K/V appended to the paged pool, pages selected, the
attention forward.  Reverse sweep, chunk c from the last: Q recomputed from X, the
attention forward recomputed, the attention backward (dK/dV added into the paged
gradient pool); the chunk's keys are seen only by queries of this and later chunks,
all done by now, so its dK/dV are complete and go back through the rotary embedding
(inverse rotation) and the projections: dX, dWq, dWk, dWv and the bias gradients.

This module only orders calls; every operation is a liboomb entry point (GEMMs on
cuBLASLt through oomb_gemm, the rotation in oomb_bias_rope, the attention path).
torch provides the buffers.  Gradient GEMMs run in fp32 (the projection GEMMs in
the layer's dtype with fp32 accumulation).
"""
from __future__ import annotations

import math
from typing import List, Optional

import torch

from . import _lib as L
from .pool import PagedKVPool


class LayerStep:
    """Weights Wq [Dm, Hq*d], Wk and Wv [Dm, Hkv*d] (the pool's dtype, device), biases
    fp32 [H*d] or None.  Selection: top-K (``top_k``, ``n_sink``) or a local window
    (``window`` >= 0)."""

    def __init__(self, pool: PagedKVPool, Wq, Wk, Wv, bq=None, bk=None, bv=None, chunk: int = 4096,
                 theta: float = 1e6, top_k: int = -1, n_sink: int = 1, window: int = -1,
                 gemm_workspace_bytes: int = 32 << 20):
        self.pool, self.chunk, self.theta = pool, chunk, theta
        self.top_k, self.n_sink, self.window = top_k, n_sink, window
        self.Hq, self.Hkv, self.d, self.P = pool.Hq, pool.Hkv, pool.d, pool.P
        self.dev = pool.device
        self.W = {"q": Wq, "k": Wk, "v": Wv}
        self.b = {"q": bq, "k": bk, "v": bv}
        self.Dm = Wq.shape[0]
        self.scale = 1.0 / math.sqrt(self.d)
        self.ws = torch.empty(gemm_workspace_bytes, dtype=torch.uint8, device=self.dev)
        # fp32 copies of the weights for the gradient GEMMs (a cast through oomb_bias_rope)
        self.W32 = {}
        for key, w in self.W.items():
            w32 = torch.empty(w.shape, dtype=torch.float32, device=self.dev)
            L.oomb_bias_rope(w, None, w32, w.numel() // (w.shape[0] * 2), 0, 0.0, 0)
            self.W32[key] = w32

    # ------------------------------------------------------------------ pieces
    def _project(self, x, key: int, H: int, pos0: int, rotate: bool):
        """[n, H, d] in the pool's dtype: rotation(pos0..) (x W + b)."""
        n = x.shape[0]
        acc = torch.empty((n, H * self.d), dtype=torch.float32, device=self.dev)
        L.oomb_gemm(x, self.W[key], acc, workspace=self.ws)
        out = torch.empty((n, H, self.d), dtype=self.pool.dtype, device=self.dev)
        L.oomb_bias_rope(acc, self.b[key], out, H, pos0, self.theta, 1 if rotate else 0)
        return out

    def _select(self, q, start: int, sel, cnt, ws_sel):
        h = self.pool.handle
        if self.window >= 0:
            L.oomb_window_select(h, start, q.shape[0], self.window, self.n_sink, sel, cnt)
        else:
            L.oomb_page_select(h, q, start, self.top_k, self.n_sink, sel, cnt, ws_sel)

    def max_sel(self) -> int:
        own = -(-self.chunk // self.P)
        if self.window >= 0:
            return self.n_sink + self.window + own
        if self.top_k < 0:
            return self.pool.max_logical
        return self.n_sink + self.top_k + own

    # ------------------------------------------------------------------ the step
    def run(self, X, dO, sel_override: Optional[List] = None) -> dict:
        """X [N, Dm] (pool dtype, device), dO [N, Hq, d] (pool dtype, device).
        ``sel_override[c]``: (sel, count) device tensors fed to chunk c's attention
        instead of the library's own selection (which is still computed and returned).
        Returns O (per chunk), sel (the library's selections, per chunk), dX, dWq, dWk,
        dWv, dbq, dbk, dbv (fp32; the bias gradients are zero where there is no bias)."""
        pool, h, dev = self.pool, self.pool.handle, self.dev
        N, Dm, Hq, Hkv, d = X.shape[0], self.Dm, self.Hq, self.Hkv, self.d
        starts = list(range(0, N, self.chunk))
        L.oomb_pool_reset(h)
        max_sel = self.max_sel()
        ws_sel = pool.workspace(L.OOMB_OP_SELECT, self.chunk)
        ws_bwd = pool.workspace(L.OOMB_OP_BWD, self.chunk)
        out = {"O": [], "sel": []}
        att = []  # the selection each chunk's attention used
        for ci, s in enumerate(starts):
            n = min(self.chunk, N - s)
            x = X[s:s + n]
            q = self._project(x, "q", Hq, s, True)
            k = self._project(x, "k", Hkv, s, True)
            v = self._project(x, "v", Hkv, s, False)
            L.oomb_kv_append(h, k, v, s)
            sel = torch.full((Hkv, max_sel), -1, dtype=torch.int32, device=dev)
            cnt = torch.zeros(Hkv, dtype=torch.int32, device=dev)
            self._select(q, s, sel, cnt, ws_sel)
            out["sel"].append((sel, cnt))
            a_sel = sel_override[ci] if sel_override is not None else (sel, cnt)
            att.append(a_sel)
            o = torch.empty_like(q)
            lse = torch.empty((Hq, n), dtype=torch.float32, device=dev)
            L.oomb_chunk_attn_fwd(h, q, s, a_sel[0], a_sel[1], self.scale, o, lse)
            out["O"].append(o)
        f32 = torch.float32
        dX = torch.empty((N, Dm), dtype=f32, device=dev)
        dW = {key: torch.zeros(self.W[key].shape, dtype=f32, device=dev) for key in "qkv"}
        db = {key: torch.zeros((1, self.W[key].shape[1]), dtype=f32, device=dev) for key in "qkv"}
        ones = torch.ones((1, self.chunk), dtype=f32, device=dev)
        for ci in range(len(starts) - 1, -1, -1):
            s = starts[ci]
            n = min(self.chunk, N - s)
            x = X[s:s + n]
            q = self._project(x, "q", Hq, s, True)  # recomputed (explainer 2.A)
            o = torch.empty_like(q)
            lse = torch.empty((Hq, n), dtype=torch.float32, device=dev)
            a_sel = att[ci]
            L.oomb_chunk_attn_fwd(h, q, s, a_sel[0], a_sel[1], self.scale, o, lse)
            dq = torch.empty_like(q)
            L.oomb_chunk_attn_bwd(h, q, o, dO[s:s + n], lse, s, a_sel[0], a_sel[1], self.scale, dq, ws_bwd)
            # the chunk's own dK/dV are complete: back through the rotation and projections
            g = {"q": torch.empty((n, Hq * d), dtype=f32, device=dev),
                 "k": torch.empty((n, Hkv * d), dtype=f32, device=dev),
                 "v": torch.empty((n, Hkv * d), dtype=f32, device=dev)}
            L.oomb_grad_gather(h, s, g["k"].view(n, Hkv, d), g["v"].view(n, Hkv, d))
            L.oomb_bias_rope(dq, None, g["q"], Hq, s, self.theta, 2)
            L.oomb_bias_rope(g["k"], None, g["k"], Hkv, s, self.theta, 2)
            x32 = torch.empty((n, Dm), dtype=f32, device=dev)
            L.oomb_bias_rope(x, None, x32, Dm // 2, 0, 0.0, 0)  # cast
            first = True
            for key in "qkv":
                L.oomb_gemm(x32, g[key], dW[key], trans_a=True, beta=1.0, workspace=self.ws)
                L.oomb_gemm(ones[:, :n], g[key], db[key], beta=1.0, workspace=self.ws)
                L.oomb_gemm(g[key], self.W32[key], dX[s:s + n], trans_b=True, beta=0.0 if first else 1.0,
                            workspace=self.ws)
                first = False
        out.update(dX=dX, dWq=dW["q"], dWk=dW["k"], dWv=dW["v"], dbq=db["q"][0], dbk=db["k"][0], dbv=db["v"][0])
        return out
