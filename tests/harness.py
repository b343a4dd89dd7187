"""Shared helpers for the GPU parity tests: run a workload through the C ABI and
through the fp64 oracle on the same seeded inputs."""
from __future__ import annotations

import math
from typing import List, Optional

import numpy as np
import torch

import oracle.oomb_oracle as O
import paged_sparse_attention_gb300 as L
from paged_sparse_attention_gb300 import synth
from paged_sparse_attention_gb300.pool import PagedKVPool

TOL = {"fp32": 1e-5, "bf16": 1e-2}


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def make_chunks(w: synth.Workload, plants: bool = True):
    pt = synth.PlantTable(w) if (plants and w.plants > 0) else None
    return [synth.make_chunk(w, c, plants=pt) for c in range(w.n_chunks)], pt


def oracle_sweep(w: synth.Workload, chunks, order, scale: Optional[float] = None):
    scale = 1.0 / math.sqrt(w.head_dim) if scale is None else scale
    return O.chunked_sweep([{k: v.double().numpy() for k, v in ch.items()} for ch in chunks], list(order),
                           w.n_kv_heads, w.page, len(order), scale, w.top_k, w.n_sink,
                           window=w.window if w.window >= 0 else None)


def pad_sel(sel_list: List[np.ndarray], max_sel: int, dev):
    Hkv = len(sel_list)
    sel = torch.full((Hkv, max_sel), -1, dtype=torch.int32)
    cnt = torch.zeros(Hkv, dtype=torch.int32)
    for h, s in enumerate(sel_list):
        sel[h, : len(s)] = torch.from_numpy(np.asarray(s, dtype=np.int32))
        cnt[h] = len(s)
    return sel.to(dev), cnt.to(dev)


class GpuSweep:
    """Forward sweep (append, select, forward) then reverse sweep (recompute
    forward, backward) through the C ABI.  ``sel_override`` feeds given
    selections to the attention calls (the GPU selection is still computed and
    kept in ``gpu_sel``).  With ``offload`` the K/V pools live in pinned host
    memory and every chunk's selected pages are prefetched on a side stream into
    the staging buffer of its parity before its attention calls.  ``staged_append``:
    the append also writes the chunk's own pages into their staging slots and only
    the history pages are gathered; "deferred": the append writes the slots only and
    the side stream writes the own pages to the host pools afterwards."""

    def __init__(self, w: synth.Workload, chunks, order, dev="cuda", sel_override=None, scale=None,
                 num_phys: Optional[int] = None, offload: bool = False, offload_grads: bool = False,
                 staged_append=False):
        self.w = w
        self.dev = torch.device(dev)
        self.scale = 1.0 / math.sqrt(w.head_dim) if scale is None else scale
        n_phys = len(order) if num_phys is None else num_phys
        max_sel = w.max_sel if sel_override is None else max(w.max_sel, max(max(len(s) for s in so)
                                                                               for so in sel_override))
        self.max_sel = max_sel
        self.pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, n_phys, w.n_pages,
                                w.torch_dtype, self.dev, page_order=torch.as_tensor(order, dtype=torch.int32),
                                offload=offload, stage_max_sel=max_sel if offload else 0,
                                offload_grads=offload_grads)
        side = torch.cuda.Stream(device=self.dev, priority=-1) if offload else None
        main = torch.cuda.current_stream(self.dev)

        def stage(c, sel, cnt):
            """Prefetch chunk c's selected pages on the side stream; main waits for them."""
            if not offload:
                return
            side.wait_stream(main)  # selection (and the chunk's own pages) written
            L.oomb_prefetch(self.pool.handle, sel, cnt, c % 2, stream=side)
            main.wait_stream(side)
            L.oomb_pool_set_stage(self.pool.handle, c % 2)
        ws_sel = self.pool.workspace(L.OOMB_OP_SELECT, w.chunk)
        ws_bwd = self.pool.workspace(L.OOMB_OP_BWD, w.chunk)
        h = self.pool.handle
        self.gpu_sel, self.O, self.LSE, self.dQ, self.O2, self.LSE2 = [], [], [], [], [], []
        dev_chunks = []
        for c, ch in enumerate(chunks):
            start, n = w.chunk_bounds(c)
            g = {k: v.to(self.dev) for k, v in ch.items()}
            dev_chunks.append(g)
            if not staged_append:
                L.oomb_kv_append(h, g["k"], g["v"], start)
            sel = torch.full((w.n_kv_heads, max_sel), -1, dtype=torch.int32, device=self.dev)
            cnt = torch.zeros(w.n_kv_heads, dtype=torch.int32, device=self.dev)
            if w.window >= 0:  # a selection needs the history only
                L.oomb_window_select(h, start, n, w.window, w.n_sink, sel, cnt)
            else:
                L.oomb_page_select(h, g["q"], start, w.top_k, w.n_sink, sel, cnt, ws_sel)
            self.gpu_sel.append([sel[i, : int(cnt[i])].cpu().numpy() for i in range(w.n_kv_heads)])
            if sel_override is not None:
                sel, cnt = pad_sel(sel_override[c], max_sel, self.dev)
            if staged_append:  # own pages into their staging slots; only the history comes from the host
                append = L.oomb_kv_append_deferred if staged_append == "deferred" else L.oomb_kv_append_staged
                append(h, g["k"], g["v"], start, cnt, max_sel, c % 2)
                side.wait_stream(main)
                L.oomb_prefetch_pages(h, sel, cnt, c % 2, 0, start // w.page, stream=side)
                if staged_append == "deferred":  # the own pages to the host pools
                    L.oomb_kv_writeback(h, sel, cnt, c % 2, start // w.page, -(-(start + n) // w.page), stream=side)
                main.wait_stream(side)
                L.oomb_pool_set_stage(h, c % 2)
            else:
                stage(c, sel, cnt)
            o = torch.empty_like(g["q"])
            lse = torch.empty(w.n_q_heads, n, dtype=torch.float32, device=self.dev)
            L.oomb_chunk_attn_fwd(h, g["q"], start, sel, cnt, self.scale, o, lse)
            self.O.append(o)
            self.LSE.append(lse)
            g["sel"], g["cnt"] = sel, cnt
        self.dQ = [None] * len(chunks)
        for c in range(len(chunks) - 1, -1, -1):
            start, n = w.chunk_bounds(c)
            g = dev_chunks[c]
            stage(c, g["sel"], g["cnt"])
            if offload_grads:  # dK/dV blocks of the selection: from the host, or carried from chunk c + 1
                prev = dev_chunks[c + 1] if c + 1 < len(chunks) else None
                with torch.cuda.stream(side):
                    L.oomb_grad_prefetch(h, g["sel"], g["cnt"], prev["sel"] if prev else None,
                                         prev["cnt"] if prev else None, c % 2, stream=side)
                    if prev is not None:
                        L.oomb_grad_carry(h, g["sel"], g["cnt"], prev["sel"], prev["cnt"], c % 2, stream=side)
                main.wait_stream(side)
            o = torch.empty_like(g["q"])
            lse = torch.empty(w.n_q_heads, n, dtype=torch.float32, device=self.dev)
            L.oomb_chunk_attn_fwd(h, g["q"], start, g["sel"], g["cnt"], self.scale, o, lse)  # recompute
            dq = torch.empty_like(g["q"])
            L.oomb_chunk_attn_bwd(h, g["q"], o, g["do"], lse, start, g["sel"], g["cnt"], self.scale, dq, ws_bwd)
            if offload_grads:  # staged dK/dV back to the host pools
                side.wait_stream(main)
                L.oomb_grad_writeback(h, g["sel"], g["cnt"], c % 2, stream=side)
            self.dQ[c] = dq
            self.O2.insert(0, o)
            self.LSE2.insert(0, lse)
        if offload:
            main.wait_stream(side)
        self.err_bits = L.oomb_check(h)
        self.dK, self.dV = self.pool.logical_grads(w.seq)


def selection_matches(w, gpu_sel, ref_pool_state, q64, start, ora_sel):
    """GPU and oracle selections agree up to near-ties (relative gap < 1e-4)."""
    cand, scores = ref_pool_state
    swaps = 0
    for h in range(w.n_kv_heads):
        ok, n = O.near_tie_ok(gpu_sel[h], ora_sel[h], cand, scores[h], w.top_k)
        if not ok:
            return False, h
        swaps += n
    return True, swaps
