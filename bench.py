"""Benchmark: one chunk-recurrent attention step (forward sweep + reverse sweep)
of one attention layer through the liboomb C ABI on one GB300 per rank.

A step = for every chunk in order: append K/V to the paged pool, select pages,
forward attention; then for every chunk in reverse: recompute the forward (not for
the last chunk, whose O and LSE are still in their buffers) and run the backward
(dQ written, dK/dV accumulated into the paged fp32 gradient pool).
This is the attention part of OOMB's chunk-recurrent training step ("Out of the
Memory Barrier", gist.science explainer 2.A-2.D) for one layer.

Metric: credited fwd+bwd attention TFLOP/s (14 d FLOPs per selected, causally
visible (query, key) pair per query head; the recomputed forward is not credited)
and tokens/s per layer.  Multi-GPU runs are independent replicas (the path has no
exchange step); `value` sums all ranks.

  python bench.py [--workload dense32k] [--steps K] [--warmup W] [--impl oomb|reference]
"""
from __future__ import annotations

import argparse
import gc
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged sparse chunk-attn fwd+bwd TFLOP/s and tokens/s/layer at 1 GB300; % roofline"
UNIT = "TFLOP/s"
# used when the machine has no measured-peaks file: GB300 figures measured earlier on
# this pool (copy 6783 GB/s; bf16 dense GEMM 1875.1 TFLOP/s burst, 1690.3 sustained),
# close to the published fallback of 6.8 TB/s and 1.9 / 1.7 PFLOP/s
FALLBACK_PEAKS = {"hbm_gbs": 6783.0, "bf16_tflops": 1875.1, "bf16_tflops_sustained": 1690.3,
                  "source": "fallback (no measured-peaks file on this machine): GB300 copy and cuBLAS bf16 "
                            "figures measured earlier on this pool"}


_T0 = time.time()


def log(msg: str) -> None:
    """Progress line on stderr (the JSON result goes alone to stdout)."""
    sys.stderr.write(f"[bench {time.time() - _T0:7.1f}s] {msg}\n")
    sys.stderr.flush()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d.setdefault("source", "measured (MEASURED_PEAKS.json)")
        return d
    return dict(FALLBACK_PEAKS)


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 200 ms."""

    def __init__(self, index: int):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 7:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ------------------------------------------------------------------ workload
class Step:
    """Device buffers and the per-chunk call sequence of one benchmark step."""

    def __init__(self, w, dev, host_inputs=False):
        import torch

        import paged_sparse_attention_gb300 as L
        from paged_sparse_attention_gb300 import synth
        from paged_sparse_attention_gb300.pool import PagedKVPool

        self.L, self.torch, self.w, self.dev = L, torch, w, dev
        self.scale = 1.0 / math.sqrt(w.head_dim)
        order = synth.page_order(w)
        self.offload = bool(w.offload)
        self.offload_grads = bool(w.offload and w.offload_grads)
        self.pool = PagedKVPool(w.n_q_heads, w.n_kv_heads, w.head_dim, w.page, w.num_phys, w.n_pages,
                                w.torch_dtype, dev, page_order=order, offload=self.offload,
                                stage_max_sel=w.max_sel if self.offload else 0, offload_grads=self.offload_grads)
        plants = synth.PlantTable(w) if w.plants > 0 else None
        # inputs generated per chunk (seeded) on the device -- or on the host and uploaded,
        # keeping the host copies, when a test needs the same tensors for the oracle --
        # and resident for the whole run
        self.chunks, self.host_chunks = [], []
        for c in range(w.n_chunks):
            if host_inputs:
                hc = synth.make_chunk(w, c, device="cpu", plants=plants)
                self.host_chunks.append(hc)
                self.chunks.append({k: v.to(dev) for k, v in hc.items()})
            else:
                self.chunks.append(synth.make_chunk(w, c, device=dev, plants=plants))
        C = w.chunk
        self.ws_sel = self.pool.workspace(L.OOMB_OP_SELECT, C)
        self.ws_bwd = self.pool.workspace(L.OOMB_OP_BWD, C)
        self.sel = torch.full((w.n_chunks, w.n_kv_heads, w.max_sel), -1, dtype=torch.int32, device=dev)
        self.cnt = torch.zeros((w.n_chunks, w.n_kv_heads), dtype=torch.int32, device=dev)
        self.o = torch.empty((C, w.n_q_heads, w.head_dim), dtype=w.torch_dtype, device=dev)
        self.lse = torch.empty((w.n_q_heads, C), dtype=torch.float32, device=dev)
        self.ob = [self.o]
        self.lseb = [self.lse]
        self.o_keep, self.lse_keep = {}, {}  # forward-sweep outputs, kept only for the no-recompute variant
        self.dq = [torch.empty_like(ch["q"]) for ch in self.chunks]
        self.fwd_events, self.bwd_events, self.app_events, self.sel_events = [], [], [], []
        self.recompute_events, self.prefetch_events = [], []  # reverse-sweep forwards; offload copies
        # the side stream runs at high priority: the block scheduler then places its small
        # transfer blocks beside the attention CTAs at once, instead of after the last of
        # a long attention grid's pending blocks
        self.side = torch.cuda.Stream(device=dev, priority=-1) if self.offload else None
        # the forward sweep's K/V write-backs (device -> host) run beside the gathers
        # (host -> device) on a stream of their own: the link moves both directions at once
        self.side_wb = torch.cuda.Stream(device=dev, priority=-1) if self.offload else None

    def run(self, record=False, no_recompute=False, wait_in=None, on_dq=None, on_fwd=None, wait_do=None,
            on_rev=None):
        """One step.  The reverse sweep recomputes each chunk's O and LSE (activations are
        not kept).  With no_recompute the forward sweep's outputs are kept per chunk and
        the reverse sweep only runs the backward (the variant without recomputation).
        wait_in[c]: an event the step waits for before it first reads chunk c's inputs;
        on_fwd(c): called once chunk c's append has been issued, on_dq(c): once chunk
        c's dQ has been issued, on_rev(c): when the reverse sweep reaches chunk c;
        wait_do[c]: an event the step waits for before chunk c's backward reads its dO
        (end-to-end copies)."""
        if self.offload:
            return self.run_offload(record, wait_in=wait_in, on_dq=on_dq, on_fwd=on_fwd, wait_do=wait_do,
                                    on_rev=on_rev, no_recompute=no_recompute)
        L, w, h, torch = self.L, self.w, self.pool.handle, self.torch
        L.oomb_pool_reset(h)
        for c, ch in enumerate(self.chunks):
            start, n = w.chunk_bounds(c)
            if wait_in is not None:
                torch.cuda.current_stream(self.dev).wait_event(wait_in[c])
            self._timed(record, self.app_events, c, L.oomb_kv_append, h, ch["k"], ch["v"], start)
            if on_fwd is not None:
                on_fwd(c)
            self._select(c, ch, start, n, record)
            if no_recompute:
                self._fwd_keep(c, ch, start, n)
            else:
                self._fwd(c, ch, start, n, record)
        if no_recompute:
            for c in range(w.n_chunks - 1, -1, -1):
                start, n = w.chunk_bounds(c)
                ch = self.chunks[c]
                L.oomb_chunk_attn_bwd(h, ch["q"], self.o_keep[c], ch["do"], self.lse_keep[c], start, self.sel[c],
                                      self.cnt[c], self.scale, self.dq[c], self.ws_bwd)
            return
        for c in range(w.n_chunks - 1, -1, -1):
            start, n = w.chunk_bounds(c)
            if on_rev is not None:
                on_rev(c)
            if c < w.n_chunks - 1:  # activations are not kept; the last chunk's are still in the buffers
                self._fwd(c, self.chunks[c], start, n, record, recompute=True)
            if wait_do is not None:
                torch.cuda.current_stream(self.dev).wait_event(wait_do[c])
            self._bwd(c, self.chunks[c], start, n, record)
            if on_dq is not None:
                on_dq(c)

    def run_offload(self, record=False, wait_in=None, on_dq=None, on_fwd=None, wait_do=None, on_rev=None,
                    no_recompute=False):
        """K/V pools (and, with offload_grads, the fp32 dK/dV pools) in pinned host memory.
        The side stream moves the selected blocks of the next chunk into the other
        staging buffer while the main stream runs the current chunk's attention (forward
        sweep: chunk c+1 is selected and appended before chunk c's forward, the append
        writing its pages into their staging slots only; the side stream then gathers
        chunk c+1's history pages while a second high-priority stream writes its own
        pages to the host pools; reverse sweep: chunk c-1's K/V and the gradient blocks
        it does not share with chunk c are staged during chunk c's backward; after it,
        the shared blocks are carried over from chunk c's staging and, on the write-back
        stream, chunk c's blocks are written back to the host)."""
        L, w, h, torch = self.L, self.w, self.pool.handle, self.torch
        main, side = torch.cuda.current_stream(self.dev), self.side
        S = w.n_chunks
        grads = self.offload_grads
        ev = lambda: torch.cuda.Event()  # noqa: E731
        L.oomb_pool_reset(h)

        app_ev = {}

        def append_select(c):
            """Selection (it needs the history only), then the append, which writes the
            chunk's own pages into their staging slots of buffer c % 2 only."""
            start, n = w.chunk_bounds(c)
            ch = self.chunks[c]
            if wait_in is not None:
                main.wait_event(wait_in[c])
            self._select(c, ch, start, n, record)
            self._timed(record, self.app_events, c, L.oomb_kv_append_deferred, h, ch["k"], ch["v"], start,
                        self.cnt[c], w.max_sel, c % 2)
            app_ev[c] = ev()
            app_ev[c].record(main)
            if on_fwd is not None:
                on_fwd(c)

        side_wb = self.side_wb

        def kv_writeback(c):
            """Chunk c's own pages, appended into staging buffer c % 2, to the host pools,
            on the write-back stream (every later gather waits for it)."""
            side_wb.wait_event(app_ev[c])
            start, n = w.chunk_bounds(c)
            if record:
                p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                p0.record(side_wb)
            L.oomb_kv_writeback(h, self.sel[c], self.cnt[c], c % 2, start // w.page, -(-(start + n) // w.page),
                                stream=side_wb)
            if record:
                p1.record(side_wb)
                self.prefetch_events.append((p0, p1, c))
            done = ev()
            done.record(side_wb)
            return done

        def side_timed(c, fn):
            if record:
                p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                p0.record(side)
            fn()
            if record:
                p1.record(side)
                self.prefetch_events.append((p0, p1, c))

        def prefetch(c, after, prev=None):
            """K/V of chunk c into staging buffer c % 2 -- in the forward sweep (prev False)
            the history pages only, the append having staged the own pages -- and in the
            reverse sweep its gradient blocks not shared with chunk prev; returns the
            side-stream event."""
            for e in after:
                side.wait_event(e)

            def work():
                if prev is False:
                    L.oomb_prefetch_pages(h, self.sel[c], self.cnt[c], c % 2, 0, w.chunk_bounds(c)[0] // w.page,
                                          stream=side)
                else:
                    L.oomb_prefetch(h, self.sel[c], self.cnt[c], c % 2, stream=side)
                if prev is not False and grads:
                    psel = self.sel[prev] if prev is not None else None
                    pcnt = self.cnt[prev] if prev is not None else None
                    L.oomb_grad_prefetch(h, self.sel[c], self.cnt[c], psel, pcnt, c % 2, stream=side)
            side_timed(c, work)
            done = ev()
            done.record(side)
            return done

        # forward sweep (K/V only)
        append_select(0)
        pf = {0: prefetch(0, [app_ev[0]], prev=False)}
        wb = {0: kv_writeback(0)}
        used = {}
        for c in range(S):
            if c + 1 < S:
                if c - 1 in wb:  # the append refills buffer (c + 1) % 2: chunk c-1's pages are on the host
                    main.wait_event(wb[c - 1])
                append_select(c + 1)
                # chunk c+1's history includes chunk c's pages: gathered after their write-back
                pf[c + 1] = prefetch(c + 1, [app_ev[c + 1], wb[c]] + ([used[c - 1]] if c - 1 in used else []),
                                     prev=False)
                wb[c + 1] = kv_writeback(c + 1)
            main.wait_event(pf[c])
            L.oomb_pool_set_stage(h, c % 2)
            start, n = w.chunk_bounds(c)
            if no_recompute:  # the forward sweep's outputs kept per chunk for the backward
                self._fwd_keep(c, self.chunks[c], start, n)
            else:
                self._fwd(c, self.chunks[c], start, n, record)
            used[c] = ev()
            used[c].record(main)
        # reverse sweep (its gathers read every page from the host pools); gradient
        # write-backs go on the write-back stream, beside the gathers
        # kv_ready[c]: chunk c's K/V (and the gradient blocks from the host) are staged, which
        # is all its recomputed forward needs; ready[c]: also the blocks carried from chunk
        # c+1, needed by its backward
        kv_ready = {S - 1: prefetch(S - 1, [used[S - 1], wb[S - 1]], prev=None)}
        ready = {S - 1: kv_ready[S - 1]}
        wbg = {}
        for c in range(S - 1, -1, -1):
            if c - 1 >= 0:
                # buffer (c-1) % 2 was last used by chunk c+1 (its backward and its write-back,
                # which also wrote host blocks this gather may read), or first by the forward sweep
                after = ([used[c + 1]] + ([wbg[c + 1]] if c + 1 in wbg else [])) if c + 1 < S else [used[S - 1]]
                kv_ready[c - 1] = ready[c - 1] = prefetch(c - 1, after, prev=c)
            if on_rev is not None:
                on_rev(c)
            main.wait_event(kv_ready[c])
            L.oomb_pool_set_stage(h, c % 2)
            start, n = w.chunk_bounds(c)
            if no_recompute:
                main.wait_event(ready[c])
                ch = self.chunks[c]
                L.oomb_chunk_attn_bwd(h, ch["q"], self.o_keep[c], ch["do"], self.lse_keep[c], start, self.sel[c],
                                      self.cnt[c], self.scale, self.dq[c], self.ws_bwd)
            else:
                if c < S - 1:  # the last chunk's O and LSE are still in the buffers
                    self._fwd(c, self.chunks[c], start, n, record, recompute=True)
                if wait_do is not None:
                    main.wait_event(wait_do[c])
                main.wait_event(ready[c])
                self._bwd(c, self.chunks[c], start, n, record)
            used[c] = ev()
            used[c].record(main)
            if on_dq is not None:
                on_dq(c)
            if grads:
                side.wait_event(used[c])
                if c - 1 >= 0:  # blocks of chunk c-1 also selected by chunk c: carried over
                    side_timed(c - 1, lambda: L.oomb_grad_carry(h, self.sel[c - 1], self.cnt[c - 1], self.sel[c],
                                                                self.cnt[c], (c - 1) % 2, stream=side))
                    ready[c - 1] = ev()
                    ready[c - 1].record(side)
                side_wb.wait_event(used[c])
                if record:
                    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    p0.record(side_wb)
                L.oomb_grad_writeback(h, self.sel[c], self.cnt[c], c % 2, stream=side_wb)
                if record:
                    p1.record(side_wb)
                    self.prefetch_events.append((p0, p1, c))
                wbg[c] = ev()
                wbg[c].record(side_wb)
        main.wait_stream(side)  # the last write-backs belong to the step
        main.wait_stream(side_wb)

    def _timed(self, record, events, c, fn, *args):
        if not record:
            return fn(*args)
        e0, e1 = self.torch.cuda.Event(enable_timing=True), self.torch.cuda.Event(enable_timing=True)
        e0.record()
        fn(*args)
        e1.record()
        events.append((e0, e1, c))

    def _select(self, c, ch, start, n, record):
        """Chunk c's pages: top-K retrieval, or the local window for window workloads."""
        L, w, h = self.L, self.w, self.pool.handle
        if w.window >= 0:
            self._timed(record, self.sel_events, c, L.oomb_window_select, h, start, n, w.window, w.n_sink,
                        self.sel[c], self.cnt[c])
        else:
            self._timed(record, self.sel_events, c, L.oomb_page_select, h, ch["q"], start, w.top_k, w.n_sink,
                        self.sel[c], self.cnt[c], self.ws_sel)

    def scored_chunks(self):
        """Chunks whose selection scores pages (top-K over more candidates than K)."""
        w = self.w
        if w.window >= 0 or w.top_k < 0:
            return set()
        return {c for c in range(w.n_chunks)
                if max(0, w.chunk_bounds(c)[0] // w.page - w.n_sink) > w.top_k}

    def hbm_bytes(self):
        """Algorithmic HBM bytes per call of append and select, per chunk."""
        w = self.w
        esz = 2 if w.dtype == "bf16" else 4
        app, sel = {}, {}
        for c in range(w.n_chunks):
            start, n = w.chunk_bounds(c)
            n_pages = -(-n // w.page)
            # read K,V; write K,V; zero dK,dV rows (whole pages; with the gradient pools in
            # host memory a state byte per block instead); summary rows
            zero = (n_pages * w.n_kv_heads if self.offload_grads
                    else n_pages * w.page * w.n_kv_heads * w.head_dim * 4 * 2)
            app[c] = (n * w.n_kv_heads * w.head_dim * esz * 2 * 2 + zero
                      + n_pages * w.n_kv_heads * w.head_dim * 4)
            n_hist = start // w.page
            cand = max(0, n_hist - w.n_sink)
            scored = w.top_k >= 0 and cand > w.top_k
            sel[c] = ((n * w.n_q_heads * w.head_dim * esz + cand * w.n_kv_heads * w.head_dim * 4
                       + 2 * cand * w.n_kv_heads * 4) if scored else 0) + w.n_kv_heads * w.max_sel * 4
        return app, sel

    def _bwd(self, c, ch, start, n, record, buf=0):
        L, torch, w = self.L, self.torch, self.w
        if record:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
        lse = self.lseb[buf] if n == w.chunk else self.lse_tail(n, buf)
        L.oomb_chunk_attn_bwd(self.pool.handle, ch["q"], self.ob[buf][:n], ch["do"], lse, start, self.sel[c],
                              self.cnt[c], self.scale, self.dq[c], self.ws_bwd)
        if record:
            e1.record()
            self.bwd_events.append((e0, e1, c))

    def _fwd_keep(self, c, ch, start, n):
        """Chunk c's forward into buffers kept for its backward (no-recompute variant)."""
        if c not in self.o_keep:
            self.o_keep[c] = self.torch.empty_like(ch["q"])
            self.lse_keep[c] = self.torch.empty((self.w.n_q_heads, n), dtype=self.torch.float32, device=self.dev)
        self.L.oomb_chunk_attn_fwd(self.pool.handle, ch["q"], start, self.sel[c], self.cnt[c], self.scale,
                                   self.o_keep[c], self.lse_keep[c])

    def _fwd(self, c, ch, start, n, record, recompute=False, buf=0):
        L, torch = self.L, self.torch
        if record:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
        lse = self.lseb[buf] if n == self.w.chunk else self.lse_tail(n, buf)
        L.oomb_chunk_attn_fwd(self.pool.handle, ch["q"], start, self.sel[c], self.cnt[c], self.scale,
                              self.ob[buf][:n], lse)
        if record:
            e1.record()
            self.fwd_events.append((e0, e1, c))
            if recompute:
                self.recompute_events.append((e0, e1, c))

    def lse_tail(self, n, buf=0):
        if not hasattr(self, "_lse_tail"):
            self._lse_tail = {}
        t = self._lse_tail.get(buf)
        if t is None or t.shape[1] != n:
            t = self._lse_tail[buf] = self.torch.empty((self.w.n_q_heads, n), dtype=self.torch.float32,
                                                       device=self.dev)
        return t

    def pairs_per_chunk(self):
        """Selected, causally visible (query, key) pairs summed over query heads, per chunk."""
        import numpy as np
        w = self.w
        sel, cnt = self.sel.cpu().numpy(), self.cnt.cpu().numpy()
        out = []
        for c in range(w.n_chunks):
            start, n = w.chunk_bounds(c)
            first_own = start // w.page
            tot = 0
            for hk in range(w.n_kv_heads):
                pages = sel[c, hk, : int(cnt[c, hk])].astype(np.int64)
                k0 = pages * w.page
                m = np.minimum(k0 + w.page, start + n) - k0  # keys present in the page
                hist = pages < first_own
                tot += int((m[hist] * n).sum())
                # own page: row at absolute position start+i sees keys <= start+i, i.e. the
                # m keys from k0 contribute sum_{x<m} (start + n - k0 - x)
                mo, ko = m[~hist], k0[~hist]
                tot += int((mo * (start + n - ko) - mo * (mo - 1) // 2).sum())
            out.append(tot * w.group)
        return out


class StackStep:
    """A stack of attention layers over one sequence, K/V and gradient pools in pinned host
    memory, run the way a model's forward and backward take them: chunk by chunk, the
    layers in order (reversed in the reverse sweep).  The transfers follow the
    explainer's 2.C: a local-window layer's history pages are staged one layer ahead
    (its page set does not depend on its queries); a top-K layer's history pages move
    while the layer's K/V projection runs (a synthetic GEMM of the layer's chunk, model
    width 3584, that the selection does not wait for); the append writes the chunk's
    own pages into their staging slots only, and a second high-priority stream writes
    them to the host pools; in the reverse sweep every layer's K/V and gradient blocks
    are staged two layers ahead, and the gradient write-backs go on the write-back
    stream.  One high-priority side stream carries the gathers."""

    def __init__(self, w, n_layers, dev, model_dim=3584):
        import torch

        import paged_sparse_attention_gb300 as L
        from paged_sparse_attention_gb300 import synth
        self.L, self.torch, self.w, self.dev = L, torch, w, dev
        self.side = torch.cuda.Stream(device=dev, priority=-1)
        self.side_wb = torch.cuda.Stream(device=dev, priority=-1)  # K/V write-backs (device -> host)
        self.layers = []
        for layer in range(n_layers):
            st = Step(synth.stack_layer(w, layer), dev)
            st.side = self.side
            self.layers.append(st)
        g = torch.Generator(device=dev)
        g.manual_seed(w.base_seed)
        self.X = torch.randn(w.chunk, model_dim, generator=g, device=dev).to(torch.bfloat16)
        self.Wkv = (torch.randn(model_dim, 2 * w.n_kv_heads * w.head_dim, generator=g, device=dev)
                    / math.sqrt(model_dim)).to(torch.bfloat16)
        self.kv_acc = torch.empty(w.chunk, 2 * w.n_kv_heads * w.head_dim, dtype=torch.float32, device=dev)
        self.gemm_ws = torch.empty(32 << 20, dtype=torch.uint8, device=dev)
        self.gemm_flops = 2 * w.chunk * model_dim * 2 * w.n_kv_heads * w.head_dim
        self.events = []  # (start, end) of every main-stream call, for the kernel time

    def _main(self, record, fn, *args, **kw):
        if not record:
            return fn(*args, **kw)
        e0, e1 = self.torch.cuda.Event(enable_timing=True), self.torch.cuda.Event(enable_timing=True)
        e0.record()
        fn(*args, **kw)
        e1.record()
        self.events.append((e0, e1))

    def run(self, record=False):
        L, w, torch = self.L, self.w, self.torch
        main, side, side_wb = torch.cuda.current_stream(self.dev), self.side, self.side_wb
        S, NL = w.n_chunks, len(self.layers)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        wb = {}  # (c, layer): the chunk's own pages are in the layer's host pools

        def mark():
            e = ev()
            e.record(main)
            return e

        for st in self.layers:
            L.oomb_pool_reset(st.pool.handle)
        items = [(c, layer) for c in range(S) for layer in range(NL)]
        staged = {}

        def select_and_stage(c, layer):
            """Selection of (c, layer) on the main stream, then its history pages staged."""
            st = self.layers[layer]
            start, n = w.chunk_bounds(c)
            self._main(record, st._select, c, st.chunks[c], start, n, False)
            e = mark()
            side.wait_event(e)
            if (c - 1, layer) in wb:  # the history includes the previous chunk's pages
                side.wait_event(wb[(c - 1, layer)])
            L.oomb_prefetch_pages(st.pool.handle, st.sel[c], st.cnt[c], c % 2, 0, start // w.page, stream=side)
            staged[(c, layer)] = True

        for i, (c, layer) in enumerate(items):
            st = self.layers[layer]
            h = st.pool.handle
            start, n = w.chunk_bounds(c)
            if (c, layer) not in staged:
                select_and_stage(c, layer)
            if i + 1 < len(items):  # a local layer next: its page set is known, stage it now
                c2, l2 = items[i + 1]
                if self.layers[l2].w.window >= 0 and (c2, l2) not in staged:
                    select_and_stage(c2, l2)
            # the layer's K/V projection (synthetic) overlaps the history transfer; the
            # append writes the chunk's own pages into their staging slots only, and the
            # write-back stream copies them to the host pools
            self._main(record, L.oomb_gemm, self.X[:n], self.Wkv, self.kv_acc[:n], workspace=self.gemm_ws)
            if (c - 2, layer) in wb:  # buffer c % 2 of this layer: chunk c-2's pages are on the host
                main.wait_event(wb[(c - 2, layer)])
            self._main(record, L.oomb_kv_append_deferred, h, st.chunks[c]["k"], st.chunks[c]["v"], start,
                       st.cnt[c], st.w.max_sel, c % 2)
            side_wb.wait_event(mark())
            L.oomb_kv_writeback(h, st.sel[c], st.cnt[c], c % 2, start // w.page, -(-(start + n) // w.page),
                                stream=side_wb)
            wb[(c, layer)] = ev()
            wb[(c, layer)].record(side_wb)
            done = ev()
            done.record(side)  # every history transfer issued so far, this item's included
            main.wait_event(done)
            L.oomb_pool_set_stage(h, c % 2)
            self._main(record, L.oomb_chunk_attn_fwd, h, st.chunks[c]["q"], start, st.sel[c], st.cnt[c], st.scale,
                       st.ob[0][:n], st.lseb[0] if n == w.chunk else st.lse_tail(n))
        # reverse sweep: every item's K/V and gradient blocks staged ahead of it
        ritems = items[::-1]
        bwd_done, ready, wbg = {}, {}, {}

        def stage_rev(c, layer):
            st = self.layers[layer]
            h = st.pool.handle
            prev = c + 1 if c + 1 < S else None
            if prev is not None:  # the carried blocks, and the host blocks written back after it
                side.wait_event(bwd_done[(prev, layer)])
                if (prev, layer) in wbg:
                    side.wait_event(wbg[(prev, layer)])
            L.oomb_prefetch(h, st.sel[c], st.cnt[c], c % 2, stream=side)
            L.oomb_grad_prefetch(h, st.sel[c], st.cnt[c], st.sel[prev] if prev is not None else None,
                                 st.cnt[prev] if prev is not None else None, c % 2, stream=side)
            if prev is not None:
                L.oomb_grad_carry(h, st.sel[c], st.cnt[c], st.sel[prev], st.cnt[prev], c % 2, stream=side)
            r = ev()
            r.record(side)
            ready[(c, layer)] = r

        side.wait_stream(main)  # the forward sweep's last reads of the staging buffers
        side.wait_stream(side_wb)  # and its write-backs: the reverse sweep gathers every page from the host
        # items are staged `ahead` items early: the previous chunk of the staged item's layer
        # (NL items after it in the reverse order) must have run its backward by then
        ahead = max(1, min(2, NL - 1))
        for j in range(min(ahead, len(ritems))):
            stage_rev(*ritems[j])
        for i, (c, layer) in enumerate(ritems):
            st = self.layers[layer]
            h = st.pool.handle
            start, n = w.chunk_bounds(c)
            if i + ahead < len(ritems):
                c2, l2 = ritems[i + ahead]
                if c2 + 1 < S and (c2 + 1, l2) not in bwd_done:
                    raise RuntimeError("stack order: the previous chunk of a layer must have run its backward")
                stage_rev(c2, l2)
            main.wait_event(ready[(c, layer)])
            L.oomb_pool_set_stage(h, c % 2)
            lse = st.lseb[0] if n == w.chunk else st.lse_tail(n)
            if c < S - 1:  # recomputed; the last chunk's O and LSE are still in the layer's buffers
                self._main(record, L.oomb_chunk_attn_fwd, h, st.chunks[c]["q"], start, st.sel[c], st.cnt[c],
                           st.scale, st.ob[0][:n], lse)
            self._main(record, L.oomb_chunk_attn_bwd, h, st.chunks[c]["q"], st.ob[0][:n], st.chunks[c]["do"], lse,
                       start, st.sel[c], st.cnt[c], st.scale, st.dq[c], st.ws_bwd)
            bwd_done[(c, layer)] = mark()
            side_wb.wait_event(bwd_done[(c, layer)])
            L.oomb_grad_writeback(h, st.sel[c], st.cnt[c], c % 2, stream=side_wb)
            wbg[(c, layer)] = ev()
            wbg[(c, layer)].record(side_wb)
        main.wait_stream(side)
        main.wait_stream(side_wb)

    def pairs(self):
        return [sum(st.pairs_per_chunk()) for st in self.layers]


def run_stack(args, w, world, dev):
    """--workload stack...: the multi-layer offload step; one JSON line."""
    import torch

    import paged_sparse_attention_gb300 as L
    from paged_sparse_attention_gb300 import synth
    n_layers = synth.STACK_LAYERS[w.name]
    log(f"stack of {n_layers} layers ({w.name}): building inputs and pools")
    stack = StackStep(w, n_layers, dev)
    for i in range(max(3, args.warmup)):
        stack.run()
        torch.cuda.synchronize()
        log(f"warm-up step {i} done")
    for st in stack.layers:
        L.oomb_check(st.pool.handle)
    pairs = stack.pairs()
    credited = sum(pairs) * 14 * w.head_dim
    stack.events = []
    launches0 = L.oomb_launch_count()
    with ClockSampler(0 if not torch.cuda.is_available() else torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with gc_paused():
            e0.record()
            for _ in range(args.steps):
                stack.run(record=True)
            e1.record()
            torch.cuda.synchronize()
    launches = L.oomb_launch_count() - launches0
    ms = reduce_max_ms(e0.elapsed_time(e1) / args.steps, world, dev)
    for st in stack.layers:
        L.oomb_check(st.pool.handle)
    kern_ms = sum(a.elapsed_time(b) for a, b in stack.events) / args.steps
    exposed = max(0.0, ms - kern_ms)
    gemm_ms_total = None
    line = {"metric": METRIC, "value": round(job_throughput(credited, ms, world) / 1e12, 3), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) Q/K/V/dO per layer, RoPE theta 1e6; no trained weights)",
            "config": dict(config_of(w, world), layers=n_layers,
                           layer_kinds=["top-%d" % w.top_k if i % 2 == 0 else "window-%d" % w.window
                                        for i in range(n_layers)],
                           kv_projection="synthetic GEMM per layer and chunk: [%d x 3584] x [3584 x %d] bf16"
                                         % (w.chunk, 2 * w.n_kv_heads * w.head_dim)),
            "tokens_per_s_per_layer": round(job_throughput(w.seq * n_layers, ms, world), 1),
            "credited_tflop_per_step": credited / 1e12,
            "main_stream_ms_per_step": round(kern_ms, 3),
            "exposed_ms_per_step": round(exposed, 3),
            "exposed_ms_per_layer": round(exposed / n_layers, 3),
            "exposed_frac_of_step": round(exposed / ms, 4),
            "gpu_launches": int(launches),
            "clocks": clk.summary()}
    del gemm_ms_total
    print(json.dumps(line), flush=True)


def state_bytes_per_10k(w) -> dict:
    """Device bytes of one layer's attention state that grow with the context, per
    10,000 tokens: K/V pools, fp32 dK/dV pools and the page summaries (the analogue,
    for this path alone, of the pages' end-to-end memory growth per 10K tokens).
    With offload the K/V pools (and with offload_grads the gradient pools) live in
    host memory and only fixed staging buffers are on the device."""
    esz = 2 if w.dtype == "bf16" else 4
    per_tok_kv = 2 * w.n_kv_heads * w.head_dim * esz
    per_tok_grad = 2 * w.n_kv_heads * w.head_dim * 4
    per_tok_sum = w.n_kv_heads * w.head_dim * 4 / w.page
    host = (per_tok_kv if w.offload else 0) + (per_tok_grad if w.offload and w.offload_grads else 0)
    dev = per_tok_kv + per_tok_grad + per_tok_sum - host
    stage = 0
    if w.offload:  # two staging buffers of max_sel blocks per KV head: K/V, and fp32 dK/dV
        blk = w.page * w.head_dim
        stage = 2 * w.n_kv_heads * w.max_sel * blk * (2 * esz + (2 * 4 if w.offload_grads else 0))
    return {"device": int(dev * 10000), "host": int(host * 10000), "fixed_staging_device": int(stage)}


def config_of(w, world: int) -> dict:
    """The `config` of the JSON line, the same for both arms."""
    tc = w.dtype == "bf16" and w.head_dim == 128 and w.page == 128
    return {"workload": w.name, "seq": w.seq, "chunk": w.chunk, "page": w.page, "top_k": w.top_k,
            **({"window_pages": w.window, "n_sink": w.n_sink} if w.window >= 0 else {}),
            "heads": f"{w.n_q_heads}/{w.n_kv_heads}", "head_dim": w.head_dim,
            "offload": ("kv+grads" if w.offload_grads else "kv") if w.offload else "none",
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "inputs larger than L2 (Q+dO of one chunk alone exceed 58 MB; all chunks resident)",
            "attention_kernels": "tcgen05" if tc else "simt"}


def host_link_bytes(w, sel, cnt, offload_grads: bool) -> dict:
    """Bytes the offload step moves over the host link per step, from the selections
    sel [S, Hkv, max_sel] and counts cnt [S, Hkv] (host arrays).  Forward sweep: each
    chunk's history blocks are gathered (its own pages are appended into their staging
    slots) and its own pages are written to the host pools; reverse sweep: every
    selected K/V block is gathered.  Gradients (offload_grads): every selected block
    is written back after its chunk's backward; a block of chunk c also selected by
    chunk c+1 is carried over on the device; any other is read from the host only if
    a chunk after c has written it back in this sweep (otherwise it is zero-filled on
    the device: the append marked it empty)."""
    S, Hkv = w.n_chunks, w.n_kv_heads
    esz = 2 if w.dtype == "bf16" else 4
    kv_blk = 2 * w.page * w.head_dim * esz   # K and V of one (page, KV head)
    g_blk = 2 * w.page * w.head_dim * 4      # dK and dV
    sets = [[set(int(x) for x in sel[c, hk, : int(cnt[c, hk])]) for hk in range(Hkv)] for c in range(S)]
    kv_in = kv_out = g_in = g_out = carried = 0
    for c in range(S):
        first_own = w.chunk_bounds(c)[0] // w.page
        for hk in range(Hkv):
            hist = sum(1 for p in sets[c][hk] if p < first_own)
            own = len(sets[c][hk]) - hist
            kv_in += (hist + len(sets[c][hk])) * kv_blk
            kv_out += own * kv_blk
    if offload_grads:
        for hk in range(Hkv):
            written = set()
            for c in range(S - 1, -1, -1):
                nxt = sets[c + 1][hk] if c + 1 < S else set()
                for p in sets[c][hk]:
                    if p in nxt:
                        carried += g_blk
                    elif p in written:
                        g_in += g_blk
                g_out += len(sets[c][hk]) * g_blk
                written |= sets[c][hk]
    return {"kv_in": kv_in, "kv_out": kv_out, "grad_in": g_in, "grad_out": g_out,
            "grad_carried_on_device": carried}


class gc_paused:
    """Python's cyclic garbage collector held off inside a timed region (reference
    counting still frees everything the steps drop): the host thread that issues a
    step's thousands of calls and events would otherwise stop for a full collection
    now and then, which shows as a stray slow step when the GPU waits on the host."""

    def __enter__(self):
        gc.collect()
        self.was = gc.isenabled()
        gc.disable()
        return self

    def __exit__(self, *exc):
        if self.was:
            gc.enable()
        return False


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` from an ncu capture recorded in
    profiles/traffic.txt, or None when there is none for this workload or the
    kernel's source has changed since (its sha256 prefix no longer matches)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split()
        if len(f) < 5 or line.startswith("#") or f[0] != workload or f[1] != kernel:
            continue
        src = os.path.join(ROOT, f[2])
        if not os.path.exists(src):
            return None
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
        return int(f[4]) if digest.startswith(f[3]) else None
    return None


def same_size_gbs(nbytes: int, dev, kind: str) -> float:
    """Bandwidth of a plain PyTorch kernel moving the same bytes from cold L2: a sum
    over nbytes (kind "read") or a copy of nbytes / 2 (kind "copy", nbytes moved in
    total).  Small transfers do not reach the large-copy peak; this is the
    size-matched reference for the append and selection calls."""
    import torch
    n = max(16, int(nbytes if kind == "read" else nbytes // 2)) // 4
    src = torch.ones(n, dtype=torch.float32, device=dev)
    dst = torch.empty_like(src) if kind == "copy" else None
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    times = []
    for i in range(7):
        flush.fill_(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        if kind == "read":
            src.sum()
        else:
            dst.copy_(src)
        e1.record()
        torch.cuda.synchronize()
        if i:
            times.append(e0.elapsed_time(e1))
    times.sort()
    return (n * 4 * (1 if kind == "read" else 2)) / (times[len(times) // 2] * 1e-3) / 1e9


def measure_graph(step, steps: int, world: int, dev) -> dict:
    """The same step captured once in a CUDA graph and replayed: every library call
    of the step (pool reset, append, selection, forward, recompute, backward) is a
    node, so the host issues one launch per step.  Returns its step time, or why
    the capture failed."""
    import torch

    import paged_sparse_attention_gb300 as L
    try:
        g = torch.cuda.CUDAGraph()
        n0 = L.oomb_launch_count()
        with torch.cuda.graph(g):
            step.run()
        per_step = L.oomb_launch_count() - n0
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = reduce_max_ms(e0.elapsed_time(e1) / steps, world, dev)
        L.oomb_check(step.pool.handle)
        return {"ms_per_step": round(ms, 3), "kernel_launches_per_step": per_step,
                "note": "one CUDA graph per step, replayed; same work as the eager step"}
    except Exception as e:  # report, do not hide: the eager numbers above stand on their own
        return {"unavailable": f"{type(e).__name__}: {str(e).splitlines()[0][:200]}"}


def reduce_max_ms(ms: float, world: int, device) -> float:
    """Step time of the whole job: the maximum over ranks (replicas run independently)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job throughput: every rank processes the same units (weak scaling) and the
    job takes as long as its slowest rank."""
    return units_per_rank * world / (ms_max * 1e-3)


def oracle_sample_seconds(w, budget_s=20.0):
    """Time the fp64 CPU oracle on a bounded sample: the forward+backward of chunk 1
    (or 0) for the query heads of KV group 0, repeated until ``budget_s``."""
    import numpy as np
    import torch

    import oracle.oomb_oracle as O
    from paged_sparse_attention_gb300 import synth

    c = 1 if w.n_chunks > 1 else 0
    plants = synth.PlantTable(w) if w.plants > 0 else None
    chunks = [synth.make_chunk(w, i, plants=plants) for i in range(c + 1)]
    G = w.group
    pool = O.OraclePool(1, w.head_dim, w.page, w.num_phys, w.n_pages)
    order = synth.page_order(w).tolist()
    used = 0
    for i, ch in enumerate(chunks):
        start, n = w.chunk_bounds(i)
        npg = -(-n // w.page)
        pool.append(ch["k"][:, :1].double().numpy(), ch["v"][:, :1].double().numpy(), start, order[used:used + npg])
        used += npg
    start, n = w.chunk_bounds(c)
    q = chunks[c]["q"][:, :G].double().numpy()
    do = chunks[c]["do"][:, :G].double().numpy()
    if w.window >= 0:
        sel = [O.window_pages(start, n, w.page, w.window, w.n_sink)]
    else:
        sel = O.select_pages(pool, q, start, w.top_k, w.n_sink)
    scale = 1.0 / math.sqrt(w.head_dim)
    # credited pairs of the sample
    kpos = np.concatenate([p * w.page + np.arange(pool.tokens_in_page(p)) for p in sel[0]])
    pairs = int(sum(int((kpos <= start + i).sum()) for i in range(n))) * G
    flops = pairs * 14 * w.head_dim
    t0 = time.perf_counter()
    reps = 0
    while True:
        o, lse = O.chunk_attn_fwd(pool, q, start, sel, scale)
        O.chunk_attn_bwd(pool, q, o, do, lse, start, sel, scale)
        reps += 1
        el = time.perf_counter() - t0
        if el > budget_s or reps >= 50:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = (f"chunk {c} ({n} queries) fwd+bwd for the {G} query heads of KV group 0, "
              f"{reps} repetition(s), fp64 numpy")
    return {"seconds": el / reps, "flops": flops, "cores": cores, "sample": sample, "tokens": n / w.n_kv_heads}


def run_reference(args, w, rank, world):
    """The CPU oracle as it stands, on host cores, on a bounded sample per step."""
    if rank != 0:
        return
    res = []
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle_sample_seconds(w, budget_s=1.0)
    for _ in range(args.steps):
        res.append(oracle_sample_seconds(w, budget_s=max(2.0, 20.0 / max(1, args.steps))))
    sec = statistics.mean(r["seconds"] for r in res)
    tflops = res[0]["flops"] / sec / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": tflops, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, world),
            "cpu_baseline": {"value": tflops, "unit": UNIT, "cores": res[0]["cores"], "kind": "oracle",
                             "sample": res[0]["sample"]},
            "e2e": {"value": tflops, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="oomb", choices=["oomb", "reference"])
    ap.add_argument("--workload", default="offload4m")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from paged_sparse_attention_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    import paged_sparse_attention_gb300 as L

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    def barrier():
        if world > 1:
            dist.barrier()

    if w.name in synth.STACK_LAYERS:
        run_stack(args, w, world, dev)
        if world > 1:
            dist.destroy_process_group()
        return
    log(f"workload {w.name}: building inputs and pool")
    step = Step(w, dev)
    torch.cuda.synchronize()
    log("warm-up")
    for i in range(max(3, args.warmup)):
        step.run()
        torch.cuda.synchronize()
        log(f"warm-up step {i} done")
    L.oomb_check(step.pool.handle)
    pairs = step.pairs_per_chunk()
    log("credited pairs counted; timed steps")
    credited = sum(pairs) * 14 * w.head_dim
    fwd_flops = {c: p * 4 * w.head_dim for c, p in enumerate(pairs)}
    bwd_flops = {c: p * 10 * w.head_dim for c, p in enumerate(pairs)}

    # ---- timed region (device-resident inputs; the step's inputs exceed L2) ----
    launches0 = L.oomb_launch_count()
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("oomb_timed_steps")  # the profiler's launch list filters on it
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with gc_paused():
            e0.record()
            for _ in range(args.steps):
                step.run(record=True)
            e1.record()
            torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        barrier()
    launches = L.oomb_launch_count() - launches0
    ms = reduce_max_ms(e0.elapsed_time(e1) / args.steps, world, dev)
    L.oomb_check(step.pool.handle)
    # end to end right after the device-resident steps, before the other variants
    e2e = None
    if not args.no_e2e:
        with ClockSampler(local) as clk_e2e:
            e2e = measure_e2e(step, args.steps, credited, world, dev)
        e2e["clocks"] = clk_e2e.summary()

    # per-kernel-call roofline: the backward (dominant) and forward calls
    bwd_ms = [a.elapsed_time(b) for a, b, _ in step.bwd_events]
    bwd_fl = [bwd_flops[c] for _, _, c in step.bwd_events]
    fwd_ms = [a.elapsed_time(b) for a, b, _ in step.fwd_events]
    fwd_fl = [fwd_flops[c] for _, _, c in step.fwd_events]
    peaks = load_peaks()
    bwd_tflops = sum(bwd_fl) / (sum(bwd_ms) * 1e-3) / 1e12
    fwd_tflops = sum(fwd_fl) / (sum(fwd_ms) * 1e-3) / 1e12
    # per-call event timings of one kernel: the burst GEMM peak; the whole seconds-long
    # step is also given against the sustained one
    peak = peaks.get("bf16_tflops", 1900.0)
    peak_sustained = peaks.get("bf16_tflops_sustained", peak)
    app_b, sel_b = step.hbm_bytes()
    def gbs(events, nbytes):
        if not events:
            return None
        t = sum(a.elapsed_time(b) for a, b, _ in events) * 1e-3
        return sum(nbytes[c] for _, _, c in events) / t / 1e9 if t > 0 else None
    app_gbs = gbs(step.app_events, app_b)
    # selection bandwidth over the calls that score pages (dense selections keep every
    # page and the window selection reads nothing: their calls only write the set)
    scored = step.scored_chunks()
    sel_gbs = gbs([e for e in step.sel_events if e[2] in scored], sel_b) if scored else None
    # size-matched references (largest call of each kind)
    app_ref = same_size_gbs(max(app_b.values()), dev, "copy") if app_gbs else None
    sel_ref = same_size_gbs(max(sel_b.values()), dev, "read") if sel_gbs else None
    hbm_peak = peaks.get("hbm_gbs", 6783.0)
    value = job_throughput(credited, ms, world) / 1e12
    tokens_per_s = job_throughput(w.seq, ms, world)
    rec_ms = sum(a.elapsed_time(b) for a, b, _ in step.recompute_events) / args.steps
    nr_ms = None
    # the variant without recompute, timed directly (forward outputs kept per chunk)
    step.run(no_recompute=True)
    torch.cuda.synchronize()
    n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with gc_paused():
        n0.record()
        for _ in range(args.steps):
            step.run(no_recompute=True)
        n1.record()
        torch.cuda.synchronize()
    nr_ms = reduce_max_ms(n0.elapsed_time(n1) / args.steps, world, dev)
    step.o_keep.clear()  # the kept outputs (30 GB at 4M tokens) are not needed again
    step.lse_keep.clear()
    graph = None if step.offload or args.no_graph else measure_graph(step, args.steps, world, dev)
    kern_ms = sum(a.elapsed_time(b) for ev in (step.fwd_events, step.bwd_events, step.app_events, step.sel_events)
                  for a, b, _ in ev) / args.steps
    prefetch = None
    if step.offload:
        S = w.n_chunks
        hb = host_link_bytes(w, step.sel.cpu().numpy(), step.cnt.cpu().numpy(), step.offload_grads)
        n_blk = [int(step.cnt[c].sum()) for c in range(S)]
        kv_blk = 2 * w.page * w.head_dim * (2 if w.dtype == "bf16" else 4)
        link_b = hb["kv_in"] + hb["kv_out"] + hb["grad_in"] + hb["grad_out"]
        pf_s = sum(a.elapsed_time(b) for a, b, _ in step.prefetch_events) * 1e-3 / args.steps
        # isolated: each of the last chunks' K/V gathers three times in a row (the first
        # gather of a page set after the step can take far longer than the repeats,
        # so it is reported on its own; the repeats give the gather's bandwidth), and
        # a plain pinned-host -> HBM copy for the link's bandwidth
        iso, first_ms = [], []
        for c in range(max(0, S - 3), S):
            for rep in range(3):
                torch.cuda.synchronize()
                g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                g0.record()
                L.oomb_prefetch(step.pool.handle, step.sel[c], step.cnt[c], rep % 2)
                g1.record()
                torch.cuda.synchronize()
                t = g0.elapsed_time(g1)
                if rep == 0:
                    first_ms.append(round(t, 3))
                else:
                    iso.append(n_blk[c] * kv_blk / (t * 1e-3) / 1e9)
        hbuf = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        dbuf.copy_(hbuf)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        for _ in range(4):
            dbuf.copy_(hbuf, non_blocking=True)
        c1.record()
        torch.cuda.synchronize()
        link = 4 * (256 << 20) / (c0.elapsed_time(c1) * 1e-3) / 1e9
        del hbuf, dbuf
        prefetch = {"link": "pinned host memory <-> HBM staging over NVLink-C2C (side stream, zero-copy kernels)",
                    "host_bytes_per_step": hb,
                    "gbs_overlapped": round(link_b / pf_s / 1e9, 1) if pf_s > 0 else None,
                    "gbs_isolated_kv_gather": round(statistics.median(iso), 1),
                    "isolated_first_call_ms": first_ms,
                    "host_link_copy_gbs": round(link, 1),
                    "side_stream_ms_per_step": round(pf_s * 1e3, 3),
                    "main_stream_kernel_ms_per_step": round(kern_ms, 3),
                    "exposed_ms_per_step": round(max(0.0, ms - kern_ms), 3),
                    "exposed_frac_of_step": round(max(0.0, ms - kern_ms) / ms, 4)}

    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "fp32",
            "data": "synthetic (seeded N(0,1) Q/K/V/dO, RoPE theta 1e6; no trained weights)",
            "config": config_of(w, world),
            "tokens_per_s_per_layer": round(tokens_per_s, 1),
            "tokens_per_s_per_layer_no_recompute": round(job_throughput(w.seq, nr_ms, world), 1) if nr_ms else None,
            "ms_per_step_no_recompute": round(nr_ms, 3) if nr_ms else None,
            "recompute_call_ms_per_step": round(rec_ms, 3),
            "credited_tflop_per_step": credited / 1e12,
            "value_frac_of_peak": round(value / peak, 4),
            "value_frac_of_sustained_peak": round(value / peak_sustained, 4),
            "state_bytes_per_10k_tokens": state_bytes_per_10k(w),
            "fwd_call_tflops": round(fwd_tflops, 2), "bwd_call_tflops": round(bwd_tflops, 2),
            "fwd_bwd_call_tflops": round((sum(fwd_fl) + sum(bwd_fl)) / ((sum(fwd_ms) + sum(bwd_ms)) * 1e-3) / 1e12, 2),
            "roofline": {"bound": "tensor", "kernel": "oomb_chunk_attn_bwd", "achieved": round(bwd_tflops, 2),
                         "peak": peak, "unit": "TFLOP/s", "frac": round(bwd_tflops / peak, 4),
                         "frac_of_sustained": round(bwd_tflops / peak_sustained, 4),
                         "fwd_frac": round(fwd_tflops / peak, 4),
                         "fwd_bwd_frac": round((sum(fwd_fl) + sum(bwd_fl)) / ((sum(fwd_ms) + sum(bwd_ms)) * 1e-3)
                                               / 1e12 / peak, 4),
                         "peak_source": peaks.get("source", "") + " (bf16 dense, burst; per-call event timings)",
                         "traffic": recorded_traffic(w.name, "oomb_chunk_attn_bwd"),
                         "traffic_unit": "DRAM bytes per launch (ncu dram__bytes_read.sum + write.sum)"},
            "append_call": {"gbs": round(app_gbs, 1) if app_gbs else None,
                            "frac_of_hbm": round(app_gbs / hbm_peak, 3) if app_gbs else None,
                            "bound": "hbm" + (" (offload: the pages go to their staging slots; the side stream "
                                              "writes them to the host pools)" if step.offload else ""),
                            "same_size_copy_gbs": round(app_ref, 1) if app_ref else None,
                            "frac_of_same_size_copy": round(app_gbs / app_ref, 3) if app_ref else None,
                            "bytes_per_token_per_kv_head": 2 * 2 * w.head_dim * (2 if w.dtype == "bf16" else 4)
                            + 2 * w.head_dim * 4},
            "select_call": {"scored_calls_per_step": len(scored),
                            "gbs": round(sel_gbs, 1) if sel_gbs else None,
                            "frac_of_hbm": round(sel_gbs / hbm_peak, 3) if sel_gbs else None,
                            "same_size_read_gbs": round(sel_ref, 1) if sel_ref else None,
                            "frac_of_same_size_read": round(sel_gbs / sel_ref, 3) if sel_ref else None},
            "prefetch_call": prefetch,
            "graph": (dict(graph, value=round(job_throughput(credited, graph["ms_per_step"], world) / 1e12, 3))
                      if graph and "ms_per_step" in graph else graph),
            "gpu_launches": int(launches),
            "clocks": clk.summary()}

    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        cb = oracle_sample_seconds(w, budget_s=15.0)
        line["cpu_baseline"] = {"value": cb["flops"] / cb["seconds"] / 1e12, "unit": UNIT, "cores": cb["cores"],
                                "kind": "oracle", "sample": cb["sample"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


class HostBuffer:
    """Page-locked host memory for the end-to-end copies: blocks of exactly 1 GiB from
    the pinned allocator (cudaHostAlloc; it rounds a request up to a power of two, so
    such blocks waste nothing), the tensors packed into them, and a block of its own for
    a tensor above 1 GiB.  Memory the driver allocates page-locked kept the copy rate
    better than pageable memory registered with cudaHostRegister (1M tokens, fresh
    machine: +0.2 % against +4.9 % end to end)."""

    BLOCK = 1 << 30

    def __init__(self):
        self.blocks, self.cur, self.off = [], None, 0

    def take(self, shape, dtype):
        import torch
        n = int(math.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        if n > self.BLOCK:
            t = torch.empty(shape, dtype=dtype, pin_memory=True)
            self.blocks.append(t)
            return t
        self.off = (self.off + 255) // 256 * 256
        if self.cur is None or self.off + n > self.BLOCK:
            self.cur = torch.empty(self.BLOCK, dtype=torch.uint8, pin_memory=True)
            self.blocks.append(self.cur)
            self.off = 0
        t = self.cur[self.off:self.off + n].view(dtype).view(shape)
        self.off += n
        return t

    def close(self):
        import torch
        torch.cuda.synchronize()
        self.blocks, self.cur = [], None


E2E_AHEAD = 3  # chunks whose inputs are uploaded ahead of the forward sweep


def measure_e2e(step, steps, credited, world, dev):
    """Same step with host-resident inputs: every step copies Q, K, V, dO of all
    chunks from page-locked host memory to the device and reads dQ (and, when the
    gradient pools are in HBM, dK/dV) back, all inside the timed region.  The uploads
    run on a copy stream, chunk by chunk, and each chunk waits only for its own
    inputs; each dQ is read back on the copy stream as soon as its backward is issued,
    and so are the chunk's dK/dV rows (token-major, gathered through the page table:
    a chunk's own pages receive nothing from the chunks the reverse sweep has left).
    With offloaded gradient pools the step's own write-backs put dK/dV in host memory;
    those bytes are counted as read back."""
    import torch
    sizes = [t.numel() * t.element_size() for ch in step.chunks for t in ch.values()]
    dq_sizes = [d.numel() * d.element_size() for d in step.dq]
    hb = HostBuffer()
    host_in = [{k: hb.take(v.shape, v.dtype) for k, v in ch.items()} for ch in step.chunks]
    for ch, hc in zip(step.chunks, host_in):
        for k in ch:
            hc[k].copy_(ch[k])
    host_dq = [hb.take(d.shape, d.dtype) for d in step.dq]
    pools_on_device = not step.offload_grads
    host_dk = host_dv = None
    w = step.w
    if pools_on_device:  # token-major dK, dV of the whole sequence; two device gather buffers
        hp = HostBuffer()
        host_dk = hp.take((w.seq, w.n_kv_heads, w.head_dim), torch.float32)
        host_dv = hp.take((w.seq, w.n_kv_heads, w.head_dim), torch.float32)
        gk = [torch.empty((w.chunk, w.n_kv_heads, w.head_dim), dtype=torch.float32, device=dev) for _ in range(2)]
        gv = [torch.empty_like(gk[0]) for _ in range(2)]
    torch.cuda.synchronize()
    bi = sum(sizes)
    bo = sum(dq_sizes) + (2 * host_dk.numel() * 4 if pools_on_device else 0)
    if not pools_on_device:  # the reverse sweep's gradient write-backs (each selected block, dK and dV)
        w = step.w
        cnt_h = step.cnt.cpu()
        bo += int(cnt_h.sum()) * 2 * w.page * w.head_dim * 4
    main = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(device=dev)
    S = len(step.chunks)

    fwd_keys = [k for k in step.chunks[0] if k != "do"]

    def one_step():
        copy.wait_stream(main)  # the previous step has finished reading the input buffers
        ready, ready_do = {}, {}

        def upload(c, keys, done):
            with torch.cuda.stream(copy):
                for k in keys:
                    step.chunks[c][k].copy_(host_in[c][k], non_blocking=True)
                done[c] = torch.cuda.Event()
                done[c].record(copy)

        def after_main():
            e = torch.cuda.Event()
            e.record(main)
            copy.wait_event(e)

        # paced, each input when it is needed: Q, K, V of chunk c + AHEAD once chunk c's
        # append has been issued (the uploads spread over the forward sweep instead of
        # taking the host link in one burst; the offload gathers share it), and dO, which
        # only the backward reads, AHEAD chunks ahead in the reverse sweep
        for c in range(min(E2E_AHEAD, S)):
            upload(c, fwd_keys, ready)

        def on_fwd(c):
            if c + E2E_AHEAD < S:
                after_main()
                upload(c + E2E_AHEAD, fwd_keys, ready)

        def on_rev(c):
            if c == S - 1:
                for c2 in range(S - 1, max(-1, S - 1 - E2E_AHEAD), -1):
                    upload(c2, ["do"], ready_do)
            elif c - E2E_AHEAD + 1 >= 0:
                after_main()
                upload(c - E2E_AHEAD + 1, ["do"], ready_do)

        read = {}

        def on_dq(c):
            if pools_on_device:  # chunk c's dK/dV rows are final: gather them for the copy
                b = c % 2
                if b in read:  # the copy of chunk c + 2 out of this buffer has finished
                    main.wait_event(read[b])
                start, n = w.chunk_bounds(c)
                step.L.oomb_grad_gather(step.pool.handle, start, gk[b][:n], gv[b][:n])
            done = torch.cuda.Event()
            done.record(main)
            copy.wait_event(done)
            with torch.cuda.stream(copy):
                host_dq[c].copy_(step.dq[c], non_blocking=True)
                if pools_on_device:
                    host_dk[start:start + n].copy_(gk[b][:n], non_blocking=True)
                    host_dv[start:start + n].copy_(gv[b][:n], non_blocking=True)
                    read[b] = torch.cuda.Event()
                    read[b].record(copy)

        step.run(wait_in=ready, on_dq=on_dq, on_fwd=on_fwd, wait_do=ready_do, on_rev=on_rev)
        main.wait_stream(copy)

    one_step()  # warm-up of the copy path
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with gc_paused():
        ev[0].record()
        for i in range(steps):
            one_step()
            ev[i + 1].record()
        torch.cuda.synchronize()
    per_step = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    ms = ev[0].elapsed_time(ev[steps]) / steps
    hb.close()
    if pools_on_device:
        hp.close()
    return {"value": round(credited / (ms * 1e-3) / 1e12 * world, 3), "unit": UNIT, "ms_per_step": round(ms, 3),
            "ms_per_step_min_max": [round(min(per_step), 3), round(max(per_step), 3)],
            "ms_each_step": [round(x, 2) for x in per_step],
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "overlap": f"uploads per chunk on a copy stream: Q, K, V {E2E_AHEAD} chunks ahead of the forward "
                       f"sweep, dO {E2E_AHEAD} chunks ahead of the reverse sweep; dQ (and dK/dV rows when the "
                       "pools are in HBM) read back as each backward is issued"}


if __name__ == "__main__":
    main()
