"""Seeded synthetic inputs for paged sparse chunk attention.

This module only draws inputs: random Q/K/V/dO per chunk, the rotary position
embedding applied to Q and K (part of the input distribution, not of the
attention method), the planted high-similarity pages of the sparse workloads,
and the shuffled order in which physical pages are handed out.  It holds none of
the attention, selection or gradient arithmetic, so both the CUDA path and the
CPU oracle can be fed from it without sharing any of the method.

Workload geometry follows Qwen2.5-7B's attention (28 query heads, 4 KV heads,
head_dim 128), the model the OOMB experiments use ("Out of the Memory Barrier",
gist.science explainer, section 4 "Experimental Results").  The pages train on
real text with trained weights; these seeded N(0,1) tensors stand in for them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

_T_PERM, _T_Q, _T_K, _T_V, _T_DO, _T_PLANT = range(6)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str            # "fp32" or "bf16"
    seq: int              # total tokens N
    chunk: int            # chunk length C (last chunk may be shorter)
    page: int             # page size P in tokens
    top_k: int            # retrieved history pages per KV head; <0 keeps all
    n_sink: int = 1       # leading pages always kept
    rope: bool = False
    rope_theta: float = 1e6
    plants: int = 0       # planted pages per (chunk, KV head)
    plant_alpha: float = 0.5
    plant_beta: float = 1.0
    base_seed: int = 1000
    offload: bool = False
    offload_grads: bool = False  # with offload: the fp32 dK/dV pools live in pinned host memory too
    window: int = -1      # >= 0: local sliding-window selection of this many history pages (no top-K)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def n_chunks(self) -> int:
        return -(-self.seq // self.chunk)

    @property
    def n_pages(self) -> int:
        return -(-self.seq // self.page)

    @property
    def num_phys(self) -> int:
        return self.n_pages

    @property
    def max_sel(self) -> int:
        own = -(-self.chunk // self.page)
        if self.window >= 0:
            return min(self.n_pages, self.n_sink + self.window + own)
        if self.top_k < 0:
            return self.n_pages
        return self.n_sink + self.top_k + own

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def chunk_bounds(self, c: int):
        start = c * self.chunk
        return start, min(self.chunk, self.seq - start)


WORKLOADS: Dict[str, Workload] = {
    # 1 layer, 2 query heads / 1 KV head, d 64, fp32, 4 chunks of 1024, page 64, dense.
    "tiny": Workload("tiny", 2, 1, 64, "fp32", 4096, 1024, 64, -1, base_seed=1000),
    # Qwen2.5-7B attention geometry, dense, 32K tokens in chunks of 4096, page 128.
    "dense32k": Workload("dense32k", 28, 4, 128, "bf16", 32768, 4096, 128, -1,
                         rope=True, base_seed=1001),
    # 128K tokens, top-64 pages + sink + own pages, 8 planted pages per chunk/head.
    "sparse128k": Workload("sparse128k", 28, 4, 128, "bf16", 131072, 4096, 128, 64,
                           rope=True, plants=8, base_seed=1002),
    # 1M tokens in chunks of 8192, top-128 pages.
    "sparse1m": Workload("sparse1m", 28, 4, 128, "bf16", 1048576, 8192, 128, 128,
                         rope=True, plants=8, base_seed=1003),
    # 4M tokens, KV pages and their fp32 gradient pages in pinned host memory; the
    # selected blocks are staged in HBM on a side stream.
    "offload4m": Workload("offload4m", 28, 4, 128, "bf16", 4194304, 8192, 128, 128,
                          rope=True, plants=8, base_seed=1004, offload=True, offload_grads=True),
    # 128K tokens with local sliding-window attention (the sparse layers of a
    # sparse-native model): the 32 pages (4K tokens) before each 4K chunk plus the
    # chunk's own pages, no sink and no top-K.
    "window128k": Workload("window128k", 28, 4, 128, "bf16", 131072, 4096, 128, -1, n_sink=0,
                           rope=True, base_seed=1005, window=32),
    # 128K tokens in chunks of 8192, top-128: the per-call shape of the 1M and 4M
    # workloads (8192 queries, up to 1 + 128 + 64 selected pages) in ~2 GB of device
    # memory, the case the kernel profiles are captured on.
    "sparse128k_chunk8k": Workload("sparse128k_chunk8k", 28, 4, 128, "bf16", 131072, 8192, 128, 128,
                                   rope=True, plants=8, base_seed=1007),
    # A stack of 4 layers over 256K tokens in chunks of 8192, K/V and gradients in pinned
    # host memory: even layers retrieve the top-128 pages, odd layers attend to a local
    # window of 32 pages (the sparse layers of a sparse-native model); each layer draws
    # its own seeded tensors (the base seed plus 101 per layer).
    "stack4x256k": Workload("stack4x256k", 28, 4, 128, "bf16", 262144, 8192, 128, 128,
                            rope=True, plants=8, base_seed=1006, offload=True, offload_grads=True, window=32),
}

STACK_LAYERS = {"stack4x256k": 4}


def stack_layer(w: Workload, layer: int) -> Workload:
    """Layer ``layer`` of a stack workload: top-K retrieval on even layers, the local
    window on odd ones, and its own seed."""
    local = layer % 2 == 1
    return dataclasses.replace(w, name=f"{w.name}_layer{layer}", base_seed=w.base_seed + 101 * (layer + 1),
                               window=w.window if local else -1, plants=0 if local else w.plants)


def scaled(w: Workload, name: str, **kw) -> Workload:
    """A copy of workload ``w`` with some fields replaced (smaller test cases)."""
    return dataclasses.replace(w, name=name, **kw)


def _gen(w: Workload, c: int, tensor: int, device) -> torch.Generator:
    seed = (w.base_seed * 1_000_003 + (c + 7) * 1013 + tensor * 7919) % (2 ** 62)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def page_order(w: Workload) -> torch.Tensor:
    """Seeded order in which the allocator hands out physical pages (int32)."""
    g = _gen(w, -1, _T_PERM, "cpu")
    return torch.randperm(w.num_phys, generator=g).to(torch.int32)


def _rope(x: torch.Tensor, pos0: int, theta: float) -> torch.Tensor:
    """Rotate-half rotary embedding at absolute positions pos0.. (fp64 angles,
    fp32 application).  x: [n, H, d] fp32."""
    n, _, d = x.shape
    half = d // 2
    inv = theta ** (-torch.arange(0, half, dtype=torch.float64, device=x.device) * 2.0 / d)
    pos = torch.arange(pos0, pos0 + n, dtype=torch.float64, device=x.device)
    ang = pos[:, None] * inv[None, :]
    cos = torch.cos(ang).to(torch.float32)[:, None, :]
    sin = torch.sin(ang).to(torch.float32)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


class PlantTable:
    """Planted pages of the sparse workloads.

    For every chunk c with non-sink history and every KV head h, a seeded unit
    vector u[c,h] is added (times alpha) to all queries of the group, and (times
    beta) to every key of ``plants`` distinct non-sink history pages, so that the
    mean-key score of those pages stands out from the noise.
    """

    def __init__(self, w: Workload):
        self.w = w
        self.q_off = {}  # c -> [Hkv, d] fp32
        self.k_off = torch.zeros(w.n_pages, w.n_kv_heads, w.head_dim, dtype=torch.float32)
        self.planted = {}  # (c, h) -> list of logical pages
        if w.plants <= 0:
            return
        for c in range(w.n_chunks):
            start, _ = w.chunk_bounds(c)
            n_hist = start // w.page
            cand = n_hist - w.n_sink
            if cand <= 0:
                continue
            g = _gen(w, c, _T_PLANT, "cpu")
            u = torch.randn(w.n_kv_heads, w.head_dim, generator=g, dtype=torch.float32)
            u = u / u.norm(dim=1, keepdim=True)
            self.q_off[c] = w.plant_alpha * u
            for h in range(w.n_kv_heads):
                pages = (torch.randperm(cand, generator=g)[: w.plants] + w.n_sink).tolist()
                self.planted[(c, h)] = sorted(pages)
                for p in pages:
                    self.k_off[p, h] += w.plant_beta * u[h]


def make_chunk(w: Workload, c: int, device="cpu", plants: Optional[PlantTable] = None,
               need_do: bool = True):
    """Q, K, V (and dO) of chunk c in the workload's dtype on ``device``.

    Q: [n, Hq, d], K/V: [n, Hkv, d], dO: [n, Hq, d], token-major.
    """
    start, n = w.chunk_bounds(c)
    f32 = torch.float32
    q = torch.randn(n, w.n_q_heads, w.head_dim, generator=_gen(w, c, _T_Q, device),
                    device=device, dtype=f32)
    k = torch.randn(n, w.n_kv_heads, w.head_dim, generator=_gen(w, c, _T_K, device),
                    device=device, dtype=f32)
    v = torch.randn(n, w.n_kv_heads, w.head_dim, generator=_gen(w, c, _T_V, device),
                    device=device, dtype=f32)
    if w.rope:
        q = _rope(q, start, w.rope_theta)
        k = _rope(k, start, w.rope_theta)
    if plants is not None and w.plants > 0:
        if c in plants.q_off:
            off = plants.q_off[c].to(device)  # [Hkv, d]
            q = q + off.repeat_interleave(w.group, dim=0)[None]
        p0 = start // w.page
        p1 = -(-(start + n) // w.page)
        koff = plants.k_off[p0:p1].to(device)  # [pages, Hkv, d]
        tok_page = (torch.arange(start, start + n, device=device) // w.page) - p0
        k = k + koff[tok_page]
    out = {"q": q.to(w.torch_dtype), "k": k.to(w.torch_dtype), "v": v.to(w.torch_dtype)}
    if need_do:
        out["do"] = torch.randn(n, w.n_q_heads, w.head_dim, generator=_gen(w, c, _T_DO, device),
                                device=device, dtype=f32).to(w.torch_dtype)
    return out
