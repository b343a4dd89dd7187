"""Device memory for a paged KV pool, allocated with torch and handed to liboomb.

torch only provides the memory (HBM, or pinned host memory for offload) and the
streams; every operation on it goes through the C entry points in _lib.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional

import torch

from . import _lib


class PagedKVPool:
    """K/V pools, the fp32 dK/dV gradient pool, page summaries and the page table
    of one attention layer, plus the library's pool object that manages them."""

    def __init__(self, n_q_heads: int, n_kv_heads: int, head_dim: int, page_size: int, num_phys_pages: int,
                 max_logical_pages: int, dtype: torch.dtype = torch.bfloat16, device="cuda",
                 page_order: Optional[torch.Tensor] = None, offload: bool = False, stage_max_sel: int = 0,
                 offload_grads: bool = False):
        self.Hq, self.Hkv, self.d, self.P = n_q_heads, n_kv_heads, head_dim, page_size
        self.num_phys, self.max_logical = num_phys_pages, max_logical_pages
        self.dtype, self.device, self.offload = dtype, torch.device(device), offload
        self.offload_grads = offload_grads
        if offload_grads and not offload:
            raise ValueError("offload_grads needs offload")
        shape = (num_phys_pages, n_kv_heads, page_size, head_dim)
        if offload:
            self.k_pool = torch.empty(shape, dtype=dtype, pin_memory=True)
            self.v_pool = torch.empty(shape, dtype=dtype, pin_memory=True)
            sshape = (2, n_kv_heads, stage_max_sel, page_size, head_dim)
            self.stage_k = torch.empty(sshape, dtype=dtype, device=self.device)
            self.stage_v = torch.empty(sshape, dtype=dtype, device=self.device)
        else:
            self.k_pool = torch.empty(shape, dtype=dtype, device=self.device)
            self.v_pool = torch.empty(shape, dtype=dtype, device=self.device)
            self.stage_k = self.stage_v = None
        if offload_grads:  # fp32 gradient pools in pinned host memory, staged blocks in HBM
            self.dk_pool = torch.zeros(shape, dtype=torch.float32, pin_memory=True)
            self.dv_pool = torch.zeros(shape, dtype=torch.float32, pin_memory=True)
            gshape = (2, n_kv_heads, stage_max_sel, page_size, head_dim)
            self.stage_dk = torch.empty(gshape, dtype=torch.float32, device=self.device)
            self.stage_dv = torch.empty(gshape, dtype=torch.float32, device=self.device)
            self.grad_state = torch.zeros((num_phys_pages, n_kv_heads), dtype=torch.uint8, device=self.device)
        else:
            self.dk_pool = torch.zeros(shape, dtype=torch.float32, device=self.device)
            self.dv_pool = torch.zeros(shape, dtype=torch.float32, device=self.device)
            self.stage_dk = self.stage_dv = self.grad_state = None
        self.summary = torch.zeros((num_phys_pages, n_kv_heads, head_dim), dtype=torch.float32, device=self.device)
        self.page_table = torch.empty(max_logical_pages, dtype=torch.int32, device=self.device)
        self.error_word = torch.zeros(_lib.OOMB_CTRL_WORDS, dtype=torch.int32, device=self.device)
        self._order = None if page_order is None else page_order.to(torch.int32).contiguous().cpu()
        d = _lib.PoolDesc()
        d.n_q_heads, d.n_kv_heads, d.head_dim, d.page_size = n_q_heads, n_kv_heads, head_dim, page_size
        d.num_phys_pages, d.max_logical_pages = num_phys_pages, max_logical_pages
        d.dtype = _lib.OOMB_FP32 if dtype == torch.float32 else _lib.OOMB_BF16
        d.k_pool, d.v_pool = self.k_pool.data_ptr(), self.v_pool.data_ptr()
        d.dk_pool, d.dv_pool = self.dk_pool.data_ptr(), self.dv_pool.data_ptr()
        d.summary, d.page_table = self.summary.data_ptr(), self.page_table.data_ptr()
        d.error_word = self.error_word.data_ptr()
        d.page_order = None if self._order is None else self._order.data_ptr()
        d.offload = 1 if offload else 0
        d.stage_k = None if self.stage_k is None else self.stage_k.data_ptr()
        d.stage_v = None if self.stage_v is None else self.stage_v.data_ptr()
        d.stage_max_sel = stage_max_sel
        d.offload_grads = 1 if offload_grads else 0
        d.stage_dk = None if self.stage_dk is None else self.stage_dk.data_ptr()
        d.stage_dv = None if self.stage_dv is None else self.stage_dv.data_ptr()
        d.grad_state = None if self.grad_state is None else self.grad_state.data_ptr()
        self.handle = _lib.oomb_pool_create(d)

    def close(self):
        if getattr(self, "handle", None):
            _lib.oomb_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover - best effort
        try:
            self.close()
        except Exception:
            pass

    # convenience views -------------------------------------------------------
    def table_host(self, n: Optional[int] = None):
        return _lib.oomb_page_table_host(self.handle, self.max_logical if n is None else n)

    @property
    def n_tokens(self) -> int:
        return _lib.oomb_pool_tokens(self.handle)

    def workspace(self, op: int, n_q: int) -> torch.Tensor:
        nbytes = _lib.oomb_workspace_size(self.handle, op, n_q)
        return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=self.device)

    def logical_grads(self, n_tokens: int):
        """dK, dV gathered to token-major [n, Hkv, d] through the host page table."""
        n_pages = -(-n_tokens // self.P)
        phys = torch.tensor(self.table_host(n_pages), dtype=torch.long, device=self.dk_pool.device)
        if self.offload_grads:
            torch.cuda.synchronize(self.device)  # write-backs into the host pools have landed
        dk = self.dk_pool[phys].permute(0, 2, 1, 3).reshape(n_pages * self.P, self.Hkv, self.d)[:n_tokens]
        dv = self.dv_pool[phys].permute(0, 2, 1, 3).reshape(n_pages * self.P, self.Hkv, self.d)[:n_tokens]
        return dk, dv

    def logical_kv(self, n_tokens: int):
        n_pages = -(-n_tokens // self.P)
        phys = torch.tensor(self.table_host(n_pages), dtype=torch.long)
        kp = self.k_pool.to(self.device) if self.offload else self.k_pool
        vp = self.v_pool.to(self.device) if self.offload else self.v_pool
        phys = phys.to(kp.device)
        k = kp[phys].permute(0, 2, 1, 3).reshape(n_pages * self.P, self.Hkv, self.d)[:n_tokens]
        v = vp[phys].permute(0, 2, 1, 3).reshape(n_pages * self.P, self.Hkv, self.d)[:n_tokens]
        return k, v
