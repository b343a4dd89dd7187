"""ctypes binding of liboomb.so: argument marshalling only.

Every function here forwards to the C entry point of the same name in
include/oomb.h, passing raw device pointers taken from torch tensors.  There is
no fallback: if liboomb.so is missing the import of the binding fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os
import re
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "liboomb.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "oomb.h")

OOMB_BF16, OOMB_FP32 = 0, 1
OOMB_CTRL_WORDS = 16  # uint32 words of a pool's control block (error bits + selection barrier state)
OOMB_OP_SELECT, OOMB_OP_BWD = 0, 1
STATUS = {0: "OK", 1: "ERR_ARG", 2: "ERR_OUT_OF_PAGES", 3: "ERR_ALIGN", 4: "ERR_DTYPE", 5: "ERR_KERNEL",
          6: "ERR_TIMEOUT", 7: "ERR_CUDA", 8: "ERR_UNSUPPORTED", 9: "ERR_WORKSPACE"}


class OombError(RuntimeError):
    def __init__(self, func: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{func}: {STATUS.get(status, status)} ({detail})")


class PoolDesc(C.Structure):
    _fields_ = [
        ("n_q_heads", C.c_int), ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("page_size", C.c_int),
        ("num_phys_pages", C.c_int), ("max_logical_pages", C.c_int), ("dtype", C.c_int),
        ("k_pool", C.c_void_p), ("v_pool", C.c_void_p), ("dk_pool", C.c_void_p), ("dv_pool", C.c_void_p),
        ("summary", C.c_void_p), ("page_table", C.c_void_p), ("error_word", C.c_void_p),
        ("page_order", C.c_void_p), ("offload", C.c_int), ("stage_k", C.c_void_p), ("stage_v", C.c_void_p),
        ("stage_max_sel", C.c_int), ("offload_grads", C.c_int), ("stage_dk", C.c_void_p),
        ("stage_dv", C.c_void_p), ("grad_state", C.c_void_p),
    ]


_lib: Optional[C.CDLL] = None


def header_symbols():
    """Names of the entry points include/oomb.h declares."""
    with open(HEADER) as f:
        txt = f.read()
    return sorted(set(re.findall(r"OOMB_API\s+[\w\s\*]+?\b(oomb_\w+)\s*\(", txt)))


def load(path: str = LIB_PATH) -> C.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run __graft_entry__.build() (nvcc, sm_103a)")
    lib = C.CDLL(path)
    vp, i32, i64, f32, sz = C.c_void_p, C.c_int, C.c_int64, C.c_float, C.c_size_t
    sig = {
        "oomb_pool_create": (i32, [C.POINTER(PoolDesc), C.POINTER(vp)]),
        "oomb_pool_destroy": (None, [vp]),
        "oomb_pool_reset": (i32, [vp, vp]),
        "oomb_kv_append": (i32, [vp, vp, vp, i64, i32, vp]),
        "oomb_kv_append_staged": (i32, [vp, vp, vp, i64, i32, vp, i32, i32, vp]),
        "oomb_kv_append_deferred": (i32, [vp, vp, vp, i64, i32, vp, i32, i32, vp]),
        "oomb_page_select_append": (i32, [vp, vp, vp, vp, i64, i32, i32, i32, vp, vp, i32, vp, sz, i32, i32, vp]),
        "oomb_kv_writeback": (i32, [vp, vp, vp, i32, i32, i64, i64, vp]),
        "oomb_page_select": (i32, [vp, vp, i64, i32, i32, i32, vp, vp, i32, vp, sz, vp]),
        "oomb_chunk_attn_fwd": (i32, [vp, vp, i64, i32, vp, vp, i32, f32, vp, vp, vp]),
        "oomb_chunk_attn_bwd": (i32, [vp, vp, vp, vp, vp, i64, i32, vp, vp, i32, f32, vp, vp, sz, vp]),
        "oomb_prefetch": (i32, [vp, vp, vp, i32, i32, vp]),
        "oomb_pool_set_stage": (i32, [vp, i32]),
        "oomb_prefetch_pages": (i32, [vp, vp, vp, i32, i32, i64, i64, vp]),
        "oomb_gemm": (i32, [i32, i32, i32, i32, i32, vp, vp, vp, i32, i32, f32, f32, vp, sz, vp]),
        "oomb_bias_rope": (i32, [vp, i32, vp, vp, i32, i32, i32, i32, i64, f32, i32, vp]),
        "oomb_grad_gather": (i32, [vp, i64, i32, vp, vp, vp]),
        "oomb_grad_prefetch": (i32, [vp, vp, vp, i32, vp, vp, i32, vp]),
        "oomb_grad_carry": (i32, [vp, vp, vp, i32, vp, vp, i32, vp]),
        "oomb_grad_writeback": (i32, [vp, vp, vp, i32, i32, vp]),
        "oomb_workspace_size": (sz, [vp, i32, i32]),
        "oomb_check": (i32, [vp, vp, C.POINTER(C.c_uint32)]),
        "oomb_page_table_host": (i32, [vp, vp, i32]),
        "oomb_pool_tokens": (i64, [vp]),
        "oomb_pool_free_pages": (i32, [vp]),
        "oomb_status_str": (C.c_char_p, [i32]),
        "oomb_uses_tensor_cores": (i32, [vp]),
        "oomb_launch_count": (C.c_uint64, []),
        "oomb_page_select_noalloc": (i32, [vp, vp, i64, i32, i32, i32, vp, vp, i32, vp]),
        "oomb_window_select": (i32, [vp, i64, i32, i32, i32, vp, vp, i32, vp]),
        "oomb_page_free": (i32, [vp, i64, i32, vp]),
        "oomb_last_cuda_error": (C.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr() if hasattr(t, "data_ptr") else int(t)


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ok(name: str, st: int):
    if st != 0:
        detail = load().oomb_status_str(st).decode()
        if st == 7:
            detail += ": " + load().oomb_last_cuda_error().decode()
        raise OombError(name, st, detail)


# ---------------------------------------------------------------- entry points
def oomb_pool_create(desc: PoolDesc) -> int:
    h = C.c_void_p()
    _ok("oomb_pool_create", load().oomb_pool_create(C.byref(desc), C.byref(h)))
    return h.value


def oomb_pool_destroy(pool: int) -> None:
    load().oomb_pool_destroy(pool)


def oomb_pool_reset(pool: int, stream=None) -> None:
    _ok("oomb_pool_reset", load().oomb_pool_reset(pool, _stream(stream)))


def oomb_kv_append(pool: int, k, v, first_token: int, n_tokens: Optional[int] = None, stream=None) -> None:
    n = k.shape[0] if n_tokens is None else n_tokens
    _ok("oomb_kv_append", load().oomb_kv_append(pool, _ptr(k), _ptr(v), first_token, n, _stream(stream)))


def oomb_kv_append_staged(pool: int, k, v, first_token: int, sel_count, max_sel: int, stage_buf: int,
                          n_tokens: Optional[int] = None, stream=None) -> None:
    n = k.shape[0] if n_tokens is None else n_tokens
    _ok("oomb_kv_append_staged", load().oomb_kv_append_staged(pool, _ptr(k), _ptr(v), first_token, n, _ptr(sel_count),
                                                              max_sel, stage_buf, _stream(stream)))


def oomb_kv_append_deferred(pool: int, k, v, first_token: int, sel_count, max_sel: int, stage_buf: int,
                            n_tokens: Optional[int] = None, stream=None) -> None:
    n = k.shape[0] if n_tokens is None else n_tokens
    _ok("oomb_kv_append_deferred", load().oomb_kv_append_deferred(pool, _ptr(k), _ptr(v), first_token, n,
                                                                  _ptr(sel_count), max_sel, stage_buf, _stream(stream)))


def oomb_kv_writeback(pool: int, sel, sel_count, stage_buf: int, first_page: int, end_page: int,
                      stream=None) -> None:
    _ok("oomb_kv_writeback", load().oomb_kv_writeback(pool, _ptr(sel), _ptr(sel_count), sel.shape[-1], stage_buf,
                                                      first_page, end_page, _stream(stream)))


def oomb_page_select(pool: int, q, q_start: int, top_k: int, n_sink: int, sel, sel_count, workspace,
                     n_q: Optional[int] = None, stream=None) -> None:
    n = q.shape[0] if n_q is None else n_q
    ws_bytes = workspace.numel() * workspace.element_size()
    _ok("oomb_page_select", load().oomb_page_select(pool, _ptr(q), q_start, n, top_k, n_sink, _ptr(sel),
                                                    _ptr(sel_count), sel.shape[-1], _ptr(workspace), ws_bytes,
                                                    _stream(stream)))


def oomb_page_free(pool: int, first_logical_page: int, n_pages: int, stream=None) -> None:
    _ok("oomb_page_free", load().oomb_page_free(pool, first_logical_page, n_pages, _stream(stream)))


def oomb_window_select(pool: int, q_start: int, n_q: int, window: int, n_sink: int, sel, sel_count,
                       stream=None) -> None:
    _ok("oomb_window_select", load().oomb_window_select(pool, q_start, n_q, window, n_sink, _ptr(sel),
                                                        _ptr(sel_count), sel.shape[-1], _stream(stream)))


def oomb_chunk_attn_fwd(pool: int, q, q_start: int, sel, sel_count, softmax_scale: float, o, lse,
                        n_q: Optional[int] = None, stream=None) -> None:
    n = q.shape[0] if n_q is None else n_q
    _ok("oomb_chunk_attn_fwd", load().oomb_chunk_attn_fwd(pool, _ptr(q), q_start, n, _ptr(sel), _ptr(sel_count),
                                                          sel.shape[-1], softmax_scale, _ptr(o), _ptr(lse),
                                                          _stream(stream)))


def oomb_chunk_attn_bwd(pool: int, q, o, d_o, lse, q_start: int, sel, sel_count, softmax_scale: float, dq,
                        workspace, n_q: Optional[int] = None, stream=None) -> None:
    n = q.shape[0] if n_q is None else n_q
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok("oomb_chunk_attn_bwd", load().oomb_chunk_attn_bwd(pool, _ptr(q), _ptr(o), _ptr(d_o), _ptr(lse), q_start, n,
                                                          _ptr(sel), _ptr(sel_count), sel.shape[-1], softmax_scale,
                                                          _ptr(dq), _ptr(workspace), ws_bytes, _stream(stream)))


def oomb_prefetch(pool: int, sel, sel_count, stage_buf: int, stream=None) -> None:
    _ok("oomb_prefetch", load().oomb_prefetch(pool, _ptr(sel), _ptr(sel_count), sel.shape[-1], stage_buf,
                                              _stream(stream)))


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return OOMB_FP32
    if t.dtype == torch.bfloat16:
        return OOMB_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def oomb_gemm(a, b, c, trans_a: bool = False, trans_b: bool = False, alpha: float = 1.0, beta: float = 0.0,
              workspace=None, stream=None) -> None:
    """c[m, n] = alpha op(a) op(b) + beta c (row-major, contiguous tensors)."""
    m, n = c.shape
    k = a.shape[0] if trans_a else a.shape[1]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok("oomb_gemm", load().oomb_gemm(m, n, k, int(trans_a), int(trans_b), _ptr(a), _ptr(b), _ptr(c), _dtype_code(a),
                                      _dtype_code(c), alpha, beta, _ptr(workspace), ws_bytes, _stream(stream)))


def oomb_bias_rope(x_in, bias, x_out, n_heads: int, pos0: int, theta: float, mode: int, stream=None) -> None:
    """x_out[i, h, :] = rotation(pos0 + i) (x_in[i, h, :] + bias[h, :]); mode 0 none, 1 forward, 2 inverse."""
    n = x_in.shape[0]
    d = x_in.numel() // (n * n_heads)
    _ok("oomb_bias_rope", load().oomb_bias_rope(_ptr(x_in), _dtype_code(x_in), _ptr(bias), _ptr(x_out),
                                                _dtype_code(x_out), n, n_heads, d, pos0, theta, mode,
                                                _stream(stream)))


def oomb_grad_gather(pool: int, first_token: int, dk, dv, stream=None) -> None:
    _ok("oomb_grad_gather", load().oomb_grad_gather(pool, first_token, dk.shape[0], _ptr(dk), _ptr(dv),
                                                    _stream(stream)))


def oomb_grad_prefetch(pool: int, sel, sel_count, prev_sel, prev_count, stage_buf: int, stream=None) -> None:
    _ok("oomb_grad_prefetch", load().oomb_grad_prefetch(pool, _ptr(sel), _ptr(sel_count), sel.shape[-1],
                                                        _ptr(prev_sel), _ptr(prev_count), stage_buf,
                                                        _stream(stream)))


def oomb_grad_carry(pool: int, sel, sel_count, prev_sel, prev_count, stage_buf: int, stream=None) -> None:
    _ok("oomb_grad_carry", load().oomb_grad_carry(pool, _ptr(sel), _ptr(sel_count), sel.shape[-1], _ptr(prev_sel),
                                                  _ptr(prev_count), stage_buf, _stream(stream)))


def oomb_grad_writeback(pool: int, sel, sel_count, stage_buf: int, stream=None) -> None:
    _ok("oomb_grad_writeback", load().oomb_grad_writeback(pool, _ptr(sel), _ptr(sel_count), sel.shape[-1],
                                                          stage_buf, _stream(stream)))


def oomb_prefetch_pages(pool: int, sel, sel_count, stage_buf: int, first_page: int, end_page: int,
                        stream=None) -> None:
    _ok("oomb_prefetch_pages", load().oomb_prefetch_pages(pool, _ptr(sel), _ptr(sel_count), sel.shape[-1], stage_buf,
                                                          first_page, end_page, _stream(stream)))


def oomb_pool_set_stage(pool: int, stage_buf: int) -> None:
    _ok("oomb_pool_set_stage", load().oomb_pool_set_stage(pool, stage_buf))


def oomb_workspace_size(pool: int, op: int, n_q: int) -> int:
    return int(load().oomb_workspace_size(pool, op, n_q))


def oomb_check(pool: int, stream=None) -> int:
    bits = C.c_uint32(0)
    st = load().oomb_check(pool, _stream(stream), C.byref(bits))
    if st != 0:
        raise OombError("oomb_check", st, f"device error bits 0x{bits.value:x}")
    return bits.value


def oomb_page_table_host(pool: int, n: int):
    buf = (C.c_int32 * n)()
    m = load().oomb_page_table_host(pool, buf, n)
    return list(buf)[:m]


def oomb_pool_tokens(pool: int) -> int:
    return int(load().oomb_pool_tokens(pool))


def oomb_pool_free_pages(pool: int) -> int:
    return int(load().oomb_pool_free_pages(pool))


def oomb_uses_tensor_cores(pool: int) -> bool:
    return bool(load().oomb_uses_tensor_cores(pool))


def oomb_launch_count() -> int:
    return int(load().oomb_launch_count())


OOMB_APPEND_POOL, OOMB_APPEND_STAGED, OOMB_APPEND_DEFERRED = 0, 1, 2


def oomb_page_select_append(pool: int, q, k, v, q_start: int, top_k: int, n_sink: int, sel, sel_count, workspace,
                            append_mode: int = OOMB_APPEND_POOL, stage_buf: int = 0, n_q: Optional[int] = None,
                            stream=None) -> None:
    """oomb_page_select and the append of the chunk's K/V (the chunk's tokens) in one call."""
    n = q.shape[0] if n_q is None else n_q
    ws_bytes = workspace.numel() * workspace.element_size()
    _ok("oomb_page_select_append", load().oomb_page_select_append(pool, _ptr(q), _ptr(k), _ptr(v), q_start, n, top_k,
                                                                  n_sink, _ptr(sel), _ptr(sel_count), sel.shape[-1],
                                                                  _ptr(workspace), ws_bytes, append_mode, stage_buf,
                                                                  _stream(stream)))


def oomb_page_select_noalloc(pool: int, q, q_start: int, top_k: int, n_sink: int, sel, sel_count,
                             n_q: Optional[int] = None, stream=None) -> None:
    """oomb_page_select with the library's static scratch instead of a workspace."""
    n = q.shape[0] if n_q is None else n_q
    _ok("oomb_page_select_noalloc", load().oomb_page_select_noalloc(pool, _ptr(q), q_start, n, top_k, n_sink,
                                                                    _ptr(sel), _ptr(sel_count), sel.shape[-1],
                                                                    _stream(stream)))
