"""Paged sparse chunk attention for GB300 (sm_103a): the hot path of OOMB's
chunk-recurrent long-context training behind the C ABI in include/oomb.h.

The CUDA library (liboomb.so) does all of the work; this package only marshals
arguments (``_lib``), provides device memory for a pool (``pool``), builds the
library (``build``) and draws seeded synthetic inputs (``synth``).
"""
from ._lib import (OOMB_APPEND_DEFERRED, OOMB_APPEND_POOL, OOMB_APPEND_STAGED, OOMB_BF16,  # noqa: F401
                   OOMB_FP32, OOMB_OP_BWD, OOMB_OP_SELECT, OombError, header_symbols, load, oomb_bias_rope,
                   oomb_check, oomb_chunk_attn_bwd, oomb_chunk_attn_fwd, oomb_gemm, oomb_grad_carry,
                   oomb_grad_gather, oomb_grad_prefetch, oomb_grad_writeback, oomb_kv_append, oomb_kv_append_deferred,
                   oomb_kv_append_staged, oomb_kv_writeback, oomb_launch_count, oomb_page_free, oomb_page_select,
                   oomb_page_select_append, oomb_page_select_noalloc, oomb_page_table_host, oomb_pool_create,
                   oomb_pool_destroy, oomb_pool_free_pages, oomb_pool_reset, oomb_pool_set_stage, oomb_pool_tokens,
                   oomb_prefetch, oomb_prefetch_pages, oomb_uses_tensor_cores, oomb_window_select, oomb_workspace_size)
