"""The multi-layer offload step (bench.StackStep): layers run chunk by chunk in model
order, local layers' pages staged one layer ahead, top-K layers' history pages moved
while a K/V projection GEMM runs, reverse-sweep blocks staged two layers ahead.  The
schedule must not change any result: every layer's selections, dQ and final
gradient pools equal those of the same layer run alone through the single-layer
offload step (selections and dK/dV bit for bit, dQ to rounding: its fp32 reductions
across thread blocks run in a run-dependent order)."""
import os
import sys

import numpy as np
import pytest
import torch

import oracle.oomb_oracle as O
import paged_sparse_attention_gb300 as L
from paged_sparse_attention_gb300 import synth

from harness import f64

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


def test_stack_schedule_matches_single_layers():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_sparse_attention_gb300 import build
    build.build()
    w = synth.scaled(synth.WORKLOADS["stack4x256k"], "stack_small", seq=3072, chunk=512, top_k=3, window=2,
                     plants=2)
    dev = torch.device("cuda")
    stack = bench.StackStep(w, 3, dev, model_dim=256)
    stack.run()
    stack.run()  # twice: the pools are reset and refilled, results must not depend on it
    torch.cuda.synchronize()
    for layer, st in enumerate(stack.layers):
        assert L.oomb_check(st.pool.handle) == 0
        ref = bench.Step(synth.stack_layer(w, layer), dev)
        ref.run()
        torch.cuda.synchronize()
        assert L.oomb_check(ref.pool.handle) == 0
        assert torch.equal(st.cnt, ref.cnt), layer
        for c in range(w.n_chunks):
            for h in range(w.n_kv_heads):
                k = int(ref.cnt[c, h])
                assert torch.equal(st.sel[c, h, :k], ref.sel[c, h, :k]), (layer, c, h)
            assert O.rel_l2(f64(st.dq[c]), f64(ref.dq[c])) < 1e-3, (layer, c)
        dk, dv = st.pool.logical_grads(w.seq)
        rdk, rdv = ref.pool.logical_grads(w.seq)
        assert torch.equal(dk, rdk) and torch.equal(dv, rdv), layer
        assert float(np.abs(f64(dk)).max()) > 0  # gradients actually flowed
        ref.pool.close()
    for st in stack.layers:
        st.pool.close()
