"""The benchmark's offload schedule (bench.Step.run_offload: selection, deferred
append into the staging slots, history gathers on one high-priority stream, K/V
and gradient write-backs on another, gradient stage-in / carry in the reverse sweep)
against the same workload with every pool in HBM: the same selections, O and LSE of
the forward sweep and the final dK/dV bit for bit, dQ to rounding (its fp32
reductions across thread blocks run in a run-dependent order), the host K/V pools
equal to the resident ones; and the same again on a second step (the pools are
reset and refilled, and state bytes of the gradient blocks restart at empty); and
the variant that keeps the forward sweep's outputs instead of recomputing them
gives the same gradients."""
import dataclasses

import pytest
import torch

import oracle.oomb_oracle as O
import paged_sparse_attention_gb300 as L
from paged_sparse_attention_gb300 import synth

from harness import f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("window", [-1, 4], ids=["topk", "window"])
def test_offload_schedule_matches_resident(window):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from paged_sparse_attention_gb300 import build
    build.build()
    base = synth.WORKLOADS["offload4m"]
    w_off = synth.scaled(base, "offload_small", seq=12 * 4096 + 1536, chunk=4096, top_k=12, plants=2,
                         window=window, n_sink=1)
    w_res = dataclasses.replace(w_off, name="resident_small", offload=False, offload_grads=False)
    dev = torch.device("cuda")
    off = bench.Step(w_off, dev)
    res = bench.Step(w_res, dev)
    assert off.offload and not res.offload
    for _ in range(2):
        res.run()
        off.run()
        torch.cuda.synchronize()
        assert L.oomb_check(off.pool.handle) == 0 and L.oomb_check(res.pool.handle) == 0
        assert torch.equal(off.cnt, res.cnt)
        for c in range(w_off.n_chunks):
            for h in range(w_off.n_kv_heads):
                k = int(res.cnt[c, h])
                assert torch.equal(off.sel[c, h, :k], res.sel[c, h, :k]), (c, h)
            assert O.rel_l2(f64(off.dq[c]), f64(res.dq[c])) < 1e-3, c
        dk, dv = off.pool.logical_grads(w_off.seq)
        rdk, rdv = res.pool.logical_grads(w_res.seq)
        assert torch.equal(dk.cpu(), rdk.cpu()) and torch.equal(dv.cpu(), rdv.cpu())
        ok, ov = off.pool.logical_kv(w_off.seq)
        rk, rv = res.pool.logical_kv(w_res.seq)
        assert torch.equal(ok.cpu(), rk.cpu()) and torch.equal(ov.cpu(), rv.cpu())
    # the forward of the last chunk (its buffers hold the forward sweep's O and LSE)
    assert torch.equal(off.ob[0], res.ob[0]) and torch.equal(off.lseb[0], res.lseb[0])
    # without the recomputed forward (outputs kept per chunk): the same gradients bit for bit
    off.run(no_recompute=True)
    torch.cuda.synchronize()
    assert L.oomb_check(off.pool.handle) == 0
    dk2, dv2 = off.pool.logical_grads(w_off.seq)
    assert torch.equal(dk2.cpu(), rdk.cpu()) and torch.equal(dv2.cpu(), rdv.cpu())
    for c in range(w_off.n_chunks):
        assert O.rel_l2(f64(off.dq[c]), f64(res.dq[c])) < 1e-3, c
    off.pool.close()
    res.pool.close()
