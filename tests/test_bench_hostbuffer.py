"""The end-to-end leg's host buffers, checked on the CPU: bench.HostBuffer packs the
step's tensors into fixed-size page-locked blocks, so a packing mistake (two
tensors sharing bytes, a tensor running past its block) would upload wrong inputs
without any error.  Page-locking needs a GPU, so the allocator is replaced here by
plain host memory; the packing logic is the bench's own."""
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _plain_host(monkeypatch, block):
    real_empty = torch.empty

    def empty(*args, pin_memory=False, **kw):
        return real_empty(*args, **kw)

    monkeypatch.setattr(torch, "empty", empty)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a, **k: None)
    monkeypatch.setattr(bench.HostBuffer, "BLOCK", block)


def _span(t):
    return t.data_ptr(), t.data_ptr() + t.numel() * t.element_size()


def test_tensors_are_disjoint_aligned_and_inside_their_blocks(monkeypatch):
    block = 1 << 16
    _plain_host(monkeypatch, block)
    hb = bench.HostBuffer()
    specs = [((100, 7, 16), torch.bfloat16),   # 22,400 B
             ((3, 5), torch.float32),          # 60 B: packing continues in the block
             ((20_000,), torch.uint8),         # does not fit the rest of block 1
             ((block // 4,), torch.float32),   # exactly one block: packed, not separate
             ((block // 4 + 1,), torch.float32),  # above a block: a block of its own
             ((1,), torch.bfloat16),
             ((40_000,), torch.uint8)]
    ts = [hb.take(s, d) for s, d in specs]
    for t, (s, d) in zip(ts, specs):
        assert tuple(t.shape) == s and t.dtype == d and t.is_contiguous()
    spans = sorted(_span(t) for t in ts)
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0, "two tensors share bytes"
    # every packed tensor lies inside one block, on a 256-byte offset
    blocks = [_span(b) for b in hb.blocks if b.dtype == torch.uint8 and b.numel() == block]
    for t in ts:
        n = t.numel() * t.element_size()
        if n > block:
            assert any(t.data_ptr() == b.data_ptr() for b in hb.blocks)
            continue
        lo, hi = _span(t)
        owner = [b for b in blocks if b[0] <= lo and hi <= b[1]]
        assert len(owner) == 1
        assert (lo - owner[0][0]) % 256 == 0
    # the bytes survive: distinct fills read back intact
    for i, t in enumerate(ts):
        t.view(torch.uint8).fill_(i + 1)
    for i, t in enumerate(ts):
        assert bool((t.view(torch.uint8) == i + 1).all())
    hb.close()
    assert hb.blocks == []


def test_blocks_are_full_size_only_when_needed(monkeypatch):
    block = 1 << 12
    _plain_host(monkeypatch, block)
    hb = bench.HostBuffer()
    for _ in range(10):
        hb.take((1000,), torch.uint8)  # 1000 B, 256-aligned: four per 4 KB block
    packed = [b for b in hb.blocks if b.numel() == block]
    assert len(packed) == 3  # 4 + 4 + 2
    hb.close()
