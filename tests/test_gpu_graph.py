"""The attention entries only enqueue work (no allocation, no synchronisation
on the call path), so a call can be captured into a CUDA graph and replayed.
A replay must give the same bits as the direct call on the same inputs (the
work split and its merge order depend only on the call's shape), and the pool
stays ready for direct calls after replays (each call's chunk counter is reset
by its own combine launch)."""
import pytest
import torch

import paged_kv_gqa_qk_gb300 as pkv
import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(wl, dev):
    return [t.to(dev) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w, wl.step_positions, wl.table)]


def test_decode_replays_from_a_graph():
    wl = W.make_decode("graph decode", (64, 512, 4096), seed=81, table_pages=64)
    dev = torch.device("cuda")
    q, k, v, qw, kw, sp, tab = _inputs(wl, dev)
    # direct call on a fresh pool: the expected bits
    K1, V1 = wl.K0.to(dev), wl.V0.to(dev)
    pool1 = pkv.PagedKVPool(K1, V1, cfg=wl.cfg)
    ref = pool1.decode(q, k, v, qw, kw, sp, tab)
    assert pool1.check_errors() == 0
    pool1.close()
    # captured call on another pool over the same initial K/V
    K2, V2 = wl.K0.to(dev), wl.V0.to(dev)
    pool2 = pkv.PagedKVPool(K2, V2, cfg=wl.cfg)
    out = torch.zeros_like(q)
    ws = pool2.workspace(wl.R, wl.pages, 0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):   # one direct call first (outside capture)
        pkv.pkv_decode(pool2.handle, q, k, v, qw, kw, sp, tab, out, ws, s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.pkv_decode(pool2.handle, q, k, v, qw, kw, sp, tab, out, ws, s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert pool2.check_errors() == 0
    assert torch.equal(K1, K2) and torch.equal(V1, V2)
    # a direct call after the replays still gives the same bits
    out2 = pool2.decode(q, k, v, qw, kw, sp, tab)
    assert pool2.check_errors() == 0 and torch.equal(out2, ref)
    pool2.close()


def test_step_replays_from_a_graph():
    wl = W.make_step("graph step", prompt_lengths=[130, 70], prompt_starts=[60, 0], decode_lengths=[90, 3, 64, 700],
                     seed=82, table_pages=14)
    dev = torch.device("cuda")
    q, k, v, qw, kw, sp, tab = _inputs(wl, dev)
    pos, prow = wl.positions.to(dev), wl.prow.to(dev)
    K1, V1 = wl.K0.to(dev), wl.V0.to(dev)
    pool1 = pkv.PagedKVPool(K1, V1, cfg=wl.cfg)
    ref = pool1.step(q, k, v, qw, kw, pos, prow, None, sp, tab)
    assert pool1.check_errors() == 0
    pool1.close()
    K2, V2 = wl.K0.to(dev), wl.V0.to(dev)
    pool2 = pkv.PagedKVPool(K2, V2, cfg=wl.cfg)
    out = torch.zeros_like(q)
    ws = pool2.workspace(wl.R, wl.pages, wl.P)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.pkv_step(pool2.handle, q, k, v, qw, kw, pos, prow, None, sp, tab, out, ws, s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert pool2.check_errors() == 0
    assert torch.equal(K1, K2) and torch.equal(V1, V2)
    pool2.close()
