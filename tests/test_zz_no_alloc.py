"""pkv_decode_static, the decode entry point for callers that cannot allocate
device memory (it runs on a scratch array compiled into the library instead
of a caller workspace), against pkv_decode with a caller workspace.

Collected last on purpose (file name), so that a run stopping at the first
failure has run every other test before this one.  It builds the library if
needed, so it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import __graft_entry__
import paged_kv_gqa_qk_gb300 as pkv
import workloads as W
from _harness import MAX_ABS, REL_L2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return pkv.load_library()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_static_scratch_matches_workspace_decode(lib):
    wl = W.config2()
    dev = torch.device("cuda")
    q, k, v, qw, kw, pos, tab = (t.to(dev) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w,
                                                    wl.step_positions, wl.table))
    # the existing entry point, with a caller workspace
    K1, V1 = wl.K0.to(dev), wl.V0.to(dev)
    pool1 = pkv.PagedKVPool(K1, V1, cfg=wl.cfg)
    ref = pool1.decode(q, k, v, qw, kw, pos, tab)
    assert pool1.check_errors() == 0
    ref64 = ref.double().cpu().numpy()

    # the no-allocation entry point, called twice in a row through the C ABI
    K2, V2 = wl.K0.to(dev), wl.V0.to(dev)
    pool2 = pkv.PagedKVPool(K2, V2, cfg=wl.cfg)
    stream = torch.cuda.current_stream()
    for call in range(2):
        out = torch.zeros_like(q)
        rc = lib.pkv_decode_static(pool2.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(qw), _ptr(kw), _ptr(pos),
                                   _ptr(tab), wl.R, wl.pages, _ptr(out), ctypes.c_void_p(stream.cuda_stream))
        assert rc == pkv.PKV_OK, pkv.pkv_strerror(rc)
        assert pool2.check_errors() == 0
        got = out.double().cpu().numpy()
        max_abs = float(np.abs(got - ref64).max())
        rel = float(np.linalg.norm(got - ref64) / np.linalg.norm(ref64))
        assert max_abs <= MAX_ABS and rel <= REL_L2, (call, max_abs, rel)
    assert torch.equal(K1, K2) and torch.equal(V1, V2)
    pool1.close()
    pool2.close()


def test_static_scratch_rejects_calls_beyond_its_size(lib):
    wl = W.config1()
    dev = torch.device("cuda")
    K, V = wl.K0.to(dev), wl.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
    rows, pages = 4096, 640
    assert pkv.pkv_workspace_bytes(pool.handle, rows, pages, 0) > pkv.PKV_STATIC_SCRATCH_BYTES
    q = torch.zeros(rows, 32, 128, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(rows, 8, 128, dtype=torch.bfloat16, device=dev)
    pos = torch.zeros(rows, dtype=torch.int32, device=dev)
    tab = torch.zeros(rows, pages, dtype=torch.int32, device=dev)
    out = torch.ones_like(q)
    w = wl.q_norm_w.to(dev)
    rc = lib.pkv_decode_static(pool.handle, _ptr(q), _ptr(kv), _ptr(kv), _ptr(w), _ptr(w), _ptr(pos), _ptr(tab),
                               rows, pages, _ptr(out), None)
    assert rc == pkv.PKV_ERANGE
    torch.cuda.synchronize()
    assert torch.equal(K.cpu(), wl.K0) and bool((out == 1).all())
    pool.close()


def _static_vs_workspace(lib, wl, ctas=0, table=True):
    """One pkv_decode (caller workspace) and two pkv_decode_static calls in a row
    on equal pools; the outputs agree within the parity tolerance and the pools
    bit for bit."""
    dev = torch.device("cuda")
    q, k, v, qw, kw, pos = (t.to(dev) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w, wl.step_positions))
    tab = wl.table.to(dev) if table else None
    pools, outs = [], []
    for static in (False, True):
        K, V = wl.K0.to(dev), wl.V0.to(dev)
        pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
        if ctas:
            pkv.pkv_set_ctas(pool.handle, ctas)
        for call in range(2 if static else 1):
            out = torch.zeros_like(q)
            if static:
                rc = lib.pkv_decode_static(pool.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(qw), _ptr(kw), _ptr(pos),
                                           _ptr(tab) if tab is not None else None, wl.R, wl.pages, _ptr(out),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
                assert rc == pkv.PKV_OK, pkv.pkv_strerror(rc)
            else:
                pool.decode(q, k, v, qw, kw, pos, tab, out=out, pages=wl.pages)
            assert pool.check_errors() == 0
            outs.append(out.double().cpu().numpy())
        pools.append(pool)
    ref = outs[0]
    for got in outs[1:]:
        max_abs = float(np.abs(got - ref).max())
        rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
        assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert torch.equal(pools[0].K, pools[1].K) and torch.equal(pools[0].V, pools[1].V)
    for pl in pools:
        pl.close()


def test_static_scratch_contiguous_rows_and_grid_sizes(lib):
    """A NULL table (contiguous rows), and grids of one CTA and of 608 CTAs
    (the grid size sets how much of the scratch the split's partials take:
    about 35 KiB a CTA, so a 1000-CTA grid no longer fits and is refused)."""
    wl = W.make_decode("decode_rows 64 x 640", (64, 1, 640), seed=34, table_pages=10, contiguous=True)
    _static_vs_workspace(lib, wl, table=False)
    small = W.make_decode("ragged", [1, 65, 640, 1000, 4097], seed=77, table_pages=70)
    _static_vs_workspace(lib, small, ctas=1)
    _static_vs_workspace(lib, small, ctas=608)
    dev = torch.device("cuda")
    K, V = small.K0.to(dev), small.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=small.cfg)
    pkv.pkv_set_ctas(pool.handle, 1000)
    assert pkv.pkv_workspace_bytes(pool.handle, small.R, small.pages, 0) > pkv.PKV_STATIC_SCRATCH_BYTES
    q, k, v, qw, kw, pos, tab = (t.to(dev) for t in (small.q, small.k, small.v, small.q_norm_w, small.k_norm_w,
                                                    small.step_positions, small.table))
    out = torch.ones_like(q)
    rc = lib.pkv_decode_static(pool.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(qw), _ptr(kw), _ptr(pos), _ptr(tab),
                               small.R, small.pages, _ptr(out), None)
    assert rc == pkv.PKV_ERANGE
    torch.cuda.synchronize()
    assert torch.equal(K.cpu(), small.K0) and bool((out == 1).all())
    pool.close()


def test_static_scratch_at_its_size_limit(lib):
    """The most rows whose scratch fits the array run (and agree with
    pkv_decode); one row more is refused with PKV_ERANGE."""
    wl1 = W.config1()
    dev = torch.device("cuda")
    probe = pkv.PagedKVPool(wl1.K0.to(dev), wl1.V0.to(dev), cfg=wl1.cfg)
    pages = 2
    lo, hi = 1, 1 << 16   # pkv_workspace_bytes grows with rows: find the largest that fits
    assert pkv.pkv_workspace_bytes(probe.handle, hi, pages, 0) > pkv.PKV_STATIC_SCRATCH_BYTES
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if pkv.pkv_workspace_bytes(probe.handle, mid, pages, 0) <= pkv.PKV_STATIC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    probe.close()
    rows = lo
    assert rows > 1000
    wl = W.make_decode("at the scratch limit", (rows, 1, 128), seed=91, table_pages=pages)
    _static_vs_workspace(lib, wl)
    over = W.make_decode("one row over the scratch limit", (rows + 1, 1, 128), seed=92, table_pages=pages)
    K, V = over.K0.to(dev), over.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=over.cfg)
    q, k, v, qw, kw, pos, tab = (t.to(dev) for t in (over.q, over.k, over.v, over.q_norm_w, over.k_norm_w,
                                                    over.step_positions, over.table))
    out = torch.ones_like(q)
    rc = lib.pkv_decode_static(pool.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(qw), _ptr(kw), _ptr(pos), _ptr(tab),
                               over.R, over.pages, _ptr(out), None)
    assert rc == pkv.PKV_ERANGE
    torch.cuda.synchronize()
    assert torch.equal(K.cpu(), over.K0) and bool((out == 1).all())
    pool.close()
