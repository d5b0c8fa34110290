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
