"""The decode attention kernel's bounded waits, run out on purpose.

Every wait inside the kernel (the shared-memory ring between its copy warp and
its compute warps, and the compute warps' meeting points) gives up after the
pool's wait limit.  A limit of 0 gives up at the first check that finds the
awaited copy not yet landed, which on any real batch happens at once.  The
call must then return, report PKV_DEVERR_TIMEOUT through pkv_check_errors
(with no CUDA error: each CTA lets its copies in flight land before it
exits), and leave the pool ready: the next call at the default limit gives
the same bits as a call on a fresh pool, and matches the oracle.  Nothing
here faults or hangs the GPU; the failure is only a wait that is told to give
up early.
"""
import pytest
import torch

import paged_kv_gqa_qk_gb300 as pkv
import workloads as W
from _harness import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("config", [1, 2])
def test_wait_limit_runs_out_then_the_pool_recovers(config):
    wl = W.CONFIGS[config]()
    dev = torch.device("cuda")
    q, k, v, qw, kw, sp, tab = (t.to(dev) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w,
                                                     wl.step_positions, wl.table))
    K, V = wl.K0.to(dev), wl.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
    pkv.pkv_set_wait_limit(pool.handle, 0)
    for _ in range(2):
        pool.decode(q, k, v, qw, kw, sp, tab)
        flags = pool.check_errors()      # synchronises: the call has returned, and no CUDA error
        assert flags & pkv.PKV_DEVERR_TIMEOUT, flags
        assert flags == pkv.PKV_DEVERR_TIMEOUT, flags
    pkv.pkv_set_wait_limit(pool.handle, 10 ** 9)
    out = pool.decode(q, k, v, qw, kw, sp, tab)
    assert pool.check_errors() == 0
    res = (out.cpu(), K.cpu(), V.cpu(), 0)
    pool.close()
    clean = run_gpu(wl)
    assert clean[3] == 0
    for a, b in zip(res[:3], clean[:3]):
        assert torch.equal(a, b)
    compare(wl, res, run_oracle(wl), label=f"config{config} after a timed-out call")


def test_wait_limit_rejects_negative_values():
    wl = W.config1()
    dev = torch.device("cuda")
    pool = pkv.PagedKVPool(wl.K0.to(dev), wl.V0.to(dev), cfg=wl.cfg)
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_set_wait_limit(pool.handle, -1)
    assert ei.value.code == pkv.PKV_EINVAL
    pool.close()
