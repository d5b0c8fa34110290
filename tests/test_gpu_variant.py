"""GPU parity of the gated-attention variant (fantasma model.zig, "Full
Attention (GQA with output gate + QK-norm + partial RoPE)"): pools whose
rotary_dim is below head_dim rotate only the first rotary_dim dims of q and k
(pairs (i, i + rotary_dim/2)), and pkv_output_gate multiplies the attention
output by sigmoid(gate).  Same bar as the other parity tests."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_qk_gb300 as pkv
import workloads as W
from _harness import MAX_ABS, REL_L2, compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def with_rot(wl, rot):
    return W.Workload(**{**wl.__dict__, "cfg": dict(wl.cfg, rotary_dim=rot)})


@pytest.mark.parametrize("rot", [32, 64, 96])
def test_partial_rope_decode(rot):
    wl = with_rot(W.make_decode("partial rope", [1, 63, 64, 65, 300, 1000, 2049], seed=50 + rot, table_pages=33), rot)
    compare(wl, run_gpu(wl), run_oracle(wl), label=f"decode rot={rot}")
    compare(wl, run_gpu(wl, ctas=7), run_oracle(wl), label=f"decode rot={rot} ctas=7")


@pytest.mark.parametrize("rot", [32, 64])
def test_partial_rope_step_and_prefill(rot):
    wl = with_rot(W.make_step("partial rope step", prompt_lengths=[70, 5, 130], prompt_starts=[60, 0, 500],
                              decode_lengths=[90, 3, 64, 65, 1], seed=60 + rot, table_pages=12), rot)
    compare(wl, run_gpu(wl), run_oracle(wl), label=f"step rot={rot}")
    pf = with_rot(W.make_prefill("partial rope prefill", [70, 5, 130, 300], [60, 0, 500, 64], seed=70 + rot,
                                 table_pages=14), rot)
    compare(pf, run_gpu(pf), run_oracle(pf), label=f"prefill rot={rot}")


def test_rotary_dim_checks():
    K = torch.zeros(8, 64, 128, dtype=torch.bfloat16, device="cuda")
    for rot, code in [(48, pkv.PKV_ENOTIMPL), (130, pkv.PKV_EINVAL), (33, pkv.PKV_EINVAL)]:
        with pytest.raises(pkv.PkvError) as ei:
            pkv.PagedKVPool(K, K.clone(), cfg=dict(oracle.DEFAULT_CONFIG, rotary_dim=rot))
        assert ei.value.code == code


def test_output_gate():
    """The gated variant end to end on a decode batch: partial RoPE (rotary_dim 32) attention, then
    out *= sigmoid(gate), against the oracle's fp64 attention times the fp64 sigmoid."""
    wl = with_rot(W.make_decode("gated", [100, 700, 64, 1500], seed=81, table_pages=24), 32)
    gen = torch.Generator().manual_seed(82)
    gate = (2 * torch.randn(wl.q.shape, generator=gen)).to(torch.bfloat16)
    dev = torch.device("cuda")
    K, V = wl.K0.to(dev), wl.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
    q, k, v, qw, kw, sp, tab = (t.to(dev) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w, wl.step_positions,
                                                     wl.table))
    out = pool.decode(q, k, v, qw, kw, sp, tab)
    pkv.pkv_output_gate(pool.handle, out, gate.to(dev))
    assert pool.check_errors() == 0
    got = out.cpu().double().numpy()
    ref = oracle.output_gate(run_oracle(wl)[0], W.bits(gate))
    max_abs = float(np.abs(got - ref).max())
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    print(f"[parity] gated decode: max-abs {max_abs:.3e} rel-L2 {rel:.3e}")
    assert max_abs <= MAX_ABS and rel <= REL_L2
    pool.close()
