"""GPU parity of pkv_linear (the q/k/v projections before the attention and
o_proj after it, y = x w^T) against the fp64 oracle.

Tolerance, from the arithmetic: the products of bf16 values are exact in fp32,
the tensor cores add them in fp32 (at most `in` additions, each off by at most
2^-23 of the running magnitude, bounded by sum_k |x_k w_ok|), and the output is
rounded once to bf16 (at most half an ulp, 2^-8 of the value).  So each element
must satisfy
    |y - y_ref| <= 2^-8 |y_ref| + in * 2^-23 * sum_k |x_k w_ok|
(the rounding bound plus the full accumulation bound)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_qk_gb300 as pkv
import workloads as W

pytestmark = pytest.mark.gpu


def check(x, w, y, label):
    xb, wb = W.bits(x), W.bits(w)
    ref = oracle.linear(xb, wb)
    mag = np.abs(oracle.bf16_to_f64(xb)) @ np.abs(oracle.bf16_to_f64(wb)).T
    got = y.float().double().numpy()
    bound = 2.0 ** -8 * np.abs(ref) + x.shape[1] * 2.0 ** -23 * mag
    err = np.abs(got - ref)
    worst = float((err / np.maximum(bound, 1e-30)).max())
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    print(f"[parity] linear {label}: worst err/bound {worst:.3f}, rel-L2 {rel:.2e}")
    assert worst <= 1.0, f"{label}: error {worst:.3f} x the bound"
    assert rel <= 4e-3


@pytest.fixture(scope="module")
def pool():
    p = pkv.PagedKVPool(torch.zeros(8, 64, 128, dtype=torch.bfloat16, device="cuda"),
                        torch.zeros(8, 64, 128, dtype=torch.bfloat16, device="cuda"))
    yield p
    p.close()


@pytest.mark.parametrize("tokens,in_f,out_f", [
    (1, 4096, 4096),      # one decode row, q_proj / o_proj
    (7, 256, 384),        # ragged token tile, 3 output tiles
    (64, 4096, 1024),     # k_proj / v_proj of the 64-row decode batch (split over the input features)
    (64, 4096, 4096),     # q_proj / o_proj of the same batch
    (64, 4096, 6144),     # q, k, v stacked for the same batch (a cluster of 6: uneven feature slices)
    (200, 512, 640),      # a 256-token tile with a ragged tail
    (300, 1024, 256),     # two token tiles, the second ragged
])
def test_linear_matches_oracle(pool, tokens, in_f, out_f):
    x, w = W.make_linear(tokens, in_f, out_f, seed=tokens * 7 + in_f + out_f)
    y = pool.linear(x.cuda(), w.cuda())
    assert pool.check_errors() == 0
    check(x, w, y.cpu(), f"{tokens}x{in_f}->{out_f}")


def test_linear_prefill_size_sampled_rows(pool):
    """q_proj over the 2048 prompt tokens of the step workload; the oracle checks every 37th row."""
    x, w = W.make_linear(2048, 4096, 4096, seed=5)
    y = pool.linear(x.cuda(), w.cuda()).cpu()
    assert pool.check_errors() == 0
    rows = list(range(0, 2048, 37)) + [2047]
    check(x[rows], w, y[rows], "2048x4096->4096 (sampled rows)")


def test_linear_repeat_is_deterministic(pool):
    x, w = W.make_linear(64, 4096, 1024, seed=9)
    xc, wc = x.cuda(), w.cuda()
    a = pool.linear(xc, wc).clone()
    b = pool.linear(xc, wc)
    assert torch.equal(a, b)


def test_linear_host_errors(pool):
    x, w = W.make_linear(4, 128, 128, seed=1)
    xc, wc = x.cuda(), w.cuda()
    y = torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as ei:   # input features not a multiple of 64
        pkv.pkv_linear(pool.handle, xc[:, :96].contiguous(), wc[:, :96].contiguous(), y)
    assert ei.value.code == pkv.PKV_ENOTIMPL
    with pytest.raises(pkv.PkvError) as ei:   # output features not a multiple of 128
        pkv.pkv_linear(pool.handle, xc, wc[:96].contiguous(), y[:, :96].contiguous())
    assert ei.value.code == pkv.PKV_ENOTIMPL
    with pytest.raises(pkv.PkvError) as ei:   # no tokens
        pkv.pkv_linear(pool.handle, xc[:0], wc, y[:0])
    assert ei.value.code == pkv.PKV_EINVAL
    torch.cuda.synchronize()
    assert not y.any()
    assert pkv.pkv_linear_workspace_bytes(pool.handle, 8, 4096, 1024) == 0


@pytest.mark.parametrize("tokens", [1, 64, 300])
def test_qkv_proj_matches_oracle(pool, tokens):
    """The fused projection writes q, k, v (each split into heads) as three separate linears would."""
    c = pool.cfg
    wq_rows, wk_rows = c.heads * c.head_dim, c.kv_heads * c.head_dim
    x, w = W.make_linear(tokens, 512, wq_rows + 2 * wk_rows, seed=40 + tokens)
    q, k, v = pool.qkv_proj(x.cuda(), w.cuda())
    assert pool.check_errors() == 0
    assert q.shape == (tokens, c.heads, c.head_dim) and k.shape == v.shape == (tokens, c.kv_heads, c.head_dim)
    check(x, w[:wq_rows], q.reshape(tokens, -1).cpu(), f"qkv q {tokens}")
    check(x, w[wq_rows:wq_rows + wk_rows], k.reshape(tokens, -1).cpu(), f"qkv k {tokens}")
    check(x, w[wq_rows + wk_rows:], v.reshape(tokens, -1).cpu(), f"qkv v {tokens}")
    # the same bits as the unfused product
    y = pool.linear(x.cuda(), w.cuda())
    assert torch.equal(torch.cat([q.reshape(tokens, -1), k.reshape(tokens, -1), v.reshape(tokens, -1)], 1), y)
