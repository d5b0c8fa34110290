"""GPU parity of the projection with the per-token work fused in
(pkv_qkv_proj_append, then pkv_decode_appended) against the fp64 oracle
composed the pages' way: q, k, v = x W^T (oracle.linear), each rounded to
bf16 (the pages' projection outputs are bf16 tensors), then oracle.decode.

Tolerances, from the arithmetic.  The tensor cores add x W^T in fp32 and the
result is rounded to bf16, so each projected element y satisfies
    |y_gpu - y| <= d(y) = 2^-8 |y| + in * 2^-23 * sum_k |x_k w_k|
(the bound test_gpu_linear checks).  Hence:
  * V (written as projected): every written element within d of the exact
    projection;
  * K: QK-norm divides k by its rms and multiplies by w, and the rotation
    mixes each element with its partner without changing the pair's length,
    so an input error d moves a normed, roped element by at most
    (d_i w_i + d_p w_p) / rms + |k_hat_i| * |d| / (sqrt(128) rms); on top of
    that comes the rounding of the written value (1 bf16 ulp);
  * untouched pool entries bit-exact; outputs within max-abs 2e-2 and
    relative-L2 5e-3 of the oracle's; error bits equal to the oracle's.
And against the unfused GPU path (pkv_qkv_proj then pkv_decode), which rounds
the same fp32 sums and runs the same norm and rotation code: the pools bit for
bit.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_qk_gb300 as pkv
import workloads as W
from _harness import MAX_ABS, REL_L2, ulp_distance_bf16

pytestmark = pytest.mark.gpu


def _projection(xb, wb):
    """Exact x W^T (fp64), its bf16 rounding, and the GPU's error bound d per element."""
    ref = oracle.linear(xb, wb)
    mag = np.abs(oracle.bf16_to_f64(xb)) @ np.abs(oracle.bf16_to_f64(wb)).T
    return ref, oracle.round_bf16(ref), 2.0 ** -8 * np.abs(ref) + xb.shape[1] * 2.0 ** -23 * mag


def _bf16_ulp(bits):
    """Size of one bf16 ulp at each value (bf16 bit patterns)."""
    e = (bits.astype(np.int32) >> 7) & 0xFF
    return np.ldexp(1.0, np.maximum(e, 1) - 127 - 7)


def _run(wl, x, w, positions=None, table=None, contiguous=False):
    cfg = wl.cfg
    H, G, D = cfg["heads"], cfg["kv_heads"], cfg["head_dim"]
    T = wl.R
    pos = wl.step_positions if positions is None else torch.as_tensor(positions, dtype=torch.int32)
    tab = wl.table if table is None else torch.as_tensor(table, dtype=torch.int32)
    xb, wb = W.bits(x), W.bits(w)
    # ---- oracle: projections rounded to bf16, then the decode step
    exact, proj, dbound = _projection(xb, wb)
    qb = proj[:, :H * D].reshape(T, H, D).copy()
    kb = proj[:, H * D:(H + G) * D].reshape(T, G, D).copy()
    vb = proj[:, (H + G) * D:].reshape(T, G, D).copy()
    Kr, Vr = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    ref, rerr = oracle.decode(Kr, Vr, qb, kb, vb, W.bits(wl.q_norm_w), W.bits(wl.k_norm_w), pos.numpy(), tab.numpy(),
                              cfg=cfg)
    v_exact = exact[:, (H + G) * D:].reshape(T, G, D)
    d_v = dbound[:, (H + G) * D:].reshape(T, G, D)
    # K: the input bound carried through QK-norm and the rotation (pairs (i, i + 64))
    k_val = oracle.bf16_to_f64(kb)
    d_k = dbound[:, H * D:(H + G) * D].reshape(T, G, D)
    wk = oracle.bf16_to_f64(W.bits(wl.k_norm_w))
    rms = np.sqrt((k_val ** 2).mean(axis=-1, keepdims=True) + cfg["eps"])
    partner = np.concatenate([np.arange(D // 2, D), np.arange(0, D // 2)])
    dw = d_k * wk
    tol_k_in = (dw + dw[..., partner]) / rms + np.abs(k_val * wk) / rms * \
        np.linalg.norm(d_k, axis=-1, keepdims=True) / (np.sqrt(D) * rms)
    # ---- GPU, fused
    dev = torch.device("cuda")
    K, V = wl.K0.to(dev), wl.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=cfg)
    xd, wd = x.to(dev), w.to(dev)
    qw, kw, posd = wl.q_norm_w.to(dev), wl.k_norm_w.to(dev), pos.to(dev)
    tabd = None if contiguous else tab.to(dev)
    out = pool.decode_layer_fused(xd, wd, qw, kw, posd, tabd, pages=tab.shape[1])
    flags = pool.check_errors()
    got_K, got_V, got = W.bits(K.cpu()), W.bits(V.cpu()), out.float().double().cpu().numpy()
    pool.close()
    # ---- GPU, unfused (the same rounding of the same fp32 sums)
    K2, V2 = wl.K0.to(dev), wl.V0.to(dev)
    pool2 = pkv.PagedKVPool(K2, V2, cfg=cfg)
    q2, k2, v2 = pool2.qkv_proj(xd, wd)
    pool2.decode(q2, k2, v2, qw, kw, posd, tabd, pages=tab.shape[1])
    assert pool2.check_errors() == rerr
    uK, uV = W.bits(K2.cpu()), W.bits(V2.cpu())
    dK, dV = uK != got_K, uV != got_V
    assert not dK.any() and not dV.any(), \
        (f"fused and unfused pools differ: K {int(dK.sum())} elements (max "
         f"{int(ulp_distance_bf16(uK[dK], got_K[dK]).max()) if dK.any() else 0} ulp, "
         f"{int(np.any(dK, axis=-1).sum())} slots), V {int(dV.sum())} elements")
    pool2.close()

    assert flags == rerr, (flags, rerr)
    K0, V0 = W.bits(wl.K0), W.bits(wl.V0)
    written = np.any(Kr != K0, axis=-1) | np.any(got_K != K0, axis=-1) | np.any(Vr != V0, axis=-1) | \
        np.any(got_V != V0, axis=-1)                                    # [G][slots]
    assert np.array_equal(got_K[~written], Kr[~written]) and np.array_equal(got_V[~written], Vr[~written])
    # slots of each (token, kv head) the oracle wrote
    S = cfg["page_size"]
    npos, ntab = pos.numpy(), tab.numpy()
    num_pages = K0.shape[1] // S
    nrows = 0
    for t in range(T):
        p = int(npos[t])
        if p < 0 or p >= cfg["max_seq"] or p >= ntab.shape[1] * S:
            continue
        if np.any((ntab[t, :p // S + 1] < 0) | (ntab[t, :p // S + 1] >= num_pages)):
            continue
        slot = int(ntab[t, p // S]) * S + p % S
        gv = oracle.bf16_to_f64(got_V[:, slot])                          # [G][D]
        assert np.all(np.abs(gv - v_exact[t]) <= d_v[t]), (t, float((np.abs(gv - v_exact[t]) / d_v[t]).max()))
        gk, rk = oracle.bf16_to_f64(got_K[:, slot]), oracle.bf16_to_f64(Kr[:, slot])
        tol = 1.01 * tol_k_in[t] + _bf16_ulp(Kr[:, slot]) + _bf16_ulp(got_K[:, slot])
        assert np.all(np.abs(gk - rk) <= tol), (t, float((np.abs(gk - rk) / tol).max()))
        nrows += 1
    max_abs = float(np.abs(got - ref).max())
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    print(f"[parity] fused {wl.name}: max-abs {max_abs:.3e} rel-L2 {rel:.3e}; written K/V of {nrows} rows "
          f"within the projection bound")
    assert max_abs <= MAX_ABS and rel <= REL_L2
    return got, flags


@pytest.mark.parametrize("rows,hidden,lo,hi", [
    (64, 4096, 512, 4096),   # the 64-row decode batch at Qwen3-8B's hidden size (split over a cluster)
    (7, 512, 1, 700),        # a ragged token tile
    (200, 512, 60, 300),     # a 256-token tile, no split
])
def test_fused_projection_decode(rows, hidden, lo, hi):
    wl = W.make_decode(f"fused {rows} rows", (rows, lo, hi), seed=50 + rows, table_pages=-(-hi // 64))
    x, w = W.make_linear(rows, hidden, 6144, seed=60 + rows)
    _run(wl, x, w)


def test_fused_projection_skips_rows_and_contiguous_rows():
    wl = W.make_decode("fused skips", [100, 70, 5, 2000, 64], seed=71, table_pages=32)
    x, w = W.make_linear(wl.R, 512, 6144, seed=72)
    pos = wl.step_positions.clone()
    table = wl.table.clone()
    pos[0] = -1                      # no step
    pos[1] = 40960                   # beyond max_seq
    table[2, 0] = wl.num_pages + 7   # not a pool page
    got, flags = _run(wl, x, w, positions=pos, table=table)
    assert flags == (pkv.PKV_DEVERR_POSITION | pkv.PKV_DEVERR_PAGE)
    for b in (0, 1, 2):
        assert not np.abs(got[b]).sum()
    rows = W.make_decode("fused contiguous rows", (16, 1, 640), seed=73, table_pages=10, contiguous=True)
    x2, w2 = W.make_linear(rows.R, 512, 6144, seed=74)
    _run(rows, x2, w2, contiguous=True)
