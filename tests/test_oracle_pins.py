"""Pins for the fp64 oracle: each check fixes the oracle against something
other than itself -- a library routine (torch's RMSNorm and scaled-dot-product
attention in fp64, torch's float32->bf16 conversion, numpy complex
arithmetic), a closed form, an invariant, or brute force on tiny inputs.

CPU only (not marked gpu).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

CFG = dict(oracle.DEFAULT_CONFIG)
D = CFG["head_dim"]


def rand_bits(rng, shape, scale=1.0):
    x = torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * scale).to(torch.bfloat16)
    return W.bits(x)


# ------------------------------------------------------------------ bf16 rounding

def test_round_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x32 = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                          (rng.standard_normal(2000) * 1e-38).astype(np.float32),   # subnormal range
                          (rng.standard_normal(2000) * 1e30).astype(np.float32)])
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(x32.astype(np.float64))
    assert np.array_equal(got, ref)


def test_round_bf16_closed_forms():
    r = lambda x: int(oracle.round_bf16(np.array([x]))[0])
    assert r(1.0) == 0x3F80
    assert r(1.0 + 2.0 ** -8) == 0x3F80           # tie -> even (down)
    assert r(1.0 + 3 * 2.0 ** -8) == 0x3F82       # tie -> even (up)
    # just above a tie in double: one rounding goes up, a detour through
    # binary32 would land exactly on the tie and go down
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert r(-2.0) == 0xC000
    assert r(2.0 ** -133) == 0x0001               # smallest subnormal
    assert r(2.0 ** -134) == 0x0000               # tie -> even (zero)
    assert r(3 * 2.0 ** -134) == 0x0002           # 1.5 quanta -> tie -> even
    assert r(3.4e38) == 0x7F80                    # beyond (max + half ulp) -> inf
    assert r(3.389e38) == 0x7F7F                  # max finite
    assert r(float("inf")) == 0x7F80


# ------------------------------------------------------------------ a2 QK-norm

def test_qk_norm_matches_torch_rms_norm():
    rng = np.random.default_rng(1)
    for _ in range(20):
        x = rand_bits(rng, D, scale=rng.uniform(0.01, 10))
        w = W.bits((torch.rand(D, dtype=torch.float32) + 0.5).to(torch.bfloat16))
        got = oracle.qk_norm(x, w)
        xt = torch.from_numpy(oracle.bf16_to_f64(x))
        wt = torch.from_numpy(oracle.bf16_to_f64(w))
        ref = torch.nn.functional.rms_norm(xt, (D,), wt, eps=1e-6).numpy()
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


def test_qk_norm_unit_rms_and_constant_vector():
    rng = np.random.default_rng(2)
    ones = W.bits(torch.ones(D, dtype=torch.bfloat16))
    x = rand_bits(rng, D)
    y = oracle.qk_norm(x, ones)
    ms = np.mean(oracle.bf16_to_f64(x) ** 2)
    assert math.isclose(np.sqrt(np.mean(y ** 2)), math.sqrt(ms / (ms + 1e-6)), rel_tol=1e-13)
    # constant vector c*1 with weight w: c / sqrt(c^2 + eps) * w
    c = 0.015625  # exactly representable; eps matters at this scale
    xc = W.bits(torch.full((D,), c, dtype=torch.bfloat16))
    w = W.bits((torch.rand(D, dtype=torch.float32) + 0.5).to(torch.bfloat16))
    yc = oracle.qk_norm(xc, w)
    np.testing.assert_allclose(yc, c / math.sqrt(c * c + 1e-6) * oracle.bf16_to_f64(w), rtol=1e-14)
    # scale invariance (up to eps)
    x2 = W.bits(torch.from_numpy(oracle.bf16_to_f64(x) * 4.0).to(torch.bfloat16))
    np.testing.assert_allclose(oracle.qk_norm(x2, ones), y, rtol=1e-6)


# ------------------------------------------------------------------ a3 RoPE

def test_rope_position_zero_is_identity():
    y = np.random.default_rng(3).standard_normal(D)
    assert np.array_equal(oracle.rope(y, 0), y)


def test_rope_equals_complex_rotation():
    """Pair (i, i+64) as the complex number y_i + j*y_{i+64}, rotated by pos * theta^(-2i/128)."""
    rng = np.random.default_rng(4)
    for pos in [1, 7, 63, 64, 1000, 40959]:
        y = rng.standard_normal(D)
        got = oracle.rope(y, pos)
        i = np.arange(D // 2)
        z = (y[:D // 2] + 1j * y[D // 2:]) * np.exp(1j * pos * np.power(1.0e6, -2.0 * i / D))
        np.testing.assert_allclose(got[:D // 2], z.real, rtol=0, atol=1e-11)
        np.testing.assert_allclose(got[D // 2:], z.imag, rtol=0, atol=1e-11)


@pytest.mark.parametrize("rot", [32, 64, 96])
def test_partial_rope_rotates_only_the_first_dims(rot):
    """rotary_dim R < head_dim (the gated variant's partial RoPE): dims from R on
    are left exactly as they are; the first R are the complex rotation of the
    pairs (i, i + R/2) by pos * theta^(-2i/R)."""
    rng = np.random.default_rng(rot)
    cfg = dict(CFG, rotary_dim=rot)
    for pos in [0, 1, 77, 40959]:
        y = rng.standard_normal(D)
        out = oracle.rope(y, pos, cfg)
        np.testing.assert_array_equal(out[rot:], y[rot:])
        i = np.arange(rot // 2)
        z = (y[:rot // 2] + 1j * y[rot // 2:rot]) * np.exp(1j * pos * np.power(1.0e6, -2.0 * i / rot))
        # angles up to ~4e4 rad: one ulp of the frequency moves them by ~1e-11
        np.testing.assert_allclose(out[:rot], np.concatenate([z.real, z.imag]), rtol=1e-10, atol=1e-10)
    # rotary_dim = head_dim is the full rotation
    y = rng.standard_normal(D)
    np.testing.assert_array_equal(oracle.rope(y, 123, dict(CFG, rotary_dim=D)), oracle.rope(y, 123, CFG))


def test_output_gate_closed_forms():
    """out * sigmoid(gate): a zero gate halves, a large gate keeps, a very negative gate zeroes."""
    out = np.array([[1.0, -3.0, 2.5, 0.0]])
    gate = W.bits(torch.tensor([[0.0, 30.0, -30.0, 5.0]], dtype=torch.bfloat16))
    got = oracle.output_gate(out, gate)
    assert got[0, 0] == 0.5
    assert abs(got[0, 1] + 3.0) < 1e-12 and abs(got[0, 2]) < 1e-12 and got[0, 3] == 0.0
    g = float(oracle.bf16_to_f64(gate)[0, 1])
    assert got[0, 1] == -3.0 / (1.0 + math.exp(-g))


def test_rope_closed_form_and_invariants():
    rng = np.random.default_rng(5)
    y = rng.standard_normal(D)
    # position 1, pair 0: angle is exactly 1 radian
    r1 = oracle.rope(y, 1)
    assert math.isclose(r1[0], y[0] * math.cos(1.0) - y[64] * math.sin(1.0), rel_tol=1e-15, abs_tol=1e-15)
    assert math.isclose(r1[64], y[64] * math.cos(1.0) + y[0] * math.sin(1.0), rel_tol=1e-15, abs_tol=1e-15)
    # every pair keeps its norm
    r = oracle.rope(y, 12345)
    np.testing.assert_allclose(r[:64] ** 2 + r[64:] ** 2, y[:64] ** 2 + y[64:] ** 2, rtol=1e-12)
    # relative position: <R(m) a, R(n) b> depends only on m - n
    a, b = rng.standard_normal(D), rng.standard_normal(D)
    for m, n, s in [(10, 3, 500), (4000, 4100, 30000)]:
        d1 = oracle.rope(a, m) @ oracle.rope(b, n)
        d2 = oracle.rope(a, m + s) @ oracle.rope(b, n + s)
        assert math.isclose(d1, d2, rel_tol=1e-9, abs_tol=1e-9)


# ------------------------------------------------------------------ a1/a5 paged attention

def scatter_contiguous(rng, K_log, V_log, num_pages, S):
    """Put a row's logical K/V [G][L][D] into a fresh pool through a random page map."""
    G, L, Dd = K_log.shape
    npg = -(-L // S)
    pages = rng.permutation(num_pages)[:npg]
    Kp = rand_bits(rng, (G, num_pages * S, Dd))
    Vp = rand_bits(rng, (G, num_pages * S, Dd))
    for j, pg in enumerate(pages):
        n = min(S, L - j * S)
        Kp[:, pg * S:pg * S + n] = K_log[:, j * S:j * S + n]
        Vp[:, pg * S:pg * S + n] = V_log[:, j * S:j * S + n]
    return Kp, Vp, pages.astype(np.int32)


def sdpa_f64(q, K, V):
    """torch scaled_dot_product_attention in float64: q [H][D], K/V [G][L][D] (GQA by repeat)."""
    H, G = q.shape[0], K.shape[0]
    Kt = torch.from_numpy(K).repeat_interleave(H // G, dim=0)
    Vt = torch.from_numpy(V).repeat_interleave(H // G, dim=0)
    qt = torch.from_numpy(q)[:, None, :]
    return torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt).squeeze(1).numpy()


def test_paged_attention_equals_contiguous_sdpa():
    rng = np.random.default_rng(6)
    G, S = CFG["kv_heads"], CFG["page_size"]
    for L in [1, 63, 64, 65, 200, 1000]:
        K_log, V_log = rand_bits(rng, (G, L, D)), rand_bits(rng, (G, L, D))
        Kp, Vp, pages = scatter_contiguous(rng, K_log, V_log, num_pages=-(-L // S) + 5, S=S)
        table = np.zeros((1, len(pages) + 2), dtype=np.int32)
        table[0, :len(pages)] = pages
        qh = rng.standard_normal((CFG["heads"], D))
        got = np.stack([oracle.attend(Kp, Vp, table, 0, L - 1, h // 4, qh[h]) for h in range(CFG["heads"])])
        ref = sdpa_f64(qh, oracle.bf16_to_f64(K_log), oracle.bf16_to_f64(V_log))
        np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(7)
    G, S = CFG["kv_heads"], CFG["page_size"]
    Kp, Vp = rand_bits(rng, (G, 4 * S, D)), rand_bits(rng, (G, 4 * S, D))
    table = np.array([[2, 0, 3, 1]], dtype=np.int32)
    qh = rng.standard_normal(D)
    # a single key returns its value exactly
    out = oracle.attend(Kp, Vp, table, 0, 0, 3, qh)
    np.testing.assert_array_equal(out, oracle.bf16_to_f64(Vp[3, 2 * S]))
    # all keys equal -> the mean of the values
    K2 = Kp.copy()
    K2[:, :, :] = Kp[:, :1, :]
    out = oracle.attend(K2, Vp, table, 0, 99, 1, qh)
    slots = [table[0, s // S] * S + s % S for s in range(100)]
    np.testing.assert_allclose(out, oracle.bf16_to_f64(Vp[1, slots]).mean(axis=0), rtol=1e-12, atol=1e-14)
    # one dominant key -> its value
    K3 = W.bits(torch.zeros((G, 4 * S, D), dtype=torch.bfloat16))
    s_dom = 77
    slot_dom = table[0, s_dom // S] * S + s_dom % S
    K3[2, slot_dom] = W.bits(torch.full((D,), 8.0, dtype=torch.bfloat16))
    out = oracle.attend(K3, Vp, table, 0, 150, 2, np.full(D, 8.0))
    np.testing.assert_allclose(out, oracle.bf16_to_f64(Vp[2, slot_dom]), rtol=1e-12, atol=1e-12)


def test_split_ranges_reassociate_exactly():
    rng = np.random.default_rng(8)
    G, S = CFG["kv_heads"], CFG["page_size"]
    Kp, Vp = rand_bits(rng, (G, 40 * S, D)), rand_bits(rng, (G, 40 * S, D))
    table = rng.permutation(40).astype(np.int32)[None, :]
    qh = rng.standard_normal(D) * 3
    pos = 40 * S - 17
    ref = oracle.attend(Kp, Vp, table, 0, pos, 5, qh)
    for _ in range(10):
        n = int(rng.integers(1, 12))
        cuts = np.sort(rng.choice(np.arange(1, pos + 1), size=n - 1, replace=False)) if n > 1 else []
        split = np.array([0, *cuts, pos + 1], dtype=np.int32)
        got = oracle.attend_split(Kp, Vp, table, 0, pos, 5, qh, split)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_page_permutation_invariance():
    wl = W.make_decode("perm", [100, 300, 64, 1], seed=11, cfg=None, table_pages=6)
    args = [W.bits(t) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w)]
    out1, _ = oracle.decode(W.bits(wl.K0).copy(), W.bits(wl.V0).copy(), *args, wl.step_positions.numpy(),
                            wl.table.numpy())
    # move every pool page to a new place and rewrite the table accordingly
    S = CFG["page_size"]
    rng = np.random.default_rng(12)
    perm = rng.permutation(wl.num_pages)             # new page of old page i is perm[i]
    K0, V0 = W.bits(wl.K0), W.bits(wl.V0)
    K1, V1 = np.empty_like(K0), np.empty_like(V0)
    for i in range(wl.num_pages):
        K1[:, perm[i] * S:(perm[i] + 1) * S] = K0[:, i * S:(i + 1) * S]
        V1[:, perm[i] * S:(perm[i] + 1) * S] = V0[:, i * S:(i + 1) * S]
    t1 = perm[wl.table.numpy()].astype(np.int32)
    out2, _ = oracle.decode(K1, V1, *args, wl.step_positions.numpy(), t1)
    np.testing.assert_array_equal(out1, out2)


# ------------------------------------------------------------------ full decode step, independent route

def complex_rope(y, pos):
    i = np.arange(D // 2)
    z = (y[:D // 2] + 1j * y[D // 2:]) * np.exp(1j * pos * np.power(1.0e6, -2.0 * i / D))
    return np.concatenate([z.real, z.imag])


def torch_norm(x_bits, w_bits):
    return torch.nn.functional.rms_norm(torch.from_numpy(oracle.bf16_to_f64(x_bits)), (D,),
                                        torch.from_numpy(oracle.bf16_to_f64(w_bits)), eps=1e-6).numpy()


def test_decode_step_against_library_route():
    """QK-norm (torch rms_norm) -> RoPE (complex rotation) -> write -> GQA (torch SDPA), all fp64."""
    wl = W.config1()
    S, G, H = CFG["page_size"], CFG["kv_heads"], CFG["heads"]
    q, k, v, qw, kw = (W.bits(t) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w))
    pos = wl.step_positions.numpy()
    table = wl.table.numpy()
    K, V = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    out, err = oracle.decode(K, V, q, k, v, qw, kw, pos, table)
    assert err == 0
    K0, V0 = W.bits(wl.K0), W.bits(wl.V0)
    written = np.zeros(K0.shape[:2], dtype=bool)
    for b in range(wl.R):
        p = int(pos[b])
        slot = table[b, p // S] * S + p % S
        for g in range(G):
            khat = complex_rope(torch_norm(k[b, g], kw), p)
            np.testing.assert_array_equal(K[g, slot], oracle.round_bf16(khat))
            np.testing.assert_array_equal(V[g, slot], v[b, g])
            written[g, slot] = True
        # contiguous logical cache of this row after the write, then SDPA
        slots = [table[b, s // S] * S + s % S for s in range(p + 1)]
        Kc, Vc = oracle.bf16_to_f64(K[:, slots]), oracle.bf16_to_f64(V[:, slots])
        qh = np.stack([complex_rope(torch_norm(q[b, h], qw), p) for h in range(H)])
        np.testing.assert_allclose(out[b], sdpa_f64(qh, Kc, Vc), rtol=1e-10, atol=1e-12)
    # untouched entries are bit-exact
    assert np.array_equal(K[~written], K0[~written]) and np.array_equal(V[~written], V0[~written])


def test_brute_force_tiny_shapes():
    """head_dim 4, 2 query heads over 1 kv head, pages of 2 positions, 3 pages: pure-Python loops."""
    cfg = dict(heads=2, kv_heads=1, head_dim=4, page_size=2, max_seq=64, rope_theta=10.0, eps=1e-6)
    rng = np.random.default_rng(13)
    K = rand_bits(rng, (1, 6, 4))
    V = rand_bits(rng, (1, 6, 4))
    q, k, v = rand_bits(rng, (1, 2, 4)), rand_bits(rng, (1, 1, 4)), rand_bits(rng, (1, 1, 4))
    qw = W.bits(torch.tensor([1.0, 0.5, 1.5, 1.25], dtype=torch.bfloat16))
    kw = W.bits(torch.tensor([0.75, 1.0, 1.0, 0.5], dtype=torch.bfloat16))
    table = np.array([[2, 0, 1]], dtype=np.int32)
    pos = 4
    Kx, Vx = K.copy(), V.copy()
    out, err = oracle.decode(Kx, Vx, q, k, v, qw, kw, np.array([pos], np.int32), table, cfg=cfg)
    assert err == 0
    f = oracle.bf16_to_f64

    def norm_rope(xb, wb):
        x, w = f(xb), f(wb)
        r = math.sqrt(sum(t * t for t in x) / 4 + 1e-6)
        y = [x[i] / r * w[i] for i in range(4)]
        res = list(y)
        for i in range(2):
            a = pos * 10.0 ** (-2 * i / 4)
            res[i] = y[i] * math.cos(a) - y[i + 2] * math.sin(a)
            res[i + 2] = y[i + 2] * math.cos(a) + y[i] * math.sin(a)
        return res

    slot_new = 1 * 2 + 0       # position 4 -> page table[0][2] = 1, offset 0
    kh = norm_rope(k[0, 0], kw)
    assert list(Kx[0, slot_new]) == list(oracle.round_bf16(np.array(kh)))
    keys = []
    for s in range(pos + 1):
        sl = table[0, s // 2] * 2 + s % 2
        keys.append((f(Kx[0, sl]), f(Vx[0, sl])))
    for h in range(2):
        qh = norm_rope(q[0, h], qw)
        z = [sum(qh[d] * kk[d] for d in range(4)) / 2.0 for kk, _ in keys]
        mz = max(z)
        e = [math.exp(t - mz) for t in z]
        o = [sum(e[s] * keys[s][1][d] for s in range(len(keys))) / sum(e) for d in range(4)]
        np.testing.assert_allclose(out[0, h], o, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------ contiguous rows: prefill_packed, decode_rows

def test_prefill_over_contiguous_rows_equals_packed_attention():
    """Prompts that each fill their own row from position 0, over the
    contiguous-row layout (identity table), give prefill_packed's result: each
    token attends to its own prompt's tokens up to itself (mask segments equal
    and positions[j] <= positions[i]), computed here from the pass's own
    normed and roped keys with torch SDPA; and token p lands at slot
    prow[p] * pages * page_size + positions[p]."""
    wl = W.make_prefill("packed", [3, 70, 1, 64], [0, 0, 0, 0], seed=41, table_pages=2, contiguous=True)
    assert wl.kind == "prefill" and wl.contiguous
    S, G, H = CFG["page_size"], CFG["kv_heads"], CFG["heads"]
    q, k, v, qw, kw = (W.bits(t) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w))
    pos, prow = wl.positions.numpy(), wl.prow.numpy()
    K, V = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    out, err = oracle.step(K, V, q, k, v, qw, kw, pos, prow, None, wl.step_positions.numpy(), wl.table.numpy())
    assert err == 0
    P = wl.P
    khat = np.stack([np.stack([oracle.round_bf16(complex_rope(torch_norm(k[t, g], kw), int(pos[t])))
                               for g in range(G)]) for t in range(P)])        # [P][G][D] bf16 bits
    for t in range(P):
        slot = int(prow[t]) * wl.pages * S + int(pos[t])
        for g in range(G):
            np.testing.assert_array_equal(K[g, slot], khat[t, g])
            np.testing.assert_array_equal(V[g, slot], v[t, g])
    for i in range(P):
        own = [j for j in range(P) if prow[j] == prow[i] and pos[j] <= pos[i]]
        qh = np.stack([complex_rope(torch_norm(q[i, h], qw), int(pos[i])) for h in range(H)])
        Kc = oracle.bf16_to_f64(khat[own].transpose(1, 0, 2))
        Vc = oracle.bf16_to_f64(v[own].transpose(1, 0, 2))
        np.testing.assert_allclose(out[i], sdpa_f64(qh, Kc, Vc), rtol=1e-10, atol=1e-12)
    assert not out[P:].any()   # the table rows take no step


# ------------------------------------------------------------------ projections (linear, no bias)

def test_linear_brute_force_and_special_cases():
    """y[t][o] = sum_k x[t][k] w[o][k]: pure-Python sums on tiny shapes, the
    identity weight returns x, a one-hot input row returns a column of w, and
    the map is linear in x."""
    rng = np.random.default_rng(11)
    x, w = rand_bits(rng, (3, 7)), rand_bits(rng, (5, 7))
    y = oracle.linear(x, w)
    xf, wf = oracle.bf16_to_f64(x), oracle.bf16_to_f64(w)
    for t in range(3):
        for o in range(5):
            ref = 0.0
            for k in range(7):
                ref += float(xf[t, k]) * float(wf[o, k])
            assert abs(y[t, o] - ref) <= 1e-12 * max(1.0, abs(ref))
    eye = W.bits(torch.eye(7, dtype=torch.bfloat16))
    np.testing.assert_array_equal(oracle.linear(x, eye), xf)
    onehot = np.zeros((1, 7), np.uint16)
    onehot[0, 4] = W.bits(torch.ones(1, dtype=torch.bfloat16))[0]
    np.testing.assert_array_equal(oracle.linear(onehot, w)[0], wf[:, 4])
    # linear in x: two inputs whose exact sum is again a bf16 value (x and x itself)
    np.testing.assert_array_equal(oracle.linear(W.bits(torch.from_numpy(2 * xf).to(torch.bfloat16)), w), 2 * y)


# ------------------------------------------------------------------ a7 prefill chunk == sequential decode

def test_step_prefill_equals_sequential_decode():
    cfg = dict(CFG)
    wl = W.make_step("tiny step", prompt_lengths=[70, 5], prompt_starts=[60, 0], decode_lengths=[90, 3],
                     seed=14, table_pages=3)
    args = [W.bits(t) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w)]
    K, V = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    pos, prow, sp, table = (wl.positions.numpy(), wl.prow.numpy(), wl.step_positions.numpy(), wl.table.numpy())
    out, err = oracle.step(K, V, *args, pos, prow, None, sp, table, cfg=cfg)
    assert err == 0
    # explicit slots give the same result
    slots = oracle.page_slots(table, prow, pos)
    Ke, Ve = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    out_e, _ = oracle.step(Ke, Ve, *args, pos, prow, slots, sp, table, cfg=cfg)
    np.testing.assert_array_equal(out, out_e)
    assert np.array_equal(K, Ke) and np.array_equal(V, Ve)
    # the same tokens one at a time as decode steps: token p is a decode row of
    # table row prow[p] at positions[p]; a one-row table holds that row.
    q, k, v, qw, kw = args
    Ks, Vs = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    P, R = wl.P, wl.R
    seq = np.zeros_like(out)
    for t in range(P + R):
        if t < P:
            r, p = int(prow[t]), int(pos[t])
        else:
            r, p = t - P, int(sp[t - P])
            if p < 0:
                continue
        o, e = oracle.decode(Ks, Vs, q[t:t + 1], k[t:t + 1], v[t:t + 1], qw, kw, np.array([p], np.int32),
                             table[r:r + 1], cfg=cfg)
        assert e == 0
        seq[t] = o[0]
    # prompt tokens see their own chunk's earlier keys either way; decode rows
    # see the whole chunk in both (their rows hold no prompt tokens)
    np.testing.assert_allclose(out, seq, rtol=1e-12, atol=1e-14)
    assert np.array_equal(K, Ks) and np.array_equal(V, Vs)
    # rows taking no step output zeros
    assert not out[P + 2:].any()


# ------------------------------------------------------------------ skipped tokens

def test_invalid_tokens_are_skipped_with_error_bits():
    wl = W.make_decode("err", [10, 70, 5], seed=15, table_pages=2)
    args = [W.bits(t) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w)]
    K, V = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    table = wl.table.numpy().copy()
    pos = wl.step_positions.numpy().copy()
    pos[0] = 40960                     # beyond max_seq (and the table)
    table[2, 0] = wl.num_pages + 3     # not a pool page
    out, err = oracle.decode(K, V, *args, pos, table)
    assert err == (oracle.ERR_POSITION | oracle.ERR_PAGE)
    assert not out[0].any() and not out[2].any() and out[1].any()
    # only row 1's slot changed
    S = CFG["page_size"]
    slot1 = table[1, 69 // S] * S + 69 % S
    mask = np.ones(K.shape[:2], dtype=bool)
    mask[:, slot1] = False
    assert np.array_equal(K[mask], W.bits(wl.K0)[mask]) and np.array_equal(V[mask], W.bits(wl.V0)[mask])
    # a row that takes no step: no write, zero output, no error
    K2, V2 = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    pos2 = wl.step_positions.numpy().copy()
    pos2[1] = -1
    out2, err2 = oracle.decode(K2, V2, *args, pos2, wl.table.numpy())
    assert err2 == 0 and not out2[1].any()


def test_explicit_slot_outside_the_pool_is_skipped():
    """The slot-check branch of the step: a prompt token whose explicit slot
    lies outside the pool (negative, or num_slots and beyond) is skipped with
    ERR_SLOT -- no write, zero output -- and nothing else changes.  The bad
    tokens are the last of their prompts, so no other token reads the slots
    they would have written: every other output, and the whole pool except
    those two slots, must equal the call with the correct slots."""
    cfg = dict(CFG)
    wl = W.make_step("slot errors", prompt_lengths=[70, 5], prompt_starts=[60, 0], decode_lengths=[90, 3],
                     seed=16, table_pages=3)
    args = [W.bits(t) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w)]
    pos, prow, sp, table = (wl.positions.numpy(), wl.prow.numpy(), wl.step_positions.numpy(), wl.table.numpy())
    slots = oracle.page_slots(table, prow, pos)
    K, V = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    ref, err = oracle.step(K, V, *args, pos, prow, slots, sp, table, cfg=cfg)
    assert err == 0
    num_slots = K.shape[1]
    bad = slots.copy()
    last0, last1 = 69, 74                   # last token of each prompt
    bad[last0] = num_slots                  # one past the pool
    bad[last1] = -3                         # negative
    Kb, Vb = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    out, errb = oracle.step(Kb, Vb, *args, pos, prow, bad, sp, table, cfg=cfg)
    assert errb == oracle.ERR_SLOT
    assert not out[last0].any() and not out[last1].any()
    keep = np.ones(out.shape[0], dtype=bool)
    keep[[last0, last1]] = False
    np.testing.assert_array_equal(out[keep], ref[keep])
    # the pool: the two skipped tokens' slots keep their old contents, all else as the good call left it
    K0, V0 = W.bits(wl.K0), W.bits(wl.V0)
    for s in (slots[last0], slots[last1]):
        assert np.array_equal(Kb[:, s], K0[:, s]) and np.array_equal(Vb[:, s], V0[:, s])
        Kb[:, s], Vb[:, s] = K[:, s], V[:, s]
    assert np.array_equal(Kb, K) and np.array_equal(Vb, V)
