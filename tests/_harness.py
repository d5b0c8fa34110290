"""Shared helpers for the GPU parity tests: run a workload through the C ABI
and through the fp64 oracle, and compare them element by element."""
import numpy as np
import torch

import oracle
import paged_kv_gqa_qk_gb300 as pkv
import workloads as W

# Output tolerances against the oracle's fp64 values (max-abs and relative L2).
MAX_ABS = 2e-2
REL_L2 = 5e-3


def run_gpu(wl: W.Workload, ctas: int = 0, explicit_slots=None, table=None, step_positions=None,
            positions=None, repeat: int = 1):
    dev = torch.device("cuda")
    K, V = wl.K0.to(dev), wl.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
    if ctas:
        pkv.pkv_set_ctas(pool.handle, ctas)
    q, k, v, qw, kw = (t.to(dev) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w))
    tab = (wl.table if table is None else torch.as_tensor(table)).to(dev)
    pages = int(tab.shape[1])
    if wl.contiguous and table is None:
        tab = None   # the library's own contiguous-row layout
    sp = (wl.step_positions if step_positions is None else torch.as_tensor(step_positions)).to(dev)
    for _ in range(repeat):
        if wl.kind == "decode":
            out = pool.decode(q, k, v, qw, kw, sp, tab, pages=pages)
        else:
            pos = (wl.positions if positions is None else torch.as_tensor(positions)).to(dev)
            slots = None if explicit_slots is None else torch.as_tensor(explicit_slots, dtype=torch.int32).to(dev)
            if wl.kind == "step":
                out = pool.step(q, k, v, qw, kw, pos, wl.prow.to(dev), slots, sp, tab, pages=pages)
            else:
                P = wl.P
                out = pool.prefill(q[:P], k[:P], v[:P], qw, kw, pos, wl.prow.to(dev), slots, tab,
                                   rows=wl.R, pages=pages)
    flags = pool.check_errors()
    res = (out.cpu(), K.cpu(), V.cpu(), flags)
    pool.close()
    return res


def run_oracle(wl: W.Workload, sel=None, table=None, step_positions=None, positions=None):
    K, V = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    args = [W.bits(t) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w)]
    tab = (wl.table if table is None else torch.as_tensor(table)).numpy()
    sp = (wl.step_positions if step_positions is None else torch.as_tensor(step_positions)).numpy()
    if wl.kind == "decode":
        out, err = oracle.decode(K, V, *args, sp, tab, cfg=wl.cfg, sel=sel)
    else:
        pos = (wl.positions if positions is None else torch.as_tensor(positions)).numpy()
        out, err = oracle.step(K, V, *args, pos, wl.prow.numpy(), None, sp, tab, cfg=wl.cfg, sel=sel)
        if wl.kind == "prefill":   # the table rows take no step: prompt outputs only
            out = out[:wl.P]
    return out, K, V, err


def ulp_distance_bf16(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between two arrays of bf16 bit patterns (uint16)."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - x, x)   # monotone map of bf16 bits to integers
    return np.abs(ordered(a) - ordered(b))


def compare(wl, gpu, ref, sel=None, label=""):
    """Assert the GPU result matches the oracle; returns (max_abs, rel_l2)."""
    out, K, V, flags = gpu
    rout, rK, rV, rerr = ref
    assert flags == rerr, f"{label}: device error bits {flags} != oracle {rerr}"
    Kb, Vb = W.bits(K), W.bits(V)
    K0 = W.bits(wl.K0)
    # V: bit-exact everywhere (written slots and untouched entries)
    assert np.array_equal(Vb, rV), f"{label}: V pool differs from the oracle"
    # K: untouched entries bit-exact, written entries within 1 bf16 ulp
    written = np.any(rK != K0, axis=-1) | np.any(Kb != K0, axis=-1)
    assert np.array_equal(Kb[~written], rK[~written]), f"{label}: untouched K entries changed"
    if written.any():
        d = ulp_distance_bf16(Kb[written], rK[written])
        if d.max() > 1:
            i = np.unravel_index(np.argmax(d), d.shape)
            gv = oracle.bf16_to_f64(Kb[written][i])
            rv = oracle.bf16_to_f64(rK[written][i])
            raise AssertionError(f"{label}: written K off by {d.max()} ulp ({(d > 1).sum()} elements > 1 ulp); "
                                 f"worst: gpu {gv!r} oracle {rv!r}, row max |k| "
                                 f"{np.abs(oracle.bf16_to_f64(rK[written][i[0]])).max():.3f}")
    got = out.float().double().numpy()
    if sel is not None:
        got, rout = got[sel], rout[sel]
    max_abs = float(np.abs(got - rout).max()) if got.size else 0.0
    nrm = float(np.linalg.norm(rout))
    rel = float(np.linalg.norm(got - rout) / nrm) if nrm > 0 else float(np.linalg.norm(got))
    print(f"[parity] {label}: max-abs {max_abs:.3e} rel-L2 {rel:.3e}")
    assert max_abs <= MAX_ABS, f"{label}: max-abs {max_abs:.3e} > {MAX_ABS}"
    assert rel <= REL_L2, f"{label}: rel-L2 {rel:.3e} > {REL_L2}"
    return max_abs, rel


def step_sm_split(prompt_lens, step_positions, kv_heads: int, sms: int, page_size: int = 64):
    """The kernels' split of a step's SMs (prompt_sms and prompt_tile_cost in
    csrc/pkv_internal.h): (SMs the prompt attention holds, the rows' attention
    CTAs resident from the start at two a SM).  prompt_lens: attended lengths
    of the prompt tokens (0 skipped); costs in 1/25 us of one SM."""
    G, S = kv_heads, page_size
    pc, pu = 0, 0
    for t0 in range(0, len(prompt_lens), 64):
        m = max(prompt_lens[t0:t0 + 64])
        if m > 0:
            pc += G * (160 + 28 * ((m + S - 1) // S))
            pu += G
    rc = 13 * G * sum(p // S + 1 for p in step_positions if p >= 0)
    n = sms
    if pc > 0 and rc > 0:
        n = (pc * sms + (pc + rc) // 2) // (pc + rc)
        n = max(n, min(pu, sms // 4), 1)
        n = sms if n > sms - 8 else n
    pgrid = min(sms, (len(prompt_lens) + 63) // 64 * G)
    kept = min(n, pgrid)
    return kept, (2 * (sms - kept) if kept < sms else 2 * sms)
