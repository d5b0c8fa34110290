"""GPU parity of the prompt-only entry (pkv_prefill, the pages' prefill_paged)
and of the contiguous-row layout (a NULL table: decode_rows, prefill_packed,
step_packed) against the fp64 oracle, with the same bar as the other parity
tests.  The oracle sees the layout as its identity page table."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_qk_gb300 as pkv
import workloads as W
from _harness import compare, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ prefill_paged

def test_prefill_chunks_over_prefilled_pages():
    """Four prompts, ragged, three of them continuing a row at a position
    inside a page (chunked prefill over keys the row already holds)."""
    wl = W.make_prefill("prefill chunks", [70, 5, 130, 300], [60, 0, 500, 64], seed=31, table_pages=14)
    ref = run_oracle(wl)
    assert ref[3] == 0
    compare(wl, run_gpu(wl), ref, label="prefill derived slots")
    slots = oracle.page_slots(wl.table.numpy(), wl.prow.numpy(), wl.positions.numpy())
    compare(wl, run_gpu(wl, explicit_slots=slots), ref, label="prefill explicit slots")
    compare(wl, run_gpu(wl, repeat=2), ref, label="prefill x2")


def test_prefill_shared_prefix_pages():
    """Two prompts whose rows list the same first pages (a shared prefix that
    neither writes) and continue past it on pages of their own."""
    wl = W.make_prefill("prefill shared prefix", [100, 33], [128, 128], seed=32, table_pages=5)
    table = wl.table.clone()
    table[1, :2] = table[0, :2]          # row 1 reads row 0's two prefix pages
    ref = run_oracle(wl, table=table)
    assert ref[3] == 0
    compare(wl, run_gpu(wl, table=table), ref, label="prefill shared prefix")


def test_prefill_2048_tokens():
    """The step mix's prompt side alone: 4 prompts, P = 2048 (each >= 64),
    continuing at U[0, 4096]; every token compared."""
    wl = W.prefill_mix()
    compare(wl, run_gpu(wl), run_oracle(wl), label="prefill P=2048 (all tokens)")


def _tile_items(lengths) -> int:
    """(64-token tile, prompt) pairs of prompts packed end to end: the prompt
    attention's work items."""
    items, t0 = 0, 0
    ends = np.cumsum(lengths)
    starts = ends - np.asarray(lengths)
    for t0 in range(0, int(ends[-1]), 64):
        items += int(((starts < t0 + 64) & (ends > t0)).sum())
    return items


@pytest.mark.parametrize("prompt_len,prompts,sorted_items", [(40, 150, True), (2, 2400, False)])
def test_prefill_many_short_prompts(prompt_len, prompts, sorted_items):
    """Many short prompts, several to a 64-token tile.  Up to 2048 work items
    (one per prompt in a tile) go longest first; more than that, and the tiles
    go in token order with all their prompts in one unit."""
    gen = torch.Generator().manual_seed(37 + prompts)
    lens = torch.randint(1, prompt_len + 1, (prompts,), generator=gen).tolist()
    starts = torch.randint(0, 301, (prompts,), generator=gen).tolist()
    assert (_tile_items(lens) <= 2048) == sorted_items
    wl = W.make_prefill(f"prefill {prompts} short prompts", lens, starts, seed=37, table_pages=6, gen=gen)
    compare(wl, run_gpu(wl), run_oracle(wl), label=f"prefill {prompts} short prompts")


@pytest.mark.parametrize("kv_heads", [2, 16])
def test_prompt_paths_other_head_counts(kv_heads):
    """Prefill and step with 4 x kv_heads query heads other than Qwen3-8B's 32:
    the prompt tokens' prepared queries (64 heads take the per-warp loop past
    its first eight heads) and each unit's copy of its four heads' rows."""
    cfg = dict(kv_heads=kv_heads, heads=4 * kv_heads)
    wl = W.make_prefill(f"prefill {kv_heads} kv heads", [70, 130, 9], [60, 0, 200], seed=38, cfg=cfg,
                        table_pages=5)
    compare(wl, run_gpu(wl), run_oracle(wl), label=f"prefill, {kv_heads} kv heads")
    wl = W.make_step(f"step {kv_heads} kv heads", [100, 40], [0, 300], [700, 64, 1, 333], seed=39, cfg=cfg,
                     table_pages=12)
    compare(wl, run_gpu(wl), run_oracle(wl), label=f"step, {kv_heads} kv heads")


def test_prefill_invalid_tokens():
    wl = W.make_prefill("prefill errors", [40, 30, 20], [0, 100, 5], seed=33, table_pages=4)
    pos = wl.positions.clone()
    pos[3] = 40960                       # beyond max_seq
    pos[45] = 4 * 64                     # beyond the table width
    table = wl.table.clone()
    table[2, 0] = wl.num_pages + 3       # not a pool page: all of prompt 2 is skipped
    gpu = run_gpu(wl, table=table, positions=pos)
    ref = run_oracle(wl, table=table, positions=pos)
    assert ref[3] == (oracle.ERR_POSITION | oracle.ERR_PAGE)
    compare(wl, gpu, ref, label="prefill errors")
    assert not gpu[0][3].float().abs().sum() and not gpu[0][45].float().abs().sum()
    assert not gpu[0][70:].float().abs().sum()


# ------------------------------------------------------------------ contiguous rows (NULL table)

@pytest.mark.parametrize("ctas", [0, 7])
def test_decode_rows_contiguous(ctas):
    """decode_rows: 64 rows of 640 positions each (10 pages a row), lengths
    U[1, 640]; the rows own their pages in pool order."""
    wl = W.make_decode("decode_rows 64 x 640", (64, 1, 640), seed=34, table_pages=10, contiguous=True)
    assert wl.contiguous and wl.num_pages == 640
    compare(wl, run_gpu(wl, ctas=ctas), run_oracle(wl), label=f"decode_rows ctas={ctas}")


def test_prefill_packed_contiguous():
    """prefill_packed: prompts each filling its own row from position 0."""
    wl = W.make_prefill("prefill_packed", [1, 64, 65, 200, 127], [0] * 5, seed=36, table_pages=4, contiguous=True)
    compare(wl, run_gpu(wl), run_oracle(wl), label="prefill_packed")


def test_step_packed_contiguous():
    """step_packed: prompts continuing their rows plus decode rows, all contiguous."""
    wl = W.make_step("step_packed", prompt_lengths=[70, 5, 130], prompt_starts=[0, 60, 100],
                     decode_lengths=[90, 3, 64, 65, 1, 640], seed=37, table_pages=10, contiguous=True)
    ref = run_oracle(wl)
    compare(wl, run_gpu(wl), ref, label="step_packed")
    compare(wl, run_gpu(wl, ctas=5), ref, label="step_packed ctas=5")


def test_contiguous_rows_must_fit_the_pool():
    """rows * pages beyond the pool is a host error, with nothing enqueued."""
    wl = W.make_decode("too wide", [10, 20], seed=38, table_pages=2, contiguous=True)
    dev = torch.device("cuda")
    K, V = wl.K0.to(dev), wl.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
    q, k, v, qw, kw, sp = (t.to(dev) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w, wl.step_positions))
    out = torch.zeros_like(q)
    ws = pool.workspace(2, 3, 0)
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_decode(pool.handle, q, k, v, qw, kw, sp, None, out, ws, pages=3)
    assert ei.value.code == pkv.PKV_ERANGE
    pos = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_prefill(pool.handle, q[:1], k[:1], v[:1], qw, kw, pos, pos, None, None, out[:1],
                        pool.workspace(0, 3, 1), rows=2, pages=3)
    assert ei.value.code == pkv.PKV_ERANGE
    torch.cuda.synchronize()
    assert not out.any()
    assert torch.equal(K.cpu(), wl.K0) and torch.equal(V.cpu(), wl.V0)
    assert pool.check_errors() == 0
    pool.close()


# ------------------------------------------------------------------ optional host pre-check

def test_host_precheck_rejects_bad_slots(monkeypatch):
    """With PKV_CHECK=1 a call whose given prompt slots disagree with the table,
    or whose written slots coincide outside page 0, is refused before anything
    is enqueued; consistent calls run and match the oracle."""
    monkeypatch.setenv("PKV_CHECK", "1")
    wl = W.make_step("checked step", prompt_lengths=[70, 5], prompt_starts=[60, 0], decode_lengths=[90, 3, 64],
                     seed=39, table_pages=3)
    slots = oracle.page_slots(wl.table.numpy(), wl.prow.numpy(), wl.positions.numpy())
    compare(wl, run_gpu(wl, explicit_slots=slots), run_oracle(wl), label="checked step")

    dev = torch.device("cuda")
    K, V = wl.K0.to(dev), wl.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
    q, k, v, qw, kw = (t.to(dev) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w))
    pos, prow, sp, tab = (t.to(dev) for t in (wl.positions, wl.prow, wl.step_positions, wl.table))
    out = torch.zeros_like(q)
    bad = slots.copy()
    bad[3] = bad[4]                          # token 3 given token 4's slot: off the table, and a duplicate
    with pytest.raises(pkv.PkvError) as ei:
        pool.step(q, k, v, qw, kw, pos, prow, torch.as_tensor(bad, dtype=torch.int32).to(dev), sp, tab, out=out)
    assert ei.value.code == pkv.PKV_EINVAL
    # two decode rows writing one slot (row 2 steps at row 0's position through row 0's pages)
    tab2 = wl.table.clone()
    tab2[2] = tab2[0]
    sp2 = wl.step_positions.clone()
    sp2[2] = sp2[0]
    with pytest.raises(pkv.PkvError) as ei:
        pool.step(q, k, v, qw, kw, pos, prow, None, sp2.to(dev), tab2.to(dev), out=out)
    assert ei.value.code == pkv.PKV_EINVAL
    torch.cuda.synchronize()
    assert not out.any()
    assert torch.equal(K.cpu(), wl.K0) and torch.equal(V.cpu(), wl.V0)
    # without the check the same call is enqueued (its result is unspecified)
    monkeypatch.delenv("PKV_CHECK")
    pool.step(q, k, v, qw, kw, pos, prow, None, sp2.to(dev), tab2.to(dev), out=out)
    torch.cuda.synchronize()
    pool.close()


def test_host_precheck_rejects_decode_rows_reading_another_rows_new_slot(monkeypatch):
    """Decode orders each row's write before its own reads only, so with
    PKV_CHECK=1 a decode call in which a row reads (at a position up to its
    own) a slot another row writes is refused, through both decode entries;
    a shared prefix (pages strictly before every sharing row's write page) is
    accepted, and pkv_step, which orders every write before every read,
    accepts the call the decode entries refuse and matches the oracle."""
    monkeypatch.setenv("PKV_CHECK", "1")
    wl = W.make_decode("cross reads", [100, 200], seed=40, table_pages=4)
    dev = torch.device("cuda")
    q, k, v, qw, kw, sp = (t.to(dev) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w, wl.step_positions))

    def refused(table):
        K, V = wl.K0.to(dev), wl.V0.to(dev)
        pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
        out = torch.zeros_like(q)
        tab = torch.as_tensor(table).to(dev)
        with pytest.raises(pkv.PkvError) as ei:
            pool.decode(q, k, v, qw, kw, sp, tab, out=out)
        assert ei.value.code == pkv.PKV_EINVAL
        with pytest.raises(pkv.PkvError) as ei:
            pkv.pkv_decode_static(pool.handle, q, k, v, qw, kw, sp, tab, out)
        assert ei.value.code == pkv.PKV_EINVAL
        torch.cuda.synchronize()
        assert not out.any() and torch.equal(K.cpu(), wl.K0) and torch.equal(V.cpu(), wl.V0)
        pool.close()

    # row 0 writes at page 1, offset 35; row 1 (position 199) reads all of its page 1
    t1 = wl.table.clone()
    t1[1, 1] = t1[0, 1]
    refused(t1)
    # the other direction: row 1's last page is row 0's write page, row 1 writes
    # offset 20 of it, which row 0 (offset 35) reads
    wl2 = W.make_decode("cross reads 2", [100, 85], seed=41, table_pages=4)
    assert wl2.meta["lengths"] == [100, 85]
    t2 = wl2.table.clone()
    t2[1, 1] = t2[0, 1]
    wl, q, k, v, qw, kw, sp = (wl2, *(t.to(dev) for t in (wl2.q, wl2.k, wl2.v, wl2.q_norm_w, wl2.k_norm_w,
                                                          wl2.step_positions)))
    refused(t2)
    # a shared prefix page (page 0, before both write pages) passes and matches the oracle
    t3 = wl.table.clone()
    t3[1, 0] = t3[0, 0]
    compare(wl, run_gpu(wl, table=t3), run_oracle(wl, table=t3), label="checked shared prefix")
    # the same rows as a step (one prompt token stands in for P > 0): writes come first, so it is accepted
    st = W.make_step("cross reads as a step", prompt_lengths=[1], prompt_starts=[0], decode_lengths=[100, 85],
                     seed=42, table_pages=4)
    t4 = st.table.clone()
    t4[1, 1] = t4[0, 1]
    compare(st, run_gpu(st, table=t4), run_oracle(st, table=t4), label="checked step cross reads")
