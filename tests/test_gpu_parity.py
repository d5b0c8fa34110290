"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle
on the same seeded inputs.

Bar (per output element / pool entry):
  * page/slot placement and untouched pool entries bit-exact, V bit-exact,
    written K within 1 bf16 ulp of the oracle's correctly rounded value;
  * attention outputs within max-abs 2e-2 and relative-L2 5e-3 of the
    oracle's fp64 result;
  * device error bits equal to the oracle's skip reasons.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_qk_gb300 as pkv
import workloads as W
from _harness import compare, run_gpu, run_oracle, step_sm_split

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ the five configurations

@pytest.mark.parametrize("ctas", [0, 1, 2, 5])
def test_config1_tiny(ctas):
    wl = W.config1()
    ma, rel = compare(wl, run_gpu(wl, ctas=ctas), run_oracle(wl), label=f"config1 ctas={ctas}")
    assert ma < 5e-3


def test_config2_decode_64_rows():
    wl = W.config2()
    compare(wl, run_gpu(wl), run_oracle(wl), label="config2")


def test_config3_long_context():
    wl = W.config3()
    compare(wl, run_gpu(wl), run_oracle(wl), label="config3")


def test_config4_shared_prefixes():
    wl = W.config4()
    compare(wl, run_gpu(wl), run_oracle(wl), label="config4")


def test_config5_step_mix():
    """Every token of the step: all 2048 prompt tokens (so every row of every
    64-token tile, every tensor-memory lane quarter and every work item of the
    prompt attention's schedule) and all 128 decode rows."""
    wl = W.config5()
    compare(wl, run_gpu(wl), run_oracle(wl), label="config5 (all tokens)")


# ------------------------------------------------------------------ tiles, ragged tails, partitions

RAGGED = [1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 191, 640, 1000, 4097]


@pytest.mark.parametrize("ctas", [0, 1, 3, 7, 1000])
def test_ragged_lengths_and_partitions(ctas):
    wl = W.make_decode("ragged", RAGGED, seed=77, table_pages=70)
    compare(wl, run_gpu(wl, ctas=ctas), run_oracle(wl), label=f"ragged ctas={ctas}")


@pytest.mark.parametrize("ctas", [0, 7])
def test_last_positions_of_the_context(ctas):
    """The largest positions the configuration allows (max_seq 40960: page 639,
    slot 63): decode rows whose step token is the context's last position, one
    page before it and at its first page, beside short rows."""
    wl = W.make_decode("max_seq", [40960, 1, 40960 - 64, 40897, 7], seed=27, table_pages=640)
    compare(wl, run_gpu(wl, ctas=ctas), run_oracle(wl), label=f"max_seq ctas={ctas}")


def test_step_prompt_ending_at_the_last_position():
    """A prompt chunk whose last token sits at position 40959 (the prompt
    attention's longest run, a tile ending on the context's last slot), a
    3-token chunk ending there too, and a decode row at the same position."""
    wl = W.make_step("max_seq step", prompt_lengths=[40, 3], prompt_starts=[40920, 40957],
                     decode_lengths=[40960, 7], seed=28, table_pages=640)
    compare(wl, run_gpu(wl), run_oracle(wl), label="max_seq step")


def test_sweep_shape_small():
    wl = W.sweep(8, 4096, seed=5)
    compare(wl, run_gpu(wl), run_oracle(wl), label="sweep 8x4096")


def test_step_small_with_explicit_slots():
    wl = W.make_step("small step", prompt_lengths=[70, 5, 130], prompt_starts=[60, 0, 500],
                     decode_lengths=[90, 3, 64, 65, 1], seed=21, table_pages=12)
    slots = oracle.page_slots(wl.table.numpy(), wl.prow.numpy(), wl.positions.numpy())
    ref = run_oracle(wl)
    compare(wl, run_gpu(wl, explicit_slots=slots), ref, label="step explicit slots")
    compare(wl, run_gpu(wl), ref, label="step derived slots")
    compare(wl, run_gpu(wl, ctas=1), ref, label="step ctas=1")
    compare(wl, run_gpu(wl, ctas=13), ref, label="step ctas=13")


def _step_sm_split(wl):
    return step_sm_split((wl.positions + 1).tolist(), wl.step_positions.tolist(), wl.cfg["kv_heads"],
                         torch.cuda.get_device_properties(0).multi_processor_count, wl.cfg["page_size"])


def test_step_prompts_beside_the_rows():
    """A step whose prompt attention keeps part of the SMs (prompt_sms) while
    the rows' attention starts on the rest: 4 prompt chunks continuing long
    rows, 64 rows of 2K-4K positions; then short rows (whole units) beside one
    small chunk, where the rows' attention CTAs that start late only claim."""
    wl = W.make_step("prompts beside rows", prompt_lengths=[128, 128, 128, 128], prompt_starts=[600, 1500, 0, 3000],
                     decode_lengths=W._uniform_int(torch.Generator().manual_seed(41), 2048, 4096, 64).tolist(),
                     seed=41, table_pages=64)
    kept, ra = _step_sm_split(wl)
    assert kept < min(torch.cuda.get_device_properties(0).multi_processor_count, 8 * 8), kept
    ref = run_oracle(wl)
    compare(wl, run_gpu(wl), ref, label="prompts beside rows")
    short = W.make_step("chunk beside short rows", prompt_lengths=[64], prompt_starts=[100],
                        decode_lengths=W._uniform_int(torch.Generator().manual_seed(42), 1, 512, 100).tolist(),
                        seed=42, table_pages=8)
    kept, ra = _step_sm_split(short)
    assert ra < 2 * torch.cuda.get_device_properties(0).multi_processor_count, ra
    compare(short, run_gpu(short), run_oracle(short), label="chunk beside short rows")


def test_step_many_prompt_tiles_beside_the_rows():
    """More prompt tiles (54 of 64 tokens) than either kernel's cost pass covers
    in one round trip, so both derive the split over several rounds; the
    prompt attention still keeps part of the SMs."""
    g = torch.Generator().manual_seed(43)
    wl = W.make_step("many prompt tiles", prompt_lengths=[550] * 6,
                     prompt_starts=W._uniform_int(g, 0, 1500, 6).tolist(),
                     decode_lengths=W._uniform_int(g, 1024, 4096, 48).tolist(), seed=43, table_pages=64)
    assert wl.P > 3072
    kept, ra = _step_sm_split(wl)
    assert kept < torch.cuda.get_device_properties(0).multi_processor_count, kept
    compare(wl, run_gpu(wl), run_oracle(wl), label="many prompt tiles")


@pytest.mark.parametrize("ctas", [0, 7])
def test_new_key_dominates(ctas):
    """Each row's new key equals its first query head's (same raw vector, same
    norm weight, same position), so that head puts ~99% of its weight on the
    key the call has just written.  A read of the page before the write would
    miss it and be off by O(1), far outside the tolerance."""
    wl = W.make_decode("own key", [1000, 1, 65, 130, 2049, 64], seed=26, table_pages=33)
    k = wl.k.clone()
    for g in range(wl.cfg["kv_heads"]):
        k[:, g] = wl.q[:, 4 * g]
    wl = W.Workload(**{**wl.__dict__, "k": k, "k_norm_w": wl.q_norm_w.clone()})
    gpu, ref = run_gpu(wl, ctas=ctas), run_oracle(wl)
    compare(wl, gpu, ref, label=f"own key ctas={ctas}")
    # the new key's value dominates the first head of every group
    S = wl.cfg["page_size"]
    vnew = wl.v.double().numpy()
    out = ref[0]
    for b, L in enumerate(wl.meta["lengths"]):
        for g in range(wl.cfg["kv_heads"]):
            assert np.abs(out[b, 4 * g] - vnew[b, g]).max() < 0.1 * max(1.0, np.abs(vnew[b, g]).max())


def test_repeated_calls_are_idempotent():
    wl = W.make_decode("repeat", [300, 5, 1000], seed=22, table_pages=16)
    compare(wl, run_gpu(wl, repeat=3), run_oracle(wl), label="repeat x3")


def test_claimed_chunks_give_the_same_bits_every_call():
    """The attention hands the last quarter of the pages out as chunks that
    whichever CTA finishes first claims.  Where a piece ends and the order in
    which pieces merge depend only on the call's shape, not on which CTA
    streamed them, so repeated calls give identical outputs (the 64-row
    U[512,4096] batch: ~18k (row, kv head, page) triples, ~1150 chunks)."""
    wl = W.make_decode("reproducible", (64, 512, 4096), seed=26, table_pages=64)
    dev = torch.device("cuda")
    K, V = wl.K0.to(dev), wl.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
    q, k, v, qw, kw, sp, tab = (t.to(dev) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w,
                                                     wl.step_positions, wl.table))
    outs = [pool.decode(q, k, v, qw, kw, sp, tab).clone() for _ in range(6)]
    assert pool.check_errors() == 0
    assert all(torch.equal(o, outs[0]) for o in outs[1:])
    pool.close()


def _streams_units_whole(wl, ctas, step_positions, pages):
    """The attention's rule for handing out every (token, kv head) unit whole,
    longest first: at most one token per prologue thread (160), no unit longer
    than 16 pages, the longest within 5/4 of a CTA's share of all pages."""
    S, G = wl.cfg["page_size"], wl.cfg["kv_heads"]
    npg = [p // S + 1 for p in step_positions.tolist() if 0 <= p < min(wl.cfg["max_seq"], pages * S)]
    C = ctas or 2 * torch.cuda.get_device_properties(0).multi_processor_count
    T = G * sum(npg)
    return len(step_positions) <= 160 and max(npg) <= 16 and 4 * max(npg) * C <= 5 * T


@pytest.mark.parametrize("rows", [64, 160, 161])
def test_short_rows_streamed_as_whole_units(rows):
    """Calls of short rows: with at most 160 rows, no unit above 16 pages and the
    longest within 5/4 of a CTA's share, each (token, kv head) is streamed whole
    by one CTA, longest first, and written out by it; the output then does not
    depend on the grid size.  A skipped row and a row with an invalid page sit
    among them; 161 rows take the slices and chunks instead."""
    wl = W.make_decode("short rows", (rows, 1, 1024), seed=40 + rows, table_pages=16)
    sp = wl.step_positions.clone()
    table = wl.table.clone()
    sp[3] = -1                        # no step
    table[5, 0] = wl.num_pages + 3    # not a pool page
    ref = run_oracle(wl, table=table, step_positions=sp)
    outs = []
    for ctas in (0, 2, 7, 1):
        whole = _streams_units_whole(wl, ctas, sp, table.shape[1])
        assert whole == (rows <= 160), (rows, ctas)
        gpu = run_gpu(wl, ctas=ctas, table=table, step_positions=sp)
        compare(wl, gpu, ref, label=f"short rows {rows} ctas={ctas}")
        outs.append(gpu[0])
    if rows <= 160:
        assert all(torch.equal(o, outs[0]) for o in outs[1:])


# ------------------------------------------------------------------ skipped tokens and device errors

def test_inactive_and_invalid_rows():
    wl = W.make_decode("errors", [100, 70, 5, 2000, 64], seed=23, table_pages=32)
    sp = wl.step_positions.clone()
    table = wl.table.clone()
    sp[0] = -1                       # no step: zero output, no write, no error
    sp[1] = 40960                    # beyond max_seq
    table[2, 0] = wl.num_pages + 7   # not a pool page
    sp[4] = 32 * 64                  # beyond the table width
    gpu = run_gpu(wl, table=table, step_positions=sp)
    ref = run_oracle(wl, table=table, step_positions=sp)
    assert ref[3] == (oracle.ERR_POSITION | oracle.ERR_PAGE)
    compare(wl, gpu, ref, label="errors")
    out = gpu[0]
    for b in (0, 1, 2, 4):
        assert not out[b].float().abs().sum()


def test_step_invalid_prompt_tokens():
    wl = W.make_step("step errors", prompt_lengths=[40, 30], prompt_starts=[0, 100], decode_lengths=[50, 10],
                     seed=24, table_pages=4)
    pos = wl.positions.clone()
    pos[3] = -5                      # negative position
    gpu_prow = wl.prow.clone()
    prow_bad = gpu_prow.clone()
    prow_bad[10] = 99                # row outside the table
    wl_bad = W.Workload(**{**wl.__dict__, "prow": prow_bad})
    gpu = run_gpu(wl_bad, positions=pos)
    ref = run_oracle(wl_bad, positions=pos)
    assert ref[3] == (oracle.ERR_POSITION | oracle.ERR_ROW)
    compare(wl_bad, gpu, ref, label="step errors")


def test_host_errors_enqueue_nothing():
    wl = W.config1()
    dev = torch.device("cuda")
    K, V = wl.K0.to(dev), wl.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
    q, k, v, qw, kw, sp, tab = (t.to(dev) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w,
                                                   wl.step_positions, wl.table))
    out = torch.zeros_like(q)
    need = pkv.pkv_workspace_bytes(pool.handle, 2, 2, 0)
    small = torch.empty(need - 256, dtype=torch.uint8, device=dev)
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_decode(pool.handle, q, k, v, qw, kw, sp, tab, out, small)
    assert ei.value.code == pkv.PKV_EWORKSPACE
    torch.cuda.synchronize()
    assert not out.any()
    assert torch.equal(K.cpu(), wl.K0) and torch.equal(V.cpu(), wl.V0)
    # unsupported shapes are refused at pool creation
    with pytest.raises(pkv.PkvError) as ei:
        pkv.pkv_pool_alloc(dict(wl.cfg, head_dim=64), 4)
    assert ei.value.code == pkv.PKV_ENOTIMPL
    pool.close()


def test_pool_alloc_owns_zeroed_memory():
    cfg = pkv.pkv_config_default()
    pool = pkv.pkv_pool_alloc(cfg, 3)
    k, v, n = pkv.pkv_pool_kv(pool)
    assert n == 3 * 64 and k and v and k % 256 == 0
    pkv.pkv_pool_free(pool)


# ------------------------------------------------------------------ partition by kv heads

def test_kv_head_shards_reproduce_full_result():
    """The attention needs no exchange between kv-head groups: running the
    library once per kv-head shard (a pool of kv_heads/n heads, the matching
    query heads) and concatenating reproduces the full result bit-exactly."""
    wl = W.make_decode("shard", [500, 64, 1300, 7], seed=25, table_pages=24)
    # one CTA: every (token, kv head) is summed in the same order whatever the shard
    full = run_gpu(wl, ctas=1)
    n = 4
    G = wl.cfg["kv_heads"] // n
    outs = []
    for r in range(n):
        g0, g1 = r * G, (r + 1) * G
        cfg = dict(wl.cfg, kv_heads=G, heads=4 * G)
        part = W.Workload(wl.name, cfg, wl.num_pages, wl.K0[g0:g1].contiguous(), wl.V0[g0:g1].contiguous(),
                          wl.q[:, 4 * g0:4 * g1].contiguous(), wl.k[:, g0:g1].contiguous(),
                          wl.v[:, g0:g1].contiguous(), wl.q_norm_w, wl.k_norm_w, wl.table, wl.step_positions)
        out, K, V, flags = run_gpu(part, ctas=1)
        assert flags == 0
        assert torch.equal(K, full[1][g0:g1]) and torch.equal(V, full[2][g0:g1])
        outs.append(out)
    assert torch.equal(torch.cat(outs, dim=1), full[0])
