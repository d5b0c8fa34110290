"""Seeded synthetic inputs for the paged-KV decode step.

This module is shared by the tests, the benchmark and the smoke check.  It
holds none of the method's arithmetic: it draws random values, lays pages
out in a pool and writes a page table, and nothing else.  Both the oracle and
the CUDA path consume what it returns.

Recipe (the same for every workload):
  * A CPU ``torch.Generator`` seeded with the workload's seed draws float32
    values that are rounded to bf16 (round-to-nearest-even).
  * q, k, v and every pre-existing pool entry ~ N(0, 1); the QK-norm weights
    ~ U[0.5, 1.5].
  * Context lengths are integers drawn uniformly, both ends inclusive; the
    step token of a row with length L sits at position L - 1 (positions
    0..L-2 are pre-filled).
  * Pool page 0 is a scratch page that no live row reads (unused table
    entries point at it); live rows take their pages, in row order, from a
    seeded permutation of pages 1..num_pages-1.  The pool holds exactly the
    pages needed plus the scratch page.
  * Shapes are Qwen3-8B's attention: 32 query heads, 8 kv heads, head_dim
    128, pages of 64 positions, MaxSeq 40960.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DEFAULT_CONFIG = dict(heads=32, kv_heads=8, head_dim=128, page_size=64, max_seq=40960,
                      rope_theta=1.0e6, eps=1.0e-6, rotary_dim=128)

# Bytes of K and V one position occupies across all kv heads (bf16).
def kv_bytes_per_position(cfg: dict) -> int:
    return 2 * cfg["kv_heads"] * cfg["head_dim"] * 2


@dataclass
class Workload:
    name: str
    cfg: dict
    num_pages: int
    K0: torch.Tensor            # bf16 [kv_heads][num_pages*page_size][head_dim], pool before the step
    V0: torch.Tensor
    q: torch.Tensor             # bf16 [P+R][heads][head_dim]
    k: torch.Tensor             # bf16 [P+R][kv_heads][head_dim]
    v: torch.Tensor
    q_norm_w: torch.Tensor      # bf16 [head_dim]
    k_norm_w: torch.Tensor
    table: torch.Tensor         # int32 [R][pages]
    step_positions: torch.Tensor  # int32 [R]; -1 = row takes no step
    positions: torch.Tensor | None = None  # int32 [P] prompt-token positions (step only)
    prow: torch.Tensor | None = None       # int32 [P] prompt-token rows (step only)
    meta: dict = field(default_factory=dict)

    @property
    def P(self) -> int:
        return 0 if self.positions is None else int(self.positions.shape[0])

    @property
    def R(self) -> int:
        return int(self.step_positions.shape[0])

    @property
    def pages(self) -> int:
        return int(self.table.shape[1])

    @property
    def kind(self) -> str:
        """"decode", "step" or "prefill" (prompt tokens only; the table rows take no step)."""
        return self.meta.get("mode") or ("decode" if self.positions is None else "step")

    @property
    def contiguous(self) -> bool:
        """True when ``table`` is the contiguous-row identity (row b owns pages b*pages ..)."""
        return bool(self.meta.get("contiguous"))


def bits(t: torch.Tensor):
    """numpy uint16 view of a bf16 tensor's bit patterns (for the oracle)."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _randn_bf16(gen: torch.Generator, shape, chunk: int = 1 << 24) -> torch.Tensor:
    n = math.prod(shape)
    out = torch.empty(n, dtype=torch.bfloat16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return out.view(*shape)


def _uniform_int(gen: torch.Generator, lo: int, hi: int, n: int) -> torch.Tensor:
    """n integers uniform on [lo, hi], both inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=gen, dtype=torch.int64)


def _pages_for(length: int, page_size: int) -> int:
    return -(-length // page_size)


def _tokens(gen: torch.Generator, cfg: dict, n: int):
    H, G, D = cfg["heads"], cfg["kv_heads"], cfg["head_dim"]
    q = _randn_bf16(gen, (n, H, D))
    k = _randn_bf16(gen, (n, G, D))
    v = _randn_bf16(gen, (n, G, D))
    qw = (torch.rand(D, generator=gen, dtype=torch.float32) + 0.5).to(torch.bfloat16)
    kw = (torch.rand(D, generator=gen, dtype=torch.float32) + 0.5).to(torch.bfloat16)
    return q, k, v, qw, kw


def contiguous_table(rows: int, pages: int) -> torch.Tensor:
    """The contiguous-row layout as a page table: row b owns pool pages b*pages .. b*pages+pages-1."""
    return torch.arange(rows * pages, dtype=torch.int32).view(rows, pages)


def make_decode(name: str, lengths, seed: int, cfg: dict | None = None, table_pages: int | None = None,
                share_groups: int = 0, share_range=(8, 32), scratch: bool = True,
                contiguous: bool = False) -> Workload:
    """A decode_paged workload: one step token per row, row b at position lengths[b]-1.

    share_groups > 0: consecutive groups of that many rows share their first
    s_g pages, s_g = min(U{share_range}, smallest write-page index in the
    group), so shared pages are full pages strictly before every write.
    contiguous: the decode_rows layout, row b owning table_pages pages of its
    own in pool order (pool of rows * table_pages pages, table the identity).
    """
    if contiguous:
        assert not share_groups and table_pages is not None
        wl = make_decode(name, lengths, seed, cfg, table_pages, scratch=False)
        R, S = wl.R, wl.cfg["page_size"]
        gen = torch.Generator().manual_seed(seed + 1)
        G, D = wl.cfg["kv_heads"], wl.cfg["head_dim"]
        num_pages = R * table_pages
        K0 = _randn_bf16(gen, (G, num_pages * S, D))
        V0 = _randn_bf16(gen, (G, num_pages * S, D))
        meta = dict(wl.meta, contiguous=True)
        return Workload(name, wl.cfg, num_pages, K0, V0, wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w,
                        contiguous_table(R, table_pages), wl.step_positions, meta=meta)
    cfg = dict(DEFAULT_CONFIG, **(cfg or {}))
    S = cfg["page_size"]
    gen = torch.Generator().manual_seed(seed)
    if isinstance(lengths, tuple) and len(lengths) == 3:       # (rows, lo, hi): drawn
        rows, lo, hi = lengths
        L = _uniform_int(gen, lo, hi, rows).tolist()
    else:
        L = [int(x) for x in lengths]
    R = len(L)
    npages = [_pages_for(x, S) for x in L]
    width = table_pages if table_pages is not None else max(npages)
    assert width >= max(npages)

    shared = [0] * R
    if share_groups:
        for g0 in range(0, R, share_groups):
            grp = range(g0, min(R, g0 + share_groups))
            draw = int(_uniform_int(gen, share_range[0], share_range[1], 1)[0])
            s_g = min([draw] + [(L[b] - 1) // S for b in grp])
            for b in grp:
                shared[b] = s_g
    # number of distinct pages: group-shared pages once, private pages per row
    seen_groups = {}
    unique_pages = 0
    for b in range(R):
        gkey = b // share_groups if share_groups else b
        if share_groups and gkey not in seen_groups:
            seen_groups[gkey] = None
            unique_pages += shared[b]
        unique_pages += npages[b] - shared[b]
    num_pages = unique_pages + (1 if scratch else 0)
    first = 1 if scratch else 0
    perm = (torch.randperm(num_pages - first, generator=gen) + first).tolist()

    table = torch.zeros(R, width, dtype=torch.int32)
    it = iter(perm)
    group_pages = {}
    for b in range(R):
        gkey = b // share_groups if share_groups else None
        if share_groups and gkey not in group_pages:
            group_pages[gkey] = [next(it) for _ in range(shared[b])]
        row_pages = (group_pages[gkey] if share_groups else []) + [next(it) for _ in range(npages[b] - shared[b])]
        table[b, :len(row_pages)] = torch.tensor(row_pages, dtype=torch.int32)

    G, D = cfg["kv_heads"], cfg["head_dim"]
    q, k, v, qw, kw = _tokens(gen, cfg, R)
    K0 = _randn_bf16(gen, (G, num_pages * S, D))
    V0 = _randn_bf16(gen, (G, num_pages * S, D))
    positions = torch.tensor([x - 1 for x in L], dtype=torch.int32)
    bpp = kv_bytes_per_position(cfg)
    if share_groups:   # a shared page is read by every row of its group but held once
        unique_positions = (sum(L) - sum(shared[b] * S for b in range(R))
                            + sum(shared[g0] * S for g0 in range(0, R, share_groups)))
    else:
        unique_positions = sum(L)
    meta = dict(lengths=L, shared_pages=shared, logical_kv_bytes=bpp * sum(L),
                unique_kv_bytes=bpp * unique_positions, seed=seed)
    return Workload(name, cfg, num_pages, K0, V0, q, k, v, qw, kw, table, positions, meta=meta)


def make_step(name: str, prompt_lengths, prompt_starts, decode_lengths, seed: int, cfg: dict | None = None,
              table_pages: int | None = None, gen: torch.Generator | None = None,
              contiguous: bool = False) -> Workload:
    """A step_paged workload: prompt chunks packed end to end, then one step per decode row.

    Table rows 0..R_d-1 are the decode rows; rows R_d..R_d+M-1 hold the M
    prompts (they take no step: step_positions -1).  Prompt j continues at
    position prompt_starts[j] over pre-filled pages and spans
    prompt_lengths[j] tokens.  contiguous: the step_packed layout (identity
    table, pool of rows * table_pages pages).
    """
    cfg = dict(DEFAULT_CONFIG, **(cfg or {}))
    S = cfg["page_size"]
    gen = gen if gen is not None else torch.Generator().manual_seed(seed)
    M = len(prompt_lengths)
    Rd = len(decode_lengths)
    R = Rd + M
    row_len = [int(x) for x in decode_lengths] + [int(s) + int(n) for s, n in zip(prompt_starts, prompt_lengths)]
    npages = [_pages_for(x, S) for x in row_len]
    width = table_pages if table_pages is not None else max(npages)
    assert width >= max(npages)
    if contiguous:
        num_pages = R * width
        table = contiguous_table(R, width)
    else:
        num_pages = sum(npages) + 1
        perm = (torch.randperm(num_pages - 1, generator=gen) + 1).tolist()
        table = torch.zeros(R, width, dtype=torch.int32)
        it = iter(perm)
        for b in range(R):
            table[b, :npages[b]] = torch.tensor([next(it) for _ in range(npages[b])], dtype=torch.int32)
    positions, prow = [], []
    for j in range(M):
        positions += list(range(int(prompt_starts[j]), int(prompt_starts[j]) + int(prompt_lengths[j])))
        prow += [Rd + j] * int(prompt_lengths[j])
    P = len(positions)
    G, D = cfg["kv_heads"], cfg["head_dim"]
    q, k, v, qw, kw = _tokens(gen, cfg, P + R)
    K0 = _randn_bf16(gen, (G, num_pages * S, D))
    V0 = _randn_bf16(gen, (G, num_pages * S, D))
    step_positions = torch.tensor([x - 1 for x in decode_lengths] + [-1] * M, dtype=torch.int32)
    bpp = kv_bytes_per_position(cfg)
    meta = dict(decode_lengths=[int(x) for x in decode_lengths], prompt_lengths=[int(x) for x in prompt_lengths],
                prompt_starts=[int(x) for x in prompt_starts],
                logical_kv_bytes=bpp * sum(int(x) for x in decode_lengths),
                prefill_attended_positions=sum(p + 1 for p in positions), seed=seed, contiguous=contiguous)
    return Workload(name, cfg, num_pages, K0, V0, q, k, v, qw, kw, table, step_positions,
                    positions=torch.tensor(positions, dtype=torch.int32),
                    prow=torch.tensor(prow, dtype=torch.int32), meta=meta)


def make_prefill(name: str, prompt_lengths, prompt_starts, seed: int, cfg: dict | None = None,
                 table_pages: int | None = None, gen: torch.Generator | None = None,
                 contiguous: bool = False) -> Workload:
    """A prefill_paged workload: make_step's prompts with no decode rows.

    Its M table rows all take no step, so q/k/v keep M unused step tokens
    after the P prompt tokens (the oracle's step form); a prefill call takes
    the first P.
    """
    wl = make_step(name, prompt_lengths, prompt_starts, [], seed, cfg, table_pages, gen, contiguous)
    wl.meta["mode"] = "prefill"
    # K/V the prompts' attention reads: each prompt's row up to its last position
    wl.meta["logical_kv_bytes"] = kv_bytes_per_position(wl.cfg) * sum(
        int(s) + int(n) for s, n in zip(prompt_starts, prompt_lengths))
    return wl


# ------------------------------------------------------------------ the five configs

def config1() -> Workload:
    """Tiny decode: 2 rows at positions 10 and 70, pool of 8 pages, table a seeded permutation."""
    cfg = dict(DEFAULT_CONFIG)
    gen = torch.Generator().manual_seed(1001)
    perm = torch.randperm(8, generator=gen).to(torch.int32)
    table = perm[:4].view(2, 2).clone()
    q, k, v, qw, kw = _tokens(gen, cfg, 2)
    G, D, S = cfg["kv_heads"], cfg["head_dim"], cfg["page_size"]
    K0 = _randn_bf16(gen, (G, 8 * S, D))
    V0 = _randn_bf16(gen, (G, 8 * S, D))
    positions = torch.tensor([10, 70], dtype=torch.int32)
    bpp = kv_bytes_per_position(cfg)
    meta = dict(lengths=[11, 71], logical_kv_bytes=bpp * 82, unique_kv_bytes=bpp * 82, seed=1001)
    return Workload("tiny: 2 rows at positions 10 and 70, pool 8 pages", cfg, 8, K0, V0, q, k, v, qw, kw,
                    table, positions, meta=meta)


def config2() -> Workload:
    """64 rows, context lengths U[512, 4096], shuffled pages."""
    return make_decode("decode 64 rows x U[512,4096]", (64, 512, 4096), seed=1002, table_pages=64)


def config3() -> Workload:
    """8 rows, context lengths U[32768, 40960] (MaxSeq 40960)."""
    return make_decode("long-context decode 8 rows x U[32768,40960]", (8, 32768, 40960), seed=1003,
                       table_pages=640)


def config4() -> Workload:
    """256 rows, lengths U[1024, 8192]; groups of 16 rows share their first 8-32 pages."""
    return make_decode("shared-prefix decode 256 rows x U[1024,8192], groups of 16 share 8-32 pages",
                       (256, 1024, 8192), seed=1004, table_pages=128, share_groups=16)


def _prompt_mix(gen: torch.Generator, M: int = 4, P: int = 2048, minlen: int = 64, start_hi: int = 4096):
    """M prompt lengths summing to P (each >= minlen) and their start positions U[0, start_hi]."""
    cuts = sorted(_uniform_int(gen, 0, P - M * minlen, M - 1).tolist())
    bounds = [0] + cuts + [P - M * minlen]
    plen = [minlen + bounds[j + 1] - bounds[j] for j in range(M)]
    starts = _uniform_int(gen, 0, start_hi, M).tolist()
    return plen, starts


def config5() -> Workload:
    """step_paged: 4 prompts totalling P=2048 (each >= 64) continuing at U[0,4096], plus 128 rows x U[1024,8192]."""
    seed = 1005
    gen = torch.Generator().manual_seed(seed)
    plen, starts = _prompt_mix(gen)
    dlen = _uniform_int(gen, 1024, 8192, 128).tolist()
    return make_step("step: 4 prompts P=2048 at U[0,4096] + 128 decode rows x U[1024,8192]",
                     plen, starts, dlen, seed=seed, table_pages=128, gen=gen)


def prefill_mix(seed: int = 1006) -> Workload:
    """prefill_paged: config5's kind of prompt side alone, 4 prompts P=2048 continuing at U[0,4096]."""
    gen = torch.Generator().manual_seed(seed)
    plen, starts = _prompt_mix(gen)
    return make_prefill("prefill: 4 prompts P=2048 at U[0,4096]", plen, starts, seed=seed, table_pages=128,
                        gen=gen)


def rows_mix(seed: int = 1007) -> Workload:
    """decode_rows: 64 contiguous rows of 640 positions (10 pages each), lengths U[1, 640]."""
    return make_decode("decode_rows 64 rows x U[1,640], 640 positions a row", (64, 1, 640), seed=seed,
                       table_pages=10, contiguous=True)


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}


def sweep(rows: int, length: int, seed: int | None = None) -> Workload:
    """Fixed-length decode, no sharing: the >=4K-context target sweep (rows in {64,128,256}, L in {4096,8192})."""
    s = seed if seed is not None else 2000 + rows + length
    return make_decode(f"decode {rows} rows x {length}", [length] * rows, seed=s,
                       table_pages=_pages_for(length, DEFAULT_CONFIG["page_size"]))


def make_linear(tokens: int, in_features: int, out_features: int, seed: int):
    """x [tokens][in] ~ N(0,1) and w [out][in] ~ N(0, 1/in), both rounded to bf16
    (outputs of order 1, as a projection of a normed hidden state gives)."""
    gen = torch.Generator().manual_seed(seed)
    x = _randn_bf16(gen, (tokens, in_features))
    w = (torch.randn(out_features, in_features, generator=gen, dtype=torch.float32) / in_features ** 0.5).to(
        torch.bfloat16)
    return x, w
