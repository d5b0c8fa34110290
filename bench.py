"""Benchmark of the paged-KV decode step (decode_paged) on GB300.

One step = one pkv_decode call over a batch: QK-norm + RoPE + KV append for
every row, split-KV attention over each row's pages, and the split combine.
The default workload is the largest single-GPU decode batch: 256 rows with
context lengths U[1024, 8192], in groups of 16 rows that share their first
8-32 pages (a shared prompt prefix), at Qwen3-8B attention shapes (32 query
heads, 8 kv heads, head_dim 128, pages of 64), synthetic and seeded.
Metric: decode rows/s (and the KV-read GB/s it implies, logical and unique),
with the attention kernel's achieved HBM bandwidth on unique bytes against
the measured copy bandwidth of the chip.  After the K timed steps the same
step runs back to back for a few seconds (the sustained pass) while the SM
clocks are sampled, and its median per-step time is reported beside
ms_per_step.

  python bench.py [--gpus N] [--steps K] [--warmup W]
                  [--workload config4|config2|config3|config5|sweepRxL|prefill|rows|linear_decode|linear_prefill|layer]
                  [--sustain-seconds S]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

Multi-GPU (torchrun, one rank per GPU): every rank runs its own batch of the
same shape (weak scaling, no data-path collective); the timed region is
bracketed by barriers and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode_paged rows/s and KV-read GB/s vs GB300 HBM roofline (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 126 << 20          # L2 of one GB300 as the driver reports it
L2_FLUSH_BYTES = 512 << 20
L2_CLEAN_BYTES = 256 << 20


def l2_flush(write_buf, read_buf):
    """Evict the step's inputs from L2: write a buffer larger than L2, then
    read another one, so that L2 is left holding clean lines (a kernel that
    follows pays no write-back of the flush's own dirty lines)."""
    import torch
    write_buf.zero_()
    torch.sum(read_buf)


# ---------------------------------------------------------------------------- distributed helpers

def dist_env():
    """(rank, world_size, local_rank) from the torchrun environment (1 process if absent)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch of the same shape (weak scaling)."""
    return base_seed + 7919 * rank


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------- workloads

def make_workload(name: str, rank: int = 0):
    import workloads as W
    if name == "config2":
        wl = W.make_decode("decode 64 rows x U[512,4096]", (64, 512, 4096), seed=rank_seed(1002, rank),
                           table_pages=64)
    elif name == "config3":
        wl = W.make_decode("long-context decode 8 rows x U[32768,40960]", (8, 32768, 40960),
                           seed=rank_seed(1003, rank), table_pages=640)
    elif name == "config4":
        wl = W.make_decode("shared-prefix decode 256 rows x U[1024,8192], groups of 16 share 8-32 pages",
                           (256, 1024, 8192), seed=rank_seed(1004, rank), table_pages=128, share_groups=16)
    elif name == "config5":
        wl = W.config5() if rank == 0 else None
        if wl is None:
            raise SystemExit("config5 runs on one rank")
    elif name == "prefill":
        wl = W.prefill_mix(seed=rank_seed(1006, rank))
    elif name == "rows":
        wl = W.rows_mix(seed=rank_seed(1007, rank))
    elif name == "short256":
        wl = W.make_decode("decode 256 short rows x U[1,1024]", (256, 1, 1024), seed=rank_seed(1008, rank),
                           table_pages=16)
    elif name.startswith("sweep"):
        r, l = name[5:].split("x")
        wl = W.sweep(int(r), int(l), seed=rank_seed(2000 + int(r) + int(l), rank))
    else:
        raise SystemExit(f"unknown workload {name}")
    return wl


# ---------------------------------------------------------------------------- measurement helpers

class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons sampled every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm"):
            if key in d:
                v = d[key]
                v = v.get("value", v) if isinstance(v, dict) else v
                return float(v), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def measured_peak_bf16():
    """Dense bf16 tensor TFLOP/s (burst) from the measured peaks, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        for key in ("bf16_tflops", "bf16_TFLOPs", "bf16"):
            if key in d:
                v = d[key]
                v = v.get("value", v) if isinstance(v, dict) else v
                return float(v), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash() -> str:
    """Hash of the decode attention kernel's sources (the kernel file and the headers it includes)."""
    h = hashlib.sha256()
    for name in ("pkv_kernels.cu", "pkv_rope.cuh", "pkv_ptx.cuh", "pkv_internal.h"):
        with open(os.path.join(ROOT, "paged_kv_gqa_qk_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per attention launch from the committed ncu summary, if the kernel is unchanged since."""
    p = os.path.join(ROOT, "profiles", "attn_kernel_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    sha = kernel_source_hash()
    for e in d.get("entries", []):
        if e.get("kernel_sha") == sha and e.get("workload") == workload:
            return e.get("dram_bytes_per_launch")
    return None


def prefill_algorithmic_flops(wl) -> int:
    """FLOPs the prompt-attention kernel must do per launch: for every prompt
    token at position p and every query head, scores against p + 1 keys and
    the weighted sum of p + 1 values, 2 * head_dim FLOPs each."""
    H, D = wl.cfg["heads"], wl.cfg["head_dim"]
    return sum(4 * H * D * (int(p) + 1) for p in wl.positions.tolist())


def attention_algorithmic_bytes(wl, unique: bool = True) -> int:
    """Bytes the decode attention kernel must move per launch: K and V of every
    attended position (4096 B each at 8 kv heads x 128 x bf16 x 2), and per
    row its page-table entries, its q (bf16, read), its new k and v (bf16,
    read, then written to the pool) and its bf16 output.  unique: a page that
    several rows share (a shared prefix) counts once."""
    import workloads as W
    S = wl.cfg["page_size"]
    L = [int(p) + 1 for p in wl.step_positions.tolist() if p >= 0]  # the rows the attention kernel serves
    kv = W.kv_bytes_per_position(wl.cfg) * sum(L)
    if unique and wl.meta.get("unique_kv_bytes") and wl.kind == "decode":
        # rows sharing prefix pages: each shared page counts once (later reads are L2 hits)
        kv = min(kv, wl.meta["unique_kv_bytes"])
    table = 4 * sum(-(-x // S) for x in L)
    H, G, D = wl.cfg["heads"], wl.cfg["kv_heads"], wl.cfg["head_dim"]
    per_row = 2 * (H * D + 2 * G * D + 2 * G * D + H * D)
    return kv + table + len(L) * per_row


def sustained_pass(step, flush, stream, ms_step_hint: float, seconds: float, block: int = 16) -> dict:
    """The same step back to back for about `seconds` (at least one block),
    timed with CUDA events on the launching stream: one pair per block of
    `block` steps when the inputs exceed L2, else one pair around each step
    with an L2 flush before it (outside the pair).  Returns the median and
    mean per-step time and the wall time the pass took."""
    import torch
    if seconds <= 0:
        return {"seconds": 0.0, "steps": 0}
    n = max(block, int(math.ceil(seconds * 1e3 / max(ms_step_hint, 1e-3))))
    n = (n + block - 1) // block * block
    per_step = []
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        if flush is None:
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(n // block + 1)]
            evs[0].record(stream)
            for b in range(n // block):
                for _ in range(block):
                    step()
                evs[b + 1].record(stream)
            stream.synchronize()
            per_step = [evs[b].elapsed_time(evs[b + 1]) / block for b in range(n // block)]
        else:
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
            for i in range(n):
                flush()
                evs[2 * i].record(stream)
                step()
                evs[2 * i + 1].record(stream)
            stream.synchronize()
            per_step = [evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(n)]
    wall = time.perf_counter() - t0
    return {"seconds": wall, "steps": n, "ms_per_step_median": statistics.median(per_step),
            "ms_per_step_mean": sum(per_step) / len(per_step),
            "timing": (f"CUDA events every {block} steps, back to back" if flush is None else
                       "CUDA events around each step, L2 flushed before each (outside the events)")}


# ---------------------------------------------------------------------------- the GPU arm

def packed(tensors, device=None, pin: bool = False):
    """One uint8 buffer holding copies of `tensors` back to back (each at a
    256-byte boundary) and views of it in their shapes and dtypes: on `device`,
    or in pinned host memory when pin.  Returns (buffer, views)."""
    import torch
    offs, off = [], 0
    for t in tensors:
        offs.append(off)
        off = (off + t.numel() * t.element_size() + 255) // 256 * 256
    flat = (torch.empty(off, dtype=torch.uint8, pin_memory=True) if pin
            else torch.empty(off, dtype=torch.uint8, device=device))
    views = []
    for t, o in zip(tensors, offs):
        v = flat[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return flat, views


def double_buffered_e2e(steps: int, sets, host_in, flush, stream, dev) -> float:
    """Wall-clock seconds of `steps` end-to-end steps.  sets[j] = (device inputs,
    run, device outputs, host outputs) for j = 0, 1: step i uses set i % 2; its
    inputs go up from the pinned host_in on one copy stream and its outputs come
    back on another, while the step before or after it runs on `stream`
    (event-fenced: a set's inputs are rewritten only after the step that read
    them, its outputs only after they were copied back)."""
    import torch
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    landed, done, fetched = ([torch.cuda.Event(), torch.cuda.Event()] for _ in range(3))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        j = i & 1
        d_in, run, d_out, h_out = sets[j]
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(done[j])
            for d, h in zip(d_in, host_in):
                d.copy_(h, non_blocking=True)
            landed[j].record(up)
        with torch.cuda.stream(stream):
            if flush is not None:
                flush()
            stream.wait_event(landed[j])
            if i >= 2:
                stream.wait_event(fetched[j])
            run()
            done[j].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(done[j])
            for h, d in zip(h_out, d_out):
                h.copy_(d, non_blocking=True)
            fetched[j].record(down)
    for st in (up, stream, down):
        st.synchronize()
    return time.perf_counter() - t0


E2E_COPIES = ("every step's inputs H2D (one copy: the inputs packed in one pinned buffer) and outputs D2H; "
              "two device buffer sets, step i+1's inputs and step i's outputs copied on their own streams while "
              "step i runs")


def run_gpu(args) -> None:
    import torch
    import paged_kv_gqa_qk_gb300 as pkv

    rank, world, local = dist_env()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    pkv.load_library()

    wl = make_workload(args.workload, rank)
    R, pages, P = wl.R, wl.pages, wl.P
    K, V = wl.K0.to(dev), wl.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
    # a prefill call takes the P prompt tokens only (its table rows take no step)
    ntok = P if wl.kind == "prefill" else P + R
    host_q, host_k, host_v = wl.q[:ntok], wl.k[:ntok], wl.v[:ntok]
    q, k, v, qw, kw, pos, tab = (t.to(dev) for t in (host_q, host_k, host_v, wl.q_norm_w, wl.k_norm_w,
                                                    wl.step_positions, wl.table))
    if wl.contiguous:
        tab = None   # the library's contiguous-row layout, no table
    out = torch.empty_like(q)
    ws = pool.workspace(0 if wl.kind == "prefill" else R, pages, P)
    stream = torch.cuda.Stream(device=dev)
    ppos = prow = None
    if wl.kind != "decode":
        ppos, prow = wl.positions.to(dev), wl.prow.to(dev)

    def make_step(b, o):
        """One call of the library on buffer set b = (q, k, v, pos, tab, ppos, prow), writing o."""
        bq, bk, bv, bpos, btab, bppos, bprow = b
        if wl.kind == "decode":
            return lambda: pkv.pkv_decode(pool.handle, bq, bk, bv, qw, kw, bpos, btab, o, ws, stream, pages=pages)
        if wl.kind == "step":  # step_paged: prompt chunks + one step per row
            return lambda: pkv.pkv_step(pool.handle, bq, bk, bv, qw, kw, bppos, bprow, None, bpos, btab, o, ws, stream,
                                        pages=pages)
        # prefill_paged: prompt chunks only
        return lambda: pkv.pkv_prefill(pool.handle, bq, bk, bv, qw, kw, bppos, bprow, None, btab, o, ws, stream,
                                       rows=R, pages=pages)

    bufs = (q, k, v, pos, tab, ppos, prow)
    step = make_step(bufs, out)
    # decode: attention, combine; step: prep, prompt attention, step-row attention, combine;
    # prefill: prep, prompt attention
    launches_per_step = {"decode": 2, "step": 4}.get(wl.kind, 2)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    flags = pkv.pkv_check_errors(pool.handle, stream)
    if flags:
        raise SystemExit(f"device error flags {flags}")

    # ---- device-timed region, inputs resident in HBM.  Pass 1 times the steps
    # as a user runs them (no events between the kernels, which would break
    # their programmatic overlap); pass 2 times the attention kernel alone
    # with events around each launch, for the roofline.
    # Workloads whose K/V fit in L2 flush it (a write larger than L2, outside
    # the timed events) before every timed step.
    logical = wl.meta["logical_kv_bytes"]
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if logical < 2 * L2_BYTES else None
    clean_buf = torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32, device=dev) if flush_buf is not None else None

    def flush():
        if flush_buf is not None:
            with torch.cuda.stream(stream):
                l2_flush(flush_buf, clean_buf)

    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 if flush_buf is None else 2 * args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        if flush_buf is None:
            evs[0].record(stream)
            for _ in range(args.steps):
                step()
            evs[1].record(stream)
        else:
            for i in range(args.steps):
                flush()
                evs[2 * i].record(stream)
                step()
                evs[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        pkv.pkv_timer_enable(pool.handle, True)
        for _ in range(args.steps):
            flush()
            step()
        torch.cuda.synchronize()
        attn_ms, attn_n = pkv.pkv_timer_read(pool.handle)
        pkv.pkv_timer_enable(pool.handle, False)
        ms_first = sum(evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(len(evs) // 2)) / args.steps
        sustained = sustained_pass(step, flush if flush_buf is not None else None, stream, ms_first,
                                   args.sustain_seconds)
    barrier(world)
    ms_total = sum(evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(len(evs) // 2))
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps

    # ---- end-to-end through the C ABI with host buffers: inputs H2D from pinned
    # memory and the output D2H, every step, inside the timed region.  As a serving
    # loop would, it keeps two device buffer sets: step i+1's inputs go up on one copy
    # stream and step i's output comes back on another while step i runs.
    # The step's inputs sit back to back in one pinned host buffer and one device
    # buffer per set, so that a step's upload is one copy.
    names = ["q", "k", "v"]
    srcs = [host_q, host_k, host_v]
    if wl.kind != "prefill":
        names.append("pos")
        srcs.append(wl.step_positions)
    if tab is not None:
        names.append("tab")
        srcs.append(wl.table)
    if wl.kind != "decode":
        names += ["ppos", "prow"]
        srcs += [wl.positions, wl.prow]
    host_flat, _ = packed(srcs, pin=True)
    host_out = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    h2d = host_flat.numel()
    d2h = host_out[0].numel() * host_out[0].element_size()
    sets = []
    for j in range(2):
        dev_flat, views = packed(srcs, device=dev)
        vb = dict(zip(names, views))
        bset = tuple(vb.get(n) for n in ("q", "k", "v", "pos", "tab", "ppos", "prow"))
        o = torch.empty_like(out)
        sets.append(([dev_flat], make_step(bset, o), [o], [host_out[j]]))
    host_in = [host_flat]
    barrier(world)
    e2e_s = double_buffered_e2e(args.steps, sets, host_in, flush, stream, dev)
    e2e_s = max_over_ranks(e2e_s, world)
    barrier(world)
    flags = pkv.pkv_check_errors(pool.handle, stream)
    if flags:
        raise SystemExit(f"device error flags {flags}")

    attn_avg_s = attn_ms / 1e3 / max(attn_n, 1)
    timing = "CUDA events around each timed launch, second timed pass of the same steps"
    if wl.kind == "prefill":
        flops = prefill_algorithmic_flops(wl)
        peak, peak_kind = measured_peak_bf16()
        roofline = {"bound": "tensor", "kernel": "prefill_kernel", "achieved": flops / attn_avg_s / 1e12,
                    "peak": peak, "peak_kind": f"{peak_kind} (dense bf16 TFLOP/s, burst)", "unit": "TFLOP/s",
                    "frac": flops / attn_avg_s / 1e12 / peak, "traffic": None,
                    "algorithmic_flops_per_launch": flops, "avg_launch_us": attn_avg_s * 1e6,
                    "timed_launches": attn_n, "timing": timing}
    else:
        plan_bytes = attention_algorithmic_bytes(wl)
        achieved = plan_bytes / attn_avg_s / 1e9
        peak, peak_kind = measured_peak_hbm()
        logical_bytes = attention_algorithmic_bytes(wl, unique=False)
        roofline = {"bound": "hbm", "kernel": "attn_kernel", "achieved": achieved, "peak": peak,
                    "peak_kind": f"{peak_kind} (hbm copy GB/s)", "unit": "GB/s", "frac": achieved / peak,
                    "traffic": ncu_traffic(args.workload), "algorithmic_bytes_per_launch": plan_bytes,
                    "bytes_counted": ("unique: each shared prefix page once" if logical_bytes != plan_bytes
                                      else "every attended position"),
                    "achieved_logical": logical_bytes / attn_avg_s / 1e9,
                    "avg_launch_us": attn_avg_s * 1e6, "timed_launches": attn_n, "timing": timing}
    # value: decode rows per second (a step's prompt tokens are reported beside it);
    # a prefill-only call has no decode rows and reports prompt tokens per second
    n_decode = int((wl.step_positions >= 0).sum()) if wl.kind != "prefill" else 0
    rows_total = (P if wl.kind == "prefill" else n_decode) * world
    unit = "tokens/s" if wl.kind == "prefill" else "rows/s"
    res = {
        "metric": METRIC,
        "value": rows_total / (ms_step / 1e3),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v/cache, U[0.5,1.5] norm weights, shuffled pages)",
        "config": {"workload": wl.name, "rows": R, "prompt_tokens": P, "table_pages": pages,
                   "pool_pages": wl.num_pages,
                   "heads": wl.cfg["heads"], "kv_heads": wl.cfg["kv_heads"], "head_dim": wl.cfg["head_dim"],
                   "page_size": wl.cfg["page_size"],
                   "sum_context": sum(wl.meta.get("lengths", wl.meta.get("decode_lengths", []))),
                   "kv_bytes_per_step": logical,
                   "l2": (f"inputs larger than L2: {logical / 1e9:.2f} GB of K/V per step vs 126 MB L2"
                          if flush_buf is None else
                          f"L2 flushed before every timed step ({L2_FLUSH_BYTES >> 20} MiB write, then a "
                          f"{L2_CLEAN_BYTES >> 20} MiB read so that L2 holds clean lines; outside the "
                          f"device-timed events, inside the e2e time): {logical / 1e6:.0f} MB of K/V per step"),
                   "parallelism": f"dp{world} (independent replicas, rows sharded by rank)"},
        "kv_gbs": logical / (ms_step / 1e3) / 1e9 * world,
        "kv_gbs_unique": wl.meta.get("unique_kv_bytes", logical) / (ms_step / 1e3) / 1e9 * world,
        "roofline": roofline,
        "e2e": {"value": rows_total * args.steps / e2e_s, "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "copies": E2E_COPIES},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "sustained": sustained,
        "gpu": torch.cuda.get_device_name(dev),
    }
    if wl.kind == "step":
        res["prompt_tokens_per_s"] = P * world / (ms_step / 1e3)
        res["config"]["decode_rows"] = n_decode
    if rank == 0 and world == 1 and not args.no_cpu_baseline and wl.kind == "decode":
        res["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)
    pool.close()
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------- the projections (pkv_linear)

LINEAR_SHAPES = (("q_proj", 4096, 4096), ("k_proj", 1024, 4096), ("v_proj", 1024, 4096), ("o_proj", 4096, 4096))
# one step: q/k/v fused in one launch (pkv_qkv_proj), then o_proj (pkv_linear)


def run_gpu_linear(args) -> None:
    """The four projections around one attention layer (q/k/v before it, o_proj
    after it) for `tokens` tokens: 64 (the decode batch) or 2048 (the prompts of
    the step workload).  One step = pkv_qkv_proj (q, k, v in one launch) and
    pkv_linear (o_proj)."""
    import torch
    import paged_kv_gqa_qk_gb300 as pkv
    import workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    pkv.load_library()
    tokens = {"linear_decode": 64, "linear_prefill": 2048}[args.workload]
    pool = pkv.PagedKVPool(torch.zeros(8, 64, 128, dtype=torch.bfloat16, device=dev),
                           torch.zeros(8, 64, 128, dtype=torch.bfloat16, device=dev))
    host_x, _ = W.make_linear(tokens, 4096, 128, seed=rank_seed(3000 + tokens, rank))
    host_a, _ = W.make_linear(tokens, 4096, 128, seed=rank_seed(3001 + tokens, rank))  # the attention output
    ws = [W.make_linear(1, i, o, seed=rank_seed(3100 + j, rank))[1].to(dev) for j, (_, o, i) in enumerate(LINEAR_SHAPES)]
    w_qkv = torch.cat(ws[:3], 0).contiguous()
    x, a = host_x.to(dev), host_a.to(dev)
    ys = [torch.empty(tokens, o, dtype=torch.bfloat16, device=dev) for _, o, _ in LINEAR_SHAPES]
    q, k, v = (ys[0].view(tokens, 32, 128), ys[1].view(tokens, 8, 128), ys[2].view(tokens, 8, 128))
    stream = torch.cuda.Stream(device=dev)

    def make_step(xb, ab, yb):
        qb, kb, vb = (yb[0].view(tokens, 32, 128), yb[1].view(tokens, 8, 128), yb[2].view(tokens, 8, 128))

        def run():
            pool.qkv_proj(xb, w_qkv, qb, kb, vb, stream=stream)
            pool.linear(ab, ws[3], yb[3], stream=stream)
        return run

    step = make_step(x, a, ys)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)  # the weights (84 MB) fit in L2
    clean_buf = torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        with torch.cuda.stream(stream):
            l2_flush(flush_buf, clean_buf)

    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush()
            evs[2 * i].record(stream)
            step()
            evs[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        pkv.pkv_timer_enable(pool.handle, True)
        for _ in range(args.steps):
            flush()
            step()
        torch.cuda.synchronize()
    barrier(world)
    ms_step = max_over_ranks(sum(evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(args.steps)), world) / args.steps
    k_ms, k_n = pkv.pkv_timer_read(pool.handle)
    pkv.pkv_timer_enable(pool.handle, False)

    host_in = [host_x.pin_memory(), host_a.pin_memory()]
    host_out = [[torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for y in ys] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    x2, a2, ys2 = x.clone(), a.clone(), [torch.empty_like(y) for y in ys]
    sets = [([x, a], make_step(x, a, ys), ys, host_out[0]), ([x2, a2], make_step(x2, a2, ys2), ys2, host_out[1])]
    barrier(world)
    e2e_s = double_buffered_e2e(args.steps, sets, host_in, flush, stream, dev)
    e2e_s = max_over_ranks(e2e_s, world)
    flags = pkv.pkv_check_errors(pool.handle, stream)
    if flags:
        raise SystemExit(f"device error flags {flags}")

    weight_bytes = sum(2 * o * i for _, o, i in LINEAR_SHAPES)
    act_bytes = sum(2 * tokens * (i + o) for _, o, i in LINEAR_SHAPES)
    flops = sum(2 * tokens * o * i for _, o, i in LINEAR_SHAPES)
    kern_s = k_ms / 1e3 / max(k_n, 1) * 2  # the two launches of one step
    timing = "CUDA events around each matrix-product launch (two per step), second timed pass"
    if tokens <= 256:   # weight streaming: bound by HBM
        peak, peak_kind = measured_peak_hbm()
        roofline = {"bound": "hbm", "kernel": "linear_kernel", "achieved": (weight_bytes + act_bytes) / kern_s / 1e9,
                    "peak": peak, "peak_kind": f"{peak_kind} (hbm copy GB/s)", "unit": "GB/s",
                    "algorithmic_bytes_per_step": weight_bytes + act_bytes}
    else:
        peak, peak_kind = measured_peak_bf16()
        roofline = {"bound": "tensor", "kernel": "linear_kernel", "achieved": flops / kern_s / 1e12,
                    "peak": peak, "peak_kind": f"{peak_kind} (dense bf16 TFLOP/s, burst)", "unit": "TFLOP/s",
                    "algorithmic_flops_per_step": flops}
    roofline.update({"frac": roofline["achieved"] / peak, "traffic": None,
                     "avg_launch_us": k_ms * 1e3 / max(k_n, 1), "timed_launches": k_n, "timing": timing})
    res = {
        "metric": METRIC,
        "value": tokens * world / (ms_step / 1e3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 activations, N(0,1/4096) bf16 weights)",
        "config": {"workload": f"projections q/k/v/o of one layer, {tokens} tokens, hidden 4096",
                   "tokens": tokens, "shapes": [list(s) for s in LINEAR_SHAPES],
                   "l2": f"L2 flushed before every timed step ({L2_FLUSH_BYTES >> 20} MiB write, then a "
                      f"{L2_CLEAN_BYTES >> 20} MiB read so that L2 holds clean lines; outside the device-timed "
                      f"events, inside the e2e time): {weight_bytes / 1e6:.0f} MB of weights",
                   "parallelism": f"dp{world} (independent replicas)"},
        "roofline": roofline,
        "e2e": {"value": tokens * args.steps * world / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "copies": E2E_COPIES},
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
        "gpu": torch.cuda.get_device_name(dev),
    }
    pool.close()
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------- one attention layer

def run_gpu_layer(args) -> None:
    """One decode step of a whole attention layer over the 64-row batch (context
    U[512,4096]) at Qwen3-8B's hidden size 4096, on synthetic weights: the q/k/v
    projection with QK-norm, RoPE and the k/v append in its epilogue
    (pkv_qkv_proj_append), the attention over the pool it wrote
    (pkv_decode_appended) and o_proj (pkv_linear) -- 3 launches of ours plus
    the attention's combine.  The same step through the unfused entries
    (pkv_qkv_proj, pkv_decode, pkv_linear) is timed beside it."""
    import torch
    import paged_kv_gqa_qk_gb300 as pkv
    import workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    pkv.load_library()
    wl = make_workload("config2", rank)
    R, pages = wl.R, wl.pages
    K, V = wl.K0.to(dev), wl.V0.to(dev)
    pool = pkv.PagedKVPool(K, V, cfg=wl.cfg)
    hidden = 4096
    host_x, _ = W.make_linear(R, hidden, 128, seed=rank_seed(3200, rank))
    w_qkv = W.make_linear(1, hidden, 6144, seed=rank_seed(3201, rank))[1].to(dev)
    w_o = W.make_linear(1, hidden, hidden, seed=rank_seed(3202, rank))[1].to(dev)
    x = host_x.to(dev)
    qw, kw, pos, tab = (t.to(dev) for t in (wl.q_norm_w, wl.k_norm_w, wl.step_positions, wl.table))
    q_hat = torch.empty(R, 32, 128, dtype=torch.float32, device=dev)
    attn = torch.empty(R, 32, 128, dtype=torch.bfloat16, device=dev)
    y = torch.empty(R, hidden, dtype=torch.bfloat16, device=dev)
    q, k, v = (torch.empty(R, h, 128, dtype=torch.bfloat16, device=dev) for h in (32, 8, 8))
    ws = pool.workspace(R, pages, 0)
    stream = torch.cuda.Stream(device=dev)

    def make_fused(xb, yb):
        def run():
            pkv.pkv_qkv_proj_append(pool.handle, xb, w_qkv, qw, kw, pos, tab, q_hat, stream)
            pkv.pkv_decode_appended(pool.handle, q_hat, pos, tab, attn, ws, stream)
            pkv.pkv_linear(pool.handle, attn.view(R, hidden), w_o, yb, None, stream)
        return run

    step_fused = make_fused(x, y)

    def step_unfused():
        pkv.pkv_qkv_proj(pool.handle, x, w_qkv, q, k, v, stream)
        pkv.pkv_decode(pool.handle, q, k, v, qw, kw, pos, tab, attn, ws, stream)
        pkv.pkv_linear(pool.handle, attn.view(R, hidden), w_o, y, None, stream)

    def timed(step, n):
        with torch.cuda.stream(stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                step()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) / n

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step_fused()
            step_unfused()
    stream.synchronize()
    if pkv.pkv_check_errors(pool.handle, stream):
        raise SystemExit("device error flags")
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms_step = max_over_ranks(timed(step_fused, args.steps), world)
        ms_unfused = max_over_ranks(timed(step_unfused, args.steps), world)
        pkv.pkv_timer_enable(pool.handle, 2)   # events around the attention launch only
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                step_fused()
        stream.synchronize()
        attn_ms, attn_n = pkv.pkv_timer_read(pool.handle)
        pkv.pkv_timer_enable(pool.handle, False)
        sustained = sustained_pass(step_fused, None, stream, ms_step, args.sustain_seconds)
    barrier(world)

    host_in = [host_x.pin_memory()]
    host_out = [[torch.empty(y.shape, dtype=y.dtype, pin_memory=True)] for _ in range(2)]
    x2, y2 = x.clone(), torch.empty_like(y)
    sets = [([x], make_fused(x, y), [y], host_out[0]), ([x2], make_fused(x2, y2), [y2], host_out[1])]
    barrier(world)
    e2e_s = double_buffered_e2e(args.steps, sets, host_in, None, stream, dev)
    e2e_s = max_over_ranks(e2e_s, world)
    if pkv.pkv_check_errors(pool.handle, stream):
        raise SystemExit("device error flags")

    S = wl.cfg["page_size"]
    L = [int(p) + 1 for p in wl.step_positions.tolist()]
    kv = W.kv_bytes_per_position(wl.cfg) * sum(L)
    attn_bytes = kv + 4 * sum(-(-n // S) for n in L) + R * (32 * 128 * 4 + 32 * 128 * 2)  # K/V, table, q_hat, out
    attn_s = attn_ms / 1e3 / max(attn_n, 1)
    peak, peak_kind = measured_peak_hbm()
    weight_bytes = 2 * hidden * (6144 + hidden)
    res = {
        "metric": METRIC,
        "value": R * world / (ms_step / 1e3),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 activations and cache, N(0,1/4096) bf16 weights, shuffled pages)",
        "config": {"workload": "attention layer decode step, 64 rows x U[512,4096], hidden 4096: q/k/v projection "
                               "with norm, RoPE and append fused, attention, o_proj",
                   "rows": R, "hidden": hidden, "table_pages": pages, "sum_context": sum(L),
                   "bytes_per_step": {"kv": kv, "weights": weight_bytes},
                   "l2": f"inputs larger than L2: {(kv + weight_bytes) / 1e9:.2f} GB of K/V and weights per step",
                   "parallelism": f"dp{world} (independent replicas)"},
        "unfused_ms_per_step": ms_unfused,
        "roofline": {"bound": "hbm", "kernel": "attn_kernel", "achieved": attn_bytes / attn_s / 1e9, "peak": peak,
                     "peak_kind": f"{peak_kind} (hbm copy GB/s)", "unit": "GB/s",
                     "frac": attn_bytes / attn_s / 1e9 / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": attn_bytes, "avg_launch_us": attn_s * 1e6,
                     "timed_launches": attn_n,
                     "timing": "CUDA events around each attention launch, a separate pass of the same steps"},
        "layer_gbs": (kv + weight_bytes) / (ms_step / 1e3) / 1e9,
        "e2e": {"value": R * args.steps * world / e2e_s, "unit": "rows/s", "h2d_bytes_per_step": host_in[0].numel() * 2,
                "d2h_bytes_per_step": host_out[0][0].numel() * 2, "copies": E2E_COPIES},
        "gpu_launches": 4 * args.steps,
        "clocks": clk.summary(),
        "sustained": sustained,
        "gpu": torch.cuda.get_device_name(dev),
    }
    pool.close()
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------- the oracle (CPU)

def _oracle_step(wl, rows, K, V, args_bits, nthreads):
    import numpy as np
    import oracle
    sel = np.asarray(rows, dtype=np.int32)
    oracle.decode(K, V, *args_bits, wl.step_positions.numpy(), wl.table.numpy(), cfg=wl.cfg, sel=sel,
                  nthreads=nthreads)


def cpu_baseline(wl, budget_s: float = 10.0) -> dict:
    """The fp64 oracle, as it stands, on the host's cores: whole decode steps over
    a bounded sample of the rows (the first rows of the same batch), repeated
    until about budget_s seconds of CPU work."""
    import workloads as W
    nthreads = os.cpu_count() or 1
    K, V = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    args_bits = [W.bits(t) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w)]
    n = min(wl.R, 8)
    rows = list(range(n))
    done = 0
    t0 = time.perf_counter()
    while True:
        _oracle_step(wl, rows, K, V, args_bits, nthreads)
        done += n
        el = time.perf_counter() - t0
        if el >= budget_s or done >= 64 * wl.R:
            break
    # the same on one core, over the first row, for about a fifth of the budget
    done1, t1 = 0, time.perf_counter()
    while True:
        _oracle_step(wl, [0], K, V, args_bits, 1)
        done1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= budget_s / 5 or done1 >= 64:
            break
    return {"value": done / el, "unit": "rows/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{n} rows (all 32 heads) of the same batch per pass, {done // n} passes, {el:.1f} s; "
                      f"every pass also writes all {wl.R} rows' k/v",
            "one_core": {"value": done1 / el1, "unit": "rows/s", "cores": 1,
                         "sample": f"row 0 of the batch, {done1} passes, {el1:.1f} s"}}


def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import workloads as W
    wl = make_workload(args.workload, 0)
    nthreads = os.cpu_count() or 1
    K, V = W.bits(wl.K0).copy(), W.bits(wl.V0).copy()
    args_bits = [W.bits(t) for t in (wl.q, wl.k, wl.v, wl.q_norm_w, wl.k_norm_w)]
    n = min(wl.R, 8)
    rows = list(range(n))
    for _ in range(args.warmup):
        _oracle_step(wl, rows, K, V, args_bits, nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(wl, rows, K, V, args_bits, nthreads)
    el = time.perf_counter() - t0
    value = n * args.steps / el
    res = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same seeded workload as the GPU arm)",
        "config": {"workload": wl.name, "rows": wl.R, "table_pages": wl.pages,
                   "sample_rows_per_step": n},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": nthreads, "kind": "oracle",
                         "sample": f"{n} rows (all 32 heads) of the batch per step; each step also writes all "
                                   f"{wl.R} rows' k/v"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    ap.add_argument("--workload", default="config4")
    ap.add_argument("--sustain-seconds", type=float, default=2.0,
                    help="length of the back-to-back pass after the timed steps (0: none)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload.startswith("linear"):
        run_gpu_linear(args)
    elif args.workload == "layer":
        run_gpu_layer(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
