"""The benchmark's reference arm on CPU: `bench.py --impl reference` times the
fp64 oracle on the host's cores and prints the contract's JSON line (one line,
from rank 0 only under torchrun), and the timing rules refuse fewer than 3
warm-up steps."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout=300):
    return subprocess.run([sys.executable] + args, cwd=ROOT, capture_output=True, text=True, timeout=timeout)


def _json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_prints_one_contract_line():
    import bench
    p = _run(["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert p.returncode == 0, p.stderr[-2000:]
    lines = _json_lines(p.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "rows/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 1, 3)
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["vs_baseline"] is None
    # the default workload: the largest single-GPU decode batch (shared prefixes)
    assert d["config"]["workload"].startswith("shared-prefix decode 256 rows x U[1024,8192]")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_under_two_ranks_prints_from_rank_0_only():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    p = _run(["-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
              "--master-port", str(port), "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
              "--warmup", "3", "--workload", "config2"])
    assert p.returncode == 0, p.stderr[-2000:]
    lines = _json_lines(p.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def test_fewer_than_three_warmup_steps_are_refused():
    p = _run(["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "2"], timeout=120)
    assert p.returncode != 0 and "warmup" in (p.stderr + p.stdout)
