"""The step's split of the SMs between the prompt attention and the rows'
attention: the rule the kernels compile (prompt_sms, prompt_tile_cost in
csrc/pkv_internal.h, built here into a small host program) against the
mirror the GPU tests use to know which path a case takes, on random and
edge-case inputs.  No GPU needed."""
import os
import random
import shutil
import subprocess

import pytest

from _harness import step_sm_split

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_gqa_qk_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <vector>
#include "pkv_internal.h"
// stdin: kv_heads sms P R, then P prompt lengths, then R step positions; stdout: kept resident
int main()
{
    int G, sms, P, R;
    if (scanf("%d %d %d %d", &G, &sms, &P, &R) != 4) return 1;
    std::vector<int> len(P), pos(R);
    for (auto& x : len) scanf("%d", &x);
    for (auto& x : pos) scanf("%d", &x);
    int64_t pc = 0, rows = 0;
    int pu = 0;
    for (int t0 = 0; t0 < P; t0 += 64) {
        int m = 0;
        for (int t = t0; t < P && t < t0 + 64; ++t) m = len[t] > m ? len[t] : m;
        pc += pkv::prompt_tile_cost(m, G);
        pu += m > 0 ? G : 0;
    }
    for (int p : pos) rows += p >= 0 ? p / pkv::kPageSize + 1 : 0;
    const int pgrid = sms < (P + 63) / 64 * G ? sms : (P + 63) / 64 * G;
    int kept = pkv::prompt_sms(pc, pkv::kSplitRowPage * G * rows, pu, sms);
    kept = kept < pgrid ? kept : pgrid;
    printf("%d %d\n", kept, kept < sms ? 2 * (sms - kept) : 2 * sms);
    return 0;
}
"""


@pytest.fixture(scope="module")
def rule(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("split_rule")
    src, exe = d / "rule.cu", d / "rule"
    src.write_text(PROGRAM)
    subprocess.run([nvcc, "-std=c++17", "-I", CSRC, "-o", str(exe), str(src)], check=True, capture_output=True)

    def run(lens, positions, G, sms):
        inp = f"{G} {sms} {len(lens)} {len(positions)}\n" + " ".join(map(str, lens)) + "\n" + \
              " ".join(map(str, positions)) + "\n"
        out = subprocess.run([str(exe)], input=inp, capture_output=True, text=True, check=True).stdout.split()
        return int(out[0]), int(out[1])
    return run


def test_rule_matches_the_mirror(rule):
    rng = random.Random(5)
    cases = [
        ([0] * 64, [100, 200], 8, 152),                      # prompts all skipped: no split
        ([10] * 5, [40000] * 64, 8, 152),                    # a small prompt beside long rows
        ([4096] * 2048, [10] * 4, 8, 152),                   # prompt-heavy: the rows keep few SMs, no split
        (list(range(1, 65)), [-1, -1], 8, 152),              # no step rows
    ]
    for _ in range(60):
        P = rng.randint(1, 3000)
        start = rng.randint(0, 8000)
        lens = [start + i + 1 if rng.random() > 0.05 else 0 for i in range(P)]
        R = rng.randint(1, 300)
        positions = [rng.randint(-1, 20000) for _ in range(R)]
        cases.append((lens, positions, rng.choice([2, 8, 16]), rng.choice([132, 148, 152])))
    splits = 0
    for lens, positions, G, sms in cases:
        got = rule(lens, positions, G, sms)
        assert got == step_sm_split(lens, positions, G, sms), (len(lens), len(positions), G, sms)
        splits += got[0] < sms
    assert splits > 10  # the random cases exercise the split, not only its absence
