"""bench.py's host-side legs on the CPU: the reference arm (the oracle timed
on the host cores over bounded samples) and the bounded cpu_baseline timer."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_w4a16", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["config"]["workload"] == "tiny_w4a16" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_bounded_oracle_timer_uses_a_prefix_of_the_sample():
    cfg = synth.CONFIGS["tiny_w4a16"]
    inp = synth.generate(cfg)
    orc = oracle.OracleMoE.from_inputs(inp, T=16)
    toks = bench.oracle_tokens(cfg, inp)
    assert np.array_equal(toks, np.arange(cfg.M))
    v, dt, cores, n, runs = bench.time_oracle_bounded(orc, toks, budget_s=0.5)
    assert 1 <= n <= cfg.M and 1 <= cores <= n and 1 <= runs <= 3
    assert v == n / dt
    big = synth.CONFIGS["large_w4a16"]
    assert big.sample == 1024      # the large workload is timed on its seeded sample
