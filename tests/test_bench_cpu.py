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


def test_stored_traffic_only_for_the_captured_case():
    # a stored ncu traffic figure belongs to one workload at its default sizes
    # and route tile: another route tile or a resized run reports none
    with open(os.path.join(ROOT, "profiles", "gemm1_traffic.json")) as f:
        tj = json.load(f)
    for name in ("decode_w4a16", "skewed_w4a16", "large_w4a16"):
        cfg = synth.CONFIGS[name]
        T = tj[name]["route_tile"]
        fam = bench.gemm_family(cfg, T, None)
        assert bench.stored_traffic(name, fam, 2 * T, cfg) == (None, None)
        assert bench.stored_traffic(name, fam, T, cfg.with_(M=cfg.M // 2)) == (None, None)
        got, src = bench.stored_traffic(name, fam, T, cfg)
        assert got is None or (got == tj[name]["dram_bytes_per_launch"] and src == tj[name]["source"])
