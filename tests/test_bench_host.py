"""Host-side checks of bench.py (no GPU): the reference arm, the fp64 oracle timed on the
host cores, prints one JSON line with the contract's keys; the byte model counts what the
round's kernels must move at least once."""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_d64_fp32",
                          "--steps", "2", "--warmup", "1", "--cpu-seconds", "0.5"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300, check=True)
    lines = [l for l in out.stdout.strip().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_round_bytes_min_counts_weights_kv_and_state():
    import bench
    from synth import get_workload
    wl = get_workload("d4096_l4_p256k_bf16")
    P = wl.prefix_len
    b = bench.round_bytes_min(wl, P)
    # weights of one [FIR-3, IIR-16, FIR-7, attention] pattern and the head, bf16
    w = (2 * 4096 * 4096 * 3 + 4 * 4096 * 4096 + 512 * 4096) * 2
    kv = 2 * P * 4096 * 2                          # K and V of every cached token, read once
    assert b > w + kv
    assert b < (w + kv) * 1.01                     # states and new rows are small beside them
    assert bench.kind_bytes(wl, P, "attn") == bench.kv_read_bytes(wl, P) == kv
