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


def test_oracle_sample_by_blocks_equals_verify_round():
    """The CPU baseline takes a round one candidate block at a time; its decisions and the
    committed state equal the oracle's whole-round call on the same inputs."""
    import numpy as np
    import bench
    import oracle
    from synth import gen_round, get_workload
    wl = get_workload("tiny_d64_fp32").replace(batch=1, n_cand=3, gamma=4, mode="sampling", q_alpha=0.5,
                                               prefix_len=40)
    smp = bench.OracleSample(wl)
    ref = [smp.state[0].clone()]
    anchor = None
    for r in range(4):
        rnd = gen_round(smp.wl1, r, anchor=anchor)
        want = oracle.verify_round(smp.tgt, ref, rnd["tokens"], rnd["q"], rnd["u"], wl.mode, wl.temperature,
                                   rule=wl.cand_rule)
        got = [smp.block() for _ in range(wl.n_cand)]
        assert got[:-1] == [0] * (wl.n_cand - 1) and got[-1] == int(want.k[0]) + 1
        assert smp.anchor[0] == want.corr[0]
        anchor = want.corr
        for a, b in zip(smp.state[0].layers, ref[0].layers):
            if a["kind"] == "attn":
                assert a["kv"].length == b["kv"].length
                np.testing.assert_array_equal(a["kv"].k[:, :a["kv"].length], b["kv"].k[:, :b["kv"].length])
            else:
                key = "tail" if a["kind"] == "fir" else "s"
                np.testing.assert_array_equal(a[key], b[key])
