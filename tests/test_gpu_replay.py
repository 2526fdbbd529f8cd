"""Replay-based recovery (evs_replay_state), the ablation that state slicing replaces
(EvSpark summary, Interpretation: slicing against a second target forward over the
accepted prefix). From the same pre-round state and the same verify, replaying the
accepted tokens must leave the state that slicing leaves: both are compared with the fp64
oracle's committed state (kv_len exact; tails, IIR states and K/V rows to 1e-5 fp32 /
2e-2 bf16)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_harness import Pair
from synth import LayerSpec, gen_round, get_workload
from test_gpu_parity import identity_drafts

pytestmark = pytest.mark.gpu


def _slice_then_replay(pair, rnd):
    """Verify + slice (checked against the oracle, which commits the same k), then the same
    verify from the same state followed by a replay instead of the slice."""
    wl = pair.wl
    pre = pair.ver.export_state()
    out = pair.run_round(rnd)
    pair.compare_state()
    dev = lambda a, dt: torch.as_tensor(a, dtype=dt).cuda().contiguous()
    toks = dev(rnd["tokens"], torch.int32)
    sampling = wl.mode == "sampling"
    q = dev(rnd["q"], torch.float32) if sampling else None
    u = dev(rnd["u"], torch.float32) if sampling else None
    pair.ver.import_state(pre)
    k, corr, cand, _ = pair.ver.verify(toks, q, u)
    pair.ver.replay(toks, k, cand)
    torch.cuda.synchronize()
    assert int(k.item()) == int(out.gk[0]) and int(corr.item()) == int(out.gc[0])
    pair.compare_state()
    return out


@pytest.mark.parametrize("k_force", [0, 3, 6])
def test_replay_equals_slice_tiny_fp32(k_force):
    wl = get_workload("tiny_d64_fp32")
    pair = Pair(wl)
    pair.import_synthetic(40)
    rnd = gen_round(wl, 7)
    rnd["tokens"] = identity_drafts(pair, rnd, wrong_at=k_force if k_force < wl.gamma else None)
    out = _slice_then_replay(pair, rnd)
    assert out.gk[0] == k_force


def test_replay_equals_slice_multi_candidate_fp32():
    wl = get_workload("tiny_d64_fp32").replace(n_cand=3, gamma=5)
    pair = Pair(wl)
    pair.import_synthetic(48)
    rnd = gen_round(wl, 1)
    rnd["tokens"] = identity_drafts(pair, rnd, wrong_at=[1, 4, 2])
    out = _slice_then_replay(pair, rnd)
    assert out.gcand[0] == 1 and out.gk[0] == 4


def test_replay_equals_slice_bf16_sampling():
    wl = get_workload("d1024_l8_p8k_bf16").replace(d=256, head_dim=128, prefix_len=300,
        layers=(LayerSpec("fir", 3), LayerSpec("iir", 16), LayerSpec("fir", 7), LayerSpec("attn", 2)))
    pair = Pair(wl)
    pair.prefill(wl.prefix_len)
    for r in range(3):
        _slice_then_replay(pair, gen_round(wl, r))


def test_replay_host_errors():
    from lossless_speculative_verify_gb300 import EvsError
    wl = get_workload("tiny_d64_fp32")
    pair = Pair(wl)
    toks = torch.as_tensor(gen_round(wl, 0)["tokens"], dtype=torch.int32).cuda()
    with pytest.raises(EvsError):          # no verify to replay
        pair.ver.replay(toks)
    wl2 = wl.replace(batch=2)
    pair2 = Pair(wl2)
    toks2 = torch.as_tensor(gen_round(wl2, 0)["tokens"], dtype=torch.int32).cuda()
    pair2.ver.verify(toks2)
    with pytest.raises(EvsError):          # one sequence only
        pair2.ver.replay(toks2)
    torch.cuda.synchronize()
    assert pair.ver.flags() == 0 and pair2.ver.flags() == 0
