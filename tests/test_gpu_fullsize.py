"""Parity at the full workload sizes, in the launch configuration the benchmark times
(same handle configuration, kernels and grids), on sampled outputs the fp64 oracle can
afford: one round from a synthetic pre-round state, every logit and IIR scan input of the
sampled sequences, the decisions (in the kernel's precision), and the sliced state
(kv_len, FIR tails, IIR states, the cache rows the round wrote)."""
import numpy as np
import pytest
import torch

from synth import gen_round, get_workload
from gpu_harness import Pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from lossless_speculative_verify_gb300.build import build
    build()


def _one_round(name, seqs, kv_dtype=np.float64):
    wl = get_workload(name)
    pair = Pair(wl, t_max=wl.prefix_len + 4 * wl.block)
    pair.import_synthetic(wl.prefix_len, kv_dtype=kv_dtype)
    out = pair.run_round(gen_round(wl, 0), seqs=seqs)
    pair.compare_state_light(seqs, rows_from=wl.prefix_len)
    assert pair.ver.flags() == 0
    assert pair.fp64_disagreements == 0, (out.gk, out.k, out.gc, out.corr, out.tie)
    return out


def test_full_size_d4096_l32_p8k_greedy():
    """32 layers, d=4096, 8192 cached tokens, gamma 12, greedy."""
    _one_round("d4096_l32_p8k_bf16", [0])


def test_full_size_d4096_l4_p256k_sampling():
    """Long context: 262144 cached tokens, 4 layers, gamma 6, sampling."""
    _one_round("d4096_l4_p256k_bf16", [0], kv_dtype=np.float32)


def test_full_size_b4c4_d4096_l8_p32k_sampling():
    """Four sequences x four candidate blocks, 32768 cached tokens each; the oracle checks
    one sequence (all four candidates; sequences are independent)."""
    _one_round("d4096_l8_p32k_b4c4_bf16", [2], kv_dtype=np.float32)
