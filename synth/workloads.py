"""Workload shapes for the replay-free block-verification path.

The five named workloads follow the synthetic stand-ins for the EvSpark measurements
("EvSpark: Lossless Speculative Decoding for Hybrid DNA Foundation Models",
Interpretation, paragraphs 1 and 3; Perspective, paragraph 1): a hybrid
short-FIR / modal-IIR / causal-attention stack over a 512-entry byte vocabulary,
with DNA bases as prefix and draft tokens.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Tuple

# Byte-token ids of the four DNA bases in the 512-entry vocabulary.
ACGT_IDS = (65, 67, 71, 84)


@dataclass(frozen=True)
class LayerSpec:
    kind: str   # "fir" | "iir" | "attn"
    param: int  # FIR taps L | IIR poles per channel N | attention heads H


def _pattern(repeats: int, fir_a: int, fir_b: int, heads: int, poles: int = 16):
    one = (LayerSpec("fir", fir_a), LayerSpec("iir", poles), LayerSpec("fir", fir_b),
           LayerSpec("attn", heads))
    return one * repeats


@dataclass(frozen=True)
class Workload:
    name: str
    d: int
    layers: Tuple[LayerSpec, ...]
    head_dim: int
    dtype: str            # "f32" or "bf16" (weights, activations and KV)
    gamma: int
    batch: int
    n_cand: int
    prefix_len: int
    mode: str             # "greedy" or "sampling"
    seed_base: int        # weights 1000+s, prefix 2000+s, rounds 3000+s*10^4+r, state 4000+s
    vocab: int = 512
    temperature: float = 1.0
    q_alpha: float = 1.0  # Dirichlet concentration of the draft distribution over ACGT
    prefix_kind: str = "uniform"  # "uniform" or "markov3"
    prefill_chunk: int = 64
    cand_rule: str = "recursive"  # several candidates under sampling: "recursive" or "max_accept"

    # ---- derived sizes -------------------------------------------------------------
    @property
    def block(self) -> int:
        return self.gamma + 1

    @property
    def rows(self) -> int:
        return self.batch * self.n_cand * self.block

    @property
    def n_layers(self) -> int:
        return len(self.layers)

    def kinds(self, kind: str):
        return [i for i, s in enumerate(self.layers) if s.kind == kind]

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # tiny fp32 stack, CPU-seconds
    "tiny_d64_fp32": Workload(
        name="tiny_d64_fp32", d=64,
        layers=(LayerSpec("fir", 3), LayerSpec("iir", 16), LayerSpec("attn", 4)),
        head_dim=16, dtype="f32", gamma=6, batch=1, n_cand=1, prefix_len=256,
        mode="greedy", seed_base=1, q_alpha=1.0, prefill_chunk=64),
    # d=1024 bf16, 8 layers, P=8192, gamma=6, sampling
    "d1024_l8_p8k_bf16": Workload(
        name="d1024_l8_p8k_bf16", d=1024, layers=_pattern(2, 3, 3, 8), head_dim=128,
        dtype="bf16", gamma=6, batch=1, n_cand=1, prefix_len=8192, mode="sampling",
        seed_base=2, q_alpha=0.5, prefill_chunk=128),
    # d=4096 bf16, 32 layers, P=8192 (order-3 Markov prefix), gamma=12, greedy
    "d4096_l32_p8k_bf16": Workload(
        name="d4096_l32_p8k_bf16", d=4096, layers=_pattern(8, 3, 7, 32), head_dim=128,
        dtype="bf16", gamma=12, batch=1, n_cand=1, prefix_len=8192, mode="greedy",
        seed_base=3, q_alpha=1.0, prefix_kind="markov3", prefill_chunk=128),
    # long context: d=4096 bf16, 4 layers, P=262144, gamma=6, sampling
    "d4096_l4_p256k_bf16": Workload(
        name="d4096_l4_p256k_bf16", d=4096, layers=_pattern(1, 3, 7, 32), head_dim=128,
        dtype="bf16", gamma=6, batch=1, n_cand=1, prefix_len=262144, mode="sampling",
        seed_base=4, q_alpha=0.5, prefill_chunk=128),
    # batched multi-candidate: B=4 x C=4, d=4096 bf16, 8 layers, P=32768, gamma=12
    "d4096_l8_p32k_b4c4_bf16": Workload(
        name="d4096_l8_p32k_b4c4_bf16", d=4096, layers=_pattern(2, 3, 7, 32), head_dim=128,
        dtype="bf16", gamma=12, batch=4, n_cand=4, prefix_len=32768, mode="sampling",
        seed_base=5, q_alpha=0.5, prefill_chunk=64),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]
