"""Seeded synthetic inputs for the replay-free verify path.

This module is the only code shared by the fp64 oracle and the CUDA path. It draws
random numbers and fixes shapes; it holds none of the method's arithmetic (no layer
math, no softmax, no acceptance). Every array it returns is a plain NumPy array in
the math convention (row vector times matrix, ``y = x @ W``).
"""
from .workloads import Workload, LayerSpec, WORKLOADS, get_workload, ACGT_IDS
from .gen import (
    round_to_bf16,
    gen_weights,
    gen_prefix,
    gen_round,
    gen_state,
    gen_table_target,
)

__all__ = [
    "Workload", "LayerSpec", "WORKLOADS", "get_workload", "ACGT_IDS",
    "round_to_bf16", "gen_weights", "gen_prefix", "gen_round", "gen_state",
    "gen_table_target",
]
