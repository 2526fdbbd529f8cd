"""Replay-free speculative block verification on GB300 (sm_103a).

The compute path lives in ``libevs.so`` (hand-written CUDA, C-ABI in include/evs.h);
this package is its binding: ``Verifier`` (one handle), ``DeviceWeights`` (weights in
the library layout), ``make_config`` and ``build`` (compiles the library in-tree).
"""
from ._lib import EvsError, load
from .api import DeviceWeights, Verifier, make_config, workspace_bytes

__all__ = ["EvsError", "load", "DeviceWeights", "Verifier", "make_config", "workspace_bytes"]
