"""The C-ABI library loads and exports every entry point include/evs.h declares; host-side
validation works without a GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from lossless_speculative_verify_gb300.build import build
    from lossless_speculative_verify_gb300 import _lib
    build()
    return _lib.load()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(evs_[a-z_0-9]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "evs_verify_block" in names and "evs_slice_state" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def _cfg(**kw):
    from lossless_speculative_verify_gb300 import make_config
    base = dict(d=64, layers=[("fir", 3), ("iir", 16), ("attn", 4)], head_dim=16, gamma=6, batch=1,
                n_cand=1, t_max=512, prefill_chunk=64, dtype="f32", mode="greedy")
    base.update(kw)
    return make_config(**base)


def test_workspace_bytes_and_validation(lib):
    from lossless_speculative_verify_gb300 import workspace_bytes
    ok = workspace_bytes(_cfg())
    assert ok > 0 and ok % 256 == 0
    assert workspace_bytes(_cfg(t_max=1024)) > ok              # KV grows with capacity
    assert workspace_bytes(_cfg(d=65)) == 0                    # width not a multiple of 64
    assert workspace_bytes(_cfg(head_dim=32)) == 0             # H * dh != d
    assert workspace_bytes(_cfg(gamma=0)) == 0
    assert workspace_bytes(_cfg(layers=[("iir", 3)])) == 0     # poles not a power of two
    assert workspace_bytes(_cfg(vocab=500)) == 0
    bad_rule = _cfg()
    bad_rule.cand_rule = 2
    assert workspace_bytes(bad_rule) == 0                      # unknown candidate rule


def test_iir_workspace_keeps_inputs_not_states(lib):
    """A verify keeps the IIR scan inputs ([B][C][gamma+1][d] fp32) for slicing, not every
    state: more poles grow the workspace by the carried state [B][d][N] complex only."""
    from lossless_speculative_verify_gb300 import workspace_bytes
    al = lambda x: (x + 255) // 256 * 256
    for B, C, g in [(1, 1, 6), (2, 3, 5)]:
        kw = dict(batch=B, n_cand=C, gamma=g, d=64)
        w1 = workspace_bytes(_cfg(layers=[("iir", 1)], **kw))
        w16 = workspace_bytes(_cfg(layers=[("iir", 16)], **kw))
        assert w16 - w1 == al(B * 64 * 16 * 8) - al(B * 64 * 1 * 8)


def test_entry_points_reject_a_null_handle(lib):
    from lossless_speculative_verify_gb300 import _lib
    null = ctypes.c_void_p()
    assert lib.evs_decode_step(null, null, null, null, null) == _lib.EVS_ERR_INVALID_ARG
    assert lib.evs_replay_state(null, null, null, null, null) == _lib.EVS_ERR_INVALID_ARG
    assert lib.evs_slice_state(null, null, null) == _lib.EVS_ERR_INVALID_ARG
    assert lib.evs_verify_block(null, null, null, null, null, null, null, null, null) == _lib.EVS_ERR_INVALID_ARG


def test_create_rejects_bad_arguments_on_the_host(lib):
    from lossless_speculative_verify_gb300 import _lib
    h = ctypes.c_void_p()
    bad = _cfg(d=65)
    w = _lib.Weights()
    st = lib.evs_create(ctypes.byref(bad), ctypes.byref(w), ctypes.c_void_p(256), 1 << 20, None,
                        ctypes.byref(h))
    assert st == _lib.EVS_ERR_INVALID_ARG and not h.value
    good = _cfg()
    st = lib.evs_create(ctypes.byref(good), ctypes.byref(w), ctypes.c_void_p(256), 1 << 20, None,
                        ctypes.byref(h))
    assert st == _lib.EVS_ERR_INVALID_ARG                      # null weight pointers
    assert lib.evs_status_str(2).decode().startswith("capacity")
    assert lib.evs_last_launch_count(None) == 0
