"""The oracle's pins have teeth: each plausible mistake below (a reversed index, a dropped
term or factor, a conjugate, a wrong boundary convention, an off-by-one snapshot, ...) is
planted in the oracle's source and executed in a fresh interpreter, and one of the pins
must then fail. Nothing is written to disk: the mutated module source is executed in
place of the module's own before the pins are imported."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RUNNER = r"""
import sys
import pytest
root, fname, old, new = sys.argv[1:5]
nodes = sys.argv[5:]
sys.path[:0] = [root, root + "/tests"]
try:
    import oracle, oracle.accept, oracle.model, oracle.verify
    mods = {"accept.py": oracle.accept, "model.py": oracle.model, "verify.py": oracle.verify,
            "__init__.py": oracle}
    for name in ("accept.py", "model.py", "verify.py", "__init__.py"):
        mod = mods[name]
        src = open(mod.__file__).read()
        if name == fname:
            if old not in src:
                sys.exit(90)
            src = src.replace(old, new, 1)
        exec(compile(src, mod.__file__, "exec"), mod.__dict__)
except Exception as e:   # the planting itself failed: not a pin's doing
    print("planting failed:", repr(e))
    sys.exit(91)
pins = root + "/tests/test_oracle_pins.py::"
sys.exit(pytest.main(["-q", "-x", "-p", "no:cacheprovider", *[pins + n for n in nodes]]))
"""

# (file, original text, planted mistake, pins of which one must fail)
MUTANTS = {
    "fir taps reversed": ("model.py", "y = y + taps[:, j] * window[Lf - 1 - j]", "y = y + taps[:, j] * window[j]",
                          ["test_fir_step_equals_numpy_convolve"]),
    "fir tail keeps the oldest input": ("model.py", "return y, window[1:].copy()", "return y, window[:-1].copy()",
                                        ["test_fir_step_equals_numpy_convolve"]),
    "iir input weight conjugated": ("model.py", "s_new = lam * s + b * u[:, None]",
                                    "s_new = lam * s + np.conj(b) * u[:, None]", ["test_iir_step_equals_scipy_lfilter"]),
    "iir readout of the old state": ("model.py", "return np.real(np.sum(c * s_new, axis=1)), s_new",
                                     "return np.real(np.sum(c * s, axis=1)), s_new",
                                     ["test_iir_step_equals_scipy_lfilter"]),
    "attention without 1/sqrt(dh)": ("model.py", "sc = K @ q / np.sqrt(q.shape[-1])", "sc = K @ q",
                                     ["test_attend_equals_scipy_softmax_and_is_permutation_invariant"]),
    "rms norm by the sum": ("model.py", "return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + EPS)",
                            "return h / np.sqrt(np.sum(h * h, axis=-1, keepdims=True) + EPS)",
                            ["test_rmsnorm_unit_rms"]),
    "attention residual dropped": ("model.py", '                h = h + o.reshape(-1) @ L["wo"]',
                                   '                h = o.reshape(-1) @ L["wo"]',
                                   ["test_block_forward_equals_sequential_decode"]),
    "query misses its own key": ("model.py", "                kv.append(k, v)\n                n = kv.length",
                                 "                n = kv.length\n                kv.append(k, v)",
                                 ["test_block_forward_equals_sequential_decode"]),
    "head without the final norm": ("model.py", "        return self.rmsnorm(h) @ self.head\n\n    # ---- independent",
                                    "        return h @ self.head\n\n    # ---- independent",
                                    ["test_block_forward_equals_sequential_decode"]),
    "acceptance at equality": ("accept.py", "        if lhs < pj:\n            continue",
                               "        if lhs <= pj:\n            continue", ["test_acceptance_boundary_is_strict"]),
    "inverse CDF closed on the right": ("accept.py", "    hit = np.nonzero(c > u * c[-1])[0]",
                                        "    hit = np.nonzero(c >= u * c[-1])[0]",
                                        ["test_inverse_cdf_boundaries_are_half_open"]),
    "residual q - p": ("accept.py",
                       "    return np.maximum(np.asarray(p, np.float64) - np.asarray(q, np.float64), 0.0)",
                       "    return np.maximum(np.asarray(q, np.float64) - np.asarray(p, np.float64), 0.0)",
                       ["test_acceptance_boundary_is_strict"]),
    "temperature ignored": ("accept.py", "    z = np.asarray(logits, dtype=np.float64) / float(temperature)",
                            "    z = np.asarray(logits, dtype=np.float64)",
                            ["test_native_decode_sampling_draws_by_inverse_cdf"]),
    "greedy ties to the highest id": ("accept.py", "    corr = int(np.argmax(p_rows[k]))",
                                      "    corr = int(len(p_rows[k]) - 1 - np.argmax(p_rows[k][::-1]))",
                                      ["test_greedy_tie_goes_to_lowest_id"]),
    "bonus from the previous row": ("accept.py",
                                    "        return j, tok, tie, empty\n    r = np.asarray(p_rows[g], np.float64)",
                                    "        return j, tok, tie, empty\n    r = np.asarray(p_rows[g - 1], np.float64)",
                                    ["test_native_decode_chain_is_the_identity_drafter_round[sampling]"]),
    "greedy compares the next row": ("accept.py",
                                     "    while k < g and int(drafts[k]) == int(np.argmax(p_rows[k])):",
                                     "    while k < g and int(drafts[k]) == int(np.argmax(p_rows[k + 1])):",
                                     ["test_slice_equals_fresh_decode_for_every_k[1]"]),
    "multi-candidate acceptance at equality": ("accept.py", "                ok = lhs < rn[x]",
                                               "                ok = lhs <= rn[x]",
                                               ["test_acceptance_boundary_is_strict"]),
    "multi-candidate test against the unnormalised residual": ("accept.py", "                ok = lhs < rn[x]",
                                                               "                ok = lhs < r[x]",
                                                               ["test_multi_candidate_recursive_chi_square"]),
    "multi-candidate revives dropped candidates": (
        "accept.py", "        keep = [c for c in alive if int(drafts[c][j]) == x_acc]",
        "        keep = [c for c in range(C) if int(drafts[c][j]) == x_acc]",
        ["test_multi_candidate_recursive_chi_square",
         "test_multi_candidate_recursive_rule_is_exact_by_enumeration"]),
    "commit the snapshot after k+1": ("verify.py", '        st.restore(bp["snaps"][b][cb][kb])',
                                      "        st.restore(bp['snaps'][b][cb][min(kb + 1, len(bp['snaps'][b][cb]) - 1)])",
                                      ["test_slice_equals_fresh_decode_for_every_k[0]"]),
    "candidates not restarted from the pre-round state": (
        "verify.py", "        for c in range(C):\n            st.restore(base)", "        for c in range(C):\n            pass",
        ["test_multi_candidate_round_commits_chosen_candidate"]),
    "decode greedy index reversed": ("verify.py", "            nxt[b] = int(np.argmax(logits[b]))",
                                     "            nxt[b] = int(np.argmax(logits[b][::-1]))",
                                     ["test_native_decode_chain_is_the_identity_drafter_round[greedy]"]),
    "decode draws at 1 - u": ("verify.py", "            nxt[b] = inverse_cdf(p, float(u[b]))",
                              "            nxt[b] = inverse_cdf(p, 1.0 - float(u[b]))",
                              ["test_native_decode_chain_is_the_identity_drafter_round[sampling]"]),
    "slice keeps the readable KV length": ("model.py", '                L["kv"].length = S["length"]',
                                           "                pass", ["test_slice_equals_fresh_decode_for_every_k[0]"]),
}


def _run(fname, old, new, nodes):
    return subprocess.run([sys.executable, "-c", RUNNER, ROOT, fname, old, new, *nodes], cwd=ROOT,
                          capture_output=True, text=True, timeout=600)


def test_unplanted_oracle_passes_the_same_pins():
    """Control: the same machinery with nothing planted passes every pin the mutants use."""
    nodes = sorted({n for *_, ns in MUTANTS.values() for n in ns})
    r = _run("accept.py", "", "", nodes)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(name):
    fname, old, new, nodes = MUTANTS[name]
    r = _run(fname, old, new, nodes)
    assert r.returncode not in (90, 91), f"{name}: could not be planted in oracle/{fname}\n{r.stdout[-500:]}"
    assert r.returncode != 90, f"{name}: the original text is no longer in oracle/{fname}"
    assert r.returncode == 1, f"{name}: no pin failed (exit {r.returncode})\n{r.stdout[-2000:]}{r.stderr[-2000:]}"
