"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each check below compares the oracle with a library routine, a closed form, an invariant
or a value printed on the EvSpark pages (tests/golden), so that a dropped term, wrong
index, sign or transposed operand in the oracle fails at least one of them.
"""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.signal
import scipy.special

import oracle
from oracle.model import fir_step, iir_step, attend
from synth import LayerSpec, gen_prefix, gen_round, gen_weights, get_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny_wl(**kw):
    base = get_workload("tiny_d64_fp32").replace(
        d=16, head_dim=4,
        layers=(LayerSpec("fir", 3), LayerSpec("iir", 4), LayerSpec("attn", 4),
                LayerSpec("fir", 7)),
        prefix_len=12)
    return base.replace(**kw)


# ---------------------------------------------------------------------------- FIR
def test_fir_step_equals_numpy_convolve():
    rng = np.random.default_rng(0)
    d, L, T = 5, 7, 19
    taps = rng.standard_normal((d, L))
    tail = rng.standard_normal((L - 1, d))
    v = rng.standard_normal((T, d))
    ys = []
    t = tail.copy()
    for i in range(T):
        y, t = fir_step(t, v[i], taps)
        ys.append(y)
    ys = np.array(ys)
    full = np.vstack([tail, v])
    for c in range(d):
        ref = np.convolve(full[:, c], taps[c], mode="valid")
        np.testing.assert_allclose(ys[:, c], ref, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(t, v[-(L - 1):])          # tail = last L-1 inputs


def test_fir_identity_and_delay_taps():
    rng = np.random.default_rng(1)
    d = 4
    tail = rng.standard_normal((2, d))
    v = rng.standard_normal(d)
    ident = np.zeros((d, 3)); ident[:, 0] = 1
    delay2 = np.zeros((d, 3)); delay2[:, 2] = 1
    y, _ = fir_step(tail, v, ident)
    np.testing.assert_array_equal(y, v)
    y, _ = fir_step(tail, v, delay2)
    np.testing.assert_array_equal(y, tail[0])                 # v_{t-2} is the oldest


# ---------------------------------------------------------------------------- IIR
def test_iir_step_equals_scipy_lfilter():
    """s_t = lam s_{t-1} + b u_t is a first-order filter: lfilter([b], [1, -lam])."""
    rng = np.random.default_rng(2)
    d, N, T = 3, 5, 23
    lam = 0.95 * np.exp(1j * rng.uniform(0, np.pi, (d, N))) * rng.uniform(0.5, 1, (d, N))
    b = rng.standard_normal((d, N)) + 1j * rng.standard_normal((d, N))
    c = rng.standard_normal((d, N)) + 1j * rng.standard_normal((d, N))
    s0 = rng.standard_normal((d, N)) + 1j * rng.standard_normal((d, N))
    u = rng.standard_normal((T, d))
    s = s0.copy()
    ys, ss = [], []
    for t in range(T):
        y, s = iir_step(s, u[t], lam, b, c)
        ys.append(y); ss.append(s)
    ys, ss = np.array(ys), np.array(ss)
    for ch in range(d):
        for n in range(N):
            ref, _ = scipy.signal.lfilter([b[ch, n]], [1, -lam[ch, n]], u[:, ch].astype(complex),
                                          zi=[lam[ch, n] * s0[ch, n]])
            np.testing.assert_allclose(ss[:, ch, n], ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ys, np.real(np.einsum("dn,tdn->td", c, ss)), atol=1e-12)


def test_iir_special_cases():
    d, T = 2, 9
    u = np.random.default_rng(3).standard_normal((T, d))
    one = np.ones((d, 1), complex)
    # real pole, b = c = 1: exponential moving sum y_t = sum_j 0.5^(t-j) u_j
    s = np.zeros((d, 1), complex)
    for t in range(T):
        y, s = iir_step(s, u[t], 0.5 * one, one, one)
        ref = sum(0.5 ** (t - j) * u[j] for j in range(t + 1))
        np.testing.assert_allclose(y, ref, atol=1e-13)
    # lam = 0: pass-through scaled by Re(c b)
    cb = np.array([[2 + 1j], [-1 + 3j]])
    s = np.full((d, 1), 7 + 7j)
    y, s = iir_step(s, u[0], 0 * one, cb, one)
    np.testing.assert_allclose(y, np.real(cb[:, 0]) * u[0], atol=1e-14)


# ---------------------------------------------------------------------------- attention
def test_attend_single_key_returns_value():
    rng = np.random.default_rng(4)
    q, k, v = rng.standard_normal(8), rng.standard_normal((1, 8)), rng.standard_normal((1, 8))
    np.testing.assert_allclose(attend(q, k, v), v[0], atol=1e-15)


def test_attend_equals_scipy_softmax_and_is_permutation_invariant():
    rng = np.random.default_rng(5)
    n, dh = 37, 16
    q, K, V = rng.standard_normal(dh), rng.standard_normal((n, dh)), rng.standard_normal((n, dh))
    w = scipy.special.softmax(K @ q / 4.0)
    np.testing.assert_allclose(attend(q, K, V), w @ V, atol=1e-13)
    perm = rng.permutation(n)
    np.testing.assert_allclose(attend(q, K[perm], V[perm]), attend(q, K, V), atol=1e-13)


def test_rmsnorm_unit_rms():
    h = np.random.default_rng(6).standard_normal((3, 64)) * 5
    x = oracle.Target.rmsnorm(h)
    np.testing.assert_allclose(np.sqrt(np.mean(x * x, axis=1)), 1.0, atol=1e-6)


# ---------------------------------------------------------------------------- Lemma 2
def _prefilled(wl, P):
    tgt = oracle.Target(wl, gen_weights(wl))
    st = tgt.empty_state()
    oracle.prefill(tgt, st, gen_prefix(wl, P)[0])
    return tgt, st


def test_block_forward_equals_sequential_decode():
    """Block-forward contract: one forward over the block from the pre-round state gives
    the same logits and per-position states as decoding the tokens one at a time."""
    wl = tiny_wl()
    tgt, st = _prefilled(wl, 12)
    toks = gen_round(wl, 0)["tokens"][0, 0]
    blk_logits, vals = tgt.block_forward(st, toks)
    seq = st.clone()
    for i, x in enumerate(toks):
        tr = []
        l = tgt.step(seq, int(x), tr)
        np.testing.assert_allclose(l, blk_logits[i], rtol=1e-10, atol=1e-10)
        for a, bv in zip(tr, vals):
            if a["kind"] == "fir":
                np.testing.assert_allclose(a["v"], bv["v"][i], atol=1e-11)
            elif a["kind"] == "iir":
                np.testing.assert_allclose(a["s"], bv["s"][i], atol=1e-10)
                np.testing.assert_allclose(a["u"], bv["u"][i], atol=1e-11)
            else:
                np.testing.assert_allclose(a["k"], bv["k"][i], atol=1e-11)
                np.testing.assert_allclose(a["v"], bv["v"][i], atol=1e-11)


# ---------------------------------------------------------------------------- Lemma 3
def _state_arrays(st):
    out = []
    for L in st.layers:
        if L["kind"] == "fir":
            out.append(L["tail"])
        elif L["kind"] == "iir":
            out.append(L["s"])
        else:
            n = L["kv"].length
            out.append((n, L["kv"].k[:, :n], L["kv"].v[:, :n]))
    return out


def _assert_same_state(a, b, tol=1e-11):
    for x, y in zip(_state_arrays(a), _state_arrays(b)):
        if isinstance(x, tuple):
            assert x[0] == y[0]
            np.testing.assert_allclose(x[1], y[1], atol=tol)
            np.testing.assert_allclose(x[2], y[2], atol=tol)
        else:
            np.testing.assert_allclose(x, y, atol=tol)


@pytest.mark.parametrize("k_force", list(range(7)))
def test_slice_equals_fresh_decode_for_every_k(k_force):
    """State restoration: the state sliced at k equals a fresh sequential decode of
    prefix || anchor, d_1..d_k, and the next round from it matches too."""
    wl = tiny_wl()
    P = 12
    tgt, st = _prefilled(wl, P)
    prefix = gen_prefix(wl, P)[0]
    # identity drafts up to k_force, then a deliberately wrong draft
    probe = st.clone()
    toks = [65]
    for i in range(wl.gamma):
        nxt = int(np.argmax(tgt.step(probe, toks[-1])))
        if i == k_force:
            nxt = (nxt + 1) % wl.vocab
        toks.append(nxt)
    toks = np.array(toks)[None, None]
    res = oracle.verify_round(tgt, [st], toks, mode="greedy")
    assert res.k[0] == k_force
    fresh = tgt.empty_state()
    oracle.prefill(tgt, fresh, np.concatenate([prefix, toks[0, 0, :k_force + 1]]))
    _assert_same_state(st, fresh)
    nxt = gen_round(wl, 1, anchor=[res.corr[0]])
    r1 = oracle.verify_round(tgt, [st], nxt["tokens"], mode="greedy")
    r2 = oracle.verify_round(tgt, [fresh], nxt["tokens"], mode="greedy")
    np.testing.assert_allclose(r1.logits, r2.logits, atol=1e-10)
    assert r1.k[0] == r2.k[0] and r1.corr[0] == r2.corr[0]


def test_worked_example_figure_1d():
    """gamma=6, three drafts accepted: FIR tail = inputs at block positions 2 and 3 (L=3),
    IIR state = s_3, readable KV advanced by 4 (tests/golden/fig1d_worked_example.json)."""
    g = json.load(open(os.path.join(GOLDEN, "fig1d_worked_example.json")))["facts"]
    wl = tiny_wl(gamma=g["gamma"], layers=(LayerSpec("fir", g["fir_len"]), LayerSpec("iir", 4),
                                           LayerSpec("attn", 4)))
    tgt, st = _prefilled(wl, 10)
    kv0 = st.kv_len
    probe = st.clone()
    toks = [67]
    for i in range(wl.gamma):
        nxt = int(np.argmax(tgt.step(probe, toks[-1])))
        if i == g["accepted_drafts"]:
            nxt = (nxt + 3) % wl.vocab
        toks.append(nxt)
    res = oracle.verify_round(tgt, [st], np.array(toks)[None, None], mode="greedy")
    assert res.k[0] == g["accepted_drafts"]
    tr = res.traces[0][0]
    fir_inputs = [tr[i][0]["v"] for i in g["fir_tail_block_positions"]]
    np.testing.assert_array_equal(st.layers[0]["tail"], np.array(fir_inputs))
    np.testing.assert_array_equal(st.layers[1]["s"], tr[g["iir_state_block_position"]][1]["s"])
    assert st.kv_len == kv0 + g["kv_len_advance"]


# ---------------------------------------------------------------------------- acceptance
def test_greedy_identity_drafter_accepts_all_and_wrong_first_draft_rejects():
    wl = tiny_wl()
    tgt, st = _prefilled(wl, 8)
    probe = st.clone()
    toks = [71]
    for _ in range(wl.gamma):
        toks.append(int(np.argmax(tgt.step(probe, toks[-1]))))
    bonus = int(np.argmax(tgt.step(probe, toks[-1])))
    r = oracle.verify_round(tgt, [st.clone()], np.array(toks)[None, None], mode="greedy")
    assert r.k[0] == wl.gamma and r.corr[0] == bonus
    bad = list(toks)
    bad[1] = (bad[1] + 1) % wl.vocab
    r = oracle.verify_round(tgt, [st.clone()], np.array(bad)[None, None], mode="greedy")
    first = int(np.argmax(tgt.step(st.clone(), toks[0])))
    assert r.k[0] == 0 and r.corr[0] == first


def _decode_chain(tgt, st, anchor, n, mode, us=None):
    toks, logits = [anchor], []
    for i in range(n):
        lg, nxt, _ = oracle.decode_step(tgt, [st], [toks[-1]], None if us is None else [us[i]], mode)
        logits.append(lg[0])
        toks.append(int(nxt[0]))
    return toks, np.array(logits)


@pytest.mark.parametrize("mode", ["greedy", "sampling"])
def test_native_decode_chain_is_the_identity_drafter_round(mode):
    """Native decoding against block verification: gamma+1 decode steps from a state give
    the drafts of an identity drafter (greedy: the argmax chain; sampling: drafts drawn
    from p itself, proposed with q = p), which a verify round accepts in full; its bonus is
    the decode's next token for the same last uniform, and the sliced state is the state
    after the decode steps."""
    wl = tiny_wl()
    tgt, st = _prefilled(wl, 9)
    rng = np.random.default_rng(11)
    us = rng.random(wl.gamma + 1)
    dec = st.clone()
    toks, logits = _decode_chain(tgt, dec, 67, wl.gamma + 1, mode, us)
    q = oracle.softmax_t(logits[:wl.gamma], wl.temperature)[None, None]
    u = np.concatenate([rng.random(wl.gamma), us[wl.gamma:]])[None, None]
    ver = st.clone()
    r = oracle.verify_round(tgt, [ver], np.array(toks[:-1])[None, None], q, u, mode, wl.temperature)
    assert r.k[0] == wl.gamma and r.corr[0] == toks[-1]
    _assert_same_state(ver, dec, tol=1e-12)


def test_native_decode_sampling_draws_by_inverse_cdf():
    """The sampled next token: over a fine grid of uniforms, each id is drawn for a share
    of the grid equal to its target probability (to the grid's resolution)."""
    rng = np.random.default_rng(5)
    lg = rng.normal(size=(1, 16)) * 2
    p = scipy.special.softmax(lg[0] / 0.7)
    grid = (np.arange(20000) + 0.5) / 20000
    ids = np.array([oracle.pick_next(lg, [g], "sampling", 0.7)[0][0] for g in grid])
    freq = np.bincount(ids, minlength=16) / len(grid)
    np.testing.assert_allclose(freq, p, atol=1.0 / len(grid) + 1e-12)
    assert oracle.pick_next(lg, None, "greedy")[0][0] == int(np.argmax(lg[0]))


def test_greedy_tie_goes_to_lowest_id():
    p = np.array([[0.1, 0.3, 0.3, 0.3], [0.25] * 4])
    k, corr, _ = oracle.greedy_accept(p, [2])
    assert k == 0 and corr == 1


def test_sampling_with_q_equal_p_always_accepts():
    rng = np.random.default_rng(7)
    V, g = 6, 4
    p = rng.dirichlet(np.ones(V), size=g + 1)
    for _ in range(200):
        d = [int(rng.integers(V)) for _ in range(g)]
        u = rng.random(g + 1)
        k, _, _, _ = oracle.sampling_accept(p, p[:g], d, u)
        assert k == g


def _bisect(pred, lo=0.0, hi=1.0, iters=64):
    """Largest x in [lo, hi) region where pred is True, for pred monotone True->False."""
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if pred(mid):
            lo = mid
        else:
            hi = mid
    return lo


def test_acceptance_probability_is_min_one_p_over_q():
    """Rejection-sampling acceptance: P(u q(d) < p(d)) over u ~ U[0,1) = min(1, p/q)."""
    for pd, qd in [(0.2, 0.5), (0.7, 0.3), (0.4, 0.4), (1e-3, 0.9)]:
        p = np.array([pd, 1 - pd]); q = np.array([qd, 1 - qd])
        acc = lambda u: oracle.sampling_accept(np.vstack([p, p]), q[None], [0], [u, 0.5])[0] == 1
        thr = _bisect(acc)
        assert abs(thr - min(1.0, pd / qd)) < 1e-15


def test_inverse_cdf_boundaries_are_half_open():
    """Inverse-transform sampling maps u in [F(v-1), F(v)) to id v, so a u exactly on F(v)
    goes to the next id (exactly representable boundaries)."""
    r = np.array([1.0, 1.0, 2.0])                     # F = 0.25, 0.5, 1.0
    assert [oracle.inverse_cdf(r, u) for u in (0.0, 0.25, 0.375, 0.5, 0.75)] == [0, 1, 1, 2, 2]
    p = np.array([[0.25, 0.25, 0.5], [0.25, 0.25, 0.5]])
    assert oracle.pick_next(np.log(p[:1]), [0.25], "sampling")[0][0] == 1


def test_acceptance_boundary_is_strict():
    """Draft d is accepted iff u q(d) < p(d), u in [0, 1): the accepted set of u is
    [0, p/q), so u exactly at p/q rejects (reading of the test at its measure-zero edge)."""
    p = np.array([[0.25, 0.75], [0.5, 0.5]])
    q = np.array([[0.5, 0.5]])
    assert oracle.sampling_accept(p, q, [0], [0.5, 0.1])[0] == 0           # 0.5 * 0.5 == 0.25
    assert oracle.sampling_accept(p, q, [0], [np.nextafter(0.5, 0), 0.1])[0] == 1
    k, _, cand, *_ = oracle.multi_candidate_accept([p, p], [q, q], [[0], [1]], [[0.5, 0.1], [0.0, 0.1]])
    assert k == 1 and cand == 1                    # first rejected at the edge, second accepted


def test_inverse_cdf_interval_lengths_are_the_distribution():
    """Inverse-transform sampling: the u-interval mapped to id v has length r_v / sum r."""
    r = np.array([0.0, 0.3, 0.0, 0.05, 0.4, 0.25]) * 3.7
    edges = [0.0]
    for v in range(len(r)):
        edges.append(_bisect(lambda u: oracle.inverse_cdf(r, u) <= v))
    lengths = np.diff(edges)
    np.testing.assert_allclose(lengths, r / r.sum(), atol=1e-15)


def _round_law(tab, ctx, gamma):
    """Exact law of the tokens one sampling round emits from context ``ctx`` (table
    target, order-1 Markov), by enumerating drafts and measuring each uniform's branch
    lengths on the black-box acceptance function (u_j for draft j, u_gamma for the draw)."""
    V = tab["p"].shape[0]
    p_of = lambda a: tab["p0"] if a is None else tab["p"][a]
    q_of = lambda a: tab["q0"] if a is None else tab["q"][a]
    law = {}

    def rec(drafts, w):
        if len(drafts) < gamma:
            prev = drafts[-1] if drafts else ctx
            for x in range(V):
                rec(drafts + [x], w * q_of(prev)[x])
            return
        ctxs = [ctx] + drafts
        p_rows = np.array([p_of(c) for c in ctxs])
        q_rows = np.array([q_of(c) for c in ctxs[:-1]])
        fn = lambda u: oracle.sampling_accept(p_rows, q_rows, drafts, u)
        # P(k >= j+1 | k >= j) from the threshold of u_j, with earlier uniforms at 0
        reach = 1.0
        for j in range(gamma + 1):
            if j < gamma:
                base = [0.0] * (gamma + 1)
                def acc(x, j=j):
                    b = list(base); b[j] = x
                    return fn(b)[0] > j
                a = _bisect(acc) if acc(0.0) else 0.0
                p_stop = reach * (1.0 - a)
            else:
                p_stop = reach
            if p_stop > 0:
                u_fix = [0.0] * (gamma + 1)
                if j < gamma:
                    u_fix[j] = 0.5 * (a + 1.0)
                edges = [0.0]
                for v in range(V):
                    def le(x, v=v):
                        b = list(u_fix); b[gamma] = x
                        return fn(b)[1] <= v
                    edges.append(_bisect(le))
                for v, ln in enumerate(np.diff(edges)):
                    if ln > 0:
                        key = tuple(drafts[:j]) + (v,)
                        law[key] = law.get(key, 0.0) + w * p_stop * ln
            if j < gamma:
                reach *= a
    rec([], 1.0)
    return law


def test_sampling_round_is_exact_by_enumeration():
    """Sequence-level exactness on a tiny target (V=4, gamma=2): the first emitted token
    has law p(. | ctx) and the first two have law p(a | ctx) p(b | a), to 1e-12."""
    from synth import gen_table_target
    V, gamma = 4, 2
    tab = gen_table_target(V, seed=11)
    law = _round_law(tab, None, gamma)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    first = np.zeros(V)
    for key, pr in law.items():
        first[key[0]] += pr
    np.testing.assert_allclose(first, tab["p0"], atol=1e-12)
    # two tokens: rounds that emit one token continue with a round from that token
    sub = {a: _round_law(tab, a, gamma) for a in range(V)}
    two = np.zeros((V, V))
    for key, pr in law.items():
        if len(key) >= 2:
            two[key[0], key[1]] += pr
        else:
            for k2, p2 in sub[key[0]].items():
                two[key[0], k2[0]] += pr * p2
    np.testing.assert_allclose(two, tab["p0"][:, None] * tab["p"], atol=1e-12)


class _U:
    """Uniforms u[c][j] of a round from a dict of values (0 where none is given)."""

    def __init__(self, vals, c=None):
        self.vals, self.c = vals, c

    def __getitem__(self, i):
        return _U(self.vals, i) if self.c is None else self.vals.get((self.c, i), 0.0)


def _explore_law(fn, V):
    """Exact law of fn(u, trace) over independent uniforms u[c][j] ~ U[0,1), for a fn that
    uses each uniform at most once: in a threshold test, traced as ("test", c, j, accepted)
    and accepted below some threshold, or in a draw, traced as ("draw", c, j, token) with
    the token non-decreasing in u. The first uniform not yet confined to an interval is
    split where its decision changes (found by bisection) and each part explored."""
    law = {}

    def decision(vals, cj):
        tr = []
        fn(_U(vals), tr)
        return next(e for e in tr if (e[1], e[2]) == cj)[3]

    def explore(fixed, w):
        vals = {cj: 0.5 * (lo + hi) for cj, (lo, hi) in fixed.items()}
        tr = []
        out = fn(_U(vals), tr)
        free = next((e for e in tr if (e[1], e[2]) not in fixed), None)
        if free is None:
            law[out] = law.get(out, 0.0) + w
            return
        kind, cj = free[0], (free[1], free[2])
        at = lambda x: {**vals, cj: x}
        if kind == "test":
            a = _bisect(lambda x: decision(at(x), cj)) if decision(at(0.0), cj) else 0.0
            parts = [(0.0, a), (a, 1.0)]
        else:
            edges = [0.0] + [_bisect(lambda x, v=v: decision(at(x), cj) <= v) for v in range(V)]
            parts = list(zip(edges[:-1], edges[1:]))
        for lo, hi in parts:
            if hi > lo:
                explore({**fixed, cj: (lo, hi)}, w * (hi - lo))

    explore({}, 1.0)
    return law


def _multi_round_law(tab, ctx, gamma, C, rule):
    """Exact law of the tokens one round with C independently drafted candidate blocks
    emits from context ctx (table target, order-1 Markov)."""
    V = tab["p"].shape[0]
    p_of = lambda a: tab["p0"] if a is None else tab["p"][a]
    q_of = lambda a: tab["q0"] if a is None else tab["q"][a]
    law = {}
    chains = []

    def rec(d, w):
        if len(d) == gamma:
            chains.append((d, w))
            return
        prev = d[-1] if d else ctx
        for x in range(V):
            rec(d + [x], w * q_of(prev)[x])

    rec([], 1.0)
    for combo in itertools.product(chains, repeat=C):
        drafts = [d for d, _ in combo]
        w = float(np.prod([wc for _, wc in combo]))
        p_rows = [[p_of(a) for a in [ctx] + d] for d in drafts]
        q_rows = [[q_of(a) for a in [ctx] + d[:-1]] for d in drafts]

        def fn(u, tr):
            if rule == "recursive":
                k, corr, c, *_ = oracle.multi_candidate_accept(p_rows, q_rows, drafts, u, trace=tr)
                return tuple(drafts[c][:k]) + (corr,)
            res = []
            for c in range(C):
                t = []
                k, corr, _, _ = oracle.sampling_accept(p_rows[c], q_rows[c], drafts[c], u[c], trace=t)
                tr.extend((e[0], c) + e[1:] for e in t)
                res.append((k, corr))
            c = max(range(C), key=lambda i: (res[i][0], -i))
            return tuple(drafts[c][:res[c][0]]) + (res[c][1],)

        for key, pr in _explore_law(fn, V).items():
            law[key] = law.get(key, 0.0) + w * pr
    return law


def _first_two(law_of, V):
    law = law_of(None)
    first = np.zeros(V)
    for key, pr in law.items():
        first[key[0]] += pr
    sub = {a: law_of(a) for a in range(V)}
    two = np.zeros((V, V))
    for key, pr in law.items():
        if len(key) >= 2:
            two[key[0], key[1]] += pr
        else:
            for k2, p2 in sub[key[0]].items():
                two[key[0], k2[0]] += pr * p2
    return sum(law.values()), first, two


def test_multi_candidate_recursive_rule_is_exact_by_enumeration():
    """Two candidate blocks drafted independently (V=3, gamma=2): with recursive rejection
    across the candidates the first emitted token has law p(. | ctx) and the first two have
    law p(a | ctx) p(b | a), to 1e-12; committing the candidate with the most accepted
    drafts instead is measurably biased on the same target."""
    from synth import gen_table_target
    V, gamma, C = 3, 2, 2
    tab = gen_table_target(V, seed=13)
    tot, first, two = _first_two(lambda a: _multi_round_law(tab, a, gamma, C, "recursive"), V)
    assert abs(tot - 1.0) < 1e-12
    np.testing.assert_allclose(first, tab["p0"], atol=1e-12)
    np.testing.assert_allclose(two, tab["p0"][:, None] * tab["p"], atol=1e-12)
    tot, first, two = _first_two(lambda a: _multi_round_law(tab, a, gamma, C, "max_accept"), V)
    assert abs(tot - 1.0) < 1e-12
    assert np.abs(two - tab["p0"][:, None] * tab["p"]).max() > 1e-3


def test_sampling_round_chi_square():
    """Seeded sampler check: first emitted token of 20000 rounds vs p (alpha = 1e-3)."""
    from scipy.stats import chisquare
    from synth import gen_table_target
    V, gamma, n = 6, 3, 20000
    tab = gen_table_target(V, seed=12)
    rng = np.random.Generator(np.random.PCG64(99))
    counts = np.zeros(V)
    for _ in range(n):
        drafts, prev = [], None
        for _ in range(gamma):
            qq = tab["q0"] if prev is None else tab["q"][prev]
            prev = int(rng.choice(V, p=qq))
            drafts.append(prev)
        ctxs = [None] + drafts
        p_rows = np.array([tab["p0"] if c is None else tab["p"][c] for c in ctxs])
        q_rows = np.array([tab["q0"] if c is None else tab["q"][c] for c in ctxs[:-1]])
        k, corr, _, _ = oracle.sampling_accept(p_rows, q_rows, drafts, rng.random(gamma + 1))
        counts[drafts[0] if k >= 1 else corr] += 1
    assert chisquare(counts, tab["p0"] * n).pvalue > 1e-3


def test_multi_candidate_recursive_chi_square():
    """Seeded sampler check of the recursive multi-candidate rule at a size the enumeration
    cannot reach (4 candidates, V=6, gamma=3): first emitted token of 20000 rounds vs p,
    and the second token given the first among rounds that emit two (alpha = 1e-3)."""
    from scipy.stats import chisquare
    from synth import gen_table_target
    V, gamma, C, n = 6, 3, 4, 20000
    tab = gen_table_target(V, seed=14)
    rng = np.random.Generator(np.random.PCG64(101))
    first = np.zeros(V)
    second = np.zeros((V, V))
    for _ in range(n):
        drafts = []
        for _ in range(C):
            d, prev = [], None
            for _ in range(gamma):
                prev = int(rng.choice(V, p=tab["q0"] if prev is None else tab["q"][prev]))
                d.append(prev)
            drafts.append(d)
        p_rows = [[tab["p0"]] + [tab["p"][a] for a in d] for d in drafts]
        q_rows = [[tab["q0"]] + [tab["q"][a] for a in d[:-1]] for d in drafts]
        k, corr, c, *_ = oracle.multi_candidate_accept(p_rows, q_rows, drafts, rng.random((C, gamma + 1)))
        out = drafts[c][:k] + [corr]
        first[out[0]] += 1
        if len(out) >= 2:
            second[out[0], out[1]] += 1
    assert chisquare(first, tab["p0"] * n).pvalue > 1e-3
    for a in range(V):
        m = second[a].sum()
        if m >= 500:
            assert chisquare(second[a], tab["p"][a] * m).pvalue > 1e-3


def test_multi_candidate_selects_longest_lowest_index():
    assert oracle.select_candidate([1, 3, 3, 0]) == 1
    assert oracle.select_candidate([0, 0, 0, 0]) == 0


def test_multi_candidate_round_commits_chosen_candidate():
    """Each candidate starts from the shared state; the committed state equals a fresh
    decode of prefix || the chosen candidate's accepted tokens."""
    wl = tiny_wl(n_cand=3, gamma=4)
    P = 10
    tgt, st = _prefilled(wl, P)
    prefix = gen_prefix(wl, P)[0]
    toks = np.zeros((1, 3, wl.gamma + 1), dtype=np.int64)
    for c, kc in enumerate([1, 3, 2]):
        probe = st.clone()
        seq = [65]
        for i in range(wl.gamma):
            nxt = int(np.argmax(tgt.step(probe, seq[-1])))
            if i == kc:
                nxt = (nxt + 1) % wl.vocab
            seq.append(nxt)
        toks[0, c] = seq
    res = oracle.verify_round(tgt, [st], toks, mode="greedy")
    assert list(res.k_c[0]) == [1, 3, 2] and res.cand[0] == 1 and res.k[0] == 3
    fresh = tgt.empty_state()
    oracle.prefill(tgt, fresh, np.concatenate([prefix, toks[0, 1, :4]]))
    _assert_same_state(st, fresh)
