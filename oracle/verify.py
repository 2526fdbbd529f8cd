"""One verify + slice round by the plain definition (test infrastructure only).

For each sequence and candidate: start from the pre-round state, consume the anchor and
the drafts one token at a time (``Target.step``), keep a snapshot of the state after each
block position, turn the logits into p = softmax(logits / T), run the acceptance rule,
and return the snapshot at the accepted index k: the state after consuming the anchor and
k drafts, with the readable KV length advanced by k+1 (EvSpark summary, Figure 1(c)-(d)).
Nothing is recomputed after acceptance.

Native decoding (``decode_step``), the baseline the block method is compared with (the
identity-drafter control of the EvSpark summary, Interpretation, is a multiple of native
throughput): one token per sequence, and the next token drawn from the new position's
softmax(logits / T) by argmax or by inverse CDF at one uniform.

With several candidates per sequence, each block is computed from the same pre-round state;
under sampling the lossless recursive rule (``multi_candidate_accept``) picks the accepted
path and the committed candidate, or, by choice, each candidate is tested alone with its own
q and uniforms and the one with the largest k is committed (lowest index on ties; the rule
for greedy either way). The committed candidate's block K/V rows, FIR tail and IIR state are
kept.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .accept import (_cdf_tie, _gap_tie, greedy_accept, inverse_cdf, multi_candidate_accept, sampling_accept,
                     select_candidate, softmax_t)


@dataclass
class RoundResult:
    logits: np.ndarray          # [B, C, T, V]
    k_c: np.ndarray             # [B, C] accepted drafts per candidate
    corr_c: np.ndarray          # [B, C]
    tie_c: np.ndarray           # [B, C] near-tie flags
    k: np.ndarray               # [B]
    corr: np.ndarray            # [B]
    cand: np.ndarray            # [B]
    tie: np.ndarray             # [B]
    traces: list = field(default_factory=list)   # [B][C][T] -> per-layer values


def prefill(target, state, tokens):
    """Consume a prefix one token at a time."""
    for x in tokens:
        target.step(state, int(x))


def block_pass(target, states, tokens):
    """Decode every candidate's block one token at a time from the pre-round state and keep
    the state after each position. ``states`` is left at the pre-round state. Returns a
    dict with logits [B, C, T, V], per-position snapshots, the block K/V rows of each
    candidate and the per-layer traces."""
    tokens = np.asarray(tokens)
    B, C, T = tokens.shape
    out = {"logits": np.zeros((B, C, T, target.wl.vocab)), "base": [], "snaps": [], "rows": [],
           "traces": []}
    for b in range(B):
        st = states[b]
        base = st.snapshot()
        snaps_c, rows_c, traces_b = [], [], []
        for c in range(C):
            st.restore(base)
            snaps, traces = [], []
            for i in range(T):
                tr = []
                out["logits"][b, c, i] = target.step(st, int(tokens[b, c, i]), tr)
                traces.append(tr)
                snaps.append(st.snapshot())
            rows = []
            for L in st.layers:
                if L["kind"] == "attn":
                    n0 = L["kv"].length - T
                    rows.append((n0, L["kv"].k[:, n0:n0 + T].copy(),
                                 L["kv"].v[:, n0:n0 + T].copy()))
            snaps_c.append(snaps)
            rows_c.append(rows)
            traces_b.append(traces)
        st.restore(base)
        out["base"].append(base)
        out["snaps"].append(snaps_c)
        out["rows"].append(rows_c)
        out["traces"].append(traces_b)
    return out


def accept_block(logits, tokens, q=None, u=None, mode="greedy", temperature=1.0, tau=0.0,
                 rule="recursive"):
    """Acceptance for every (sequence, candidate) of a block from its logits [B, C, T, V];
    returns k_c, corr_c, tie_c [B, C] and the committed k, corr, cand, tie [B].

    Sampling with several candidates follows ``rule``: "recursive" (lossless, recursive
    rejection across the candidates; k_c is then each candidate's depth on the accepted
    path and corr_c the correction for the committed candidate, -1 for the others) or
    "max_accept" (each candidate alone, the most accepted drafts committed). Greedy is the
    same under both."""
    tokens = np.asarray(tokens)
    B, C, T = tokens.shape
    k_c = np.zeros((B, C), np.int64)
    corr_c = np.zeros((B, C), np.int64)
    tie_c = np.zeros((B, C), bool)
    if mode == "sampling" and C > 1 and rule == "recursive":
        k = np.zeros(B, np.int64)
        corr = np.zeros(B, np.int64)
        cand = np.zeros(B, np.int64)
        for b in range(B):
            p = [softmax_t(np.asarray(logits[b, c], np.float64), temperature) for c in range(C)]
            kb, cb, lead, tie, _, depth = multi_candidate_accept(p, q[b], tokens[b, :, 1:], u[b], tau)
            k[b], corr[b], cand[b] = kb, cb, lead
            k_c[b] = depth
            corr_c[b] = -1
            corr_c[b, lead] = cb
            tie_c[b] = tie
        return k_c, corr_c, tie_c, k, corr, cand, tie_c.any(axis=1)
    for b in range(B):
        for c in range(C):
            lg = np.asarray(logits[b, c], np.float64)
            p = softmax_t(lg, temperature)
            if mode == "greedy":
                k, corr, tie = greedy_accept(p, tokens[b, c, 1:], lg, tau)
            else:
                k, corr, tie, _ = sampling_accept(p, q[b, c], tokens[b, c, 1:], u[b, c], tau)
            k_c[b, c], corr_c[b, c], tie_c[b, c] = k, corr, tie
    cand = np.array([select_candidate(k_c[b]) for b in range(B)], np.int64)
    k = k_c[np.arange(B), cand]
    corr = corr_c[np.arange(B), cand]
    return k_c, corr_c, tie_c, k, corr, cand, tie_c.any(axis=1)


def commit(states, bp, k, cand):
    """State slicing at block index k[b] of candidate cand[b]: the chosen candidate's block
    K/V rows become the cache rows after the prefix, then each sequence returns to its
    snapshot at k (readable KV length advanced by k+1, FIR tail and IIR state at k)."""
    for b, st in enumerate(states):
        cb, kb = int(cand[b]), int(k[b])
        st.restore(bp["base"][b])
        it = iter(bp["rows"][b][cb])
        for L in st.layers:
            if L["kind"] == "attn":
                n0, kr, vr = next(it)
                T = kr.shape[1]
                L["kv"].k[:, n0:n0 + T] = kr
                L["kv"].v[:, n0:n0 + T] = vr
        st.restore(bp["snaps"][b][cb][kb])


def verify_round(target, states, tokens, q=None, u=None, mode="greedy", temperature=1.0,
                 tau=0.0, rule="recursive") -> RoundResult:
    """``states`` is a list (one ``SeqState`` per sequence), updated in place to the
    sliced state. tokens int [B, C, gamma+1]; q [B, C, gamma, V]; u [B, C, gamma+1]."""
    bp = block_pass(target, states, tokens)
    k_c, corr_c, tie_c, k, corr, cand, tie = accept_block(bp["logits"], tokens, q, u, mode,
                                                          temperature, tau, rule)
    commit(states, bp, k, cand)
    return RoundResult(logits=bp["logits"], k_c=k_c, corr_c=corr_c, tie_c=tie_c, k=k, corr=corr,
                       cand=cand, tie=tie, traces=bp["traces"])


def pick_next(logits, u=None, mode="greedy", temperature=1.0, tau=0.0):
    """The next token of native decoding from each sequence's logits [B, V]: the argmax
    (lowest id on ties) in greedy mode, the inverse CDF of softmax(logits / T) at u[b] in
    sampling mode. Returns next [B] and the near-tie flags [B] (the same tests as the
    acceptance rule's)."""
    logits = np.asarray(logits, np.float64)
    B = logits.shape[0]
    nxt = np.zeros(B, np.int64)
    tie = np.zeros(B, bool)
    for b in range(B):
        if mode == "greedy":
            nxt[b] = int(np.argmax(logits[b]))
            tie[b] = _gap_tie(logits[b], tau)
        else:
            p = softmax_t(logits[b], temperature)
            nxt[b] = inverse_cdf(p, float(u[b]))
            tie[b] = _cdf_tie(p, float(u[b]), tau)
    return nxt, tie


def decode_step(target, states, tokens, u=None, mode="greedy", temperature=1.0, tau=0.0):
    """One step of native decoding: sequence b consumes tokens[b] (its state advances in
    place) and draws its next token. Returns logits [B, V], next [B], near-tie flags [B]."""
    logits = np.stack([target.step(st, int(x)) for st, x in zip(states, tokens)])
    nxt, tie = pick_next(logits, u, mode, temperature, tau)
    return logits, nxt, tie
