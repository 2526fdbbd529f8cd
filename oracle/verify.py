"""One verify + slice round by the plain definition (test infrastructure only).

For each sequence and candidate: start from the pre-round state, consume the anchor and
the drafts one token at a time (``Target.step``), keep a snapshot of the state after each
block position, turn the logits into p = softmax(logits / T), run the acceptance rule,
and return the snapshot at the accepted index k: the state after consuming the anchor and
k drafts, with the readable KV length advanced by k+1 (EvSpark summary, Figure 1(c)-(d)).
Nothing is recomputed after acceptance.

With several candidates per sequence, each is verified from the same pre-round state with
its own q and uniforms; the candidate with the largest k is committed (lowest index on
ties), together with its block K/V rows, FIR tail and IIR state.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .accept import greedy_accept, sampling_accept, select_candidate, softmax_t


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


def verify_round(target, states, tokens, q=None, u=None, mode="greedy", temperature=1.0,
                 tau=0.0) -> RoundResult:
    """``states`` is a list (one ``SeqState`` per sequence), updated in place to the
    sliced state. tokens int [B, C, gamma+1]; q [B, C, gamma, V]; u [B, C, gamma+1]."""
    tokens = np.asarray(tokens)
    B, C, T = tokens.shape
    g = T - 1
    V = target.wl.vocab
    res = RoundResult(logits=np.zeros((B, C, T, V)), k_c=np.zeros((B, C), np.int64),
                      corr_c=np.zeros((B, C), np.int64), tie_c=np.zeros((B, C), bool),
                      k=np.zeros(B, np.int64), corr=np.zeros(B, np.int64),
                      cand=np.zeros(B, np.int64), tie=np.zeros(B, bool))
    for b in range(B):
        st = states[b]
        base = st.snapshot()
        snaps_c, rows_c, traces_b = [], [], []
        for c in range(C):
            st.restore(base)
            snaps, logits, traces = [], [], []
            for i in range(T):
                tr = []
                logits.append(target.step(st, int(tokens[b, c, i]), tr))
                traces.append(tr)
                snaps.append(st.snapshot())
            rows = []
            for L in st.layers:
                if L["kind"] == "attn":
                    n0 = L["kv"].length - T
                    rows.append((n0, L["kv"].k[:, n0:n0 + T].copy(),
                                 L["kv"].v[:, n0:n0 + T].copy()))
            logits = np.asarray(logits)
            p = softmax_t(logits, temperature)
            if mode == "greedy":
                k, corr, tie = greedy_accept(p, tokens[b, c, 1:], logits, tau)
            else:
                k, corr, tie, _ = sampling_accept(p, q[b, c], tokens[b, c, 1:], u[b, c], tau)
            res.logits[b, c] = logits
            res.k_c[b, c], res.corr_c[b, c], res.tie_c[b, c] = k, corr, tie
            snaps_c.append(snaps)
            rows_c.append(rows)
            traces_b.append(traces)
        cb = select_candidate(res.k_c[b])
        kb = int(res.k_c[b, cb])
        # commit: the chosen candidate's block K/V rows become the cache rows after the
        # prefix, then the state returns to its snapshot at block index k
        it = iter(rows_c[cb])
        for L in st.layers:
            if L["kind"] == "attn":
                n0, kr, vr = next(it)
                L["kv"].k[:, n0:n0 + T] = kr
                L["kv"].v[:, n0:n0 + T] = vr
        st.restore(snaps_c[cb][kb])
        res.k[b], res.corr[b], res.cand[b] = kb, res.corr_c[b, cb], cb
        res.tie[b] = bool(res.tie_c[b].any())
        res.traces.append(traces_b)
    return res
