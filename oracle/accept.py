"""Lossless acceptance rules, fp64 (test infrastructure only).

Greedy (ReaDy summary, section 3.1 and appendix D.2; EvSpark summary, Figure 1(c)):
the accepted prefix is the longest run of drafts equal to the target's argmax; the
target's argmax at the first mismatch (or after the last draft, the bonus) becomes the
correction. Ties in argmax go to the lowest token id.

Rejection sampling (EvSpark, Figure 1(c): the correction may be sampled; ReaDy, appendix D.2,
the target distribution is preserved): draft d_j is accepted with probability
min(1, p_j(d_j) / q_j(d_j)), realised as the strict test u_j * q_j(d_j) < p_j(d_j) with
u_j uniform in [0, 1); at the first rejection the correction is drawn from
max(0, p_j - q_j) renormalised; if every draft is accepted the bonus is drawn from
p_{gamma+1}. Both draws use the last uniform, u_gamma, by inverse CDF over ascending ids.

Several candidates per sequence: either each candidate is tested alone and the one with
the most accepted drafts is committed (``select_candidate``; exact for greedy, not for
sampling), or the lossless recursive rule of ``multi_candidate_accept``.

Indexing: ``p_rows[i]`` is the target distribution computed at block position i (after
consuming the anchor and drafts 1..i), i.e. the distribution for draft i+1; ``q_rows[j]``
and ``drafts[j]`` are draft j+1's proposal distribution and token.
"""
from __future__ import annotations

import numpy as np


def softmax_t(logits, temperature=1.0):
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def residual(p, q):
    """Unnormalised residual distribution max(0, p - q)."""
    return np.maximum(np.asarray(p, np.float64) - np.asarray(q, np.float64), 0.0)


def inverse_cdf(r, u):
    """Smallest id v with sum_{w<=v} r_w > u * sum(r) (ascending ids).

    If rounding leaves no such id, the last id with positive mass is returned.
    """
    r = np.asarray(r, np.float64)
    c = np.cumsum(r)
    hit = np.nonzero(c > u * c[-1])[0]
    if hit.size:
        return int(hit[0])
    return int(np.nonzero(r > 0)[0][-1])


def _gap_tie(logits, tau):
    if tau <= 0:
        return False
    l = np.sort(np.asarray(logits, np.float64))
    rms = np.sqrt(np.mean(l * l))
    return (l[-1] - l[-2]) < tau * rms


def _cdf_tie(r, u, tau):
    if tau <= 0:
        return False
    c = np.cumsum(np.asarray(r, np.float64))
    return bool(np.min(np.abs(c - u * c[-1])) < tau * c[-1])


def greedy_accept(p_rows, drafts, logits=None, tau=0.0):
    """Returns (k, correction, near_tie). Near-tie: top-2 logit gap below tau * rms
    at any position whose argmax was consulted."""
    g = len(drafts)
    k = 0
    while k < g and int(drafts[k]) == int(np.argmax(p_rows[k])):
        k += 1
    corr = int(np.argmax(p_rows[k]))
    tie = False
    if logits is not None:
        tie = any(_gap_tie(logits[i], tau) for i in range(k + 1))
    return k, corr, tie


def sampling_accept(p_rows, q_rows, drafts, u, tau=0.0, trace=None):
    """Returns (k, correction, near_tie, residual_was_empty). ``trace``, when a list,
    receives ("test", j, accepted) and ("draw", gamma, token) in order."""
    g = len(drafts)
    tie = False
    for j in range(g):
        d = int(drafts[j])
        pj, qj = float(p_rows[j][d]), float(q_rows[j][d])
        lhs = float(u[j]) * qj
        if tau > 0 and abs(lhs - pj) < tau * pj:
            tie = True
        if trace is not None:
            trace.append(("test", j, lhs < pj))
        if lhs < pj:
            continue
        r = residual(p_rows[j], q_rows[j])
        empty = not (r.sum() > 0)
        if empty:
            r = np.asarray(p_rows[j], np.float64)
        tie = tie or _cdf_tie(r, float(u[g]), tau)
        tok = inverse_cdf(r, float(u[g]))
        if trace is not None:
            trace.append(("draw", g, tok))
        return j, tok, tie, empty
    r = np.asarray(p_rows[g], np.float64)
    tie = tie or _cdf_tie(r, float(u[g]), tau)
    tok = inverse_cdf(r, float(u[g]))
    if trace is not None:
        trace.append(("draw", g, tok))
    return g, tok, tie, False


def multi_candidate_accept(p_rows, q_rows, drafts, u, tau=0.0, trace=None):
    """Lossless verification of several candidate blocks of one sequence: rejection
    sampling applied recursively across the candidates, which form a token tree whose
    equal prefixes are merged (the multi-candidate / tree verification the EvSpark summary
    cites as related work; ReaDy appendix D.2 for the single-chain rule it extends).

    p_rows [C][gamma+1][V]: each candidate's target distributions along its own block;
    q_rows [C][gamma][V], drafts [C][gamma], u [C][gamma+1].

    At depth j the alive candidates (whose drafts 1..j equal the accepted path; all of them
    at j = 0) are tried in index order against the current distribution r (p at the path's
    position j, taken from the lowest alive candidate): draft x of candidate c is accepted
    iff u[c][j] q_c(x) < r(x); after a rejection r becomes max(0, r - q_c) renormalised
    (left unchanged, and the round marked, if that has no mass). On acceptance the alive
    set shrinks to the candidates whose draft j+1 is x. If every alive candidate is
    rejected the correction is drawn from r, and after gamma acceptances the bonus from p
    at the end of the path, both by inverse CDF at u[lead][gamma] (lead: the lowest alive
    index), which is the committed candidate.

    Returns (k, correction, committed candidate, near_tie, residual_was_empty, depth [C]):
    depth[c] is how many of candidate c's drafts lie on the accepted path. ``trace``, when
    a list, receives ("test", c, j, accepted) and ("draw", c, gamma, token) in order."""
    C, g = len(drafts), len(drafts[0])
    alive = list(range(C))
    depth = np.zeros(C, np.int64)
    tie = empty = False
    for j in range(g + 1):
        lead = alive[0]
        r = np.asarray(p_rows[lead][j], np.float64)
        x_acc = None
        if j < g:
            for c in alive:
                x = int(drafts[c][j])
                qc = np.asarray(q_rows[c][j], np.float64)
                rn = r / r.sum()
                lhs = float(u[c][j]) * qc[x]
                if tau > 0 and abs(lhs - rn[x]) < tau * rn[x]:
                    tie = True
                ok = lhs < rn[x]
                if trace is not None:
                    trace.append(("test", c, j, ok))
                if ok:
                    x_acc = x
                    break
                res = residual(rn, qc)
                if res.sum() > 0:
                    r = res
                else:
                    empty = True
        if x_acc is None:
            depth[alive] = j
            ug = float(u[lead][g])
            tie = tie or _cdf_tie(r, ug, tau)
            tok = inverse_cdf(r, ug)
            if trace is not None:
                trace.append(("draw", lead, g, tok))
            return j, tok, lead, tie, empty, depth
        keep = [c for c in alive if int(drafts[c][j]) == x_acc]
        for c in alive:
            if c not in keep:
                depth[c] = j
        alive = keep
    raise AssertionError("unreachable")


def select_candidate(ks):
    """Multi-candidate commit: the candidate with the most accepted drafts, lowest
    index on ties."""
    ks = np.asarray(ks)
    return int(np.argmax(ks))
