"""Lossless acceptance rules, fp64 (test infrastructure only).

Greedy (ReaDy summary, section 3.1 and appendix D.2; EvSpark summary, Figure 1(c)):
the accepted prefix is the longest run of drafts equal to the target's argmax; the
target's argmax at the first mismatch (or after the last draft, the bonus) becomes the
correction. Ties in argmax go to the lowest token id.

Rejection sampling (EvSpark, Figure 1(c) "sampled correction"; ReaDy, appendix D.2,
the target distribution is preserved): draft d_j is accepted with probability
min(1, p_j(d_j) / q_j(d_j)), realised as the strict test u_j * q_j(d_j) < p_j(d_j) with
u_j uniform in [0, 1); at the first rejection the correction is drawn from
max(0, p_j - q_j) renormalised; if every draft is accepted the bonus is drawn from
p_{gamma+1}. Both draws use the last uniform, u_gamma, by inverse CDF over ascending ids.

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


def sampling_accept(p_rows, q_rows, drafts, u, tau=0.0):
    """Returns (k, correction, near_tie, residual_was_empty)."""
    g = len(drafts)
    tie = False
    for j in range(g):
        d = int(drafts[j])
        pj, qj = float(p_rows[j][d]), float(q_rows[j][d])
        lhs = float(u[j]) * qj
        if tau > 0 and abs(lhs - pj) < tau * pj:
            tie = True
        if lhs < pj:
            continue
        r = residual(p_rows[j], q_rows[j])
        empty = not (r.sum() > 0)
        if empty:
            r = np.asarray(p_rows[j], np.float64)
        tie = tie or _cdf_tie(r, float(u[g]), tau)
        return j, inverse_cdf(r, float(u[g])), tie, empty
    r = np.asarray(p_rows[g], np.float64)
    tie = tie or _cdf_tie(r, float(u[g]), tau)
    return g, inverse_cdf(r, float(u[g])), tie, False


def select_candidate(ks):
    """Multi-candidate commit: the candidate with the most accepted drafts, lowest
    index on ties."""
    ks = np.asarray(ks)
    return int(np.argmax(ks))
