"""Seeded generators (NumPy PCG64) for weights, prefixes, draft rounds and pre-round state.

Seeds: weights 1000+s, prefix 2000+s, round r 3000+s*10^4+r, synthetic state 4000+s,
where s is the workload's ``seed_base``. Draw order inside each generator is fixed, so a
given (workload, seed) always yields the same arrays on any machine.

Value distributions follow the synthetic workload descriptions: every matrix N(0, 1/d);
FIR taps N(0, 1/L); IIR poles lambda = r*exp(i*theta) with r ~ U[0.5, 0.99] and
theta ~ U[0, pi]; IIR input and readout coefficients complex normal with variance 1 and
1/16; DNA prefixes uniform over ACGT or from an order-3 Markov chain with Dirichlet(0.3)
transition rows; draft distributions q Dirichlet(alpha) over the four bases with drafts
drawn from q; uniforms in [0, 1).
"""
from __future__ import annotations

import numpy as np

from .workloads import ACGT_IDS, Workload

_ACGT = np.asarray(ACGT_IDS, dtype=np.int32)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32.

    A storage-format conversion for generated inputs of bf16 workloads, so that both
    sides start from the same representable values. Finite inputs only.
    """
    a = np.array(x, dtype=np.float32, copy=True, order="C")
    flat = a.reshape(-1).view(np.uint32)
    step = 1 << 24
    for lo in range(0, flat.size, step):
        b = flat[lo:lo + step]
        lsb = (b >> np.uint32(16)) & np.uint32(1)
        b += np.uint32(0x7FFF) + lsb
        b &= np.uint32(0xFFFF0000)
    return a


def _normal(rng, shape, std, bf16):
    out = np.empty(shape, dtype=np.float32)
    rng.standard_normal(out=out, dtype=np.float32)
    out *= np.float32(std)
    return round_to_bf16(out) if bf16 else out


def _cnormal(rng, shape, var):
    re = np.empty(shape, dtype=np.float32)
    im = np.empty(shape, dtype=np.float32)
    rng.standard_normal(out=re, dtype=np.float32)
    rng.standard_normal(out=im, dtype=np.float32)
    s = np.float32(np.sqrt(var / 2.0))
    return (re * s + 1j * (im * s)).astype(np.complex64)


def gen_weights(wl: Workload) -> dict:
    """Random-init target weights, math convention (``y = x @ W``).

    Returns {"embed": [V,d], "head": [d,V], "layers": [dict per layer]}; FIR layers hold
    w_in, taps [d,L], w_out; IIR layers w_in, lam/b/c complex64 [d,N], w_out; attention
    layers wq, wk, wv, wo. Matrices are bf16-representable float32 for bf16 workloads.
    """
    rng = _rng(1000 + wl.seed_base)
    d, V = wl.d, wl.vocab
    bf = wl.dtype == "bf16"
    std = 1.0 / np.sqrt(d)
    w = {"embed": _normal(rng, (V, d), std, bf), "layers": []}
    for spec in wl.layers:
        if spec.kind == "fir":
            L = spec.param
            w["layers"].append({
                "kind": "fir",
                "w_in": _normal(rng, (d, d), std, bf),
                "taps": _normal(rng, (d, L), 1.0 / np.sqrt(L), False),
                "w_out": _normal(rng, (d, d), std, bf),
            })
        elif spec.kind == "iir":
            N = spec.param
            w_in = _normal(rng, (d, d), std, bf)
            r = rng.uniform(0.5, 0.99, size=(d, N))
            th = rng.uniform(0.0, np.pi, size=(d, N))
            lam = (r * np.exp(1j * th)).astype(np.complex64)
            b = _cnormal(rng, (d, N), 1.0)
            c = _cnormal(rng, (d, N), 1.0 / 16.0)
            w["layers"].append({
                "kind": "iir", "w_in": w_in, "lam": lam, "b": b, "c": c,
                "w_out": _normal(rng, (d, d), std, bf),
            })
        elif spec.kind == "attn":
            w["layers"].append({
                "kind": "attn",
                "wq": _normal(rng, (d, d), std, bf),
                "wk": _normal(rng, (d, d), std, bf),
                "wv": _normal(rng, (d, d), std, bf),
                "wo": _normal(rng, (d, d), std, bf),
            })
        else:
            raise ValueError(spec.kind)
    w["head"] = _normal(rng, (d, V), std, bf)
    return w


def gen_prefix(wl: Workload, length: int | None = None) -> np.ndarray:
    """DNA prefix tokens, int32 [B, P]."""
    P = wl.prefix_len if length is None else length
    rng = _rng(2000 + wl.seed_base)
    B = wl.batch
    if wl.prefix_kind == "uniform":
        return _ACGT[rng.integers(0, 4, size=(B, P))]
    if wl.prefix_kind == "markov3":
        trans = rng.dirichlet(np.full(4, 0.3), size=64)      # 64 contexts x 4 bases
        cdf = np.cumsum(trans, axis=1)
        idx = np.empty((B, P), dtype=np.int64)
        idx[:, :3] = rng.integers(0, 4, size=(B, min(3, P)))
        u = rng.random(size=(B, P))
        for t in range(3, P):
            ctx = idx[:, t - 3] * 16 + idx[:, t - 2] * 4 + idx[:, t - 1]
            nxt = (u[:, t, None] >= cdf[ctx]).sum(axis=1)
            idx[:, t] = np.minimum(nxt, 3)
        return _ACGT[idx]
    raise ValueError(wl.prefix_kind)


def gen_round(wl: Workload, r: int, anchor: np.ndarray | None = None) -> dict:
    """One verification round's generated inputs.

    tokens int32 [B, C, gamma+1] (position 0 is the anchor, shared by the candidates of a
    sequence; positions 1..gamma are drafts drawn from q), q float32 [B, C, gamma, V]
    (mass only on ACGT), u float32 [B, C, gamma+1] in [0, 1): u[..., j] for the test of
    draft j+1, u[..., gamma] for the correction / bonus draw.
    """
    rng = _rng(3000 + wl.seed_base * 10_000 + r)
    B, C, g, V = wl.batch, wl.n_cand, wl.gamma, wl.vocab
    if anchor is None:
        anchor = _ACGT[rng.integers(0, 4, size=B)]
    probs = rng.dirichlet(np.full(4, wl.q_alpha), size=(B, C, g)).astype(np.float32)
    q = np.zeros((B, C, g, V), dtype=np.float32)
    q[..., _ACGT] = probs
    cdf = np.cumsum(probs.astype(np.float64), axis=-1)
    ud = rng.random(size=(B, C, g))
    pick = np.minimum((ud[..., None] >= cdf).sum(axis=-1), 3)
    tokens = np.empty((B, C, g + 1), dtype=np.int32)
    tokens[:, :, 0] = np.asarray(anchor, dtype=np.int32)[:, None]
    tokens[:, :, 1:] = _ACGT[pick]
    u = rng.random(size=(B, C, g + 1), dtype=np.float32)
    return {"tokens": tokens, "q": q, "u": u}


def gen_state(wl: Workload, P: int | None = None) -> dict:
    """Synthetic pre-round state of the stated shapes and value ranges.

    kv_len int32 [B] = P; per attention layer K and V float32 [B, H, P, dh] ~ N(0, 1)
    (bf16-representable for bf16 workloads, the magnitude of x_hat @ W_k with unit-rms
    x_hat and N(0, 1/d) weights); per FIR layer the last L-1 inputs float32 [B, L-1, d]
    ~ N(0, 1); per IIR layer the modal state complex64 [B, d, N] ~ CN(0, 4).
    """
    P = wl.prefix_len if P is None else P
    rng = _rng(4000 + wl.seed_base)
    B, d, dh = wl.batch, wl.d, wl.head_dim
    bf = wl.dtype == "bf16"
    st = {"kv_len": np.full(B, P, dtype=np.int32), "layers": []}
    for spec in wl.layers:
        if spec.kind == "attn":
            H = spec.param
            st["layers"].append({"kind": "attn",
                                 "k": _normal(rng, (B, H, P, dh), 1.0, bf),
                                 "v": _normal(rng, (B, H, P, dh), 1.0, bf)})
        elif spec.kind == "fir":
            st["layers"].append({"kind": "fir",
                                 "tail": _normal(rng, (B, spec.param - 1, d), 1.0, False)})
        else:
            st["layers"].append({"kind": "iir", "s": _cnormal(rng, (B, d, spec.param), 4.0)})
    return st


def gen_table_target(V: int, seed: int, alpha: float = 1.0) -> dict:
    """Tiny autoregressive target and draft tables for exactness checks of acceptance.

    p[a] is the target's next-token distribution after token a, q[a] the drafter's
    (order-1 Markov, both float64 [V, V]); p0 and q0 are the distributions at the first
    position. Entries of q are kept away from zero so every token can be drafted.
    """
    rng = _rng(seed)
    p = rng.dirichlet(np.full(V, alpha), size=V)
    q = rng.dirichlet(np.full(V, alpha), size=V) * 0.9 + 0.1 / V
    p0 = rng.dirichlet(np.full(V, alpha))
    q0 = rng.dirichlet(np.full(V, alpha)) * 0.9 + 0.1 / V
    return {"p": p, "q": q, "p0": p0, "q0": q0}
