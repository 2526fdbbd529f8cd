"""fp64 hybrid FIR / modal-IIR / attention target, decoded one token at a time.

Test infrastructure only (see the package docstring). Reading of the layer internals
(the pages name only the three state classes: finite FIR windows, modal IIR states and
attention caches; EvSpark summary, Figure 1(d) and Interpretation paragraph 1):

  h <- E[x]
  per layer:  xh = h / sqrt(mean(h^2) + 1e-6)
    FIR-L   v = xh W_in;  y = sum_{j<L} w[:, j] * v_{t-j};  h += y W_out
            state: the last L-1 inputs v (the FIR inputs Figure 1(d) carries over)
    IIR-N   u = xh W_in;  s_t = lam * s_{t-1} + b * u_t  (N complex poles per channel)
            y = Re sum_n c_n s_{t,n};  h += y W_out;  state: s
    attn    q, k, v = xh W_q, xh W_k, xh W_v;  per head o = softmax(q K^T / sqrt(dh)) V
            over the readable cache plus the new key; h += o W_o;  state: K, V, length
  logits = (h / rms(h)) W_head

``Target.step`` is the definition (sequential decode). ``Target.block_forward`` is an
independent block form (convolution, closed-form modal sum, masked attention matrix)
used only to check the block-forward contract (Lemma 2) against the step form.
"""
from __future__ import annotations

import copy

import numpy as np

EPS = 1e-6


def fir_step(tail, v, taps):
    """One depthwise FIR step (EvSpark summary, Figure 1(d): a finite window of the last L-1
    inputs is the FIR state). tail [L-1, d] holds the previous inputs, oldest first;
    returns y = sum_j taps[:, j] * v_{t-j} and the new tail (the last L-1 inputs)."""
    Lf = taps.shape[1]
    window = np.vstack([tail, v[None]])          # v_{t-L+1} .. v_t
    y = np.zeros_like(v)
    for j in range(Lf):
        y = y + taps[:, j] * window[Lf - 1 - j]
    return y, window[1:].copy()


def iir_step(s, u, lam, b, c):
    """One modal IIR step (EvSpark summary, Figure 1(d): the modal state s is the IIR state):
    s' = lam * s + b * u (per channel, N poles), y = Re sum_n c s'."""
    s_new = lam * s + b * u[:, None]
    return np.real(np.sum(c * s_new, axis=1)), s_new


def attend(q, K, V):
    """Single-query attention over rows [0, n) of K, V: softmax(K q / sqrt(dh)) V (EvSpark
    summary, Figure 1(d): the query reads the readable KV prefix)."""
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    sc = K @ q / np.sqrt(q.shape[-1])
    sc = sc - sc.max()
    w = np.exp(sc)
    return (w / w.sum()) @ V


class KVBuffer:
    """Append-only key/value rows of one attention layer of one sequence.

    Rows [0, length) are readable. Shortening ``length`` is the KV part of state
    restoration: rows past it are unreadable and are overwritten by the next append.
    """

    def __init__(self, H, dh, cap, k=None, v=None, length=0, dtype=np.float64):
        self.k = np.zeros((H, cap, dh), dtype=dtype)
        self.v = np.zeros((H, cap, dh), dtype=dtype)
        if k is not None:
            self.k[:, :k.shape[1]] = k
            self.v[:, :v.shape[1]] = v
        self.length = length

    def append(self, k, v):
        if self.length >= self.k.shape[1]:
            grow = max(64, self.k.shape[1])
            self.k = np.concatenate([self.k, np.zeros_like(self.k[:, :grow])], axis=1)
            self.v = np.concatenate([self.v, np.zeros_like(self.v[:, :grow])], axis=1)
        self.k[:, self.length] = k
        self.v[:, self.length] = v
        self.length += 1


class SeqState:
    """Decode state of one sequence: per-layer FIR tail, IIR modal state, KV buffer."""

    def __init__(self, layers):
        self.layers = layers  # list of dicts {"kind", ...}

    @property
    def kv_len(self):
        for L in self.layers:
            if L["kind"] == "attn":
                return L["kv"].length
        return None

    def snapshot(self):
        """Copy of the O(1) states; KV represented by its readable length only (EvSpark
        summary, Figure 1(d): slicing keeps the state at k and shortens the KV prefix)."""
        snap = []
        for L in self.layers:
            if L["kind"] == "fir":
                snap.append({"kind": "fir", "tail": L["tail"].copy()})
            elif L["kind"] == "iir":
                snap.append({"kind": "iir", "s": L["s"].copy()})
            else:
                snap.append({"kind": "attn", "length": L["kv"].length})
        return snap

    def restore(self, snap):
        """Return to a snapshot: shorten readable KV, put back FIR tail and IIR state."""
        for L, S in zip(self.layers, snap):
            if L["kind"] == "fir":
                L["tail"] = S["tail"].copy()
            elif L["kind"] == "iir":
                L["s"] = S["s"].copy()
            else:
                L["kv"].length = S["length"]

    def clone(self):
        return copy.deepcopy(self)


class Target:
    def __init__(self, wl, weights):
        self.wl = wl
        f = np.float64
        self.E = np.asarray(weights["embed"], dtype=f)
        self.head = np.asarray(weights["head"], dtype=f)
        self.layers = []
        for spec, W in zip(wl.layers, weights["layers"]):
            assert spec.kind == W["kind"]
            if spec.kind == "fir":
                self.layers.append({"kind": "fir", "L": spec.param,
                                    "w_in": np.asarray(W["w_in"], f),
                                    "taps": np.asarray(W["taps"], f),
                                    "w_out": np.asarray(W["w_out"], f)})
            elif spec.kind == "iir":
                self.layers.append({"kind": "iir", "N": spec.param,
                                    "w_in": np.asarray(W["w_in"], f),
                                    "lam": np.asarray(W["lam"], np.complex128),
                                    "b": np.asarray(W["b"], np.complex128),
                                    "c": np.asarray(W["c"], np.complex128),
                                    "w_out": np.asarray(W["w_out"], f)})
            else:
                self.layers.append({"kind": "attn", "H": spec.param, "dh": wl.head_dim,
                                    "wq": np.asarray(W["wq"], f), "wk": np.asarray(W["wk"], f),
                                    "wv": np.asarray(W["wv"], f), "wo": np.asarray(W["wo"], f)})

    # ---- state -------------------------------------------------------------------------
    def empty_state(self, kv_cap=64) -> SeqState:
        d = self.wl.d
        layers = []
        for L in self.layers:
            if L["kind"] == "fir":
                layers.append({"kind": "fir", "tail": np.zeros((L["L"] - 1, d))})
            elif L["kind"] == "iir":
                layers.append({"kind": "iir", "s": np.zeros((d, L["N"]), np.complex128)})
            else:
                layers.append({"kind": "attn", "kv": KVBuffer(L["H"], L["dh"], kv_cap)})
        return SeqState(layers)

    def state_from_arrays(self, st: dict, b: int, extra=64, kv_dtype=np.float64) -> SeqState:
        """State of sequence b from a generated state dict (see ``synth.gen_state``)."""
        layers = []
        n = int(st["kv_len"][b])
        for L, S in zip(self.layers, st["layers"]):
            if L["kind"] == "fir":
                layers.append({"kind": "fir", "tail": np.asarray(S["tail"][b], np.float64)})
            elif L["kind"] == "iir":
                layers.append({"kind": "iir", "s": np.asarray(S["s"][b], np.complex128)})
            else:
                kv = KVBuffer(L["H"], L["dh"], n + extra, S["k"][b][:, :n], S["v"][b][:, :n],
                              length=n, dtype=kv_dtype)
                layers.append({"kind": "attn", "kv": kv})
        return SeqState(layers)

    # ---- definition: one token ---------------------------------------------------------
    @staticmethod
    def rmsnorm(h):
        return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + EPS)

    def step(self, st: SeqState, x: int, trace: list | None = None) -> np.ndarray:
        """Consume token x: update ``st`` in place and return the next-token logits. This is
        the definition every other form is checked against (sequential decode; EvSpark
        summary, Interpretation paragraph 1, Lemmas 2 and 3)."""
        h = self.E[x].copy()
        for L, S in zip(self.layers, st.layers):
            xh = self.rmsnorm(h)
            if L["kind"] == "fir":
                v = xh @ L["w_in"]
                y, S["tail"] = fir_step(S["tail"], v, L["taps"])
                h = h + y @ L["w_out"]
                if trace is not None:
                    trace.append({"kind": "fir", "v": v})
            elif L["kind"] == "iir":
                u = xh @ L["w_in"]
                y, S["s"] = iir_step(S["s"], u, L["lam"], L["b"], L["c"])
                h = h + y @ L["w_out"]
                if trace is not None:
                    trace.append({"kind": "iir", "s": S["s"].copy(), "u": u})
            else:
                H, dh = L["H"], L["dh"]
                q = (xh @ L["wq"]).reshape(H, dh)
                k = (xh @ L["wk"]).reshape(H, dh)
                v = (xh @ L["wv"]).reshape(H, dh)
                kv = S["kv"]
                kv.append(k, v)
                n = kv.length
                o = np.empty((H, dh))
                for hh in range(H):
                    o[hh] = attend(q[hh], kv.k[hh, :n], kv.v[hh, :n])
                h = h + o.reshape(-1) @ L["wo"]
                if trace is not None:
                    trace.append({"kind": "attn", "k": k, "v": v})
        return self.rmsnorm(h) @ self.head

    # ---- independent block form (for the block-forward contract check) -----------------
    def block_forward(self, st: SeqState, tokens) -> tuple[np.ndarray, list]:
        """Forward over a whole block from ``st`` without mutating it.

        FIR as a per-channel ``numpy.convolve`` over [tail || block inputs]; IIR by the
        closed-form modal sum y_t = Re sum_n c_n (lam_n^{t+1} s_{-1,n}
        + b_n sum_{j<=t} lam_n^{t-j} u_j); attention as one masked score matrix over
        [readable prefix || block]. Returns logits [T, V] and per-layer block values
        (FIR inputs v [T,d], IIR states s [T,d,N], attention k, v [T,H,dh]).
        """
        tokens = np.asarray(tokens)
        T = len(tokens)
        h = self.E[tokens].copy()                                   # [T, d]
        layer_vals = []
        for L, S in zip(self.layers, st.layers):
            xh = self.rmsnorm(h)
            if L["kind"] == "fir":
                v = xh @ L["w_in"]                                  # [T, d]
                full = np.vstack([S["tail"], v])                    # [L-1+T, d]
                y = np.empty_like(v)
                for c in range(v.shape[1]):
                    y[:, c] = np.convolve(full[:, c], L["taps"][c], mode="valid")
                h = h + y @ L["w_out"]
                layer_vals.append({"kind": "fir", "v": v})
            elif L["kind"] == "iir":
                u = xh @ L["w_in"]                                  # [T, d]
                lam, b, c = L["lam"], L["b"], L["c"]
                t = np.arange(T)
                # powers lam^(t-j) for j <= t, zero above the diagonal
                expo = t[:, None] - t[None, :]
                mask = expo >= 0
                pw = np.where(mask[:, :, None, None],
                              lam[None, None] ** np.maximum(expo, 0)[:, :, None, None], 0)
                s_forced = np.einsum("tjdn,jd->tdn", pw, u) * b[None]
                s_free = (lam[None] ** (t[:, None, None] + 1)) * S["s"][None]
                s_all = s_forced + s_free                           # [T, d, N]
                y = np.real(np.sum(c[None] * s_all, axis=2))
                h = h + y @ L["w_out"]
                layer_vals.append({"kind": "iir", "s": s_all, "u": u})
            else:
                H, dh = L["H"], L["dh"]
                q = (xh @ L["wq"]).reshape(T, H, dh)
                k = (xh @ L["wk"]).reshape(T, H, dh)
                v = (xh @ L["wv"]).reshape(T, H, dh)
                n0 = S["kv"].length
                o = np.empty((T, H, dh))
                for hh in range(H):
                    Kall = np.vstack([S["kv"].k[hh, :n0].astype(np.float64), k[:, hh]])
                    Vall = np.vstack([S["kv"].v[hh, :n0].astype(np.float64), v[:, hh]])
                    sc = q[:, hh] @ Kall.T / np.sqrt(dh)            # [T, n0+T]
                    causal = np.arange(T)[:, None] >= np.arange(T)[None, :]
                    allow = np.hstack([np.ones((T, n0), bool), causal])
                    sc = np.where(allow, sc, -np.inf)
                    sc = sc - sc.max(axis=1, keepdims=True)
                    w = np.exp(sc)
                    o[:, hh] = (w / w.sum(axis=1, keepdims=True)) @ Vall
                h = h + o.reshape(T, -1) @ L["wo"]
                layer_vals.append({"kind": "attn", "k": k, "v": v})
        return self.rmsnorm(h) @ self.head, layer_vals
