"""Shared helpers for the GPU parity tests: build an oracle / library pair on the same
seeded inputs and compare them."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from synth import gen_prefix, gen_round, gen_state, gen_weights

# Tolerances (relative L2 error, per tensor and per row): fp32 1e-5, bf16 2e-2.
TOL = {"f32": 1e-5, "bf16": 2e-2}
# Near-tie thresholds used when comparing discrete decisions.
TAU = {"f32": 1e-5, "bf16": 2e-2}

# Worst errors seen per compared quantity: name -> [per-tensor, worst row, tolerance]
MARGINS: dict = {}
# Discrete decisions against the fp64 oracle's own, per workload variant (wl_key) ->
# {"rounds", "near_ties", "fp64_disagreements" (unflagged), "near_tie_disagreements"}
DECISIONS: dict = {}


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def rel_rows(a, b, lead: int) -> float:
    """Worst error over rows, each row's L2 error relative to max(its own norm, the RMS row
    norm of the reference): the first `lead` axes index the rows, the rest form one row.
    A row of typical or larger norm is held to a plain relative bound; a row whose norm is
    small by chance is measured against the typical row, so a wholly wrong row, channel or
    tile still shows as an error of order one."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    n = int(np.prod(b.shape[:lead])) if lead else 1
    a = a.reshape(n, -1)
    b = b.reshape(n, -1)
    if a.size == 0:
        return 0.0
    nb = np.linalg.norm(b, axis=1)
    floor = np.sqrt(np.mean(nb * nb))
    den = np.maximum(nb, floor)
    return float(np.max(np.linalg.norm(a - b, axis=1) / np.where(den > 0, den, 1.0)))


def check_close(name, a, b, lead, tol):
    """Assert the per-tensor relative error and the worst per-row error (rel_rows) are both
    within tol; records both. Returns the larger."""
    e = rel_l2(a, b)
    r = rel_rows(a, b, lead)
    m = MARGINS.setdefault(name, [0.0, 0.0, tol])
    m[0], m[1] = max(m[0], e), max(m[1], r)
    assert e <= tol, f"{name}: rel err {e:.3e} (tol {tol:g})"
    assert r <= tol, f"{name}: worst row rel err {r:.3e} (tol {tol:g}; whole tensor {e:.3e})"
    return max(e, r)


def wl_key(wl) -> str:
    """A name for a workload variant by its shape (tests replace fields of the named ones)."""
    kinds = "".join({"fir": "F", "iir": "I", "attn": "A"}[x.kind] + str(x.param) for x in wl.layers)
    return (f"d{wl.d}_{kinds}_b{wl.batch}c{wl.n_cand}_g{wl.gamma}_{wl.mode}_{wl.dtype}"
            + (f"_v{wl.vocab}" if wl.vocab != 512 else "")
            + (f"_{wl.cand_rule}" if wl.n_cand > 1 and wl.mode == "sampling" else ""))


def tally_decisions(wl, own, gk, gc, gcand):
    """Count the library's committed (k, correction, candidate) against the fp64 oracle's
    own decisions, per sequence: near-ties the oracle flags are counted apart; returns the
    number of unflagged disagreements."""
    tie = np.asarray(own[6], bool)
    agree = (np.asarray(gk) == own[3]) & (np.asarray(gc) == own[4])
    if wl.n_cand > 1:
        agree &= np.asarray(gcand) == own[5]
    bad = int((~agree & ~tie).sum())
    rec = DECISIONS.setdefault(wl_key(wl), {"rounds": 0, "near_ties": 0, "fp64_disagreements": 0,
                                            "near_tie_disagreements": 0})
    rec["rounds"] += len(tie)
    rec["near_ties"] += int(tie.sum())
    rec["fp64_disagreements"] += bad
    rec["near_tie_disagreements"] += int((~agree & tie).sum())
    return bad


def layer_list(wl):
    return [(s.kind, s.param) for s in wl.layers]


def make_verifier(wl, weights, t_max, near_tie_tau=None):
    from lossless_speculative_verify_gb300 import DeviceWeights, Verifier, make_config
    tau = TAU[wl.dtype] if near_tie_tau is None else near_tie_tau
    cfg = make_config(wl.d, layer_list(wl), wl.head_dim, wl.gamma, wl.batch, wl.n_cand, t_max,
                      wl.prefill_chunk, wl.dtype, wl.mode, wl.temperature, tau, wl.vocab, wl.cand_rule)
    dw = DeviceWeights(layer_list(wl), weights, wl.dtype)
    return Verifier(cfg, dw)


def _select(st, seqs):
    out = {"kv_len": st["kv_len"][seqs], "layers": []}
    for L in st["layers"]:
        out["layers"].append({k: (v[seqs] if k != "kind" else v) for k, v in L.items()})
    return out


class RoundOut:
    """own / kern: oracle decisions (k_c, corr_c, tie_c, k, corr, cand, tie) from its own
    fp64 logits and from the library's fp32 logits; gk, gc, gcand: the library's."""

    def __init__(self, own, kern, gk, gc, gcand, bp):
        self.own, self.kern, self.gk, self.gc, self.gcand, self.bp = own, kern, gk, gc, gcand, bp
        self.k, self.corr, self.cand, self.tie = own[3], own[4], own[5], own[6]


class _Res:
    def __init__(self, bp):
        self.logits, self.traces = bp["logits"], bp["traces"]


class Pair:
    """Oracle and library driven in lockstep."""

    def __init__(self, wl, t_max=None, weights=None):
        self.wl = wl
        self.weights = gen_weights(wl) if weights is None else weights
        self.tgt = oracle.Target(wl, self.weights)
        self.t_max = t_max or (wl.prefix_len + 16 * (wl.gamma + 1))
        self.ver = make_verifier(wl, self.weights, self.t_max)
        self.states = [self.tgt.empty_state() for _ in range(wl.batch)]

    # ---- state ---------------------------------------------------------------------------
    def prefill(self, P):
        toks = gen_prefix(self.wl, P)
        for b in range(self.wl.batch):
            oracle.prefill(self.tgt, self.states[b], toks[b])
        self.ver.prefill(torch.as_tensor(toks, dtype=torch.int32).cuda().contiguous())

    def import_synthetic(self, P, kv_dtype=np.float64):
        st = gen_state(self.wl, P)
        self.states = [self.tgt.state_from_arrays(st, b, kv_dtype=kv_dtype) for b in range(self.wl.batch)]
        self.ver.import_state(st)

    def oracle_state_arrays(self):
        """Oracle states in the library's import/export format."""
        B = self.wl.batch
        n = max(s.kv_len or 0 for s in self.states)
        out = {"kv_len": np.array([s.kv_len or 0 for s in self.states], np.int32), "layers": []}
        for li, spec in enumerate(self.wl.layers):
            if spec.kind == "attn":
                H, dh = spec.param, self.wl.head_dim
                K = np.zeros((B, H, n, dh))
                V = np.zeros((B, H, n, dh))
                for b, s in enumerate(self.states):
                    kv = s.layers[li]["kv"]
                    K[b, :, :kv.length] = kv.k[:, :kv.length]
                    V[b, :, :kv.length] = kv.v[:, :kv.length]
                out["layers"].append({"kind": "attn", "k": K, "v": V})
            elif spec.kind == "fir":
                out["layers"].append({"kind": "fir",
                                      "tail": np.stack([s.layers[li]["tail"] for s in self.states])})
            else:
                out["layers"].append({"kind": "iir",
                                      "s": np.stack([s.layers[li]["s"] for s in self.states])})
        return out

    def compare_state(self, tol=None, seqs=None, kv_from=0):
        """Exported library state against the oracle's. seqs limits the sequences compared;
        kv_from skips cache rows below it (rows the round did not touch)."""
        tol = TOL[self.wl.dtype] if tol is None else tol
        g = self.ver.export_state()
        o = self.oracle_state_arrays()
        if seqs is not None:
            g = _select(g, seqs)
            o = _select(o, seqs)
        np.testing.assert_array_equal(g["kv_len"], o["kv_len"])
        worst = 0.0
        for li, (a, b) in enumerate(zip(g["layers"], o["layers"])):
            if a["kind"] == "attn":
                for bb in range(len(o["kv_len"])):
                    n = int(o["kv_len"][bb])
                    for key in ("k", "v"):
                        # rows: (head, cache row)
                        e = check_close(f"{self.wl.dtype} cache {key} (per head, row)",
                                        a[key][bb, :, kv_from:n], b[key][bb, :, kv_from:n], 2, tol)
                        worst = max(worst, e)
            elif a["kind"] == "fir":
                # rows: (sequence, tail row)
                e = check_close(f"{self.wl.dtype} FIR tail (per sequence, row)", a["tail"], b["tail"], 2, tol)
                worst = max(worst, e)
            else:
                # rows: (sequence, channel), the channel's N complex poles
                e = check_close(f"{self.wl.dtype} IIR state (per sequence, channel)",
                                np.stack([a["s"].real, a["s"].imag], axis=-1),
                                np.stack([b["s"].real, b["s"].imag], axis=-1), 2, tol)
                worst = max(worst, e)
        return worst

    def compare_state_light(self, seqs, rows_from, tol=None):
        """Sliced state of the given sequences through read-only views of the library's
        buffers (no full export): kv_len, FIR tails, IIR states and the cache rows from
        rows_from to kv_len (the rows a round writes)."""
        wl = self.wl
        tol = TOL[wl.dtype] if tol is None else tol
        B, d, dh = wl.batch, wl.d, wl.head_dim
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        kvl = self.ver.buffer(7, -1, torch.int32, (B,)).cpu().numpy()
        for b in seqs:
            st = self.states[b]
            assert kvl[b] == st.kv_len, (b, kvl[b], st.kv_len)
            for li, spec in enumerate(wl.layers):
                L = st.layers[li]
                if spec.kind == "fir":
                    t = self.ver.buffer(8, li, torch.float32, (B, spec.param - 1, d))[b].cpu().numpy()
                    check_close(f"{wl.dtype} FIR tail (per sequence, row)", t, L["tail"], 1, tol)
                elif spec.kind == "iir":
                    t = self.ver.buffer(9, li, torch.float32, (B, d, spec.param, 2))[b].cpu().numpy()
                    check_close(f"{wl.dtype} IIR state (per sequence, channel)", t,
                                np.stack([L["s"].real, L["s"].imag], axis=-1), 1, tol)
                else:
                    H = spec.param
                    n = st.kv_len
                    for which, arr, key in ((3, L["kv"].k, "k"), (4, L["kv"].v, "v")):
                        c = self.ver.buffer(which, li, tdt, (B, H, self.t_max, dh))[b, :, rows_from:n]
                        check_close(f"{wl.dtype} cache {key} (per head, row)", c.float().cpu().numpy(),
                                    arr[:, rows_from:n], 2, tol)

    # ---- one round -------------------------------------------------------------------------
    def round_inputs(self, r, anchor=None):
        rnd = gen_round(self.wl, r, anchor=anchor)
        return rnd

    def run_round(self, rnd, check_block=True, tol=None, seqs=None):
        """Verify + slice on both sides from the current (identical) state.

        Decisions are checked in two ways: (1) the oracle's acceptance applied to the
        library's fp32 logits (the kernel's precision) must give exactly the library's k,
        correction and candidate unless a near-tie at fp32 resolution (tau 1e-5) is flagged;
        (2) the oracle's own fp64 decisions are returned for callers that compare them too.
        The oracle then commits the state at the library's (k, candidate), so both sides stay
        in lockstep and every slice is compared exactly."""
        wl = self.wl
        tol = TOL[wl.dtype] if tol is None else tol
        dev = lambda a, dt: torch.as_tensor(a, dtype=dt).cuda().contiguous()
        toks = dev(rnd["tokens"], torch.int32)
        sampling = wl.mode == "sampling"
        q = dev(rnd["q"], torch.float32) if sampling else None
        u = dev(rnd["u"], torch.float32) if sampling else None
        sq = list(range(wl.batch)) if seqs is None else list(seqs)
        sub = lambda a: None if a is None else np.asarray(a)[sq]
        states = [self.states[b] for b in sq]
        bp = oracle.block_pass(self.tgt, states, sub(rnd["tokens"]))
        own = oracle.accept_block(bp["logits"], sub(rnd["tokens"]), sub(rnd["q"]), sub(rnd["u"]),
                                  wl.mode, wl.temperature, TAU[wl.dtype], wl.cand_rule)
        k, corr, cand, tie = self.ver.verify(toks, q, u)
        self.round_launches = self.ver.launches          # kernels of the verify call
        torch.cuda.synchronize()
        if check_block:
            self.check_block(bp, tol, sq)
        B, C, T, V = wl.batch, wl.n_cand, wl.block, wl.vocab
        glog = self.ver.buffer(0, -1, torch.float32, (B, C, T, V)).cpu().numpy()[sq]
        kern = oracle.accept_block(glog, sub(rnd["tokens"]), sub(rnd["q"]), sub(rnd["u"]), wl.mode,
                                   wl.temperature, TAU["f32"], wl.cand_rule)
        gk, gc, gcand = k.cpu().numpy()[sq], corr.cpu().numpy()[sq], cand.cpu().numpy()[sq]
        gcand = gcand if C > 1 else np.zeros_like(gk)
        if C > 1:   # per-candidate words: accepted drafts (or depth on the path), corrections
            gkc = self.ver.buffer(10, -1, torch.int32, (B, C)).cpu().numpy()[sq]
            gcc = self.ver.buffer(11, -1, torch.int32, (B, C)).cpu().numpy()[sq]
        for i in range(len(sq)):
            if kern[6][i]:
                continue
            assert gk[i] == kern[3][i] and gc[i] == kern[4][i] and gcand[i] == kern[5][i], \
                (sq[i], gk, gc, gcand, kern[3:6])
            if C > 1:
                np.testing.assert_array_equal(gkc[i], kern[0][i])
                np.testing.assert_array_equal(gcc[i], kern[1][i])
        self.fp64_disagreements = tally_decisions(wl, own, gk, gc, gcand)
        oracle.commit(states, bp, gk, gcand)
        self.ver.slice(k, cand)
        self.round_launches += self.ver.launches         # plus the slice
        return RoundOut(own, kern, gk, gc, gcand, bp)

    def check_block(self, res, tol, sq=None):
        """Block forward outputs: logits, IIR scan inputs, FIR inputs, block K/V. (Each IIR
        state s_t enters the logits through the readout; the sliced s_k is compared after
        the slice.)"""
        res = _Res(res)
        wl = self.wl
        B, C, T, V, d = wl.batch, wl.n_cand, wl.block, wl.vocab, wl.d
        sq = list(range(B)) if sq is None else sq
        lg = self.ver.buffer(0, -1, torch.float32, (B, C, T, V)).cpu().numpy()[sq]
        # rows: (sequence, candidate, block position)
        check_close(f"{wl.dtype} logits (per sequence, candidate, position)", lg, res.logits, 3, tol)
        for li, spec in enumerate(wl.layers):
            if spec.kind == "iir":
                uin = self.ver.buffer(2, li, torch.float32, (B, C, T, d)).cpu().numpy()[sq]
                ref = np.array([[[res.traces[b][c][i][li]["u"] for i in range(T)] for c in range(C)]
                                for b in range(len(sq))])
                check_close(f"{wl.dtype} IIR scan inputs (per sequence, candidate, position)", uin, ref, 3, tol)
            elif spec.kind == "fir":
                Lm1 = spec.param - 1
                stage = self.ver.buffer(1, li, torch.float32, (B, C, Lm1 + T, d)).cpu().numpy()[sq]
                ref = np.array([[[res.traces[b][c][i][li]["v"] for i in range(T)] for c in range(C)]
                                for b in range(len(sq))])
                check_close(f"{wl.dtype} FIR block inputs (per sequence, candidate, position)",
                            stage[:, :, Lm1:], ref, 3, tol)
            elif C > 1:
                H, dh = spec.param, wl.head_dim
                tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
                for which, key in ((5, "k"), (6, "v")):
                    blk = self.ver.buffer(which, li, tdt, (B, C, H, T, dh)).float().cpu().numpy()[sq]
                    ref = np.array([[[res.traces[b][c][i][li][key] for i in range(T)] for c in range(C)]
                                    for b in range(len(sq))])                 # [B,C,T,H,dh]
                    # rows: (sequence, candidate, head, block position)
                    check_close(f"{wl.dtype} block {key} rows (per head, position)", blk,
                                ref.transpose(0, 1, 3, 2, 4), 4, tol)

    def resync_from_oracle(self):
        self.ver.import_state(self.oracle_state_arrays())
