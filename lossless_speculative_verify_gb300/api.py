"""Thin Python surface over the evs C-ABI (PyTorch supplies device memory and streams).

Every method marshals tensors into pointers and calls one entry point of ``libevs.so``;
none of the method's arithmetic happens here.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import _lib as L

_KIND = {"fir": L.LAYER_FIR, "iir": L.LAYER_IIR, "attn": L.LAYER_ATTN}


def _vp(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _dev(x, device, dt):
    if isinstance(x, torch.Tensor):
        return x.to(device=device, dtype=dt).contiguous()
    return torch.as_tensor(np.asarray(x, np.float32)).to(device).to(dt).contiguous()


class _DeviceArray:
    """Exposes a raw device pointer through __cuda_array_interface__ (for torch.as_tensor)."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(int(s) for s in shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}


def make_config(d, layers, head_dim, gamma, batch, n_cand, t_max, prefill_chunk, dtype, mode,
                temperature=1.0, near_tie_tau=0.0, vocab=512, cand_rule="recursive") -> L.Config:
    """layers: sequence of (kind, param) with kind in {"fir", "iir", "attn"}; cand_rule:
    "recursive" (lossless) or "max_accept", for several candidates under sampling."""
    cfg = L.Config()
    cfg.d, cfg.vocab, cfg.n_layers = d, vocab, len(layers)
    for i, (kind, param) in enumerate(layers):
        cfg.layer_kind[i] = _KIND[kind]
        cfg.layer_param[i] = param
    cfg.head_dim, cfg.gamma, cfg.batch, cfg.n_cand = head_dim, gamma, batch, n_cand
    cfg.t_max, cfg.prefill_chunk = t_max, prefill_chunk
    cfg.dtype = L.DTYPE_BF16 if dtype == "bf16" else L.DTYPE_F32
    cfg.mode = L.MODE_SAMPLING if mode == "sampling" else L.MODE_GREEDY
    cfg.temperature, cfg.near_tie_tau = temperature, near_tie_tau
    cfg.cand_rule = {"recursive": L.CAND_RECURSIVE, "max_accept": L.CAND_MAX_ACCEPT}[cand_rule]
    return cfg


def workspace_bytes(cfg: L.Config) -> int:
    return int(L.load().evs_workspace_bytes(C.byref(cfg)))


class DeviceWeights:
    """Target weights on the device in the library's layout.

    Input is the math convention (``y = x @ W``): embed [V,d], head [d,V]; FIR w_in, taps
    [d,L], w_out; IIR w_in, lam/b/c complex [d,N], w_out; attention wq, wk, wv, wo. Matrices
    become out-major (transposed), q/k/v are stacked into one [3d, d] matrix and complex
    coefficients become interleaved (re, im) fp32 pairs.
    """

    def __init__(self, layers, w: dict, dtype: str, device="cuda"):
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.keep = []

        def dev(a, dt=tdt, transpose=False):
            t = torch.as_tensor(np.ascontiguousarray(a, dtype=np.float32)).to(device)
            if transpose:
                t = t.t()
            t = t.to(dt).contiguous()
            self.keep.append(t)
            return t

        def cplx(a):
            a = np.ascontiguousarray(a, dtype=np.complex64)
            return dev(a.view(np.float32).reshape(a.shape + (2,)), torch.float32)

        s = L.Weights()
        s.embed = _vp(dev(w["embed"]))
        s.head = _vp(dev(w["head"], transpose=True))
        for i, ((kind, _), W) in enumerate(zip(layers, w["layers"])):
            lw = s.layer[i]
            if kind == "fir":
                lw.w_in = _vp(dev(W["w_in"], transpose=True))
                lw.w_out = _vp(dev(W["w_out"], transpose=True))
                lw.fir_taps = _vp(dev(W["taps"], torch.float32))
            elif kind == "iir":
                lw.w_in = _vp(dev(W["w_in"], transpose=True))
                lw.w_out = _vp(dev(W["w_out"], transpose=True))
                lw.iir_lambda = _vp(cplx(W["lam"]))
                lw.iir_b = _vp(cplx(W["b"]))
                lw.iir_c = _vp(cplx(W["c"]))
            else:
                qkv = np.concatenate([W["wq"], W["wk"], W["wv"]], axis=1)   # [d, 3d]
                lw.w_qkv = _vp(dev(qkv, transpose=True))
                lw.w_o = _vp(dev(W["wo"], transpose=True))
        self.struct = s


class Verifier:
    """One evs handle: workspace, state and the verify / slice calls."""

    def __init__(self, cfg: L.Config, weights: DeviceWeights, device="cuda", stream=None):
        self.lib = L.load()
        self.cfg = cfg
        self.weights = weights
        self.device = torch.device(device)
        nbytes = workspace_bytes(cfg)
        if nbytes == 0:
            raise ValueError("invalid evs configuration")
        self.ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        base = (self.ws.data_ptr() + 255) & ~255
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        h = C.c_void_p()
        L.check(self.lib.evs_create(C.byref(cfg), C.byref(weights.struct), C.c_void_p(base), nbytes,
                                    C.c_void_p(self.stream.cuda_stream), C.byref(h)), "evs_create")
        self.h = h
        B, Cn = cfg.batch, cfg.n_cand
        z = lambda n: torch.zeros(n, dtype=torch.int32, device=self.device)
        self.k, self.corr, self.cand, self.tie = z(B), z(B), z(B), z(B)
        self.next, self.next_tie = z(B), z(B)
        self.kinds = [cfg.layer_kind[i] for i in range(cfg.n_layers)]
        self.params = [cfg.layer_param[i] for i in range(cfg.n_layers)]

    # ---- calls -------------------------------------------------------------------------
    def prefill(self, tokens: torch.Tensor):
        assert tokens.dtype == torch.int32 and tokens.is_contiguous()
        L.check(self.lib.evs_prefill(self.h, _vp(tokens), tokens.shape[-1]), "evs_prefill")

    def verify(self, tokens, q=None, u=None, anchor=None, out=None):
        k, corr, cand, tie = out if out is not None else (self.k, self.corr, self.cand, self.tie)
        L.check(self.lib.evs_verify_block(self.h, _vp(tokens), _vp(anchor), _vp(q), _vp(u), _vp(k),
                                          _vp(corr), _vp(cand), _vp(tie)), "evs_verify_block")
        return k, corr, cand, tie

    def slice(self, k=None, cand=None):
        k = self.k if k is None else k
        cand = self.cand if cand is None else cand
        L.check(self.lib.evs_slice_state(self.h, _vp(k), _vp(cand)), "evs_slice_state")

    def replay(self, tokens, k=None, cand=None, anchor=None):
        """Replay-based recovery after a verify (ablation of slice; one sequence only)."""
        k = self.k if k is None else k
        cand = self.cand if cand is None else cand
        L.check(self.lib.evs_replay_state(self.h, _vp(tokens), _vp(anchor), _vp(k), _vp(cand)),
                "evs_replay_state")

    def decode(self, tokens, u=None, out=None):
        """One native decode step: consume tokens [B], return (next [B], near_tie [B])."""
        nxt, tie = out if out is not None else (self.next, self.next_tie)
        L.check(self.lib.evs_decode_step(self.h, _vp(tokens), _vp(u), _vp(nxt), _vp(tie)), "evs_decode_step")
        return nxt, tie

    def reset(self):
        L.check(self.lib.evs_reset(self.h), "evs_reset")

    def set_stream(self, stream):
        self.stream = stream
        L.check(self.lib.evs_set_stream(self.h, C.c_void_p(stream.cuda_stream)), "evs_set_stream")

    @property
    def launches(self) -> int:
        return int(self.lib.evs_last_launch_count(self.h))

    def profile(self, on: bool):
        L.check(self.lib.evs_profile_enable(self.h, 1 if on else 0), "evs_profile_enable")

    def profile_read(self) -> dict:
        """{kind: (launches, ms)} since the previous read (see EVS_K_* in evs.h)."""
        n = len(L.KERNEL_KINDS)
        la = (C.c_int32 * n)()
        ms = (C.c_float * n)()
        L.check(self.lib.evs_profile_read(self.h, la, ms, n), "evs_profile_read")
        return {k: (int(la[i]), float(ms[i])) for i, k in enumerate(L.KERNEL_KINDS)}

    def flags(self, clear=True) -> int:
        f = C.c_uint32()
        L.check(self.lib.evs_device_flags(self.h, C.byref(f), 1 if clear else 0), "evs_device_flags")
        return int(f.value)

    # ---- state ---------------------------------------------------------------------------
    def import_state(self, st: dict):
        """st: {"kv_len": int [B], "layers": [{"k","v"} [B,H,P,dh] | {"tail"} [B,L-1,d] |
        {"s"} complex [B,d,N]]} as NumPy arrays or tensors."""
        tdt = torch.bfloat16 if self.cfg.dtype == L.DTYPE_BF16 else torch.float32
        view = L.StateView()
        kv = (C.c_int32 * self.cfg.batch)(*[int(x) for x in np.asarray(st["kv_len"])])
        view.kv_len = kv
        keep = []
        stride = 1
        for i, S in enumerate(st["layers"]):
            if self.kinds[i] == L.LAYER_ATTN:
                kt, vt = _dev(S["k"], self.device, tdt), _dev(S["v"], self.device, tdt)
                stride = kt.shape[2]
                keep += [kt, vt]
                view.k[i], view.v[i] = kt.data_ptr(), vt.data_ptr()
            elif self.kinds[i] == L.LAYER_FIR:
                t = torch.as_tensor(np.asarray(S["tail"], np.float32)).to(self.device).contiguous()
                keep.append(t)
                view.fir_tail[i] = t.data_ptr()
            else:
                s = np.ascontiguousarray(S["s"], dtype=np.complex64)
                t = torch.as_tensor(s.view(np.float32).reshape(s.shape + (2,))).to(self.device).contiguous()
                keep.append(t)
                view.iir_state[i] = t.data_ptr()
        view.t_stride = stride
        torch.cuda.synchronize(self.device)        # sources may come from another stream
        L.check(self.lib.evs_import_state(self.h, C.byref(view)), "evs_import_state")
        del keep

    def export_state(self, rows: int | None = None) -> dict:
        """State as NumPy arrays in the import format (K/V rows [0, max kv_len))."""
        cfg = self.cfg
        B, d, dh = cfg.batch, cfg.d, cfg.head_dim
        tdt = torch.bfloat16 if cfg.dtype == L.DTYPE_BF16 else torch.float32
        kvl = self.buffer(L.BUF_KV_LEN, -1, torch.int32, (B,)).cpu().numpy()
        n = int(kvl.max()) if rows is None else rows
        view = L.StateView()
        host_len = (C.c_int32 * B)()
        view.kv_len = host_len
        view.t_stride = max(n, 1)
        bufs = []
        for i in range(cfg.n_layers):
            kind, p = self.kinds[i], self.params[i]
            if kind == L.LAYER_ATTN:
                kt = torch.zeros((B, p, max(n, 1), dh), dtype=tdt, device=self.device)
                vt = torch.zeros_like(kt)
                view.k[i], view.v[i] = kt.data_ptr(), vt.data_ptr()
                bufs.append(("attn", kt, vt))
            elif kind == L.LAYER_FIR:
                t = torch.zeros((B, p - 1, d), dtype=torch.float32, device=self.device)
                view.fir_tail[i] = t.data_ptr()
                bufs.append(("fir", t))
            else:
                t = torch.zeros((B, d, p, 2), dtype=torch.float32, device=self.device)
                view.iir_state[i] = t.data_ptr()
                bufs.append(("iir", t))
        L.check(self.lib.evs_export_state(self.h, C.byref(view)), "evs_export_state")
        out = {"kv_len": np.array(host_len[:], dtype=np.int32), "layers": []}
        for b in bufs:
            if b[0] == "attn":
                out["layers"].append({"kind": "attn", "k": b[1][:, :, :n].float().cpu().numpy(),
                                      "v": b[2][:, :, :n].float().cpu().numpy()})
            elif b[0] == "fir":
                out["layers"].append({"kind": "fir", "tail": b[1].cpu().numpy()})
            else:
                a = b[1].cpu().numpy()
                out["layers"].append({"kind": "iir", "s": a[..., 0] + 1j * a[..., 1]})
        return out

    def buffer(self, which: int, layer: int, dtype, shape) -> torch.Tensor:
        """Read-only tensor view of an internal buffer (see EVS_BUF_* in evs.h)."""
        info = L.BufferInfo()
        L.check(self.lib.evs_debug_buffer(self.h, which, layer, C.byref(info)), "evs_debug_buffer")
        typestr = {torch.float32: "<f4", torch.int32: "<i4", torch.bfloat16: "<i2"}[dtype]
        n = int(np.prod(shape))
        esize = 2 if dtype == torch.bfloat16 else 4
        assert n * esize <= info.bytes, "requested view larger than the buffer"
        t = torch.as_tensor(_DeviceArray(info.ptr, shape, typestr), device=self.device)
        if dtype == torch.bfloat16:
            t = t.view(torch.bfloat16)
        return t

    def close(self):
        if getattr(self, "h", None):
            self.lib.evs_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
