#!/usr/bin/env python
"""Benchmark: verified tokens/s of verify + slice rounds on one GB300 (or N replicas).

One step = one round of the hot path: block forward over [anchor, d_1..d_gamma] through
every FIR / modal-IIR / attention layer, softmax + acceptance, and state slicing at the
accepted index, for every sequence (and candidate) of the workload. Inputs are seeded and
synthetic (random-init weights of the stated shapes, a synthetic pre-round state of
P cached tokens, drafts drawn from Dirichlet q over ACGT), resident in HBM before the
timed region; L2 is flushed before every timed step.

The headline is the largest single-GPU workload (4 sequences x 4 candidate blocks of
gamma = 12 at width 4096, 8 layers, 32768 cached tokens each); the other bf16 workloads
are measured the same way under "also", each for about a second of timed rounds.

--impl reference times the fp64 CPU oracle (the definition the library is checked
against) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "d4096_l8_p32k_b4c4_bf16"
ALSO_WORKLOADS = ("d1024_l8_p8k_bf16", "d4096_l32_p8k_bf16", "d4096_l4_p256k_bf16",
                  "d4096_l8_p32k_b4c4_bf16")
METRIC = "verified tokens/s (verify+slice rounds)"
UNIT = "tokens/s"
N_INPUTS = 64            # distinct generated rounds the timed loops cycle through


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="evs", choices=["evs", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--also-seconds", type=float, default=1.2,
                    help="timed seconds of rounds for each secondary workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-also", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-decode", action="store_true", help="skip the native-decode control leg")
    ap.add_argument("--no-ablation", action="store_true", help="skip the slice / replay ablation leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--no-profile", action="store_true", help="skip the per-kind event profile")
    ap.add_argument("--prefix", type=int, default=None,
                    help="cached tokens per sequence instead of the workload's (small profiling "
                         "cases; the workload name then carries the override)")
    return ap.parse_args()


# ------------------------------------------------------------------------------- byte model
def es(wl):
    return 2 if wl.dtype == "bf16" else 4


def weight_bytes(wl):
    d, e = wl.d, es(wl)
    tot = wl.vocab * d * e
    for s in wl.layers:
        tot += (4 if s.kind == "attn" else 2) * d * d * e
    return tot


def kv_read_bytes(wl, P):
    return sum(1 for s in wl.layers if s.kind == "attn") * wl.batch * P * wl.d * 2 * es(wl)


def round_bytes_min(wl, P):
    """Weights read once + KV prefix read once + block K/V written + FIR/IIR state read and
    written once (per round)."""
    d, e, B = wl.d, es(wl), wl.batch
    kv_w = sum(1 for s in wl.layers if s.kind == "attn") * wl.rows * d * 2 * e
    st = 0
    for s in wl.layers:
        if s.kind == "fir":
            st += 2 * B * (s.param - 1) * d * 4
        elif s.kind == "iir":
            st += 2 * B * d * s.param * 8
    return weight_bytes(wl) + kv_read_bytes(wl, P) + kv_w + st


def kind_bytes(wl, P, kind):
    """Algorithmic bytes one round moves through kernels of one kind."""
    d, e, M = wl.d, es(wl), wl.rows
    if kind == "gemm":
        tot = 0
        for s in wl.layers:
            n_in = 3 * d if s.kind == "attn" else d
            tot += n_in * d * e + M * d * e + M * n_in * 4          # W_in / W_qkv
            tot += d * d * e + M * d * e + 2 * M * d * 4            # W_out / W_o (+ residual)
        tot += wl.vocab * d * e + M * d * e + M * wl.vocab * 4    # head
        return tot
    if kind == "attn":
        return kv_read_bytes(wl, P)
    return None


# ------------------------------------------------------------------------------- clocks
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown"}


class Clocks:
    """SM clock, power and throttle reasons sampled during a timed region.

    NVML (the library nvidia-smi reads) is polled from a thread every 2 ms, so a region of a
    few milliseconds still gets samples; without NVML, nvidia-smi is run at its 200 ms
    period. Only reads: nothing is set."""

    def __init__(self, device_index=0, uuid=None, period=0.002):
        self.sm, self.mx, self.reasons, self.power = [], [], set(), []
        self.p = None
        self.src = None
        self._stop = threading.Event()
        try:
            self._nvml_start(device_index, uuid, period)
            self.src = "nvml"
        except (OSError, AttributeError, RuntimeError):
            self._smi_start(device_index)

    def _nvml_start(self, index, uuid, period):
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        n = ctypes.c_uint()
        ok = False
        if uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(h)) == 0
        if not ok and lib.nvmlDeviceGetCount_v2(ctypes.byref(n)) == 0 and n.value == 1:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) == 0
        if not ok:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) == 0
        if not ok:
            raise RuntimeError("no NVML handle")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.lib, self.h = lib, h

        def poll():
            mhz, mx, mw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
            rs = ctypes.c_ulonglong()
            while not self._stop.is_set():
                if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:       # NVML_CLOCK_SM
                    self.sm.append(float(mhz.value))
                if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                    self.mx.append(float(mx.value))
                if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) == 0:
                    self.power.append(mw.value / 1e3)
                if reasons_fn(h, ctypes.byref(rs)) == 0:
                    for bit, name in _NVML_REASONS.items():
                        if rs.value & bit:
                            self.reasons.add(name)
                time.sleep(period)

        self.t = threading.Thread(target=poll, daemon=True)
        self.t.start()

    def _smi_start(self, index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
            self.src = "nvidia-smi"
        except OSError:
            self.p = None

    def stop(self):
        if self.src == "nvml":
            self._stop.set()
            self.t.join()
        elif self.p is not None:
            self.p.terminate()
            self.p.wait()
            self.f.seek(0)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in self.f.read().strip().splitlines():
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    self.sm.append(float(parts[1]))
                    self.mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        self.reasons.add(n)
            os.unlink(self.f.name)
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"], "samples": 0}
        return {"sm_mhz": statistics.median(self.sm) if self.sm else None,
                "sm_max_mhz": max(self.mx) if self.mx else None, "reasons": sorted(self.reasons),
                "samples": len(self.sm), "power_w_max": max(self.power) if self.power else None,
                "source": self.src}


# ------------------------------------------------------------------------------- CPU oracle
class OracleSample:
    """The fp64 oracle (as it stands) on one sequence of the workload: its weights and a
    synthetic state of P cached tokens for that sequence. Sequences are independent, so one
    sequence's rounds are a bounded sample whose verified tokens per second is the
    workload's rate on these cores. A round is taken one candidate block at a time (the
    oracle's block pass over one candidate from the pre-round state, which leaves the state
    unchanged), and after the last candidate the acceptance rule and the commit."""

    def __init__(self, wl):
        import oracle
        from synth import gen_state, gen_weights
        self.oracle = oracle
        self.wl1 = wl.replace(batch=1)
        self.tgt = oracle.Target(self.wl1, gen_weights(self.wl1))
        st = gen_state(self.wl1)
        self.state = [self.tgt.state_from_arrays(st, 0, extra=4096, kv_dtype=np.float32)]
        del st
        self.anchor = None
        self.rounds = 0
        self.cur = None

    def block(self, round_base=0):
        """One candidate block of the current round (a new round when none is open); after
        the last candidate, acceptance and commit. Returns the verified tokens the block
        completed (0 until the round's last block)."""
        from synth import gen_round
        wl, o = self.wl1, self.oracle
        C, T = wl.n_cand, wl.block
        if self.cur is None:
            rnd = gen_round(wl, round_base + self.rounds, anchor=self.anchor)
            bp = {"logits": np.zeros((1, C, T, wl.vocab)), "base": None, "snaps": [[None] * C],
                  "rows": [[None] * C], "traces": [[None] * C]}
            self.cur = [rnd, bp, 0]
        rnd, bp, c = self.cur
        one = o.block_pass(self.tgt, self.state, rnd["tokens"][:, c:c + 1])
        bp["logits"][0, c] = one["logits"][0, 0]
        bp["base"] = one["base"]
        for key in ("snaps", "rows", "traces"):
            bp[key][0][c] = one[key][0][0]
        self.cur[2] = c + 1
        if c + 1 < C:
            return 0
        acc = o.accept_block(bp["logits"], rnd["tokens"], rnd["q"], rnd["u"], wl.mode, wl.temperature, 0.0,
                             wl.cand_rule)
        k, corr, cand = acc[3], acc[4], acc[5]
        o.commit(self.state, bp, k, cand)
        self.anchor = corr
        self.rounds += 1
        self.cur = None
        return int((k + 1).sum())

    def run(self, seconds, round_base=0):
        """Whole consecutive rounds until `seconds` elapse (at least one)."""
        tokens, n = 0, 0
        t0 = time.perf_counter()
        while True:
            for _ in range(self.wl1.n_cand):
                tokens += self.block(round_base)
            n += 1
            if time.perf_counter() - t0 >= seconds:
                break
        return tokens, n, time.perf_counter() - t0

    def describe(self, n, dt, batch):
        wl = self.wl1
        steps = wl.n_cand * wl.block
        return (f"{n} consecutive rounds of one of the workload's {batch} sequences (all {wl.n_cand} "
                f"candidate blocks: {steps} sequential fp64 decode steps per round) of {wl.name}, from a "
                f"synthetic state of {wl.prefix_len} cached tokens, {dt:.1f} s")


def oracle_rate(wl, seconds):
    s = OracleSample(wl)
    tokens, n, dt = s.run(seconds)
    return {"value": tokens / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": s.describe(n, dt, wl.batch), "us_per_round": dt / n * 1e6 * wl.batch}


# ------------------------------------------------------------------------------- ranks
def aggregate(ms, e2e_ms, tokens, e2e_tokens, device):
    """Whole-job figures over the ranks of the process group (if any): the slowest rank's
    times, the sum of every rank's verified tokens."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms, e2e_ms, tokens, e2e_tokens
    t = torch.tensor([ms, e2e_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    c = torch.tensor([tokens, e2e_tokens], dtype=torch.int64, device=device)
    dist.all_reduce(c)
    return float(t[0]), float(t[1]), int(c[0]), int(c[1])


def traffic_per_round(wl, kind):
    """DRAM bytes one round's launches of a kernel kind moved in an ncu capture, as recorded
    in profiles/traffic.txt, if the kernel source is unchanged since (else None)."""
    import hashlib
    src = {"gemm": "gemm_tc.cu", "attn": "attn_fa.cu"}.get(kind)
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if src is None or not os.path.exists(path):
        return None
    digest = hashlib.sha256(open(os.path.join(ROOT, "lossless_speculative_verify_gb300", "csrc", src),
                                 "rb").read()).hexdigest()[:16]
    for line in open(path):
        f = line.split()
        if len(f) == 4 and f[0] == wl.name and f[1] == kind and f[3] == digest:
            return float(f[2])
    return None


def dominant_roofline(wl, P, prof, n_rounds, round_ms, pk, pk_kind):
    """Roofline of the kernel kind that takes the most time in a round. Its time per round
    is the sum of its launches' event-bracketed durations (every launch between two events,
    which only lengthens it: the events also break the overlap of dependent launches), an
    upper bound on its time, capped at the graph-timed round; the achieved bandwidth is
    therefore a lower bound."""
    if not prof:
        return None
    known = {k: v for k, v in prof.items() if v[0] > 0 and kind_bytes(wl, P, k) is not None}
    if not known:
        return None
    dom = max(known, key=lambda k: known[k][1])
    t_ev = known[dom][1] / n_rounds
    t_ms = min(t_ev, round_ms)
    b = kind_bytes(wl, P, dom)
    achieved = b / (t_ms / 1e3) / 1e9
    tot = sum(v[1] for v in prof.values())
    return {"bound": "hbm", "kernel": {"attn": "attn_fa_kernel", "gemm": "gemm_tc_kernel"}[dom],
            "kind": dom, "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": traffic_per_round(wl, dom),
            "algorithmic_bytes_per_round": b, "us_per_round": t_ms * 1e3,
            "event_us_per_round": t_ev * 1e3, "share_of_event_time": known[dom][1] / tot,
            "peak_source": f"hbm_gbs, {pk_kind}",
            "timing": f"sum of the kind's event-bracketed launches over {n_rounds} graph-replayed rounds "
                      "(an upper bound on its time), capped at the graph-timed round"}


# ------------------------------------------------------------------------------- GPU arm
def run_evs(args, wl, rank, world, steps, warmup, seconds=None, headline=True):
    """Measure one workload. With `seconds`, the timed rounds continue until that much device
    time has been timed (at least `steps` rounds), in chunks between which the synthetic
    pre-round state is imported again (untimed), so the cached length stays within a few
    blocks of P."""
    import torch
    from lossless_speculative_verify_gb300.build import build
    from lossless_speculative_verify_gb300 import DeviceWeights, Verifier, make_config
    from synth import gen_round, gen_state, gen_weights

    build()
    dev = torch.device("cuda", torch.cuda.current_device())
    P, T = wl.prefix_len, wl.block
    n_prof = 8
    n_abl = 8                                       # rounds of the slice / replay ablation
    chunk = max(1, max(64, P // 64) // T) if seconds else None
    # rows the state can grow by before it is imported again (or over the whole run)
    span = (chunk if chunk else warmup + steps) + 2 * steps + 2 * n_prof + 2 * n_abl + 4
    dec_steps = warmup + steps + 2
    t_max = (P + span * T + dec_steps + 255) // 256 * 256
    weights = gen_weights(wl)
    layers = [(s.kind, s.param) for s in wl.layers]
    dw = DeviceWeights(layers, weights, wl.dtype, dev)
    del weights
    cfg = make_config(wl.d, layers, wl.head_dim, wl.gamma, wl.batch, wl.n_cand, t_max,
                      wl.prefill_chunk, wl.dtype, wl.mode, wl.temperature, 0.0, wl.vocab, wl.cand_rule)
    s = torch.cuda.Stream(dev)
    ver = Verifier(cfg, dw, dev, stream=s)
    # synthetic pre-round state: O(1) FIR / IIR states from the seeded generator, KV rows
    # N(0,1) drawn on the device (seeded), P rows per sequence
    st = gen_state(wl, 0)
    st["kv_len"] = np.full(wl.batch, P, np.int32)
    g = torch.Generator(device=dev)
    g.manual_seed(4000 + wl.seed_base + 7919 * rank)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    for li, spec in enumerate(wl.layers):
        if spec.kind == "attn":
            shape = (wl.batch, spec.param, P, wl.head_dim)
            st["layers"][li]["k"] = torch.randn(shape, generator=g, device=dev).to(tdt)
            st["layers"][li]["v"] = torch.randn(shape, generator=g, device=dev).to(tdt)
    ver.import_state(st)
    # generated rounds' inputs resident in HBM (and pinned on the host for the e2e leg)
    rin = [gen_round(wl, r) for r in range(N_INPUTS)]
    sampling = wl.mode == "sampling"
    host = {"tokens": torch.as_tensor(np.stack([r["tokens"] for r in rin])).pin_memory()}
    if sampling:
        host["q"] = torch.as_tensor(np.stack([r["q"] for r in rin])).pin_memory()
        host["u"] = torch.as_tensor(np.stack([r["u"] for r in rin])).pin_memory()
    devin = {k: v.to(dev) for k, v in host.items()}
    buf = {k: torch.empty_like(v[0]) for k, v in devin.items()}
    ver.corr.fill_(65)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    tok_acc = torch.zeros(wl.batch, dtype=torch.int64, device=dev)

    def one_round():
        ver.verify(buf["tokens"], buf.get("q"), buf.get("u"), anchor=ver.corr)
        ver.slice()

    def load_inputs(r, src):
        for k in buf:
            buf[k].copy_(src[k][r % N_INPUTS], non_blocking=True)

    with torch.cuda.stream(s):
        load_inputs(0, devin)
    one_round()                                     # eager round: loads every kernel
    graph = None
    with torch.cuda.stream(s):
        ver.verify(buf["tokens"], buf.get("q"), buf.get("u"), anchor=ver.corr)
        lv = ver.launches
        ver.slice()
        launches_round = lv + ver.launches
        if not args.no_graph:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                one_round()
    replay = graph.replay if graph is not None else one_round
    r = 1

    def reimport():
        s.synchronize()
        ver.import_state(st)
        s.synchronize()

    with torch.cuda.stream(s):
        for _ in range(warmup):
            load_inputs(r, devin)
            replay()
            r += 1
    if chunk:
        reimport()
    s.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(dev.index, str(getattr(torch.cuda.get_device_properties(dev), "uuid", "") or "")) \
        if rank == 0 else None
    kv_view = ver.buffer(7, -1, torch.int32, (wl.batch,))      # readable lengths (read only)
    ms, done, kv_rows = 0.0, 0, 0.0
    while True:
        n = chunk or steps
        kv0 = float(kv_view.double().mean())
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(s):
            for i in range(n):
                flush.zero_()
                evs[i][0].record(s)
                load_inputs(r, devin)
                replay()
                evs[i][1].record(s)
                tok_acc += ver.k + 1
                r += 1
        s.synchronize()
        ms += sum(a.elapsed_time(b) for a, b in evs)
        done += n
        kv_rows += n * (kv0 + float(kv_view.double().mean())) / 2   # cached rows grow linearly
        if not chunk or (done >= steps and ms >= seconds * 1e3) or done >= 100000:
            break
        reimport()
    torch.cuda.synchronize()
    tokens = int(tok_acc.sum().item())
    clk = clocks.stop() if clocks is not None else None
    if chunk:
        reimport()
    out = dict(ms=ms, steps=done, tokens=tokens, clocks=clk, graph=graph is not None,
               launches_round=launches_round, P_timed=kv_rows / done, n_prof=n_prof)
    out["ablation"] = None if args.no_ablation else replay_ablation(ver, s, wl, lambda i: load_inputs(i, devin),
                                                                    buf, r, n_abl)
    r += 2 * n_abl
    # per-kind kernel time: the library brackets every launch with events; the bracketed
    # rounds are captured in a graph (events become graph nodes, no host gaps) and replayed
    out["prof"], out["prof_mode"] = (None, None) if args.no_profile else \
        kind_profile(ver, s, flush, lambda i: load_inputs(i, devin), one_round, r, n_prof)
    r += 2 * n_prof
    if chunk:
        reimport()
    out["dec_ms"] = None if args.no_decode else decode_control(args, ver, s, flush, wl, steps, warmup)
    if headline and not args.no_e2e:
        if chunk:
            reimport()
        out.update(e2e_leg(ver, s, flush, wl, host, buf, r, steps))
        r += steps
    out["flags"] = ver.flags()
    ms, e2e_ms, tokens, e2e_tokens = aggregate(out["ms"], out.get("e2e_ms", 0.0), out["tokens"],
                                               out.get("e2e_tokens", 0), dev)
    out.update(ms=ms, e2e_ms=e2e_ms, tokens=tokens, e2e_tokens=e2e_tokens)
    del ver, st, devin, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def e2e_leg(ver, s, flush, wl, host, buf, r0, steps):
    """End to end through the public API, one C-ABI call per step of the round: pinned
    host inputs copied in (tokens, q, u), evs_verify_block and evs_slice_state called
    eagerly, the accepted length and correction read back to the host; events bracket each
    step from the first copy to the last, and the host waits for every step's result."""
    import torch
    out_host = torch.empty((2, wl.batch), dtype=torch.int32).pin_memory()
    anchor = ver.corr
    e2e_ms, e2e_tokens = 0.0, 0
    with torch.cuda.stream(s):
        for i in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            for k in buf:
                buf[k].copy_(host[k][(r0 + i) % N_INPUTS], non_blocking=True)
            ver.verify(buf["tokens"], buf.get("q"), buf.get("u"), anchor=anchor)
            ver.slice()
            out_host[0].copy_(ver.k, non_blocking=True)
            out_host[1].copy_(ver.corr, non_blocking=True)
            b.record(s)
            s.synchronize()
            e2e_ms += a.elapsed_time(b)
            e2e_tokens += int(out_host[0].sum()) + wl.batch
    h2d = sum(v[0].numel() * v.element_size() for v in host.values())
    d2h = out_host.numel() * out_host.element_size()
    return {"e2e_ms": e2e_ms, "e2e_tokens": e2e_tokens, "h2d": h2d, "d2h": d2h}


def kind_profile(ver, s, flush, load, one_round, r0, n):
    """{kind: (launches, ms)} over n rounds, every launch bracketed by two events."""
    import torch
    ver.profile(True)
    with torch.cuda.stream(s):
        for i in range(n):                      # eager pass fills the event pool
            load(r0 + i)
            one_round()
    ver.profile_read()
    mode = "graph"
    try:
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp, stream=s):
            for i in range(n):
                load(r0 + n + i)
                one_round()
        ver.profile(False)
        with torch.cuda.stream(s):
            flush.zero_()
            gp.replay()
        prof = ver.profile_read()
    except Exception:                          # event nodes unsupported: eager numbers
        ver.profile(True)
        mode = "eager"
        with torch.cuda.stream(s):
            for i in range(n):
                load(r0 + n + i)
                one_round()
        prof = ver.profile_read()
    ver.profile(False)
    return prof, f"{mode} replay of {n} rounds"


def replay_ablation(ver, s, wl, load, buf, r0, n):
    """State recovery after a verify, two ways, on the same rounds (one sequence only): the
    slice, and the replay ablation (k read back, then a second committed forward over the
    accepted tokens). Each is bracketed by events on the stream after an eager verify; the
    replay's bracket includes the host round trip for k. Returns mean µs of each."""
    import torch
    if wl.batch != 1:
        return None
    anc = torch.empty_like(ver.corr)
    out = {}
    for leg in ("slice", "replay"):
        tot, acc = 0.0, 0
        for i in range(n):
            with torch.cuda.stream(s):
                load(r0 + i + (n if leg == "replay" else 0))
                anc.copy_(ver.corr)
                ver.verify(buf["tokens"], buf.get("q"), buf.get("u"), anchor=anc)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s)
                if leg == "slice":
                    ver.slice()
                else:
                    ver.replay(buf["tokens"], anchor=anc)
                b.record(s)
            s.synchronize()
            tot += a.elapsed_time(b)
            acc += int(ver.k.item()) + 1
        out[f"{leg}_us"] = round(tot / n * 1e3, 2)
        out[f"{leg}_tokens_per_round"] = acc / n
    out["replay_over_slice"] = out["replay_us"] / out["slice_us"]
    return out


def decode_control(args, ver, s, flush, wl, K, W):
    """Native decoding on the same handle and state: one token per sequence per step (the
    target's own loop), timed like the rounds (graph replay, L2 flushed before each step).
    Returns ms per step."""
    import torch
    B = wl.batch
    dev = ver.next.device
    g = torch.Generator(device=dev)
    g.manual_seed(5000 + wl.seed_base)
    u = torch.rand(B, generator=g, device=dev) if wl.mode == "sampling" else None
    with torch.cuda.stream(s):
        ver.next.fill_(65)
        ver.decode(ver.next, u)                        # eager step: next token in place
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            ver.decode(ver.next, u)
    step = graph.replay if graph is not None else (lambda: ver.decode(ver.next, u))
    with torch.cuda.stream(s):
        for _ in range(W):
            step()
    s.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(s):
        for i in range(K):
            flush.zero_()
            evs[i][0].record(s)
            step()
            evs[i][1].record(s)
    s.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / K


def control_line(wl, round_ms, dec_ms):
    """The identity-drafter control against native throughput: a drafter that always agrees
    gets every draft accepted, gamma+1 tokens per sequence per round. The round's kernels do
    the same work whatever the tokens (only the slice copies depend on k), so the measured
    round time stands for it."""
    if dec_ms is None:
        return None
    B, T = wl.batch, wl.gamma + 1
    return {"native_us_per_step": round(dec_ms * 1e3, 2), "native_tokens_per_s": B / (dec_ms / 1e3),
            "identity_drafter_tokens_per_s": B * T / (round_ms / 1e3),
            "identity_drafter_vs_native": T * dec_ms / round_ms}


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def workload_record(wl, out, pk, pk_kind):
    """µs per round, throughput and both rooflines of one measured workload."""
    K = out["steps"]
    round_ms = out["ms"] / K
    bmin = round_bytes_min(wl, out["P_timed"])
    rec = {"us_per_round": round(round_ms * 1e3, 2), "value": out["tokens"] / (out["ms"] / 1e3), "unit": UNIT,
           "steps": K, "timed_s": round(out["ms"] / 1e3, 3),
           "round_roofline": {"bytes_min": bmin, "us_at_peak": bmin / (pk["hbm_gbs"] * 1e9) * 1e6,
                              "frac": bmin / (pk["hbm_gbs"] * 1e9) / (round_ms / 1e3)},
           "roofline": dominant_roofline(wl, out["P_timed"], out["prof"], out["n_prof"], round_ms, pk, pk_kind),
           "kernels": None if not out["prof"] else
           {k: {"launches": v[0], "ms": round(v[1], 4)} for k, v in out["prof"].items() if v[0]},
           "kernel_profile": out["prof_mode"],
           "clocks": out["clocks"], "device_flags": out["flags"],
           "decode_control": control_line(wl, round_ms, out["dec_ms"]),
           "recovery_ablation": out["ablation"]}
    c = out["clocks"] or {}
    if c.get("sm_mhz"):
        rec["us_x_ghz"] = round(round_ms * 1e3 * c["sm_mhz"] / 1e3, 2)
    return rec


def reference_arm(args, wl):
    """The fp64 oracle as it stands on the host cores. Each step is one candidate block of
    one sequence (gamma+1 sequential decode steps; after a sequence's last candidate block,
    its acceptance and commit): every n_cand consecutive steps complete one sequence-round.
    The value is the verified tokens of the completed rounds over the time of their
    steps."""
    t_all = time.perf_counter()
    smp = OracleSample(wl)
    C = wl.n_cand
    for i in range(args.warmup):
        smp.block()
    while smp.cur is not None:                       # timed steps start at a round boundary
        smp.block()
    tokens, t_done, t_open, blocks, rounds = 0, 0.0, 0.0, 0, 0
    for i in range(args.steps):
        t0 = time.perf_counter()
        got = smp.block(round_base=1000)
        t_open += time.perf_counter() - t0
        blocks += 1
        if smp.cur is None:                          # a round completed with this block
            tokens += got
            t_done += t_open
            t_open = 0.0
            rounds += 1
    if rounds == 0:                                  # fewer steps than candidates: finish one
        while smp.cur is not None:
            t0 = time.perf_counter()
            tokens += smp.block(round_base=1000)
            t_open += time.perf_counter() - t0
        t_done, rounds = t_open, 1
    value = tokens / t_done
    sample = (f"per step one candidate block of one of the workload's {wl.batch} sequences ({wl.block} sequential "
              f"fp64 decode steps of {wl.name} from a synthetic state of {wl.prefix_len} cached tokens); "
              f"{rounds} sequence-rounds of {C} blocks completed in {t_done:.1f} s")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t_all}
    print(json.dumps(line))


def main():
    args = parse()
    from synth import get_workload
    wl = get_workload(args.workload)
    if args.prefix is not None:
        wl = wl.replace(prefix_len=args.prefix, name=f"{wl.name}@prefix{args.prefix}")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            reference_arm(args, wl)
        return
    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    else:
        torch.cuda.set_device(0)
    K = args.steps
    out = run_evs(args, wl, rank, world, K, args.warmup)
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    pk, pk_kind = peaks()
    rec = workload_record(wl, out, pk, pk_kind)
    line = {
        "metric": METRIC, "value": out["tokens"] / (out["ms"] / 1e3), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": out["ms"] / K,
        "us_per_round": out["ms"] / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "d": wl.d, "layers": wl.n_layers, "gamma": wl.gamma,
                   "batch": wl.batch, "n_cand": wl.n_cand, "prefix_tokens": wl.prefix_len,
                   "mode": wl.mode, "l2": "flushed (256 MiB write) before every timed step",
                   "graph": out["graph"], "parallelism": f"replicas x{world}"},
        "round_roofline": rec["round_roofline"],
        "roofline": rec["roofline"],
        "kernels": rec["kernels"], "kernel_profile": rec["kernel_profile"],
        "gpu_launches": out["launches_round"] * K,
        "clocks": out["clocks"], "device_flags": out["flags"],
        "decode_control": rec["decode_control"],
        "recovery_ablation": rec["recovery_ablation"],
    }
    if "us_x_ghz" in rec:
        line["us_x_ghz"] = rec["us_x_ghz"]
    if "e2e_ms" in out and out["e2e_ms"] > 0:
        line["e2e"] = {"value": out["e2e_tokens"] / (out["e2e_ms"] / 1e3), "unit": UNIT,
                       "h2d_bytes_per_step": out["h2d"], "d2h_bytes_per_step": out["d2h"],
                       "path": "eager evs_verify_block + evs_slice_state per step, pinned host inputs "
                               "copied in and k / correction read back inside the timed region"}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_rate(wl, args.cpu_seconds)
    if world == 1 and not args.no_also:
        # the other bf16 workloads, about a second of timed rounds each, with their own
        # clocks, dominant-kernel roofline and round roofline
        also = {}
        for name in ALSO_WORKLOADS:
            if name == wl.name:
                continue
            w2 = get_workload(name)
            o2 = run_evs(args, w2, rank, world, max(K, 10), 3, seconds=args.also_seconds, headline=False)
            also[name] = workload_record(w2, o2, pk, pk_kind)
        line["also"] = also
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
