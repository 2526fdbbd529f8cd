#!/usr/bin/env python
"""Benchmark: verified tokens/s of verify + slice rounds on one GB300 (or N replicas).

One step = one round of the hot path: block forward over [anchor, d_1..d_gamma] through
every FIR / modal-IIR / attention layer, softmax + acceptance, and state slicing at the
accepted index, for every sequence (and candidate) of the workload. Inputs are seeded and
synthetic (random-init weights of the stated shapes, a synthetic pre-round state of
P cached tokens, drafts drawn from Dirichlet q over ACGT), resident in HBM before the
timed region; L2 is flushed before every timed step.

--impl reference times the fp64 CPU oracle (the definition the library is checked
against) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "d1024_l8_p8k_bf16"
METRIC = "verified tokens/s (verify+slice rounds)"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="evs", choices=["evs", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-also", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-decode", action="store_true", help="skip the native-decode control leg")
    ap.add_argument("--no-ablation", action="store_true", help="skip the slice / replay ablation leg")
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
class Clocks:
    def __init__(self, index=0):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={index}", f"--query-gpu={q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------- CPU oracle
def oracle_rate(wl, seconds, rounds_from=0):
    """Oracle (as it stands) on a bounded sample: consecutive rounds from a synthetic state
    of P cached tokens until `seconds` elapse (at least one round)."""
    import oracle
    from synth import gen_round, gen_state, gen_weights
    w = gen_weights(wl)
    tgt = oracle.Target(wl, w)
    st = gen_state(wl)
    states = [tgt.state_from_arrays(st, b, extra=4096, kv_dtype=np.float32) for b in range(wl.batch)]
    del st
    tokens, rounds, steps = 0, 0, 0
    t0 = time.perf_counter()
    anchor = None
    while True:
        rnd = gen_round(wl, rounds_from + rounds, anchor=anchor)
        res = oracle.verify_round(tgt, states, rnd["tokens"], rnd["q"], rnd["u"], wl.mode,
                                  wl.temperature, rule=wl.cand_rule)
        anchor = res.corr
        tokens += int((res.k + 1).sum())
        rounds += 1
        steps += wl.rows
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": tokens / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{rounds} consecutive rounds ({steps} sequential fp64 decode steps) of "
                      f"{wl.name} from a synthetic state of {wl.prefix_len} cached tokens, "
                      f"{dt:.1f} s", "us_per_round": dt / rounds * 1e6}


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


# ------------------------------------------------------------------------------- GPU arm
def run_evs(args, wl, rank, world, light=False):
    import torch
    from lossless_speculative_verify_gb300.build import build
    from lossless_speculative_verify_gb300 import DeviceWeights, Verifier, make_config
    from synth import gen_round, gen_state, gen_weights

    build()
    dev = torch.device("cuda", torch.cuda.current_device())
    K, W = args.steps, args.warmup
    P, T = wl.prefix_len, wl.block
    n_prof = min(K, 8)
    n_abl = min(K, 8)                               # rounds of the slice / replay ablation
    rounds = W + 2 * K + 2 * n_prof + 2 * n_abl + 2
    dec_steps = W + K + 2                           # native decode steps of the control leg
    t_max = (P + rounds * T + dec_steps + 255) // 256 * 256
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
    del st
    # all rounds' inputs resident in HBM (and pinned on the host for the e2e leg)
    rin = [gen_round(wl, r) for r in range(rounds)]
    sampling = wl.mode == "sampling"
    host = {"tokens": torch.as_tensor(np.stack([r["tokens"] for r in rin])).pin_memory()}
    if sampling:
        host["q"] = torch.as_tensor(np.stack([r["q"] for r in rin])).pin_memory()
        host["u"] = torch.as_tensor(np.stack([r["u"] for r in rin])).pin_memory()
    devin = {k: v.to(dev) for k, v in host.items()}
    buf = {k: torch.empty_like(v[0]) for k, v in devin.items()}
    out_host = torch.empty((2, wl.batch), dtype=torch.int32).pin_memory()
    ver.corr.fill_(65)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    tok_acc = torch.zeros(wl.batch, dtype=torch.int64, device=dev)

    def one_round():
        ver.verify(buf["tokens"], buf.get("q"), buf.get("u"), anchor=ver.corr)
        ver.slice()

    def load_inputs(r, src):
        for k in buf:
            buf[k].copy_(src[k][r], non_blocking=True)

    with torch.cuda.stream(s):
        load_inputs(0, devin)
    one_round()                                     # eager round: loads every kernel
    launches_round = None
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
    with torch.cuda.stream(s):
        for _ in range(W):
            load_inputs(r % rounds, devin)
            replay()
            r += 1
    s.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(dev.index) if rank == 0 else None
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(s):
        for i in range(K):
            flush.zero_()
            evs[i][0].record(s)
            load_inputs(r % rounds, devin)
            replay()
            evs[i][1].record(s)
            tok_acc += ver.k + 1
            r += 1
    s.synchronize()
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs)
    tokens = int(tok_acc.sum().item())
    clk = clocks.stop() if clocks is not None else None
    abl = None if args.no_ablation else replay_ablation(ver, s, wl, lambda i: load_inputs(i % rounds, devin), buf,
                                                          r, n_abl)
    r += 2 * n_abl
    dec_ms = None if args.no_decode else decode_control(args, ver, s, flush, wl, K, W)
    if light:
        return dict(ms=ms, tokens=tokens, clocks=clk, flags=ver.flags(), graph=graph is not None, dec_ms=dec_ms,
                    ablation=abl)
    # end-to-end through the public API: pinned host inputs in, accepted length and
    # correction out, every step
    e2e_ms = 0.0
    e2e_tokens = 0
    with torch.cuda.stream(s):
        for i in range(K):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            load_inputs(r % rounds, host)
            replay()
            out_host[0].copy_(ver.k, non_blocking=True)
            out_host[1].copy_(ver.corr, non_blocking=True)
            b.record(s)
            s.synchronize()
            e2e_ms += a.elapsed_time(b)
            e2e_tokens += int(out_host[0].sum()) + wl.batch
            r += 1
    h2d = sum(v[0].numel() * v.element_size() for v in host.values())
    d2h = out_host.numel() * out_host.element_size()
    # per-kind kernel time: the library brackets every launch with events; the bracketed
    # rounds are captured in a graph (events become graph nodes, no host gaps) and replayed
    ver.profile(True)
    with torch.cuda.stream(s):
        for i in range(n_prof):                 # eager pass fills the event pool
            load_inputs(r % rounds, devin)
            one_round()
            r += 1
    ver.profile_read()
    prof_mode = "graph"
    try:
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp, stream=s):
            for i in range(n_prof):
                load_inputs((r + i) % rounds, devin)
                one_round()
        ver.profile(False)
        with torch.cuda.stream(s):
            flush.zero_()
            gp.replay()
        r += n_prof
        prof = ver.profile_read()
    except Exception:                          # event nodes unsupported: eager numbers
        ver.profile(True)
        prof_mode = "eager"
        with torch.cuda.stream(s):
            for i in range(n_prof):
                load_inputs(r % rounds, devin)
                one_round()
                r += 1
        prof = ver.profile_read()
    ver.profile(False)
    flags = ver.flags()
    ms, e2e_ms, tokens, e2e_tokens = aggregate(ms, e2e_ms, tokens, e2e_tokens, dev)
    return dict(ms=ms, tokens=tokens, e2e_ms=e2e_ms, e2e_tokens=e2e_tokens, h2d=h2d, d2h=d2h,
                prof=prof, n_prof=n_prof, prof_mode=prof_mode, launches_round=launches_round, clocks=clk,
                flags=flags, graph=graph is not None, dec_ms=dec_ms, ablation=abl)


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


def main():
    args = parse()
    from synth import get_workload
    wl = get_workload(args.workload)
    if args.prefix is not None:
        wl = wl.replace(prefix_len=args.prefix, name=f"{wl.name}@prefix{args.prefix}")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        # the oracle arm: each step a bounded sample of the same workload
        tot_tokens, tot_s, samples = 0, 0.0, []
        t_all = time.perf_counter()
        per = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
        for i in range(args.warmup + args.steps):
            res = oracle_rate(wl, per if i >= args.warmup else 0.0, rounds_from=i * 1000)
            if i >= args.warmup:
                samples.append(res)
        value = statistics.median(r["value"] for r in samples)
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": wl.name},
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                                 "sample": samples[0]["sample"]},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "wall_s": time.perf_counter() - t_all}
        print(json.dumps(line))
        return
    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    else:
        torch.cuda.set_device(0)
    out = run_evs(args, wl, rank, world)
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    K = args.steps
    pk, pk_kind = peaks()
    round_s = out["ms"] / K / 1e3
    P_mid = wl.prefix_len + (args.warmup + K) * 1          # cached rows during the timed rounds
    bmin = round_bytes_min(wl, P_mid)
    prof = out["prof"]
    dom = max((k for k in prof if prof[k][0] > 0), key=lambda k: prof[k][1])
    dom_bytes = kind_bytes(wl, P_mid, dom)
    roof = None
    if dom_bytes is not None and prof[dom][1] > 0:
        rounds_prof = out["n_prof"]
        achieved = dom_bytes * rounds_prof / (prof[dom][1] / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "traffic": traffic_per_round(wl, dom),
                "algorithmic_bytes_per_round": dom_bytes, "peak_source": pk_kind,
                "share_of_round": prof[dom][1] / sum(v[1] for v in prof.values()),
                "timing": f"event pairs around each launch, {out['prof_mode']} replay of {out['n_prof']} rounds"}
    line = {
        "metric": METRIC, "value": out["tokens"] / (out["ms"] / 1e3), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": out["ms"] / K,
        "us_per_round": out["ms"] / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "d": wl.d, "layers": wl.n_layers, "gamma": wl.gamma,
                   "batch": wl.batch, "n_cand": wl.n_cand, "prefix_tokens": wl.prefix_len,
                   "mode": wl.mode, "l2": "flushed (256 MiB write) before every timed step",
                   "graph": out["graph"], "parallelism": f"replicas x{world}"},
        "round_roofline": {"bytes_min": bmin, "us_at_peak": bmin / (pk["hbm_gbs"] * 1e9) * 1e6,
                           "frac": bmin / (pk["hbm_gbs"] * 1e9) / round_s},
        "roofline": roof,
        "kernels": {k: {"launches": v[0], "ms": round(v[1], 4)} for k, v in prof.items() if v[0]},
        "e2e": {"value": out["e2e_tokens"] / (out["e2e_ms"] / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": out["h2d"], "d2h_bytes_per_step": out["d2h"]},
        "gpu_launches": out["launches_round"] * K,
        "clocks": out["clocks"], "device_flags": out["flags"],
        "decode_control": control_line(wl, out["ms"] / K, out["dec_ms"]),
        "recovery_ablation": out["ablation"],
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_rate(wl, args.cpu_seconds)
    if world == 1 and not args.no_also:
        # the other bf16 workloads, measured the same way with fewer steps (context for the
        # roofline targets on the 4096-wide and long-context shapes)
        also = {}
        for name in ("d4096_l32_p8k_bf16", "d4096_l4_p256k_bf16", "d4096_l8_p32k_b4c4_bf16"):
            if name == wl.name:
                continue
            w2 = get_workload(name)
            sub = argparse.Namespace(**vars(args))
            sub.steps, sub.warmup = max(5, K // 4), 3
            o2 = run_evs(sub, w2, rank, world, light=True)
            r_s = o2["ms"] / sub.steps / 1e3
            b2 = round_bytes_min(w2, w2.prefix_len + sub.warmup + sub.steps)
            also[name] = {"us_per_round": round(r_s * 1e6, 2), "value": o2["tokens"] / (o2["ms"] / 1e3),
                          "unit": UNIT, "steps": sub.steps, "bytes_min": b2,
                          "round_roofline_frac": round(b2 / (pk["hbm_gbs"] * 1e9) / r_s, 4),
                          "clocks": o2["clocks"], "device_flags": o2["flags"],
                          "decode_control": control_line(w2, o2["ms"] / sub.steps, o2["dec_ms"]),
                          "recovery_ablation": o2["ablation"]}
            torch.cuda.empty_cache()
        line["also"] = also
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
