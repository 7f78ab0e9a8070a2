#!/usr/bin/env python3
"""Benchmark of the routed-expert MXFP4 MoE layer on GB300.

Default workload (``--workload gptoss128``): the gpt-oss-120b-shaped layer,
K = I = 2880, 128 experts, top-4 softmax routing, one MoE call at each of
T = 1, 4, 16 and 32 tokens per step (the metric's "1-32 tokens"). Each call
uses its own layer's weights (8 distinct layers, 1.69 GB of packed weights
each), so between two uses of one layer the other calls stream >= 2 GB and
the 129 MB L2 holds nothing useful: inputs are larger than L2.

``--workload prefill`` times the glm256 prefill chunk (T = 8192, 65,536
token-expert pairs) instead.

Printed: one JSON line (rank 0). ``value`` is microseconds per MoE call
(whole job: all calls of all ranks / time), taken from CUDA-graph replays of
the step with events on the replay stream. ``roofline`` is the dominant kernel
(decode phase 1, gate/up projection) timed with CUDA events around each of its
launches over a second timed pass. ``e2e`` repeats the metric through the C-ABI
with host buffers (pinned host -> device copies of each call's activations and
routing, device -> host copy of its output, inside the timed region).
``--impl reference`` times the CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mxfp4_mixture_experts_gb300 import synth  # noqa: E402

PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = ("\u00b5s per MoE layer call and achieved HBM GB/s vs peak at 1\u201332 tokens; "
          "prefill TFLOP/s")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: one independent copy of the workload per GPU)
# ---------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate_us_per_call(max_elapsed_ms: float, calls_per_rank: int, world: int) -> float:
    """Whole-job microseconds per MoE call: every rank runs calls_per_rank calls
    in (at most) max_elapsed_ms."""
    return max_elapsed_ms * 1000.0 / (calls_per_rank * world)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(self.rows), "reasons": reasons}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def touched_experts(ids: torch.Tensor, E: int) -> int:
    v = ids[(ids >= 0) & (ids < E)]
    return int(torch.unique(v).numel())


def expert_bytes(K: int, I: int) -> int:
    """Packed bytes + scales of one expert (w13 and w2)."""
    return 3 * I * K // 2 + 3 * I * K // 32


def w13_bytes(K: int, I: int) -> int:
    return 2 * I * K // 2 + 2 * I * K // 32


class DecodeWorkload:
    name = "gptoss128"
    tokens = (1, 4, 16, 32)
    layers = 8

    def __init__(self, dev):
        from mxfp4_mixture_experts_gb300 import moe
        self.moe = moe
        self.shape = synth.SHAPES[self.name]
        s = self.shape
        self.dev = dev
        self.L = []
        for l in range(self.layers):
            T = self.tokens[l % len(self.tokens)]
            rng = np.random.Generator(np.random.PCG64(l))
            hidden, logits, ids, w = synth.draw_activations(s, T, rng)
            w13, s13, w2, s2 = synth.draw_weights_cuda(s, seed=0, layer=l, device=dev)
            ly = dict(T=T, hidden=hidden.to(dev), ids=ids.to(dev), w=w.to(dev), w13=w13, s13=s13,
                      w2=w2, s2=s2, out=torch.empty(T, s.K, dtype=torch.bfloat16, device=dev),
                      host_hidden=hidden.pin_memory(), host_ids=ids.pin_memory(),
                      host_w=w.pin_memory(),
                      host_out=torch.empty(T, s.K, dtype=torch.bfloat16).pin_memory())
            ly["D"] = touched_experts(ly["ids"], s.E)
            self.L.append(ly)
        Tmax = max(self.tokens)
        self.ws = moe.new_workspace(Tmax, s.K, s.I, s.E, s.topk, dev)
        self.calls_per_step = len(self.tokens)

    def step_layers(self, step: int):
        n = self.calls_per_step
        return [self.L[(step * n + i) % self.layers] for i in range(n)]

    def call(self, ly, stream=None):
        self.moe.forward(ly["hidden"], ly["ids"], ly["w"], ly["w13"], ly["s13"], ly["w2"],
                         ly["s2"], out=ly["out"], workspace=self.ws, stream=stream)

    def call_e2e(self, ly, stream):
        ly["hidden"].copy_(ly["host_hidden"], non_blocking=True)
        ly["ids"].copy_(ly["host_ids"], non_blocking=True)
        ly["w"].copy_(ly["host_w"], non_blocking=True)
        self.call(ly, stream)
        ly["host_out"].copy_(ly["out"], non_blocking=True)

    def e2e_bytes(self, ly):
        T, K, k = ly["T"], self.shape.K, self.shape.topk
        return T * K * 2 + 2 * T * k * 4, T * K * 2

    def alg_bytes(self, ly):
        s = self.shape
        return ly["D"] * expert_bytes(s.K, s.I) + 4 * ly["T"] * s.K

    def config(self):
        return decode_config(self.shape, self.tokens, self.layers)


def decode_config(s, tokens, layers):
    return {"workload": "gptoss128 decode: MoE layer K=I=2880, 128 experts, top-4 softmax "
                        "routing, one call at each of T=1,4,16,32 tokens per step",
            "K": s.K, "I": s.I, "E": s.E, "topk": s.topk, "tokens": list(tokens),
            "layers": layers,
            "l2": "inputs larger than L2: 8 distinct layers (1.69 GB packed each) rotate",
            "weights": "uniform random MXFP4 bytes, E8M0 scales 118..124 (synthetic)"}


# ---------------------------------------------------------------------------
def time_graph_loop(wl, steps: int, warmup: int, dist: Dist):
    """Headline timing: each step is captured once as a CUDA graph (two graphs
    alternate over the layer ring) and replayed."""
    stream = torch.cuda.Stream()
    n_graphs = wl.layers // wl.calls_per_step
    graphs = []
    with torch.cuda.stream(stream):
        for gi in range(n_graphs):          # eager warm-up of every layer first
            for ly in wl.step_layers(gi):
                wl.call(ly)
    stream.synchronize()
    for gi in range(n_graphs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for ly in wl.step_layers(gi):
                wl.call(ly)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for s in range(warmup):
            graphs[s % n_graphs].replay()
    stream.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    time.sleep(0.3)
    t_wall = time.perf_counter()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for s in range(steps):
            graphs[s % n_graphs].replay()
        e1.record(stream)
    stream.synchronize()
    t_wall = time.perf_counter() - t_wall
    torch.cuda.synchronize()
    dist.barrier()
    ck = clocks.stop()
    return e0.elapsed_time(e1), ck, t_wall


def time_phases(wl, steps: int, warmup: int):
    """Per-kernel durations: events recorded by the library around each kernel."""
    from mxfp4_mixture_experts_gb300 import moe
    stream = torch.cuda.Stream()
    per_T = {T: [] for T in wl.tokens}
    w13 = []          # (alg bytes, ms) per phase-1 launch
    with torch.cuda.stream(stream):
        for s in range(warmup + steps):
            recs = []
            for ly in wl.step_layers(s):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                moe.set_phase_events(ev)
                wl.call(ly)
                recs.append((ly, ev))
            moe.set_phase_events(None)
            stream.synchronize()
            if s < warmup:
                continue
            for ly, ev in recs:
                t13 = ev[0].elapsed_time(ev[1])
                t2 = ev[1].elapsed_time(ev[2])
                tc = ev[2].elapsed_time(ev[3])
                per_T[ly["T"]].append((t13 + t2 + tc, ly, (t13, t2, tc)))
                sh = wl.shape
                w13.append((ly["D"] * w13_bytes(sh.K, sh.I), t13))
    return per_T, w13


def time_e2e(wl, steps: int, warmup: int):
    stream = torch.cuda.Stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    h2d = d2h = 0
    with torch.cuda.stream(stream):
        for s in range(warmup):
            for ly in wl.step_layers(s):
                wl.call_e2e(ly, stream)
        stream.synchronize()
        e0.record(stream)
        for s in range(steps):
            for ly in wl.step_layers(s):
                wl.call_e2e(ly, stream)
                a, b = wl.e2e_bytes(ly)
                h2d += a
                d2h += b
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1), h2d // steps, d2h // steps


def cpu_oracle_sample(wl, budget_s: float = 15.0):
    """The oracle as it stands, timed on this host on single calls of the
    workload (smallest T first) until about budget_s of CPU work."""
    from oracle import mxfp4_moe_oracle as O
    times, sample = [], []
    t_start = time.perf_counter()
    for ly in sorted(wl.L, key=lambda l: l["T"]):
        if time.perf_counter() - t_start > budget_s and times:
            break
        ids = ly["ids"].cpu().numpy().astype(np.int64)
        E = wl.shape.E
        used = np.unique(ids[(ids >= 0) & (ids < E)])
        idx = torch.as_tensor(used, device=ly["w13"].device)
        host = [t.index_select(0, idx).cpu().numpy() for t in (ly["w13"], ly["s13"], ly["w2"], ly["s2"])]
        remap = np.full(E, -1)
        remap[used] = np.arange(len(used))
        sub = remap[ids]
        hb = ly["hidden"].cpu().view(torch.int16).numpy().view(np.uint16)
        w = ly["w"].cpu().numpy()
        t0 = time.perf_counter()
        O.forward(hb, sub, w, *host)
        times.append(time.perf_counter() - t0)
        sample.append(ly["T"])
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        cores = os.cpu_count()
    us = statistics.mean(times) * 1e6
    return {"value": us, "unit": "us_per_moe_call", "cores": cores, "kind": "oracle",
            "sample": f"{len(times)} single oracle calls of the same workload at T={sample} "
                      f"(float64 numpy, {sum(times):.1f} s of CPU work)"}


# ---------------------------------------------------------------------------
def run_ours(args, dist: Dist):
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks()
    if args.workload != "gptoss128":
        raise SystemExit(f"workload {args.workload} is not wired into the benchmark yet")
    wl = DecodeWorkload(dev)
    elapsed_ms, clocks, t_wall = time_graph_loop(wl, args.steps, args.warmup, dist)
    elapsed_ms = dist.max(elapsed_ms)
    calls = args.steps * wl.calls_per_step
    value = aggregate_us_per_call(elapsed_ms, calls, dist.world)
    per_T_raw, w13 = time_phases(wl, args.steps, min(args.warmup, 3))
    e2e_ms, h2d, d2h = time_e2e(wl, args.steps, args.warmup)
    e2e_ms = dist.max(e2e_ms)
    per_T = {}
    hbm = peaks["hbm_gbs"]
    for T, recs in per_T_raw.items():
        ms = statistics.median([r[0] for r in recs])
        b = statistics.mean([wl.alg_bytes(r[1]) for r in recs])
        phases = [round(statistics.median([r[2][i] for r in recs]) * 1000, 2) for i in range(3)]
        per_T[str(T)] = {"us": round(ms * 1000, 2), "phase_us": phases, "alg_bytes": int(b),
                         "gbs": round(b / (ms * 1e-3) / 1e9, 1),
                         "frac_of_8tbs": round(b / (ms * 1e-3) / 8e12, 3),
                         "frac_of_measured": round(b / (ms * 1e-3) / 1e9 / hbm, 3)}
    tot_b = sum(b for b, _ in w13)
    tot_ms = sum(t for _, t in w13)
    achieved = tot_b / (tot_ms * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "us_per_call",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": wl.config(),
        "per_T": per_T,
        "roofline": {"kernel": "decode_kernel<1> (w13 gate/up + SwiGLU)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 3), "peak_kind": peak_kind,
                     "traffic": None,
                     "alg_bytes_per_launch": int(tot_b / max(len(w13), 1)),
                     "avg_launch_us": round(tot_ms / max(len(w13), 1) * 1000, 2)},
        "e2e": {"value": round(aggregate_us_per_call(e2e_ms, calls, dist.world), 3),
                "unit": "us_per_call", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": 3 * calls,
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if dist.rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_oracle_sample(wl)
    return out


def run_reference(args, dist: Dist):
    """The CPU oracle as the reference arm, on the same workload."""
    if dist.rank != 0:
        return None
    from oracle import mxfp4_moe_oracle as O
    s = synth.SHAPES["gptoss128"]
    rng = np.random.Generator(np.random.PCG64(0))
    T = 1
    hidden, _, ids, w = synth.draw_activations(s, T, rng)
    ids = ids.numpy().astype(np.int64)
    used = np.unique(ids)
    remap = np.full(s.E, -1)
    remap[used] = np.arange(len(used))
    g = np.random.Generator(np.random.PCG64(1))
    n = len(used)
    w13 = g.integers(0, 256, (n, 2 * s.I, s.K // 2), dtype=np.uint8)
    s13 = g.integers(118, 125, (n, 2 * s.I, s.K // 32), dtype=np.uint8)
    w2 = g.integers(0, 256, (n, s.K, s.I // 2), dtype=np.uint8)
    s2 = g.integers(118, 125, (n, s.K, s.I // 32), dtype=np.uint8)
    hb = hidden.view(torch.int16).numpy().view(np.uint16)
    args_ = (hb, remap[ids], w.numpy(), w13, s13, w2, s2)
    for _ in range(args.warmup):
        O.forward(*args_)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.forward(*args_)
    el = time.perf_counter() - t0
    us = el / args.steps * 1e6
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        cores = os.cpu_count()
    return {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us_per_call",
            "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": decode_config(s, DecodeWorkload.tokens, DecodeWorkload.layers),
            "cpu_baseline": {"value": round(us, 1), "unit": "us_per_call", "cores": cores,
                             "kind": "oracle",
                             "sample": "each step: one T=1 call of the workload (4 touched "
                                       "experts), float64 numpy oracle"},
            "e2e": {"value": round(us, 1), "unit": "us_per_call", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_profile_case(args):
    """`--profile-case NAME:T`: warm-up + steps forward calls of one layer of a
    workload, no timing; the command profilers (ncu) run."""
    from mxfp4_mixture_experts_gb300 import moe
    name, T = args.profile_case.split(":")
    T = int(T)
    shape = synth.SHAPES[name]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hidden, _, ids, w = synth.draw_activations(shape, T, np.random.Generator(np.random.PCG64(T)))
    w13, s13, w2, s2 = synth.draw_weights_cuda(shape, seed=0, layer=0, device=dev)
    hidden, ids, w = hidden.to(dev), ids.to(dev), w.to(dev)
    ws = moe.new_workspace(T, shape.K, shape.I, shape.E, shape.topk, dev)
    out = torch.empty(T, shape.K, dtype=torch.bfloat16, device=dev)
    for _ in range(args.warmup + args.steps):
        moe.forward(hidden, ids, w, w13, s13, w2, s2, out=out, workspace=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": args.profile_case, "calls": args.warmup + args.steps,
                      "touched_experts": touched_experts(ids, shape.E)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gptoss128", choices=["gptoss128", "prefill"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", default=None,
                    help="NAME:T -- run warmup+steps calls of one layer, untimed (for ncu)")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    dist = Dist()
    try:
        if args.impl == "reference":
            out = run_reference(args, dist)
        else:
            if args.gpus != dist.world and dist.world > 1:
                raise SystemExit("--gpus must match WORLD_SIZE")
            out = run_ours(args, dist)
        if out is not None and dist.rank == 0:
            print(json.dumps(out), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
