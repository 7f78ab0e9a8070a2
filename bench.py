#!/usr/bin/env python3
"""Benchmark of the routed-expert MXFP4 MoE layer on GB300.

Default workload (``--workload gptoss128``): the gpt-oss-120b-shaped layer,
K = I = 2880, 128 experts, top-4 softmax routing, one MoE call at each of
T = 1, 4, 16 and 32 tokens per step (the metric's "1-32 tokens"). Each call
uses its own layer's weights (8 distinct layers, 1.69 GB of packed weights
each), so between two uses of one layer the other calls stream >= 2 GB and
the 129 MB L2 holds nothing useful: inputs are larger than L2.

``--workload prefill`` times the prefill chunk on the 6144 x 2048 shape
instead (T = 8192 tokens, 256 experts, top-8 sigmoid routing: 65,536
token-expert pairs) and reports TFLOP/s of the two grouped GEMMs; the default
line carries the same measurement, shorter, under ``prefill``.

Printed: one JSON line (rank 0). ``value`` is microseconds per MoE call
(whole job: all calls of all ranks / time), taken from CUDA-graph replays of
two steps at a time (the 8 calls on the 8 layers, the pages' chain of 8
calls) with events on the replay stream. ``per_T`` and ``roofline`` come
from a second pass at each T: a chain of 8 calls (one cooperative decode
launch each: w13 + SwiGLU, w2, combine) on 8 distinct layers captured in one
graph, median replay time / 8 (the pages' protocol), against the touched
experts' packed bytes. ``e2e`` repeats the metric through the C-ABI
with host buffers: every step copies its calls' activations and routing up
from one pinned host buffer (one copy) and their outputs down (one copy),
inside the timed region.
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
                      host_w=w.pin_memory())
            ly["D"] = touched_experts(ly["ids"], s.E)
            self.L.append(ly)
        Tmax = max(self.tokens)
        self.ws = moe.new_workspace(Tmax, s.K, s.I, s.E, s.topk, dev)
        self.calls_per_step = len(self.tokens)
        self._pack_steps()

    def _pack_steps(self):
        """The end-to-end pass moves a step the way a serving loop does: the
        step's inputs (every call's hidden rows, routing ids and weights) sit
        in one pinned host buffer and go up in one copy, and the step's outputs
        come back in one copy. Each call reads and writes views of the two
        device buffers."""
        def align(n):
            return (n + 255) // 256 * 256
        self.packs = []
        n = self.calls_per_step
        for g in range(self.layers // n):
            lys = self.L[g * n:(g + 1) * n]
            srcs = [t for ly in lys for t in (ly["host_hidden"], ly["host_ids"], ly["host_w"])]
            offs, o = [], 0
            for t in srcs:
                offs.append(o)
                o += align(t.numel() * t.element_size())
            host_in = torch.zeros(o, dtype=torch.uint8).pin_memory()
            for t, off in zip(srcs, offs):
                nb = t.numel() * t.element_size()
                host_in[off:off + nb].copy_(t.contiguous().view(-1).view(torch.uint8))
            dev_in = torch.empty(o, dtype=torch.uint8, device=self.dev)
            views = []
            for t, off in zip(srcs, offs):
                nb = t.numel() * t.element_size()
                views.append(dev_in[off:off + nb].view(t.dtype).view(t.shape))
            out_offs, oo = [], 0
            for ly in lys:
                out_offs.append(oo)
                oo += align(ly["out"].numel() * 2)
            dev_out = torch.empty(oo, dtype=torch.uint8, device=self.dev)
            host_out = torch.empty(oo, dtype=torch.uint8).pin_memory()
            outs = [dev_out[off:off + ly["out"].numel() * 2].view(torch.bfloat16).view(ly["out"].shape)
                    for ly, off in zip(lys, out_offs)]
            calls = [(ly, views[3 * i], views[3 * i + 1], views[3 * i + 2], outs[i])
                     for i, ly in enumerate(lys)]
            h2d = sum(t.numel() * t.element_size() for t in srcs)
            d2h = sum(ly["out"].numel() * 2 for ly in lys)
            self.packs.append(dict(host_in=host_in, dev_in=dev_in, dev_out=dev_out,
                                   host_out=host_out, calls=calls, h2d=h2d, d2h=d2h))

    def step_e2e(self, step: int, stream):
        """One step end to end: its inputs up in one copy, its calls, its
        outputs down in one copy. Returns the bytes moved each way."""
        pk = self.packs[step % len(self.packs)]
        pk["dev_in"].copy_(pk["host_in"], non_blocking=True)
        for ly, hidden, ids, w, out in pk["calls"]:
            self.moe.forward(hidden, ids, w, ly["w13"], ly["s13"], ly["w2"], ly["s2"], out=out,
                             workspace=self.ws, stream=stream)
        pk["host_out"].copy_(pk["dev_out"], non_blocking=True)
        return pk["h2d"], pk["d2h"]

    def step_layers(self, step: int):
        n = self.calls_per_step
        return [self.L[(step * n + i) % self.layers] for i in range(n)]

    def call(self, ly, stream=None):
        self.moe.forward(ly["hidden"], ly["ids"], ly["w"], ly["w13"], ly["s13"], ly["w2"],
                         ly["s2"], out=ly["out"], workspace=self.ws, stream=stream)

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


class PrefillWorkload:
    """One prefill chunk: T = 8192 tokens on the 6144 x 2048, 256-expert,
    top-8 shape. 4.8 GB of packed weights and 805 MB of permuted activations
    per call: inputs larger than L2."""
    name = "prefill256"
    T = 8192

    def __init__(self, dev):
        from mxfp4_mixture_experts_gb300 import moe
        self.moe = moe
        self.shape = s = synth.SHAPES[self.name]
        self.dev = dev
        rng = np.random.Generator(np.random.PCG64(self.T))
        hidden, logits, ids, w = synth.draw_activations(s, self.T, rng)
        self.w13, self.s13, self.w2, self.s2 = synth.draw_weights_cuda(s, seed=0, layer=0,
                                                                      device=dev)
        self.hidden, self.ids, self.w = hidden.to(dev), ids.to(dev), w.to(dev)
        self.host_hidden, self.host_ids, self.host_w = (hidden.pin_memory(), ids.pin_memory(),
                                                        w.pin_memory())
        self.out = torch.empty(self.T, s.K, dtype=torch.bfloat16, device=dev)
        self.host_out = torch.empty(self.T, s.K, dtype=torch.bfloat16).pin_memory()
        self.ws = moe.new_workspace(self.T, s.K, s.I, s.E, s.topk, dev)
        ids_np = ids.numpy()
        self.routes = int(((ids_np >= 0) & (ids_np < s.E)).sum())
        self.D = touched_experts(self.ids, s.E)

    def flops(self):
        """(GEMM1, GEMM2) multiply-add flops: 2 per MAC over the valid routes."""
        s = self.shape
        return 2.0 * self.routes * s.K * 2 * s.I, 2.0 * self.routes * s.I * s.K

    def call(self, stream=None):
        self.moe.forward(self.hidden, self.ids, self.w, self.w13, self.s13, self.w2, self.s2,
                         out=self.out, workspace=self.ws, path=2, stream=stream)

    def call_e2e(self, stream):
        self.hidden.copy_(self.host_hidden, non_blocking=True)
        self.ids.copy_(self.host_ids, non_blocking=True)
        self.w.copy_(self.host_w, non_blocking=True)
        self.call(stream)
        self.host_out.copy_(self.out, non_blocking=True)

    def e2e_bytes(self):
        s = self.shape
        return self.T * s.K * 2 + 2 * self.T * s.topk * 4, self.T * s.K * 2

    def config(self):
        s = self.shape
        return {"workload": "prefill chunk: MoE layer K=6144, I=2048, 256 experts, top-8 "
                            "sigmoid routing, T=8192 tokens (65,536 token-expert pairs)",
                "K": s.K, "I": s.I, "E": s.E, "topk": s.topk, "tokens": self.T,
                "l2": "inputs larger than L2: 4.8 GB packed weights, 805 MB permuted "
                      "activations per call",
                "weights": "uniform random MXFP4 bytes, E8M0 scales 118..124 (synthetic)"}


def time_prefill(wl: PrefillWorkload, steps: int, warmup: int, dist: Dist):
    """Graph-replayed calls (headline), then per-kernel events, then e2e."""
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        wl.call()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        wl.call()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
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
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    t_wall = time.perf_counter() - t_wall
    torch.cuda.synchronize()
    dist.barrier()
    ck = clocks.stop()
    ms = e0.elapsed_time(e1)
    # per kernel: events 0..4 around route+gather, GEMM1, GEMM2, combine
    from mxfp4_mixture_experts_gb300 import moe
    phases = []
    with torch.cuda.stream(stream):
        for i in range(warmup + steps):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            moe.set_phase_events(ev)
            wl.call()
            moe.set_phase_events(None)
            stream.synchronize()
            if i >= warmup:
                phases.append([ev[j].elapsed_time(ev[j + 1]) for j in range(4)])
    # end to end through the public call with host buffers
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            wl.call_e2e(stream)
        stream.synchronize()
        e0.record(stream)
        for _ in range(steps):
            wl.call_e2e(stream)
        e1.record(stream)
    stream.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    return ms, phases, e2e_ms, ck, t_wall


def prefill_cpu_sample(wl: PrefillWorkload, budget_s: float = 15.0):
    """The oracle on a bounded sample of the chunk's tokens (first 4 tokens,
    then more until about budget_s), scaled to TFLOP/s."""
    from oracle import mxfp4_moe_oracle as O
    s = wl.shape
    ids = wl.ids.cpu().numpy().astype(np.int64)
    hb = wl.hidden.cpu().view(torch.int16).numpy().view(np.uint16)
    w = wl.w.cpu().numpy()
    done, flops, el = 0, 0.0, 0.0
    n = 4
    while el < budget_s and done + n <= wl.T:
        tok = np.arange(done, done + n)
        sub = ids[tok]
        used = np.unique(sub[(sub >= 0) & (sub < s.E)])
        remap = np.full(s.E, -1)
        remap[used] = np.arange(len(used))
        idx = torch.as_tensor(used, device=wl.w13.device)
        host = [t.index_select(0, idx).cpu().numpy() for t in (wl.w13, wl.s13, wl.w2, wl.s2)]
        t0 = time.perf_counter()
        O.forward(hb[tok], remap[sub], w[tok], *host)
        el += time.perf_counter() - t0
        flops += 2.0 * int(((sub >= 0) & (sub < s.E)).sum()) * 3 * s.I * s.K
        done += n
        n *= 2
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        cores = os.cpu_count()
    return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"the first {done} of the chunk's 8192 tokens through the float64 numpy "
                      f"oracle ({el:.1f} s of CPU work), flops of the sampled routes / time"}


def run_prefill(args, dist: Dist, steps: int, warmup: int, cpu: bool):
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks()
    wl = PrefillWorkload(dev)
    ms, phases, e2e_ms, clocks, t_wall = time_prefill(wl, steps, warmup, dist)
    ms, e2e_ms = dist.max(ms), dist.max(e2e_ms)
    f1, f2 = wl.flops()
    tflops = (f1 + f2) * dist.world * steps / (ms * 1e-3) / 1e12
    med = [statistics.median([p[j] for p in phases]) for j in range(4)]
    peak = peaks["bf16_tflops"]
    g1 = f1 / (med[1] * 1e-3) / 1e12
    g2 = f2 / (med[2] * 1e-3) / 1e12
    # GEMM1's algorithmic bytes: the w13 packed bytes and scales of the touched
    # experts, the routed token rows, h written; DRAM traffic from the
    # recorded ratio while the prefill sources hash the same
    s = wl.shape
    b1 = wl.D * w13_bytes(s.K, s.I) + wl.routes * s.K * 2 + wl.routes * s.I * 2
    rec = recorded_traffic("prefill")
    traffic1 = int(rec["gemm1_dram_over_alg"] * b1) if rec is not None else None
    out = {
        "metric": METRIC, "value": round(tflops, 1), "unit": "TFLOP/s",
        "n_gpus": dist.world, "steps": steps, "warmup": warmup,
        "ms_per_step": round(ms / steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": wl.config(),
        "phase_ms": {"route_gather": round(med[0], 4), "gemm1": round(med[1], 4),
                     "gemm2": round(med[2], 4), "combine": round(med[3], 4)},
        "gemm_tflops": {"gemm1": round(g1, 1), "gemm2": round(g2, 1)},
        "roofline": {"kernel": "gemm_kernel<1> (w13 grouped GEMM + SwiGLU)", "bound": "tensor",
                     "achieved": round(g1, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(g1 / peak, 3), "peak_kind": peak_kind + " bf16 burst",
                     "traffic": traffic1,
                     "traffic_source": "profiles/prefill_traffic.json" if traffic1 else None,
                     "alg_bytes_per_launch": int(b1), "alg_flops_per_launch": f1,
                     "avg_launch_us": round(med[1] * 1000, 1)},
        "e2e": {"value": round((f1 + f2) * dist.world * steps / (e2e_ms * 1e-3) / 1e12, 1),
                "unit": "TFLOP/s", "h2d_bytes_per_step": wl.e2e_bytes()[0],
                "d2h_bytes_per_step": wl.e2e_bytes()[1]},
        "gpu_launches": 5 * steps,
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if cpu and dist.rank == 0:
        out["cpu_baseline"] = prefill_cpu_sample(wl)
    del wl
    torch.cuda.empty_cache()
    return out


CHAIN = 8          # calls (distinct layers) per timed chain


def time_chain(fwd, calls, stream, reps: int = 20, warmup: int = 3, cold_reps: int = 3):
    """The pages' timing protocol ("MXFP4 MoE decode kernels", Measured
    results: a chain of 8 calls in a graph, median of replays): the CHAIN
    calls, each on its own layer's weights so that no call finds its experts
    in L2 from the call before, are captured back to back in one CUDA graph;
    each replay is timed with CUDA events on the replay stream and the median
    replay time / CHAIN is the time per call. The cold cross-check times a
    graph of [1 GiB L2 scrub, one call] against a graph of the scrub alone;
    the difference is one call that starts with nothing in L2.
    calls: list of (args, kwargs) for fwd. Returns (us per call, cold us)."""
    with torch.cuda.stream(stream):
        for a, k in calls:
            fwd(*a, **k)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for a, k in calls:
            fwd(*a, **k)
    times = []
    with torch.cuda.stream(stream):
        for r in range(warmup + reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            stream.synchronize()
            if r >= warmup:
                times.append(e0.elapsed_time(e1) / len(calls))
    scrub = torch.empty(1 << 30, dtype=torch.uint8, device=calls[0][0][0].device)
    gs, gc = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(gs, stream=stream):
        scrub.fill_(1)
    a, k = calls[0]
    with torch.cuda.graph(gc, stream=stream):
        scrub.fill_(2)
        fwd(*a, **k)
    ts, tc = [], []
    with torch.cuda.stream(stream):
        for r in range(1 + cold_reps):
            for gr, lst in ((gs, ts), (gc, tc)):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                gr.replay()
                e1.record(stream)
                stream.synchronize()
                if r >= 1:
                    lst.append(e0.elapsed_time(e1))
    del g, gs, gc, scrub
    return statistics.median(times) * 1000, (statistics.median(tc) - statistics.median(ts)) * 1000


def per_call_figures(us: float, alg_bytes: float, hbm_gbs: float):
    gbs = alg_bytes / (us * 1e-6) / 1e9
    return {"us": round(us, 2), "alg_bytes": int(alg_bytes), "gbs": round(gbs, 1),
            "frac_of_8tbs": round(gbs / 8000.0, 3), "frac_of_measured": round(gbs / hbm_gbs, 3)}


def measure_configs(dev, hbm_gbs: float, reps: int = 10):
    """The other decode workload shapes (the 32-expert single layer, the
    6144 x 2048 256-expert layer at T = 1, 8, 32 and the wide-K skewed layer
    at T = 1 .. 32) and the gpt-oss form of the 2880 x 2880 128-expert layer
    (interleaved gate/up rows, biases, SwiGLU-OAI): microseconds per call and
    GB/s of the touched experts' packed bytes, from chains of 8 calls on 8
    distinct layers (time_chain)."""
    from mxfp4_mixture_experts_gb300 import moe
    out = {}
    stream = torch.cuda.Stream()
    for name in ("single32", "glm256", "widek256", "gptoss128_oai"):
        oai = name.endswith("_oai")
        sh = synth.SHAPES[name[:-4] if oai else name]
        Ts = (1, 4, 16, 32) if name in ("single32", "gptoss128_oai") else sh.tokens
        layers = [synth.draw_weights_cuda(sh, seed=0, layer=l, device=dev) for l in range(CHAIN)]
        biases = ([tuple(b.to(dev) for b in synth.draw_biases(sh, seed=0, layer=l))
                   for l in range(CHAIN)] if oai else None)
        res = {}
        for T in Ts:
            ws = moe.new_workspace(T, sh.K, sh.I, sh.E, sh.topk, dev)
            calls, D = [], []
            for l, (w13, s13, w2, s2) in enumerate(layers):
                rng = np.random.Generator(np.random.PCG64(1000 * T + l))
                hidden, _, ids, w = synth.draw_activations(sh, T, rng)
                x, ids, w = hidden.to(dev), ids.to(dev), w.to(dev)
                y = torch.empty(T, sh.K, dtype=torch.bfloat16, device=dev)
                if oai:   # the gpt-oss form: the same bytes, interleaved rows, biases
                    b13, b2 = biases[l]
                    calls.append(((x, ids, w, w13, s13, b13, w2, s2, b2), dict(out=y, workspace=ws)))
                else:
                    calls.append(((x, ids, w, w13, s13, w2, s2), dict(out=y, workspace=ws)))
                D.append(touched_experts(ids, sh.E))
            us, cold = time_chain(moe.forward_oai if oai else moe.forward, calls, stream, reps=reps)
            alg = statistics.mean(D) * expert_bytes(sh.K, sh.I) + 4 * T * sh.K
            res[str(T)] = dict(per_call_figures(us, alg, hbm_gbs), touched=D,
                               cold_us=round(cold, 2))
            del calls, ws
        out[name] = {"K": sh.K, "I": sh.I, "E": sh.E, "topk": sh.topk, "per_T": res}
        if oai:
            out[name]["form"] = "gpt-oss: interleaved gate/up rows, f32 biases, SwiGLU-OAI"
        del layers, biases
        torch.cuda.empty_cache()
    return out


def measure_router(dev, reps: int = 20):
    """The router step (logits -> top-k ids and weights) at the gpt-oss decode
    size (T = 32, E = 128, top-4 softmax) and the prefill chunk (T = 8192,
    E = 256, top-8 sigmoid): microseconds per call from CUDA-graph replays of
    single calls with events around each replay."""
    from mxfp4_mixture_experts_gb300 import moe
    stream = torch.cuda.Stream()
    out = {}
    for name, T, E, k, scoring in (("gptoss128_t32", 32, 128, 4, "softmax_topk"),
                                   ("prefill256_t8192", 8192, 256, 8, "sigmoid_renorm")):
        g = torch.Generator(device=dev).manual_seed(T + E)
        logits = torch.randn(T, E, device=dev, generator=g)
        ids = torch.empty(T, k, dtype=torch.int32, device=dev)
        w = torch.empty(T, k, dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            moe.router(logits, k, scoring, topk_ids=ids, topk_weights=w)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            moe.router(logits, k, scoring, topk_ids=ids, topk_weights=w)
        times = []
        with torch.cuda.stream(stream):
            for r in range(reps + 3):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                stream.synchronize()
                if r >= 3:
                    times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        out[name] = {"T": T, "E": E, "topk": k, "scoring": scoring, "us": round(ms * 1000, 2),
                     "logit_bytes": 4 * T * E}
    return out


def measure_encode(dev, hbm_gbs: float, reps: int = 10):
    """The MXFP4 encoder on the w13 rows of 16 gpt-oss-120b experts (bf16
    [16 x 5760, 2880], N(0, 0.02), 531 MB in; larger than L2): microseconds
    per call from CUDA-graph replays with events around each replay, and GB/s
    of its algorithmic bytes (2 + 17/32 per value: bf16 in, codes and scales
    out) against the measured copy bandwidth."""
    from mxfp4_mixture_experts_gb300 import moe
    stream = torch.cuda.Stream()
    rows, cols = 16 * 5760, 2880
    g = torch.Generator(device=dev).manual_seed(64)
    x = (0.02 * torch.randn(rows, cols, device=dev, generator=g)).to(torch.bfloat16)
    out = {"rows": rows, "cols": cols}
    for rule in ("ocp", "quark"):
        with torch.cuda.stream(stream):
            moe.encode(x, rule)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            moe.encode(x, rule)
        times = []
        with torch.cuda.stream(stream):
            for r in range(reps + 3):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                stream.synchronize()
                if r >= 3:
                    times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        alg = rows * cols * (2 + 17 / 32)
        out[rule] = {"us": round(ms * 1000, 1), "alg_bytes": int(alg),
                     "gbs": round(alg / (ms * 1e-3) / 1e9, 1),
                     "frac_of_measured": round(alg / (ms * 1e-3) / 1e9 / hbm_gbs, 3)}
        del graph
    del x
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
def time_graph_loop(wl, steps: int, warmup: int, dist: Dist):
    """Headline timing, the pages' protocol ("MXFP4 MoE decode kernels",
    Measured results: a chain of 8 calls in a graph): two steps -- the 8
    calls on the 8 distinct layers, T = 1, 4, 16, 32 twice -- are captured in
    one CUDA graph and replayed; an odd step count ends with a graph of one
    step. CUDA events on the replay stream bracket all `steps` steps."""
    stream = torch.cuda.Stream()
    per_graph = wl.layers // wl.calls_per_step          # 2 steps: every layer once
    with torch.cuda.stream(stream):                      # eager warm-up of every layer first
        for gi in range(per_graph):
            for ly in wl.step_layers(gi):
                wl.call(ly)
    stream.synchronize()
    g_chain, g_one = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_chain, stream=stream):
        for gi in range(per_graph):
            for ly in wl.step_layers(gi):
                wl.call(ly)
    with torch.cuda.graph(g_one, stream=stream):
        for ly in wl.step_layers(0):
            wl.call(ly)
    with torch.cuda.stream(stream):
        for s in range(warmup):
            g_chain.replay()
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
        for s in range(steps // per_graph):
            g_chain.replay()
        for s in range(steps % per_graph):
            g_one.replay()
        e1.record(stream)
    stream.synchronize()
    t_wall = time.perf_counter() - t_wall
    torch.cuda.synchronize()
    dist.barrier()
    ck = clocks.stop()
    return e0.elapsed_time(e1), ck, t_wall


def time_per_T(wl, reps: int):
    """Per-call time at each T of the headline workload: chains of CHAIN calls
    at one T on the workload's 8 distinct layers (time_chain), with the
    touched experts' algorithmic bytes of each call."""
    stream = torch.cuda.Stream()
    s = wl.shape
    out = {}
    for T in wl.tokens:
        ws = wl.moe.new_workspace(T, s.K, s.I, s.E, s.topk, wl.dev)
        calls, alg = [], []
        for l, ly in enumerate(wl.L[:CHAIN]):
            rng = np.random.Generator(np.random.PCG64(1000 * T + l))
            hidden, _, ids, w = synth.draw_activations(s, T, rng)
            x, ids, w = hidden.to(wl.dev), ids.to(wl.dev), w.to(wl.dev)
            y = torch.empty(T, s.K, dtype=torch.bfloat16, device=wl.dev)
            calls.append(((x, ids, w, ly["w13"], ly["s13"], ly["w2"], ly["s2"]),
                          dict(out=y, workspace=ws)))
            alg.append(touched_experts(ids, s.E) * expert_bytes(s.K, s.I) + 4 * T * s.K)
        us, cold = time_chain(wl.moe.forward, calls, stream, reps=reps)
        out[T] = (us, statistics.mean(alg), cold)
        del calls, ws
    return out


# Sources that make up each kernel: a profile summary under profiles/ records
# their hash next to the DRAM traffic ncu measured, and the bench reports that
# traffic only while the hash still matches (a changed kernel reports null).
KERNEL_SOURCES = {
    "decode": ["decode.cu", "decode_common.cuh", "common.cuh", "route.cuh", "kernels.h"],
    "prefill": ["prefill.cu", "prefill.h", "common.cuh", "route.cuh"],
}


def kernel_hash(kind: str) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mxfp4_mixture_experts_gb300", "csrc")
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kind: str):
    """The DRAM-traffic record of profiles/<kind>_traffic.json (written with
    the ncu capture it summarises), if its kernel hash is the current one,
    else None."""
    path = os.path.join(ROOT, "profiles", f"{kind}_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    return rec if rec.get("kernel_hash") == kernel_hash(kind) else None


def time_e2e(wl, steps: int, warmup: int):
    """End to end through the C ABI from pinned host buffers: every step copies
    its inputs up (one copy), runs its calls and copies its outputs down (one
    copy), all inside the timed region."""
    stream = torch.cuda.Stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    h2d = d2h = 0
    with torch.cuda.stream(stream):
        for s in range(warmup):
            wl.step_e2e(s, stream)
        stream.synchronize()
        e0.record(stream)
        for s in range(steps):
            a, b = wl.step_e2e(s, stream)
            h2d += a
            d2h += b
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1), h2d // steps, d2h // steps


def _oracle_inputs(ly, E):
    """Host copies of one bench layer's call for the oracle: only the experts
    the call touches, relabelled 0..n-1 (the oracle is pinned invariant under
    expert relabelling)."""
    ids = ly["ids"].cpu().numpy().astype(np.int64)
    used = np.unique(ids[(ids >= 0) & (ids < E)])
    idx = torch.as_tensor(used, device=ly["w13"].device)
    host = [t.index_select(0, idx).cpu().numpy() for t in (ly["w13"], ly["s13"], ly["w2"], ly["s2"])]
    remap = np.full(E, -1)
    remap[used] = np.arange(len(used))
    hb = ly["hidden"].cpu().view(torch.int16).numpy().view(np.uint16)
    return (hb, remap[ids], ly["w"].cpu().numpy(), *host)


def _host_cores():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        return os.cpu_count()


def cpu_oracle_sample(wl):
    """The oracle as it stands, timed on this host on one call at each T of
    the workload's mix (the first layer of each T; value = the mean over the
    T, as the headline's). The oracle rows of those calls also give the
    parity figures of the GPU's outputs of the same calls: rel_l2 against the
    bf16-intermediate oracle (the pages' reference) and the unrounded one,
    and the largest absolute error, over every row."""
    from oracle import mxfp4_moe_oracle as O
    times, parity = {}, {}
    for T in wl.tokens:
        ly = next(l for l in wl.L if l["T"] == T)
        args = _oracle_inputs(ly, wl.shape.E)
        t0 = time.perf_counter()
        ya = O.forward(*args, intermediate="bf16")
        times[T] = time.perf_counter() - t0
        yb = O.forward(*args, intermediate="fp32")
        got = ly["out"].float().cpu().numpy().astype(np.float64)
        parity[str(T)] = {"rows": int(T),
                          "rel_l2_bf16_intermediate": float(np.linalg.norm(got - ya) / np.linalg.norm(ya)),
                          "rel_l2_fp32_intermediate": float(np.linalg.norm(got - yb) / np.linalg.norm(yb)),
                          "max_abs_err": float(np.abs(got - ya).max()),
                          "max_abs_ref": float(np.abs(ya).max())}
    us = statistics.mean(times.values()) * 1e6
    cpu = {"value": round(us, 1), "unit": "us_per_moe_call", "cores": _host_cores(),
           "kind": "oracle",
           "sample": f"one oracle call at each T={list(times)} of the workload (float64 numpy, "
                     f"{sum(times.values()):.1f} s of CPU work); value = mean over the T"}
    return cpu, parity


# ---------------------------------------------------------------------------
def run_ours(args, dist: Dist):
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks()
    if args.workload == "prefill":
        return run_prefill(args, dist, args.steps, args.warmup, not args.no_cpu_baseline)
    wl = DecodeWorkload(dev)
    elapsed_ms, clocks, t_wall = time_graph_loop(wl, args.steps, args.warmup, dist)
    elapsed_ms = dist.max(elapsed_ms)
    calls = args.steps * wl.calls_per_step
    value = aggregate_us_per_call(elapsed_ms, calls, dist.world)
    per_T_raw = time_per_T(wl, reps=max(args.steps, 10))
    e2e_ms, h2d, d2h = time_e2e(wl, args.steps, args.warmup)
    e2e_ms = dist.max(e2e_ms)
    hbm = peaks["hbm_gbs"]
    per_T = {str(T): dict(per_call_figures(us, b, hbm), cold_us=round(cold, 2))
             for T, (us, b, cold) in per_T_raw.items()}
    # roofline: the T = 32 calls (the bandwidth-bound end of the decode range);
    # a launch's duration = the chain's time per call (kernel + the gap to the
    # next launch of the chain)
    big = max(wl.tokens)
    us32, b32, _ = per_T_raw[big]
    achieved = b32 / (us32 * 1e-6) / 1e9
    rec = recorded_traffic("decode")
    traffic = None
    if rec is not None:   # ncu DRAM bytes / algorithmic bytes of a launch at this T, scaled
        traffic = int(rec["dram_over_alg"][str(big)] * b32)
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "us_per_call",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": wl.config(),
        "per_T": per_T,
        "roofline": {"kernel": f"decode_kernel (w13 + SwiGLU, w2, combine: one launch per call), "
                               f"T = {big} calls",
                     "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 3), "peak_kind": peak_kind,
                     "traffic": traffic,
                     "traffic_source": "profiles/decode_traffic.json" if traffic is not None else None,
                     "alg_bytes_per_launch": int(b32),
                     "avg_launch_us": round(us32, 2),
                     "timing": f"chains of {CHAIN} calls on {CHAIN} distinct layers at T = {big}, "
                               "median replay / calls"},
        "e2e": {"value": round(aggregate_us_per_call(e2e_ms, calls, dist.world), 3),
                "unit": "us_per_call", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": calls,
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if dist.rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"], out["parity"] = cpu_oracle_sample(wl)
    del wl
    torch.cuda.empty_cache()
    if not args.no_configs:
        out["configs"] = measure_configs(dev, hbm)
        out["router"] = measure_router(dev)
        out["encode"] = measure_encode(dev, hbm)
    if not args.no_prefill:
        pf = run_prefill(args, dist, 10, 3, False)
        out["prefill"] = {k: pf[k] for k in ("value", "unit", "ms_per_step", "config",
                                             "phase_ms", "gemm_tflops", "roofline", "e2e",
                                             "gpu_launches", "clocks")}
    return out


def run_reference(args, dist: Dist):
    """The CPU oracle as the reference arm, on the same workload: each step is
    one call at the next T of the mix 1, 4, 16, 32 (the routing of the GPU
    arm's layer of that T, random packed weights for the experts it touches);
    value = the mean over the T of the mean time per call, as the headline's."""
    if dist.rank != 0:
        return None
    from oracle import mxfp4_moe_oracle as O
    s = synth.SHAPES["gptoss128"]
    tokens = DecodeWorkload.tokens
    calls = {}
    for l, T in enumerate(tokens):
        hidden, _, ids, w = synth.draw_activations(s, T, np.random.Generator(np.random.PCG64(l)))
        ids = ids.numpy().astype(np.int64)
        used = np.unique(ids)
        remap = np.full(s.E, -1)
        remap[used] = np.arange(len(used))
        g = np.random.Generator(np.random.PCG64(100 + l))
        n = len(used)
        w13 = g.integers(0, 256, (n, 2 * s.I, s.K // 2), dtype=np.uint8)
        s13 = g.integers(118, 125, (n, 2 * s.I, s.K // 32), dtype=np.uint8)
        w2 = g.integers(0, 256, (n, s.K, s.I // 2), dtype=np.uint8)
        s2 = g.integers(118, 125, (n, s.K, s.I // 32), dtype=np.uint8)
        hb = hidden.view(torch.int16).numpy().view(np.uint16)
        calls[T] = (hb, remap[ids], w.numpy(), w13, s13, w2, s2)
    for i in range(args.warmup):
        O.forward(*calls[tokens[i % len(tokens)]])
    per_T = {T: [] for T in tokens}
    t_all = time.perf_counter()
    for i in range(args.steps):
        T = tokens[i % len(tokens)]
        t0 = time.perf_counter()
        O.forward(*calls[T])
        per_T[T].append(time.perf_counter() - t0)
    el = time.perf_counter() - t_all
    us = statistics.mean(statistics.mean(v) for v in per_T.values() if v) * 1e6
    cores = _host_cores()
    return {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us_per_call",
            "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": decode_config(s, tokens, DecodeWorkload.layers),
            "per_T_us": {str(T): round(statistics.mean(v) * 1e6, 1) for T, v in per_T.items() if v},
            "cpu_baseline": {"value": round(us, 1), "unit": "us_per_call", "cores": cores,
                             "kind": "oracle",
                             "sample": "each step: one call at the next T of the mix 1, 4, 16, "
                                       "32 (float64 numpy oracle, touched experts only); value "
                                       "= mean over the T of the mean time per call"},
            "e2e": {"value": round(us, 1), "unit": "us_per_call", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_profile_case(args):
    """`--profile-case NAME:T`: warm-up + steps forward calls of one layer of a
    workload, no timing; the command profilers (ncu) run."""
    from mxfp4_mixture_experts_gb300 import moe
    name, T = args.profile_case.split(":")
    T = int(T)
    if name in synth.SHAPES:
        shape = synth.SHAPES[name]
    else:   # "K,I,E,topk": a smaller layer of the same kind, for counter captures
        K, I, E, k = (int(v) for v in name.split(","))
        shape = synth.custom_shape(K, I, E, k, scoring="sigmoid_renorm")
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
    ap.add_argument("--no-configs", action="store_true",
                    help="leave the other decode workload shapes out of the default line")
    ap.add_argument("--no-prefill", action="store_true",
                    help="leave the shorter prefill measurement out of the default line")
    ap.add_argument("--profile-case", default=None,
                    help="NAME:T or K,I,E,topk:T -- run warmup+steps calls of one layer, "
                         "untimed (for ncu)")
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
