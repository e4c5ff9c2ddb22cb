#!/usr/bin/env python
"""Denoise steps/s of one uniform-state denoising step over a 256-token canvas
(V = 262144, d = 2816, prefix 8192, 16 q / 8 kv heads) on one GB300, with the
roofline of its dominant kernel.

One timed "step" is one pass of the whole hot path over the canvas: embedding +
RMSNorm, q/k/v + RoPE, attention over prefix + canvas, output projection, LM
head with softmax statistics, entropy-bounded accept / renoise with the stop
test, p0 . E with Gumbel-max sampling, and the self-conditioning FFW.  The
temperature follows the 48-step schedule (step s uses tau_{s mod 48}); the
canvas state carries over from step to step as in the real loop.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(no data-path collective); the value is the steps of all ranks divided by the
slowest rank's time.  --impl reference times the CPU oracle on the host cores
instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from block_diffusion_text_gb300 import synth  # noqa: E402

METRIC = "denoise steps/s (C=256, V=262144)"
UNIT = "denoise steps/s"
DEFAULT_WORKLOAD = "loop_v262k_c256_p8k"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-loop", action="store_true")
    ap.add_argument("--no-variants", action="store_true")
    return ap.parse_args()


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend=backend)
    return world, rank, local


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), tc=float(p["bf16_tflops"]),
                    tc_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, tc=1900.0, tc_sustained=1700.0, src="fallback")


# ---------------------------------------------------------------- clocks --
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            uuid = str(device_index)
        self.cmd = ["nvidia-smi", f"--id={uuid}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "20"]
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def mark(self, t0, t1):
        """Host-clock bounds of the timed region; only samples inside it are reported."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        if self.window is not None:
            inside = [p for t, p in self.samples if self.window[0] <= t <= self.window[1] + 0.025]
        else:
            inside = [p for _, p in self.samples]
        n_all = len(self.samples)
        self.samples = inside
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "samples_total": n_all}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in self.samples if num(s[0]) is not None]
        mx = [num(s[1]) for s in self.samples if num(s[1]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for s in self.samples for n, v in zip(names, s[4:8]) if v.lower() == "active"})
        pw = [num(s[2]) for s in self.samples if num(s[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "sm_mhz_min": min(sm) if sm else None, "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(self.samples), "window": "timed region only"}


# ------------------------------------------------------- algorithmic work --
def stage_work(d: synth.Dims):
    """Algorithmic FLOPs and HBM bytes per step of each stage: what the method must compute and
    move (weights and E read once, the stage's own inputs and outputs), not what a kernel happens
    to store for itself (the exp(s - m) tiles, split partials, statistics).  Every stage of the
    step is listed, so their sum of roofline times is the step's roofline."""
    M, V, D = d.B * d.C, d.V, d.d
    nq, nkv = d.Hq * d.hd, d.Hkv * d.hd
    T = d.P + d.C
    bf = 2.0
    w = {}
    w["embed"] = (0.0, bf * M * D * 3 + 4.0 * M)                       # E rows, z, a
    w["qkv"] = (2.0 * M * D * (nq + 2 * nkv), bf * D * (nq + 2 * nkv) + bf * M * D + bf * M * (nq + 2 * nkv))
    w["attn"] = (4.0 * d.B * d.Hq * d.C * T * d.hd, bf * 2 * d.B * d.Hkv * T * d.hd + bf * 2 * M * nq)
    w["oproj"] = (2.0 * M * nq * D, bf * nq * D + bf * M * nq + bf * 2 * M * D)
    w["lmhead"] = (2.0 * M * V * D, bf * V * D + bf * M * D + 4.0 * M)  # E + h (+ alpha)
    w["selfcond"] = (2.0 * M * V * D, bf * V * D + bf * M * D)          # E + u
    w["ffw"] = (4.0 * M * D * d.F, bf * 2 * D * d.F + bf * 2 * M * D + bf * M * d.F)
    w["sampler"] = (0.0, 4.0 * M * 4)                                   # entropy, argmax, tokens, accept
    return w


def kernel_work(d: synth.Dims):
    """(FLOPs, algorithmic bytes) per launch of the timed kernel slots."""
    w = stage_work(d)
    return {"lmhead": w["lmhead"], "selfcond": w["selfcond"], "attn": w["attn"]}


def fp8_lmhead_work(d: synth.Dims):
    """The FP8 LM head: the same FLOPs, E4M3 codes of E and h plus their per-row scales."""
    M, V, D = d.B * d.C, d.V, d.d
    return (2.0 * M * V * D, 1.0 * V * D + 4.0 * V + 1.0 * M * D + 4.0 * M + 4.0 * M)


def step_roofline(d: synth.Dims, peaks):
    """T_roof = sum over stages of max(FLOPs / tensor peak, bytes / HBM peak), with E read once per
    step for the two vocabulary products together (their bytes are counted once).  Sustained bf16
    tensor peak: the step runs back to back."""
    w = stage_work(d)
    w = dict(w)
    fl = w["lmhead"][0] + w["selfcond"][0]
    w["vocab"] = (fl, 2.0 * d.V * d.d + 2.0 * 2 * d.M * d.d + 4.0 * d.M)
    del w["lmhead"], w["selfcond"]
    tc, bw = peaks["tc_sustained"] * 1e12, peaks["hbm"] * 1e9
    per = {k: max(f / tc, b / bw) for k, (f, b) in w.items()}
    return sum(per.values()), per


def _traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it still matches the source."""
    try:
        import hashlib
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            t = json.load(f)
        e = t.get(kernel)
        if not e:
            return None
        srcs = {e["source"]: e["source_sha256"], **e.get("also", {})}
        for rel, sha in srcs.items():
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != sha:
                    return None
        return float(e["bytes_per_launch_full_size"])
    except Exception:
        return None


# ------------------------------------------------------------ CPU oracle --
def oracle_full_step(dims, w_np, x, z, a, nthreads, tau=0.8, step=0, seed=0):
    """Seconds of one full oracle step (every stage, every row) on `nthreads` host threads."""
    import oracle
    t0 = time.perf_counter()
    oracle.denoise_step(dims, w_np, x, z, a, tau=tau, b=0.1, seed=seed, step=step,
                        want=("H", "tokens_out", "z_out", "n_acc"), nthreads=nthreads)
    return time.perf_counter() - t0


def _oracle_inputs_from(w, x, z, a):
    wn = synth.to_numpy_f32(w)
    return wn, x.cpu().numpy(), z.float().cpu().numpy(), a.cpu().numpy()


def run_reference(args, world, rank):
    """The oracle as it stands, on the host cores.  Each timed step is one full oracle step (every
    stage for every row of the canvas); the warm-up steps run the oracle's front stages (a..h) only,
    since the oracle has no state that a full warm-up step would prepare."""
    if rank != 0:
        return
    import oracle
    dims, seed = synth.workload(args.workload)
    nthreads = os.cpu_count() or 1
    w = synth.make_weights(dims, seed, device="cpu")
    x, z, a = synth.make_canvas(dims, seed, device="cpu")
    wn, xn, zn, an = _oracle_inputs_from(w, x, z, a)
    del w
    taus = oracle.tau_schedule(48, 0.8, 0.4)
    for s in range(args.warmup):
        oracle.denoise_step(dims, wn, xn, zn, an, tau=taus[s % 48], b=0.1, seed=seed, step=s % 48, rows=[],
                            want=("h",), nthreads=nthreads)
    times = []
    t_all = time.perf_counter()
    for s in range(args.steps):
        times.append(oracle_full_step(dims, wn, xn, zn, an, nthreads, tau=taus[s % 48], step=s % 48, seed=seed))
    t_all = time.perf_counter() - t_all
    value = args.steps / t_all
    sample = (f"each timed step is one full oracle step: all {dims.M} rows through every stage "
              f"(front, LM head, sampler, p0.E, FFW); warm-up steps run the front stages only")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_all / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": _config(dims, args.workload),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                             "sample": sample, "step_s": [round(t, 3) for t in times]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _config(dims, name):
    return {"workload": name, "V": dims.V, "d": dims.d, "C": dims.C, "B": dims.B, "P": dims.P,
            "Hq": dims.Hq, "Hkv": dims.Hkv, "hd": dims.hd, "F": dims.F, "tau": "0.8->0.4 over 48 steps",
            "b": 0.1, "l2": f"inputs larger than L2 (E alone is {2 * dims.V * dims.d / 1e9:.2f} GB)"}


# ------------------------------------------------------------- our path ---
def run_ours(args, world, rank, local):
    from block_diffusion_text_gb300 import dg
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dims, seed = synth.workload(args.workload)
    w = synth.make_weights(dims, seed, device=dev)
    x, z, a = synth.make_canvas(dims, seed, device=dev)
    x0, z0 = x.clone(), z.clone()
    model = dg.Model(dims, w)
    canvas = dg.Canvas(x, z, a)
    taus = dg.tau_schedule(48)
    outbuf = None
    slots = dg.PROF_SLOTS
    timed_slots = tuple(k for k in slots if k != "moe" or dims.n_exp > 0)

    def step(s, events=None):
        nonlocal outbuf
        outbuf = dg.denoise_step(model, canvas, tau=taus[s % 48], b=0.1, seed=seed, step=s % 48,
                                 out=outbuf, events=events)

    stream = torch.cuda.current_stream()
    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    if model.status() != 0:
        raise RuntimeError("device status word set during warm-up")

    # per-kernel events of the timed steps (recorded once so that the handles exist)
    ev = []
    for _ in range(args.steps):
        row = [None] * (2 * len(slots))
        for name in timed_slots:
            k = slots.index(name)
            for e in (0, 1):
                t = torch.cuda.Event(enable_timing=True)
                t.record(stream)
                row[2 * k + e] = t
        ev.append(row)
    torch.cuda.synchronize()

    # Eager reference: the same steps launched one by one from the host.
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n_eager = min(args.steps, 20)
    e0.record(stream)
    for s in range(n_eager):
        step(args.warmup + s)
    e1.record(stream)
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / n_eager

    # The K timed steps captured into one CUDA graph (no host work inside the
    # timed region), and the same steps with an event before and after every
    # kernel in a second graph: event-record nodes cost ~2 us each, so the
    # per-kernel durations come from that instrumented replay, run right after.
    def capture(events, keep=False):
        try:
            g = torch.cuda.CUDAGraph(keep_graph=True) if keep else torch.cuda.CUDAGraph()
        except TypeError:
            g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap):
            for s in range(args.steps):
                step(args.warmup + n_eager + s, events=ev[s] if events else None)
        torch.cuda.synchronize()
        return g
    graph = capture(False, keep=True)
    graph_kernels = _kernel_nodes(graph)
    if hasattr(graph, "instantiate"):
        graph.instantiate()
    graph_ev = capture(True)

    clocks = ClockSampler(local)
    _barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    h0 = time.time()
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    clocks.mark(h0, time.time())
    _barrier(world)
    clk = clocks.stop()
    elapsed_ms = t0.elapsed_time(t1)
    graph_ev.replay()
    torch.cuda.synchronize()
    if model.status() != 0:
        raise RuntimeError("device status word set during the timed steps")
    per_kernel = {}
    for name in timed_slots:
        k = slots.index(name)
        per_kernel[name] = statistics.mean(ev[s][2 * k].elapsed_time(ev[s][2 * k + 1]) for s in range(args.steps))
    max_ms = _max_over_ranks(elapsed_ms, world)
    value = world * args.steps / (max_ms / 1e3)

    # end to end through the public API with host buffers: the step's inputs
    # (tokens, z, alpha) go up from pinned host memory and its results (tokens,
    # z, entropy, accept mask) come back, each as one contiguous copy; two host
    # buffers alternate, so a step's results are the next step's inputs.
    e2e = None
    if not args.no_e2e:
        io_dev, io_host, views = _e2e_buffers(dims, dev)
        tok_d, z_d, a_d, ent_d, acc_d = views(io_dev)
        tok_d.copy_(x0)
        z_d.copy_(z0)
        a_d.copy_(a)
        io_host[0].copy_(io_dev)
        io_host[1].copy_(io_dev)
        e_canvas = dg.Canvas(tok_d, z_d, a_d)
        e_out = dict(entropy=ent_d, accept=acc_d, argmax=torch.empty_like(tok_d),
                     n_acc=torch.empty(dims.B, dtype=torch.int32, device=dev),
                     mean_H=torch.empty(dims.B, dtype=torch.float32, device=dev),
                     stop=torch.empty(dims.B, dtype=torch.int32, device=dev))
        n_in = _e2e_input_bytes(dims)
        h2d, d2h = n_in, io_dev.numel()
        ksteps = min(args.steps, 50)

        def e2e_body(s):
            src, dst = io_host[s % 2], io_host[(s + 1) % 2]
            io_dev[:n_in].copy_(src[:n_in], non_blocking=True)
            dg.denoise_step(model, e_canvas, tau=taus[s % 48], b=0.1, seed=seed, step=s % 48, out=e_out)
            dst.copy_(io_dev, non_blocking=True)

        def e2e_eager(s):
            e2e_body(s)
            torch.cuda.current_stream().synchronize()

        def timed(fn):
            _barrier(world)
            torch.cuda.synchronize()
            tt = time.perf_counter()
            for s in range(ksteps):
                fn(s)
            torch.cuda.synchronize()
            return _max_over_ranks(time.perf_counter() - tt, world)

        for s in range(3):
            e2e_eager(s)
        eager_s = timed(e2e_eager)
        # The same per-step work replayed from CUDA graphs, one per step of the
        # schedule (the copies and the step captured together; the host still
        # waits for every step's results before the next one starts).
        graphs = []
        cap = torch.cuda.Stream()
        for s in range(48):
            g = torch.cuda.CUDAGraph()
            cap.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(g, stream=cap):
                e2e_body(s)
            graphs.append(g)
        torch.cuda.synchronize()

        def e2e_graph(s):
            graphs[s % 48].replay()
            torch.cuda.current_stream().synchronize()

        for s in range(3):
            e2e_graph(s)
        graph_s = timed(e2e_graph)
        e2e = {"value": world * ksteps / graph_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": ksteps,
               "mode": "per step: pinned host -> device copy of tokens, z, alpha; the step; device -> host "
                       "copy of tokens, z, alpha, entropy, accept; host waits for the results; replayed from "
                       "a CUDA graph of those three per schedule step",
               "host_launched_value": world * ksteps / eager_s}

    # rooflines: per kernel against both bounds (algorithmic work), and the whole step
    peaks = _peaks()
    work = kernel_work(dims)
    rl = {}
    for name, (fl, by) in work.items():
        if name not in per_kernel:
            continue
        sec = per_kernel[name] / 1e3
        t_tc = fl / (peaks["tc_sustained"] * 1e12)
        t_hbm = by / (peaks["hbm"] * 1e9)
        bound = "tensor" if t_tc >= t_hbm else "hbm"
        tc_frac = fl / sec / 1e12 / peaks["tc_sustained"]
        hbm_frac = by / sec / 1e9 / peaks["hbm"]
        if bound == "tensor":
            ach, peak, unit, frac = fl / sec / 1e12, peaks["tc_sustained"], "TFLOP/s", tc_frac
        else:
            ach, peak, unit, frac = by / sec / 1e9, peaks["hbm"], "GB/s", hbm_frac
        rl[name] = {"bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": frac,
                    "traffic": _traffic(name), "ms": per_kernel[name],
                    "tflops": fl / sec / 1e12, "gbs": by / sec / 1e9,
                    "tensor_frac": tc_frac, "hbm_frac": hbm_frac,
                    "algorithmic": {"flop": fl, "bytes": by},
                    "peak_note": ("of measured" if peaks["src"] == "measured" else "of fallback")
                    + (" sustained bf16" if bound == "tensor" else " HBM copy")}
    dominant = max(rl, key=lambda k: rl[k]["ms"])
    dom = rl[dominant]
    t_roof, t_stage = step_roofline(dims, peaks)
    step_s = max_ms / args.steps / 1e3
    step_rl = {"t_roof_ms": t_roof * 1e3, "steps_per_s_roof": 1.0 / t_roof, "frac": t_roof / step_s,
               "canvas_tokens_per_s_roof": dims.M / t_roof, "canvas_tokens_frac": t_roof / step_s,
               "stage_roof_ms": {k: round(v * 1e3, 4) for k, v in t_stage.items()},
               "note": "sum over stages of max(FLOPs / sustained bf16 peak, algorithmic bytes / HBM peak); "
                       "E read once per step for both vocabulary products"}

    # Variants of the same step, each captured as K' steps in one CUDA graph: the FP8 LM head
    # (E4M3 E and h on the kind::f8f6f4 tensor cores) and masked confidence decoding (the
    # second sampler, [MASK] = the last token id)
    variants = None
    if rank == 0 and not args.no_variants:
        variants = {}
        kv = min(args.steps, 50)

        def time_graph(fn, n):
            cap = torch.cuda.Stream()
            cap.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                for s in range(n):
                    fn(s)
            torch.cuda.synchronize()
            g.replay()  # warm replay
            torch.cuda.synchronize()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            g.replay()
            a1.record(stream)
            torch.cuda.synchronize()
            return a0.elapsed_time(a1) / n

        m8 = dg.Model(dims, w, fp8_head=True)
        c8 = dg.Canvas(x0.clone(), z0.clone(), a)
        o8 = [None]
        lm_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(slots))] for _ in range(kv)]
        for row in lm_ev:  # recorded once so that the handles exist before the capture
            for e in row:
                e.record(stream)

        def step8(s, events=None):
            o8[0] = dg.denoise_step(m8, c8, tau=taus[s % 48], b=0.1, seed=seed, step=s % 48, out=o8[0],
                                    events=events)
        for s in range(3):
            step8(s)
        torch.cuda.synchronize()
        ms8 = time_graph(step8, kv)
        time_graph(lambda s: step8(s, events=lm_ev[s]), kv)
        k = slots.index("lmhead")
        lm8 = statistics.mean(lm_ev[s][2 * k].elapsed_time(lm_ev[s][2 * k + 1]) for s in range(kv))
        fl8, by8 = fp8_lmhead_work(dims)
        pk8 = 2.0 * peaks["tc_sustained"]
        variants["fp8_lm_head"] = {
            "value": 1e3 / ms8, "unit": UNIT, "ms_per_step": ms8, "steps": kv, "dtype": "e4m3 x e4m3 -> f32",
            "lmhead_ms": lm8, "lmhead_bf16_ms": per_kernel.get("lmhead"),
            "lmhead_roofline": {"bound": "tensor", "achieved": fl8 / (lm8 / 1e3) / 1e12, "peak": pk8,
                                "unit": "TFLOP/s", "frac": fl8 / (lm8 / 1e3) / 1e12 / pk8,
                                "hbm_gbs": by8 / (lm8 / 1e3) / 1e9, "algorithmic": {"flop": fl8, "bytes": by8},
                                "peak_note": "2 x measured sustained bf16 (the nominal fp8 / bf16 ratio)"},
            "note": "the lmhead slot includes the per-step E4M3 quantization of h"}
        if m8.status() != 0:
            raise RuntimeError("device status word set in the FP8 variant")
        del m8, c8, o8

        # the MoE FFN after the attention block (128 experts, top 8 + shared, Fe 768, 84 hot experts:
        # the pages' canvas-level activation), same workload otherwise
        dmoe = dataclasses.replace(dims, n_exp=128, top_k=8, Fe=768, moe_hot=84)
        wm = dict(w)
        wm.update({k: v for k, v in synth.make_weights(dmoe, seed + 1, device=dev).items()
                   if k in ("Wr", "We1", "We2")})
        mm = dg.Model(dmoe, wm)
        cmo = dg.Canvas(x0.clone(), z0.clone(), a)
        om = [None]
        dbg_run = dg.denoise_step(mm, cmo, tau=taus[0], b=0.1, seed=seed, step=0, debug=True)
        n_active = int(torch.unique(dbg_run["debug"]["moe_idx"]).numel()) + 1  # + the shared expert
        del dbg_run
        mo_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(slots))] for _ in range(kv)]
        for row in mo_ev:
            for e in row:
                e.record(stream)

        def stepmo(s, events=None):
            om[0] = dg.denoise_step(mm, cmo, tau=taus[s % 48], b=0.1, seed=seed, step=s % 48, out=om[0],
                                    events=events)
        for s in range(3):
            stepmo(s)
        torch.cuda.synchronize()
        msmo = time_graph(stepmo, kv)
        time_graph(lambda s: stepmo(s, events=mo_ev[s]), kv)
        k = slots.index("moe")
        moe_ms = statistics.mean(mo_ev[s][2 * k].elapsed_time(mo_ev[s][2 * k + 1]) for s in range(kv))
        wbytes = 2.0 * n_active * 2 * dmoe.Fe * dmoe.d + 2.0 * dmoe.n_exp * dmoe.d  # active experts + router
        mflop = 2.0 * dmoe.M * (dmoe.top_k + 1) * 2 * dmoe.Fe * dmoe.d
        variants["moe_ffn"] = {
            "value": 1e3 / msmo, "unit": UNIT, "ms_per_step": msmo, "steps": kv,
            "config": {"n_exp": 128, "top_k": 8, "shared": 1, "Fe": dmoe.Fe, "hot_experts": 84},
            "experts_active": n_active, "moe_ms": moe_ms,
            "moe_roofline": {"bound": "hbm", "achieved": wbytes / (moe_ms / 1e3) / 1e9, "peak": peaks["hbm"],
                             "unit": "GB/s", "frac": wbytes / (moe_ms / 1e3) / 1e9 / peaks["hbm"],
                             "algorithmic": {"bytes": wbytes, "flop": mflop},
                             "tflops": mflop / (moe_ms / 1e3) / 1e12,
                             "note": "bytes: the active experts' two matrices (each read once per step) and the "
                                     "router; the block's kernels: RMSNorm, router, plan, gather, two grouped "
                                     "GEMMs, combine"}}
        if mm.status() != 0:
            raise RuntimeError("device status word set in the MoE variant")
        del mm, cmo, om, wm

        mask_id = dims.V - 1
        cm = dg.Canvas(dg.canvas_init_masked(dims.B, dims.C, mask_id, device=dev), z0.clone(), a)
        om = [None]
        tok_m0 = cm.tokens.clone()

        def stepm(s):
            if s % 16 == 0:
                cm.tokens.copy_(tok_m0)  # a fresh all-[MASK] canvas every 16 steps
            om[0] = dg.denoise_step(model, cm, tau=1.0, b=0.0, seed=seed, step=s % 16, out=om[0],
                                    masked=(mask_id, 16))
        for s in range(3):
            stepm(s)
        torch.cuda.synchronize()
        msm = time_graph(stepm, 48)
        variants["masked_confidence"] = {
            "value": 1e3 / msm, "unit": UNIT, "ms_per_step": msm, "steps": 48,
            "note": "masked confidence decoding, 16 steps per canvas (reveal ceil(unresolved / steps left))"}
        if model.status() != 0:
            raise RuntimeError("device status word set in the masked variant")

    # the annealed loop itself (dg_denoise_canvas, up to 48 steps with adaptive stop) from the
    # benchmark's initial canvas, and the commit of its result
    loop = None
    if rank == 0 and not args.no_loop:
        lc = dg.Canvas(x0.clone(), z0.clone(), a)
        torch.cuda.synchronize()
        tl = time.perf_counter()
        res = dg.denoise_canvas(model, lc, seed=seed, N=48)
        torch.cuda.synchronize()
        tl = time.perf_counter() - tl
        acc = res["accepted"].cpu().numpy()
        taken = res["steps_taken"].cpu().tolist()
        per_step = [int(v) for v in acc[0] if v >= 0]
        loop = {"steps_taken": taken, "converged": res["converged"].cpu().tolist(),
                "accepted_per_step": per_step,
                "mean_accepted_per_step": float(sum(per_step) / max(len(per_step), 1)),
                "ms": tl * 1e3, "steps_per_s": sum(taken) / tl,
                "note": "one dg_denoise_canvas call, host clock (the loop reads its 4-byte stop count "
                        "every 4 steps)"}
        if model.status() != 0:
            raise RuntimeError("device status word set during the loop")
        # commit of the loop's x0 at position P (into rows P..P+C-1 of a cache with room for it)
        Kx = torch.zeros(dims.B, dims.Hkv, dims.P + dims.C, dims.hd, dtype=torch.bfloat16, device=dev)
        Vx = torch.zeros_like(Kx)
        xh = res["xhat0"]
        for _ in range(3):
            dg.commit_block(model, xh, cache=(Kx, Vx, dims.P))
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(20):
            dg.commit_block(model, xh, cache=(Kx, Vx, dims.P))
        c1.record(stream)
        torch.cuda.synchronize()
        loop["commit_ms"] = c0.elapsed_time(c1) / 20
        del Kx, Vx

    if graph_kernels is not None:
        gpu_launches, launch_src = graph_kernels, "kernel nodes of the timed CUDA graph"
    else:
        launches_per_step = len(dg.PROF_SLOTS) + (1 if _attn_splits(dims) > 1 else 0)
        gpu_launches, launch_src = launches_per_step * args.steps, "one per profiled stage (lower bound)"

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": _config(dims, args.workload),
            "canvas_tokens_per_s": value * dims.B * dims.C,
            "roofline": {"bound": dom["bound"], "achieved": dom["achieved"], "peak": dom["peak"],
                         "unit": dom["unit"], "frac": dom["frac"], "traffic": dom["traffic"],
                         "kernel": dominant, "peak_note": dom["peak_note"],
                         "tensor_frac": dom["tensor_frac"], "hbm_frac": dom["hbm_frac"]},
            "step_roofline": step_rl,
            "loop": loop,
            "variants": variants,
            "kernels": rl,
            "kernel_ms": {k: round(v, 5) for k, v in per_kernel.items()},
            "timing": "K steps captured in one CUDA graph, CUDA events around its replay; per-kernel "
                      "times from an event-instrumented replay of the same steps; "
                      f"eager host-launched step for comparison: {eager_ms:.4f} ms",
            "clocks": clk,
            "e2e": e2e,
            "gpu_launches": gpu_launches, "gpu_launches_source": launch_src}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            nthreads = os.cpu_count() or 1
            wn, xn, zn, an = _oracle_inputs_from(w, x0, z0, a)
            t = oracle_full_step(dims, wn, xn, zn, an, nthreads, seed=seed)
            line["cpu_baseline"] = {"value": 1.0 / t, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                                    "sample": f"one full oracle step: all {dims.M} rows through every stage",
                                    "step_s": round(t, 3)}
        except Exception as e:  # the baseline is reported, not required
            line["cpu_baseline"] = {"value": None, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                                    "sample": f"failed: {e!r}"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def _e2e_offsets(dims):
    """Byte offsets of tokens, z, alpha, entropy, accept in the e2e I/O block (256-byte aligned)."""
    M = dims.B * dims.C
    sizes = (4 * M, 2 * M * dims.d, 4 * M, 4 * M, M)
    offs, o = [], 0
    for n in sizes:
        offs.append(o)
        o = (o + n + 255) // 256 * 256
    return offs, sizes, o


def _e2e_input_bytes(dims):
    offs, sizes, _ = _e2e_offsets(dims)
    return offs[2] + sizes[2]  # tokens, z, alpha


def _e2e_buffers(dims, dev):
    offs, sizes, total = _e2e_offsets(dims)
    io_dev = torch.zeros(total, dtype=torch.uint8, device=dev)
    io_host = [torch.zeros(total, dtype=torch.uint8).pin_memory() for _ in range(2)]
    M = dims.B * dims.C

    def views(buf):
        v = lambda k, dt: buf[offs[k]:offs[k] + sizes[k]].view(dt)
        return (v(0, torch.int32).view(dims.B, dims.C), v(1, torch.bfloat16).view(dims.B, dims.C, dims.d),
                v(2, torch.float32).view(dims.B, dims.C), v(3, torch.float32).view(dims.B, dims.C),
                v(4, torch.uint8).view(dims.B, dims.C))
    return io_dev, io_host, views


def _kernel_nodes(graph):
    """Kernel nodes in a captured CUDA graph (driver API through ctypes), or None."""
    try:
        import ctypes
        cu = ctypes.CDLL("libcuda.so.1")
        h = ctypes.c_void_p(graph.raw_cuda_graph())
        n = ctypes.c_size_t(0)
        if cu.cuGraphGetNodes(h, None, ctypes.byref(n)) != 0:
            return None
        nodes = (ctypes.c_void_p * n.value)()
        if cu.cuGraphGetNodes(h, nodes, ctypes.byref(n)) != 0:
            return None
        kind = ctypes.c_int(-1)
        count = 0
        for i in range(n.value):
            if cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(kind)) != 0:
                return None
            count += kind.value == 0  # CU_GRAPH_NODE_TYPE_KERNEL
        return count
    except Exception:
        return None


def _attn_splits(dims):
    """Key splits of the attention launch (mirrors the library's choice; used to count launches)."""
    T = dims.P + dims.C
    if dims.hd == 128 and dims.P % 128 == 0:
        units = math.ceil(math.ceil(dims.Hq // dims.Hkv * dims.C / 128) / 2) * dims.B * dims.Hkv
        ns, blk = min(152 // units, math.ceil(T / 256), 64), 128
    else:
        units = math.ceil(dims.C / 64) * dims.B * dims.Hq
        ns, blk = min(math.ceil(3 * 152 / units), math.ceil(T / 256), 64), 64
    ns = max(ns, 1)
    kps = math.ceil(math.ceil(T / ns) / blk) * blk
    return math.ceil(T / kps)


def main():
    args = _args()
    world, rank, local = _dist()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
