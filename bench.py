#!/usr/bin/env python
"""Benchmark of the tensor-parallel layer forward on one B300 (per GPU).

Headline: decode weight-stream GB/s on a Qwen2.5-1.5B-shaped stack -- 28
serial pre-norm decoder layers (D=1536, SwiGLU F=8960, 12 Q / 2 KV heads of
128), TP=2 logical shards, distinct random weights per layer (2.6 GB, far
larger than the 126 MB L2, so no flush is needed) -- decoding one batch of
each size in {1, 8, 32, 64} per step.  GB/s counts the unique projection
weight bytes each forward must read (93,585,408 per layer).

Alongside: prefill TFLOP/s of the Llama-3.1-70B-shaped MLP (X[4096, 8192],
F=28672, TP=8), flops 2*B*D*2F + 2*B*F*D.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With torchrun (N > 1) every rank runs an independent replica (weak scaling,
no collective on the data path); value = units of all ranks / max time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic_inputs as si  # noqa: E402

METRIC = "decode weight-stream GB/s & prefill TFLOP/s per TP-sharded layer, 1×B300"
QW = si.QWEN_DECODE
LD = si.LLAMA_DECODE
LP = si.LLAMA_PREFILL


def layer_bytes(D, F, n_q, n_kv, hd):
    return 2 * ((n_q + 2 * n_kv) * hd * D + D * n_q * hd + 3 * D * F)


QWEN_LAYER_BYTES = layer_bytes(QW["D"], QW["F"], QW["n_q"], QW["n_kv"], QW["head_dim"])
LLAMA_LAYER_BYTES = layer_bytes(LD["D"], LD["F"], LD["n_q"], LD["n_kv"], LD["head_dim"])
PREFILL_FLOPS = 2 * LP["B"] * LP["D"] * 2 * LP["F"] + 2 * LP["B"] * LP["F"] * LP["D"]


def args_parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=QW["n_layers"])
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-llama", action="store_true", help="skip the Llama-3.1-70B-shaped decode stack")
    ap.add_argument("--no-cases", action="store_true", help="skip the sharded-matmul cases and shard_reduce")
    ap.add_argument("--no-lm-head", action="store_true", help="skip the vocabulary-parallel lm_head lines")
    ap.add_argument("--no-w8", action="store_true", help="skip the weight-only int8 MLP lines")
    ap.add_argument("--no-unfused", action="store_true",
                    help="skip timing the unfused decode path beside the fused one")
    ap.add_argument("--model", "--lm-head-model", dest="model", choices=["llama-3.1-70b", "qwen2.5-1.5b"],
                    default=None, help="with --only lm_head or --only w8: one model's shape only "
                                       "(--batches selects the batch sizes)")
    ap.add_argument("--llama-layers", type=int, default=LD["n_layers"],
                    help="layers of the Llama-3.1-70B-shaped decode stack (small captures)")
    ap.add_argument("--only", choices=["decode", "prefill", "llama", "lm_head", "w8", "cases"], default=None,
                    help="run one workload only (small cases for profiling); prints that workload's line")
    ap.add_argument("--batches", type=str, default=None, help="decode batch sizes, comma-separated")
    ap.add_argument("--phase-trace", action="store_true",
                    help="per-phase timeline of the fused decode stack from the instrumented library "
                         "(build it with: python mlp_megatron_tp_layer_b300/build.py --trace); with "
                         "--model, --batches and --layers; prints one JSON line per batch size")
    ap.add_argument("--prefill-tokens", type=int, default=LP["B"])
    ap.add_argument("--block", choices=["serial", "parallel"], default="serial", help="with --phase-trace")
    return ap.parse_args()


# ------------------------------------------------------------ distributed

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["smax"] for r in rows),
                "samples": len(loaded), "power_w_max": max(r["power"] for r in rows), "reasons": sorted(reasons)}


FUSED_SOURCES = ("decode_fused.cu", "ptx.cuh", "epilogue.cuh", "internal.h")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fused_stack_traffic.txt")


def fused_source_hash():
    import hashlib
    h = hashlib.sha256()
    for name in FUSED_SOURCES:
        with open(os.path.join(ROOT, "mlp_megatron_tp_layer_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def fused_traffic(batches):
    """Mean DRAM bytes per launch of the fused stack over the given batch sizes,
    from the committed ncu summary, or None if it is missing or was taken on
    different kernel sources."""
    try:
        kv = dict(line.strip().split("=", 1) for line in open(TRAFFIC_FILE)
                  if "=" in line and not line.startswith("#"))
    except OSError:
        return None
    if kv.get("source_sha256_16") != fused_source_hash():
        return None
    try:
        vals = [float(kv[f"qwen_28_layers_b{B}"]) for B in batches]
    except KeyError:
        return None
    return sum(vals) / len(vals)


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


# ------------------------------------------------------------- workloads

def qwen_stack(n_layers, device):
    return [si.layer_weights(QW["D"], QW["F"], QW["n_q"], QW["n_kv"], QW["head_dim"], seed=0, layer=l,
                             prefix="qwen", device=device) for l in range(n_layers)]


def cpu_baseline(layers_dev, budget_s):
    """The oracle, as it stands, on the host cores: one Qwen-shaped layer decoded
    at each batch size, repeated until the budget is used; GB/s of weights."""
    import numpy as np
    from oracle import tp_layer as O
    try:
        from threadpoolctl import threadpool_info
        cores = max([int(p.get("num_threads", 1)) for p in threadpool_info()] + [1])
    except Exception:  # noqa: BLE001
        cores = len(os.sched_getaffinity(0))
    W = {k: v.to("cpu", torch.float64).numpy() for k, v in layers_dev[0].items()}
    xs = {B: si.activations(B, QW["D"], seed=1, name=f"bench.x{B}").to(torch.float64).numpy()
          for B in QW["batches"]}
    def timed(budget):
        n = 0
        t0 = time.perf_counter()
        while True:
            for B in QW["batches"]:
                O.decoder_layer(xs[B], W, QW["n_q"], QW["n_kv"], QW["head_dim"], QW["tp"])
                n += 1
            if time.perf_counter() - t0 > budget:
                break
        return n, time.perf_counter() - t0

    n, dt = timed(budget_s)
    single, why = None, None
    try:
        single = oracle_one_thread(W, xs, budget_s / 4)
    except Exception as e:  # noqa: BLE001
        why = f"{type(e).__name__}: {e}"[:300]
    del np
    out = {"value": n * QWEN_LAYER_BYTES / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
           "single_thread_value": single,
           "sample": f"{n // len(QW['batches'])} passes of one Qwen-shaped TP=2 layer over B in "
                     f"{list(QW['batches'])} (numpy float64), {dt:.1f} s; then the same in a child process "
                     f"with every BLAS/OpenMP pool at one thread, for a quarter of that budget"}
    if why:
        out["single_thread_error"] = why
    return out


ONE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                  "NUMEXPR_NUM_THREADS", "VECLIB_MAXIMUM_THREADS")


def oracle_one_thread(W, xs, budget_s):
    """GB/s of the oracle decoding one Qwen-shaped layer at every batch size in
    a child process whose thread pools are all limited to one thread by the
    environment (set before numpy loads its BLAS); the arrays go by file."""
    import numpy as np
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    try:
        np.savez(path, **{f"W_{k}": v for k, v in W.items()}, **{f"x_{B}": v for B, v in xs.items()})
        code = (
            "import sys, time, numpy as np\n"
            f"sys.path.insert(0, {ROOT!r})\n"
            "from oracle import tp_layer as O\n"
            "z = np.load(sys.argv[1])\n"
            "W = {k[2:]: z[k] for k in z.files if k.startswith('W_')}\n"
            "xs = [z[k] for k in z.files if k.startswith('x_')]\n"
            f"n, t0 = 0, time.perf_counter()\n"
            "while True:\n"
            "    for x in xs:\n"
            f"        O.decoder_layer(x, W, {QW['n_q']}, {QW['n_kv']}, {QW['head_dim']}, {QW['tp']})\n"
            "        n += 1\n"
            f"    if time.perf_counter() - t0 > {budget_s}:\n"
            "        break\n"
            "print(n, time.perf_counter() - t0)\n")
        env = dict(os.environ, **{k: "1" for k in ONE_THREAD_ENV})
        r = subprocess.run([sys.executable, "-c", code, path], env=env, capture_output=True, text=True,
                           timeout=budget_s * 4 + 120)
        if r.returncode != 0:
            raise RuntimeError(r.stderr.strip().splitlines()[-1] if r.stderr.strip() else f"rc {r.returncode}")
        n, dt = r.stdout.split()
        return int(n) * QWEN_LAYER_BYTES / float(dt) / 1e9
    finally:
        os.unlink(path)


def run_reference(args, rank, world):
    """--impl reference: the oracle timed on the host cores, same metric and workload."""
    if rank != 0:
        return
    import numpy as np
    from oracle import tp_layer as O
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    W = {k: v.to("cpu", torch.float64).numpy() for k, v in qwen_stack(1, dev)[0].items()}
    xs = {B: si.activations(B, QW["D"], seed=1, name=f"bench.x{B}").to(torch.float64).numpy()
          for B in QW["batches"]}

    def step():
        for B in QW["batches"]:
            O.decoder_layer(xs[B], W, QW["n_q"], QW["n_kv"], QW["head_dim"], QW["tp"])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    try:
        from threadpoolctl import threadpool_info
        cores = max([int(p.get("num_threads", 1)) for p in threadpool_info()] + [1])
    except Exception:  # noqa: BLE001
        cores = len(os.sched_getaffinity(0))
    units = args.steps * len(QW["batches"]) * QWEN_LAYER_BYTES
    value = units / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "Qwen2.5-1.5B-shaped decode layer, TP=2 logical shards, B in {1,8,32,64} "
                                   "(one layer per step: a bounded sample of the 28-layer stack)"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} steps x one layer x 4 batches"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    del np
    print(json.dumps(line), flush=True)


def profile_pass(tpl, fn, stream):
    """Per-launch device times of one call of fn: fn is captured into a CUDA
    graph with the library's launch timing on (event-record nodes around every
    kernel), replayed, and the last replay's times returned as [(tag, ms)]."""
    tpl.profile_enable(8192)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    rec = tpl.profile_records()
    tpl.profile_disable()
    del g
    return rec


def run_decode(args, tpl, dev, world, peaks, peak_kind, stream):
    """The headline: the decode stack at every batch size, graph-replayed."""
    D, F, n_q, n_kv, hd, tp = QW["D"], QW["F"], QW["n_q"], QW["n_kv"], QW["head_dim"], QW["tp"]
    batches = [int(b) for b in args.batches.split(",")] if args.batches else list(QW["batches"])
    L = args.layers

    layers = qwen_stack(L, dev)
    xs = {B: si.activations(B, D, seed=1, name=f"bench.x{B}", device=dev) for B in batches}
    ys = {B: torch.empty_like(xs[B]) for B in batches}
    ws = tpl.workspace(max(tpl.decoder_workspace_bytes(B, D, F, n_q, n_kv, hd, tp) for B in batches), dev)

    def forward(B, x=None, y=None):
        tpl.tp_decoder_stack(xs[B] if x is None else x, layers, n_q, n_kv, hd, tp,
                             out=ys[B] if y is None else y, ws=ws)

    def eager_step():
        for B in batches:
            forward(B)

    # launch list and per-kernel device times (inside a graph, events around each launch)
    eager_step()
    torch.cuda.synchronize()
    recs = profile_pass(tpl, eager_step, stream)
    # launch_rmsnorm scopes also hold one small zeroing kernel
    launches_per_step = len(recs) + sum(1 for t, _ in recs if t == "rmsnorm")

    # CUDA graphs: one per batch size, replaying the library's launches
    graphs = {}
    with torch.cuda.stream(stream):
        for B in batches:
            forward(B)
    torch.cuda.synchronize()
    for B in batches:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            forward(B)
        graphs[B] = g
    torch.cuda.synchronize()

    def step():
        for B in batches:
            graphs[B].replay()

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    for _ in range(args.warmup):
        step()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    clk = clocks.stop()
    ms = max_over_ranks(ms, world)
    units_per_step = L * len(batches) * QWEN_LAYER_BYTES
    value = units_per_step * args.steps * world / (ms / 1e3) / 1e9

    # per-batch breakdown
    per_batch = {}
    for B in batches:
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(max(3, args.steps // 2)):
            graphs[B].replay()
        b.record()
        torch.cuda.synchronize()
        t = a.elapsed_time(b) / max(3, args.steps // 2)
        per_batch[str(B)] = {"ms_per_forward": t, "GB/s": L * QWEN_LAYER_BYTES / (t / 1e3) / 1e9,
                             "TFLOP/s": 2 * B * L * QWEN_LAYER_BYTES / 2 / (t / 1e3) / 1e12}

    # end to end: pinned host x in, host y out, inside the timed region
    hx = {B: xs[B].to("cpu").pin_memory() for B in batches}
    hy = {B: torch.empty_like(hx[B]).pin_memory() for B in batches}
    with torch.cuda.stream(stream):
        for B in batches:
            xs[B].copy_(hx[B], non_blocking=True)
    torch.cuda.synchronize()
    h2d = sum(hx[B].numel() * hx[B].element_size() for B in batches)
    d2h = sum(hy[B].numel() * hy[B].element_size() for B in batches)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            for B in batches:
                xs[B].copy_(hx[B], non_blocking=True)
                graphs[B].replay()
                hy[B].copy_(ys[B], non_blocking=True)
            stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e = {"value": units_per_step * args.steps * world / e2e_s / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    # roofline of the dominant kernel (largest total device time in the launch list)
    tot = {}
    for tag, t in recs:
        n, s = tot.get(tag, (0, 0.0))
        tot[tag] = (n + 1, s + t)
    dom = max(tot, key=lambda k: tot[k][1])
    # algorithmic bytes of one launch of each step: the weights it must stream
    # once plus its activation input and output (per-layer steps launch L times
    # per forward, the fused stack once per forward for all L layers)
    alg = {"gateup": lambda B: L * (2 * F * D * 2 + B * D * 2 + B * F * 2),
           "down": lambda B: L * (D * F * 2 + B * F * 2 + B * D * 4),
           "qkv": lambda B: L * ((n_q + 2 * n_kv) * hd * D * 2 + B * D * 2),
           "oproj": lambda B: L * (D * n_q * hd * 2 + B * n_q * hd * 2),
           "fused_stack": lambda B: L * QWEN_LAYER_BYTES + 2 * B * D * 2}
    roof = None
    if dom in alg:
        total_bytes = sum(alg[dom](B) for B in batches)
        n_launch, t_ms = tot[dom]
        achieved = total_bytes / (t_ms / 1e3) / 1e9
        traffic = fused_traffic(batches) if dom == "fused_stack" and L == QW["n_layers"] else None
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "peak_kind": peak_kind,
                "launches": n_launch, "avg_launch_us": t_ms / n_launch * 1e3,
                "algorithmic_bytes_per_launch_avg": total_bytes / n_launch}
    share = {k: {"launches": v[0], "ms": v[1], "share": v[1] / sum(x[1] for x in tot.values())}
             for k, v in sorted(tot.items(), key=lambda kv: -kv[1][1])}
    # per batch size: average device time of each step of one layer (us)
    per_fwd = len(recs) // len(batches)
    for bi, B in enumerate(batches):
        grp = recs[bi * per_fwd:(bi + 1) * per_fwd]
        agg = {}
        for tag, t in grp:
            n, s_ = agg.get(tag, (0, 0.0))
            agg[tag] = (n + 1, s_ + t)
        per_batch[str(B)]["kernel_us"] = {k: round(v[1] / v[0] * 1e3, 2) for k, v in agg.items()}
        per_batch[str(B)]["sum_kernel_us_per_layer"] = round(sum(v[1] for v in agg.values()) / L * 1e3, 2)
    # the unfused path (one launch per projection and reduction, graph-
    # replayed) beside the fused one, per batch size: what the automatic path
    # choice rests on
    if not args.no_unfused:
        for B in batches:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                tpl.tp_decoder_stack(xs[B], layers, n_q, n_kv, hd, tp, out=ys[B], ws=ws, path=tpl.PATH_UNFUSED)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                tpl.tp_decoder_stack(xs[B], layers, n_q, n_kv, hd, tp, out=ys[B], ws=ws, path=tpl.PATH_UNFUSED)
            t = time_ms(g.replay, max(3, args.steps // 4))
            per_batch[str(B)]["unfused"] = {"ms_per_forward": t, "GB/s": L * QWEN_LAYER_BYTES / (t / 1e3) / 1e9}
            del g
    out = {"value": value, "ms": ms, "batches": batches, "L": L, "roofline": roof, "e2e": e2e,
           "gpu_launches": launches_per_step * args.steps, "clocks": clk, "per_batch": per_batch,
           "kernel_share": share, "layers": layers}
    return out


def run_parallel_block(args, tpl, dev, layers, peaks, stream):
    """The same Qwen-shaped stack in the parallel (PaLM) arrangement of the
    pages (y = x + Attn(RMSNorm x) + MLP(RMSNorm x), one shared reduction per
    layer): weight-stream GB/s per batch size, graph-replayed."""
    D, F, n_q, n_kv, hd, tp = QW["D"], QW["F"], QW["n_q"], QW["n_kv"], QW["head_dim"], QW["tp"]
    L = len(layers)
    out = {"workload": f"Qwen2.5-1.5B-shaped decode, parallel block, {L} layers, TP=2", "per_batch": {}}
    for B in QW["batches"]:
        x = si.activations(B, D, seed=1, name=f"bench.x{B}", device=dev)
        y = torch.empty_like(x)
        ws = tpl.workspace(tpl.decoder_workspace_bytes(B, D, F, n_q, n_kv, hd, tp), dev)
        with torch.cuda.stream(stream):
            tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, out=y, ws=ws, block=tpl.BLOCK_PARALLEL)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, out=y, ws=ws, block=tpl.BLOCK_PARALLEL)
        t = time_ms(g.replay, max(5, args.steps // 2))
        gbs = L * QWEN_LAYER_BYTES / (t / 1e3) / 1e9
        out["per_batch"][str(B)] = {"ms_per_forward": t, "GB/s": gbs, "frac_of_peak": gbs / peaks["hbm_gbs"]}
        del g
    return out


def run_llama_decode(args, tpl, dev, world, peaks, peak_kind, stream):
    """Llama-3.1-70B-shaped decode stack (8 layers, TP=8, 13.69 GB of weights),
    one graph-replayed forward per batch size: weight-stream GB/s per batch."""
    D, F, n_q, n_kv, hd, tp = LD["D"], LD["F"], LD["n_q"], LD["n_kv"], LD["head_dim"], LD["tp"]
    L = args.llama_layers
    batches = list(LD["batches"])
    if args.only == "llama" and args.batches:
        batches = [int(b) for b in args.batches.split(",")]
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=0, layer=l, prefix="llama", device=dev) for l in range(L)]
    xs = {B: si.activations(B, D, seed=3, name=f"llama.x{B}", device=dev) for B in batches}
    ys = {B: torch.empty_like(xs[B]) for B in batches}
    ws = tpl.workspace(max(tpl.decoder_workspace_bytes(B, D, F, n_q, n_kv, hd, tp) for B in batches), dev)
    graphs = {}
    with torch.cuda.stream(stream):
        for B in batches:
            tpl.tp_decoder_stack(xs[B], layers, n_q, n_kv, hd, tp, out=ys[B], ws=ws)
    torch.cuda.synchronize()
    for B in batches:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            tpl.tp_decoder_stack(xs[B], layers, n_q, n_kv, hd, tp, out=ys[B], ws=ws)
        graphs[B] = g
    out = {"workload": f"Llama-3.1-70B-shaped decode stack: {L} layers D=8192 F=28672 64Q/8KV x128, TP=8 "
                       f"logical shards, {L * LLAMA_LAYER_BYTES / 1e9:.2f} GB of weights per forward",
           "per_batch": {}}
    reps = max(3, args.steps // 4)
    for B in batches:
        warm_up(graphs[B].replay, n_min=2)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            graphs[B].replay()
        b.record()
        torch.cuda.synchronize()
        t = a.elapsed_time(b) / reps
        gbs = L * LLAMA_LAYER_BYTES / (t / 1e3) / 1e9
        out["per_batch"][str(B)] = {"ms_per_forward": t, "GB/s": gbs, "frac_of_peak": gbs / peaks["hbm_gbs"]}
    if not args.no_unfused:
        for B in batches:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                tpl.tp_decoder_stack(xs[B], layers, n_q, n_kv, hd, tp, out=ys[B], ws=ws, path=tpl.PATH_UNFUSED)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                tpl.tp_decoder_stack(xs[B], layers, n_q, n_kv, hd, tp, out=ys[B], ws=ws, path=tpl.PATH_UNFUSED)
            t = time_ms(g.replay, reps)
            out["per_batch"][str(B)]["unfused"] = {"ms_per_forward": t,
                                                   "GB/s": L * LLAMA_LAYER_BYTES / (t / 1e3) / 1e9}
            del g
    del layers, graphs
    torch.cuda.empty_cache()
    return out


# Vocabulary-parallel lm_head shapes: the models' vocabularies and hidden sizes
# with the TP degree of their decode configurations.
LM_HEADS = {
    "llama-3.1-70b": {"D": 8192, "V": 128256, "tp": 8, "batches": (1, 8, 64, 128)},
    "qwen2.5-1.5b": {"D": 1536, "V": 151936, "tp": 2, "batches": (1, 8, 32, 64)},
}


def run_lm_head(args, tpl, dev, peaks, stream, k=1):
    """Greedy next-token selection through the vocabulary-parallel lm_head:
    per-shard top-k in the GEMM epilogue, then the candidate exchange.  One
    graph-replayed call per batch size; GB/s counts the weight and input bytes
    (V*D*2 + B*D*2), the logits never being written."""
    out = {}
    reps = max(5, args.steps // 2)
    for name, c in LM_HEADS.items():
        if args.only == "lm_head" and args.model not in (None, name):
            continue
        D, V, tp = c["D"], c["V"], c["tp"]
        batches = c["batches"]
        if args.only == "lm_head" and args.batches:
            batches = tuple(int(b) for b in args.batches.split(","))
        x_all, W = si.lm_head(max(batches), D, V, seed=0, device=dev)
        res = {"workload": f"{name}-shaped lm_head: W[{V}, {D}] bf16 ({V * D * 2 / 1e9:.2f} GB), "
                           f"TP={tp} vocabulary shards, top-{k} per shard then exchange",
               "per_batch": {}}
        for B in batches:
            x = x_all[:B].contiguous()
            idx = torch.empty(B, k, dtype=torch.int32, device=dev)
            val = torch.empty(B, k, dtype=torch.float32, device=dev)
            ws = tpl.workspace(tpl.vocab_topk_workspace_bytes(B, V, tp, k), dev)
            with torch.cuda.stream(stream):
                tpl.vocab_parallel_topk(x, W, tp, k, out=(idx, val), ws=ws)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                tpl.vocab_parallel_topk(x, W, tp, k, out=(idx, val), ws=ws)
            warm_up(g.replay)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            t = a.elapsed_time(b) / reps
            gbs = (V * D * 2 + B * D * 2) / (t / 1e3) / 1e9
            res["per_batch"][str(B)] = {"ms": t, "GB/s": gbs, "frac_of_peak": gbs / peaks["hbm_gbs"]}
            del g
        out[name] = res
        del x_all, W
        torch.cuda.empty_cache()
    return out


# Weight-only int8 decode MLP shapes (the decode configurations' MLPs).
W8_MLPS = {
    "qwen2.5-1.5b": {"D": 1536, "F": 8960, "tp": 2, "batches": (1, 8, 32, 64)},
    "llama-3.1-70b": {"D": 8192, "F": 28672, "tp": 8, "batches": (1, 8, 32, 64)},
}
L2_BYTES = 126 * 2 ** 20


def run_w8_mlp(args, tpl, dev, peaks, stream):
    """Decode MLP with int8 weights against the same MLP in bf16.  Enough
    distinct weight copies are cycled that every timed pass streams more than
    three L2s of int8 weights; GB/s counts the bytes each MLP must read
    (int8 codes + float32 scales, or bf16 weights) per forward."""
    out = {}
    reps = max(3, args.steps // 5)
    for name, c in W8_MLPS.items():
        if args.only == "w8" and args.model not in (None, name):
            continue
        D, F, tp = c["D"], c["F"], c["tp"]
        batches = c["batches"]
        if args.only == "w8" and args.batches:
            batches = tuple(int(b) for b in args.batches.split(","))
        b8 = 3 * D * F + 4 * (2 * F + D * tp)
        b16 = 3 * D * F * 2
        copies = max(1, math.ceil(3 * L2_BYTES / b8))
        weights = []
        for i in range(copies):
            Wg = si.normal((F, D), 0.02, 0, f"{name}.w8.Wg{i}", device=dev)
            Wu = si.normal((F, D), 0.02, 0, f"{name}.w8.Wu{i}", device=dev)
            Wd = si.normal((D, F), 0.02, 0, f"{name}.w8.Wd{i}", device=dev)
            q = tpl.quantize_w8(Wg) + tpl.quantize_w8(Wu) + tpl.quantize_w8(Wd, groups=tp)
            weights.append(((Wg, Wu, Wd), q))
        res = {"workload": f"{name}-shaped decode MLP D={D} F={F}, TP={tp}: int8 weights "
                           f"({b8 / 1e6:.1f} MB) vs bf16 ({b16 / 1e6:.1f} MB), {copies} weight copies cycled",
               "per_batch": {}}
        for B in batches:
            x = si.activations(B, D, seed=5, name=f"{name}.w8.x{B}", device=dev)
            y8 = torch.empty(B, D, dtype=torch.bfloat16, device=dev)
            y16 = torch.empty_like(y8)
            ws8 = tpl.workspace(tpl.mlp_w8_workspace_bytes(B, D, F, tp), dev)
            ws16 = torch.empty(tpl.mlp_workspace_bytes(B, D, F, tp), dtype=torch.uint8, device=dev)
            times = {}
            for kind in ("w8", "bf16"):
                def call():
                    for (Wg, Wu, Wd), q in weights:
                        if kind == "w8":
                            tpl.tp_mlp_forward_w8(x, *q, tp, out=y8, ws=ws8)
                        else:
                            tpl.tp_mlp_forward(x, Wg, Wu, Wd, tp, out=y16, ws=ws16)
                with torch.cuda.stream(stream):
                    call()
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    call()
                warm_up(g.replay)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for _ in range(reps):
                    g.replay()
                b.record()
                torch.cuda.synchronize()
                times[kind] = a.elapsed_time(b) / reps / copies
                del g
            gbs = b8 / (times["w8"] / 1e3) / 1e9
            res["per_batch"][str(B)] = {"ms_int8": times["w8"], "ms_bf16": times["bf16"],
                                        "speedup": times["bf16"] / times["w8"], "int8_GB/s": gbs,
                                        "frac_of_peak": gbs / peaks["hbm_gbs"],
                                        "bf16_GB/s": b16 / (times["bf16"] / 1e3) / 1e9}
        out[name] = res
        del weights
        torch.cuda.empty_cache()
    return out


def warm_up(fn, min_ms=10.0, n_min=3):
    """Untimed calls of fn: at least n_min of them and at least min_ms of wall
    time.  Three calls alone left the first batch size timed after new weights
    were created about 6 us slow on an 85 us lm_head call."""
    for _ in range(n_min):
        fn()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    while (time.perf_counter() - t0) * 1e3 < min_ms:
        fn()
        torch.cuda.synchronize()


def time_ms(fn, reps):
    """Average device time of fn over reps calls (CUDA events, after warm_up)."""
    warm_up(fn)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def run_cases_and_reduce(args, tpl, dev, peaks, peak_kind):
    """The four sharded-matmul cases at A[512,8192] . B[8192,28672], X = 8 (TFLOP/s,
    bf16 output), and shard_reduce over 8 fp32 partial planes of a [4096, 8192] output."""
    SC = si.SHARDED_CASES
    d = si.sharded_case_operands(SC["I"], SC["J"], SC["K"], seed=0, device=dev)
    flops = 2 * SC["I"] * SC["J"] * SC["K"]
    cases = {}
    for name, case, mode, gather in (("1", 1, 0, 0), ("2", 2, 0, 0), ("3 all-reduce", 3, 0, 0),
                                     ("3 reduce-scatter", 3, 1, 0), ("3 via partials", 3, 0, 0),
                                     ("4 gather B", 4, 0, 0), ("4 gather A", 4, 0, 1)):
        want_p = name == "3 via partials"
        P = torch.empty((SC["X"], SC["I"], SC["K"]), dtype=torch.float32, device=dev) if want_p else None
        ws = tpl.workspace(tpl.case_workspace_bytes(case, mode, SC["I"], SC["J"], SC["K"], SC["X"]), dev)
        k_sh = (case == 3 and mode == 1) or (case == 4 and gather == 1)
        C = torch.empty((SC["X"], SC["I"], SC["K"] // SC["X"]) if k_sh else (SC["I"], SC["K"]), dtype=torch.bfloat16,
                        device=dev)
        t = time_ms(lambda: tpl.sharded_matmul(case, d["A"], d["Bt"], SC["X"], mode, gather, out=C,
                                               partials=P if want_p else None, ws=ws), max(10, args.steps))
        cases[name] = {"ms": t, "TFLOP/s": flops / (t / 1e3) / 1e12}
    del d
    rows, cols, tp = LP["B"], LP["D"], LP["tp"]
    Pr = si.normal((tp, rows, cols), 1.0, 0, "bench.partials", torch.float32, device=dev)
    Yr = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
    t = time_ms(lambda: tpl.shard_reduce(Pr, tpl.ALLREDUCE, out=Yr), max(10, args.steps))
    nbytes = tp * rows * cols * 4 + rows * cols * 2
    red = {"workload": f"shard_reduce: {tp} fp32 planes [{rows}, {cols}] -> bf16", "ms": t,
           "GB/s": nbytes / (t / 1e3) / 1e9, "frac_of_peak": nbytes / (t / 1e3) / 1e9 / peaks["hbm_gbs"],
           "peak_kind": peak_kind}
    del Pr, Yr
    return {"workload": f"sharded matmul A[{SC['I']},{SC['J']}] . B[{SC['J']},{SC['K']}], X={SC['X']}, bf16 out",
            "per_case": cases}, red


def run_prefill(args, tpl, dev, world, peaks, peak_kind, stream):
    """Llama-3.1-70B-shaped prefill MLP (TP=8), fused shard reduce."""
    T = args.prefill_tokens
    P = si.prefill_mlp(T, LP["D"], LP["F"], seed=0, device=dev)
    Yp = torch.empty((T, LP["D"]), dtype=torch.bfloat16, device=dev)
    pws = tpl.workspace(tpl.mlp_workspace_bytes(T, LP["D"], LP["F"], LP["tp"]), dev)

    def pstep():
        tpl.tp_mlp_forward(P["X"], P["Wg"], P["Wu"], P["Wd"], LP["tp"], out=Yp, ws=pws)

    for _ in range(max(3, args.warmup)):
        pstep()
    precs = profile_pass(tpl, pstep, stream)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    psteps = max(5, args.steps // 5)
    a.record()
    for _ in range(psteps):
        pstep()
    b.record()
    torch.cuda.synchronize()
    pms = max_over_ranks(a.elapsed_time(b) / psteps, world)
    gu = [t for tag, t in precs if tag == "gateup"]
    dn = [t for tag, t in precs if tag == "down"]
    gu_flops = 2 * T * LP["D"] * 2 * LP["F"]
    dn_flops = 2 * T * LP["F"] * LP["D"]
    flops = gu_flops + dn_flops
    prefill = {"workload": f"Llama-3.1-70B-shaped prefill MLP X[{T},8192], F=28672, TP=8, fused shard reduce",
               "value": flops / (pms / 1e3) / 1e12 * world, "unit": "TFLOP/s", "ms_per_step": pms,
               "roofline": {"bound": "tensor", "kernel": "gateup", "achieved": gu_flops / (gu[0] / 1e3) / 1e12,
                            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": gu_flops / (gu[0] / 1e3) / 1e12 / peaks["bf16_tflops"],
                            "traffic": None, "peak_kind": peak_kind + " burst"} if gu else None,
               "down_TFLOP/s": dn_flops / (dn[0] / 1e3) / 1e12 if dn else None,
               "launches_per_step": len(precs)}
    del P
    return prefill


TRACE_EVENTS = ("act_ready", "mma_start", "first_ticket", "drained", "fin_start", "published", "w_first",
                "act_wait", "mma_first_unit_done", "w_last", "acc_first", "act_last")


def run_phase_trace(args):
    """Per-phase event times of one fused-stack launch (instrumented library):
    for every phase, the median and the maximum over CTAs of each event, in us
    from the launch's first stamp.  Not a benchmark number: the stamps add a
    few stores per phase."""
    os.environ["TPL_LIBRARY"] = os.path.join(ROOT, "mlp_megatron_tp_layer_b300", "libtpl_trace.so")
    import numpy as np
    import mlp_megatron_tp_layer_b300 as tpl
    model = args.model or "qwen2.5-1.5b"
    cfg = QW if model.startswith("qwen") else LD
    D, F, n_q, n_kv, hd, tp = cfg["D"], cfg["F"], cfg["n_q"], cfg["n_kv"], cfg["head_dim"], cfg["tp"]
    L = min(args.layers, 4) if model.startswith("qwen") else min(args.llama_layers, 2)
    block = tpl.BLOCK_PARALLEL if args.block == "parallel" else tpl.BLOCK_SERIAL
    prefix = "qwen" if model.startswith("qwen") else "llama"
    layers = [si.layer_weights(D, F, n_q, n_kv, hd, seed=0, layer=l, prefix=prefix, device="cuda") for l in range(L)]
    batches = [int(b) for b in args.batches.split(",")] if args.batches else list(cfg["batches"])
    kinds = ["QKV", "GATEUP", "OPROJ", "DOWN"] if block == tpl.BLOCK_PARALLEL else ["QKV", "OPROJ", "GATEUP", "DOWN"]
    for B in batches:
        x = si.activations(B, D, seed=1, name=f"bench.x{B}", device="cuda")
        for _ in range(3):
            y = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, block=block, path=tpl.PATH_FUSED)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        y = tpl.tp_decoder_stack(x, layers, n_q, n_kv, hd, tp, block=block, path=tpl.PATH_FUSED)
        b.record()
        torch.cuda.synchronize()
        tr = tpl.fused_trace().astype(np.float64)
        t0 = tr[tr > 0].min()
        tr = np.where(tr > 0, (tr - t0) / 1e3, np.nan)
        phases = []
        for k in range(1, 4 * L + 1):
            row = {"phase": k, "layer": (k - 1) // 4, "kind": kinds[(k - 1) % 4]}
            for e, name in enumerate(TRACE_EVENTS):
                v = tr[:, k, e]
                v = v[~np.isnan(v)]
                if v.size:
                    row[name] = [round(float(np.median(v)), 2), round(float(v.max()), 2)]
            phases.append(row)
        print(json.dumps({"phase_trace": model, "block": args.block, "B": B, "layers": L,
                          "launch_us": round(a.elapsed_time(b) * 1e3, 1), "events": "[median, max] us over CTAs",
                          "phases": phases}), flush=True)
        del y


def main():
    args = args_parse()
    if args.phase_trace:
        run_phase_trace(args)
        return
    rank, world = dist_init()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import mlp_megatron_tp_layer_b300 as tpl
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks, peak_kind = measured_peaks()
    stream = torch.cuda.Stream(device=dev)

    if args.only == "prefill":
        pre = run_prefill(args, tpl, dev, world, peaks, peak_kind, stream)
        if rank == 0:
            print(json.dumps(dict(pre, metric=METRIC, n_gpus=world, steps=args.steps, warmup=args.warmup)),
                  flush=True)
        return
    if args.only == "w8":
        w8 = run_w8_mlp(args, tpl, dev, peaks, stream)
        if rank == 0:
            print(json.dumps(dict(w8_mlp=w8, metric=METRIC, n_gpus=world, steps=args.steps)), flush=True)
        return
    if args.only == "lm_head":
        lm = run_lm_head(args, tpl, dev, peaks, stream)
        if rank == 0:
            print(json.dumps(dict(lm_head=lm, metric=METRIC, n_gpus=world, steps=args.steps)), flush=True)
        return
    if args.only == "cases":
        cases, reduce_line = run_cases_and_reduce(args, tpl, dev, peaks, peak_kind)
        if rank == 0:
            print(json.dumps(dict(sharded_matmul=cases, shard_reduce=reduce_line, metric=METRIC, n_gpus=world,
                                  steps=args.steps)), flush=True)
        return
    if args.only == "llama":
        ll = run_llama_decode(args, tpl, dev, world, peaks, peak_kind, stream)
        if rank == 0:
            print(json.dumps(dict(ll, metric=METRIC, n_gpus=world, steps=args.steps)), flush=True)
        return

    dec = run_decode(args, tpl, dev, world, peaks, peak_kind, stream)
    parallel = None
    if args.only is None:
        parallel = run_parallel_block(args, tpl, dev, dec["layers"], peaks, stream)
    llama = None
    if not args.no_llama and args.only is None:
        llama = run_llama_decode(args, tpl, dev, world, peaks, peak_kind, stream)
    prefill = None
    if not args.no_prefill and args.only is None:
        prefill = run_prefill(args, tpl, dev, world, peaks, peak_kind, stream)

    lm_head = None
    if not args.no_lm_head and args.only is None:
        lm_head = run_lm_head(args, tpl, dev, peaks, stream)

    w8 = None
    if not args.no_w8 and args.only is None:
        w8 = run_w8_mlp(args, tpl, dev, peaks, stream)

    cases = reduce_line = None
    if not args.no_cases and args.only is None:
        cases, reduce_line = run_cases_and_reduce(args, tpl, dev, peaks, peak_kind)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.only is None:
        cpu = cpu_baseline(dec["layers"], args.cpu_seconds)

    if rank == 0:
        L, batches = dec["L"], dec["batches"]
        line = {"metric": METRIC, "value": dec["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": dec["ms"] / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": f"Qwen2.5-1.5B-shaped decode: {L} serial pre-norm layers D=1536 F=8960 "
                                       f"12Q/2KV heads x128, TP=2 logical shards, one forward per B in "
                                       f"{list(batches)} per step",
                           "global_batch": sum(batches), "parallelism": "tp2 logical shards; 1 replica per GPU",
                           "l2": f"weights {L * QWEN_LAYER_BYTES / 1e9:.2f} GB per forward > 126 MB L2; no flush",
                           "graphs": "one CUDA graph per batch size"},
                "roofline": dec["roofline"], "cpu_baseline": cpu, "e2e": dec["e2e"],
                "gpu_launches": dec["gpu_launches"], "clocks": dec["clocks"],
                "per_batch": dec["per_batch"], "kernel_share": dec["kernel_share"],
                "qwen_decode_parallel_block": parallel, "llama_decode": llama,
                "prefill": prefill, "lm_head_topk": lm_head, "mlp_int8_weights": w8, "sharded_matmul": cases,
                "shard_reduce": reduce_line}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
