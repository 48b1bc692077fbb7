"""Benchmark of the block-FP8 MoE layer forward on GB300.

One step = one decode forward at each batch size of three layers, on
seeded synthetic inputs resident in HBM:
  small          E=128 H=2048 I=512 top_k=8, T in {1,2,4,8,16}, down scales
                 padded to stride 8;
  padded_skewed  E=256 H=2560 I=640 top_k=8, T in {1,8,32}, down scales
                 padded to stride 6, router logits +2 on 16 hot experts;
  wide           E=256 H=7168 I=2048 top_k=8, T in {1,4,16,64} (11.3 GB of
                 e4m3 weights).
The metric is the decode routed-weight HBM bandwidth: bytes of the distinct
routed experts' e4m3 weights and valid bf16 block scales, divided by the
device time of the forwards (CUDA events on the launching stream).  The
headline `value` aggregates every forward of up to 16 tokens (the range the
decode target is stated for); each layer's numbers, per T, are beside it.
Each forward takes the path the library's gate chooses for it (--path auto):
the W8A16 decode kernels for the small and skewed layers, the tcgen05 W8A8
grouped GEMMs for the wide layer, whose 14 KiB activation rows leave the
decode weight ring too few stages.  `value_decode_path` is the same
aggregate with every forward forced onto the decode kernels, and --path
decode makes that the headline.

No forward finds its weights in L2.  Two ways to ensure it (--l2), for the
small and skewed layers:
  rotate (default): consecutive forwards read different copies of the weight
      banks, as the layers of a model do (16 and 8 copies, far larger than
      L2); nothing else runs between forwards.
  flush: one weight bank; a 256 MiB buffer is written before every forward.
      The written lines sit dirty in L2, so the forward's reads also pay for
      their write-back to HBM.
The wide layer keeps one bank: each of its forwards reads more than twice
the L2 capacity.  For the small layer the line also reports the other L2
mode, eager launches and the W8A8 decode option.  Each timed forward is a
replay of a CUDA graph captured from the library call (one graph per batch
size and weight bank), as a serving loop would run it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--l2 rotate|flush]

--impl reference times the float64 CPU oracle (the only baseline the pages
allow here) on a bounded sample of the small-expert workload.  Under
torchrun (N > 1) every rank runs an independent replica (the layer has no
exchange step on one GPU per token batch); value = bytes of all ranks / max
time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_fp8_mixture_route_gb300 import api, synthetic as syn  # noqa: E402

DECODE_TS = [1, 2, 4, 8, 16]   # the small-expert workload (oracle sample, end to end)
SHAPE = syn.DECODE_SMALL
WORKLOAD = ("decode, batches of up to 16 tokens of three layers: E=128 H=2048 I=512 (T=1,2,4,8,16); "
            "E=256 H=2560 I=640 skewed (T=1,8); E=256 H=7168 I=2048 (T=1,4,16); top_k=8")
METRIC = "decode routed-weight HBM GB/s"
DECODE_KERNEL = "chain"   # --decode-kernel: the chained decode kernels or the single persistent one
FORCE = None              # --path: None = the library's own gate per call; "decode" = the W8A16 decode path


def routed_bytes(shape: syn.MoeShape, ids: torch.Tensor) -> tuple[int, int]:
    """(distinct routed experts, bytes of their weights + valid block scales)."""
    E, H, I = shape.E, shape.H, shape.I
    v = ids[(ids >= 0) & (ids < E)]
    D = int(torch.unique(v).numel())
    per = 2 * I * H + H * I + 2 * ((2 * I // 128) * (H // 128)) + 2 * ((H // 128) * (I // 128))
    return D, D * per


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.dev = dev_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self):
        if not self.p:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def profile_traffic(kernel: str, workload: str = None):
    """(DRAM bytes of one launch, captured workload, its algorithmic bytes)
    of `kernel` (on `workload` if given, else its first line) from the
    committed ncu summary profiles/traffic.txt, if the source file it was
    captured from has not changed since (else None).
    Line format: kernel workload dram_bytes algorithmic_bytes source sha256[:16]."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split()
        if len(f) < 6 or line.startswith("#") or f[0] != kernel or (workload and f[1] != workload):
            continue
        src = os.path.join(ROOT, "block_fp8_mixture_route_gb300", "csrc", f[4])
        if os.path.exists(src) and hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] == f[5]:
            return float(f[2]), f[1], float(f[3])
    return None


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def allreduce_sum(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t)
    return float(t.item())


def aggregate(step_bytes: int, step_tokens: int, steps: int, dev_ms: float, world: int):
    """Whole-job numbers of the replicas: bytes and tokens summed over the
    ranks, device time the maximum over them.  Returns (GB/s, tokens/s,
    max ms)."""
    dev_ms_max = allreduce_max(dev_ms, world)
    total_bytes = allreduce_sum(step_bytes * steps, world)
    total_tokens = allreduce_sum(step_tokens * steps, world)
    return total_bytes / (dev_ms_max / 1e3) / 1e9, total_tokens / (dev_ms_max / 1e3), dev_ms_max


# ----------------------------------------------------------------- oracle
def oracle_sample(problems, budget_s: float = 12.0):
    """Time the float64 oracle (gathered mode) on whole forwards of the
    workload, smallest T first, until ~budget_s of CPU work; returns
    (routed bytes processed, seconds, description)."""
    from oracle import moe_oracle as mo
    from oracle.host_inputs import oracle_args
    done_bytes, secs, parts = 0, 0.0, []
    for T in DECODE_TS:
        prob = problems[T]
        args, _ = oracle_args(prob)
        _, nbytes = routed_bytes(SHAPE, prob["topk_ids"])
        t0 = time.perf_counter()
        mo.forward(*args, mode="gathered", act="bf16")
        dt = time.perf_counter() - t0
        done_bytes += nbytes
        secs += dt
        parts.append(f"T={T}")
        if secs > budget_s:
            break
    return done_bytes, secs, "full forwards of the workload at " + ",".join(parts)


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


def make_problems(device):
    w13, w13s, w2, w2s = syn.make_weights(SHAPE, 0, device)
    probs = {}
    for T in DECODE_TS:
        ids, w = syn.make_routing(T, SHAPE.E, SHAPE.k, 0, device, "softmax", step=T)
        probs[T] = dict(hidden=syn.make_hidden(T, SHAPE.H, 0, device, step=T), topk_ids=ids, topk_weights=w,
                        w13=w13, w13_scale=w13s, w2=w2, w2_scale=w2s)
    return probs


def run_reference(args, world, rank):
    if rank != 0:
        return
    probs = make_problems("cuda" if torch.cuda.is_available() else "cpu")
    for _ in range(args.warmup):
        oracle_sample(probs, budget_s=0.5)
    tb, ts = 0, 0.0
    desc = ""
    for _ in range(args.steps):
        b, s, desc = oracle_sample(probs, budget_s=8.0)
        tb += b
        ts += s
    v = tb / ts / 1e9
    cores = cpu_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * ts / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "decode_kernel": DECODE_KERNEL, "l2": "n/a (host)"},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class Feed:
    """The inputs of forward number j of one decode workload and what runs
    before it (--l2).  `banks` copies of the weight banks are rotated when
    one forward's weights could fit in L2; a workload whose every forward
    reads far more than L2 (the wide layer) keeps a single bank."""

    def __init__(self, wl, probs, mode: str, dev, banks: int):
        """mode: "rotate" (`banks` copies of the banks, read in turn), "flush"
        (one bank, a 256 MiB write before every forward) or "single" (one
        bank, nothing in between)."""
        self.wl, self.probs, self.mode, self.j = wl, probs, mode, 0
        self.nb = banks if mode == "rotate" else 1
        self.banks = None
        if mode == "rotate":
            p = probs[wl.ts[0]]
            bank0 = (p["w13"], p["w13_scale"], p["w2"], p["w2_scale"])
            self.banks = [bank0] + [tuple(t.clone() for t in bank0) for _ in range(self.nb - 1)]
        props = torch.cuda.get_device_properties(dev)
        self.flush = torch.empty(max(256 << 20, 2 * getattr(props, "L2_cache_size", 128 << 20)),
                                 dtype=torch.uint8, device=dev) if mode == "flush" else None

    def n_banks(self) -> int:
        return self.nb

    def problem(self, T, bank):
        if self.banks is None:
            return self.probs[T]
        w = self.banks[bank]
        return dict(self.probs[T], w13=w[0], w13_scale=w[1], w2=w[2], w2_scale=w[3])

    def next_bank(self):
        """Run the pre-forward step (flush mode) and return forward j's weight bank."""
        j, self.j = self.j, self.j + 1
        if self.mode == "flush":
            self.flush.zero_()
        return j % self.n_banks()

    def next(self, T):
        """Run the pre-forward step (flush mode) and return forward j's problem."""
        return self.problem(T, self.next_bank())

    def describe(self) -> str:
        if self.mode == "flush":
            return "flushed (256 MiB write) before every forward"
        if self.mode == "single":
            return "one weight bank; every forward reads more than twice the L2 capacity"
        return (f"weights rotated over {self.nb} copies of the banks "
                f"({self.nb * bank_bytes(self.wl.shape) / 1e9:.1f} GB); no flush")


def bank_bytes(shape) -> int:
    return shape.E * 3 * shape.H * shape.I


def hold_stream(s, ms: float):
    """Occupy stream s with a bounded spin kernel of about `ms` milliseconds,
    so that the host queues the launches that follow before the device
    reaches them: a forward's events then time the device work, not the
    host's launch overhead (the decode forwards are tens of microseconds)."""
    with torch.cuda.stream(s):
        torch.cuda._sleep(int(ms * 2.0e6))


def capture_forwards(wl, feed, s, outs, force):
    """One CUDA graph per (T, weight bank) of the library's forward, captured
    on stream s (the library is capture-safe once its workspace is sized):
    replays launch the forward's kernels without host work in between."""
    graphs = {}
    for T in wl.ts:
        for bank in range(feed.n_banks()):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                api.forward_problem(feed.problem(T, bank), out=outs[T], stream=s, force_path=force,
                                    decode_kernel=DECODE_KERNEL)
            graphs[(T, bank)] = g
    with torch.cuda.stream(s):
        for g in graphs.values():
            g.replay()
    s.synchronize()
    return graphs


def timed_forwards(wl, feed, s, outs, steps, graphs=None, decode_act=None, force=None):
    """Device time of every forward of `steps` steps: {T: [ms per forward]}.
    With `graphs`, each forward is a replay of its captured graph."""
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in wl.ts]
          for _ in range(steps)]
    hold_stream(s, 2.0 + 0.5 * steps * len(wl.ts) * wl.hold_scale)
    with torch.cuda.stream(s):
        for k in range(steps):
            for i, T in enumerate(wl.ts):
                bank = feed.next_bank()
                ev[k][i][0].record(s)
                if graphs is not None:
                    graphs[(T, bank)].replay()
                else:
                    api.forward_problem(feed.problem(T, bank), out=outs[T], stream=s, force_path=force,
                                        decode_act=decode_act, decode_kernel=DECODE_KERNEL)
                ev[k][i][1].record(s)
    s.synchronize()
    return {T: [ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(steps)] for i, T in enumerate(wl.ts)}


class Workload:
    """One decode workload: a layer shape, its token counts and routing."""

    def __init__(self, name, shape, ts, routing, banks, desc, hold_scale=1.0):
        self.name, self.shape, self.ts, self.routing, self.banks = name, shape, ts, routing, banks
        self.desc, self.hold_scale = desc, hold_scale

    def problems(self, dev):
        w13, w13s, w2, w2s = syn.make_weights(self.shape, 0, dev)
        probs = {}
        for T in self.ts:
            ids, w = syn.make_routing(T, self.shape.E, self.shape.k, 0, dev, self.routing, step=T)
            probs[T] = dict(hidden=syn.make_hidden(T, self.shape.H, 0, dev, step=T), topk_ids=ids, topk_weights=w,
                            w13=w13, w13_scale=w13s, w2=w2, w2_scale=w2s)
        return probs


# The decode workloads (small fine-grained experts, padded-scale skewed
# routing, wide experts); the headline aggregates their batches of up to 16
# tokens, the range the decode target is stated for.
WORKLOADS = [
    Workload("small", syn.DECODE_SMALL, [1, 2, 4, 8, 16], "softmax", 16,
             "E=128 H=2048 I=512 top_k=8 T={1,2,4,8,16}, w2-scale stride 8"),
    Workload("padded_skewed", syn.PADDED_SKEWED, [1, 8, 32], "hot", 8,
             "E=256 H=2560 I=640 top_k=8 T={1,8,32}, w2-scale stride 6, +2 logits on 16 hot experts"),
    Workload("wide", syn.DECODE_WIDE, [1, 4, 16, 64], "softmax", 1,
             "E=256 H=7168 I=2048 top_k=8 T={1,4,16,64}, 11.3 GB bank", hold_scale=20.0),
]
HEADLINE_T_MAX = 16


DECODE_KERNELS = ["decode_prep_kernel", "decode_gemm1_kernel", "decode_gemm2_kernel", "decode_combine_kernel"]
PREFILL_KERNELS = ["route", "act_quant_permute_kernel", "prefill_gemm_kernel<1>", "prefill_gemm_kernel<2>",
                   "prefill_combine_kernel"]


def kernel_names(path: str, n: int) -> list:
    """Names of the stage-timed kernels of one forward (the route of the
    prefill path is one stage whatever its launch count)."""
    if path == "decode":
        return DECODE_KERNELS[:n] if n == 4 else ["decode_fused_kernel"][:n]
    return PREFILL_KERNELS[:n]


def kernel_bytes(name: str, shape, T: int, D: int) -> int:
    """Algorithmic bytes of one launch: what the kernel must read and write
    at least (weights and valid scales of the D routed experts it streams,
    its activation inputs once, its outputs once)."""
    E, H, I, k = shape.E, shape.H, shape.I, shape.k
    S = T * k
    w13 = D * (2 * I * H + 2 * ((2 * I // 128) * (H // 128)))
    w2 = D * (H * I + 2 * ((H // 128) * (I // 128)))
    return {
        "decode_prep_kernel": 4 * S + 2 * T * H + 2 * T * H,
        "decode_gemm1_kernel": w13 + 2 * T * H + 4 * S * I,
        "decode_gemm2_kernel": w2 + 4 * S * I + 4 * S * H,
        "decode_combine_kernel": 4 * S * H + 2 * T * H,
        "decode_fused_kernel": w13 + w2 + 2 * T * H + 2 * T * H,
        "route": 4 * S + 4 * S,
        "act_quant_permute_kernel": 2 * T * H + S * H + 4 * S * (H // 128),
        "prefill_gemm_kernel<1>": w13 + S * H + S * I + 4 * S * ((H // 128) + (I // 128)),
        "prefill_gemm_kernel<2>": w2 + S * I + 2 * S * H + 4 * S * (I // 128),
        "prefill_combine_kernel": 2 * S * H + 2 * T * H,
    }[name]


def roofline_entry(name, nbytes, ms, n, steps, hbm, src, share):
    """The `roofline` object for the dominant kernel: its algorithmic bytes
    per launch over its average stage-timed launch duration, against the
    measured copy bandwidth; traffic = ncu DRAM bytes of one captured launch
    (committed summary) while the kernel's source is unchanged."""
    achieved = nbytes / (ms / 1e3) / 1e9
    tr = profile_traffic(name)
    return {"kernel": name, "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": tr[0] if tr else None,
            "traffic_case": ({"workload": tr[1], "algorithmic_bytes": tr[2]} if tr else None),
            "launches_timed": n, "share_of_kernel_time": share,
            "algorithmic_bytes": "per launch: the routed experts' e4m3 weights and valid bf16 scales the kernel "
                                 "streams, its activation inputs read once and its outputs written once; "
                                 "summed over one launch per timed forward (every layer and T), over their "
                                 "summed stage-timed durations",
            "peak_source": f"{src} hbm_gbs (copy, burst)"}


def algorithmic_bytes(shape, T, D) -> int:
    """Least bytes a decode forward moves: the routed experts' weights and
    valid block scales, the activations read and the output written."""
    return D * routed_per_expert(shape) + 2 * T * shape.H * 2


def routed_per_expert(shape) -> int:
    E, H, I = shape.E, shape.H, shape.I
    return 2 * I * H + H * I + 2 * ((2 * I // 128) * (H // 128)) + 2 * ((H // 128) * (I // 128))


def measure_workload(wl, dev, s, steps, warmup, l2="rotate", graphs_on=True, extras=False):
    """Time one decode workload; returns a dict of per-T results (and, with
    extras, the other L2 mode, eager launches and the W8A8 option)."""
    probs = wl.problems(dev)
    shp = wl.shape
    api.moe_fp8_block_reserve(max(wl.ts), shp.k, shp.H, shp.I, shp.E, stream=s)
    mode = "single" if wl.banks == 1 else l2
    feed = Feed(wl, probs, mode, dev, wl.banks)
    outs = {T: torch.empty(T, shp.H, dtype=torch.bfloat16, device=dev) for T in wl.ts}
    info = {T: routed_bytes(shp, probs[T]["topk_ids"]) for T in wl.ts}
    with torch.cuda.stream(s):
        for _ in range(warmup):
            for T in wl.ts:
                for force in {FORCE, "decode"}:
                    api.forward_problem(feed.next(T), out=outs[T], stream=s, force_path=force,
                                        decode_kernel=DECODE_KERNEL)
    s.synchronize()
    launches, paths = {}, {}
    for T in wl.ts:
        with torch.cuda.stream(s):
            api.forward_problem(feed.next(T), out=outs[T], stream=s, force_path=FORCE, decode_kernel=DECODE_KERNEL)
        launches[T] = api.moe_fp8_block_last_launches()
        paths[T] = "decode" if api.moe_fp8_block_last_path() == 1 else "prefill"
    s.synchronize()
    graphs = capture_forwards(wl, feed, s, outs, FORCE) if graphs_on else None
    # the headline's timed forwards, marked for an ncu launch list restricted
    # to them (ncu --nvtx --nvtx-include "headline/")
    torch.cuda.nvtx.range_push("headline")
    per_T = timed_forwards(wl, feed, s, outs, steps, graphs, force=FORCE)
    torch.cuda.nvtx.range_pop()
    kern = kernel_durations(wl, feed, s, max(3, steps // 2))
    # where the library's gate takes the prefill path, the forced decode path too
    per_T_decode = {T: per_T[T] for T in wl.ts if paths[T] == "decode"}
    other = [T for T in wl.ts if paths[T] != "decode"]
    if other:
        sub_wl = Workload(wl.name, wl.shape, other, wl.routing, wl.banks, wl.desc, wl.hold_scale)
        dgraphs = capture_forwards(sub_wl, feed, s, outs, "decode") if graphs_on else None
        per_T_decode.update(timed_forwards(sub_wl, feed, s, outs, steps, dgraphs, force="decode"))
        del dgraphs
    res = {"workload": wl.desc, "l2": feed.describe(), "per_T": per_T, "info": info, "kern": kern,
           "launches": launches, "paths": paths, "per_T_decode": per_T_decode}
    if extras:
        alt = Feed(wl, probs, "flush" if mode == "rotate" else "rotate", dev, wl.banks)
        alt_graphs = capture_forwards(wl, alt, s, outs, FORCE) if graphs_on else None
        alt_T = timed_forwards(wl, alt, s, outs, steps, alt_graphs, force=FORCE)
        res["alt"] = (alt.describe(), alt_T)
        res["eager"] = timed_forwards(wl, feed, s, outs, steps, force=FORCE)
        with torch.cuda.stream(s):
            for T in wl.ts:
                api.forward_problem(feed.next(T), out=outs[T], stream=s, force_path="decode", decode_act="e4m3",
                                    decode_kernel=DECODE_KERNEL)
        res["w8a8"] = timed_forwards(wl, feed, s, outs, steps, decode_act="e4m3", force="decode")
        res["feed"] = feed
    else:
        del feed, probs, graphs
        torch.cuda.empty_cache()
    return res


def kernel_durations(wl, feed, s, reps):
    """Median device time of each kernel of a decode forward per T, from CUDA
    events the library records around its kernels (stage-timing mode:
    moe_fp8_block_set_stage_events).  Returns {T: [ms per kernel]}."""
    import ctypes
    from block_fp8_mixture_route_gb300 import _lib
    lib = _lib.load()
    res = {}
    for T in wl.ts:
        with torch.cuda.stream(s):
            api.forward_problem(feed.next(T), stream=s, force_path=FORCE, decode_kernel=DECODE_KERNEL)
        n = api.moe_fp8_block_last_launches()
        if api.moe_fp8_block_last_path() == 2:
            n = len(PREFILL_KERNELS)   # the route is one stage whatever its launch count
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        for e in evs:          # torch creates the event handle on first record
            e.record(s)
        s.synchronize()
        arr = (ctypes.c_void_p * (n + 1))(*[e.cuda_event for e in evs])
        times = []
        for _ in range(reps):
            hold_stream(s, 1.0 * wl.hold_scale)
            with torch.cuda.stream(s):
                prob = feed.next(T)
                _lib.check(lib.moe_fp8_block_set_stage_events(arr, n + 1), "set_stage_events")
                api.forward_problem(prob, stream=s, force_path=FORCE, decode_kernel=DECODE_KERNEL)
            s.synchronize()
            times.append([evs[i].elapsed_time(evs[i + 1]) for i in range(n)])
        res[T] = [statistics.median(t[i] for t in times) for i in range(n)]
    return res


# ------------------------------------------------------------------ ours
def run_ours(args, world, rank, local):
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    s = torch.cuda.Stream(device=dev)
    hbm, _, src = peaks()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    results = {}
    for wl in WORKLOADS:
        results[wl.name] = measure_workload(wl, dev, s, args.steps, args.warmup, l2=args.l2,
                                            graphs_on=not args.no_graph, extras=(wl.name == "small"))
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    ck = clocks.stop()

    # headline: all decode-size forwards (up to 16 tokens), each on the path
    # the library's gate takes (or the forced one)
    step_bytes = step_tokens = 0
    dev_ms = dec_ms = 0.0
    kern_tot = {}   # kernel name -> [algorithmic bytes, summed median ms, launches per step]
    gpu_launches = 0
    per_wl = {}
    for wl in WORKLOADS:
        r = results[wl.name]
        rows = {}
        for T in wl.ts:
            D, nbytes = r["info"][T]
            med = statistics.median(r["per_T"][T])
            path = r["paths"][T]
            names = kernel_names(path, len(r["kern"][T]))
            rows[str(T)] = {"distinct_experts": D, "routed_MB": nbytes / 1e6, "path": path, "us": 1e3 * med,
                            "GB_s": nbytes / (med / 1e3) / 1e9, "frac_of_hbm_peak": nbytes / (med / 1e3) / 1e9 / hbm,
                            "kernels_us": {n: round(1e3 * x, 2) for n, x in zip(names, r["kern"][T])},
                            "launches": r["launches"][T]}
            dmed = statistics.median(r["per_T_decode"][T])
            if path != "decode":
                rows[str(T)]["decode_path_us"] = 1e3 * dmed
                rows[str(T)]["decode_path_GB_s"] = nbytes / (dmed / 1e3) / 1e9
            # the roofline's kernel totals cover every timed forward (as an ncu
            # launch list of the timed region does); the headline T <= 16
            for n, x in zip(names, r["kern"][T]):
                kt = kern_tot.setdefault(n, [0, 0.0, 0])
                kt[0] += kernel_bytes(n, wl.shape, T, D)
                kt[1] += x
                kt[2] += 1
            gpu_launches += r["launches"][T] * args.steps
            if T <= HEADLINE_T_MAX:
                step_bytes += nbytes
                step_tokens += T
                dev_ms += sum(r["per_T"][T])
                dec_ms += sum(r["per_T_decode"][T])
        head = [T for T in wl.ts if T <= HEADLINE_T_MAX]
        wb = sum(r["info"][T][1] for T in head)
        wms = sum(statistics.median(r["per_T"][T]) for T in head)
        per_wl[wl.name] = {"workload": wl.desc, "l2": r["l2"], "GB_s_T_le_16": wb / (wms / 1e3) / 1e9,
                           "frac_of_hbm_peak_T_le_16": wb / (wms / 1e3) / 1e9 / hbm, "per_T": rows}
    value, tok_s, dev_ms_max = aggregate(step_bytes, step_tokens, args.steps, dev_ms, world)
    dec_value, _, _ = aggregate(step_bytes, step_tokens, args.steps, dec_ms, world)
    # the dominant kernel: most summed device time over the timed forwards
    dom = max(kern_tot, key=lambda n: kern_tot[n][1])
    dom_bytes, dom_ms, dom_n = kern_tot[dom]
    dom_achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    kern_all_ms = sum(v[1] for v in kern_tot.values())

    small = results["small"]
    sb = sum(small["info"][T][1] for T in WORKLOADS[0].ts)
    alt_desc, alt_T = small["alt"]
    alt_value = sb * args.steps / (sum(sum(v) for v in alt_T.values()) / 1e3) / 1e9
    eager_value = sb * args.steps / (sum(sum(v) for v in small["eager"].values()) / 1e3) / 1e9
    w8a8_value = sb * args.steps / (sum(sum(v) for v in small["w8a8"].values()) / 1e3) / 1e9

    # end to end through the host-buffer entry point (pinned host inputs/outputs), small experts
    e2e_v, h2d, d2h = e2e_hostio(small["feed"], s, args.steps, args.warmup)
    small.pop("feed")
    torch.cuda.empty_cache()
    prefill = prefill_leg(dev, s, max(5, args.steps)) if not args.no_prefill and world == 1 else None
    host_exp = host_experts_leg(dev, s, 5) if not args.no_prefill and world == 1 else None

    if rank != 0:
        return
    cpu = None
    if world == 1:
        probs = make_problems(dev)
        b, secs, desc = oracle_sample(probs)
        cpu = {"value": b / secs / 1e9, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": desc}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dev_ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3xbf16->f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "decode_kernel": DECODE_KERNEL,
                   "l2": {n: v["l2"] for n, v in per_wl.items()},
                   "launch": "CUDA graph replay per forward" if not args.no_graph else "eager",
                   "path": "decode (forced)" if FORCE == "decode" else
                   "the library's gate per call (W8A16 decode kernels, or the tcgen05 W8A8 grouped GEMMs)",
                   "replicas": world},
        "frac_of_hbm_peak": value / hbm, "peak_source": src,
        "value_decode_path": {"path": "the W8A16 decode kernels for every forward (forced)", "value": dec_value,
                              "frac_of_hbm_peak": dec_value / hbm},
        "tok_per_s": tok_s,
        "workloads": per_wl,
        "value_small_other_l2": {"l2": alt_desc, "value": alt_value, "frac_of_hbm_peak": alt_value / hbm},
        "value_small_eager": {"launch": "eager (no CUDA graph)", "value": eager_value,
                              "frac_of_hbm_peak": eager_value / hbm},
        "value_small_w8a8": {"decode_act": "e4m3 (W8A8), eager", "value": w8a8_value,
                             "frac_of_hbm_peak": w8a8_value / hbm,
                             "us": {str(T): 1e3 * statistics.median(small["w8a8"][T]) for T in WORKLOADS[0].ts}},
        "roofline": roofline_entry(dom, dom_bytes, dom_ms, dom_n, args.steps, hbm, src,
                                   share=dom_ms / kern_all_ms),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_v, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "call": "moe_fp8_block_forward_hostio through the C ABI on the small-expert workload; page-locked "
                        "host inputs read and the output written in place by the kernels"},
        "prefill": prefill,
        "host_experts": host_exp,
        "gpu_launches": gpu_launches,
        "clocks": ck,
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)


def e2e_hostio(feed, s, steps, warmup):
    """End to end through the C ABI with HOST buffers: each forward reads its
    page-locked inputs and writes its output across the host link inside the
    timed region.  Descriptors are built once per buffer, as a C caller
    would, so the time is the library's and not the Python binding's."""
    import ctypes
    from block_fp8_mixture_route_gb300 import _lib
    lib = _lib.load()
    P = ctypes.byref
    probs = feed.probs
    host = {T: (probs[T]["hidden"].cpu().pin_memory(), probs[T]["topk_ids"].cpu().pin_memory(),
                probs[T]["topk_weights"].cpu().pin_memory(),
                torch.empty(T, SHAPE.H, dtype=torch.bfloat16).pin_memory()) for T in DECODE_TS}
    hdesc = {T: [api.desc(x) for x in host[T]] for T in DECODE_TS}
    wdesc = {}
    opt = api._options(None, "decode", decode_kernel=DECODE_KERNEL)
    sp = ctypes.c_void_p(s.cuda_stream)
    total_b, total_s = 0, 0.0
    h2d = sum(T * SHAPE.H * 2 + T * SHAPE.k * 8 for T in DECODE_TS)
    d2h = sum(T * SHAPE.H * 2 for T in DECODE_TS)
    for k in range(warmup + steps):
        for T in DECODE_TS:
            dx, di, dw, do = hdesc[T]
            with torch.cuda.stream(s):
                w = feed.next(T)
            key = w["w13"].data_ptr()
            if key not in wdesc:
                wdesc[key] = ([api.desc(w[n]) for n in ("w13", "w13_scale", "w2", "w2_scale")],
                              w["w13_scale"].stride(1), w["w2_scale"].stride(1))
            (d13, d13s, d2, d2s), s13, s2 = wdesc[key]
            s.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            rc = lib.moe_fp8_block_forward_hostio(P(dx), P(di), P(dw), P(d13), P(d13s), s13, P(d2), P(d2s), s2,
                                                  P(do), sp, P(opt))
            e1.record(s)
            s.synchronize()
            _lib.check(rc, "moe_fp8_block_forward_hostio")
            if k >= warmup:
                total_s += e0.elapsed_time(e1) / 1e3
                total_b += routed_bytes(SHAPE, probs[T]["topk_ids"])[1]
    return total_b / total_s / 1e9, h2d, d2h


PREFILL_CASES = [(1024, "softmax"), (4096, "softmax"), (4096, "zipf"), (16384, "softmax"), (16384, "zipf")]
HOST_EXPERT_TS = [1, 4, 16]


def host_experts_leg(dev, s, reps):
    """The small-expert layer with its expert banks in page-locked host
    memory (moe_fp8_block_forward_host_experts): routed-weight GB/s per T,
    against the host link's read rate measured here as a 1 GiB page-locked
    host-to-device copy."""
    shp = syn.DECODE_SMALL
    dw = syn.make_weights(shp, 0, dev)
    hw = []
    for t in dw:
        h = torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        hw.append(h)
    del dw
    torch.cuda.empty_cache()
    src = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    link = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            dst.copy_(src, non_blocking=True)
            e1.record(s)
        s.synchronize()
        link.append(src.numel() / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del src, dst
    link_gbs = max(link)
    rows, tb, tms = {}, 0, 0.0
    for T in HOST_EXPERT_TS:
        ids, w = syn.make_routing(T, shp.E, shp.k, 0, dev, "softmax", step=T)
        x = syn.make_hidden(T, shp.H, 0, dev, step=T)
        out = torch.empty(T, shp.H, dtype=torch.bfloat16, device=dev)
        D, nbytes = routed_bytes(shp, ids)
        times = []
        for r in range(reps + 2):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                e0.record(s)
                api.moe_fp8_block_forward_host_experts(x, ids, w, hw[0], hw[1], hw[1].stride(1), hw[2], hw[3],
                                                       hw[3].stride(1), out=out, stream=s)
                e1.record(s)
            s.synchronize()
            if r >= 2:
                times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        rows[str(T)] = {"distinct_experts": D, "us": 1e3 * ms, "GB_s": nbytes / (ms / 1e3) / 1e9}
        tb += nbytes
        tms += ms
    value = tb / (tms / 1e3) / 1e9
    return {"layer": "E=128 H=2048 I=512 top_k=8, expert banks in page-locked host memory", "value": value,
            "unit": "GB/s", "link_GB_s": link_gbs, "frac_of_link": value / link_gbs,
            "link": "1 GiB page-locked host-to-device copy, best of 3", "per_T": rows}


def prefill_leg(dev, s, reps):
    """Prefill grouped GEMM workload (E=128, H=2048, I=512, top_k=8): FP8
    TFLOPS = 6*T*k*H*I / forward time, per-kernel times from stage events."""
    import ctypes
    from block_fp8_mixture_route_gb300 import _lib
    lib = _lib.load()
    shp = syn.PREFILL
    w13, w13s, w2, w2s = syn.make_weights(shp, 0, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # prefill reads are compute-bound
    hbm_peak, bf16_peak, src = peaks()
    fp8_peak = 2.0 * bf16_peak
    # the least bytes a prefill forward moves: every expert's weights and valid
    # block scales (all are routed at these sizes), x in and out
    per_expert = (2 * shp.I * shp.H + shp.H * shp.I + 2 * ((2 * shp.I // 128) * (shp.H // 128))
                  + 2 * ((shp.H // 128) * (shp.I // 128)))
    res = {}
    for T, routing in PREFILL_CASES:
        ids, w = syn.make_routing(T, shp.E, shp.k, 0, dev, routing, step=T)
        prob = dict(hidden=syn.make_hidden(T, shp.H, 0, dev, step=T), topk_ids=ids, topk_weights=w, w13=w13,
                    w13_scale=w13s, w2=w2, w2_scale=w2s)
        out = torch.empty(T, shp.H, dtype=torch.bfloat16, device=dev)
        flops = 6.0 * T * shp.k * shp.H * shp.I
        with torch.cuda.stream(s):
            for _ in range(3):
                api.forward_problem(prob, out=out, stream=s, force_path="prefill")
        s.synchronize()
        times = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                flush.zero_()
                e0.record(s)
                api.forward_problem(prob, out=out, stream=s, force_path="prefill")
                e1.record(s)
            s.synchronize()
            times.append(e0.elapsed_time(e1))
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        for e in evs:
            e.record(s)
        s.synchronize()
        arr = (ctypes.c_void_p * 6)(*[e.cuda_event for e in evs])
        st = []
        for _ in range(max(3, reps // 2)):
            with torch.cuda.stream(s):
                flush.zero_()
                _lib.check(lib.moe_fp8_block_set_stage_events(arr, 6), "set_stage_events")
                api.forward_problem(prob, out=out, stream=s, force_path="prefill")
            s.synchronize()
            st.append([evs[i].elapsed_time(evs[i + 1]) for i in range(5)])
        stage = [statistics.median(x[i] for x in st) for i in range(5)]
        ms = statistics.median(times)
        g1f, g2f = 4.0 * T * shp.k * shp.H * shp.I, 2.0 * T * shp.k * shp.H * shp.I
        min_bytes = shp.E * per_expert + 2 * 2 * T * shp.H
        bound_s = max(flops / (fp8_peak * 1e12), min_bytes / (hbm_peak * 1e9))
        res[f"T{T}_{routing}"] = {
            "us": 1e3 * ms, "tflops": flops / (ms / 1e3) / 1e12, "frac_of_fp8_peak": flops / (ms / 1e3) / 1e12 / fp8_peak,
            "frac_of_roofline": bound_s / (ms / 1e3),
            "roofline_bound": "tensor" if flops / (fp8_peak * 1e12) >= min_bytes / (hbm_peak * 1e9) else "hbm",
            "stage_us": {n: round(1e3 * v, 2) for n, v in
                         zip(("route", "act_quant_permute", "gemm1", "gemm2", "combine"), stage)},
            "gemm1_tflops": g1f / (stage[2] / 1e3) / 1e12, "gemm2_tflops": g2f / (stage[3] / 1e3) / 1e12,
        }
        if (T, routing) == (4096, "softmax"):
            # DRAM bytes of one launch of each GEMM from the committed ncu
            # capture of this case, beside the launch's algorithmic bytes
            # (null once the kernel source has changed since the capture)
            tr = {}
            for name, key in (("prefill_gemm_kernel<1>", "gemm1"), ("prefill_gemm_kernel<2>", "gemm2")):
                t = profile_traffic(name, "prefill_T4096")
                alg = kernel_bytes(name, shp, T, shp.E)
                tr[key] = {"dram_bytes": t[0] if t else None, "algorithmic_bytes": alg,
                           "ratio": t[0] / alg if t else None}
            res[f"T{T}_{routing}"]["traffic"] = tr
    res["fp8_peak_tflops"] = fp8_peak
    res["peak_source"] = f"2 x {src} bf16_tflops (burst)"
    return res


PROFILE_CASES = ("decode_T16", "decode_T1", "prefill_T4096", "prefill_T16384", "wide_T16", "wide_T1", "wide32_T4")
# gate sweeps: layer -> token counts.  wide: T = round(32 r), r = T*k/E = 0.1 .. 1.0;
# small: r = T*k/E = 0.0625 .. 1.0
SWEEPS = {
    "wide": (syn.DECODE_WIDE, (1, 3, 6, 10, 13, 16, 19, 22, 26, 29, 32)),
    "small": (syn.DECODE_SMALL, (1, 2, 3, 4, 6, 8, 10, 12, 16)),
}


def gate_sweep(which: str = "wide", reps: int = 5):
    """Decode against prefill for r = T*k/E up to 1.0 on the wide-expert
    layer (E=256, H=7168, I=2048, top_k=8, about 11 GB of e4m3 weights) or
    the small-expert one (E=128, H=2048, I=512): median forward time of each
    path after an L2 flush.  Prints one JSON object (not a bench line): the
    data behind the default gate."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    shp, sweep_ts = SWEEPS[which]
    w13, w13s, w2, w2s = syn.make_weights(shp, 0, dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)
    rows = []
    for T in sweep_ts:
        ids, w = syn.make_routing(T, shp.E, shp.k, 0, dev, "softmax", step=T)
        prob = dict(hidden=syn.make_hidden(T, shp.H, 0, dev, step=T), topk_ids=ids, topk_weights=w, w13=w13,
                    w13_scale=w13s, w2=w2, w2_scale=w2s)
        out = torch.empty(T, shp.H, dtype=torch.bfloat16, device=dev)
        D, nbytes = routed_bytes(shp, ids)
        row = {"T": T, "r": T * shp.k / shp.E, "distinct_experts": D, "routed_GB": nbytes / 1e9}
        for path in ("decode", "prefill"):
            with torch.cuda.stream(s):
                for _ in range(2):
                    api.forward_problem(prob, out=out, stream=s, force_path=path)
            s.synchronize()
            times = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(s):
                    flush.zero_()
                    e0.record(s)
                    api.forward_problem(prob, out=out, stream=s, force_path=path)
                    e1.record(s)
                s.synchronize()
                times.append(e0.elapsed_time(e1))
            ms = statistics.median(times)
            row[f"{path}_us"] = 1e3 * ms
            row[f"{path}_GB_s"] = nbytes / (ms / 1e3) / 1e9
        row["faster"] = "decode" if row["decode_us"] <= row["prefill_us"] else "prefill"
        rows.append(row)
    cross = next((r["r"] for r in rows if r["faster"] == "prefill"), None)
    print(json.dumps({"gate_sweep": rows,
                      "workload": f"E={shp.E} H={shp.H} I={shp.I} top_k={shp.k}, softmax routing",
                      "default_gate": "decode while T*k <= E and the decode gate/up ring has >= 4 stages",
                      "first_r_where_prefill_is_faster": cross}), flush=True)


def profile_case(name: str, reps: int = 3):
    """Run `reps` forwards of one case and nothing else (no timing, no
    oracle): the command an ncu capture of a single kernel wraps."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    s = torch.cuda.Stream(device=dev)
    if name.startswith("decode"):
        T = int(name.split("_T")[1])
        prob = make_problems(dev)[T]
        path, H = "decode", SHAPE.H
    elif name.startswith("wide"):
        # the wide layer at a decode batch size, on the path the library's gate
        # takes; wide32: the same expert shape with 32 experts (1.4 GB of
        # weights, a case small enough for a full ncu capture)
        T = int(name.split("_T")[1])
        shp = syn.DECODE_WIDE if name.startswith("wide_") else syn.MoeShape(E=32, H=7168, I=2048, k=8)
        w13, w13s, w2, w2s = syn.make_weights(shp, 0, dev)
        ids, w = syn.make_routing(T, shp.E, shp.k, 0, dev, "softmax", step=T)
        prob = dict(hidden=syn.make_hidden(T, shp.H, 0, dev, step=T), topk_ids=ids, topk_weights=w, w13=w13,
                    w13_scale=w13s, w2=w2, w2_scale=w2s)
        path, H = None, shp.H
    else:
        T = int(name.split("_T")[1])
        shp = syn.PREFILL
        w13, w13s, w2, w2s = syn.make_weights(shp, 0, dev)
        ids, w = syn.make_routing(T, shp.E, shp.k, 0, dev, "softmax", step=T)
        prob = dict(hidden=syn.make_hidden(T, shp.H, 0, dev, step=T), topk_ids=ids, topk_weights=w, w13=w13,
                    w13_scale=w13s, w2=w2, w2_scale=w2s)
        path, H = "prefill", shp.H
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    with torch.cuda.stream(s):
        for _ in range(reps):
            api.forward_problem(prob, out=out, stream=s, force_path=path)
    s.synchronize()
    print(json.dumps({"profile_case": name, "reps": reps, "launches_per_forward": api.moe_fp8_block_last_launches()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill leg")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of CUDA-graph replays of each forward")
    ap.add_argument("--l2", choices=("rotate", "flush"), default="rotate",
                    help="how forwards are kept from finding their weights in L2 (see the module docstring)")
    ap.add_argument("--gate-sweep", choices=tuple(SWEEPS), default=None,
                    help="time decode against prefill for r = T*k/E up to 1.0 on one layer (one JSON object)")
    ap.add_argument("--path", choices=("auto", "decode"), default="auto",
                    help="auto (default): each forward takes the path the library's gate chooses; decode: force "
                         "the W8A16 decode kernels")
    ap.add_argument("--decode-kernel", choices=("chain", "fused"), default="chain",
                    help="decode kernels: four chained launches (default) or one persistent launch")
    ap.add_argument("--profile-case", choices=PROFILE_CASES, default=None,
                    help="only run 3 forwards of one case (for ncu captures); prints no bench line")
    args = ap.parse_args()
    global DECODE_KERNEL, FORCE
    DECODE_KERNEL = args.decode_kernel
    FORCE = None if args.path == "auto" else "decode"
    if args.profile_case:
        profile_case(args.profile_case)
        return
    if args.gate_sweep:
        gate_sweep(args.gate_sweep)
        return
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
