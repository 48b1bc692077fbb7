"""Benchmark of the block-FP8 MoE layer forward on GB300.

One step = one forward at each batch size of the decode workload with small
fine-grained experts (E=128, H=2048, I=512, top_k=8, T in {1,2,4,8,16}, down
scales padded to stride 8), on seeded synthetic inputs resident in HBM.  The
metric is the decode routed-weight HBM bandwidth: bytes of the distinct
routed experts' e4m3 weights and valid bf16 block scales, divided by the
device time of the forwards (CUDA events on the launching stream).

No forward finds its weights in L2.  Two ways to ensure it (--l2):
  rotate (default): consecutive forwards read different copies of the weight
      banks, as the layers of a model do (16 copies, 6.4 GB, far larger
      than L2); nothing else runs between forwards.
  flush: one weight bank; a 256 MiB buffer is written before every forward.
      The written lines sit dirty in L2, so the forward's reads also pay for
      their write-back to HBM.
The line reports the chosen mode as `value` and the other one beside it.
Each timed forward is a replay of a CUDA graph captured from the library
call (one graph per batch size and weight bank), as a serving loop would
run it; `value_eager` times the same forwards launched eagerly.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--l2 rotate|flush]

--impl reference times the float64 CPU oracle (the only baseline the pages
allow here) on a bounded sample of the same workload.  Under torchrun
(N > 1) every rank runs an independent replica (the layer has no exchange
step on one GPU per token batch); value = bytes of all ranks / max time.
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

DECODE_TS = [1, 2, 4, 8, 16]
SHAPE = syn.DECODE_SMALL
WORKLOAD = "decode E=128 H=2048 I=512 top_k=8 T={1,2,4,8,16} w2-scale stride 8"
METRIC = "decode routed-weight HBM GB/s"
N_LAYERS = 16   # weight-bank copies in --l2 rotate


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


def profile_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if
    the kernel source has not changed since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = open(os.path.join(ROOT, "block_fp8_mixture_route_gb300", "csrc", "decode.cu"), "rb").read()
    sha = hashlib.sha256(src).hexdigest()[:16]
    for line in open(path):
        f = line.split()
        if len(f) >= 4 and not line.startswith("#") and f[0] == kernel and f[1] == workload and f[3] == sha:
            return float(f[2])
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
        "config": {"workload": WORKLOAD, "l2": "n/a (host)"},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class Feed:
    """The inputs of forward number j and what runs before it (--l2)."""

    def __init__(self, probs, mode: str, dev):
        self.probs, self.mode, self.j = probs, mode, 0
        self.banks = None
        if mode == "rotate":
            p = probs[DECODE_TS[0]]
            bank0 = (p["w13"], p["w13_scale"], p["w2"], p["w2_scale"])
            self.banks = [bank0] + [tuple(t.clone() for t in bank0) for _ in range(N_LAYERS - 1)]
        props = torch.cuda.get_device_properties(dev)
        self.flush = torch.empty(max(256 << 20, 2 * getattr(props, "L2_cache_size", 128 << 20)),
                                 dtype=torch.uint8, device=dev) if mode == "flush" else None

    def n_banks(self) -> int:
        return N_LAYERS if self.mode == "rotate" else 1

    def problem(self, T, bank):
        if self.mode == "flush":
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
        return f"weights rotated over {N_LAYERS} copies of the banks ({N_LAYERS * bank_bytes() / 1e9:.1f} GB); no flush"


def bank_bytes() -> int:
    E, H, I = SHAPE.E, SHAPE.H, SHAPE.I
    return E * 3 * H * I


def hold_stream(s, ms: float):
    """Occupy stream s with a bounded spin kernel of about `ms` milliseconds,
    so that the host queues the launches that follow before the device
    reaches them: a forward's events then time the device work, not the
    host's launch overhead (the decode forwards are tens of microseconds)."""
    with torch.cuda.stream(s):
        torch.cuda._sleep(int(ms * 2.0e6))


def capture_forwards(feed, s, outs):
    """One CUDA graph per (T, weight bank) of the library's forward, captured
    on stream s (the library is capture-safe once its workspace is sized):
    replays launch the forward's kernels without host work in between."""
    graphs = {}
    for T in DECODE_TS:
        for bank in range(feed.n_banks()):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                api.forward_problem(feed.problem(T, bank), out=outs[T], stream=s, force_path="decode")
            graphs[(T, bank)] = g
    with torch.cuda.stream(s):
        for g in graphs.values():
            g.replay()
    s.synchronize()
    return graphs


def timed_forwards(feed, s, outs, steps, graphs=None, decode_act=None):
    """Device time of every forward of `steps` steps: {T: [ms per forward]}.
    With `graphs`, each forward is a replay of its captured graph."""
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in DECODE_TS]
          for _ in range(steps)]
    hold_stream(s, 2.0 + 0.5 * steps * len(DECODE_TS))
    with torch.cuda.stream(s):
        for k in range(steps):
            for i, T in enumerate(DECODE_TS):
                bank = feed.next_bank()
                ev[k][i][0].record(s)
                if graphs is not None:
                    graphs[(T, bank)].replay()
                else:
                    api.forward_problem(feed.problem(T, bank), out=outs[T], stream=s, force_path="decode",
                                        decode_act=decode_act)
                ev[k][i][1].record(s)
    s.synchronize()
    return {T: [ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(steps)] for i, T in enumerate(DECODE_TS)}


# ------------------------------------------------------------------ ours
def run_ours(args, world, rank, local):
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    probs = make_problems(dev)
    s = torch.cuda.Stream(device=dev)
    api.moe_fp8_block_reserve(max(DECODE_TS), SHAPE.k, SHAPE.H, SHAPE.I, SHAPE.E, stream=s)
    feed = Feed(probs, args.l2, dev)
    alt = Feed(probs, "flush" if args.l2 == "rotate" else "rotate", dev)
    outs = {T: torch.empty(T, SHAPE.H, dtype=torch.bfloat16, device=dev) for T in DECODE_TS}
    info = {T: routed_bytes(SHAPE, probs[T]["topk_ids"]) for T in DECODE_TS}
    step_bytes = sum(b for _, b in info.values())
    step_tokens = sum(DECODE_TS)

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    # warm-up
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            for T in DECODE_TS:
                api.forward_problem(feed.next(T), out=outs[T], stream=s, force_path="decode")
    s.synchronize()
    launches_per_step = 0
    for T in DECODE_TS:
        with torch.cuda.stream(s):
            api.forward_problem(feed.next(T), out=outs[T], stream=s, force_path="decode")
        launches_per_step += api.moe_fp8_block_last_launches()
    s.synchronize()

    graphs = capture_forwards(feed, s, outs) if not args.no_graph else None
    alt_graphs = capture_forwards(alt, s, outs) if not args.no_graph else None

    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    per_T = timed_forwards(feed, s, outs, args.steps, graphs)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    ck = clocks.stop()
    dev_ms = sum(sum(v) for v in per_T.values())
    value, tok_s, dev_ms_max = aggregate(step_bytes, step_tokens, args.steps, dev_ms, world)
    # the same measurement with the other way of keeping weights out of L2
    with torch.cuda.stream(s):
        for T in DECODE_TS:
            api.forward_problem(alt.next(T), out=outs[T], stream=s, force_path="decode")
    alt_T = timed_forwards(alt, s, outs, args.steps, alt_graphs)
    alt_value = step_bytes * args.steps / (sum(sum(v) for v in alt_T.values()) / 1e3) / 1e9
    # and with eager launches instead of graph replays
    eager_T = timed_forwards(feed, s, outs, args.steps)
    eager_value = step_bytes * args.steps / (sum(sum(v) for v in eager_T.values()) / 1e3) / 1e9
    # the decode path's W8A8 mode (activations quantised per token per 128
    # columns), eager launches
    with torch.cuda.stream(s):
        for T in DECODE_TS:
            api.forward_problem(feed.next(T), out=outs[T], stream=s, force_path="decode", decode_act="e4m3")
    w8a8_T = timed_forwards(feed, s, outs, args.steps, decode_act="e4m3")
    w8a8_value = step_bytes * args.steps / (sum(sum(v) for v in w8a8_T.values()) / 1e3) / 1e9

    # dominant kernel (decode GEMM1) timed with CUDA events between the stages
    st_ms = stage_durations(feed, s, args.steps)
    g1_ms = {T: st_ms[T][1] for T in DECODE_TS}
    g1_bytes = {T: info[T][0] * (2 * SHAPE.I * SHAPE.H + 2 * (2 * SHAPE.I // 128) * (SHAPE.H // 128))
                + T * SHAPE.H * 2 + T * SHAPE.k * SHAPE.I * 4 for T in DECODE_TS}
    g1_achieved = sum(g1_bytes.values()) / (sum(g1_ms.values()) / 1e3) / 1e9
    hbm, _, src = peaks()

    # end to end through the host-buffer entry point (pinned host inputs/outputs)
    e2e_v, h2d, d2h = e2e_hostio(feed, s, args.steps, args.warmup)
    prefill = prefill_leg(dev, s, max(5, args.steps)) if not args.no_prefill else None

    if rank != 0:
        return
    cpu = None
    if world == 1:
        b, secs, desc = oracle_sample(probs)
        cpu = {"value": b / secs / 1e9, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": desc}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dev_ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3xbf16->f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": feed.describe(),
                   "launch": "CUDA graph replay per forward" if graphs is not None else "eager",
                   "path": "decode (forced)", "replicas": world},
        "frac_of_hbm_peak": value / hbm, "peak_source": src,
        "value_other_l2": {"l2": alt.describe(), "value": alt_value, "frac_of_hbm_peak": alt_value / hbm},
        "value_eager": {"launch": "eager (no CUDA graph)", "value": eager_value, "frac_of_hbm_peak": eager_value / hbm},
        "value_w8a8": {"decode_act": "e4m3 (W8A8), eager", "value": w8a8_value, "frac_of_hbm_peak": w8a8_value / hbm,
                       "us": {str(T): 1e3 * statistics.median(w8a8_T[T]) for T in DECODE_TS}},
        "tok_per_s": tok_s,
        "per_T": {str(T): {"distinct_experts": info[T][0], "routed_MB": info[T][1] / 1e6,
                           "us": 1e3 * statistics.median(per_T[T]),
                           "GB_s": info[T][1] / (statistics.median(per_T[T]) / 1e3) / 1e9}
                  for T in DECODE_TS},
        "stage_us": {str(T): {n: round(1e3 * v, 2) for n, v in zip(("prep", "gemm1", "gemm2", "combine"), st_ms[T])}
                     for T in DECODE_TS},
        "roofline": {"kernel": "decode_gemm1", "bound": "hbm", "achieved": g1_achieved, "peak": hbm,
                     "unit": "GB/s", "frac": g1_achieved / hbm,
                     "traffic": profile_traffic("decode_gemm1_kernel", "decode_small_T16"),
                     "traffic_launch": "T=16 launch (ncu capture); achieved aggregates T=1..16",
                     "algorithmic_bytes_T16": g1_bytes[16],
                     "achieved_T16": g1_bytes[16] / (g1_ms[16] / 1e3) / 1e9,
                     "peak_source": f"{src} hbm_gbs (copy, burst)"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_v, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "call": "moe_fp8_block_forward_hostio through the C ABI; page-locked host inputs read and the "
                        "output written in place by the kernels"},
        "prefill": prefill,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": ck,
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)


def stage_durations(feed, s, steps):
    """Median device time of each kernel of the decode path per T, from CUDA
    events the library records between its kernels (stage-timing mode:
    moe_fp8_block_set_stage_events).  Returns {T: [prep, gemm1, gemm2, combine]} in ms."""
    import ctypes
    from block_fp8_mixture_route_gb300 import _lib
    lib = _lib.load()
    res = {}
    for T in DECODE_TS:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        for e in evs:          # torch creates the event handle on first record
            e.record(s)
        s.synchronize()
        arr = (ctypes.c_void_p * 5)(*[e.cuda_event for e in evs])
        times = []
        for _ in range(max(steps, 3)):
            hold_stream(s, 1.0)
            with torch.cuda.stream(s):
                prob = feed.next(T)
                _lib.check(lib.moe_fp8_block_set_stage_events(arr, 5), "set_stage_events")
                api.forward_problem(prob, stream=s, force_path="decode")
            s.synchronize()
            times.append([evs[i].elapsed_time(evs[i + 1]) for i in range(4)])
        res[T] = [statistics.median(t[i] for t in times) for i in range(4)]
    return res


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
    opt = api._options(None, "decode")
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
    res["fp8_peak_tflops"] = fp8_peak
    res["peak_source"] = f"2 x {src} bf16_tflops (burst)"
    return res


PROFILE_CASES = ("decode_T16", "decode_T1", "prefill_T4096", "prefill_T16384")
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
    ap.add_argument("--profile-case", choices=PROFILE_CASES, default=None,
                    help="only run 3 forwards of one case (for ncu captures); prints no bench line")
    args = ap.parse_args()
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
