"""Benchmark of the GB300 MoE router: effective HBM GB/s of the top-K router
forward/backward and the aux-score forward/backward at 8192 tokens.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

One step is one pass of the router's hot path over one batch of synthetic
tokens: top-K forward, aux-score forward, top-K backward, aux-score backward
(softmax, fp32 logits, 8192 tokens x 2304 experts, K = 36).  The timed steps
run back to back, with no flush, over N rotating buffer sets (inputs and
outputs) whose bytes per kernel launch together exceed 3x L2, so that every
kernel reads its inputs from HBM and pays the write-back of whatever its
predecessors left dirty in L2.  value = algorithmic bytes of the K steps / the
time between CUDA events around them; the per-kernel events inside the region
give the roofline.  The same kernels timed one at a time with L2 flushed
before each launch are reported under "isolated".

Algorithmic bytes per token row of E experts (d = bytes per logit):
  top-K fwd  E (d + d + 1 + 4)   logits in; probs, map, scores out (+ bias 4E once)
  top-K bwd  E (d + 1 + 4 + d)   grad_probs, map, scores in; grad_logits out
  aux fwd    softmax E (d + 4 + 1); sigmoid E (d + 4 + 1 + 4)
  aux bwd    E (4 + 4 + d)       grad_scores, saved scores in; grad_logits out

Under torchrun (N > 1) every rank routes its own 8192-token batch (token rows
are independent: no collective on the data path), the timed region is
bracketed by barriers, the times are the max over ranks and value is the
bytes of all ranks over that time ("weak" scaling).

--impl reference times the CPU oracle (float64 numpy, one row at a time, the
test suite's reference) on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "t8192_e2304_k36"
METRIC = "effective HBM GB/s of router top-k fwd/bwd vs GB300 peak, 8192 tokens"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ---------------------------------------------------------------------------
# byte accounting
# ---------------------------------------------------------------------------
def bytes_per_launch(op: str, T: int, E: int, d: int, sf: str = "softmax",
                     bias: bool = False) -> int:
    if op == "topk_fwd":
        return T * E * (2 * d + 5) + (4 * E if bias else 0)
    if op == "topk_bwd":
        return T * E * (2 * d + 5)
    if op == "aux_fwd":
        return T * E * (d + 5 + (4 if sf == "sigmoid" else 0))
    if op == "aux_bwd":
        return T * E * (8 + d)
    raise ValueError(op)


def next_row_bytes(op: str, T: int, E: int, K: int, d: int) -> int:
    """Algorithmic bytes of the compact, maps and aux-loss launches."""
    if op == "compact_fwd":      # logits in; weights, indices, expanded rows out
        return T * E * d + T * K * 12
    if op == "expert_maps":      # indices in; offsets and three [T K] maps out
        return T * K * 4 + (E + 1) * 4 + 3 * T * K * 4
    if op == "aux_loss_fwd":     # aux scores and map in; tokens and the loss out
        return T * E * 5 + E * 4 + 4
    if op == "aux_loss_bwd":     # tokens and grad in; grad [T, E] out
        return T * E * 4 + E * 4 + 4
    raise ValueError(op)


def _strip_comments(src: str) -> str:
    """C/C++/CUDA source without comments and whitespace (string literals
    kept), so that the hash below moves only when code changes."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return "".join(out)


def kernel_source_hash() -> str:
    """Hash of the code of the CUDA sources and the public header they include
    (comments and whitespace ignored)."""
    h = hashlib.sha256()
    for sub in (os.path.join("score_top_expert_gb300", "csrc"), "include"):
        d = os.path.join(ROOT, sub)
        if not os.path.isdir(d):
            continue
        for name in sorted(os.listdir(d)):
            with open(os.path.join(d, name), encoding="utf-8") as f:
                h.update(name.encode() + _strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def hbm_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernels changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("kernel_source_hash") != kernel_source_hash():
        return None
    e = t.get("kernels", {}).get(f"{kernel}@{workload}")
    return None if e is None else int(e["dram_bytes_per_launch"])


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self) -> dict:
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                rows.append(dict(sm=float(f[0]), max=float(f[1]), power=float(f[2]),
                                 hw=f[4], hwt=f[5], swt=f[6], swp=f[7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "samples": 0}
        load = [r for r in rows if r["power"] > 0.25 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in load:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                            ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(load), "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class Step:
    """Inputs and outputs of one router step on the device."""

    def __init__(self, R, torch, case, args, dev, sf="softmax", packed=False):
        """packed: the inputs (logits, grad_probs, grad_scores) are views into
        one device buffer (in_buf) and the outputs into another (out_buf), so
        that a host round trip takes one copy each way."""
        self.R, self.torch = R, torch
        T, E = case.logits.shape
        dt = torch.float32 if case.dtype == "f32" else torch.bfloat16
        self.dt = dt
        self.K, self.sf = args["K"], sf
        self.c, self.ng, self.gk = args["scaling_factor"], args["num_groups"], args["group_topk"]
        f32, b8 = torch.float32, torch.bool
        ins = [("x", dt), ("g", dt), ("gs", f32)]
        outs = [("probs", dt), ("rmap", b8), ("scores", f32), ("gx", dt), ("q", f32),
                ("amap", b8), ("agx", dt)] + ([("inter", f32)] if sf == "sigmoid" else [])
        if packed:
            self.in_buf, views = _carve(torch, dev, (T, E), ins)
            for (n, _), v in zip(ins, views):
                setattr(self, n, v)
            self.out_buf, views = _carve(torch, dev, (T, E), outs)
            for (n, _), v in zip(outs, views):
                setattr(self, n, v)
            self.x.copy_(torch.from_numpy(case.logits).to(dt))
            self.g.copy_(torch.from_numpy(case.grad_probs).to(dt))
            self.gs.copy_(torch.from_numpy(case.grad_scores))
        else:
            self.x = torch.from_numpy(case.logits).to(dev).to(dt)
            self.g = torch.from_numpy(case.grad_probs).to(dev).to(dt)
            self.gs = torch.from_numpy(case.grad_scores).to(dev)
            for n, t in outs:
                setattr(self, n, torch.empty(T, E, dtype=t, device=dev))
        if sf != "sigmoid":
            self.inter = None
        self.bias = None if case.expert_bias is None else torch.from_numpy(case.expert_bias).to(dev)
        self.T, self.E, self.d = T, E, (4 if dt == torch.float32 else 2)

    def ops(self):
        R = self
        return [
            ("topk_fwd", lambda: R.R.router_topk_fwd(
                R.x, R.K, R.sf, R.ng, R.gk, R.c, R.bias, probs=R.probs, routing_map=R.rmap,
                scores=R.scores)),
            ("aux_fwd", lambda: R.R.router_aux_scores_fwd(
                R.x, R.K, R.sf, scores=R.q, routing_map=R.amap, intermediate=R.inter)),
            ("topk_bwd", lambda: R.R.router_topk_bwd(
                R.g, R.rmap, R.scores, R.K, R.sf, R.c, grad_logits=R.gx)),
            ("aux_bwd", lambda: R.R.router_aux_scores_bwd(
                R.gs, R.inter if R.inter is not None else R.q, R.K, R.sf, R.dt,
                grad_logits=R.agx)),
        ]

    def bytes(self, op):
        return bytes_per_launch(op, self.T, self.E, self.d, self.sf, self.bias is not None)


def _carve(torch, dev, shape, specs):
    """One uint8 device buffer holding a [shape] tensor of each dtype in
    ``specs`` back to back (each at a 256-byte boundary); returns the buffer
    and the tensor views."""
    n = shape[0] * shape[1]
    sizes = [n * torch.empty(0, dtype=t).element_size() for _, t in specs]
    offs, off = [], 0
    for b in sizes:
        offs.append(off)
        off += (b + 255) // 256 * 256
    buf = torch.empty(off, dtype=torch.uint8, device=dev)
    views = [buf[o:o + b].view(t).view(shape) for o, b, (_, t) in zip(offs, sizes, specs)]
    return buf, views


class L2Flush:
    """Evict L2 with clean lines: write one buffer larger than L2, then read
    another one of the same size (the write-backs of the first happen during
    the read, not during the next timed kernel)."""

    def __init__(self, torch, dev):
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n = max(2 * l2, 256 << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.zeros(n // 4096, 4096, dtype=torch.float32, device=dev)
        self.acc = torch.empty(4096, dtype=torch.float32, device=dev)
        self.torch = torch
        self.mib = n * 4 >> 20

    def zero_(self):
        self.w.zero_()
        self.torch.sum(self.r, dim=0, out=self.acc)


def time_ops(torch, stream, flush, ops, reps, warmup):
    """Per-op device times (ms) over ``reps`` passes, L2 flushed before each op."""
    for _ in range(warmup):
        for _, fn in ops:
            flush.zero_()
            fn()
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in ops] for _ in range(reps)]
    torch.cuda._sleep(2_000_000)  # let the host run ahead of the GPU
    for r in range(reps):
        for i, (_, fn) in enumerate(ops):
            flush.zero_()
            ev[r][i][0].record(stream)
            fn()
            ev[r][i][1].record(stream)
    torch.cuda.synchronize()
    return [[ev[r][i][0].elapsed_time(ev[r][i][1]) for r in range(reps)]
            for i in range(len(ops))]


def rotating_sets(R, torch, case, args, dev, sf, l2, make=None):
    """Buffer sets (Step objects) for back-to-back timing: enough that the
    bytes of one kernel launch over all sets exceed 3x L2, so a launch never
    finds its inputs in L2 from the previous use of its set."""
    make = make or (lambda: Step(R, torch, case, args, dev, sf))
    first = make()
    per_launch = min(first.bytes(n) for n, _ in first.ops())
    nsets = max(2, -(-3 * l2 // per_launch))
    return [first] + [make() for _ in range(nsets - 1)]


def graph_us(torch, stream, fns, reps_per_fn=3, replays=10):
    """Device µs per launch: a CUDA graph of the launches ``fns`` repeated
    ``reps_per_fn`` times back to back, median over ``replays`` replays."""
    g = torch.cuda.CUDAGraph()
    for fn in fns:
        fn()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        for fn in fns * reps_per_fn:
            fn()
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(replays):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    del g
    return statistics.median(times) / (len(fns) * reps_per_fn)


def gpu_arm(a, world, rank, local):
    import torch

    import score_top_expert_gb300.router as R
    from score_top_expert_gb300 import build
    from score_top_expert_gb300.workloads import make_workload

    build.build()
    R.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    peak, peak_kind = hbm_peak()

    case, args = make_workload(WORKLOAD)
    sets = rotating_sets(R, torch, case, args, dev, "softmax", l2)
    nsets = len(sets)
    step = sets[0]
    set_ops = [st.ops() for st in sets]
    names = [n for n, _ in set_ops[0]]
    step_bytes = sum(step.bytes(n) for n in names)

    # ---- the timed region: K steps back to back over the rotating sets -------
    # W eager warm-up steps, then one CUDA graph of exactly K steps (step r on
    # set r mod N), replayed untimed for about half a second inside the clock
    # sampler's window and then once between CUDA events.
    for w in range(a.warmup):
        for _, fn in set_ops[w % nsets]:
            fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for r in range(a.steps):
            for _, fn in set_ops[r % nsets]:
                fn()
    graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t_load = time.perf_counter()
        while time.perf_counter() - t_load < 0.5:
            graph.replay()
            torch.cuda.synchronize()
        barrier(world)
        wall0 = time.perf_counter()
        t_all0.record(stream)
        graph.replay()
        t_all1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        wall1 = time.perf_counter()
    region_ms = max_over_ranks(t_all0.elapsed_time(t_all1), world, dev)
    value = world * step_bytes * a.steps / (region_ms * 1e-3) / 1e9
    del graph

    # per kernel: each one back to back over the same sets (a CUDA graph of
    # three rounds, median of ten replays), the dominant one for the roofline
    kern = {}
    for n, v in steady_step_ops(torch, stream, sets, peak).items():
        us = max_over_ranks(v["us"], world, dev)
        gbs = step.bytes(n) / (us * 1e-6) / 1e9
        kern[n] = dict(avg_us=round(us, 2), gbs=round(gbs, 1), frac=round(gbs / peak, 4),
                       bytes=step.bytes(n))
    dom = max(kern, key=lambda n: kern[n]["avg_us"])

    # the same steps launched eagerly from the host, one after another
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000)  # let the host run ahead of the GPU
    ev0.record(stream)
    for r in range(a.steps):
        for _, fn in set_ops[r % nsets]:
            fn()
    ev1.record(stream)
    torch.cuda.synchronize()
    eager_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)

    # ---- the same kernels one at a time, L2 flushed before each launch --------
    flush = L2Flush(torch, dev)
    iso = isolated(torch, stream, flush, step, peak, reps=max(20, min(a.steps, 200)))

    # ---- end to end through the public API with host buffers ----------------
    del sets, set_ops
    torch.cuda.empty_cache()
    e2e = e2e_arm(torch, R, stream, max(3, min(a.steps, 20)), world, dev, case, args)

    if rank != 0:
        return None
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": round(region_ms / a.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} softmax: router_topk_fwd + router_aux_scores_fwd"
                               " + router_topk_bwd + router_aux_scores_bwd",
                   "tokens": 8192, "experts": 2304, "topk": 36, "score_func": "softmax",
                   "logits_dtype": "f32", "tokens_per_gpu": 8192,
                   "parallelism": f"data-parallel x{world} (independent token batches)",
                   "l2": f"inputs larger than L2: steps rotate over {nsets} buffer sets "
                         f"({nsets} x {min(step.bytes(n) for n in names) >> 20} MiB and more "
                         f"per kernel > 3 x {l2 >> 20} MiB L2), kernels back to back, "
                         "no flush",
                   "peak_hbm_gbs": peak, "peak_kind": peak_kind},
        "gpu_launches": len(names) * a.steps,
        "timing": f"one CUDA graph of the {a.steps} steps between CUDA events",
        "kernel_sum_ms_per_step": round(sum(k["avg_us"] for k in kern.values()) * 1e-3, 4),
        "eager_ms_per_step": round(eager_ms / a.steps, 4),
        "wall_s": round(wall1 - wall0, 3),
        "kernels": kern,
        "roofline": {"bound": "hbm", "kernel": dom,
                     "achieved": kern[dom]["gbs"], "peak": peak, "unit": "GB/s",
                     "frac": kern[dom]["frac"], "peak_kind": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": kern[dom]["bytes"],
                     "traffic": traffic_for(dom, WORKLOAD)},
        "isolated": iso,
        "e2e": e2e,
        "clocks": clk.summary(),
    }
    if not a.no_extra:
        out["target_matrix"] = target_matrix(torch, R, stream, dev, peak, l2)
        out["breakdown"] = breakdown(torch, R, stream, dev, peak, l2)
        out["next_rows"] = next_rows(torch, R, stream, L2Flush(torch, dev), dev, peak, l2)
        out["decode_us"] = decode_latency(torch, R, stream, dev)
        out["decode_eager_us"] = decode_eager(torch, R, stream, dev)
        out["decode_maps_us"] = decode_latency(torch, R, stream, dev, maps=True)
    out["cpu_baseline"] = cpu_baseline(a.cpu_seconds)
    return out


def isolated(torch, stream, flush, step, peak, reps):
    """The step's kernels one launch at a time, L2 flushed with clean lines
    before each (a kernel's own writes may stay dirty in L2 after its end
    event, so its write-back goes untimed): mean µs per kernel and the step's
    effective GB/s."""
    ops = step.ops()
    t = time_ops(torch, stream, flush, ops, reps, 3)
    res = {"protocol": f"one launch at a time, L2 flushed before each (write of {flush.mib} "
                       f"MiB, then a read of another {flush.mib} MiB), mean of {reps}"}
    total_us, total_b = 0.0, 0
    for i, (n, _) in enumerate(ops):
        us = sum(t[i]) / len(t[i]) * 1e3
        gbs = step.bytes(n) / (us * 1e-6) / 1e9
        res[n] = {"us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}
        total_us += us
        total_b += step.bytes(n)
    gbs = total_b / (total_us * 1e-6) / 1e9
    res["step"] = {"us": round(total_us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}
    return res


def e2e_arm(torch, R, stream, reps, world, dev, case, args):
    """Same step through the public API with host buffers: every step copies
    its inputs in from pinned host memory, makes the four router calls and
    copies every output back.  The inputs sit in one device buffer and the
    outputs in another (the router writes into caller-placed views), so each
    direction is one copy per step.  Reported: steps pipelined over two
    device buffer sets (inputs of step i+1 in flight while step i computes and
    step i-1's outputs come back, on three streams ordered by events); beside
    it the same steps one after another on one stream, and the host-link copy
    ceilings measured on the same buffers."""
    steps = [Step(R, torch, case, args, dev, "softmax", packed=True) for _ in range(2)]
    step = steps[0]
    hin = torch.empty(step.in_buf.numel(), dtype=torch.uint8, pin_memory=True)
    hin.copy_(step.in_buf)
    houts = [torch.empty(st.out_buf.numel(), dtype=torch.uint8, pin_memory=True)
             for st in steps]
    h2d = int(hin.numel())
    d2h = int(houts[0].numel())
    step_bytes = sum(step.bytes(n) for n, _ in step.ops())

    def copy_in(st):
        st.in_buf.copy_(hin, non_blocking=True)

    def copy_out(st, hout):
        hout.copy_(st.out_buf, non_blocking=True)

    # one after another on one stream
    def serial_one():
        copy_in(step)
        for _, fn in step.ops():
            fn()
        copy_out(step, houts[0])

    for _ in range(2):
        serial_one()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        serial_one()
    e1.record(stream)
    torch.cuda.synchronize()
    serial_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)

    # pipelined over two buffer sets
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))

    def pipelined(n, first=None, last=None):
        done_cmp, done_out = [None, None], [None, None]
        for i in range(n):
            k = i % 2
            st = steps[k]
            with torch.cuda.stream(s_in):
                if i == 0 and first is not None:
                    first.record(s_in)
                if done_cmp[k] is not None:
                    s_in.wait_event(done_cmp[k])  # step i-2 has read this set's inputs
                copy_in(st)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in)
                if done_out[k] is not None:
                    s_cmp.wait_event(done_out[k])  # step i-2's outputs are back on the host
                for _, fn in st.ops():
                    fn()
                done_cmp[k] = torch.cuda.Event()
                done_cmp[k].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_cmp[k])
                copy_out(st, houts[k])
                done_out[k] = torch.cuda.Event()
                done_out[k].record(s_out)
        if last is not None:
            last.record(s_out)

    pipelined(2)
    torch.cuda.synchronize()
    barrier(world)
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    pipelined(reps, p0, p1)
    torch.cuda.synchronize()
    ms = max_over_ranks(p0.elapsed_time(p1), world, dev)

    # host-link ceilings on the same buffers: each direction alone, and both
    # at once on two streams (what the pipeline overlaps)
    def copy_gbs(fns_streams, nbytes):
        for _ in range(2):
            for fn, st in fns_streams:
                with torch.cuda.stream(st):
                    fn()
        torch.cuda.synchronize()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        uniq = list({id(st): st for _, st in fns_streams}.values())
        for st in uniq:
            st.wait_event(c0)
        for _ in range(reps):
            for fn, st in fns_streams:
                with torch.cuda.stream(st):
                    fn()
        for st in uniq:
            ev = torch.cuda.Event()
            ev.record(st)
            stream.wait_event(ev)
        c1.record(stream)
        torch.cuda.synchronize()
        return nbytes * reps / (c0.elapsed_time(c1) * 1e-3) / 1e9

    d2h_gbs = copy_gbs([(lambda: copy_out(step, houts[0]), s_out)], d2h)
    h2d_gbs = copy_gbs([(lambda: copy_in(step), s_in)], h2d)
    both_ms_per = (h2d / h2d_gbs + d2h / d2h_gbs) / 1e9  # if serialised
    bidir_gbs = copy_gbs([(lambda: copy_in(steps[1]), s_in),
                          (lambda: copy_out(step, houts[0]), s_out)], h2d + d2h)
    ms_per = ms / reps
    return {"value": round(world * step_bytes * reps / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms_per, 4),
            "pipelined": "two device buffer sets; one copy in, the four router calls and one "
                         "copy out per step, on three streams ordered by events",
            "serial": {"value": round(world * step_bytes * reps / (serial_ms * 1e-3) / 1e9, 1),
                       "ms_per_step": round(serial_ms / reps, 4)},
            "copy_ceiling_d2h_gbs": round(d2h_gbs, 1),
            "copy_ceiling_h2d_gbs": round(h2d_gbs, 1),
            "copy_ceiling_bidirectional_gbs": round(bidir_gbs, 1),
            "copies_alone_ms_per_step": round(both_ms_per * 1e3, 4),
            "d2h_rate_gbs": round(d2h / (ms_per * 1e-3) / 1e9, 1),
            "d2h_rate_frac_of_ceiling": round(d2h / (ms_per * 1e-3) / 1e9 / d2h_gbs, 3)}


def copy_ceiling(torch, stream, flush, dev, nbytes, peak, l2=None):
    """A device-to-device copy moving the same bytes as one launch (half read,
    half written), timed like the router kernels: isolated (L2 flushed before
    each copy, median of 20) or, given l2, back to back over rotating buffer
    pairs totalling more than 3x L2 (CUDA graph)."""
    half = max(nbytes // 2, 16)
    if l2 is None:
        src = torch.empty(half, dtype=torch.uint8, device=dev)
        dst = torch.empty(half, dtype=torch.uint8, device=dev)
        t = time_ops(torch, stream, flush, [("copy", lambda: dst.copy_(src))], 20, 3)
        us = statistics.median(t[0]) * 1e3
    else:
        n = max(2, -(-3 * l2 // (2 * half)))
        pairs = [(torch.empty(half, dtype=torch.uint8, device=dev),
                  torch.empty(half, dtype=torch.uint8, device=dev)) for _ in range(n)]
        us = graph_us(torch, stream, [lambda s=s_, d=d_: d.copy_(s) for s_, d_ in pairs])
        del pairs
    gbs = 2 * half / (us * 1e-6) / 1e9
    return {"us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 3)}


def time_step_ops(torch, stream, flush, st, peak):
    """The four kernels of one Step, each timed in isolation (L2 flushed
    before every launch, median of 20): µs, effective GB/s, fraction of peak."""
    ops = st.ops()
    t = time_ops(torch, stream, flush, ops, 20, 3)
    row = {}
    for i, (n, _) in enumerate(ops):
        med = statistics.median(t[i])
        gbs = st.bytes(n) / (med * 1e-3) / 1e9
        row[n] = {"us": round(med * 1e3, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 3)}
    return row


def steady_step_ops(torch, stream, sets, peak):
    """The four kernels of a list of rotating buffer sets, each timed back to
    back over the sets (CUDA graph of 3 rounds, median of 10 replays)."""
    row = {}
    first = sets[0]
    for i, (n, _) in enumerate(first.ops()):
        us = graph_us(torch, stream, [st.ops()[i][1] for st in sets])
        gbs = first.bytes(n) / (us * 1e-6) / 1e9
        row[n] = {"us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 3)}
    return row


def breakdown(torch, R, stream, dev, peak, l2):
    """Per-kernel effective GB/s on the other benchmark workloads in both
    protocols (back to back over rotating buffer sets, and isolated with L2
    flushed before each launch), with a plain device copy of the top-K
    forward's bytes beside each (copy_ceiling)."""
    from score_top_expert_gb300.workloads import make_workload
    flush = L2Flush(torch, dev)
    res = {}
    for name, sfs, dts in (("t8192_e256_k8", ("softmax", "sigmoid"), ("f32", "bf16")),
                           ("t16384_e256_k8_grouped", ("sigmoid",), ("bf16",)),
                           ("t1024_e64_k4", ("softmax",), ("f32",))):
        for dt in dts:
            case, args = make_workload(name, dtype=dt)
            for sf in sfs:
                sets = rotating_sets(R, torch, case, args, dev, sf, l2)
                b = sets[0].bytes("topk_fwd")
                res[f"{name}/{sf}/{dt}"] = {
                    "steady": steady_step_ops(torch, stream, sets, peak),
                    "isolated": time_step_ops(torch, stream, flush, sets[0], peak),
                    "copy_ceiling": {"steady": copy_ceiling(torch, stream, flush, dev, b, peak,
                                                            l2),
                                     "isolated": copy_ceiling(torch, stream, flush, dev, b,
                                                              peak)}}
                del sets
                torch.cuda.empty_cache()
    return res


# (E, K) pairs of the before/after table on the TransformerEngine page
# ("[Common] Optimize fused router forward/backward kernels", benchmark
# results), all at 8192 fp32 tokens; the sweep adds the pairs it leaves out
SWEEP_E = (512, 2304)
SWEEP_K = (4, 8, 22, 36)


def k_sweep(a):
    """Every (E, K) of SWEEP_E x SWEEP_K under both score functions, the four
    kernels timed back to back over rotating buffer sets and in isolation
    (L2 flushed before each launch); one JSON line."""
    import torch

    import score_top_expert_gb300.router as R
    from score_top_expert_gb300 import build
    from score_top_expert_gb300.workloads import make_workload
    build.build()
    R.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    flush = L2Flush(torch, dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    peak, peak_kind = hbm_peak()
    res = {}
    for E, name in zip(SWEEP_E, ("t8192_e512_k22", "t8192_e2304_k36")):
        for K in SWEEP_K:
            case, args = make_workload(name, K=K)
            for sf in ("softmax", "sigmoid"):
                sets = rotating_sets(R, torch, case, args, dev, sf, l2)
                res[f"e{E}_k{K}/{sf}"] = {
                    "steady": steady_step_ops(torch, stream, sets, peak),
                    "isolated": time_step_ops(torch, stream, flush, sets[0], peak)}
                del sets
                torch.cuda.empty_cache()
    assert R.device_status() == 0
    return {"sweep": "router kernels over (E, K), 8192 fp32 tokens: steady = back to back "
                     "over rotating buffer sets (CUDA graph, median of 10 replays); "
                     "isolated = L2 flushed before each launch, median of 20",
            "peak_gbs": peak, "peak_kind": peak_kind, "results": res}


# the target matrix: E x K x score function at 8192 fp32 tokens (the pairs of
# the TransformerEngine page's softmax and sigmoid tables, "[Common] Optimize
# fused router forward/backward kernels", Performance)
MATRIX_E = ((512, "t8192_e512_k22"), (2304, "t8192_e2304_k36"))
MATRIX_K = (22, 36)
MATRIX_TARGET = 0.6


def target_matrix(torch, R, stream, dev, peak, l2):
    """The four kernels at every (E, K, score function) of the target matrix,
    back to back over rotating buffer sets (more than 3x L2 per kernel), with
    a device copy of the top-K forward's bytes under the same protocol, and
    the whole step of four kernels."""
    from score_top_expert_gb300.workloads import make_workload
    res = {"protocol": "CUDA graph of 3 rounds of back-to-back launches over N rotating "
                       "buffer sets (> 3x L2 of bytes per launch), median of 10 replays, "
                       "no flush", "target_frac": MATRIX_TARGET, "cells": {}}
    below = []
    for E, name in MATRIX_E:
        for K in MATRIX_K:
            case, args = make_workload(name, K=K)
            for sf in ("softmax", "sigmoid"):
                sets = rotating_sets(R, torch, case, args, dev, sf, l2)
                row = steady_step_ops(torch, stream, sets, peak)
                first = sets[0]
                step_fns = [fn for st in sets for _, fn in st.ops()]
                us = graph_us(torch, stream, step_fns) * len(first.ops())
                sb = sum(first.bytes(n) for n, _ in first.ops())
                row["step"] = {"us": round(us, 2), "gbs": round(sb / (us * 1e-6) / 1e9, 1),
                               "frac": round(sb / (us * 1e-6) / 1e9 / peak, 3)}
                row["copy_ceiling"] = copy_ceiling(torch, stream, None, dev,
                                                   first.bytes("topk_fwd"), peak, l2)
                row["buffer_sets"] = len(sets)
                key = f"e{E}_k{K}/{sf}"
                res["cells"][key] = row
                below += [f"{key}/{n}" for n, _ in first.ops()
                          if row[n]["frac"] < MATRIX_TARGET]
                del sets, first, step_fns
                torch.cuda.empty_cache()
    res["below_target"] = below
    return res


def next_rows(torch, R, stream, flush, dev, peak, l2):
    """The compact forward, the expert maps and the aux loss on the benchmark
    workloads: back to back over rotating copies of each call's buffers (more
    than 3x L2 of bytes per launch; CUDA graph, median of 10 replays), and in
    isolation (L2 flushed before each launch; median of 20)."""
    from score_top_expert_gb300.workloads import make_workload
    res = {}
    for name in ("t8192_e512_k22", "t8192_e2304_k36"):
        case, args = make_workload(name)
        T, E, K = case.logits.shape[0], case.logits.shape[1], args["K"]
        x0 = torch.from_numpy(case.logits).to(dev)
        i32 = torch.int32

        def compact_set():
            x = x0.clone()
            w = torch.empty(T, K, device=dev)
            idx = torch.empty(T, K, dtype=i32, device=dev)
            tei = torch.empty(T, K, dtype=i32, device=dev)
            return lambda: R.router_topk_fwd_compact(
                x, K, "softmax", topk_weights=w, topk_indices=idx, token_expert_indices=tei)

        _, idx0, *_ = R.router_topk_fwd_compact(x0, K, "softmax")

        def maps_set():
            idx = idx0.clone()
            out = {"expert_first_token_offset": torch.empty(E + 1, dtype=i32, device=dev)}
            for nm in ("permuted_to_unpermuted", "unpermuted_to_permuted", "permuted_experts"):
                out[nm] = torch.empty(T * K, dtype=i32, device=dev)
            ws = torch.empty(R.lib().router_expert_maps_workspace_bytes(T, E), dtype=torch.uint8,
                             device=dev)
            return lambda: R.router_expert_maps(idx, E, out=out, workspace=ws)

        q0, amap0, _ = R.router_aux_scores_fwd(x0, K, "softmax")

        def loss_fwd_set():
            q, amap = q0.clone(), amap0.clone()
            loss = torch.empty(1, device=dev)
            tok = torch.empty(E, dtype=i32, device=dev)
            lws = torch.empty(max(16, R.lib().router_aux_loss_workspace_bytes(T, E)),
                              dtype=torch.uint8, device=dev)
            return lambda: R.router_aux_loss_fwd(q, amap, K, 0.01, loss=loss,
                                                 tokens_per_expert=tok, workspace=lws)

        _, tok0 = R.router_aux_loss_fwd(q0, amap0, K, 0.01)

        def loss_bwd_set():
            gl = torch.ones(1, device=dev)
            tok = tok0.clone()
            gq = torch.empty(T, E, device=dev)
            return lambda: R.router_aux_loss_bwd(gl, tok, T, K, 0.01, grad_aux_scores=gq)

        row = {}
        for n, make in (("compact_fwd", compact_set), ("expert_maps", maps_set),
                        ("aux_loss_fwd", loss_fwd_set), ("aux_loss_bwd", loss_bwd_set)):
            b = next_row_bytes(n, T, E, K, 4)
            nsets = min(96, max(2, -(-3 * l2 // b)))
            fns = [make() for _ in range(nsets)]
            us = graph_us(torch, stream, fns)
            t = time_ops(torch, stream, flush, [(n, fns[0])], 20, 3)
            iso = statistics.median(t[0]) * 1e3
            row[n] = {"us": round(us, 2), "gbs": round(b / (us * 1e-6) / 1e9, 1),
                      "frac": round(b / (us * 1e-6) / 1e9 / peak, 3), "bytes": b,
                      "isolated": {"us": round(iso, 2),
                                   "frac": round(b / (iso * 1e-6) / 1e9 / peak, 3)}}
            del fns
            torch.cuda.empty_cache()
        row["expert_maps"]["launches"] = ("a one-block kernel zeroing the barrier counter and "
                                          "one cooperative launch (three launches beyond one "
                                          "wave)")
        row["aux_loss_fwd"]["launches"] = "a one-block kernel zeroing the counters and one launch"
        res[f"{name}/softmax/f32"] = row
        del x0, q0, amap0
        torch.cuda.empty_cache()
    return res


def decode_eager(torch, R, stream, dev):
    """Decode latency per call including launch overhead: 200 calls of the
    top-K forward through the Python binding, one after another on the
    stream without a graph (1, 2, 4 rows x 512 experts, K = 8, softmax)."""
    from score_top_expert_gb300.workloads import make_case
    res = {}
    for T in (1, 2, 4):
        case = make_case(T, 512, 8, seed=77 + T)
        x = torch.from_numpy(case.logits).to(dev)
        p = torch.empty(T, 512, device=dev)
        m = torch.empty(T, 512, dtype=torch.bool, device=dev)
        s = torch.empty(T, 512, device=dev)
        for _ in range(20):
            R.router_topk_fwd(x, 8, "softmax", probs=p, routing_map=m, scores=s)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(200):
            R.router_topk_fwd(x, 8, "softmax", probs=p, routing_map=m, scores=s)
        torch.cuda.synchronize()
        res[f"T{T}_K8"] = round((time.perf_counter() - t0) / 200 * 1e6, 2)
    return res


def decode_latency(torch, R, stream, dev, maps=False):
    """Decode sweep: 1, 2, 4 rows x 512 experts, softmax, K in 1..10: device
    time per launch from a CUDA graph of 100 launches (L2-warm).  With maps:
    the router with expert maps (one fused launch) instead of the top-K
    forward."""
    from score_top_expert_gb300.workloads import make_case
    res = {}
    for T in (1, 2, 4):
        case = make_case(T, 512, 10, seed=77 + T)
        x = torch.from_numpy(case.logits).to(dev)
        p = torch.empty(T, 512, device=dev)
        m = torch.empty(T, 512, dtype=torch.bool, device=dev)
        s = torch.empty(T, 512, device=dev)
        ws = torch.empty(R.lib().router_expert_maps_workspace_bytes(T, 512), dtype=torch.uint8,
                         device=dev)
        for K in (1, 2, 4, 6, 8, 10):
            w = torch.empty(T, K, device=dev)
            idx = torch.empty(T, K, dtype=torch.int32, device=dev)
            mo = {"expert_first_token_offset": torch.empty(513, dtype=torch.int32, device=dev)}
            for nm in ("permuted_to_unpermuted", "unpermuted_to_permuted", "permuted_experts"):
                mo[nm] = torch.empty(T * K, dtype=torch.int32, device=dev)

            def launch():
                if maps:
                    R.router_topk_fwd_maps(x, K, "softmax", topk_weights=w, topk_indices=idx,
                                           token_expert_indices=False, out=mo,
                                           workspace=ws)
                else:
                    R.router_topk_fwd(x, K, "softmax", probs=p, routing_map=m, scores=s)
            launch()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(100):
                    launch()
            g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(5):
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            res[f"T{T}_K{K}"] = round(e0.elapsed_time(e1) * 1e3 / 500, 2)
    return res


# ---------------------------------------------------------------------------
# CPU oracle
# ---------------------------------------------------------------------------
def oracle_step(O, case, K, rows):
    """The oracle over ``rows`` token rows of the workload: the same four ops."""
    x = case.logits[rows]
    f = O.topk_fwd(x, K, "softmax")
    a = O.aux_scores_fwd(x, K, "softmax")
    O.topk_bwd(case.grad_probs[rows], f["routing_map"], f["scores"], "softmax")
    O.aux_scores_bwd(case.grad_scores[rows], a["saved"], "softmax")


def _oracle_rows_worker(arg):
    """One process of the all-cores oracle run: chunks i, i + n, ... of 128
    rows until the time budget is spent.  Returns (rows, seconds)."""
    i, n, seconds = arg
    import oracle.router_oracle as O
    from score_top_expert_gb300.workloads import make_workload
    case, args = make_workload(WORKLOAD)
    K, T = args["K"], case.logits.shape[0]
    chunk, done, c = 128, 0, i
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds and (c + 1) * chunk <= T:
        oracle_step(O, case, K, slice(c * chunk, (c + 1) * chunk))
        done += chunk
        c += n
    return done, time.perf_counter() - t0


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for placing the
    oracle's timing."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(seconds: float):
    """The oracle on the host: all cores (one process per core, rows split
    between them; the reported value) and one thread."""
    import multiprocessing as mp

    import oracle.router_oracle as O
    from score_top_expert_gb300.workloads import make_workload
    case, args = make_workload(WORKLOAD)
    E, K = case.logits.shape[1], args["K"]
    row_bytes = sum(bytes_per_launch(op, 1, E, 4) for op in
                    ("topk_fwd", "aux_fwd", "topk_bwd", "aux_bwd"))
    done, t0 = 0, time.perf_counter()
    chunk = 128
    while time.perf_counter() - t0 < seconds and done + chunk <= case.logits.shape[0]:
        oracle_step(O, case, K, slice(done, done + chunk))
        done += chunk
    dt = time.perf_counter() - t0
    single = {"value": round(row_bytes * done / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
              "sample": f"first {done} of 8192 token rows of {WORKLOAD} (softmax, fp32): "
                        f"the four ops, float64 numpy, one thread, {dt:.1f} s"}
    n = max(1, os.cpu_count() or 1)
    try:
        # spawn: the parent process has a CUDA context
        with mp.get_context("spawn").Pool(n) as pool:
            res = pool.map(_oracle_rows_worker, [(i, n, seconds) for i in range(n)])
        rows = sum(r for r, _ in res)
        wall = max(t for _, t in res)
        allc = {"value": round(row_bytes * rows / wall / 1e9, 4), "cores": n,
                "sample": f"{rows} of 8192 token rows of {WORKLOAD} (softmax, fp32) split in "
                          f"128-row chunks over {n} processes: the four ops, float64 numpy, "
                          f"{wall:.1f} s"}
    except Exception as exc:  # a host without process pools still gets the one-thread figure
        allc = None
        single["note"] = f"all-cores run unavailable: {type(exc).__name__}"
    model = cpu_model()
    if allc is None:
        return dict(single, kind="oracle", cpu_model=model)
    return {"value": allc["value"], "unit": "GB/s", "cores": allc["cores"], "kind": "oracle",
            "cpu_model": model, "sample": allc["sample"], "single_thread": single}


def reference_arm(a, world, rank):
    """The oracle as the reference arm: each step runs the four ops over a
    bounded sample of the workload's rows on the host cores."""
    if rank != 0:
        return None
    import oracle.router_oracle as O
    from score_top_expert_gb300.workloads import make_workload
    case, args = make_workload(WORKLOAD)
    E, K = case.logits.shape[1], args["K"]
    rows_per_step = 64
    row_bytes = sum(bytes_per_launch(op, 1, E, 4) for op in
                    ("topk_fwd", "aux_fwd", "topk_bwd", "aux_bwd"))
    for w in range(a.warmup):
        oracle_step(O, case, K, slice(w * rows_per_step, (w + 1) * rows_per_step))
    times = []
    for s in range(a.steps):
        lo = (s * rows_per_step) % (8192 - rows_per_step)
        t0 = time.perf_counter()
        oracle_step(O, case, K, slice(lo, lo + rows_per_step))
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = row_bytes * rows_per_step * a.steps / total / 1e9
    sample = (f"{rows_per_step} token rows per step of {WORKLOAD} (softmax, fp32): the four "
              "ops, float64 numpy, one thread")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": round(total / a.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{WORKLOAD} softmax: the four router ops (bounded sample)",
                       "tokens": 8192, "experts": 2304, "topk": 36},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def profile_run(a):
    """Untimed steps for an ncu capture, no flush.  --profile-ops step: the
    four router ops once per step, steps rotating over the headline's buffer
    sets; next: the compact forward, the expert maps, the aux-loss forward and
    backward."""
    import torch

    import score_top_expert_gb300.router as R
    from score_top_expert_gb300 import build
    from score_top_expert_gb300.workloads import make_workload
    build.build()
    dev = torch.device("cuda", 0)
    case, args = make_workload(a.profile)
    if a.profile_ops == "step":
        # the bench's own protocol: back to back over rotating buffer sets
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        sets = rotating_sets(R, torch, case, args, dev, a.profile_score, l2)
        ops = []
        for w in range(a.warmup + a.steps):
            ops += [fn for _, fn in sets[w % len(sets)].ops()]
        for fn in ops:
            fn()
        torch.cuda.synchronize()
        print(f"profile run done: {a.profile} {a.profile_ops} {a.profile_score}, "
              f"{a.warmup + a.steps} steps over {len(sets)} buffer sets")
        return
    else:
        T, E = case.logits.shape
        K = args["K"]
        x = torch.from_numpy(case.logits).to(dev)
        w = torch.empty(T, K, device=dev)
        idx = torch.empty(T, K, dtype=torch.int32, device=dev)
        tei = torch.empty(T, K, dtype=torch.int32, device=dev)
        ws = torch.empty(R.lib().router_expert_maps_workspace_bytes(T, E), dtype=torch.uint8,
                         device=dev)
        q, amap, _ = R.router_aux_scores_fwd(x, K, "softmax")
        lws = torch.empty(R.lib().router_aux_loss_workspace_bytes(T, E), dtype=torch.uint8,
                          device=dev)
        loss = torch.empty(1, device=dev)
        tok = torch.empty(E, dtype=torch.int32, device=dev)
        gl = torch.ones(1, device=dev)
        gq = torch.empty(T, E, device=dev)
        ops = [lambda: R.router_topk_fwd_compact(x, K, "softmax", topk_weights=w,
                                                 topk_indices=idx, token_expert_indices=tei),
               lambda: R.router_expert_maps(idx, E, workspace=ws),
               lambda: R.router_aux_loss_fwd(q, amap, K, 0.01, loss=loss,
                                             tokens_per_expert=tok, workspace=lws),
               lambda: R.router_aux_loss_bwd(gl, tok, T, K, 0.01, grad_aux_scores=gq)]
    for _ in range(a.warmup + a.steps):
        for fn in ops:
            fn()
    torch.cuda.synchronize()
    print(f"profile run done: {a.profile} {a.profile_ops} {a.profile_score}, "
          f"{a.warmup + a.steps} steps")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="length of the CPU-oracle baseline sample")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the per-workload breakdown and the decode sweep")
    ap.add_argument("--profile", default=None, metavar="WORKLOAD",
                    help="run W + K untimed steps of the four ops on a named workload "
                         "(softmax; for ncu captures) and print nothing else")
    ap.add_argument("--profile-score", default="softmax", choices=("softmax", "sigmoid"))
    ap.add_argument("--profile-ops", default="step", choices=("step", "next"),
                    help="with --profile: the four router ops, or the compact forward, "
                         "expert maps and aux loss")
    ap.add_argument("--sweep-k", action="store_true",
                    help="time the four kernels over E in {512, 2304} x K in {4, 8, 22, 36} "
                         "(softmax and sigmoid) and print that table instead")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if a.profile:
        profile_run(a)
        return
    if a.sweep_k:
        print(json.dumps(k_sweep(a)), flush=True)
        return
    if a.impl == "reference":
        out = reference_arm(a, world, rank)
    else:
        out = gpu_arm(a, world, rank, local)
    if out is not None:
        print(json.dumps(out), flush=True)
    if world > 1 and a.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
