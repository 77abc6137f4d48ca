#!/usr/bin/env python
"""Benchmark: TFLOP/s of the training products of linear layers on GB300.

One step = every product of the 2B-class decoder layer set (q, k, v, o
2304->2304; gate, up 2304->5760; down 5760->2304) at T = 1,024, 2,048 and
4,096 tokens, each as forward, input gradient and weight gradient, in bf16 and
in fp16 with FP32 accumulation: 126 products, 5.25 TFLOP.  Inputs are seeded
synthetic tensors resident in HBM (1.95 GB, far above the L2); L2 is also
flushed (a 256 MiB write) before every step, outside the timed events.  The
step is one captured CUDA graph of the library calls in training order, the
products that a training step may run side by side (the q, k and v
projections, gate and up, a layer's input and weight gradients) on parallel
branches (`--serial-step`: one product at a time); CUDA events inside it
mark the step (`value`).  The roofline entry times the dominant launch class
(one kernel identity at one product shape): its launches of the step, with
the same tensors and plans, replayed back to back in a graph of their own
(L2 flushed before each replay), events around each replay.

Printed on stdout (rank 0): first one `row {...}` line per measured row of the
other product sets (the 135M-class step, every distinct 2B-class product
alone with warm and rotated operands, FP32 operands, rank-16 LoRA, batched
and fused attention in bf16 and fp16), then ONE compact JSON line, the
headline, last.  `value` is the whole-job TFLOP/s (all ranks' flops / the
slowest rank's time).  Also in it: the same step end to end through the
public API with pinned host inputs and outputs copied every step (`e2e`), the
oracle on the host cores on a bounded sample (`cpu_baseline`), the roofline
fraction of the dominant launch class and SM clocks sampled during the timed
region.

`--impl reference` times the fp64 CPU oracle on the same workload instead
(bounded samples per step, host cores).

`python bench.py probe OP D0 D1 D2 [--dtype bf16|f16|f32] [--out same|f32]
[--plan "bn splits [raster]"] [--reps R]` times one product alone through the
public entry points (the command the ncu summaries are captured with): OP is
fwd|dgrad|wgrad or fwd_lora|dgrad_lora (dims T d_in d_out; rank 16, scale 2),
one of the attention products
qk|pv|do_vt|pt_do|ds_k|dst_q or the fused attn_fwd / attn_bwd (dims heads s d), or
lora_down|lora_up|lora_grad and their _f32w forms (dims T d_in d_out, rank 16); --plan writes a
one-line tile table for the shape and loads it first.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gemms_linear_layers_gb300 import inputs, workloads  # noqa: E402

METRIC = "TFLOPS per training GEMM (fwd/dgrad/wgrad, bf16/fp16) and % of GB300 dense peak"
STEP_SETS = {
    "2b": (workloads.DECODER_2B,
           "2B-class decoder layer set (q/k/v/o 2304x2304, gate/up 2304->5760, down 5760->2304) at T=1024, 2048 "
           "and 4096, fwd+dgrad+wgrad, bf16 and fp16 (126 products)"),
    "135m": (workloads.DECODER_135M,
             "135M-class decoder layer set (q/o 576x576, k/v 576->192, gate/up 576->1536, down 1536->576, head "
             "576->49152) at T=2048, fwd+dgrad+wgrad, bf16 and fp16 (48 products)"),
}
L2_FLUSH_BYTES = 256 << 20
PROFILES_DIR = os.path.join(ROOT, "profiles")
CSRC_DIR = os.path.join(ROOT, "gemms_linear_layers_gb300", "csrc")


# the sources the step's kernels are built from: the 16-bit GEMM kernels (single
# CTAs, pairs, cluster split) and their launches, the split and tail
# reductions, the PTX wrappers, the shared declarations and the tensor maps
STEP_KERNEL_SOURCES = ("gemm_simt.cu", "gemm_tc.cuh", "gemm_tc2.cuh", "gemm_tc_cs.cuh", "gemm_tc_launch.cuh",
                       "gemm_tc_nn.cu", "gemm_tc_nt.cu", "gemm_tc_tn.cu", "ptx.cuh", "tg_internal.h", "tmap.cpp")


def kernel_sources_digest(csrc=None) -> str:
    """SHA-1 over the sources that decide what a kernel of the step reads and
    writes (STEP_KERNEL_SOURCES that exist; not the host planner, whose
    changes show up as a different kernel identity, nor the units whose
    kernels are not in the step), name and bytes in name order."""
    csrc = csrc or CSRC_DIR
    h = hashlib.sha1()
    for name in sorted(os.listdir(csrc)):
        if name in STEP_KERNEL_SOURCES:
            h.update(name.encode())
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def profiled_traffic(kernel_key: str, profiles=None, digest=None):
    """DRAM bytes (read + write) per launch of the launch class `kernel_key`,
    from a committed ncu summary that names it and records the digest of the
    kernel sources it was captured from; None when no summary matches or the
    kernels changed since the counters were taken."""
    profiles = profiles or PROFILES_DIR
    digest = digest or kernel_sources_digest()
    if not os.path.isdir(profiles):
        return None
    pat = re.compile(r"^- (bench_kernel_key|traffic_bytes_per_launch|kernel_sources_sha1): `([^`]*)`")
    for name in sorted(os.listdir(profiles)):
        if not name.endswith(".md"):
            continue
        fields = {}
        with open(os.path.join(profiles, name)) as f:
            for line in f:
                m = pat.match(line)
                if m:
                    fields[m.group(1)] = m.group(2)
        if fields.get("bench_kernel_key") == kernel_key and fields.get("kernel_sources_sha1") == digest:
            try:
                return int(fields["traffic_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [x for x in sm if x > 0.5 * (mx or max(sm))] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ products
class Product:
    def __init__(self, layer, op, dtype, T, d_in, d_out):
        self.layer, self.op, self.dtype = layer, op, dtype
        self.T, self.d_in, self.d_out = T, d_in, d_out
        if op == "fwd":
            self.M, self.N, self.K = T, d_out, d_in
        elif op == "dgrad":
            self.M, self.N, self.K = T, d_in, d_out
        else:
            self.M, self.N, self.K = d_out, d_in, T
        self.flops = workloads.flops(self.M, self.N, self.K)
        self.graph = None
        self.call = ""
        self.launches = 1
        self.kernel = "?"

    @property
    def name(self):
        return f"{self.layer}.{self.op}.T{self.T}.{str(self.dtype)[6:]}"

    @property
    def launch_class(self):
        """The kernel identity at this product's shape: launches of one class
        do the same work, so a per-launch figure of the class is well defined."""
        return f"{self.kernel} @ {self.M}x{self.N}x{self.K}"


def step_token_counts(cfg):
    T = cfg["T"]
    return tuple(T) if isinstance(T, (tuple, list)) else (T,)


def build_step(device, only=None, cfg=None):
    """Inputs, outputs and workspaces of every product of the step (or of the
    products named in `only`), on the device.  Every layer has its own
    tensors, as in a training step."""
    from gemms_linear_layers_gb300 import _binding as tg
    cfg = cfg or workloads.DECODER_2B
    prods = []
    for dtype in cfg["dtypes"]:
        for T in step_token_counts(cfg):
            for layer, d_in, d_out in cfg["layers"]:
                names = [Product(layer, op, dtype, T, d_in, d_out).name for op in ("fwd", "dgrad", "wgrad")]
                if only and not any(n in only for n in names):
                    continue
                X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag=f"bench-{layer}", device=device)
                t = {"X": X, "W": W, "dY": dY,
                     "Y": torch.empty(T, d_out, dtype=dtype, device=device),
                     "dX": torch.empty(T, d_in, dtype=dtype, device=device),
                     "dW": torch.empty(d_out, d_in, dtype=dtype, device=device)}
                for op in ("fwd", "dgrad", "wgrad"):
                    p = Product(layer, op, dtype, T, d_in, d_out)
                    if only and p.name not in only:
                        continue
                    opcode = {"fwd": tg.TG_OP_GEMM_FWD, "dgrad": tg.TG_OP_GEMM_DGRAD,
                              "wgrad": tg.TG_OP_GEMM_WGRAD}[op]
                    n = tg.tg_workspace_size(opcode, T, d_out, d_in, 0, dtype, dtype)
                    p.ws = torch.empty(max(n, 16), dtype=torch.uint8, device=device) if n else None
                    p.t = t
                    prods.append(p)
    return prods


def run_product(p):
    from gemms_linear_layers_gb300 import _binding as tg
    t = p.t
    if p.op == "fwd":
        tg.tg_gemm_fwd(t["X"], t["W"], Y=t["Y"], ws=p.ws)
    elif p.op == "dgrad":
        tg.tg_gemm_dgrad(t["dY"], t["W"], dX=t["dX"], ws=p.ws)
    else:
        tg.tg_gemm_wgrad(t["dY"], t["X"], dW=t["dW"], ws=p.ws)


def kernel_key(call: str) -> str:
    """'tc nt bn=256' style identity of the kernel a call ran (from tg_last_call)."""
    f = call.split()
    path = f[1] if len(f) > 1 else "?"
    if path == "ffma":
        return f"ffma {f[2]}" + (" +reduce" if any(x.startswith("splits=") and x != "splits=1" for x in f) else "")
    if path not in ("tc", "tc3"):
        return f"{path} {f[2] if len(f) > 2 else ''}".strip()
    bn = next((x for x in f if x.startswith("bn=")), "bn=?")
    sp = next((x for x in f if x.startswith("splits=")), "splits=1")
    deep = " deep" if "deep" in f else ""
    pair = " pair" if "pair" in f else (" cs" if "cs" in f else "")
    tail = " +tail" if any(x.startswith("tail=") for x in f) else ""
    sk = " sk" if "sk" in f else ""
    return f"{path} {f[2]} {bn}{deep}{pair}{sk}" + (" +reduce" if sp != "splits=1" else "") + tail


def launches_of(call: str) -> int:
    """Kernel launches of one call: the product, plus the ordered reduction
    of split or tail-split partials when the plan has one."""
    f = call.split()
    split = any(x.startswith("splits=") and x != "splits=1" for x in f)
    tail = any(x.startswith("tail=") for x in f)
    return 2 if (split or tail) else 1


def capture(prods, stream):
    from gemms_linear_layers_gb300 import _binding as tg
    for p in prods:  # warm-up call: sets kernel attributes, records the plan
        with torch.cuda.stream(stream):
            run_product(p)
        p.call = tg.tg_last_call()
        p.launches = launches_of(p.call)
        p.kernel = kernel_key(p.call)
    torch.cuda.synchronize()
    for p in prods:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run_product(p)
        p.graph = g
    torch.cuda.synchronize()


def probe_products(prods, stream, flush, reps=2):
    """Untimed pass: each product's own graph between events, in step order,
    to find the launch class with the largest share of the step."""
    per_prod = {p.name: 0.0 for p in prods}
    with torch.cuda.stream(stream):
        for _ in range(reps):
            flush.add_(1)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(prods) + 1)]
            ev[0].record(stream)
            for i, p in enumerate(prods):
                p.graph.replay()
                ev[i + 1].record(stream)
            torch.cuda.synchronize()
            for i, p in enumerate(prods):
                per_prod[p.name] += ev[i].elapsed_time(ev[i + 1]) / reps
    return per_prod


def external_event():
    """A timing event that becomes an event-record node when captured."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None


# The order of a training step's linear-layer products, as waves of products
# that have no data dependence on each other: forward q, k, v together, o,
# gate and up together, down, head; backward from the head down, each
# layer's input and weight gradients together (both need only dY and the
# layer's own input or weight), gate/up and q/k/v as groups.
FWD_WAVES = [["q", "k", "v"], ["o"], ["gate", "up"], ["down"], ["head"]]
BWD_WAVES = [["head"], ["down"], ["gate", "up"], ["o"], ["q", "k", "v"]]


def step_waves(prods):
    """The step's products as a list of waves (lists of products that may run
    concurrently); each (dtype, token count) set one after the other."""
    by = {(p.layer, p.op, p.dtype, p.T): p for p in prods}
    waves = []
    for dtype, T in dict.fromkeys((p.dtype, p.T) for p in prods):
        for group in FWD_WAVES:
            w = [by[(l, "fwd", dtype, T)] for l in group if (l, "fwd", dtype, T) in by]
            if w:
                waves.append(w)
        for group in BWD_WAVES:
            w = [by[(l, op, dtype, T)] for l in group for op in ("dgrad", "wgrad") if (l, op, dtype, T) in by]
            if w:
                waves.append(w)
    placed = {id(p) for w in waves for p in w}
    waves += [[p] for p in prods if id(p) not in placed]
    return waves


def graph_waves(prods, concurrent=True):
    """The waves of the step graph: with `concurrent`, the step's waves, a
    stream-K launch taken out to run alone after the rest of its wave (it
    waits on its own later CTAs, which need every SM it may occupy); without,
    one product per wave in training order."""
    if not concurrent:
        return [[q] for w in step_waves(prods) for q in w]
    out = []
    for w in step_waves(prods):
        alone = [p for p in w if " sk" in p.kernel]
        rest = [p for p in w if not any(p is q for q in alone)]
        if rest:
            out.append(rest)
        out += [[p] for p in alone]
    return out


def capture_step(prods, stream, concurrent=True):
    """One graph for the whole step: the waves of `graph_waves`, the products
    of a wave on parallel branches (fork/join through events on side
    streams).  External events mark the step's start and end."""
    e0, e1 = external_event(), external_event()
    if e0 is None:
        return None
    waves = graph_waves(prods, concurrent)
    width = max(len(w) for w in waves)
    side = [torch.cuda.Stream() for _ in range(width)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        e0.record()
        for w in waves:
            if len(w) == 1:
                branches = [(stream, w[0])]
            else:
                fork = torch.cuda.Event()
                fork.record(stream)
                branches = []
                for i, p in enumerate(w):
                    side[i].wait_event(fork)
                    branches.append((side[i], p))
            for st, p in branches:
                with torch.cuda.stream(st):
                    run_product(p)
            if len(w) > 1:
                for st, _ in branches:
                    j = torch.cuda.Event()
                    j.record(st)
                    stream.wait_event(j)
        e1.record()
    torch.cuda.synchronize()
    return g, e0, e1


def timed_steps(step, n_warm, n_steps, stream, flush):
    """Per step: flush L2 (untimed), replay the step graph, read its events;
    the total ms of the timed steps."""
    g, e0, e1 = step
    total_ms = 0.0
    for s in range(n_warm + n_steps):
        with torch.cuda.stream(stream):
            flush.add_(1)
            g.replay()
        torch.cuda.synchronize()
        if s >= n_warm:
            total_ms += e0.elapsed_time(e1)
    return total_ms


def capture_dominant(dprods, stream, rounds=3):
    """One graph of the dominant launch class's products of the step (same
    tensors, workspaces and plans as in the step), `rounds` passes back to
    back between two events: inside a graph, events around each launch would
    cut it off from the launch before it (measured: 37.6 us bracketed against
    32.0 us per launch back to back for the 4,096-token q/k/v/o weight
    gradient), so the class is timed as a run of its own launches."""
    e0, e1 = external_event(), external_event()
    if e0 is None:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        e0.record()
        for _ in range(rounds):
            for p in dprods:
                run_product(p)
        e1.record()
    torch.cuda.synchronize()
    return g, e0, e1, rounds * len(dprods)


def timed_dominant(dg, n_warm, n_steps, stream, flush):
    """Per replay: flush L2 (untimed), replay the dominant-class graph; the
    average ms per launch of the class."""
    g, e0, e1, n = dg
    total = 0.0
    for s in range(n_warm + n_steps):
        with torch.cuda.stream(stream):
            flush.add_(1)
            g.replay()
        torch.cuda.synchronize()
        if s >= n_warm:
            total += e0.elapsed_time(e1)
    return total / (n_steps * n)


def timed_steps_per_product(prods, n_warm, n_steps, stream, flush, dominant):
    """Fallback when events cannot be captured: each product's own graph,
    events between them on the launching stream."""
    total_ms, dom_ms = 0.0, 0.0
    with torch.cuda.stream(stream):
        for s in range(n_warm + n_steps):
            flush.add_(1)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(prods) + 1)]
            ev[0].record(stream)
            for i, p in enumerate(prods):
                p.graph.replay()
                ev[i + 1].record(stream)
            torch.cuda.synchronize()
            if s >= n_warm:
                total_ms += ev[0].elapsed_time(ev[-1])
                dom_ms += sum(ev[i].elapsed_time(ev[i + 1]) for i, p in enumerate(prods)
                              if p.launch_class == dominant)
    return total_ms, dom_ms


def by_launch_class(prods, per_prod):
    """{launch class: {ms, flops, n, products}} from a probe pass."""
    out = {}
    for p in prods:
        k = out.setdefault(p.launch_class, {"ms": 0.0, "flops": 0, "n": 0, "products": [], "launches": 0})
        k["ms"] += per_prod[p.name]
        k["flops"] += p.flops
        k["n"] += 1
        k["launches"] += p.launches
        k["products"].append(p.name)
    return out


# ------------------------------------------------------------------ e2e
def e2e_steps(prods, n_steps, stream):
    """The step through the public API with pinned host buffers: every step
    copies its inputs host->device and its outputs device->host.  Copies and
    products form a pipeline over the step's (dtype, token count) sets (the
    smallest first, the next smallest last): a set's X and W come in, then
    its dY, while the set before it computes; each product starts as soon as its own operands have arrived,
    and each result goes out on a second copy stream as soon as the product
    that writes it is done, while later sets come in.  Steps do not overlap."""
    groups = {}
    for p in prods:
        groups.setdefault((p.layer, p.dtype, p.T), []).append(p)
    # the smallest set first (the first products wait for it alone) and the
    # next smallest last (its outputs are what still crosses the link after
    # the last product): the large sets in between, while both directions of
    # the link are busy
    size = {}
    for p in prods:
        size[(p.dtype, p.T)] = size.get((p.dtype, p.T), 0) + p.M * p.N
    by_size = sorted(dict.fromkeys((p.dtype, p.T) for p in prods), key=lambda k: size[k])
    sets = by_size[:1] + by_size[:1:-1] + by_size[1:2] if len(by_size) > 2 else by_size
    h2d = d2h = 0
    host = {}
    for key, ps in groups.items():
        t = ps[0].t
        for n in ("X", "W", "dY", "Y", "dX", "dW"):
            host[(key, n)] = (t[n], torch.empty(t[n].shape, dtype=t[n].dtype).pin_memory())
            if n in ("X", "W", "dY"):
                host[(key, n)][1].copy_(t[n].cpu())
                h2d += t[n].numel() * t[n].element_size()
            else:
                d2h += t[n].numel() * t[n].element_size()
    needs = {"fwd": ("X", "W"), "dgrad": ("dY", "W"), "wgrad": ("dY", "X")}
    writes = {"fwd": "Y", "dgrad": "dX", "wgrad": "dW"}
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    times = []
    for step in range(n_steps + 1):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s_in.wait_event(a)
        s_out.wait_event(a)
        arrived = {}
        for dt, T in sets:  # operands in, set by set: X and W of every layer of the set, then its dY
            keys = [k for k in groups if k[1] == dt and k[2] == T]
            for names in (("X", "W"), ("dY",)):
                for key in keys:
                    with torch.cuda.stream(s_in):
                        for n in names:
                            dev, h = host[(key, n)]
                            dev.copy_(h, non_blocking=True)
                            arrived[(key, n)] = torch.cuda.Event()
                            arrived[(key, n)].record(s_in)
        for dt, T in sets:  # products set by set, forwards first, as their operands arrive
            keys = [k for k in groups if k[1] == dt and k[2] == T]
            for ops in (("fwd",), ("dgrad", "wgrad")):
                for key in keys:
                    for p in groups[key]:
                        if p.op not in ops:
                            continue
                        for n in needs[p.op]:
                            stream.wait_event(arrived[(key, n)])
                        with torch.cuda.stream(stream):
                            run_product(p)
                        done = torch.cuda.Event()
                        done.record(stream)
                        s_out.wait_event(done)
                        with torch.cuda.stream(s_out):  # its result out
                            dev, h = host[(key, writes[p.op])]
                            h.copy_(dev, non_blocking=True)
        out_done = torch.cuda.Event()
        out_done.record(s_out)
        stream.wait_event(out_done)
        b.record(stream)
        if step > 0:
            times.append((a, b))
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in times)
    return ms, h2d, d2h


# ------------------------------------------------------------------ oracle
def oracle_sample(target_s, cfg=None):
    """The fp64 oracle on the host cores over a bounded sample of the step:
    the first output rows of each of its products (same shapes, same input
    recipe and seeds).  Returns (flops, seconds, rows per product)."""
    import numpy as np

    import oracle
    cfg = cfg or workloads.DECODER_2B
    key = id(cfg)
    cache = oracle_sample.__dict__.setdefault("cache", {})
    if key not in cache:
        jobs = []
        for dtype in cfg["dtypes"]:
            for T in step_token_counts(cfg):
                for layer, d_in, d_out in cfg["layers"]:
                    X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag=f"bench-{layer}")
                    for op in ("fwd", "dgrad", "wgrad"):
                        jobs.append((op, X, W, dY))
        cache[key] = {"jobs": jobs, "sec_per_row": None}
    c = cache[key]

    def run(rows):
        flops = 0
        t0 = time.perf_counter()
        for op, X, W, dY in c["jobs"]:
            if op == "fwd":
                M, N, K = X.shape[0], W.shape[0], X.shape[1]
            elif op == "dgrad":
                M, N, K = dY.shape[0], W.shape[1], dY.shape[1]
            else:
                M, N, K = dY.shape[1], X.shape[1], dY.shape[0]
            r = min(rows, M)
            ii = np.repeat(np.arange(r), N)
            jj = np.tile(np.arange(N), r)
            bi = np.zeros_like(ii)
            if op == "fwd":
                oracle.gemm_fwd(X, W, sample=(bi, ii, jj))
            elif op == "dgrad":
                oracle.gemm_dgrad(dY, W, sample=(bi, ii, jj))
            else:
                oracle.gemm_wgrad(dY, X, sample=(bi, ii, jj))
            flops += 2 * r * N * K
        return flops, time.perf_counter() - t0

    if c["sec_per_row"] is None:
        f, t = run(1)  # calibration
        c["sec_per_row"] = t
    rows = max(1, int(target_s / max(c["sec_per_row"], 1e-4)))
    f, t = run(rows)
    return f, t, rows


def cpu_baseline(target_s=12.0, cfg=None):
    import oracle
    cfg = cfg or workloads.DECODER_2B
    n = len(cfg["dtypes"]) * len(step_token_counts(cfg)) * len(cfg["layers"]) * 3
    f, t, rows = oracle_sample(target_s, cfg)
    return {"value": round(f / t / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"first {rows} output row(s) of each of the {n} products ({f / 2e9:.2f} GMAC), "
                      f"fp64 naive loops, {t:.1f} s"}


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg, workload = STEP_SETS[args.set]
    steps, warm = args.steps, args.warmup
    t0 = time.perf_counter()
    # each step: a sample of the workload, sized so the whole run takes ~2 minutes
    per_step_s = max(0.5, 120.0 / max(1, steps + warm))
    total_f = total_t = 0.0
    rows = 0
    for s in range(warm + steps):
        f, t, rows = oracle_sample(per_step_s, cfg)
        if s >= warm:
            total_f += f
            total_t += t
    value = total_f / total_t / 1e12
    n = len(cfg["dtypes"]) * len(step_token_counts(cfg)) * len(cfg["layers"]) * 3
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": steps, "warmup": warm, "ms_per_step": round(1000 * total_t / steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic", "config": {"workload": workload, "parallelism": "host threads"},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.threads(),
                             "kind": "oracle",
                             "sample": f"each step: first {rows} output row(s) of all {n} products"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": round(time.perf_counter() - t0, 1)}
    print(json.dumps(line), flush=True)


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (a replicated job takes as long as its
    slowest replica); x itself when no process group with several ranks is
    up."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_step: float, steps: int, total_ms: float) -> float:
    """Whole-job throughput: every replica's work over the slowest replica's time."""
    return world * flops_per_step * steps / (total_ms / 1e3) / 1e12


# ------------------------------------------------------------------ rows
FP32_LANES_PER_SM = 128  # FP32 FMA units per SM (4 sub-partitions x 32)


def fp32_peak_tflops(sms=None, mhz=None):
    """FP32 CUDA-core peak: SMs x FMA units x 2 flop x the maximum SM clock
    (152 x 128 x 2 x 2,070 MHz = 80.5 TFLOP/s on a GB300)."""
    if sms is None:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
    if mhz is None:
        try:
            out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits", "-i", "0"],
                                 capture_output=True, text=True, timeout=20).stdout.split()
            mhz = float(out[0])
        except Exception:
            mhz = 2070.0
    return sms * FP32_LANES_PER_SM * 2 * mhz / 1e6


def bars_of(rows):
    """The rows against the targets they are held to: the smallest tensor
    fraction (rotated operands) over the 2,048- and 4,096-token products of
    the 2B-class set (target 0.70), the smallest weight-gradient / forward
    ratio (target 0.85) and the smallest HBM fraction of the rank-16 LoRA
    down, up and gradient products (target 0.70)."""
    fr = [r["frac_cold"] for r in rows if r.get("set") == "2B" and r["T"] >= 2048 and r["op"] != "wgrad_acc"]
    wf = [r["wgrad_over_fwd"] for r in rows if r.get("set") == "2B" and "wgrad_over_fwd" in r]
    lo = [r["frac_of_hbm"] for r in rows if r.get("set") == "LoRA" and r["op"] in ("down", "up", "grad")]
    out = {}
    if fr:
        out["min_tensor_frac_T2048_4096"] = min(fr)
    if wf:
        out["min_wgrad_over_fwd"] = min(wf)
    if lo:
        out["min_lora_hbm_frac"] = min(lo)
    return out


def time_calls(stream, make_call, reps=10, sets=1):
    """Median per-launch ms of one call over 5 replays of a graph of `reps`
    launches (cycling through `sets` operand sets), and its call record."""
    from gemms_linear_layers_gb300 import _binding as tg
    calls = [make_call(i) for i in range(sets)]
    for c in calls:
        c()
    torch.cuda.synchronize()
    call = tg.tg_last_call()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for r in range(reps):
            calls[r % sets]()
    res = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        res.append(a.elapsed_time(b) / reps)
    del g
    return statistics.median(res), call


def step_row(stream, pk, cfg, workload, steps=10):
    """A whole layer-set step (as the headline measures it) on its own."""
    prods = build_step("cuda", cfg=cfg)
    capture(prods, stream)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    step = capture_step(prods, stream)
    flops = sum(p.flops for p in prods)
    if step:
        total_ms = timed_steps(step, 3, steps, stream, flush)
    else:
        total_ms, _ = timed_steps_per_product(prods, 3, steps, stream, flush, None)
    tf = flops * steps / (total_ms / 1e3) / 1e12
    return {"set": "step", "workload": workload, "products": len(prods), "ms_per_step": round(total_ms / steps, 4),
            "tflops": round(tf, 1), "frac_of_peak": round(tf / pk["bf16_tflops"], 3)}


def measure_rows(stream, pk, budget_s=150.0):
    """One timing row per distinct product of the other product sets, each
    alone: CUDA graph of R launches, L2-sized buffer rotation for the
    HBM-bound ones (and, beside the warm figure, for the 2B-class products),
    median of 5 replays."""
    from gemms_linear_layers_gb300 import _binding as tg
    rows = []
    t_start = time.perf_counter()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size

    # the 135M-class step (the earlier headline) as one row
    rows.append(step_row(stream, pk, workloads.DECODER_135M, STEP_SETS["135m"][1]))
    torch.cuda.empty_cache()

    # 2B-class layers: each distinct product alone, warm (same operands every
    # launch) and cold (operand sets rotated so that the bytes between two
    # uses of a set exceed twice the L2)
    for T in workloads.DECODER_2B["T"]:
        for dtype in workloads.DECODER_2B["dtypes"]:
            for d_in, d_out, names in ((2304, 2304, "q,k,v,o"), (2304, 5760, "gate,up"), (5760, 2304, "down")):
                per_set = (T * d_in + d_out * d_in + T * d_out) * 2  # operand bytes of one set
                sets = max(1, int(2 * l2 // per_set) + 1)
                data = [inputs.layer_inputs(T, d_in, d_out, dtype, tag=f"rows{i}", device="cuda")
                        for i in range(sets)]
                outs = [{"fwd": torch.empty(T, d_out, dtype=dtype, device="cuda"),
                         "dgrad": torch.empty(T, d_in, dtype=dtype, device="cuda"),
                         "wgrad": torch.empty(d_out, d_in, dtype=dtype, device="cuda"),
                         "wgrad_acc": torch.zeros(d_out, d_in, dtype=torch.float32, device="cuda")}
                        for _ in range(sets)]
                ws = torch.empty(1 << 28, dtype=torch.uint8, device="cuda")
                res = {}
                for op in ("fwd", "dgrad", "wgrad", "wgrad_acc"):
                    def fn(i, op=op):
                        X, W, dY = data[i]
                        o = outs[i][op]
                        return {"fwd": lambda: tg.tg_gemm_fwd(X, W, Y=o, ws=ws),
                                "dgrad": lambda: tg.tg_gemm_dgrad(dY, W, dX=o, ws=ws),
                                "wgrad": lambda: tg.tg_gemm_wgrad(dY, X, dW=o, ws=ws),
                                "wgrad_acc": lambda: tg.tg_gemm_wgrad_accumulate(dY, X, o, ws=ws)}[op]
                    ms_w, call = time_calls(stream, fn, reps=10, sets=1)
                    ms_c, _ = time_calls(stream, fn, reps=max(10, 2 * sets), sets=sets)
                    M, N, K = {"fwd": (T, d_out, d_in), "dgrad": (T, d_in, d_out), "wgrad": (d_out, d_in, T),
                               "wgrad_acc": (d_out, d_in, T)}[op]
                    tf_w = workloads.flops(M, N, K) / ms_w / 1e9
                    tf_c = workloads.flops(M, N, K) / ms_c / 1e9
                    res[op] = tf_c
                    rows.append({"set": "2B", "layer": names, "T": T, "op": op, "dtype": str(dtype)[6:],
                                 "M": M, "N": N, "K": K, "us_warm": round(ms_w * 1000, 2),
                                 "us_cold": round(ms_c * 1000, 2), "tflops_cold": round(tf_c, 1),
                                 "frac_warm": round(tf_w / pk["bf16_tflops"], 3),
                                 "frac_cold": round(tf_c / pk["bf16_tflops"], 3), "bound": "tensor",
                                 "operand_sets": sets, "kernel": kernel_key(call)})
                rows[-2]["wgrad_over_fwd"] = round(res["wgrad"] / res["fwd"], 3)
                rows[-1]["acc_over_wgrad"] = round(res["wgrad_acc"] / res["wgrad"], 3)
                del data, outs, ws
                torch.cuda.empty_cache()
    # the LoRA branch added inside the layer product (one pass over the output)
    # against the product followed by the branch's read-modify-write pass
    for name, d_in, d_out in (("q", 2304, 2304), ("gate", 2304, 5760), ("down", 5760, 2304)):
        T, r, dt = 4096, 16, torch.bfloat16
        X, W, dY = inputs.layer_inputs(T, d_in, d_out, dt, tag="rowsf", device="cuda")
        _, A, B, H, _ = inputs.lora_inputs(T, d_in, d_out, r, dt, tag="rowsf", device="cuda")
        dH = inputs.normal((T, r), 0.01, torch.float32, 7, device="cuda")
        dH16, At = dH.to(dt), A.t().contiguous()
        Y = torch.empty(T, d_out, dtype=dt, device="cuda")
        dX = torch.empty(T, d_in, dtype=dt, device="cuda")
        ws = torch.empty(1 << 28, dtype=torch.uint8, device="cuda")
        pairs = {
            "fwd_lora": (lambda i: (lambda: tg.tg_gemm_fwd_lora(X, W, H, B, 2.0, Y=Y, ws=ws)),
                         lambda i: (lambda: (tg.tg_gemm_fwd(X, W, Y=Y, ws=ws), tg.tg_lora_up_add(H, B, Y, 2.0))),
                         workloads.flops(T, d_out, d_in) + workloads.flops(T, d_out, r)),
            "dgrad_lora": (lambda i: (lambda: tg.tg_gemm_dgrad_lora(dY, W, dH, A, 2.0, dX=dX, ws=ws)),
                           lambda i: (lambda: (tg.tg_gemm_dgrad(dY, W, dX=dX, ws=ws),
                                               tg.tg_lora_up_add(dH16, At, dX, 2.0))),
                           workloads.flops(T, d_in, d_out) + workloads.flops(T, d_in, r)),
        }
        for op, (fused, separate, fl) in pairs.items():
            ms_f, call = time_calls(stream, fused, reps=10)
            ms_s, _ = time_calls(stream, separate, reps=10)
            tf = fl / ms_f / 1e9
            rows.append({"set": "LoRA-fused", "layer": name, "T": T, "op": op, "dtype": "bf16", "r": r,
                         "us_fused": round(ms_f * 1000, 2), "us_product_then_add": round(ms_s * 1000, 2),
                         "speedup": round(ms_s / ms_f, 3), "tflops": round(tf, 1),
                         "frac_of_peak": round(tf / pk["bf16_tflops"], 3), "bound": "tensor",
                         "kernel": call.split(" [")[0][:80]})
        del X, W, dY, A, B, H, dH, dH16, At, Y, dX, ws
        torch.cuda.empty_cache()
    # FP32 operands (the CUDA-core FFMA kernel): the 2B-class layers at T=2048
    # and the 135M-class head, against the FP32 CUDA-core peak
    f32_peak = fp32_peak_tflops()
    for names, T, d_in, d_out in (("q,k,v,o", 2048, 2304, 2304), ("gate,up", 2048, 2304, 5760),
                                  ("down", 2048, 5760, 2304), ("head", 2048, 576, 49152)):
        dt = torch.float32
        X, W, dY = inputs.layer_inputs(T, d_in, d_out, dt, tag="rows32", device="cuda")
        outs = {"fwd": torch.empty(T, d_out, dtype=dt, device="cuda"),
                "dgrad": torch.empty(T, d_in, dtype=dt, device="cuda"),
                "wgrad": torch.empty(d_out, d_in, dtype=dt, device="cuda")}
        ws = torch.empty(1 << 28, dtype=torch.uint8, device="cuda")
        for op in ("fwd", "dgrad", "wgrad"):
            fn = {"fwd": lambda i: (lambda: tg.tg_gemm_fwd(X, W, Y=outs["fwd"], ws=ws)),
                  "dgrad": lambda i: (lambda: tg.tg_gemm_dgrad(dY, W, dX=outs["dgrad"], ws=ws)),
                  "wgrad": lambda i: (lambda: tg.tg_gemm_wgrad(dY, X, dW=outs["wgrad"], ws=ws))}[op]
            ms, call = time_calls(stream, fn, reps=5)
            M, N, K = {"fwd": (T, d_out, d_in), "dgrad": (T, d_in, d_out), "wgrad": (d_out, d_in, T)}[op]
            tf = workloads.flops(M, N, K) / ms / 1e9
            key = kernel_key(call)
            row = {"set": "FP32", "layer": names, "T": T, "op": op, "dtype": "fp32", "M": M, "N": N, "K": K,
                   "us": round(ms * 1000, 2), "tflops": round(tf, 2), "kernel": key,
                   "frac_of_fp32_alu": round(tf / f32_peak, 3)}
            if key.startswith("tc3"):
                # three bf16 parts per operand: six 16-bit MMAs per product term, so
                # the ceiling is a sixth of the 16-bit tensor peak
                row.update({"bound": "tensor (three-part split)", "peak_tflops": round(pk["bf16_tflops"] / 6, 1),
                            "frac_of_peak": round(6 * tf / pk["bf16_tflops"], 3)})
            else:
                row.update({"bound": "alu", "peak_tflops": round(f32_peak, 1), "frac_of_peak": round(tf / f32_peak, 3)})
            rows.append(row)
        del X, W, dY, outs, ws
    # rank-16 LoRA, bf16, T=4096: effective HBM bandwidth
    cfg = workloads.LORA_2B
    T, r = cfg["T"], cfg["r"]
    for name, d_in, d_out in cfg["layers"]:
        if name in ("k", "v", "o", "up"):
            continue  # same shapes as q / gate
        dt = torch.bfloat16
        big = max(d_in, d_out) * T * 2
        sets = max(1, int(2 * l2 // big) + 1)
        data = [inputs.lora_inputs(T, d_in, d_out, r, dt, tag=f"rows{i}", device="cuda") for i in range(sets)]
        Hs = [torch.empty(T, r, dtype=dt, device="cuda") for _ in range(sets)]
        Ys = [torch.empty(T, d_out, dtype=dt, device="cuda") for _ in range(sets)]
        grads = [{"dA": torch.empty(r, d_in, dtype=dt, device="cuda"),
                  "dB": torch.empty(d_out, r, dtype=dt, device="cuda"),
                  "dX": torch.empty(T, d_in, dtype=dt, device="cuda")} for _ in range(sets)]
        wsn = tg.tg_workspace_size(tg.TG_OP_LORA_GRAD, T, d_in, d_out, r, dt, dt)
        wss = [torch.empty(max(wsn, 16), dtype=torch.uint8, device="cuda") for _ in range(sets)]
        # FP32 factors (as an optimizer keeps them) with the same bf16 activations
        f32 = [inputs.lora_inputs(T, d_in, d_out, r, torch.float32, tag=f"rows{i}", device="cuda")[1:3]
               for i in range(sets)]
        grads32 = [{"dA": torch.empty(r, d_in, dtype=torch.float32, device="cuda"),
                    "dB": torch.empty(d_out, r, dtype=torch.float32, device="cuda"),
                    "dX": torch.empty(T, d_in, dtype=dt, device="cuda")} for _ in range(sets)]
        wsn32 = max(tg.tg_workspace_size(op, *dims, dt, dt) for op, dims in (
            (tg.TG_OP_LORA_DOWN_F32W, (T, d_in, r, 0)), (tg.TG_OP_LORA_UP_F32W, (T, d_out, r, 0)),
            (tg.TG_OP_LORA_GRAD_F32W, (T, d_in, d_out, r))))
        wss32 = [torch.empty(max(wsn32, 16), dtype=torch.uint8, device="cuda") for _ in range(sets)]
        specs = [
            ("down", lambda i: (lambda: tg.tg_lora_down(data[i][0], data[i][1], H=Hs[i])),
             (T * d_in + r * d_in + T * r) * 2, 2 * T * d_in * r),
            ("up", lambda i: (lambda: tg.tg_lora_up(data[i][3], data[i][2], Y=Ys[i])),
             (T * r + d_out * r + T * d_out) * 2, 2 * T * d_out * r),
            # the branch added into the base output: Y read and written
            ("up_add", lambda i: (lambda: tg.tg_lora_up_add(data[i][3], data[i][2], Ys[i], 2.0)),
             (T * r + d_out * r + 2 * T * d_out) * 2, 2 * T * d_out * r),
            # reads dY, X, H, A, B; writes dX, dA, dB
            ("grad", lambda i: (lambda: tg.tg_lora_grad(*data[i], outs=grads[i], ws=wss[i])),
             (T * d_out + 2 * T * d_in + T * r + 2 * r * d_in + 2 * d_out * r) * 2,
             4 * T * r * (d_in + d_out)),
            # the same with dX added into the base layer's input gradient: dX also read
            ("grad_add", lambda i: (lambda: tg.tg_lora_grad_add(*data[i], grads[i]["dX"], 2.0,
                                                                 outs={"dA": grads[i]["dA"], "dB": grads[i]["dB"]},
                                                                 ws=wss[i])),
             (T * d_out + 3 * T * d_in + T * r + 2 * r * d_in + 2 * d_out * r) * 2,
             4 * T * r * (d_in + d_out)),
            # FP32 factors: 4-byte A and B, read once by a split into 16-bit parts
            ("down_f32w", lambda i: (lambda: tg.tg_lora_down_f32w(data[i][0], f32[i][0], H=Hs[i], ws=wss32[i])),
             (T * d_in + T * r) * 2 + r * d_in * 4, 2 * T * d_in * r),
            ("up_f32w", lambda i: (lambda: tg.tg_lora_up_f32w(data[i][3], f32[i][1], Y=Ys[i], ws=wss32[i])),
             (T * r + T * d_out) * 2 + d_out * r * 4, 2 * T * d_out * r),
            ("grad_f32w", lambda i: (lambda: tg.tg_lora_grad_f32w(data[i][0], f32[i][0], f32[i][1], data[i][3],
                                                                  data[i][4], outs=grads32[i], ws=wss32[i])),
             (T * d_out + 2 * T * d_in + T * r) * 2 + (2 * r * d_in + 2 * d_out * r) * 4,
             4 * T * r * (d_in + d_out)),
        ]
        for op, fn, nbytes, fl in specs:
            ms, call = time_calls(stream, fn, reps=max(10, sets * 2), sets=sets)
            gbs = nbytes / ms / 1e6
            rows.append({"set": "LoRA", "layer": name, "T": T, "op": op, "dtype": "bf16", "d_in": d_in,
                         "d_out": d_out, "us": round(ms * 1000, 2), "gbs": round(gbs, 1),
                         "frac_of_hbm": round(gbs / pk["hbm_gbs"], 3), "bound": "hbm",
                         "tflops": round(fl / ms / 1e9, 2), "kernel": call.split(" [")[0][:60]})
        del data, Hs, Ys, grads, wss, f32, grads32, wss32
        torch.cuda.empty_cache()
    # attention, s = 1024 / 2048 / 4096, bf16 and fp16
    acfg = workloads.ATTENTION
    for dt in acfg["dtypes"]:
        for s in acfg["s"]:
            if time.perf_counter() - t_start > budget_s:
                break
            h, d = acfg["heads"], acfg["d"]
            # operand sets rotated so that the bytes touched between two uses of a
            # set exceed twice the L2: every launch reads from HBM
            per_set = 3 * h * s * s * 2 + 6 * h * s * d * 2
            sets = max(1, int(2 * l2 // per_set) + 1)
            ts = [inputs.attn_inputs(h, s, d, dt, tag="rows" if i == 0 else f"rows{i}", device="cuda")
                  for i in range(sets)]
            for op in ("qk", "pv", "do_vt", "pt_do", "ds_k", "dst_q"):
                a, b = inputs.ATTN_OPERANDS[op]
                ss_out = op in ("qk", "do_vt")
                Cs = [torch.empty(h, s, s if ss_out else d, dtype=dt, device="cuda") for _ in range(sets)]
                ms, call = time_calls(stream, lambda i: (lambda: tg.tg_bmm_attn(op, ts[i][a], ts[i][b], C=Cs[i])),
                                      reps=max(5, 2 * sets), sets=sets)
                t, C = ts[0], Cs[0]
                nbytes = (t[a].numel() + t[b].numel() + C.numel()) * 2
                fl = 2 * h * s * s * d
                gbs = nbytes / ms / 1e6
                rows.append({"set": "attention", "s": s, "op": op, "dtype": str(dt)[6:], "us": round(ms * 1000, 2),
                             "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 3),
                             "tflops": round(fl / ms / 1e9, 1), "bound": "hbm", "kernel": kernel_key(call),
                             "operand_sets": sets})
                del C, Cs
            # the fused forward, softmax(Q K^T / 8) V without the [s, s] matrices (tensor-bound)
            Os = [torch.empty(h, s, d, dtype=dt, device="cuda") for _ in range(sets)]
            ms, call = time_calls(stream, lambda i: (lambda: tg.tg_attn_fwd(ts[i]["Q"], ts[i]["K"], ts[i]["V"],
                                                                            O=Os[i])),
                                  reps=max(5, 2 * sets), sets=sets)
            fl = 4 * h * s * s * d
            rows.append({"set": "attention", "s": s, "op": "fused_fwd", "dtype": str(dt)[6:],
                         "us": round(ms * 1000, 2), "tflops": round(fl / ms / 1e9, 1),
                         "frac_of_peak": round(fl / ms / 1e9 / pk["bf16_tflops"], 3),
                         "bound": "tensor", "kernel": call.split(" [")[0][:40], "operand_sets": sets})
            # the fused backward: dQ, dK, dV without the [s, s] matrices (counted as its
            # four products dV, dP, dQ, dK: 8 h s^2 d flops)
            gs = [{k: torch.empty(h, s, d, dtype=dt, device="cuda") for k in ("dQ", "dK", "dV")} for _ in range(sets)]
            wsb = torch.empty(max(16, tg.tg_workspace_size(tg.TG_OP_ATTN_BWD, h, s, d, 0, dt, dt)), dtype=torch.uint8,
                              device="cuda")
            ms, call = time_calls(stream, lambda i: (lambda: tg.tg_attn_bwd(ts[i]["Q"], ts[i]["K"], ts[i]["V"],
                                                                            ts[i]["dO"], outs=gs[i], ws=wsb)),
                                  reps=max(3, 2 * sets), sets=sets)
            fl = 8 * h * s * s * d
            rows.append({"set": "attention", "s": s, "op": "fused_bwd", "dtype": str(dt)[6:],
                         "us": round(ms * 1000, 2), "tflops": round(fl / ms / 1e9, 1),
                         "frac_of_peak": round(fl / ms / 1e9 / pk["bf16_tflops"], 3),
                         "bound": "tensor", "kernel": call.split(" [")[0][:40], "operand_sets": sets})
            del Os, gs, wsb, t, ts
            torch.cuda.empty_cache()
    return rows


# ------------------------------------------------------------------ probe
PROBE_LAYOUT = {"fwd": "nt", "dgrad": "nn", "wgrad": "tn", "qk": "nt", "do_vt": "nt", "pv": "nn", "ds_k": "nn",
          "pt_do": "tn", "dst_q": "tn"}
PROBE_NAME = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}


def probe_main(argv=None):
    """`bench.py probe OP D0 D1 D2 ...`: one product through the public entry
    points, alone, optionally with a forced plan (see the module docstring)."""
    import tempfile

    from gemms_linear_layers_gb300 import _binding as tg
    ap = argparse.ArgumentParser(prog="bench.py probe")
    ap.add_argument("op")
    ap.add_argument("dims", type=int, nargs=3)
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f16", "f32"],
                    help="f32: FP32 operands and output (layer products only, CUDA-core kernel)")
    ap.add_argument("--out", default="same", choices=["same", "f32"])
    ap.add_argument("--plan", default=None, help='"bn splits [raster]"; splits may be sk')
    ap.add_argument("--reps", type=int, default=20)
    a = ap.parse_args(argv)
    dtype = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[a.dtype]
    if dtype == torch.float32 and a.op not in ("fwd", "dgrad", "wgrad"):
        raise SystemExit("--dtype f32 applies to fwd, dgrad and wgrad only")
    out_dtype = dtype if a.out == "same" else torch.float32
    dev = "cuda"
    if a.op in ("fwd", "dgrad", "wgrad"):
        T, d_in, d_out = a.dims
        X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="probe", device=dev)
        M, N, K = {"fwd": (T, d_out, d_in), "dgrad": (T, d_in, d_out), "wgrad": (d_out, d_in, T)}[a.op]
        batch = 1
        out = torch.empty(M, N, dtype=out_dtype, device=dev)
        fn = {"fwd": lambda ws: tg.tg_gemm_fwd(X, W, Y=out, ws=ws),
              "dgrad": lambda ws: tg.tg_gemm_dgrad(dY, W, dX=out, ws=ws),
              "wgrad": lambda ws: tg.tg_gemm_wgrad(dY, X, dW=out, ws=ws)}[a.op]
    elif a.op.startswith("lora"):  # rank 16; --dtype applies to the activations
        T, d_in, d_out = a.dims
        X, A, B, H, dY = inputs.lora_inputs(T, d_in, d_out, 16, dtype, tag="probe", device=dev)
        M, N, K, batch = T, 16, d_in, 1
        outs = {"dA": torch.empty(16, d_in, dtype=out_dtype, device=dev),
                "dB": torch.empty(d_out, 16, dtype=out_dtype, device=dev),
                "dX": torch.empty(T, d_in, dtype=out_dtype, device=dev)}
        Hout = torch.empty(T, 16, dtype=out_dtype, device=dev)
        Yout = torch.empty(T, d_out, dtype=out_dtype, device=dev)
        # FP32 factors (the *_f32w forms): A, B drawn in fp32, dA, dB FP32
        _, A32, B32, _, _ = inputs.lora_inputs(T, d_in, d_out, 16, torch.float32, tag="probe", device=dev)
        outs32 = {"dA": torch.empty(16, d_in, dtype=torch.float32, device=dev),
                  "dB": torch.empty(d_out, 16, dtype=torch.float32, device=dev),
                  "dX": torch.empty(T, d_in, dtype=out_dtype, device=dev)}
        fn = {"lora_down": lambda ws: tg.tg_lora_down(X, A, H=Hout, ws=ws),
              "lora_up": lambda ws: tg.tg_lora_up(H, B, Y=Yout, ws=ws),
              "lora_grad": lambda ws: tg.tg_lora_grad(X, A, B, H, dY, outs=outs, ws=ws),
              "lora_down_f32w": lambda ws: tg.tg_lora_down_f32w(X, A32, H=Hout, ws=ws),
              "lora_up_f32w": lambda ws: tg.tg_lora_up_f32w(H, B32, Y=Yout, ws=ws),
              "lora_grad_f32w": lambda ws: tg.tg_lora_grad_f32w(X, A32, B32, H, dY, outs=outs32, ws=ws)}[a.op]
        base = a.op.replace("_f32w", "")
        wb = 4 if a.op.endswith("_f32w") else 2  # bytes of a factor element
        nbytes = {"lora_down": (T * d_in + T * 16) * 2 + 16 * d_in * wb,
                  "lora_up": (T * 16 + T * d_out) * 2 + 16 * d_out * wb,
                  "lora_grad": (T * d_out + 2 * T * d_in + T * 16) * 2 + (2 * 16 * d_in + 2 * 16 * d_out) * wb}[base]
    elif a.op in ("fwd_lora", "dgrad_lora"):  # the layer product with a rank-16 LoRA branch inside it
        T, d_in, d_out = a.dims
        X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="probe", device=dev)
        _, A, B, H, _ = inputs.lora_inputs(T, d_in, d_out, 16, dtype, tag="probe", device=dev)
        dH = inputs.normal((T, 16), 0.01, torch.float32, 7, device=dev)
        M, N, K, batch = (T, d_out, d_in + 16, 1) if a.op == "fwd_lora" else (T, d_in, d_out + 16, 1)
        out = torch.empty(M, N, dtype=out_dtype, device=dev)
        fn = ((lambda ws: tg.tg_gemm_fwd_lora(X, W, H, B, 2.0, Y=out, ws=ws)) if a.op == "fwd_lora"
              else (lambda ws: tg.tg_gemm_dgrad_lora(dY, W, dH, A, 2.0, dX=out, ws=ws)))
    elif a.op == "attn_bwd":  # the fused backward (counted as its four products dV, dP, dQ, dK: 8 h s^2 d flops)
        h, s, d = a.dims
        t = inputs.attn_inputs(h, s, d, dtype, tag="probe", device=dev)
        M, N, K, batch = s, s, 4 * d, h
        outs = {k: torch.empty(h, s, d, dtype=out_dtype, device=dev) for k in ("dQ", "dK", "dV")}
        fn = lambda ws: tg.tg_attn_bwd(t["Q"], t["K"], t["V"], t["dO"], outs=outs, ws=ws)  # noqa: E731
    elif a.op == "attn_fwd":  # the fused forward (counted as its two products: 4 h s^2 d flops)
        h, s, d = a.dims
        t = inputs.attn_inputs(h, s, d, dtype, tag="probe", device=dev)
        M, N, K, batch = s, s, 2 * d, h
        out = torch.empty(h, s, d, dtype=out_dtype, device=dev)
        fn = lambda ws: tg.tg_attn_fwd(t["Q"], t["K"], t["V"], O=out)  # noqa: E731
    else:
        h, s, d = a.dims
        t = inputs.attn_inputs(h, s, d, dtype, tag="probe", device=dev)
        x, y = inputs.ATTN_OPERANDS[a.op]
        ss = a.op in ("qk", "do_vt")
        M, N, K, batch = (s, s, d, h) if ss else (s, d, s, h)
        out = torch.empty(h, s, s if ss else d, dtype=out_dtype, device=dev)
        fn = lambda ws: tg.tg_bmm_attn(a.op, t[x], t[y], C=out, ws=ws)  # noqa: E731
    if a.plan:
        f = tempfile.NamedTemporaryFile("w", suffix=".txt", delete=False)
        f.write(f"{PROBE_LAYOUT[a.op]} {PROBE_NAME[dtype]} {PROBE_NAME[out_dtype]} {M} {N} {K} {batch} {a.plan}\n")
        f.close()
        assert tg.tg_load_table(f.name) == 0
        os.unlink(f.name)
    ws = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        fn(ws)
    torch.cuda.synchronize()
    plan = tg.tg_last_call()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(a.reps):
            fn(ws)
    times = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / a.reps)
    ms = statistics.median(times)
    st = tg.tg_stream_status(stream)
    if a.op.startswith("lora"):
        print(f"{a.op} T={a.dims[0]} d_in={a.dims[1]} d_out={a.dims[2]}: {ms * 1e3:.2f} us, "
              f"{nbytes / ms / 1e6:.0f} GB/s, status {st} [{plan}]", flush=True)
    else:
        print(f"{a.op} M={M} N={N} K={K} batch={batch}: {ms * 1e3:.2f} us, "
              f"{workloads.flops(M, N, K, batch) / ms / 1e9:.0f} TFLOP/s, status {st} [{plan}]", flush=True)
    return 0 if st == 0 else 1


# ------------------------------------------------------------------ main
MODE_CONCURRENT = ("one CUDA graph per step, independent products on parallel branches; dominant class: its "
                   "launches replayed back to back, 3 rounds per replay, L2 flushed per replay")
MODE_SERIAL = ("one CUDA graph per step, products in training order; dominant class: its launches replayed "
               "back to back, 3 rounds per replay, L2 flushed per replay")
MODE_PER_PRODUCT = "one CUDA graph per product; events between them on the launching stream"


def headline(value, ms_step, world, steps, warmup, workload, token_counts, products, table, step_flops, resident,
             mode, roofline, launches, clocks):
    """The headline JSON object (e2e, cpu_baseline and bars are added to it
    afterwards); printed as the last stdout line, kept under 2 KB."""
    return {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16,fp16 (fp32 accumulate)", "data": "synthetic",
            "config": {"workload": workload, "T": token_counts, "products_per_step": products, "tile_table": table,
                       "gflop_per_step": round(step_flops / 1e9, 2), "parallelism": f"replicas x{world}",
                       "l2": f"step inputs {resident / 1e9:.2f} GB resident in HBM; L2 flushed before every step "
                             "(256 MiB write, untimed)",
                       "timing": mode},
            "roofline": roofline, "gpu_launches": launches, "clocks": clocks}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tg", choices=["tg", "reference"])
    ap.add_argument("--set", default="2b", choices=sorted(STEP_SETS),
                    help="layer set of the headline step (default: the 2B-class set at 1,024-4,096 tokens)")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-product rows of the other sets")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--per-product-graphs", action="store_true",
                    help="time with one graph per product instead of one graph per step")
    ap.add_argument("--serial-step", action="store_true",
                    help="one product at a time in training order (default: the step's independent products on "
                         "parallel graph branches)")
    ap.add_argument("--only", default=None,
                    help="comma-separated products to run, e.g. gate.fwd.T4096.bfloat16 (profiling a single kernel)")
    ap.add_argument("--rows-out", default=None, help="also write the rows to this JSON file")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args)

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()
    from gemms_linear_layers_gb300 import _binding as tg
    # the library loads its shipped tile table (or $TG_TABLE) at first use
    table = os.environ.get("TG_TABLE", tg.DEFAULT_TABLE)
    table = table if table and os.path.exists(table) else None
    pk = peaks()
    cfg, workload = STEP_SETS[args.set]
    stream = torch.cuda.Stream()
    only = set(args.only.split(",")) if args.only else None
    prods = build_step("cuda", only, cfg)
    if not prods:
        raise SystemExit(f"--only {args.only}: no such product")
    capture(prods, stream)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    step_flops = sum(p.flops for p in prods)
    seen = {}
    for p in prods:
        for n in ("X", "W", "dY"):
            seen[id(p.t[n])] = p.t[n].numel() * p.t[n].element_size()
    resident = sum(seen.values())

    # untimed probe: per-product times and the dominant launch class
    per_prod = probe_products(prods, stream, flush)
    classes = by_launch_class(prods, per_prod)
    dom_name, dom = max(classes.items(), key=lambda kv: kv[1]["ms"])
    # the headline step (the independent products side by side unless
    # --serial-step); the dominant class timed as a run of its own launches
    step = dg = None
    if not args.per_product_graphs:
        step = capture_step(prods, stream, concurrent=not args.serial_step)
        if step:
            dg = capture_dominant([p for p in prods if p.launch_class == dom_name], stream)
    mode = (MODE_PER_PRODUCT if not step else MODE_SERIAL if args.serial_step else MODE_CONCURRENT)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        if step:
            total_ms = timed_steps(step, args.warmup, args.steps, stream, flush)
            avg_launch_ms = timed_dominant(dg, args.warmup, args.steps, stream, flush)
        else:
            total_ms, dom_ms = timed_steps_per_product(prods, args.warmup, args.steps, stream, flush, dom_name)
            avg_launch_ms = dom_ms / (dom["n"] * args.steps)
    torch.cuda.synchronize()
    if world > 1:
        total_ms = max_over_ranks(total_ms, "cuda")
        torch.distributed.barrier()
    st = tg.tg_stream_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after the timed region: {tg.tg_status_string(st)}")

    ms_step = total_ms / args.steps
    value = job_tflops(world, step_flops, args.steps, total_ms)

    flops_per_launch = dom["flops"] / dom["n"]
    achieved = flops_per_launch / (avg_launch_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / pk["bf16_tflops"], 4), "traffic": profiled_traffic(dom_name),
                "kernel": dom_name, "launches_per_step": dom["n"],
                "gflop_per_launch": round(flops_per_launch / 1e9, 3),
                "peak_source": f"{pk['source']} bf16 burst (fp16 same nominal rate)",
                "ms_per_launch": round(avg_launch_ms, 5),
                "share_of_step": round(avg_launch_ms * dom["n"] / ms_step, 3)}

    launches = sum(p.launches for p in prods) * args.steps  # the step's timed region
    if dg is not None:  # and the dominant class's
        launches += dg[3] // len([p for p in prods if p.launch_class == dom_name]) * args.steps * sum(
            p.launches for p in prods if p.launch_class == dom_name)
    line = headline(value, ms_step, world, args.steps, args.warmup,
                    workload if not only else f"{workload}; only {sorted(only)}", list(step_token_counts(cfg)),
                    len(prods), os.path.relpath(table, ROOT) if table else None, step_flops, resident, mode,
                    roofline, launches, clk.summary())

    if rank == 0:
        if not args.no_e2e:
            e2e_n = min(args.steps, 3)
            ms, h2d, d2h = e2e_steps(prods, e2e_n, stream)
            line["e2e"] = {"value": round(step_flops * e2e_n / (ms / 1e3) / 1e12 * world, 2), "unit": "TFLOP/s",
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                           "ms_per_step": round(ms / e2e_n, 3)}
        if world == 1 and not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline(cfg=cfg)
        classes_ms = {k: round(v["ms"], 4) for k, v in sorted(classes.items(), key=lambda kv: -kv[1]["ms"])}
        print("row " + json.dumps({"set": "probe", "ms_per_step_by_launch_class": classes_ms}), flush=True)
        if not args.no_rows:
            del prods, step, dg
            torch.cuda.empty_cache()
            rows = measure_rows(stream, pk)
            for r in rows:
                print("row " + json.dumps(r), flush=True)
            line["bars"] = bars_of(rows)
            if args.rows_out:
                with open(args.rows_out, "w") as f:
                    json.dump(rows, f, indent=1)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    if len(sys.argv) > 1 and sys.argv[1] == "probe":
        import __graft_entry__
        __graft_entry__.build()
        sys.exit(probe_main(sys.argv[2:]))
    main()
