"""On-device sweep that fills the shape-keyed tile table (tables/gb300.txt).

The analogue of the page's tuning run ("Twice the training speed on a BC-250
from tuned matrix kernels", section "Tuning the kernels": benchmark a set of
kernel designs for the list of sizes training uses and keep the winners in a
file the library reads; section "What got in the way": the winners must be
looked up with the same key they were stored under, and the speed-up has to
be confirmed through the normal call path).  Here a design is (tile width,
single CTA or CTA pair, split count or schedule, raster order) of the
tensor-core kernel; each candidate is timed
through the public entry point with a one-line table that forces it, and the
fastest per shape is written with the same key the library looks up.
Each candidate is timed as a training step meets it: by default every call
reads operands that are not in L2 (operand sets rotated beyond twice the L2
size, the state a step's products find after the previous ones streamed
their own); `--warm` times one operand set over and over instead.

Usage (on the GPU): python -m gemms_linear_layers_gb300.sweep [--out PATH] [--sets 2b,135m,attn]
"""
from __future__ import annotations

import argparse
import os
import statistics
import sys
import tempfile
import time

import torch

from . import _binding as tg
from . import inputs, workloads

HERE = os.path.dirname(os.path.abspath(__file__))
DEFAULT_OUT = os.path.join(HERE, "tables", "gb300.txt")
BNS = (64, 128, 144, 192, 256)
PAIR_BNS = (128, 192, 256)
SPLITS = (1, 2, 3, 4, 6, 8, 12, 16)


def cold_sets(set_bytes: int, warm: bool) -> int:
    """Operand sets to rotate through so that no call finds its operands in L2."""
    if warm:
        return 1
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    return max(1, min(24, 2 * l2 // max(set_bytes, 1) + 1))


class Rotating:
    """A call over `len(calls)` operand sets, taking the next set each time."""

    def __init__(self, calls):
        self.calls = calls
        self.i = 0

    @property
    def sets(self) -> int:
        return len(self.calls)

    def __call__(self):
        c = self.calls[self.i % len(self.calls)]
        self.i += 1
        return c()


def shapes(sets, warm=False):
    """(layout, M, N, K, batch, make_call) for every distinct product."""
    out = []
    seen = set()

    def add(key, make):
        if key not in seen:
            seen.add(key)
            out.append((*key, make))

    if "2b" in sets or "135m" in sets:
        groups = []
        if "135m" in sets:
            groups.append((workloads.DECODER_135M["T"], workloads.LAYERS_135M))
        if "2b" in sets:
            for T in workloads.DECODER_2B["T"]:
                groups.append((T, workloads.LAYERS_2B))
        for T, layers in groups:
            for _, d_in, d_out in layers:
                for lay, op, key in (("nt", "fwd", (T, d_out, d_in)), ("nn", "dgrad", (T, d_in, d_out)),
                                     ("tn", "wgrad", (d_out, d_in, T))):
                    add((lay, *key, 1), lambda T=T, a=d_in, b=d_out, op=op: layer_call(op, T, a, b, warm=warm))
    if "attn" in sets:
        h, d = workloads.ATTENTION["heads"], workloads.ATTENTION["d"]
        for s in workloads.ATTENTION["s"]:
            add(("nt", s, s, d, h), lambda s=s: attn_call("qk", h, s, d, warm=warm))
            add(("nn", s, d, s, h), lambda s=s: attn_call("pv", h, s, d, warm=warm))
            add(("tn", s, d, s, h), lambda s=s: attn_call("pt_do", h, s, d, warm=warm))
    return out


def layer_call(op, T, d_in, d_out, dtype=torch.bfloat16, warm=False):
    n = cold_sets((T * d_in + d_out * d_in + T * d_out) * dtype.itemsize, warm)
    ws = torch.empty(1 << 29, dtype=torch.uint8, device="cuda")
    calls = []
    for i in range(n):
        X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag=f"sweep{i}", device="cuda")
        if op == "fwd":
            Y = torch.empty(T, d_out, dtype=dtype, device="cuda")
            calls.append(lambda X=X, W=W, Y=Y: tg.tg_gemm_fwd(X, W, Y=Y, ws=ws))
        elif op == "dgrad":
            dX = torch.empty(T, d_in, dtype=dtype, device="cuda")
            calls.append(lambda dY=dY, W=W, dX=dX: tg.tg_gemm_dgrad(dY, W, dX=dX, ws=ws))
        else:
            dW = torch.empty(d_out, d_in, dtype=dtype, device="cuda")
            calls.append(lambda dY=dY, X=X, dW=dW: tg.tg_gemm_wgrad(dY, X, dW=dW, ws=ws))
    return Rotating(calls)


def attn_call(op, h, s, d, dtype=torch.bfloat16, warm=False):
    a, b = inputs.ATTN_OPERANDS[op]
    out_cols = s if op in ("qk", "do_vt") else d
    elems = {"Q": s * d, "K": s * d, "V": s * d, "dO": s * d, "P": s * s, "dS": s * s}
    n = cold_sets(h * (elems[a] + elems[b] + s * out_cols) * dtype.itemsize, warm)
    ws = torch.empty(1 << 29, dtype=torch.uint8, device="cuda")
    calls = []
    for i in range(n):
        t = inputs.attn_inputs(h, s, d, dtype, tag=f"sweep{i}", device="cuda")
        C = torch.empty(h, s, out_cols, dtype=dtype, device="cuda")
        calls.append(lambda t=t, C=C: tg.tg_bmm_attn(op, t[a], t[b], C=C, ws=ws))
    return Rotating(calls)


def time_call(call, stream, reps):
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(reps):
            call()
    res = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        res.append(a.elapsed_time(b) / reps)
    return statistics.median(res)


def candidates(M, N, K, batch, sms, stream_k=False):
    kb = -(-K // 64)
    for bn in BNS:
        tiles = batch * -(-M // 128) * -(-N // bn)
        for s in SPLITS:
            if s > kb:
                break
            kps = -(-kb // s)
            if -(-kb // kps) != s:
                continue
            if s > 1 and tiles * s > 8 * sms:
                continue
            for raster in ("m", "n"):
                yield bn, s, raster
        # tail split: whole tiles in full waves, the last partial wave cut along K
        if bn % 64 == 0 and tiles > sms and tiles % sms:
            for ts in (2, 4, 8):
                if -(-kb // -(-kb // ts)) >= 2:
                    for raster in ("m", "n"):
                        yield bn, f"t{ts}", raster
        # split-K across a cluster, added on chip: one wave of tiles x N CTAs
        if bn != 144:
            for cs in range(2, 9):
                if cs > kb or tiles * cs > sms or -(-kb // -(-kb // cs)) != cs:
                    continue
                for raster in ("m", "n"):
                    yield bn, f"c{cs}", raster
        # stream-K: an equal share of tile x K-block iterations per CTA
        # (its partial tiles are 64-column multiples)
        # (offered only on request: its CTAs wait for each other, so a table
        # entry that selects it needs the GPU to itself)
        if stream_k and bn % 64 == 0 and tiles * kb >= sms and tiles * 4 >= sms:
            for raster in ("m", "n"):
                yield bn, "sk", raster
    # CTA pairs: 256-row tiles on two SMs, data-parallel or split
    if M > 128:
        for bn in PAIR_BNS:
            tiles = batch * -(-M // 256) * -(-N // bn)
            for s in SPLITS:
                if s > kb:
                    break
                kps = -(-kb // s)
                if -(-kb // kps) != s:
                    continue
                if s > 1 and tiles * s > 4 * sms:
                    continue
                for raster in ("m", "n"):
                    yield f"{bn}p", s, raster
            if stream_k and tiles * kb >= sms // 2 and tiles * 4 >= sms // 2:
                for raster in ("m", "n"):
                    yield f"{bn}p", "sk", raster
            # tail split over the pairs' last partial wave
            pairs = sms // 2
            if tiles > pairs and tiles % pairs:
                for ts in (2, 4, 8, 13, 16):
                    if -(-kb // -(-kb // ts)) >= 2:
                        for raster in ("m", "n"):
                            yield f"{bn}p", f"t{ts}", raster


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=DEFAULT_OUT)
    ap.add_argument("--sets", default="2b,135m,attn")
    ap.add_argument("--budget-s", type=float, default=900.0)
    ap.add_argument("--only", default=None, help="comma-separated layouts or MxNxKxbatch keys to sweep")
    ap.add_argument("-v", "--verbose", action="store_true", help="print every candidate's time")
    ap.add_argument("--warm", action="store_true", help="time one operand set repeatedly (operands in L2)")
    ap.add_argument("--stream-k", action="store_true",
                    help="also offer stream-K plans (their CTAs wait for each other: the GPU must be otherwise idle)")
    args = ap.parse_args(argv)
    sets = set(args.sets.split(","))
    stream = torch.cuda.Stream()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    name = torch.cuda.get_device_name(0)
    t0 = time.time()
    lines = []
    tmpdir = tempfile.mkdtemp()
    only = set(args.only.split(",")) if args.only else None
    for layout, M, N, K, batch, make in shapes(sets, warm=args.warm):
        if only and layout not in only and f"{M}x{N}x{K}x{batch}" not in only:
            continue
        if time.time() - t0 > args.budget_s:
            print(f"budget exhausted before {layout} {M}x{N}x{K}x{batch}", flush=True)
            break
        call = make()
        flops = 2 * M * N * K * batch
        reps = max(3, min(50, int(2e13 / max(flops, 1))), call.sets)
        # the heuristic's own choice, for the record
        tg.tg_load_table(None)
        base_ms = time_call(call, stream, reps)
        base_plan = tg.tg_last_call()
        best = None
        for bn, s, raster in candidates(M, N, K, batch, sms, stream_k=args.stream_k):
            path = os.path.join(tmpdir, "one.txt")
            with open(path, "w") as f:
                f.write(f"{layout} bf16 bf16 {M} {N} {K} {batch} {bn} {s} {raster}\n")
            assert tg.tg_load_table(path) == 0
            try:
                ms = time_call(call, stream, reps)
            except Exception as e:  # a candidate that cannot run (e.g. workspace) is skipped
                print(f"  skip bn={bn} s={s} {raster}: {e}", flush=True)
                continue
            plan = tg.tg_last_call()
            assert "table=hit" in plan, plan
            if args.verbose:
                print(f"  bn={bn} splits={s} raster={raster}: {ms * 1e3:.2f} us", flush=True)
            if best is None or ms < best[0]:
                best = (ms, bn, s, raster)
        tg.tg_load_table(None)
        ms, bn, s, raster = best
        tf = flops / ms / 1e9
        temp = "warm" if call.sets == 1 and args.warm else f"cold, {call.sets} operand sets"
        print(f"{layout} {M}x{N}x{K}x{batch}: best bn={bn} splits={s} raster={raster} {ms * 1e3:.1f} us "
              f"{tf:.0f} TFLOP/s ({temp}; heuristic {base_ms * 1e3:.1f} us: {base_plan})", flush=True)
        for din in ("bf16", "f16"):
            for dout in (din, "f32"):
                lines.append(f"{layout} {din} {dout} {M} {N} {K} {batch} {bn} {s} {raster}"
                             f"   # {ms * 1e3:.1f} us {'warm' if args.warm else 'cold'}, {tf:.0f} TFLOP/s")
        del call
        torch.cuda.empty_cache()
    os.makedirs(os.path.dirname(args.out), exist_ok=True)
    if os.path.exists(args.out):
        # a sweep updates its entries and keeps every other line (shapes of
        # other sets, or left out by --only)
        swept = {" ".join(l.split()[:7]) for l in lines}
        kept = []
        for l in open(args.out):
            body = l.split("#")[0].split()
            if len(body) >= 7 and " ".join(body[:7]) not in swept:
                kept.append(l.rstrip("\n"))
        lines = kept + lines
    with open(args.out, "w") as f:
        f.write("# tile table for the tensor-core kernel: op in out M N K batch bn splits raster\n")
        f.write(f"# last written by `python -m gemms_linear_layers_gb300.sweep --sets {args.sets}"
                f"{' --warm' if args.warm else ''}` on {name} ({sms} SMs), which kept the entries of shapes it did "
                f"not time; timings are bf16 and apply to fp16 and FP32 outputs too; cold = operand sets rotated "
                f"beyond 2 x L2\n")
        for l in lines:
            f.write(l + "\n")
    print(f"wrote {len(lines)} entries to {args.out} in {time.time() - t0:.0f} s", flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
