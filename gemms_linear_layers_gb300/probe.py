"""Time one product through the public entry points, optionally forcing its plan.

Used to compare schedules of a single shape and to give a profiler exactly one
kind of kernel launch:

    python -m gemms_linear_layers_gb300.probe wgrad 2048 2304 2304 [--plan "256 sk n"] [--reps 20]

`op` is fwd|dgrad|wgrad (dims: T d_in d_out; --dtype f32 for FP32 operands), one of the attention products
qk|pv|do_vt|pt_do|ds_k|dst_q or the fused attn_fwd (dims: heads s d), or lora_down|lora_up|lora_grad
(dims: T d_in d_out, rank 16).  --plan "bn splits [raster]"
writes a one-line tile table for this shape and loads it first.
"""
from __future__ import annotations

import argparse
import os
import statistics
import sys
import tempfile

import torch

from . import _binding as tg
from . import inputs, workloads

LAYOUT = {"fwd": "nt", "dgrad": "nn", "wgrad": "tn", "qk": "nt", "do_vt": "nt", "pv": "nn", "ds_k": "nn",
          "pt_do": "tn", "dst_q": "tn"}
NAME = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}


def main(argv=None):
    ap = argparse.ArgumentParser()
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
    elif a.op.startswith("lora"):
        T, d_in, d_out = a.dims
        X, A, B, H, dY = inputs.lora_inputs(T, d_in, d_out, 16, dtype, tag="probe", device=dev)
        M, N, K, batch = T, 16, d_in, 1
        outs = {"dA": torch.empty(16, d_in, dtype=out_dtype, device=dev),
                "dB": torch.empty(d_out, 16, dtype=out_dtype, device=dev),
                "dX": torch.empty(T, d_in, dtype=out_dtype, device=dev)}
        Hout = torch.empty(T, 16, dtype=out_dtype, device=dev)
        Yout = torch.empty(T, d_out, dtype=out_dtype, device=dev)
        fn = {"lora_down": lambda ws: tg.tg_lora_down(X, A, H=Hout, ws=ws),
              "lora_up": lambda ws: tg.tg_lora_up(H, B, Y=Yout, ws=ws),
              "lora_grad": lambda ws: tg.tg_lora_grad(X, A, B, H, dY, outs=outs, ws=ws)}[a.op]
        nbytes = {"lora_down": (T * d_in + 16 * d_in + T * 16) * 2,
                  "lora_up": (T * 16 + 16 * d_out + T * d_out) * 2,
                  "lora_grad": (T * d_out + 2 * T * d_in + T * 16 + 2 * 16 * d_in + 2 * 16 * d_out) * 2}[a.op]
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
        f.write(f"{LAYOUT[a.op]} {NAME[dtype]} {NAME[out_dtype]} {M} {N} {K} {batch} {a.plan}\n")
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


if __name__ == "__main__":
    sys.exit(main())
