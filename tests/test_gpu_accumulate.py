"""GPU parity of the accumulating weight gradient, dW (FP32) += dY^T X.

The product is the weight gradient of page "Twice the training speed on a
BC-250 from tuned matrix kernels", section "Where the time went", with FP32
accumulation ("Tuning the kernels"); adding it into an FP32 gradient buffer
is the gradient accumulation a training step across micro-batches does.  The
expected value is the initial buffer plus the oracle's fp64 product; the FP32
tolerance covers the product's rounding and the one final addition.  Every
schedule that writes C is forced through a one-line tile table.
"""
import os
import tempfile

import numpy as np
import pytest
import torch

import oracle
from gemms_linear_layers_gb300 import _binding as tg
from gemms_linear_layers_gb300 import inputs
from parity import assert_close, gather, sample_coords

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gemms_linear_layers_gb300 import build
    build.build()
    tg.lib()
    assert tg.tg_load_table(tg.DEFAULT_TABLE if os.path.exists(tg.DEFAULT_TABLE) else None) == 0


def _with_table(line, fn):
    with tempfile.NamedTemporaryFile("w", suffix=".txt", delete=False) as f:
        f.write(line + "\n")
    assert tg.tg_load_table(f.name) == 0
    try:
        return fn()
    finally:
        os.unlink(f.name)
        assert tg.tg_load_table(tg.DEFAULT_TABLE if os.path.exists(tg.DEFAULT_TABLE) else None) == 0


# (T, d_in, d_out, table width, schedule token, record marker): every path that writes dW
CASES = [
    (1024, 576, 576, "64", "1", "splits=1"),
    (2048, 576, 576, "128", "4", "splits=4"),            # split partials, then the ordered reduction adds
    (4096, 512, 384, "256", "sk", "sk grid="),           # stream-K owners add their tile
    (2048, 2304, 2304, "256", "t4", " tail="),           # whole tiles add, tail pieces through the reduction
    (1000, 296, 200, "144", "1", "bn=144"),              # the 16-column tail store of a 144-wide tile
    (1024, 512, 768, "256p", "1", " pair"),              # CTA pairs
    (2048, 576, 1536, "192p", "3", " pair"),             # pairs with split partials
    (4096, 2304, 2304, "256p", "sk", " pair sk"),        # stream-K on pairs
    (4096, 2304, 2304, "256p", "t8", " tail="),          # tail split on pairs
    (2048, 576, 192, "64", "c4", " cs"),                 # split-K inside a cluster (on-chip sum, then the add)
]


def _check(T, d_in, d_out, dtype, dW0, got, times=1):
    X, _, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="acc")
    if d_out * d_in * T <= 3 * 10 ** 9:
        C, S = oracle.gemm_wgrad(dY, X)
        base = dW0.double().cpu().numpy()
    else:  # full rows, full columns and random elements, each an exact fp64 dot product
        co = sample_coords(d_out, d_in, rows=32, cols=32, rand=4096, seed=77)
        C, S = oracle.gemm_wgrad(dY, X, sample=co)
        base = gather(dW0, co)
        got = gather(got, co)
    assert_close(got, base + times * C, np.abs(base) + times * S, f"wgrad accumulate {T}x{d_in}->{d_out}",
                 torch.float32)


@pytest.mark.parametrize("dtype", (torch.bfloat16, torch.float16))
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c[:5])))
def test_accumulate_every_schedule(case, dtype):
    T, d_in, d_out, bn, sched, marker = case
    dname = {torch.bfloat16: "bf16", torch.float16: "f16"}[dtype]
    line = f"tn {dname} f32 {d_out} {d_in} {T} 1 {bn} {sched}"
    X, _, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="acc")
    dW0 = inputs.normal((d_out, d_in), 0.5, torch.float32, 4242, device="cuda")
    Xc, dYc = X.cuda(), dY.cuda()

    def go():
        outs = []
        for _ in range(2):  # twice from the same start: bitwise equal
            dW = dW0.clone()
            tg.tg_gemm_wgrad_accumulate(dYc, Xc, dW)
            outs.append(dW)
        return outs, tg.tg_last_call()

    (a, b), call = _with_table(line, go)
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    assert marker in call and "table=hit" in call and call.startswith("wgrad_accumulate"), call
    assert torch.equal(a, b), "accumulation not reproducible"
    _check(T, d_in, d_out, dtype, dW0, a)


def test_accumulate_cuda_core_path():
    """A row pitch that is not a multiple of 16 bytes takes the CUDA-core
    kernel, which adds as well."""
    T, d_in, d_out = 300, 300, 200  # X rows of 600 bytes
    X, _, dY = inputs.layer_inputs(T, d_in, d_out, torch.bfloat16, tag="acc")
    dW0 = inputs.normal((d_out, d_in), 0.5, torch.float32, 4243, device="cuda")
    dW = dW0.clone()
    tg.tg_gemm_wgrad_accumulate(dY.cuda(), X.cuda(), dW)
    assert tg.tg_last_call().startswith("wgrad_accumulate simt"), tg.tg_last_call()
    _check(T, d_in, d_out, torch.bfloat16, dW0, dW)


def test_accumulate_small_integers_exact():
    """Small-integer operands and buffer: every partial sum and the addition
    are exact in FP32, so the result equals the integer sum bitwise."""
    T, d_in, d_out = 4096, 384, 256
    X = inputs.small_int((T, d_in), -2, 2, torch.bfloat16, 31)
    dY = inputs.small_int((T, d_out), -2, 2, torch.bfloat16, 32)
    dW0 = inputs.small_int((d_out, d_in), -100, 100, torch.float32, 33, device="cuda")
    for line in (f"tn bf16 f32 {d_out} {d_in} {T} 1 128 4", f"tn bf16 f32 {d_out} {d_in} {T} 1 256p 1",
                 f"tn bf16 f32 {d_out} {d_in} {T} 1 64 c8", f"tn bf16 f32 {d_out} {d_in} {T} 1 128 sk"):
        dW = dW0.clone()
        _with_table(line, lambda: tg.tg_gemm_wgrad_accumulate(dY.cuda(), X.cuda(), dW))
        C, _ = oracle.gemm_wgrad(dY, X)
        assert np.array_equal(dW.cpu().double().numpy(), dW0.cpu().double().numpy() + C), line


def test_accumulate_empty_reduction_leaves_the_buffer():
    dY = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    X = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    dW0 = inputs.normal((64, 128), 1.0, torch.float32, 4244, device="cuda")
    dW = dW0.clone()
    tg.tg_gemm_wgrad_accumulate(dY, X, dW)
    torch.cuda.synchronize()
    assert torch.equal(dW, dW0)
    assert "nothing to add" in tg.tg_last_call()


def test_accumulate_in_replayed_cuda_graph():
    """A captured accumulation adds once per replay (three replays: three
    products added to the buffer)."""
    T, d_in, d_out = 2048, 576, 576
    X, _, dY = inputs.layer_inputs(T, d_in, d_out, torch.bfloat16, tag="acc")
    Xc, dYc = X.cuda(), dY.cuda()
    dW0 = inputs.normal((d_out, d_in), 0.5, torch.float32, 4245, device="cuda")
    dW = dW0.clone()
    n = tg.tg_workspace_size(tg.TG_OP_GEMM_WGRAD, T, d_out, d_in, 0, torch.bfloat16, torch.float32)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        tg.tg_gemm_wgrad_accumulate(dYc, Xc, torch.empty_like(dW), ws=ws)  # warm-up (attributes) outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        tg.tg_gemm_wgrad_accumulate(dYc, Xc, dW, ws=ws)
    dW.copy_(dW0)
    for _ in range(3):
        with torch.cuda.stream(stream):
            g.replay()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    _check(T, d_in, d_out, torch.bfloat16, dW0, dW, times=3)
