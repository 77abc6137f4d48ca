"""Independent products side by side, as a training step may run them.

The q, k and v projections of one layer input, and a layer's input and
weight gradients, do not depend on each other; the benchmark step runs them
on parallel streams inside one captured CUDA graph (fork and join through
events).  Each call carries its own workspace and the library keeps no other
state that two calls in flight could share, so the results must be the bits
of the same calls made one at a time (every schedule is deterministic).
Shapes: the 2B-class layers at 1,024 / 2,048 / 4,096 tokens with the shipped
tile table, which picks split-K, tail-split and whole-tile plans among them.
Page "Twice the training speed on a BC-250 from tuned matrix kernels",
section "Where the time went" (the three products of each layer).
"""
import os

import pytest
import torch

from gemms_linear_layers_gb300 import _binding as tg
from gemms_linear_layers_gb300 import inputs

pytestmark = pytest.mark.gpu

LAYERS = (("q", 2304, 2304), ("k", 2304, 2304), ("gate", 2304, 5760), ("down", 5760, 2304))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gemms_linear_layers_gb300 import build
    build.build()
    assert tg.tg_load_table(tg.DEFAULT_TABLE if os.path.exists(tg.DEFAULT_TABLE) else None) == 0


def _products(T, dtype):
    """(name, call(stream), output) for the forward, input and weight gradient
    of each layer, each with its own output buffer."""
    prods = []
    for name, d_in, d_out in LAYERS:
        X, W, dY = (t.cuda() for t in inputs.layer_inputs(T, d_in, d_out, dtype, tag=f"conc-{name}"))
        Y = torch.empty(T, d_out, dtype=dtype, device="cuda")
        dX = torch.empty(T, d_in, dtype=dtype, device="cuda")
        dW = torch.empty(d_out, d_in, dtype=dtype, device="cuda")
        prods.append((f"{name}.fwd", lambda s, X=X, W=W, Y=Y: tg.tg_gemm_fwd(X, W, Y=Y, stream=s), Y))
        prods.append((f"{name}.dgrad", lambda s, dY=dY, W=W, dX=dX: tg.tg_gemm_dgrad(dY, W, dX=dX, stream=s), dX))
        prods.append((f"{name}.wgrad", lambda s, dY=dY, X=X, dW=dW: tg.tg_gemm_wgrad(dY, X, dW=dW, stream=s), dW))
    return prods


def _side_by_side(prods, streams, main):
    """Every product on its own stream, forked from and joined to `main`."""
    fork = torch.cuda.Event()
    fork.record(main)
    for (_, call, _), s in zip(prods, streams):
        s.wait_event(fork)
        with torch.cuda.stream(s):
            call(s)
        done = torch.cuda.Event()
        done.record(s)
        main.wait_event(done)


@pytest.mark.parametrize("dtype", (torch.bfloat16, torch.float16), ids=("bf16", "fp16"))
@pytest.mark.parametrize("T", (1024, 2048, 4096))
def test_independent_products_side_by_side(T, dtype):
    prods = _products(T, dtype)
    ref = {}
    for name, call, out in prods:  # one at a time, on the default stream
        call(None)
        torch.cuda.synchronize()
        ref[name] = out.clone()
    main = torch.cuda.Stream()
    streams = [torch.cuda.Stream() for _ in prods]
    for _, _, out in prods:
        out.fill_(float("nan"))
    main.wait_stream(torch.cuda.current_stream())  # after the fills
    _side_by_side(prods, streams, main)
    torch.cuda.synchronize()
    for name, _, out in prods:
        assert torch.equal(out, ref[name]), name
        assert tg.tg_stream_status(streams[[p[0] for p in prods].index(name)]) == 0

    # the same inside one captured graph, replayed twice
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=main):
        _side_by_side(prods, streams, main)
    for _ in range(2):
        for _, _, out in prods:
            out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for name, _, out in prods:
            assert torch.equal(out, ref[name]), name
