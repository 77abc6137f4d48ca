"""The weight-gradient entry point for callers that cannot allocate.

tg_gemm_wgrad_noalloc serves code that may not call cudaMalloc or lend a
workspace (a host framework that owns all device memory through its own pool,
or a process with a fixed memory budget): it runs the same kernels as
tg_gemm_wgrad with the split-K scratch in the library's own static array.

These checks call it through the C ABI twice in a row (different shapes, so
the second call reuses scratch the first one filled) and compare its output
with the fp64 oracle's product, within the tolerance the other parity tests
use, and bit for bit with the regular entry point's output on the same plan
(both sum the split partials in the same fixed order).  The file sorts last
so that a run stopping at the first failure has already run every other
test; it also passes when run on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gemms_linear_layers_gb300 import _binding as tg
from gemms_linear_layers_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu


def _call_noalloc(dY, X, dW):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    T, d_out = dY.shape
    d_in = X.shape[1]
    return tg.lib().tg_gemm_wgrad_noalloc(ctypes.c_void_p(dY.data_ptr()), ctypes.c_void_p(X.data_ptr()),
                                          ctypes.c_void_p(dW.data_ptr()), T, d_out, d_in,
                                          tg._DT[dY.dtype], tg._DT[dW.dtype], stream)


def test_noalloc_wgrad_matches_regular_entry_point_twice_in_a_row(tmp_path):
    import os
    from gemms_linear_layers_gb300 import build
    build.build()
    # two shapes whose plans split the token reduction into FP32 partials (so
    # the scratch is used): forced by a table, whatever the shipped one picks
    cases = [(2048, 576, 576, torch.bfloat16, torch.bfloat16), (16384, 192, 128, torch.float16, torch.float32)]
    table = tmp_path / "split.txt"
    table.write_text("tn bf16 bf16 576 576 2048 1 128 4\ntn f16 f32 128 192 16384 1 64 8\n")
    assert tg.tg_load_table(str(table)) == 0
    try:
        for T, d_in, d_out, dtype, out_dtype in cases:
            need = tg.tg_workspace_size(tg.TG_OP_GEMM_WGRAD, T, d_out, d_in, 0, dtype, out_dtype)
            assert 0 < need <= 32 << 20, need
            X, _, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="noalloc")
            Xc, dYc = X.cuda(), dY.cuda()
            regular = tg.tg_gemm_wgrad(dYc, Xc, out_dtype=out_dtype)
            dW = torch.full((d_out, d_in), float("nan"), dtype=out_dtype, device="cuda")
            assert _call_noalloc(dYc, Xc, dW) == 0, tg.tg_last_call()
            torch.cuda.synchronize()
            assert tg.tg_stream_status() == 0
            C, S = oracle.gemm_wgrad(dY, X)
            assert_close(dW, C, S, f"noalloc wgrad {T}x{d_in}->{d_out} vs the oracle", out_dtype)
            assert torch.equal(dW, regular), f"noalloc wgrad {T}x{d_in}->{d_out} differs from tg_gemm_wgrad"
    finally:
        assert tg.tg_load_table(tg.DEFAULT_TABLE if os.path.exists(tg.DEFAULT_TABLE) else None) == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(tmp_path):
    """A plan whose split partials exceed the 32 MiB array is refused, and
    nothing is launched.  A one-line tile table forces 16 splits here."""
    import os
    T, d_in, d_out = 4096, 1024, 1024
    table = tmp_path / "t.txt"
    table.write_text(f"tn bf16 bf16 {d_out} {d_in} {T} 1 256 16\n")
    assert tg.tg_load_table(str(table)) == 0
    try:
        need = tg.tg_workspace_size(tg.TG_OP_GEMM_WGRAD, T, d_out, d_in, 0, torch.bfloat16, torch.bfloat16)
        assert need == 16 * d_out * d_in * 4 > 32 << 20
        dev = "cuda"
        dY = torch.zeros(T, d_out, dtype=torch.bfloat16, device=dev)
        X = torch.zeros(T, d_in, dtype=torch.bfloat16, device=dev)
        dW = torch.full((d_out, d_in), 5.0, dtype=torch.bfloat16, device=dev)
        assert _call_noalloc(dY, X, dW) == 4
        assert "static array" in tg.tg_last_call()
        torch.cuda.synchronize()
        assert bool((dW == 5.0).all())  # nothing ran
    finally:
        assert tg.tg_load_table(tg.DEFAULT_TABLE if os.path.exists(tg.DEFAULT_TABLE) else None) == 0
