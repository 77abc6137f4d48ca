"""GPU parity of the layer products with a LoRA branch added inside them.

Page "Twice the training speed on a BC-250 from tuned matrix kernels",
section "What's left": fusing the small element-wise operations; here the
LoRA branch's addition into the base layer's output (forward) and input
gradient, without a second pass over that tensor:
    tg_gemm_fwd_lora:   Y  = X W^T + scale H B^T
    tg_gemm_dgrad_lora: dX = dY W  + scale dH A     (dH FP32)
Each result is compared with the oracle's two fp64 products added in fp64,
with the bound 1e-5 (S_base + |scale| S_lora) (+ one output ulp for 16-bit
outputs).  Every call goes through the C ABI via the ctypes binding.
"""
import math
import os

import pytest
import torch

import oracle
from gemms_linear_layers_gb300 import _binding as tg
from gemms_linear_layers_gb300 import inputs
from parity import assert_close, gather, sample_coords

pytestmark = pytest.mark.gpu
DT16 = (torch.bfloat16, torch.float16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gemms_linear_layers_gb300 import build
    build.build()
    assert tg.tg_load_table(tg.DEFAULT_TABLE if os.path.exists(tg.DEFAULT_TABLE) else None) == 0


def lora_layer_inputs(T, d_in, d_out, r, dtype, tag):
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag=tag)
    _, A, B, H, _ = inputs.lora_inputs(T, d_in, d_out, r, dtype, tag=tag)
    # dH = dY B in FP32 as the LoRA gradient keeps it: drawn on its own with that spread
    dH = inputs.normal((T, r), inputs.STD_G * inputs.STD_LORA * math.sqrt(d_out), torch.float32,
                       inputs.seed_for(tag, T, d_in, d_out, r, "dH"))
    return X, W, dY, A, B, H, dH


def ref_fwd(X, W, H, B, scale, sample=None):
    C1, S1 = oracle.gemm_fwd(X, W, sample=sample)
    C2, S2 = oracle.gemm_fwd(H, B, sample=sample)
    return C1 + scale * C2, S1 + abs(scale) * S2


def ref_dgrad(dY, W, dH, A, scale, sample=None):
    C1, S1 = oracle.gemm_dgrad(dY, W, sample=sample)
    C2, S2 = oracle.gemm_dgrad(dH, A, sample=sample)
    return C1 + scale * C2, S1 + abs(scale) * S2


# (T, d_in, d_out, r): whole and ragged tiles, odd and largest ranks on the
# tensor-core path; a row pitch of 13 elements and a rank above 32 take the
# CUDA-core path
SHAPES = [(256, 128, 192, 16), (200, 136, 264, 16), (130, 72, 40, 8), (64, 64, 64, 32), (300, 192, 520, 1),
          (100, 13, 24, 16), (96, 64, 80, 48)]


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("scale", [2.0, -0.5, 0.3])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fwd_and_dgrad_with_lora(shape, scale, dtype, out_kind):
    T, d_in, d_out, r = shape
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    X, W, dY, A, B, H, dH = lora_layer_inputs(T, d_in, d_out, r, dtype, "fused")
    y = tg.tg_gemm_fwd_lora(X.cuda(), W.cuda(), H.cuda(), B.cuda(), scale, out_dtype=out_dtype)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    path = "simt" if (d_in * 2) % 16 or r > 32 else "tc"
    assert f"fwd_lora {path}" in call, call
    C, S = ref_fwd(X, W, H, B, scale)
    assert_close(y, C, S, f"fwd_lora {shape} scale={scale} [{call}]", out_dtype)
    dx = tg.tg_gemm_dgrad_lora(dY.cuda(), W.cuda(), dH.cuda(), A.cuda(), scale, out_dtype=out_dtype)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    path = "simt" if (d_in * 2) % 16 or r > 32 else "tc"
    assert f"dgrad_lora {path}" in call, call
    C, S = ref_dgrad(dY, W, dH, A, scale)
    assert_close(dx, C, S, f"dgrad_lora {shape} scale={scale} [{call}]", out_dtype)


@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("layer", [("q", 2304, 2304), ("gate", 2304, 5760), ("down", 5760, 2304)],
                         ids=lambda l: l[0])
@pytest.mark.parametrize("T", [1024, 4096])
def test_2b_layers_with_rank16_lora(T, layer, dtype):
    """The 2B-class projections with their rank-16 LoRA branch, scale 2
    (alpha 32 / r 16): 128 rows, 128 columns and 8,192 random elements of Y
    and dX against the oracle."""
    name, d_in, d_out = layer
    X, W, dY, A, B, H, dH = lora_layer_inputs(T, d_in, d_out, 16, dtype, "fused2b")
    y = tg.tg_gemm_fwd_lora(X.cuda(), W.cuda(), H.cuda(), B.cuda(), 2.0)
    call = tg.tg_last_call()
    co = sample_coords(T, d_out, seed=T + d_out)
    C, S = ref_fwd(X, W, H, B, 2.0, sample=co)
    assert_close(gather(y, co), C, S, f"fwd_lora {name} T={T} [{call}]", dtype)
    dx = tg.tg_gemm_dgrad_lora(dY.cuda(), W.cuda(), dH.cuda(), A.cuda(), 2.0)
    call = tg.tg_last_call()
    co = sample_coords(T, d_in, seed=T + d_in + 1)
    C, S = ref_dgrad(dY, W, dH, A, 2.0, sample=co)
    assert_close(gather(dx, co), C, S, f"dgrad_lora {name} T={T} [{call}]", dtype)
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0


def test_rank_zero_is_the_plain_product():
    """r = 0 runs the plain product: the same bits as tg_gemm_fwd / _dgrad."""
    T, d_in, d_out = 512, 256, 384
    X, W, dY = (t.cuda() for t in inputs.layer_inputs(T, d_in, d_out, torch.bfloat16, tag="r0"))
    H = torch.empty(T, 0, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(d_out, 0, dtype=torch.bfloat16, device="cuda")
    A = torch.empty(0, d_in, dtype=torch.bfloat16, device="cuda")
    dH = torch.empty(T, 0, dtype=torch.float32, device="cuda")
    assert torch.equal(tg.tg_gemm_fwd_lora(X, W, H, B, 3.0), tg.tg_gemm_fwd(X, W))
    assert torch.equal(tg.tg_gemm_dgrad_lora(dY, W, dH, A, 3.0), tg.tg_gemm_dgrad(dY, W))


def test_small_integers_exact():
    """Integer operands, an integer scale and integer dH: every FP32 partial
    sum is an exact integer, so the FP32 output equals the oracle bit for bit
    (both 16-bit parts of scale h carry the exact value)."""
    T, d_in, d_out, r = 384, 256, 320, 16
    X = inputs.small_int((T, d_in), -2, 2, torch.bfloat16, 11)
    W = inputs.small_int((d_out, d_in), -2, 2, torch.bfloat16, 12)
    dY = inputs.small_int((T, d_out), -2, 2, torch.bfloat16, 13)
    H = inputs.small_int((T, r), -2, 2, torch.bfloat16, 14)
    B = inputs.small_int((d_out, r), -2, 2, torch.bfloat16, 15)
    A = inputs.small_int((r, d_in), -2, 2, torch.bfloat16, 16)
    dH = inputs.small_int((T, r), -3, 3, torch.float32, 17)
    y = tg.tg_gemm_fwd_lora(X.cuda(), W.cuda(), H.cuda(), B.cuda(), 3.0, out_dtype=torch.float32)
    C, _ = ref_fwd(X, W, H, B, 3.0)
    assert torch.equal(y.cpu().double(), torch.from_numpy(C)), tg.tg_last_call()
    dx = tg.tg_gemm_dgrad_lora(dY.cuda(), W.cuda(), dH.cuda(), A.cuda(), -2.0, out_dtype=torch.float32)
    C, _ = ref_dgrad(dY, W, dH, A, -2.0)
    assert torch.equal(dx.cpu().double(), torch.from_numpy(C)), tg.tg_last_call()
