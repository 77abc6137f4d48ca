"""GPU parity of the FP32-input layer products (the CUDA-core FFMA kernel).

Page "Twice the training speed on a BC-250 from tuned matrix kernels",
section "Where the time went" (the three products of a linear layer, each in
its own layout; the page times their FP32 versions too) and section
"Checking the results are right" (every product against a float64 CPU
product).  FP32 operands are exact in the fp64 oracle; the output is FP32
and is held to the FP32 bound |C - C*| <= 1e-5 sum_k |a b|.
"""
import numpy as np
import pytest
import torch

import oracle
from gemms_linear_layers_gb300 import _binding as tg
from gemms_linear_layers_gb300 import inputs
from parity import assert_close, gather, sample_coords

pytestmark = pytest.mark.gpu
F32 = torch.float32
OPS = ("fwd", "dgrad", "wgrad")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gemms_linear_layers_gb300 import build
    build.build()
    tg.lib()


def run(op, X, W, dY):
    if op == "fwd":
        return tg.tg_gemm_fwd(X, W)
    if op == "dgrad":
        return tg.tg_gemm_dgrad(dY, W)
    return tg.tg_gemm_wgrad(dY, X)


def ref(op, X, W, dY, sample=None):
    if op == "fwd":
        return oracle.gemm_fwd(X, W, sample=sample)
    if op == "dgrad":
        return oracle.gemm_dgrad(dY, W, sample=sample)
    return oracle.gemm_wgrad(dY, X, sample=sample)


# (T, d_in, d_out): one element, odd sizes (scalar loads), tile edges and ragged tails,
# a width that is not a multiple of 4 (no 16-byte loads), and a long reduction that splits
LADDER = [(1, 1, 1), (7, 5, 13), (16, 16, 16), (64, 64, 64), (129, 65, 257), (1000, 999, 1001),
          (256, 4096, 128), (3000, 64, 40)]


def fp32_path(op, T, d_in, d_out):
    """'tc3' (three bf16 parts on the tensor cores) when the row pitches of both
    operands are multiples of 8 elements and the output's of 4, else 'ffma'."""
    lda, ldb, N = {"fwd": (d_in, d_in, d_out), "dgrad": (d_out, d_in, d_in), "wgrad": (d_out, d_in, d_in)}[op]
    return "tc3" if lda % 8 == 0 and ldb % 8 == 0 and N % 4 == 0 else "ffma"


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("shape", LADDER, ids=lambda s: "x".join(map(str, s)))
def test_fp32_ladder(shape, op):
    T, d_in, d_out = shape
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, F32, tag="f32")
    got = run(op, X.cuda(), W.cuda(), dY.cuda())
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    assert f" {fp32_path(op, *shape)} " in call, call
    C, S = ref(op, X, W, dY)
    assert got.dtype == F32 and tuple(got.shape) == C.shape
    assert_close(got, C, S, f"fp32 {op} {shape} [{call}]", F32)


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("shape", [(2048, 2304, 2304), (2048, 576, 49152), (4096, 2304, 5760)],
                         ids=("2b-qkvo-T2048", "135m-head", "2b-gate-T4096"))
def test_fp32_config_sizes(shape, op):
    """Configuration sizes: sampled rows, columns and elements (each an exact
    fp64 dot product), and the same bits from a second run (split-K included)."""
    T, d_in, d_out = shape
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, F32, tag="f32cfg")
    dev = [t.cuda() for t in (X, W, dY)]
    a = run(op, *dev)
    b = run(op, *dev)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    assert torch.equal(a, b), "not reproducible"
    M, N = a.shape
    co = sample_coords(M, N, rows=8, cols=8, rand=2048, seed=M + N)
    C, S = ref(op, X, W, dY, sample=co)
    assert_close(gather(a, co), C, S, f"fp32 {op} {shape} [{call}]", F32)


@pytest.mark.parametrize("op", OPS)
def test_fp32_small_integers_exact(op):
    """Integer operands in [-3, 3]: every product and partial sum is an exact
    FP32 integer, so any summation order (splits included) gives the oracle's
    value bitwise."""
    T, d_in, d_out = 2048, 576, 192  # the weight gradient splits its 2,048-long sums
    X = inputs.small_int((T, d_in), -3, 3, F32, 41)
    W = inputs.small_int((d_out, d_in), -3, 3, F32, 42)
    dY = inputs.small_int((T, d_out), -3, 3, F32, 43)
    got = run(op, X.cuda(), W.cuda(), dY.cuda())
    torch.cuda.synchronize()
    C, _ = ref(op, X, W, dY)
    assert np.array_equal(got.cpu().double().numpy(), C), tg.tg_last_call()


@pytest.mark.parametrize("shape", [(1000, 300, 200), (8192, 576, 192), (1000, 296, 200)],
                         ids=("ffma", "tensor-cores", "tensor-cores-small"))
def test_fp32_weight_gradient_accumulates(shape):
    """dW += dY^T X with FP32 operands, on the CUDA cores (a row pitch of 300
    floats) and on the tensor cores (three-part split), unsplit and split
    (added by the ordered reduction)."""
    T, d_in, d_out = shape
    X, _, dY = inputs.layer_inputs(T, d_in, d_out, F32, tag="f32acc")
    dW0 = inputs.normal((d_out, d_in), 0.5, F32, 4246)
    dW = dW0.cuda()
    tg.tg_gemm_wgrad_accumulate(dY.cuda(), X.cuda(), dW)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert f" {fp32_path('wgrad', T, d_in, d_out)} " in call, call
    C, S = oracle.gemm_wgrad(dY, X)
    base = dW0.double().numpy()
    assert_close(dW, base + C, np.abs(base) + S, f"fp32 wgrad accumulate {shape} [{call}]", F32)


def test_fp32_empty_reduction_and_sizes():
    X = torch.empty(0, 32, dtype=F32, device="cuda")
    W = torch.randn(16, 32, device="cuda")
    assert tg.tg_gemm_fwd(X, W).shape == (0, 16)
    dY = torch.empty(0, 16, dtype=F32, device="cuda")
    dW = tg.tg_gemm_wgrad(dY, X)  # K = T = 0: an empty sum is zero
    torch.cuda.synchronize()
    assert torch.count_nonzero(dW) == 0


@pytest.mark.parametrize("op", OPS)
def test_fp32_wide_exponents_on_the_tensor_cores(op):
    """FP32 operands whose magnitudes span twelve decades, with all 24
    significand bits in use: the three bf16 parts carry each value exactly, so
    the tensor-core path holds the bound wherever the magnitudes fall."""
    T, d_in, d_out = 512, 384, 256
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, F32, tag="f32wide")
    spread = lambda shape, seed: torch.pow(10.0, inputs.normal(shape, 2.0, F32, seed).clamp(-6, 6))
    X, W, dY = X * spread(X.shape, 51), W * spread(W.shape, 52), dY * spread(dY.shape, 53)
    got = run(op, X.cuda(), W.cuda(), dY.cuda())
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert " tc3 " in call, call
    C, S = ref(op, X, W, dY)
    assert_close(got, C, S, f"fp32 wide {op} [{call}]", F32)
