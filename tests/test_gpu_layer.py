"""GPU parity of the three layer products against the fp64 oracle.

Page "Twice the training speed on a BC-250 from tuned matrix kernels":
section "Where the time went" (forward, input-gradient and weight-gradient
products, each in its own layout) and section "Checking the results are
right" (shapes from 1x1x1 up to training sizes, each against a float64 CPU
product).  Every call goes through the C ABI via the ctypes binding.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from gemms_linear_layers_gb300 import _binding as tg
from gemms_linear_layers_gb300 import inputs, workloads
from parity import assert_close, exact_rne_fraction, gather, sample_coords

pytestmark = pytest.mark.gpu
DT16 = (torch.bfloat16, torch.float16)
OPS = ("fwd", "dgrad", "wgrad")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gemms_linear_layers_gb300 import build
    build.build()
    tg.lib()
    # the table the library ships (the launch configuration bench.py times)
    assert tg.tg_load_table(tg.DEFAULT_TABLE if os.path.exists(tg.DEFAULT_TABLE) else None) == 0


def run(op, X, W, dY, out_dtype):
    if op == "fwd":
        return tg.tg_gemm_fwd(X, W, out_dtype=out_dtype)
    if op == "dgrad":
        return tg.tg_gemm_dgrad(dY, W, out_dtype=out_dtype)
    return tg.tg_gemm_wgrad(dY, X, out_dtype=out_dtype)


def ref(op, X, W, dY, sample=None):
    if op == "fwd":
        return oracle.gemm_fwd(X, W, sample=sample)
    if op == "dgrad":
        return oracle.gemm_dgrad(dY, W, sample=sample)
    return oracle.gemm_wgrad(dY, X, sample=sample)


def out_shape(op, T, d_in, d_out):
    return {"fwd": (T, d_out), "dgrad": (T, d_in), "wgrad": (d_out, d_in)}[op]


def check_full(op, T, d_in, d_out, dtype, out_dtype, tag="ladder"):
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag=tag)
    got = run(op, X.cuda(), W.cuda(), dY.cuda(), out_dtype)
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    C, S = ref(op, X, W, dY)
    assert tuple(got.shape) == C.shape
    assert_close(got, C, S, f"{op} {T}x{d_in}->{d_out} {dtype}->{out_dtype} [{tg.tg_last_call()}]", out_dtype)
    return got, C


# (T, d_in, d_out): unaligned tiny shapes (CUDA-core path), tile edges and
# ragged tails in every dimension (tensor-core path), a multi-tile square
LADDER = [(1, 1, 1), (1, 8, 8), (7, 13, 5), (16, 16, 16), (64, 64, 64), (128, 64, 256),
          (129, 72, 40), (200, 136, 264), (8, 8, 8), (300, 192, 520), (1000, 1000, 1000)]


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("shape", LADDER, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("op", OPS)
def test_ladder(op, shape, dtype, out_kind):
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    check_full(op, *shape, dtype, out_dtype)


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("op", OPS)
def test_single_layer_576_to_1536(op, out_kind):
    cfg = workloads.SINGLE_LAYER
    (_, d_in, d_out), = cfg["layers"]
    dtype = torch.bfloat16
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    got, C = check_full(op, cfg["T"], d_in, d_out, dtype, out_dtype, tag="single")
    if out_dtype == dtype:
        assert exact_rne_fraction(got, C, dtype) > 0.95


@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("layer", workloads.LAYERS_135M, ids=lambda l: l[0])
@pytest.mark.parametrize("op", OPS)
def test_decoder_135m_T2048(op, layer, dtype):
    name, d_in, d_out = layer
    T = workloads.DECODER_135M["T"]
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="135m")
    got = run(op, X.cuda(), W.cuda(), dY.cuda(), dtype)
    torch.cuda.synchronize()
    M, N = out_shape(op, T, d_in, d_out)
    if M * N * (d_in if op == "fwd" else d_out if op == "dgrad" else T) <= 2 * 10 ** 9:
        C, S = ref(op, X, W, dY)
        assert_close(got, C, S, f"{op} {name} [{tg.tg_last_call()}]", dtype)
    else:
        co = sample_coords(M, N, seed=inputs.seed_for(op, name) % 1000)
        C, S = ref(op, X, W, dY, sample=co)
        assert_close(gather(got, co), C, S, f"{op} {name} sampled [{tg.tg_last_call()}]", dtype)


@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("T", workloads.DECODER_2B["T"])
@pytest.mark.parametrize("dims", [(2304, 2304), (2304, 5760), (5760, 2304)], ids=["qkvo", "gate_up", "down"])
@pytest.mark.parametrize("op", OPS)
def test_decoder_2b(op, dims, T, dtype):
    """Every product of the 2B-class set, bf16 and fp16 at every token count:
    128 full rows, 128 full columns and 8,192 random elements of the output
    against the oracle."""
    d_in, d_out = dims
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="2b")
    got = run(op, X.cuda(), W.cuda(), dY.cuda(), dtype)
    torch.cuda.synchronize()
    M, N = out_shape(op, T, d_in, d_out)
    co = sample_coords(M, N, rows=128, cols=128, rand=8192, seed=T + d_in + d_out)
    C, S = ref(op, X, W, dY, sample=co)
    assert_close(gather(got, co), C, S, f"{op} {T}x{d_in}->{d_out} sampled [{tg.tg_last_call()}]", dtype)


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", DT16)
def test_small_integers_exact(op, dtype):
    """Integer inputs: every FP32 partial sum is an exact integer, so the
    FP32 output must equal the oracle bit for bit (any summation order)."""
    T, d_in, d_out = 512, 384, 256
    X = inputs.small_int((T, d_in), -2, 2, dtype, 1)
    W = inputs.small_int((d_out, d_in), -2, 2, dtype, 2)
    dY = inputs.small_int((T, d_out), -2, 2, dtype, 3)
    got = run(op, X.cuda(), W.cuda(), dY.cuda(), torch.float32)
    C, _ = ref(op, X, W, dY)
    assert np.array_equal(got.cpu().double().numpy(), C), tg.tg_last_call()


def test_long_reduction_integers_exact_with_split():
    """Weight gradient over 16,384 tokens (split across the GPU): still exact."""
    T, d_in, d_out = 16384, 192, 128
    X = inputs.small_int((T, d_in), -1, 1, torch.bfloat16, 4)
    dY = inputs.small_int((T, d_out), -1, 1, torch.bfloat16, 5)
    got = tg.tg_gemm_wgrad(dY.cuda(), X.cuda(), out_dtype=torch.float32)
    assert "splits=1 " not in tg.tg_last_call(), tg.tg_last_call()
    C, _ = oracle.gemm_wgrad(dY, X)
    assert np.array_equal(got.cpu().double().numpy(), C)


@pytest.mark.parametrize("op", OPS)
def test_runs_are_bitwise_identical(op):
    T, d_in, d_out = 2048, 576, 1536
    X, W, dY = (t.cuda() for t in inputs.layer_inputs(T, d_in, d_out, torch.bfloat16, tag="det"))
    outs = [run(op, X, W, dY, torch.float32) for _ in range(3)]
    outs += [run(op, X, W, dY, torch.bfloat16).float() for _ in range(2)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert torch.equal(outs[3], outs[4])


def test_empty_and_zero_reduction():
    dev = "cuda"
    X = torch.zeros(0, 64, dtype=torch.bfloat16, device=dev)
    W = torch.ones(32, 64, dtype=torch.bfloat16, device=dev)
    assert tg.tg_gemm_fwd(X, W).shape == (0, 32)
    # K = 0: zeros, whatever the output held
    X = torch.zeros(16, 0, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(24, 0, dtype=torch.bfloat16, device=dev)
    Y = torch.full((16, 24), 7.0, device=dev)
    tg.tg_gemm_fwd(X, W, Y=Y, out_dtype=torch.float32)
    assert torch.count_nonzero(Y) == 0
    dY = torch.zeros(0, 24, dtype=torch.bfloat16, device=dev)
    Xe = torch.zeros(0, 16, dtype=torch.bfloat16, device=dev)
    dW = torch.full((24, 16), 3.0, dtype=torch.bfloat16, device=dev)
    tg.tg_gemm_wgrad(dY, Xe, dW=dW)
    assert torch.count_nonzero(dW) == 0


def test_workspace_too_small_is_an_error():
    T, d_in, d_out = 16384, 192, 128
    need = tg.tg_workspace_size(tg.TG_OP_GEMM_WGRAD, T, d_out, d_in, 0, torch.bfloat16, torch.bfloat16)
    assert need > 0
    dY = torch.zeros(T, d_out, dtype=torch.bfloat16, device="cuda")
    X = torch.zeros(T, d_in, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(d_out, d_in, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    import ctypes
    st = tg.lib().tg_gemm_wgrad(ctypes.c_void_p(dY.data_ptr()), ctypes.c_void_p(X.data_ptr()),
                                ctypes.c_void_p(dW.data_ptr()), T, d_out, d_in, 0, 0,
                                ctypes.c_void_p(ws.data_ptr()), need - 16,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 4


def test_bounded_wait_reports_timeout_and_context_survives():
    assert tg.tg_stream_status() == 0
    assert tg.tg_wait_probe(2000) == 0          # 2 ms wait on a barrier nothing completes
    assert tg.tg_stream_status() == 6           # TG_ERR_DEVICE_TIMEOUT, word cleared
    assert tg.tg_stream_status() == 0
    check_full("fwd", 256, 128, 192, torch.bfloat16, torch.float32, tag="after-timeout")


def test_table_entry_is_used(tmp_path):
    T, d_in, d_out = 2048, 576, 576
    p = tmp_path / "table.txt"
    p.write_text(f"fwd bf16 bf16 {T} {d_out} {d_in} 1 64 3\n")
    assert tg.tg_load_table(str(p)) == 0
    try:
        got, _ = check_full("fwd", T, d_in, d_out, torch.bfloat16, torch.bfloat16, tag="table")
        call = tg.tg_last_call()
        assert "table=hit" in call and "bn=64" in call and "splits=3" in call, call
    finally:
        assert tg.tg_load_table(None) == 0
    check_full("fwd", T, d_in, d_out, torch.bfloat16, torch.bfloat16, tag="table")
    assert "table=miss" in tg.tg_last_call()
    assert tg.tg_load_table(tg.DEFAULT_TABLE if os.path.exists(tg.DEFAULT_TABLE) else None) == 0


@pytest.mark.parametrize("op", OPS)
def test_heuristic_plans_without_table(op):
    """Shapes of the layer sets with no table loaded: the cost-model plans."""
    assert tg.tg_load_table(None) == 0
    try:
        for T, d_in, d_out in ((2048, 576, 49152), (1024, 2304, 5760)):
            X, W, dY = inputs.layer_inputs(T, d_in, d_out, torch.bfloat16, tag="heur")
            got = run(op, X.cuda(), W.cuda(), dY.cuda(), torch.bfloat16)
            assert "table=miss" in tg.tg_last_call()
            M, N = out_shape(op, T, d_in, d_out)
            co = sample_coords(M, N, rows=16, cols=16, rand=2048, seed=7)
            C, S = ref(op, X, W, dY, sample=co)
            assert_close(gather(got, co), C, S, f"{op} heuristic [{tg.tg_last_call()}]", torch.bfloat16)
    finally:
        assert tg.tg_load_table(tg.DEFAULT_TABLE if os.path.exists(tg.DEFAULT_TABLE) else None) == 0


# --------------------------------------------------------------- stream-K
SK_CASES = [
    # (op, T, d_in, d_out, bn): tiles vs 152 CTAs: fewer tiles than CTAs (every
    # tile cut into several pieces), about one tile per CTA, many tiles per CTA
    ("wgrad", 4096, 2304, 2304, 256),
    ("wgrad", 16384, 192, 128, 64),
    ("dgrad", 2048, 576, 49152, 192),
    ("fwd", 1000, 520, 1000, 128),
    ("fwd", 2048, 576, 1536, 256),
    # CTA pairs ("p"): a pair's partials come from the CTA of the same rank
    # in each later pair; ragged edges; one partial per pair and several
    ("wgrad", 4096, 2304, 2304, "256p"),
    ("wgrad", 2048, 2304, 2304, "256p"),
    ("dgrad", 2048, 576, 49152, "192p"),
    ("fwd", 1000, 520, 1000, "128p"),
    ("wgrad", 16384, 384, 256, "128p"),
]


def _with_table(line, fn):
    import tempfile
    with tempfile.NamedTemporaryFile("w", suffix=".txt", delete=False) as f:
        f.write(line + "\n")
    assert tg.tg_load_table(f.name) == 0
    try:
        return fn()
    finally:
        os.unlink(f.name)
        assert tg.tg_load_table(tg.DEFAULT_TABLE if os.path.exists(tg.DEFAULT_TABLE) else None) == 0


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("case", SK_CASES, ids=lambda c: "-".join(map(str, c)))
def test_stream_k_schedule(case, out_kind):
    op, T, d_in, d_out, bn = case
    dtype = torch.bfloat16
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    M, N = out_shape(op, T, d_in, d_out)
    K = {"fwd": d_in, "dgrad": d_out, "wgrad": T}[op]
    lay = {"fwd": "nt", "dgrad": "nn", "wgrad": "tn"}[op]
    dname = {torch.bfloat16: "bf16", torch.float32: "f32"}
    line = f"{lay} bf16 {dname[out_dtype]} {M} {N} {K} 1 {bn} sk"
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="sk")
    Xc, Wc, dYc = X.cuda(), W.cuda(), dY.cuda()

    def go():
        outs = [run(op, Xc, Wc, dYc, out_dtype) for _ in range(3)]
        return outs, tg.tg_last_call()

    outs, call = _with_table(line, go)
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    assert "sk grid=" in call and "table=hit" in call, call
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2]), "stream-K not deterministic"
    if M * N * K <= 3 * 10 ** 9:
        C, S = ref(op, X, W, dY)
        assert_close(outs[0], C, S, f"{op} stream-K [{call}]", out_dtype)
    else:
        co = sample_coords(M, N, rows=32, cols=32, rand=4096, seed=3)
        C, S = ref(op, X, W, dY, sample=co)
        assert_close(gather(outs[0], co), C, S, f"{op} stream-K sampled [{call}]", out_dtype)


@pytest.mark.parametrize("bn", ["128", "128p"])
def test_stream_k_small_integers_exact(bn):
    T, d_in, d_out = 8192, 384, 256
    X = inputs.small_int((T, d_in), -2, 2, torch.float16, 8)
    dY = inputs.small_int((T, d_out), -2, 2, torch.float16, 9)
    line = f"tn f16 f32 {d_out} {d_in} {T} 1 {bn} sk"
    got = _with_table(line, lambda: tg.tg_gemm_wgrad(dY.cuda(), X.cuda(), out_dtype=torch.float32))
    C, _ = oracle.gemm_wgrad(dY, X)
    assert np.array_equal(got.cpu().double().numpy(), C)


def test_stream_k_attention_batch():
    h, s, d = 36, 1024, 64
    t = inputs.attn_inputs(h, s, d, torch.bfloat16, tag="sk")
    line = f"tn bf16 bf16 {s} {d} {s} {h} 64 sk"
    got = _with_table(line, lambda: tg.tg_bmm_attn("pt_do", t["P"].cuda(), t["dO"].cuda()))
    call = tg.tg_last_call()
    co = sample_coords(s, d, batch=h, rows=16, cols=16, rand=2048, seed=5)
    C, S = oracle.bmm_attn("pt_do", t["P"], t["dO"], sample=co)
    assert_close(gather(got, co), C, S, f"attn pt_do stream-K [{call}]", torch.bfloat16)


@pytest.mark.parametrize("bn", ["256", "256p"])
def test_stream_k_in_replayed_cuda_graph(bn):
    """A captured stream-K launch reuses one flag value on every replay: each
    replay must still wait for this replay's partial tiles."""
    T, d_in, d_out = 2048, 2304, 2304
    line = f"tn bf16 bf16 {d_out} {d_in} {T} 1 {bn} sk"
    X, W, dY = (t.cuda() for t in inputs.layer_inputs(T, d_in, d_out, torch.bfloat16, tag="skg"))
    dW = torch.empty(d_out, d_in, dtype=torch.bfloat16, device="cuda")
    n = tg.tg_workspace_size(tg.TG_OP_GEMM_WGRAD, T, d_out, d_in, 0, torch.bfloat16, torch.bfloat16)

    def go():
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            tg.tg_gemm_wgrad(dY, X, dW=dW, ws=ws)
        torch.cuda.synchronize()
        assert "sk grid=" in tg.tg_last_call()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            tg.tg_gemm_wgrad(dY, X, dW=dW, ws=ws)
        for i in range(4):
            # new inputs in place, then replay; compare with a direct call
            dY.copy_(inputs.normal((T, d_out), 0.01, torch.bfloat16, 100 + i, device="cuda"))
            with torch.cuda.stream(stream):
                g.replay()
            torch.cuda.synchronize()
            want = tg.tg_gemm_wgrad(dY, X, ws=torch.empty(n, dtype=torch.uint8, device="cuda"))
            torch.cuda.synchronize()
            assert torch.equal(dW, want), f"replay {i} differs from a direct call"
        assert tg.tg_stream_status() == 0

    _with_table(line, go)


# 144-column tiles (a width that is not a multiple of 64: the last 16 columns
# of every tile leave through their own store box); ragged N in every layout
W144_CASES = [("fwd", 300, 200, 520), ("dgrad", 300, 520, 200), ("wgrad", 520, 296, 200),
              ("fwd", 1000, 1000, 1000)]


@pytest.mark.parametrize("splits", [1, 2])
@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("case", W144_CASES, ids=lambda c: "-".join(map(str, c)))
def test_tile_width_144(case, dtype, out_kind, splits):
    op, T, d_in, d_out = case
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    M, N = out_shape(op, T, d_in, d_out)
    K = {"fwd": d_in, "dgrad": d_out, "wgrad": T}[op]
    lay = {"fwd": "nt", "dgrad": "nn", "wgrad": "tn"}[op]
    dname = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}
    line = f"{lay} {dname[dtype]} {dname[out_dtype]} {M} {N} {K} 1 144 {splits}"
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="w144")
    got = _with_table(line, lambda: run(op, X.cuda(), W.cuda(), dY.cuda(), out_dtype))
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    assert "bn=144" in call and "table=hit" in call, call
    C, S = ref(op, X, W, dY)
    assert_close(got, C, S, f"{op} bn=144 [{call}]", out_dtype)


def test_tile_width_144_full_size_wgrad():
    """The square weight gradient of the 2B-class attention projections at
    2,048 tokens with 144-column tiles (288 tiles: about two waves)."""
    T, d_in, d_out = 2048, 2304, 2304
    line = f"tn bf16 bf16 {d_out} {d_in} {T} 1 144 1"
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, torch.bfloat16, tag="w144f")
    got = _with_table(line, lambda: tg.tg_gemm_wgrad(dY.cuda(), X.cuda()))
    call = tg.tg_last_call()
    assert "bn=144" in call, call
    co = sample_coords(d_out, d_in, rows=32, cols=32, rand=4096, seed=144)
    C, S = oracle.gemm_wgrad(dY, X, sample=co)
    assert_close(gather(got, co), C, S, f"wgrad bn=144 full size [{call}]", torch.bfloat16)


# Tail split: the tiles past the last whole wave of 152 CTAs are cut along K
# into FP32 partial tiles that a second kernel adds in split order.  Cases
# with ragged M/N edge tiles in the tail, every layout, a batch.
TAIL_CASES = [("fwd", 2000, 576, 1528, 64, 4), ("dgrad", 2048, 1536, 576, 64, 3),
              ("wgrad", 2048, 576, 2304, 64, 4), ("wgrad", 2048, 2304, 2304, 256, 4),
              # CTA pairs: 256-row tiles, a wave of 76 pairs
              ("wgrad", 4096, 2304, 2304, "256p", 13), ("fwd", 2000, 1000, 2304, "128p", 4),
              ("dgrad", 4096, 1536, 1000, "192p", 3)]


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("case", TAIL_CASES, ids=lambda c: "-".join(map(str, c)))
def test_tail_split_schedule(case, dtype, out_kind):
    op, T, d_in, d_out, bn, ts = case
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    M, N = out_shape(op, T, d_in, d_out)
    K = {"fwd": d_in, "dgrad": d_out, "wgrad": T}[op]
    lay = {"fwd": "nt", "dgrad": "nn", "wgrad": "tn"}[op]
    dname = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}
    line = f"{lay} {dname[dtype]} {dname[out_dtype]} {M} {N} {K} 1 {bn} t{ts}"
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="tail")
    Xc, Wc, dYc = X.cuda(), W.cuda(), dY.cuda()
    outs = _with_table(line, lambda: [run(op, Xc, Wc, dYc, out_dtype) for _ in range(2)])
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    assert " tail=" in call and "table=hit" in call, call
    assert torch.equal(outs[0], outs[1]), "tail split not deterministic"
    if M * N * K <= 3 * 10 ** 9:
        C, S = ref(op, X, W, dY)
        assert_close(outs[0], C, S, f"{op} tail split [{call}]", out_dtype)
    else:
        co = sample_coords(M, N, rows=32, cols=32, rand=4096, seed=7)
        C, S = ref(op, X, W, dY, sample=co)
        assert_close(gather(outs[0], co), C, S, f"{op} tail split sampled [{call}]", out_dtype)


# Cluster split-K: the K ranges of one 128 x bn tile on the CTAs of a cluster,
# their FP32 partial tiles added through distributed shared memory.  Ragged
# M, N and K (a short last range), every layout, 2 to 8 ranks.
CLUSTER_CASES = [("fwd", 2048, 1536, 576, 192, 3), ("dgrad", 2048, 576, 1536, 192, 3),
                 ("wgrad", 2048, 576, 576, 64, 8), ("wgrad", 2048, 576, 192, 64, 8),
                 ("fwd", 300, 200, 520, 128, 2), ("dgrad", 300, 520, 200, 256, 3),
                 ("wgrad", 1000, 296, 200, 64, 5), ("fwd", 1000, 1000, 1000, 64, 7)]


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("case", CLUSTER_CASES, ids=lambda c: "-".join(map(str, c)))
def test_cluster_split_schedule(case, dtype, out_kind):
    op, T, d_in, d_out, bn, cs = case
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    M, N = out_shape(op, T, d_in, d_out)
    K = {"fwd": d_in, "dgrad": d_out, "wgrad": T}[op]
    lay = {"fwd": "nt", "dgrad": "nn", "wgrad": "tn"}[op]
    dname = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}
    line = f"{lay} {dname[dtype]} {dname[out_dtype]} {M} {N} {K} 1 {bn} c{cs}"
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="cs")
    Xc, Wc, dYc = X.cuda(), W.cuda(), dY.cuda()
    outs = _with_table(line, lambda: [run(op, Xc, Wc, dYc, out_dtype) for _ in range(3)])
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    assert f"bn={bn} cs" in call and "table=hit" in call, call
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2]), "cluster split not deterministic"
    C, S = ref(op, X, W, dY)
    assert_close(outs[0], C, S, f"{op} cluster split [{call}]", out_dtype)


def test_cluster_split_small_integers_exact():
    """FP32 output of small-integer operands is exact whatever the order of
    the partial sums: the on-chip reduction must equal the oracle bitwise."""
    T, d_in, d_out = 4096, 576, 192
    X = inputs.small_int((T, d_in), -2, 2, torch.bfloat16, 21)
    dY = inputs.small_int((T, d_out), -2, 2, torch.bfloat16, 22)
    line = f"tn bf16 f32 {d_out} {d_in} {T} 1 64 c8"
    got = _with_table(line, lambda: tg.tg_gemm_wgrad(dY.cuda(), X.cuda(), out_dtype=torch.float32))
    assert " cs" in tg.tg_last_call()
    C, _ = oracle.gemm_wgrad(dY, X)
    assert np.array_equal(got.cpu().double().numpy(), C)


def test_cluster_split_attention_batch_and_graph():
    """A batch of heads (one cluster per tile of every head), replayed from a
    CUDA graph with new inputs."""
    h, s, d = 4, 512, 64
    t = inputs.attn_inputs(h, s, d, torch.bfloat16, tag="cs")
    line = f"nn bf16 bf16 {s} {d} {s} {h} 64 c4"
    P, V = t["P"].cuda(), t["V"].cuda()

    def go():
        out = tg.tg_bmm_attn("pv", P, V)
        call = tg.tg_last_call()
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        C = torch.empty_like(out)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            tg.tg_bmm_attn("pv", P, V, C=C)
        V.mul_(2)  # exact in bf16: the replay must see the new values
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        return out, C, call

    out, replayed, call = _with_table(line, go)
    assert " cs" in call, call
    C, S = oracle.bmm_attn("pv", t["P"], t["V"])
    assert_close(out, C, S, f"attn pv cluster split [{call}]", torch.bfloat16)
    assert_close(replayed, 2 * C, 2 * S, f"attn pv cluster split replay [{call}]", torch.bfloat16)


# CTA pairs: 256-row tiles computed by two CTAs of a cluster (one MMA of
# M = 256 across both SMs).  Ragged M, N and K; K-major and MN-major B halves
# of 64, 96 and 128 rows/columns; the 4-D chunked operand views (widths that
# are multiples of 64) and the per-chunk boxes (other widths); split partials.
PAIR_CASES = [("fwd", 300, 200, 520, 128, 1), ("dgrad", 300, 520, 200, 192, 1),
              ("wgrad", 520, 296, 200, 256, 1), ("fwd", 1000, 1000, 1000, 256, 2),
              ("wgrad", 1024, 512, 768, 256, 1), ("dgrad", 1024, 768, 512, 128, 3),
              ("wgrad", 1024, 576, 576, 192, 1), ("fwd", 512, 640, 384, 192, 1)]


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: "-".join(map(str, c)))
def test_cta_pair_schedule(case, dtype, out_kind):
    op, T, d_in, d_out, bn, splits = case
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    M, N = out_shape(op, T, d_in, d_out)
    K = {"fwd": d_in, "dgrad": d_out, "wgrad": T}[op]
    lay = {"fwd": "nt", "dgrad": "nn", "wgrad": "tn"}[op]
    dname = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}
    line = f"{lay} {dname[dtype]} {dname[out_dtype]} {M} {N} {K} 1 {bn}p {splits}"
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, dtype, tag="pair")
    Xc, Wc, dYc = X.cuda(), W.cuda(), dY.cuda()
    outs = _with_table(line, lambda: [run(op, Xc, Wc, dYc, out_dtype) for _ in range(2)])
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    assert f"bn={bn} pair" in call and "table=hit" in call, call
    assert torch.equal(outs[0], outs[1]), "pair schedule not deterministic"
    C, S = ref(op, X, W, dY)
    assert_close(outs[0], C, S, f"{op} pair [{call}]", out_dtype)


def test_cta_pair_attention_batch():
    """Batched scores Q K^T (four heads) on CTA pairs."""
    h, s, d = 4, 512, 64
    t = inputs.attn_inputs(h, s, d, torch.bfloat16, tag="pair")
    line = f"nt bf16 bf16 {s} {s} {d} {h} 256p 1"
    got = _with_table(line, lambda: tg.tg_bmm_attn("qk", t["Q"].cuda(), t["K"].cuda()))
    call = tg.tg_last_call()
    assert " pair" in call, call
    C, S = oracle.bmm_attn("qk", t["Q"], t["K"])
    assert_close(got, C, S, f"attn qk pair [{call}]", torch.bfloat16)


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_cta_pair_full_size_head(op):
    """The vocabulary head of the 135M-class model at 2,048 tokens on CTA
    pairs, sampled against the oracle, and replayed from a CUDA graph."""
    T, d_in, d_out = 2048, 576, 49152
    M, N = out_shape(op, T, d_in, d_out)
    K = {"fwd": d_in, "dgrad": d_out, "wgrad": T}[op]
    lay = {"fwd": "nt", "dgrad": "nn", "wgrad": "tn"}[op]
    bn, splits = {"fwd": (256, 1), "dgrad": (192, 2), "wgrad": (192, 1)}[op]
    line = f"{lay} bf16 bf16 {M} {N} {K} 1 {bn}p {splits}"
    X, W, dY = inputs.layer_inputs(T, d_in, d_out, torch.bfloat16, tag="pairhead")
    Xc, Wc, dYc = X.cuda(), W.cuda(), dY.cuda()

    def go():
        first = run(op, Xc, Wc, dYc, torch.bfloat16)
        call = tg.tg_last_call()
        out = torch.empty_like(first)
        n = tg.tg_workspace_size({"fwd": tg.TG_OP_GEMM_FWD, "dgrad": tg.TG_OP_GEMM_DGRAD,
                                  "wgrad": tg.TG_OP_GEMM_WGRAD}[op], T, d_out, d_in, 0,
                                 torch.bfloat16, torch.bfloat16)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            if op == "fwd":
                tg.tg_gemm_fwd(Xc, Wc, Y=out, ws=ws)
            elif op == "dgrad":
                tg.tg_gemm_dgrad(dYc, Wc, dX=out, ws=ws)
            else:
                tg.tg_gemm_wgrad(dYc, Xc, dW=out, ws=ws)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        return first, out, call

    first, replayed, call = _with_table(line, go)
    assert tg.tg_stream_status() == 0
    assert f"bn={bn} pair" in call, call
    assert torch.equal(first, replayed), "graph replay differs from the direct call"
    co = sample_coords(M, N, rows=32, cols=32, rand=4096, seed=256)
    C, S = ref(op, X, W, dY, sample=co)
    assert_close(gather(first, co), C, S, f"{op} head pair [{call}]", torch.bfloat16)


def test_tail_split_attention_batch():
    h, s, d = 36, 1024, 64
    t = inputs.attn_inputs(h, s, d, torch.bfloat16, tag="tail")
    line = f"tn bf16 bf16 {s} {d} {s} {h} 64 t2"
    got = _with_table(line, lambda: tg.tg_bmm_attn("pt_do", t["P"].cuda(), t["dO"].cuda()))
    call = tg.tg_last_call()
    assert " tail=" in call, call
    co = sample_coords(s, d, batch=h, rows=16, cols=16, rand=2048, seed=9)
    C, S = oracle.bmm_attn("pt_do", t["P"], t["dO"], sample=co)
    assert_close(gather(got, co), C, S, f"attn pt_do tail split [{call}]", torch.bfloat16)


def test_tail_split_small_integers_exact():
    """Integer-valued inputs: every split and the reduction are exact, so the
    result equals the oracle bit for bit."""
    T, d_in, d_out = 2048, 576, 2304
    X = inputs.small_int((T, d_in), -2, 2, torch.bfloat16, 21)
    dY = inputs.small_int((T, d_out), -2, 2, torch.bfloat16, 22)
    line = f"tn bf16 f32 {d_out} {d_in} {T} 1 64 t4"
    got = _with_table(line, lambda: tg.tg_gemm_wgrad(dY.cuda(), X.cuda(), out_dtype=torch.float32))
    assert " tail=" in tg.tg_last_call()
    C, _ = oracle.gemm_wgrad(dY, X)
    assert np.array_equal(got.cpu().double().numpy(), C)
