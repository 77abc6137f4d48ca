"""GPU parity of the batched attention products and the rank-16 LoRA products.

Page "Twice the training speed on a BC-250 from tuned matrix kernels",
section "Tuning the kernels" (the rank-16 LoRA matrices and the batched
products inside attention) and section "Checking the results are right"
(batched attention checked against a float64 CPU product).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from gemms_linear_layers_gb300 import _binding as tg
from gemms_linear_layers_gb300 import inputs, workloads
from parity import assert_close, gather, sample_coords, sample_coords_every_batch

pytestmark = pytest.mark.gpu
DT16 = (torch.bfloat16, torch.float16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gemms_linear_layers_gb300 import build
    build.build()
    # the table the library ships (the launch configuration bench.py times)
    assert tg.tg_load_table(tg.DEFAULT_TABLE if os.path.exists(tg.DEFAULT_TABLE) else None) == 0


# --------------------------------------------------------------- attention
ATTN_SEED = {op: i for i, op in enumerate(oracle.ATTN_OPS)}

@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("op", oracle.ATTN_OPS)
@pytest.mark.parametrize("hsd", [(3, 256, 64), (2, 200, 64), (1, 136, 16)], ids=lambda t: "x".join(map(str, t)))
def test_attention_small(hsd, op, dtype, out_kind):
    h, s, d = hsd
    t = inputs.attn_inputs(h, s, d, dtype, tag="small")
    a, b = inputs.ATTN_OPERANDS[op]
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    got = tg.tg_bmm_attn(op, t[a].cuda(), t[b].cuda(), out_dtype=out_dtype)
    C, S = oracle.bmm_attn(op, t[a], t[b])
    assert_close(got, C, S, f"attn {op} {hsd} [{tg.tg_last_call()}]", out_dtype)


@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("s", workloads.ATTENTION["s"])
def test_attention_full_size(s, dtype):
    """36 heads, head_dim 64: all six products, sampled against the oracle:
    128 full rows and 128 full columns dealt over the heads (each head has
    at least three of each) plus 8,192 random elements."""
    h, d = workloads.ATTENTION["heads"], workloads.ATTENTION["d"]
    t = inputs.attn_inputs(h, s, d, dtype, tag="attn")
    dev = {k: v.cuda() for k, v in t.items()}
    for op in oracle.ATTN_OPS:
        a, b = inputs.ATTN_OPERANDS[op]
        got = tg.tg_bmm_attn(op, dev[a], dev[b])
        M, N = (s, s) if op in ("qk", "do_vt") else (s, d)
        co = sample_coords_every_batch(M, N, h, seed=s + ATTN_SEED[op])
        C, S = oracle.bmm_attn(op, t[a], t[b], sample=co)
        assert_close(gather(got, co), C, S, f"attn {op} s={s} [{tg.tg_last_call()}]", dtype)
        del got


# -------------------------------------------------------------------- LoRA
def lora_check(T, d_in, d_out, r, dtype, out_dtype, tag):
    X, A, B, H, dY = inputs.lora_inputs(T, d_in, d_out, r, dtype, tag=tag)
    Xc, Ac, Bc, Hc, dYc = (t.cuda() for t in (X, A, B, H, dY))
    h = tg.tg_lora_down(Xc, Ac, out_dtype=out_dtype)
    C, S = oracle.lora_down(X, A)
    assert_close(h, C, S, f"lora_down {T}x{d_in} r={r} [{tg.tg_last_call()}]", out_dtype)
    y = tg.tg_lora_up(Hc, Bc, out_dtype=out_dtype)
    C, S = oracle.lora_up(H, B)
    assert_close(y, C, S, f"lora_up {T}x{d_out} r={r} [{tg.tg_last_call()}]", out_dtype)
    g = tg.tg_lora_grad(Xc, Ac, Bc, Hc, dYc, out_dtype=out_dtype, want_dH=True)
    torch.cuda.synchronize()
    ref = oracle.lora_grad(X, A, B, H, dY)
    assert_close(g["dH"], *ref["dH"], f"lora dH {T} {d_in}->{d_out} [{tg.tg_last_call()}]", None)
    for name in ("dB", "dA", "dX"):
        assert_close(g[name], *ref[name], f"lora {name} {T} {d_in}->{d_out} [{tg.tg_last_call()}]", out_dtype)
    # without the optional dH output the results are the same bits
    g2 = tg.tg_lora_grad(Xc, Ac, Bc, Hc, dYc, out_dtype=out_dtype)
    for name in ("dA", "dB", "dX"):
        assert torch.equal(g[name], g2[name]), name


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("shape", [(256, 128, 192, 16), (200, 72, 40, 16), (130, 264, 136, 16),
                                   (64, 64, 64, 8), (33, 24, 40, 4)], ids=lambda t: "x".join(map(str, t)))
def test_lora_small(shape, dtype, out_kind):
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    lora_check(*shape, dtype, out_dtype, tag="small")


@pytest.mark.parametrize("layer", [("q", 2304, 2304), ("gate", 2304, 5760), ("down", 5760, 2304)],
                         ids=lambda l: l[0])
def test_lora_2b_T4096(layer):
    """Rank-16 LoRA on the 2B-class projections at 4,096 tokens, bf16: full check."""
    _, d_in, d_out = layer
    lora_check(workloads.LORA_2B["T"], d_in, d_out, 16, torch.bfloat16, torch.bfloat16, tag="lora2b")


def test_lora_grad_deterministic():
    T, d_in, d_out, r = 4096, 2304, 5760, 16
    t = [x.cuda() for x in inputs.lora_inputs(T, d_in, d_out, r, torch.bfloat16, tag="det")]
    a = tg.tg_lora_grad(*t, out_dtype=torch.float32, want_dH=True)
    b = tg.tg_lora_grad(*t, out_dtype=torch.float32, want_dH=True)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_lora_grad_counters_from_any_workspace_and_in_a_replayed_graph():
    """The gradient's second pass adds each column block's partials in the
    CTA that arrives last, counted on per-block counters in the workspace:
    a workspace full of garbage, and the same call replayed in a CUDA graph,
    give the same bits as the first call (the first pass clears the
    counters, the last CTA resets its block's)."""
    T, d_in, d_out, r = 4096, 2304, 2304, 16
    t = [x.cuda() for x in inputs.lora_inputs(T, d_in, d_out, r, torch.bfloat16, tag="cnt")]
    ref = tg.tg_lora_grad(*t, out_dtype=torch.float32)
    n = tg.tg_workspace_size(tg.TG_OP_LORA_GRAD, T, d_in, d_out, r, torch.bfloat16, torch.float32)
    ws = torch.full((n,), 0xA5, dtype=torch.uint8, device="cuda")
    outs = {k: torch.full_like(v, float("nan")) for k, v in ref.items()}
    got = tg.tg_lora_grad(*t, out_dtype=torch.float32, outs=outs, ws=ws)
    for k in ref:
        assert torch.equal(got[k], ref[k]), k
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            tg.tg_lora_grad(*t, out_dtype=torch.float32, outs=outs, ws=ws, stream=s)
    for _ in range(2):
        for v in outs.values():
            v.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(outs[k], ref[k]), k
    assert tg.tg_stream_status() == 0 and tg.tg_stream_status(s) == 0


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("case", [(256, 192, 16, 2.0), (130, 136, 16, -0.5), (4096, 2304, 16, 0.125),
                                  (64, 64, 8, 2.0), (33, 40, 4, 1.0)], ids=lambda c: "x".join(map(str, c)))
def test_lora_up_add_into_the_base_output(case, dtype, out_kind):
    """Y += scale H B^T: the LoRA branch added into the base layer's output
    (one rounding to Y's type).  Rank 16 takes the streaming kernel, other
    ranks the CUDA-core path."""
    import numpy as np
    T, d_out, r, scale = case
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    _, _, B, H, _ = inputs.lora_inputs(T, 64, d_out, r, dtype, tag="upadd")
    Y0 = inputs.normal((T, d_out), 0.05, out_dtype, 555)  # the base layer's output
    Hc, Bc = H.cuda(), B.cuda()
    outs = []
    for _ in range(2):  # the same start twice: the same bits
        Y = Y0.cuda()
        tg.tg_lora_up_add(Hc, Bc, Y, scale)
        outs.append(Y)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    assert ("lora_up_add stream" in call) == (r == 16), call
    C, S = oracle.lora_up(H, B)
    base = Y0.double().numpy()
    assert_close(outs[0], base + scale * C, np.abs(base) + abs(scale) * S, f"lora_up_add {T}x{d_out} r={r} [{call}]",
                 out_dtype)


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("case", [(256, 128, 192, 16, 2.0), (130, 264, 136, 16, -0.5),
                                  (4096, 2304, 5760, 16, 0.125), (64, 64, 64, 8, 2.0), (33, 24, 40, 4, 1.0)],
                         ids=lambda c: "x".join(map(str, c)))
def test_lora_grad_add_into_the_base_dgrad(case, dtype, out_kind):
    """dX += scale dH A on top of the base layer's input gradient, dA and dB
    scaled, dH unscaled (one rounding of each FP32 result).  Rank 16 takes
    the streaming kernels, other ranks the CUDA-core path."""
    import numpy as np
    T, d_in, d_out, r, scale = case
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    X, A, B, H, dY = inputs.lora_inputs(T, d_in, d_out, r, dtype, tag="gradadd")
    dX0 = inputs.normal((T, d_in), 0.002, out_dtype, 556)  # the base layer's input gradient
    dev = [t.cuda() for t in (X, A, B, H, dY)]
    outs = []
    for _ in range(2):  # the same start twice: the same bits
        outs.append(tg.tg_lora_grad_add(*dev, dX0.cuda(), scale, want_dH=True))
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    for k in outs[0]:
        assert torch.equal(outs[0][k], outs[1][k]), k
    assert ("lora_grad_add stream" in call) == (r == 16), call
    ref = oracle.lora_grad(X, A, B, H, dY)
    what = f"{T} {d_in}->{d_out} r={r} scale={scale} [{call}]"
    assert_close(outs[0]["dH"], *ref["dH"], f"lora_grad_add dH {what}", None)
    for name in ("dA", "dB"):
        C, S = ref[name]
        assert_close(outs[0][name], scale * C, abs(scale) * S, f"lora_grad_add {name} {what}", out_dtype)
    C, S = ref["dX"]
    base = dX0.double().numpy()
    assert_close(outs[0]["dX"], base + scale * C, np.abs(base) + abs(scale) * S, f"lora_grad_add dX {what}",
                 out_dtype)


@pytest.mark.parametrize("shape", [(1000, 576, 1536, 16), (100, 40, 24, 8)], ids=lambda t: "x".join(map(str, t)))
def test_lora_grad_add_unit_scale_on_zero_is_the_plain_gradient(shape):
    """scale 1 added into a zero dX multiplies and adds exactly: the bits of
    tg_lora_grad, on the streaming kernels and on the CUDA-core path."""
    dev = [t.cuda() for t in inputs.lora_inputs(*shape, torch.bfloat16, tag="unit")]
    g = tg.tg_lora_grad(*dev, want_dH=True)
    dX = torch.zeros_like(g["dX"])
    h = tg.tg_lora_grad_add(*dev, dX, 1.0, want_dH=True)
    torch.cuda.synchronize()
    for k in ("dA", "dB", "dX", "dH"):
        assert torch.equal(g[k], h[k]), k


def test_lora_grad_add_rank_zero_leaves_dX():
    T, d_in, d_out = 64, 32, 48
    X = torch.randn(T, d_in, device="cuda").to(torch.bfloat16)
    dY = torch.randn(T, d_out, device="cuda").to(torch.bfloat16)
    A = torch.empty(0, d_in, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(d_out, 0, dtype=torch.bfloat16, device="cuda")
    H = torch.empty(T, 0, dtype=torch.bfloat16, device="cuda")
    dX0 = torch.randn(T, d_in, device="cuda").to(torch.bfloat16)
    dX = dX0.clone()
    tg.tg_lora_grad_add(X, A, B, H, dY, dX, 3.0)
    torch.cuda.synchronize()
    assert torch.equal(dX, dX0)


# ------------------------------------------------------- FP32 LoRA factors
F32_SHAPES = [(256, 128, 192, 16), (130, 264, 136, 16), (4096, 2304, 5760, 16), (64, 64, 64, 8), (33, 24, 40, 4)]


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("shape", F32_SHAPES, ids=lambda t: "x".join(map(str, t)))
def test_lora_fp32_factors(shape, dtype, out_kind):
    """16-bit activations with FP32 A and B (not rounded to 16 bits): the
    down, up and gradient products against the oracle on the FP32 factors;
    dA and dB come out in FP32.  Rank 16 takes the streaming kernels with
    the factors split into hi + lo parts, other ranks the CUDA cores."""
    T, d_in, d_out, r = shape
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    X, _, _, H, dY = inputs.lora_inputs(T, d_in, d_out, r, dtype, tag="w32")
    _, A, B, _, _ = inputs.lora_inputs(T, d_in, d_out, r, torch.float32, tag="w32")
    Xc, Ac, Bc, Hc, dYc = (t.cuda() for t in (X, A, B, H, dY))
    stream_path = r == 16
    h = tg.tg_lora_down_f32w(Xc, Ac, out_dtype=out_dtype)
    call = tg.tg_last_call()
    assert ("lora_down_f32w stream" in call) == stream_path, call
    C, S = oracle.lora_down(X, A)
    assert_close(h, C, S, f"lora_down_f32w {shape} [{call}]", out_dtype)
    y = tg.tg_lora_up_f32w(Hc, Bc, out_dtype=out_dtype)
    call = tg.tg_last_call()
    assert ("lora_up_f32w stream" in call) == stream_path, call
    C, S = oracle.lora_up(H, B)
    assert_close(y, C, S, f"lora_up_f32w {shape} [{call}]", out_dtype)
    g = tg.tg_lora_grad_f32w(Xc, Ac, Bc, Hc, dYc, out_dtype=out_dtype, want_dH=True)
    g2 = tg.tg_lora_grad_f32w(Xc, Ac, Bc, Hc, dYc, out_dtype=out_dtype, want_dH=True)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    assert ("lora_grad_f32w stream" in call) == stream_path, call
    ref = oracle.lora_grad(X, A, B, H, dY)
    assert_close(g["dH"], *ref["dH"], f"lora_grad_f32w dH {shape} [{call}]", None)
    for name in ("dA", "dB"):
        assert g[name].dtype == torch.float32
        assert_close(g[name], *ref[name], f"lora_grad_f32w {name} {shape} [{call}]", torch.float32)
    assert_close(g["dX"], *ref["dX"], f"lora_grad_f32w dX {shape} [{call}]", out_dtype)
    for k in g:
        assert torch.equal(g[k], g2[k]), k


@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("g", [1e-4, 1e-6])
def test_lora_grad_small_output_gradients(g, dtype):
    """Output gradients far below the config's N(0, 1e-2): the FP32 dH = dY B
    enters the 16-bit MMAs of dA and dX as hi + lo parts with the lo part
    stored times 2^11, which keeps fp16's lo part out of its subnormal range,
    so the relative bound holds at every gradient size (and bf16 is
    unchanged).  Full check at a 2B-class width."""
    T, d_in, d_out, r = 1024, 2304, 2304, 16
    X, A, B, H, _ = inputs.lora_inputs(T, d_in, d_out, r, dtype, tag="smallg")
    dY = inputs.normal((T, d_out), g, dtype, inputs.seed_for("smallg", g, str(dtype)))
    got = tg.tg_lora_grad(*(t.cuda() for t in (X, A, B, H, dY)), out_dtype=torch.float32, want_dH=True)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    ref = oracle.lora_grad(X, A, B, H, dY)
    for name in ("dH", "dB", "dA", "dX"):
        assert_close(got[name], *ref[name], f"lora_grad dY~N(0,{g}) {name} [{call}]", None)


@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("w", [1e-4, 1e-5])
def test_lora_fp32_factors_small(w, dtype):
    """FP32 factors far smaller than N(0, 0.02): their lo parts (stored times
    2^11) keep their precision in fp16 down to the range the header states
    (|w| above about 1.5e-6: a hi part in fp16's subnormal range carries 2^-25
    absolutely, the scaled lo part 2^-36), so down, up and the gradient hold
    the relative bound."""
    T, d_in, d_out, r = 1024, 2304, 2304, 16
    X, _, _, H, dY = inputs.lora_inputs(T, d_in, d_out, r, dtype, tag="w32s")
    A = inputs.normal((r, d_in), w, torch.float32, inputs.seed_for("w32s", w, "A"))
    B = inputs.normal((d_out, r), w, torch.float32, inputs.seed_for("w32s", w, "B"))
    Xc, Ac, Bc, Hc, dYc = (t.cuda() for t in (X, A, B, H, dY))
    h = tg.tg_lora_down_f32w(Xc, Ac, out_dtype=torch.float32)
    C, S = oracle.lora_down(X, A)
    assert_close(h, C, S, f"lora_down_f32w A~N(0,{w}) [{tg.tg_last_call()}]", None)
    y = tg.tg_lora_up_f32w(Hc, Bc, out_dtype=torch.float32)
    C, S = oracle.lora_up(H, B)
    assert_close(y, C, S, f"lora_up_f32w B~N(0,{w}) [{tg.tg_last_call()}]", None)
    got = tg.tg_lora_grad_f32w(Xc, Ac, Bc, Hc, dYc, out_dtype=torch.float32, want_dH=True)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    ref = oracle.lora_grad(X, A, B, H, dY)
    for name in ("dH", "dB", "dA", "dX"):
        assert_close(got[name], *ref[name], f"lora_grad_f32w factors~N(0,{w}) {name} [{call}]", None)


def test_lora_fp32_factors_use_the_low_part():
    """With FP32 outputs the error against the FP32 factors is far below what
    rounding the factors to bf16 first would give: the lo parts are used."""
    T, d_in, d_out, r = 4096, 2304, 2304, 16
    X, _, _, H, dY = inputs.lora_inputs(T, d_in, d_out, r, torch.bfloat16, tag="w32lo")
    _, A, B, _, _ = inputs.lora_inputs(T, d_in, d_out, r, torch.float32, tag="w32lo")
    h = tg.tg_lora_down_f32w(X.cuda(), A.cuda(), out_dtype=torch.float32).cpu().double().numpy()
    y = tg.tg_lora_up_f32w(H.cuda(), B.cuda(), out_dtype=torch.float32).cpu().double().numpy()
    for got, exact, rounded in ((h, oracle.lora_down(X, A)[0], oracle.lora_down(X, A.to(torch.bfloat16))[0]),
                                (y, oracle.lora_up(H, B)[0], oracle.lora_up(H, B.to(torch.bfloat16))[0])):
        err = np.abs(got - exact).max()
        err_rounded = np.abs(rounded - exact).max()
        assert err < 0.02 * err_rounded, (err, err_rounded)


# ------------------------------------------------------ fused attention forward
ATTN_SCALE = 0.125  # 1 / sqrt(64)


def attn_scale(S, E, scale=ATTN_SCALE):
    """Error scale of the fused forward: the products' 1e-5 S_O plus the FP32
    rounding of each logit (64 terms, at most 64 * 2^-24 * E) carried through
    the exponential, twice over (the row's normaliser too): the bound is
    (1e-5 + 2 scale 64 2^-24 E) S_O, written as 1e-5 times the value returned."""
    return S * (1.0 + (2.0 * scale * 64 * 2.0 ** -24 * np.asarray(E))[..., None] / 1e-5)


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("hs", [(2, 256), (3, 200), (1, 65), (1, 1), (2, 130)], ids=lambda t: "x".join(map(str, t)))
def test_attn_fwd_small(hs, dtype, out_kind):
    """Fused softmax(scale Q K^T) V against the oracle, full check: whole and
    ragged key blocks, a single key, rows past the last whole query block."""
    h, s = hs
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    t = inputs.attn_inputs(h, s, 64, dtype, tag="fused")
    got = tg.tg_attn_fwd(t["Q"].cuda(), t["K"].cuda(), t["V"].cuda(), out_dtype=out_dtype)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert "attn_fwd fused" in call, call
    O, S, E = oracle.attn_fwd(t["Q"], t["K"], t["V"], ATTN_SCALE)
    assert_close(got, O, attn_scale(S, E), f"attn_fwd {hs} [{call}]", out_dtype)


@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("s", workloads.ATTENTION["s"])
def test_attn_fwd_full_size(s, dtype):
    """36 heads, head_dim 64, bf16 and fp16: sampled rows (each a full softmax
    over all keys) against the oracle, and the same bits from a second run."""
    h, d = workloads.ATTENTION["heads"], workloads.ATTENTION["d"]
    t = inputs.attn_inputs(h, s, d, dtype, tag="attn")
    dev = [t[n].cuda() for n in ("Q", "K", "V")]
    a = tg.tg_attn_fwd(*dev, out_dtype=torch.float32)
    b = tg.tg_attn_fwd(*dev, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    rng = np.random.default_rng(s)
    hh = np.concatenate([rng.integers(0, h, 384), [0, h - 1, 0, h - 1]])
    ii = np.concatenate([rng.integers(0, s, 384), [0, 0, s - 1, s - 1]])
    O, S, E = oracle.attn_fwd(t["Q"], t["K"], t["V"], ATTN_SCALE, rows=(hh, ii))
    got = a[torch.from_numpy(hh).cuda(), torch.from_numpy(ii).cuda()]
    assert_close(got, O, attn_scale(S, E), f"attn_fwd s={s}", torch.float32)


@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("scale", [1.0, -0.5, 3.0])
def test_attn_fwd_running_maximum_refreshed(scale, dtype):
    """Logits with a spread of tens (scale 1 to 3 on N(0,1) inputs, and keys
    whose size grows along the sequence): the running maximum of a row is
    overtaken block after block, so the partial output and sum are rescaled
    many times, and most weights are far below the row's largest (fp16 keeps
    their low parts).  Full check against the oracle."""
    h, s, d = 2, 1000, 64
    t = inputs.attn_inputs(h, s, d, dtype, tag="refresh")
    grow = torch.linspace(0.25, 2.0, s).reshape(1, s, 1)
    K = (t["K"].float() * grow).to(dtype)
    got = tg.tg_attn_fwd(t["Q"].cuda(), K.cuda(), t["V"].cuda(), scale=scale, out_dtype=torch.float32)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    O, S, E = oracle.attn_fwd(t["Q"], K, t["V"], scale)
    assert_close(got, O, attn_scale(S, E, abs(scale)), f"attn_fwd scale={scale} [{call}]", torch.float32)


def logit_terms_max(Q, K):
    """Per head, the largest sum_k |q_ik k_jk| over query i and key j (the
    size of the largest logit's terms)."""
    q, k = np.abs(oracle.decode(Q)), np.abs(oracle.decode(K))
    return np.array([(q[h] @ k[h].T).max() for h in range(q.shape[0])])


def attn_bwd_scale(S, E, scale):
    """Error scale of the fused backward: the products' 1e-5 times the
    oracle's sums of absolute terms, plus the FP32 rounding of the logits
    (at most 64 2^-24 E each) carried through the probabilities into dV, dS
    and D (four times over, generously); E per head, broadcast over rows."""
    E = np.asarray(E, dtype=np.float64).reshape(-1, 1, 1)
    return S * (1.0 + 4.0 * abs(scale) * 64 * 2.0 ** -24 * E / 1e-5)


def check_attn_bwd(t, scale, out_dtype, what, heads=None, dO=None):
    Q, K, V = t["Q"], t["K"], t["V"]
    dO = t["dO"] if dO is None else dO
    got = tg.tg_attn_bwd(Q.cuda(), K.cuda(), V.cuda(), dO.cuda(), scale=scale, out_dtype=out_dtype)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert tg.tg_stream_status() == 0
    assert "attn_bwd fused" in call, call
    for h in (range(Q.shape[0]) if heads is None else heads):
        sl = slice(h, h + 1)
        ref = oracle.attn_bwd(Q[sl], K[sl], V[sl], dO[sl], scale)
        E = logit_terms_max(Q[sl], K[sl])
        for name in ("dQ", "dK", "dV"):
            C, S = ref[name]
            assert_close(got[name][sl], C, attn_bwd_scale(S, E, scale), f"{what} {name} head {h} [{call}]",
                         out_dtype)
    return got


@pytest.mark.parametrize("out_kind", ["f32", "same"])
@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("hs", [(2, 256), (3, 200), (1, 65), (1, 1), (2, 130), (1, 384)],
                         ids=lambda t: "x".join(map(str, t)))
def test_attn_bwd_small(hs, dtype, out_kind):
    """Fused backward (dQ, dK, dV of <dO, softmax(scale Q K^T) V>) against the
    oracle's chain rule in fp64, every element: whole and ragged blocks of
    queries and keys, a single position."""
    h, s = hs
    out_dtype = torch.float32 if out_kind == "f32" else dtype
    t = inputs.attn_inputs(h, s, 64, dtype, tag="fusedbwd")
    check_attn_bwd(t, ATTN_SCALE, out_dtype, f"attn_bwd {hs}")


@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("s", workloads.ATTENTION["s"])
def test_attn_bwd_full_size(s, dtype):
    """36 heads, head_dim 64: every element of dQ, dK and dV of three heads
    (first, middle, last) against the oracle, and the same bits from a
    second run."""
    h, d = workloads.ATTENTION["heads"], workloads.ATTENTION["d"]
    t = inputs.attn_inputs(h, s, d, dtype, tag="attn")
    a = check_attn_bwd(t, ATTN_SCALE, torch.float32, f"attn_bwd s={s}", heads=(0, h // 2, h - 1))
    b = tg.tg_attn_bwd(t["Q"].cuda(), t["K"].cuda(), t["V"].cuda(), t["dO"].cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("scale", [1.0, -0.5, 3.0])
def test_attn_bwd_wide_logits(scale, dtype):
    """Logits with a spread of tens and keys growing along the sequence (as
    in the forward's refresh test): the row statistics' running maximum is
    overtaken block after block and most probabilities are far below the
    row's largest.  Full check."""
    h, s, d = 2, 1000, 64
    t = dict(inputs.attn_inputs(h, s, d, dtype, tag="refreshbwd"))
    grow = torch.linspace(0.25, 2.0, s).reshape(1, s, 1)
    t["K"] = (t["K"].float() * grow).to(dtype)
    check_attn_bwd(t, scale, torch.float32, f"attn_bwd scale={scale}")


@pytest.mark.parametrize("dtype", DT16)
@pytest.mark.parametrize("g", [1e-4, 1e-7, 30.0])
def test_attn_bwd_gradient_magnitudes(g, dtype):
    """Output gradients far smaller and far larger than the config's N(0, 1e-2):
    the power-of-two scaling of dS keeps fp16's hi + lo parts out of its
    subnormal range and below its overflow, so the bound holds at every size."""
    h, s, d = 2, 300, 64
    t = inputs.attn_inputs(h, s, d, dtype, tag="gscale")
    dO = inputs.normal((h, s, d), g, dtype, inputs.seed_for("gscale", g, str(dtype), "dO"))
    check_attn_bwd(t, ATTN_SCALE, torch.float32, f"attn_bwd dO~N(0,{g})", dO=dO)


def test_attn_fwd_zero_scale_is_the_mean():
    """A zero scale weighs every key alike: O is the mean of V's rows."""
    h, s, d = 2, 300, 64
    t = inputs.attn_inputs(h, s, d, torch.bfloat16, tag="fused0")
    got = tg.tg_attn_fwd(t["Q"].cuda(), t["K"].cuda(), t["V"].cuda(), scale=0.0, out_dtype=torch.float32)
    mean = t["V"].double().mean(dim=1, keepdim=True).expand(h, s, d).numpy()
    S = t["V"].double().abs().mean(dim=1, keepdim=True).expand(h, s, d).numpy()
    assert_close(got, mean, S, "attn_fwd scale 0", torch.float32)


def test_lora_up_fp32_factor_unaligned_takes_the_cuda_cores():
    """The up product reads an FP32 B with 16-byte loads; a B that starts 4
    bytes past a 16-byte boundary goes to the CUDA-core path, same result."""
    T, d_out, r = 256, 192, 16
    _, _, _, H, _ = inputs.lora_inputs(T, 64, d_out, r, torch.bfloat16, tag="w32u")
    _, _, B, _, _ = inputs.lora_inputs(T, 64, d_out, r, torch.float32, tag="w32u")
    buf = torch.empty(d_out * r + 1, dtype=torch.float32, device="cuda")
    Bu = buf[1:].view(d_out, r)
    Bu.copy_(B.cuda())
    y = tg.tg_lora_up_f32w(H.cuda(), Bu, out_dtype=torch.float32)
    call = tg.tg_last_call()
    torch.cuda.synchronize()
    assert "simt" in call, call
    C, S = oracle.lora_up(H, B)
    assert_close(y, C, S, f"lora_up_f32w unaligned B [{call}]", torch.float32)
