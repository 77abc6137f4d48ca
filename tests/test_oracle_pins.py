"""Pins for the CPU oracle, each independent of the code it checks.

The oracle restates the products of a linear layer in fp64 (page "Twice the
training speed on a BC-250 from tuned matrix kernels", sections "Where the
time went", "Tuning the kernels" and "Checking the results are right").
These tests tie it to things other than itself: exact rational arithmetic,
NumPy's float64 and int64 matmul, hand-worked fixtures, closed forms,
transpose identities and finite differences.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from gemms_linear_layers_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DT16 = (torch.bfloat16, torch.float16)
DTIN = DT16 + (torch.float32,)  # the layer products also take FP32 operands
U = 2.0 ** -53


def f64(t):
    """Exact float64 values through torch's own conversion (not the oracle's)."""
    return t.to(torch.float64).numpy()


def rand16(shape, dtype, seed, spread=True):
    t = inputs.normal(shape, 1.0, torch.float32, seed)
    if spread:  # vary magnitudes over several binades
        g = torch.Generator().manual_seed(seed + 1)
        t = t * torch.pow(2.0, torch.randint(-6, 7, tuple(shape), generator=g).float())
    return t.to(dtype)


# ---------------------------------------------------------------------------
# decoding and rounding
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", DT16)
def test_decode_every_16bit_pattern(dtype):
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    vals = bits.view(dtype)
    ref = vals.to(torch.float64).numpy()
    got = oracle.decode(vals)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def _golden_round_cases():
    cases = []
    with open(os.path.join(GOLDEN, "round16_cases.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            val, dt, hexbits = line.split()
            m, e = val.split("*2^")
            cases.append((float(Fraction(int(m)) * Fraction(2) ** int(e)),
                          torch.bfloat16 if dt == "bf16" else torch.float16, int(hexbits, 16)))
    return cases


def test_round16_golden_cases():
    cases = _golden_round_cases()
    assert len(cases) >= 25
    for x, dtype, want in cases:
        got = int(oracle.round16(np.array([x]), dtype)[0])
        assert got == want, (x, dtype, hex(got), hex(want))


@pytest.mark.parametrize("dtype", DT16)
def test_round16_matches_torch_on_binary32(dtype):
    g = torch.Generator().manual_seed(7)
    x = torch.randn(200000, generator=g) * torch.pow(2.0, torch.randint(-30, 20, (200000,), generator=g).float())
    # add exact ties for the 16-bit grid: k + 1/2 quanta
    k = torch.randint(1, 1 << 10, (5000,), generator=g).float()
    ties = (k + 0.5) * 2.0 ** -8
    x = torch.cat([x, ties, -ties])
    want = x.to(dtype).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round16(x.to(torch.float64).numpy(), dtype)
    assert np.array_equal(got, want)


def test_round16_f16_matches_numpy_on_doubles():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(200000) * np.exp2(rng.integers(-28, 18, 200000))
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = oracle.round16(x, torch.float16)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# the products: hand-worked fixture, brute force, NumPy, integers
# ---------------------------------------------------------------------------
def _read_layer_fixture():
    out = {}
    with open(os.path.join(GOLDEN, "layer_products_2x3x2.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            name, rest = line.split(None, 1)
            out[name] = np.array([[float(v) for v in row.split()] for row in rest.split(";")])
    return out


@pytest.mark.parametrize("dtype", DT16)
def test_hand_worked_layer(dtype):
    fx = _read_layer_fixture()
    X, W, dY = (torch.tensor(fx[n]).to(dtype) for n in ("X", "W", "dY"))
    assert np.array_equal(oracle.gemm_fwd(X, W)[0], fx["Y"])
    assert np.array_equal(oracle.gemm_dgrad(dY, W)[0], fx["dX"])
    assert np.array_equal(oracle.gemm_wgrad(dY, X)[0], fx["dW"])


def _exact(op, A, B):
    """Exact rational products written from the page's definitions."""
    a = [[Fraction(float(v)) for v in row] for row in A.to(torch.float64).tolist()]
    b = [[Fraction(float(v)) for v in row] for row in B.to(torch.float64).tolist()]
    if op == "fwd":    # Y[t][o] = sum_i X[t][i] W[o][i]
        T, d_in, d_out = len(a), len(a[0]), len(b)
        return [[sum((a[t][i] * b[o][i] for i in range(d_in)), Fraction(0)) for o in range(d_out)]
                for t in range(T)], [[sum((abs(a[t][i] * b[o][i]) for i in range(d_in)), Fraction(0))
                                      for o in range(d_out)] for t in range(T)], d_in
    if op == "dgrad":  # dX[t][i] = sum_o dY[t][o] W[o][i]
        T, d_out, d_in = len(a), len(a[0]), len(b[0])
        return [[sum((a[t][o] * b[o][i] for o in range(d_out)), Fraction(0)) for i in range(d_in)]
                for t in range(T)], [[sum((abs(a[t][o] * b[o][i]) for o in range(d_out)), Fraction(0))
                                      for i in range(d_in)] for t in range(T)], d_out
    # wgrad: dW[o][i] = sum_t dY[t][o] X[t][i]
    T, d_out, d_in = len(a), len(a[0]), len(b[0])
    return [[sum((a[t][o] * b[t][i] for t in range(T)), Fraction(0)) for i in range(d_in)]
            for o in range(d_out)], [[sum((abs(a[t][o] * b[t][i]) for t in range(T)), Fraction(0))
                                      for i in range(d_in)] for o in range(d_out)], T


def _operands(op, T, d_in, d_out, dtype, seed):
    X = rand16((T, d_in), dtype, seed)
    W = rand16((d_out, d_in), dtype, seed + 100)
    dY = rand16((T, d_out), dtype, seed + 200)
    return {"fwd": (X, W), "dgrad": (dY, W), "wgrad": (dY, X)}[op]


ORACLE_OP = {"fwd": oracle.gemm_fwd, "dgrad": oracle.gemm_dgrad, "wgrad": oracle.gemm_wgrad}


@pytest.mark.parametrize("dtype", DTIN)
@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_bruteforce_rational_all_tiny_shapes(op, dtype):
    for T, d_in, d_out in itertools.product(range(1, 5), repeat=3):
        A, B = _operands(op, T, d_in, d_out, dtype, seed=T * 100 + d_in * 10 + d_out)
        C, S = ORACLE_OP[op](A, B)
        ex, exs, K = _exact(op, A, B)
        ex = np.array([[float(v) for v in row] for row in ex])
        exs = np.array([[float(v) for v in row] for row in exs])
        # fp64 recursive summation: |err| <= (K-1) u S, |err(S)| likewise
        bound = max(K - 1, 0) * U * 1.0001 * exs
        assert np.all(np.abs(C - ex) <= bound), (op, T, d_in, d_out)
        assert np.all(np.abs(S - exs) <= bound), (op, T, d_in, d_out)


LADDER = [(1, 1, 1), (1, 8, 8), (7, 5, 13), (16, 16, 16), (64, 64, 64), (33, 129, 65), (200, 96, 300)]


@pytest.mark.parametrize("dtype", DTIN)
@pytest.mark.parametrize("T,d_in,d_out", LADDER)
def test_numpy_float64_matmul(T, d_in, d_out, dtype):
    X = rand16((T, d_in), dtype, 1)
    W = rand16((d_out, d_in), dtype, 2)
    dY = rand16((T, d_out), dtype, 3)
    x, w, g = f64(X), f64(W), f64(dY)
    for op, (A, B), ref, K in (("fwd", (X, W), x @ w.T, d_in), ("dgrad", (dY, W), g @ w, d_out),
                               ("wgrad", (dY, X), g.T @ x, T)):
        C, S = ORACLE_OP[op](A, B)
        assert C.shape == ref.shape
        # both are fp64 sums of K exact products in different orders
        assert np.all(np.abs(C - ref) <= 2 * K * U * S + 1e-300), op


@pytest.mark.parametrize("dtype", DTIN)
def test_small_integer_inputs_are_exact(dtype):
    T, d_in, d_out = 96, 700, 40
    X = inputs.small_int((T, d_in), -2, 2, dtype, 5)
    W = inputs.small_int((d_out, d_in), -2, 2, dtype, 6)
    dY = inputs.small_int((T, d_out), -2, 2, dtype, 7)
    xi, wi, gi = (t.to(torch.int64).numpy() for t in (X, W, dY))
    assert np.array_equal(oracle.gemm_fwd(X, W)[0], (xi @ wi.T).astype(np.float64))
    assert np.array_equal(oracle.gemm_dgrad(dY, W)[0], (gi @ wi).astype(np.float64))
    assert np.array_equal(oracle.gemm_wgrad(dY, X)[0], (gi.T @ xi).astype(np.float64))


# ---------------------------------------------------------------------------
# closed forms and identities
# ---------------------------------------------------------------------------
def test_permutation_and_ones_closed_forms():
    n, T = 24, 9
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(3))
    P = torch.zeros(n, n)
    P[torch.arange(n), perm] = 1.0          # P[j][perm[j]] = 1
    P = P.to(torch.bfloat16)
    X = rand16((T, n), torch.bfloat16, 9)
    x = f64(X)
    # forward with W = P: Y[t][j] = X[t][perm[j]]
    assert np.array_equal(oracle.gemm_fwd(X, P)[0], x[:, perm.numpy()])
    # input gradient with W = P: dX[t][perm[j]] = dY[t][j]
    dX = oracle.gemm_dgrad(X, P)[0]
    assert np.array_equal(dX[:, perm.numpy()], x)
    # weight gradient with X = I (T = n): dW[o][i] = dY[i][o]
    G = rand16((n, 5), torch.bfloat16, 10)
    I = torch.eye(n).to(torch.bfloat16)
    assert np.array_equal(oracle.gemm_wgrad(G, I)[0], f64(G).T)
    # all ones: every entry equals the reduction length
    ones = torch.ones(7, 33).to(torch.float16)
    assert np.all(oracle.gemm_fwd(ones, torch.ones(5, 33).to(torch.float16))[0] == 33)
    assert np.all(oracle.gemm_wgrad(ones, torch.ones(7, 4).to(torch.float16))[0] == 7)


@pytest.mark.parametrize("dtype", DT16)
def test_transpose_identities_bitwise(dtype):
    T, d_in, d_out = 37, 53, 29
    X = rand16((T, d_in), dtype, 21)
    W = rand16((d_out, d_in), dtype, 22)
    G = rand16((T, d_out), dtype, 23)
    # fwd(X, W)^T = fwd(W, X)
    assert np.array_equal(oracle.gemm_fwd(X, W)[0].T, oracle.gemm_fwd(W, X)[0])
    # dgrad(G, W) = fwd(G, W^T)
    assert np.array_equal(oracle.gemm_dgrad(G, W)[0], oracle.gemm_fwd(G, W.T.contiguous())[0])
    # wgrad(G, X) = fwd(G^T, X^T)
    assert np.array_equal(oracle.gemm_wgrad(G, X)[0],
                          oracle.gemm_fwd(G.T.contiguous(), X.T.contiguous())[0])


def _loss_fwd(X, W, G):
    Y, _ = oracle.gemm_fwd(X, W)
    return float(np.sum(f64(G) * Y))


def test_finite_differences_dgrad_wgrad():
    """L(X, W) = <G, X W^T> is linear in X and in W, so a central difference
    with step 1 is exact up to fp64 rounding: dL/dX = G W, dL/dW = G^T X."""
    T, d_in, d_out = 5, 7, 6
    X = rand16((T, d_in), torch.bfloat16, 31).to(torch.float64)
    W = rand16((d_out, d_in), torch.bfloat16, 32).to(torch.float64)
    G = rand16((T, d_out), torch.bfloat16, 33).to(torch.float64)
    dX, _ = oracle.gemm_dgrad(G, W)
    dW, _ = oracle.gemm_wgrad(G, X)
    scale = float(np.sum(np.abs(f64(G)) @ np.abs(f64(W)))) + float(np.sum(np.abs(f64(G)).T @ np.abs(f64(X))))
    for t, i in itertools.product(range(T), range(d_in)):
        E = torch.zeros_like(X)
        E[t, i] = 1.0
        fd = (_loss_fwd(X + E, W, G) - _loss_fwd(X - E, W, G)) / 2.0
        assert abs(fd - dX[t, i]) <= 1e-12 * scale
    for o, i in itertools.product(range(d_out), range(d_in)):
        E = torch.zeros_like(W)
        E[o, i] = 1.0
        fd = (_loss_fwd(X, W + E, G) - _loss_fwd(X, W - E, G)) / 2.0
        assert abs(fd - dW[o, i]) <= 1e-12 * scale


def test_finite_differences_lora():
    """L = <G, (X A^T) B^T>; linear in each of X, A, B separately."""
    T, d_in, d_out, r = 6, 10, 9, 4
    X = rand16((T, d_in), torch.bfloat16, 41).to(torch.float64)
    A = rand16((r, d_in), torch.bfloat16, 42).to(torch.float64)
    B = rand16((d_out, r), torch.bfloat16, 43).to(torch.float64)
    G = rand16((T, d_out), torch.bfloat16, 44).to(torch.float64)

    def loss(X, A, B):
        H, _ = oracle.lora_down(X, A)
        Y, _ = oracle.lora_up(torch.from_numpy(H), B)
        return float(np.sum(f64(G) * Y))

    H = torch.from_numpy(oracle.lora_down(X, A)[0])
    g = oracle.lora_grad(X, A, B, H, G)
    scale = 1e-12 * (1.0 + float(np.sum(np.abs(f64(G)))) * float(np.max(np.abs(f64(B)))) *
                     float(np.max(np.abs(f64(A)))) * float(np.max(np.abs(f64(X)))) * d_in * r)
    for name, P, shape in (("dX", 0, (T, d_in)), ("dA", 1, (r, d_in)), ("dB", 2, (d_out, r))):
        args = [X, A, B]
        for idx in itertools.product(*(range(s) for s in shape)):
            E = torch.zeros(shape, dtype=torch.float64)
            E[idx] = 1.0
            plus = list(args)
            minus = list(args)
            plus[P] = args[P] + E
            minus[P] = args[P] - E
            fd = (loss(*plus) - loss(*minus)) / 2.0
            assert abs(fd - g[name][0][idx]) <= scale, (name, idx)
    # dH = G B is the gradient with respect to H
    assert np.allclose(g["dH"][0], f64(G) @ f64(B), rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# attention products
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", DT16)
def test_attention_products_against_numpy(dtype):
    h, s, d = 3, 40, 16
    t = inputs.attn_inputs(h, s, d, dtype, tag="pin")
    v = {k: f64(x) for k, x in t.items()}
    ref = {
        "qk": v["Q"] @ v["K"].transpose(0, 2, 1),
        "pv": v["P"] @ v["V"],
        "do_vt": v["dO"] @ v["V"].transpose(0, 2, 1),
        "pt_do": v["P"].transpose(0, 2, 1) @ v["dO"],
        "ds_k": v["dS"] @ v["K"],
        "dst_q": v["dS"].transpose(0, 2, 1) @ v["Q"],
    }
    for op in oracle.ATTN_OPS:
        a, b = inputs.ATTN_OPERANDS[op]
        C, S = oracle.bmm_attn(op, t[a], t[b])
        assert C.shape == ref[op].shape, op
        K = t[a].shape[2] if op in ("qk", "do_vt") else s
        assert np.all(np.abs(C - ref[op]) <= 2 * K * U * S + 1e-300), op


def test_attention_gradients_by_finite_differences():
    """dV = P^T dO, dP = dO V^T from <dO, P V>; dQ = dS K, dK = dS^T Q from <dS, Q K^T>."""
    h, s, d = 2, 5, 3
    g = torch.Generator().manual_seed(51)
    Q, K, V, dO = (torch.randn(h, s, d, generator=g, dtype=torch.float64) for _ in range(4))
    P, dS = (torch.randn(h, s, s, generator=g, dtype=torch.float64) for _ in range(2))

    def l_pv(P, V):
        return float(np.sum(dO.numpy() * oracle.bmm_attn("pv", P, V)[0]))

    def l_qk(Q, K):
        return float(np.sum(dS.numpy() * oracle.bmm_attn("qk", Q, K)[0]))

    grads = {"pt_do": oracle.bmm_attn("pt_do", P, dO)[0], "do_vt": oracle.bmm_attn("do_vt", dO, V)[0],
             "ds_k": oracle.bmm_attn("ds_k", dS, K)[0], "dst_q": oracle.bmm_attn("dst_q", dS, Q)[0]}
    for name, fn, args, pos in (("pt_do", l_pv, [P, V], 1), ("do_vt", l_pv, [P, V], 0),
                                ("ds_k", l_qk, [Q, K], 0), ("dst_q", l_qk, [Q, K], 1)):
        shape = args[pos].shape
        for idx in itertools.product(*(range(n) for n in shape)):
            E = torch.zeros(shape, dtype=torch.float64)
            E[idx] = 1.0
            plus, minus = list(args), list(args)
            plus[pos] = args[pos] + E
            minus[pos] = args[pos] - E
            fd = (fn(*plus) - fn(*minus)) / 2.0
            assert abs(fd - grads[name][idx]) <= 1e-11, (name, idx)


def test_sampled_product_equals_full():
    T, d_in, d_out = 50, 70, 30
    X = rand16((T, d_in), torch.float16, 61)
    W = rand16((d_out, d_in), torch.float16, 62)
    C, S = oracle.gemm_fwd(X, W)
    rng = np.random.default_rng(0)
    ii, jj = rng.integers(0, T, 100), rng.integers(0, d_out, 100)
    c, s = oracle.gemm_fwd(X, W, sample=(np.zeros(100, np.int64), ii, jj))
    assert np.array_equal(c, C[ii, jj]) and np.array_equal(s, S[ii, jj])


def test_thread_count_does_not_change_results():
    X = rand16((64, 300), torch.bfloat16, 71)
    W = rand16((48, 300), torch.bfloat16, 72)
    a, _ = oracle.gemm_fwd(X, W, nthreads=1)
    b, _ = oracle.gemm_fwd(X, W, nthreads=4)
    assert np.array_equal(a, b)


def test_ulp16():
    assert oracle.ulp16(1.0, torch.bfloat16) == 2.0 ** -7
    assert oracle.ulp16(1.5, torch.float16) == 2.0 ** -10
    assert oracle.ulp16(0.0, torch.float16) == 2.0 ** -24
    assert oracle.ulp16(1e-9, torch.float16) == 2.0 ** -24
    assert oracle.ulp16(-3.0, torch.bfloat16) == 2.0 ** -6


# ---------------------------------------------------------------------------
# the pins catch planted mistakes (mutated copies of the oracle, CPU only)
# ---------------------------------------------------------------------------
MUTATIONS = [
    ("for (int64_t k = 0; k < K; ++k) {\n        double p", "for (int64_t k = 0; k < K - 1; ++k) {\n        double p"),
    ("        c += p;", "        c -= p;"),
    ("v = ldexp((double)(m + 1024), e - 25);", "v = ldexp((double)(m + 1024), e - 24);"),
    ("load(B, bdt, b * b_bs + k * b_rs + j * b_cs);\n        c += p;",
     "load(B, bdt, b * b_bs + j * b_rs + k * b_cs);\n        c += p;"),
]


@pytest.mark.parametrize("mutation", range(len(MUTATIONS)))
def test_pins_catch_planted_mistakes(mutation, tmp_path):
    import ctypes
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTATIONS[mutation]
    assert src.count(old) == 1
    (tmp_path / "m.c").write_text(src.replace(old, new))
    so = str(tmp_path / "m.so")
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", so, str(tmp_path / "m.c"), "-lm"],
                   check=True)
    lib = ctypes.CDLL(so)
    i64 = ctypes.c_int64
    lib.oracle_gemm.argtypes = [ctypes.c_void_p, ctypes.c_int, i64, i64, i64, ctypes.c_void_p, ctypes.c_int,
                                i64, i64, i64, i64, i64, i64, i64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    caught = False
    for dtype in DT16:
        for T, d_in, d_out in ((3, 4, 2), (4, 3, 4)):
            X, W = _operands("fwd", T, d_in, d_out, dtype, seed=99)
            C = np.zeros((T, d_out))
            S = np.zeros((T, d_out))
            lib.oracle_gemm(X.data_ptr(), oracle.BF16 if dtype == torch.bfloat16 else oracle.F16,
                            T * d_in, d_in, 1, W.data_ptr(),
                            oracle.BF16 if dtype == torch.bfloat16 else oracle.F16,
                            d_out * d_in, 1, d_in, 1, T, d_out, d_in, C.ctypes.data, S.ctypes.data, 1)
            ex, exs, K = _exact("fwd", X, W)
            ex = np.array([[float(v) for v in row] for row in ex])
            exs = np.array([[float(v) for v in row] for row in exs])
            if not np.all(np.abs(C - ex) <= (K - 1) * U * 1.0001 * exs):
                caught = True
    assert caught, MUTATIONS[mutation]


# ---------------------------------------------------------------------------
# fused attention forward (softmax between the two products)
# ---------------------------------------------------------------------------
def _attn_bruteforce(q, k, v, scale):
    """softmax(scale q k^T) v with Python loops and math.exp, one row at a time."""
    import math
    h, s, d = q.shape
    out = np.zeros((h, s, d))
    for b in range(h):
        for i in range(s):
            x = [scale * sum(q[b, i, t] * k[b, j, t] for t in range(d)) for j in range(s)]
            mx = max(x)
            w = [math.exp(xj - mx) for xj in x]
            tot = sum(w)
            for t in range(d):
                out[b, i, t] = sum(w[j] * v[b, j, t] for j in range(s)) / tot
    return out


@pytest.mark.parametrize("dtype", DT16)
def test_attn_fwd_bruteforce_tiny(dtype):
    for h, s, d in ((1, 1, 1), (1, 2, 3), (2, 3, 2), (1, 5, 4)):
        Q, K, V = (rand16((h, s, d), dtype, 300 + i) for i in range(3))
        O, S, _ = oracle.attn_fwd(Q, K, V, 0.37)
        ref = _attn_bruteforce(f64(Q), f64(K), f64(V), 0.37)
        assert np.all(np.abs(O - ref) <= 1e-13 * S + 1e-300), (h, s, d)


def test_attn_fwd_closed_forms():
    h, s, d = 2, 40, 64
    V = rand16((h, s, d), torch.bfloat16, 310)
    K = rand16((h, s, d), torch.bfloat16, 311)
    # Q = 0: every key weighs 1/s, O is the mean of V's rows
    O, _, _ = oracle.attn_fwd(torch.zeros(h, s, d, dtype=torch.bfloat16), K, V, 0.125)
    mean = f64(V).mean(axis=1, keepdims=True)
    assert np.allclose(O, np.broadcast_to(mean, O.shape), rtol=0, atol=1e-14 * np.abs(f64(V)).max())
    # V = 1: each row of the softmax sums to one
    Q = rand16((h, s, d), torch.bfloat16, 312)
    O, _, _ = oracle.attn_fwd(Q, K, torch.ones(h, s, d, dtype=torch.bfloat16), 0.125)
    assert np.all(np.abs(O - 1.0) <= 1e-14)
    # one key far ahead of the others: its row of V comes out
    Qd = torch.zeros(h, s, d)
    Qd[:, :, 0] = 4.0
    Kd = torch.zeros(h, s, d)
    Kd[:, 7, 0] = 64.0  # logit 0.125 * 256 = 32 for key 7, 0 for the rest
    O, _, _ = oracle.attn_fwd(Qd.to(torch.bfloat16), Kd.to(torch.bfloat16), V, 0.125)
    want = np.broadcast_to(f64(V)[:, 7:8, :], O.shape)
    assert np.all(np.abs(O - want) <= (s * math.exp(-32.0)) * 2 * np.abs(f64(V)).max())


def test_attn_fwd_is_the_two_products_with_a_softmax_between():
    """The same result from the C oracle's batched products and a NumPy softmax."""
    h, s, d = 3, 50, 64
    Q, K, V = (rand16((h, s, d), torch.float16, 320 + i, spread=False) for i in range(3))
    O, S, _ = oracle.attn_fwd(Q, K, V, 0.125)
    logits, _ = oracle.bmm_attn("qk", Q, K)
    x = 0.125 * logits
    p = np.exp(x - x.max(axis=2, keepdims=True))
    p /= p.sum(axis=2, keepdims=True)
    ref = np.einsum("hij,hjd->hid", p, f64(V))
    assert np.all(np.abs(O - ref) <= 1e-12 * S)


def test_attn_fwd_sampled_rows_match_the_full_result():
    h, s, d = 3, 70, 64
    Q, K, V = (rand16((h, s, d), torch.bfloat16, 330 + i, spread=False) for i in range(3))
    O, S, E = oracle.attn_fwd(Q, K, V, 0.125)
    hh, ii = np.array([0, 2, 1, 2]), np.array([0, 69, 33, 5])
    Or, Sr, Er = oracle.attn_fwd(Q, K, V, 0.125, rows=(hh, ii))
    assert np.allclose(Or, O[hh, ii], rtol=1e-13, atol=0) and np.allclose(Sr, S[hh, ii], rtol=1e-13, atol=0)
    assert np.array_equal(Er, E[hh, ii])


def test_attn_bwd_finite_differences():
    """The attention gradients are the derivatives of L = <dO, O(Q, K, V)>:
    fp64 central differences on every input element of a small case."""
    h, s, d, scale = 2, 5, 3, 0.6
    Q, K, V, dO = (rand16((h, s, d), torch.float32, 340 + i, spread=False) for i in range(4))
    g = oracle.attn_bwd(Q, K, V, dO, scale)
    base = {"Q": f64(Q), "K": f64(K), "V": f64(V)}
    do = f64(dO)

    def loss(t):
        O, _, _ = oracle.attn_fwd(torch.from_numpy(t["Q"]), torch.from_numpy(t["K"]), torch.from_numpy(t["V"]),
                                  scale)
        return float((O * do).sum())

    eps = 1e-6
    for name in ("Q", "K", "V"):
        want = np.zeros_like(base[name])
        for idx in np.ndindex(*base[name].shape):
            tp = {k: v.copy() for k, v in base.items()}
            tm = {k: v.copy() for k, v in base.items()}
            tp[name][idx] += eps
            tm[name][idx] -= eps
            want[idx] = (loss(tp) - loss(tm)) / (2 * eps)
        got, S = g["d" + name]
        assert np.all(np.abs(got - want) <= 1e-6 * (S + 1.0)), name


def test_attn_bwd_value_gradient_is_p_transposed_times_do():
    """dV = P^T dO with P from the oracle's own softmax of the C oracle's logits."""
    h, s, d = 2, 30, 64
    Q, K, V, dO = (rand16((h, s, d), torch.bfloat16, 350 + i, spread=False) for i in range(4))
    dV, S = oracle.attn_bwd(Q, K, V, dO, 0.125)["dV"]
    logits, _ = oracle.bmm_attn("qk", Q, K)
    x = 0.125 * logits
    p = np.exp(x - x.max(axis=2, keepdims=True))
    p /= p.sum(axis=2, keepdims=True)
    assert np.all(np.abs(dV - np.einsum("hij,hid->hjd", p, f64(dO))) <= 1e-12 * S)


@pytest.mark.parametrize("scale", [0.6, -0.6])
def test_attn_bwd_error_scales_bound_the_values(scale):
    """Each error scale is a sum of magnitudes of the terms the gradient sums
    (for dQ and dK the terms carry the factor scale, so their magnitudes carry
    |scale|): it is non-negative and at least the magnitude of the value, for
    a negative scale too.  The finite differences of the same case pin the
    values."""
    h, s, d = 2, 5, 3
    Q, K, V, dO = (rand16((h, s, d), torch.float32, 360 + i, spread=False) for i in range(4))
    g = oracle.attn_bwd(Q, K, V, dO, scale)
    for name in ("dQ", "dK", "dV"):
        val, S = g[name]
        assert np.all(S >= 0), name
        assert np.all(np.abs(val) <= S * (1 + 1e-12)), name
