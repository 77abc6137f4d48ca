"""CPU oracle for the training products of a linear layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library's product path never does,
and this package imports nothing from the library: the two share no code.

What it computes (page "Twice the training speed on a BC-250 from tuned matrix
kernels"):

* section "Where the time went": each linear layer runs three products, the
  forward pass, the gradient for its input and the gradient for its weight,
  each in its own memory layout;
* section "Tuning the kernels": bf16 and fp16 inputs with FP32 accumulation,
  plus the rank-16 LoRA matrices and the batched products inside attention;
* section "Checking the results are right": every product is checked against
  a float64 product on the CPU.

So the oracle is the exact definition, evaluated in fp64 over the exact values
of the 16-bit inputs (``oracle.c``): ``C[b,i,j] = sum_k A(b,i,k) B(b,k,j)``
with k ascending, together with the error scale ``S = sum_k |A B|``.  Each
product below is that one loop nest with its own index map.

Pins (``tests/test_oracle_pins.py``), each independent of the code it checks:

* ``gemm`` (all index maps): exact rational brute force on every shape up to
  4x4x4; NumPy float64 matmul on the same inputs; exact integer results for
  small-integer inputs (against NumPy int64 matmul); closed forms for
  permutation and all-ones operands; transpose identities linking the three
  layouts; fp64 finite differences showing that dgrad and wgrad are the
  gradients of L = <G, X W^T>.
* ``lora_*``: finite differences of L = <G, X A^T B^T> for dA, dB, dX, and
  the same brute-force/NumPy pins for the individual products.
* ``bmm_attn``: the six products against NumPy batched matmul, and finite
  differences of <dO, P V> and <dS, Q K^T>.
* ``attn_fwd`` (softmax between the products): Python-loop brute force with
  math.exp, closed forms (Q = 0 gives the mean of V; V = 1 gives 1; one
  dominant key gives its row of V), the C oracle's logits with a NumPy
  softmax, and sampled rows against the full result.
* ``attn_bwd``: fp64 finite differences of <dO, attn_fwd(Q, K, V)> for every
  input element, and dV against P^T dO.
* ``round16``: hand-derived tie, subnormal and overflow cases
  (``tests/golden/round16_cases.txt``), torch's binary32->bf16/fp16 RNE on
  binary32 inputs and NumPy's float64->float16 conversion on doubles.

Nothing here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# element type codes (must match oracle.c)
BF16, F16, F32, F64 = 0, 1, 2, 3
_CODE = {torch.bfloat16: BF16, torch.float16: F16, torch.float32: F32, torch.float64: F64}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (-O2, no fast-math, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
            lib.oracle_gemm.argtypes = [vp, ip, i64, i64, i64, vp, ip, i64, i64, i64,
                                        i64, i64, i64, i64, dp, dp, ip]
            lib.oracle_gemm.restype = None
            lib.oracle_gemm_at.argtypes = [vp, ip, i64, i64, i64, vp, ip, i64, i64, i64,
                                           i64, i64, vp, vp, vp, dp, dp, ip]
            lib.oracle_gemm_at.restype = None
            lib.oracle_round16.argtypes = [dp, i64, ip, vp]
            lib.oracle_round16.restype = None
            lib.oracle_decode.argtypes = [vp, ip, i64, dp]
            lib.oracle_decode.restype = None
            lib.oracle_version.restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    """Host threads the oracle uses: every core this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _as_buffer(t):
    """(contiguous CPU tensor, type code) for a torch tensor or numpy array."""
    if isinstance(t, np.ndarray):
        t = torch.from_numpy(np.ascontiguousarray(t))
    t = t.detach().to("cpu").contiguous()
    if t.dtype not in _CODE:
        t = t.to(torch.float64)
    return t, _CODE[t.dtype]


# --------------------------------------------------------------------------
# the one product, with explicit index maps
# --------------------------------------------------------------------------
def gemm(A, a_map, B, b_map, batch, M, N, K, nthreads=None, want_s=True):
    """C[b,i,j] = sum_k A(b,i,k) B(b,k,j); a_map = (bs, rs, cs) element strides.

    Returns (C, S) as float64 numpy arrays shaped [batch, M, N] (S is None when
    want_s is False).
    """
    lib = _load()
    a, adt = _as_buffer(A)
    b, bdt = _as_buffer(B)
    C = np.zeros((batch, M, N), dtype=np.float64)
    S = np.zeros((batch, M, N), dtype=np.float64) if want_s else None
    if batch * M * N > 0:
        lib.oracle_gemm(a.data_ptr(), adt, *a_map, b.data_ptr(), bdt, *b_map,
                        batch, M, N, K, C.ctypes.data,
                        S.ctypes.data if want_s else None,
                        nthreads if nthreads else threads())
    return C, S


def gemm_at(A, a_map, B, b_map, K, bi, ii, jj, nthreads=None):
    """The product at sampled coordinates; returns (C, S) float64 vectors."""
    lib = _load()
    a, adt = _as_buffer(A)
    b, bdt = _as_buffer(B)
    bi = np.ascontiguousarray(bi, dtype=np.int64)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    n = len(ii)
    C = np.zeros(n, dtype=np.float64)
    S = np.zeros(n, dtype=np.float64)
    if n:
        lib.oracle_gemm_at(a.data_ptr(), adt, *a_map, b.data_ptr(), bdt, *b_map, K, n,
                           bi.ctypes.data, ii.ctypes.data, jj.ctypes.data,
                           C.ctypes.data, S.ctypes.data, nthreads if nthreads else threads())
    return C, S


# --------------------------------------------------------------------------
# index maps of the layer's products.  Shapes use the page's names:
# X[T, d_in] activations, W[d_out, d_in] weight, dY[T, d_out] output gradient.
# --------------------------------------------------------------------------
def _maps_fwd(M, N, K):
    # Y[M=T, N=d_out] = X[T, d_in] . W[d_out, d_in]^T ; X(i,k)=X[i*K+k], W^T(k,j)=W[j*K+k]
    return (M * K, K, 1), (N * K, 1, K)


def _maps_dgrad(M, N, K):
    # dX[M=T, N=d_in] = dY[T, K=d_out] . W[d_out, d_in] ; dY(i,k)=dY[i*K+k], W(k,j)=W[k*N+j]
    return (M * K, K, 1), (K * N, N, 1)


def _maps_wgrad(M, N, K):
    # dW[M=d_out, N=d_in] = dY[K=T, d_out]^T . X[T, d_in] ; dY^T(i,k)=dY[k*M+i], X(k,j)=X[k*N+j]
    return (K * M, 1, M), (K * N, N, 1)


def gemm_fwd(X, W, sample=None, nthreads=None):
    """Forward product Y = X W^T.  X [T, d_in], W [d_out, d_in] -> [T, d_out]."""
    T, d_in = X.shape
    d_out = W.shape[0]
    am, bm = _maps_fwd(T, d_out, d_in)
    return _run(X, am, W, bm, 1, T, d_out, d_in, sample, nthreads)


def gemm_dgrad(dY, W, sample=None, nthreads=None):
    """Input gradient dX = dY W.  dY [T, d_out], W [d_out, d_in] -> [T, d_in]."""
    T, d_out = dY.shape
    d_in = W.shape[1]
    am, bm = _maps_dgrad(T, d_in, d_out)
    return _run(dY, am, W, bm, 1, T, d_in, d_out, sample, nthreads)


def gemm_wgrad(dY, X, sample=None, nthreads=None):
    """Weight gradient dW = dY^T X, summed over tokens.  -> [d_out, d_in]."""
    T, d_out = dY.shape
    d_in = X.shape[1]
    am, bm = _maps_wgrad(d_out, d_in, T)
    return _run(dY, am, X, bm, 1, d_out, d_in, T, sample, nthreads)


def _run(A, am, B, bm, batch, M, N, K, sample, nthreads):
    if sample is None:
        C, S = gemm(A, am, B, bm, batch, M, N, K, nthreads)
        if batch == 1:
            return C[0], S[0]
        return C, S
    bi, ii, jj = sample
    return gemm_at(A, am, B, bm, K, bi, ii, jj, nthreads)


# --------------------------------------------------------------------------
# batched products inside attention: tensors [batch, rows, cols]
# --------------------------------------------------------------------------
ATTN_OPS = ("qk", "pv", "do_vt", "pt_do", "ds_k", "dst_q")


def bmm_attn(op, A, B, sample=None, nthreads=None):
    """One of the six attention products (no mask, no softmax, no scaling).

    qk:    S  = Q  K^T   Q,K [h,s,d]      -> [h,s,s]
    pv:    O  = P  V     P [h,s,s], V [h,s,d] -> [h,s,d]
    do_vt: dP = dO V^T   dO,V [h,s,d]     -> [h,s,s]
    pt_do: dV = P^T dO   P [h,s,s], dO [h,s,d] -> [h,s,d]
    ds_k:  dQ = dS K     dS [h,s,s], K [h,s,d] -> [h,s,d]
    dst_q: dK = dS^T Q   dS [h,s,s], Q [h,s,d] -> [h,s,d]
    """
    if op in ("qk", "do_vt"):  # forward layout, K = d
        h, s, d = A.shape
        am, bm = _maps_fwd(s, s, d)
        return _run(A, am, B, bm, h, s, s, d, sample, nthreads)
    if op in ("pv", "ds_k"):  # input-gradient layout, K = s
        h, s, _ = A.shape
        d = B.shape[2]
        am, bm = _maps_dgrad(s, d, s)
        return _run(A, am, B, bm, h, s, d, s, sample, nthreads)
    if op in ("pt_do", "dst_q"):  # weight-gradient layout, K = s
        h, s, _ = A.shape
        d = B.shape[2]
        am, bm = _maps_wgrad(s, d, s)
        return _run(A, am, B, bm, h, s, d, s, sample, nthreads)
    raise ValueError(f"unknown attention product {op!r}")


def attn_fwd(Q, K, V, scale, rows=None):
    """Attention forward with the softmax between the two products, in fp64
    over the exact input values: O[h,i] = sum_j P[h,i,j] V[h,j] with
    P[h,i,:] = softmax_j(scale * sum_k Q[h,i,k] K[h,j,k]) (no mask).

    Returns (O, S_O, E): O [h,s,d]; the error scale S_O = sum_j P |V|; and per
    row E = max_j sum_k |Q K| (the size of the largest logit's terms), from
    which the FP32 rounding of the logits is bounded.  rows = (heads, row
    indices) restricts the result to those rows (each a full softmax over all
    keys); then O, S_O are [n, d] and E [n].
    Written from the definition: the softmax is exp(x - max) / sum exp(x - max),
    with NumPy float64 matrix products and exponentials.
    """
    q, k, v = decode(Q), decode(K), decode(V)
    if rows is not None:
        hh, ii = (np.asarray(x, dtype=np.int64) for x in rows)
        qs = q[hh, ii]                                  # [n, d]
        logits = np.einsum("nd,njd->nj", qs, k[hh])     # [n, s]
        terms = np.einsum("nd,njd->nj", np.abs(qs), np.abs(k[hh]))
        x = scale * logits
        p = np.exp(x - x.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        return np.einsum("nj,njd->nd", p, v[hh]), np.einsum("nj,njd->nd", p, np.abs(v[hh])), terms.max(axis=1)
    x = scale * np.einsum("hid,hjd->hij", q, k)
    p = np.exp(x - x.max(axis=2, keepdims=True))
    p /= p.sum(axis=2, keepdims=True)
    terms = np.einsum("hid,hjd->hij", np.abs(q), np.abs(k)).max(axis=2)
    return np.einsum("hij,hjd->hid", p, v), np.einsum("hij,hjd->hid", p, np.abs(v)), terms


def attn_bwd(Q, K, V, dO, scale):
    """Gradients of L = <dO, O> for O = softmax(scale Q K^T) V (the forward of
    attn_fwd), in fp64 over the exact input values, written from the chain
    rule: with P the softmax weights,
        dV = P^T dO,   dP = dO V^T,   dS = P * (dP - rowsum(dO * O)),
        dQ = scale dS K,   dK = scale dS^T Q.
    Returns a dict of (value, error scale) pairs for dQ, dK, dV; the scales are
    the same sums with every term replaced by its absolute value.
    """
    q, k, v, do = decode(Q), decode(K), decode(V), decode(dO)
    x = scale * np.einsum("hid,hjd->hij", q, k)
    p = np.exp(x - x.max(axis=2, keepdims=True))
    p /= p.sum(axis=2, keepdims=True)
    o = np.einsum("hij,hjd->hid", p, v)
    dv = np.einsum("hij,hid->hjd", p, do)
    dp = np.einsum("hid,hjd->hij", do, v)
    delta = np.einsum("hid,hid->hi", do, o)[..., None]
    ds = p * (dp - delta)
    dq = scale * np.einsum("hij,hjd->hid", ds, k)
    dk = scale * np.einsum("hij,hid->hjd", ds, q)
    ads = p * (np.abs(dp) + np.abs(delta))
    asc = abs(scale)
    return {"dQ": (dq, asc * np.einsum("hij,hjd->hid", ads, np.abs(k))),
            "dK": (dk, asc * np.einsum("hij,hid->hjd", ads, np.abs(q))),
            "dV": (dv, np.einsum("hij,hid->hjd", p, np.abs(do)))}


# --------------------------------------------------------------------------
# rank-r LoRA products (section "Tuning the kernels": the rank-16 LoRA
# matrices).  A [r, d_in], B [d_out, r]; no alpha/r scaling (the page gives
# none); outputs overwrite.
# --------------------------------------------------------------------------
def lora_down(X, A, nthreads=None):
    """H = X A^T: [T, d_in] x [r, d_in] -> [T, r]."""
    return gemm_fwd(X, A, nthreads=nthreads)


def lora_up(H, B, nthreads=None):
    """Y = H B^T: [T, r] x [d_out, r] -> [T, d_out]."""
    return gemm_fwd(H, B, nthreads=nthreads)


def lora_grad(X, A, B, H, dY, nthreads=None):
    """Gradients of the LoRA branch Y = (X A^T) B^T given dY.

    dH = dY B (kept in fp64, unrounded), dB = dY^T H, dA = dH^T X, dX = dH A.
    For dA and dX, whose input dH is itself a product, the error scale is
    the chained one: S2 = sum over both reductions of |each product term|,
    i.e. (sum_o |dY B|) applied to |X| or |A|.
    Returns a dict of (value, scale) pairs.
    """
    dH, S_dH = gemm_dgrad(dY, B, nthreads=nthreads)
    dB, S_dB = gemm_wgrad(dY, H, nthreads=nthreads)
    dA, _ = gemm_wgrad(torch.from_numpy(dH), X, nthreads=nthreads)
    dX, _ = gemm_dgrad(torch.from_numpy(dH), A, nthreads=nthreads)
    # chained scales: S_dH >= 0, so sum |S_dH * x| = sum S_dH |x|
    _, S_dA = gemm_wgrad(torch.from_numpy(S_dH), X, nthreads=nthreads)
    _, S_dX = gemm_dgrad(torch.from_numpy(S_dH), A, nthreads=nthreads)
    return {"dH": (dH, S_dH), "dB": (dB, S_dB), "dA": (dA, S_dA), "dX": (dX, S_dX)}


# --------------------------------------------------------------------------
# rounding to the 16-bit output types, and their unit in the last place
# --------------------------------------------------------------------------
def round16(x, dtype) -> np.ndarray:
    """RNE from float64 straight to bf16/fp16; returns the uint16 bit patterns."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    code = BF16 if dtype == torch.bfloat16 else F16
    lib.oracle_round16(x.ctypes.data, x.size, code, out.ctypes.data)
    return out


def decode(t) -> np.ndarray:
    """Exact float64 values of a bf16/fp16/fp32 tensor."""
    lib = _load()
    b, code = _as_buffer(t)
    out = np.zeros(tuple(b.shape), dtype=np.float64)
    lib.oracle_decode(b.data_ptr(), code, b.numel(), out.ctypes.data)
    return out


def ulp16(x, dtype) -> np.ndarray:
    """Spacing of the bf16/fp16 grid at |x|: 2^(max(e, emin) - (p - 1))."""
    p, emin = (8, -126) if dtype == torch.bfloat16 else (11, -14)
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(a)
    e = np.where(a > 0, e - 1, emin)
    return np.ldexp(1.0, np.maximum(e, emin) - (p - 1))


__all__ = ["build", "threads", "gemm", "gemm_at", "gemm_fwd", "gemm_dgrad", "gemm_wgrad",
           "bmm_attn", "ATTN_OPS", "lora_down", "lora_up", "lora_grad", "round16", "decode",
           "ulp16", "BF16", "F16", "F32", "F64"]
