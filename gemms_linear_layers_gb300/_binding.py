"""ctypes binding of libtg.so: the same entry points as include/tg.h.

Each function takes torch CUDA tensors, checks that their shapes agree,
allocates the output (and the workspace the call asks for) with torch's
caching allocator when the caller passes none, and calls the C entry point on
the current CUDA stream.  No arithmetic happens here: every product runs in
the library's kernels.  If libtg.so has not been built the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtg.so")
DEFAULT_TABLE = os.path.join(_PKG, "tables", "gb300.txt")
_lock = threading.Lock()
_lib = None

TG_BF16, TG_F16, TG_F32 = 0, 1, 2
_DT = {torch.bfloat16: TG_BF16, torch.float16: TG_F16, torch.float32: TG_F32}

TG_OP_GEMM_FWD, TG_OP_GEMM_DGRAD, TG_OP_GEMM_WGRAD = 0, 1, 2
TG_OP_LORA_DOWN, TG_OP_LORA_UP, TG_OP_LORA_GRAD, TG_OP_BMM_ATTN = 3, 4, 5, 6
TG_OP_LORA_DOWN_F32W, TG_OP_LORA_UP_F32W, TG_OP_LORA_GRAD_F32W = 7, 8, 9
TG_OP_ATTN_BWD = 10
TG_OP_GEMM_FWD_LORA, TG_OP_GEMM_DGRAD_LORA = 11, 12
ATTN_OPS = {"qk": 0, "pv": 1, "do_vt": 2, "pt_do": 3, "ds_k": 4, "dst_q": 5}
SIZE_MAX = (1 << 64) - 1

# every symbol include/tg.h declares, with (restype, argtypes)
_vp, _i64, _sz, _i = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
SIGNATURES = {
    "tg_gemm_fwd": (_i, [_vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _vp, _sz, _vp]),
    "tg_gemm_dgrad": (_i, [_vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _vp, _sz, _vp]),
    "tg_gemm_wgrad": (_i, [_vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _vp, _sz, _vp]),
    "tg_gemm_fwd_lora": (_i, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, ctypes.c_float, _i, _i, _vp, _sz, _vp]),
    "tg_gemm_dgrad_lora": (_i, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, ctypes.c_float, _i, _i, _vp, _sz,
                                _vp]),
    "tg_gemm_wgrad_accumulate": (_i, [_vp, _vp, _vp, _i64, _i64, _i64, _i, _vp, _sz, _vp]),
    "tg_gemm_wgrad_noalloc": (_i, [_vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _vp]),
    "tg_lora_down": (_i, [_vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _vp, _sz, _vp]),
    "tg_lora_up": (_i, [_vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _vp, _sz, _vp]),
    "tg_lora_up_add": (_i, [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_float, _i, _i, _vp, _sz, _vp]),
    "tg_lora_grad": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i, _i,
                          _vp, _sz, _vp]),
    "tg_lora_down_f32w": (_i, [_vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _vp, _sz, _vp]),
    "tg_lora_up_f32w": (_i, [_vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _vp, _sz, _vp]),
    "tg_lora_grad_f32w": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i, _i,
                               _vp, _sz, _vp]),
    "tg_attn_fwd": (_i, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_float, _i, _i, _vp]),
    "tg_attn_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_float, _i, _i, _vp, _sz, _vp]),
    "tg_lora_grad_add": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, ctypes.c_float,
                              _i, _i, _vp, _sz, _vp]),
    "tg_bmm_attn": (_i, [_i, _vp, _vp, _vp, _i64, _i64, _i64, _i, _i, _vp, _sz, _vp]),
    "tg_workspace_size": (_sz, [_i, _i64, _i64, _i64, _i64, _i, _i]),
    "tg_stream_status": (_i, [_vp]),
    "tg_status_string": (ctypes.c_char_p, [_i]),
    "tg_load_table": (_i, [ctypes.c_char_p]),
    "tg_version": (_i, []),
    "tg_last_call": (_sz, [ctypes.c_char_p, _sz]),
    "tg_plan_describe": (_sz, [_i, _i64, _i64, _i64, _i64, _i, _i, _i, ctypes.c_char_p, _sz]),
    "tg_wait_probe": (_i, [_i64, _vp]),
}


class TGError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: tg status {status} ({lib().tg_status_string(status).decode()})")


def lib() -> ctypes.CDLL:
    """The loaded libtg.so (built in-tree by gemms_linear_layers_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m gemms_linear_layers_gb300.build` (needs nvcc)")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(l, name)
                fn.restype = res
                fn.argtypes = args
            _lib = l
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise TGError(status, where)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _keep(buf, stream):
    """A workspace allocated here is freed on return; tell the caching
    allocator which stream still uses it."""
    if buf is not None and stream is not None:
        buf.record_stream(stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def _need(t, name, ndim):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor, got shape {tuple(t.shape)}")
    return t


def _out(out, shape, dtype, device, name):
    if out is None:
        return torch.empty(shape, dtype=dtype, device=device)
    _need(out, name, len(shape))
    if tuple(out.shape) != tuple(shape) or out.dtype != dtype:
        raise ValueError(f"{name} must be {tuple(shape)} {dtype}, got {tuple(out.shape)} {out.dtype}")
    return out


def _workspace(op, dims, din, dout, ws, device):
    n = lib().tg_workspace_size(op, *dims, din, dout)
    if n == SIZE_MAX:
        raise ValueError(f"invalid sizes {dims} for workspace query {op}")
    if n == 0:
        return ctypes.c_void_p(0), 0, None
    if ws is not None and ws.numel() * ws.element_size() >= n:
        return ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(), ws
    buf = torch.empty(n, dtype=torch.uint8, device=device)
    return ctypes.c_void_p(buf.data_ptr()), n, buf


# --------------------------------------------------------------------------
def tg_gemm_fwd(X, W, Y=None, out_dtype=None, ws=None, stream=None):
    """Y[T, d_out] = X[T, d_in] W[d_out, d_in]^T."""
    _need(X, "X", 2), _need(W, "W", 2)
    T, d_in = X.shape
    d_out = W.shape[0]
    if W.shape[1] != d_in or W.dtype != X.dtype:
        raise ValueError("W must be [d_out, d_in] with X's dtype")
    Y = _out(Y, (T, d_out), out_dtype or X.dtype, X.device, "Y")
    wp, wn, keep = _workspace(TG_OP_GEMM_FWD, (T, d_out, d_in, 0), _DT[X.dtype], _DT[Y.dtype], ws, X.device)
    _check(lib().tg_gemm_fwd(_ptr(X), _ptr(W), _ptr(Y), T, d_out, d_in, _DT[X.dtype], _DT[Y.dtype], wp, wn,
                             _stream(stream)), "tg_gemm_fwd")
    _keep(keep, stream)
    return Y


def tg_gemm_dgrad(dY, W, dX=None, out_dtype=None, ws=None, stream=None):
    """dX[T, d_in] = dY[T, d_out] W[d_out, d_in]."""
    _need(dY, "dY", 2), _need(W, "W", 2)
    T, d_out = dY.shape
    d_in = W.shape[1]
    if W.shape[0] != d_out or W.dtype != dY.dtype:
        raise ValueError("W must be [d_out, d_in] with dY's dtype")
    dX = _out(dX, (T, d_in), out_dtype or dY.dtype, dY.device, "dX")
    wp, wn, keep = _workspace(TG_OP_GEMM_DGRAD, (T, d_out, d_in, 0), _DT[dY.dtype], _DT[dX.dtype], ws, dY.device)
    _check(lib().tg_gemm_dgrad(_ptr(dY), _ptr(W), _ptr(dX), T, d_out, d_in, _DT[dY.dtype], _DT[dX.dtype], wp, wn,
                               _stream(stream)), "tg_gemm_dgrad")
    _keep(keep, stream)
    return dX


def tg_gemm_wgrad(dY, X, dW=None, out_dtype=None, ws=None, stream=None):
    """dW[d_out, d_in] = dY[T, d_out]^T X[T, d_in]."""
    _need(dY, "dY", 2), _need(X, "X", 2)
    T, d_out = dY.shape
    d_in = X.shape[1]
    if X.shape[0] != T or X.dtype != dY.dtype:
        raise ValueError("X must be [T, d_in] with dY's dtype")
    dW = _out(dW, (d_out, d_in), out_dtype or dY.dtype, dY.device, "dW")
    wp, wn, keep = _workspace(TG_OP_GEMM_WGRAD, (T, d_out, d_in, 0), _DT[dY.dtype], _DT[dW.dtype], ws, dY.device)
    _check(lib().tg_gemm_wgrad(_ptr(dY), _ptr(X), _ptr(dW), T, d_out, d_in, _DT[dY.dtype], _DT[dW.dtype], wp, wn,
                               _stream(stream)), "tg_gemm_wgrad")
    _keep(keep, stream)
    return dW



def tg_gemm_fwd_lora(X, W, H, B, scale, Y=None, out_dtype=None, ws=None, stream=None):
    """Y = X W^T + scale H B^T in one product: X [T, d_in], W [d_out, d_in], H [T, r], B [d_out, r]."""
    _need(X, "X", 2)
    _need(W, "W", 2)
    _need(H, "H", 2)
    _need(B, "B", 2)
    T, d_in = X.shape
    d_out, r = W.shape[0], H.shape[1]
    if W.shape[1] != d_in or H.shape[0] != T or tuple(B.shape) != (d_out, r):
        raise ValueError("shapes do not match")
    if not (W.dtype == H.dtype == B.dtype == X.dtype):
        raise ValueError("X, W, H, B must share a dtype")
    Y = _out(Y, (T, d_out), out_dtype or X.dtype, X.device, "Y")
    wp, wn, keep = _workspace(TG_OP_GEMM_FWD_LORA, (T, d_out, d_in, r), _DT[X.dtype], _DT[Y.dtype], ws, X.device)
    _check(lib().tg_gemm_fwd_lora(_ptr(X), _ptr(W), _ptr(H), _ptr(B), _ptr(Y), T, d_out, d_in, r, float(scale),
                                  _DT[X.dtype], _DT[Y.dtype], wp, wn, _stream(stream)), "tg_gemm_fwd_lora")
    _keep(keep, stream)
    return Y


def tg_gemm_dgrad_lora(dY, W, dH, A, scale, dX=None, out_dtype=None, ws=None, stream=None):
    """dX = dY W + scale dH A in one product: dY [T, d_out], W [d_out, d_in], dH [T, r] FP32, A [r, d_in]."""
    _need(dY, "dY", 2)
    _need(W, "W", 2)
    _need(A, "A", 2)
    T, d_out = dY.shape
    d_in, r = W.shape[1], A.shape[0]
    if W.shape[0] != d_out or A.shape[1] != d_in or tuple(dH.shape) != (T, r):
        raise ValueError("shapes do not match")
    if dH.dtype != torch.float32 or not dH.is_contiguous() or dH.device != dY.device:
        raise ValueError("dH must be a contiguous FP32 tensor on the device of dY")
    if not (W.dtype == A.dtype == dY.dtype):
        raise ValueError("dY, W, A must share a dtype")
    dX = _out(dX, (T, d_in), out_dtype or dY.dtype, dY.device, "dX")
    wp, wn, keep = _workspace(TG_OP_GEMM_DGRAD_LORA, (T, d_out, d_in, r), _DT[dY.dtype], _DT[dX.dtype], ws, dY.device)
    _check(lib().tg_gemm_dgrad_lora(_ptr(dY), _ptr(W), _ptr(dH), _ptr(A), _ptr(dX), T, d_out, d_in, r, float(scale),
                                    _DT[dY.dtype], _DT[dX.dtype], wp, wn, _stream(stream)), "tg_gemm_dgrad_lora")
    _keep(keep, stream)
    return dX


def tg_gemm_wgrad_accumulate(dY, X, dW, ws=None, stream=None):
    """dW[d_out, d_in] += dY[T, d_out]^T X[T, d_in], dW an FP32 tensor."""
    _need(dY, "dY", 2), _need(X, "X", 2)
    T, d_out = dY.shape
    d_in = X.shape[1]
    if X.shape[0] != T or X.dtype != dY.dtype:
        raise ValueError("X must be [T, d_in] with dY's dtype")
    if dW is None or dW.dtype != torch.float32 or tuple(dW.shape) != (d_out, d_in) or not dW.is_contiguous():
        raise ValueError("dW must be a contiguous FP32 [d_out, d_in] tensor")
    wp, wn, keep = _workspace(TG_OP_GEMM_WGRAD, (T, d_out, d_in, 0), _DT[dY.dtype], _DT[torch.float32], ws, dY.device)
    _check(lib().tg_gemm_wgrad_accumulate(_ptr(dY), _ptr(X), _ptr(dW), T, d_out, d_in, _DT[dY.dtype], wp, wn,
                                          _stream(stream)), "tg_gemm_wgrad_accumulate")
    _keep(keep, stream)
    return dW
def tg_gemm_wgrad_noalloc(dY, X, dW, stream=None):
    """dW = dY^T X without any device allocation by the library (the split-K
    scratch is the library's own static array); dW must be given."""
    _need(dY, "dY", 2), _need(X, "X", 2), _need(dW, "dW", 2)
    T, d_out = dY.shape
    d_in = X.shape[1]
    if X.shape[0] != T or X.dtype != dY.dtype or tuple(dW.shape) != (d_out, d_in):
        raise ValueError("inconsistent shapes or dtypes")
    _check(lib().tg_gemm_wgrad_noalloc(_ptr(dY), _ptr(X), _ptr(dW), T, d_out, d_in, _DT[dY.dtype], _DT[dW.dtype],
                                       _stream(stream)), "tg_gemm_wgrad_noalloc")
    return dW


def tg_lora_down(X, A, H=None, out_dtype=None, ws=None, stream=None):
    """H[T, r] = X[T, d_in] A[r, d_in]^T."""
    _need(X, "X", 2), _need(A, "A", 2)
    T, d_in = X.shape
    r = A.shape[0]
    if A.shape[1] != d_in or A.dtype != X.dtype:
        raise ValueError("A must be [r, d_in] with X's dtype")
    H = _out(H, (T, r), out_dtype or X.dtype, X.device, "H")
    wp, wn, keep = _workspace(TG_OP_LORA_DOWN, (T, d_in, r, 0), _DT[X.dtype], _DT[H.dtype], ws, X.device)
    _check(lib().tg_lora_down(_ptr(X), _ptr(A), _ptr(H), T, d_in, r, _DT[X.dtype], _DT[H.dtype], wp, wn,
                              _stream(stream)), "tg_lora_down")
    _keep(keep, stream)
    return H


def tg_lora_up(H, B, Y=None, out_dtype=None, ws=None, stream=None):
    """Y[T, d_out] = H[T, r] B[d_out, r]^T."""
    _need(H, "H", 2), _need(B, "B", 2)
    T, r = H.shape
    d_out = B.shape[0]
    if B.shape[1] != r or B.dtype != H.dtype:
        raise ValueError("B must be [d_out, r] with H's dtype")
    Y = _out(Y, (T, d_out), out_dtype or H.dtype, H.device, "Y")
    wp, wn, keep = _workspace(TG_OP_LORA_UP, (T, d_out, r, 0), _DT[H.dtype], _DT[Y.dtype], ws, H.device)
    _check(lib().tg_lora_up(_ptr(H), _ptr(B), _ptr(Y), T, d_out, r, _DT[H.dtype], _DT[Y.dtype], wp, wn,
                            _stream(stream)), "tg_lora_up")
    _keep(keep, stream)
    return Y



def tg_lora_up_add(H, B, Y, scale, ws=None, stream=None):
    """Y[T, d_out] += scale * H[T, r] B[d_out, r]^T (one rounding to Y's type)."""
    _need(H, "H", 2), _need(B, "B", 2)
    T, r = H.shape
    d_out = B.shape[0]
    if B.shape[1] != r or B.dtype != H.dtype:
        raise ValueError("B must be [d_out, r] with H's dtype")
    if Y is None or tuple(Y.shape) != (T, d_out) or not Y.is_contiguous():
        raise ValueError("Y must be a contiguous [T, d_out] tensor")
    wp, wn, keep = _workspace(TG_OP_LORA_UP, (T, d_out, r, 0), _DT[H.dtype], _DT[Y.dtype], ws, H.device)
    _check(lib().tg_lora_up_add(_ptr(H), _ptr(B), _ptr(Y), T, d_out, r, float(scale), _DT[H.dtype], _DT[Y.dtype],
                                wp, wn, _stream(stream)), "tg_lora_up_add")
    _keep(keep, stream)
    return Y
def tg_lora_grad(X, A, B, H, dY, out_dtype=None, want_dH=False, outs=None, ws=None, stream=None):
    """Gradients of Y = (X A^T) B^T: returns dict dA, dB, dX (and dH in FP32 when asked)."""
    for t, n in ((X, "X"), (A, "A"), (B, "B"), (H, "H"), (dY, "dY")):
        _need(t, n, 2)
    T, d_in = X.shape
    r = A.shape[0]
    d_out = B.shape[0]
    if A.shape[1] != d_in or B.shape[1] != r or H.shape != (T, r) or dY.shape != (T, d_out):
        raise ValueError("inconsistent LoRA shapes")
    od = out_dtype or X.dtype
    outs = dict(outs or {})
    dA = _out(outs.get("dA"), (r, d_in), od, X.device, "dA")
    dB = _out(outs.get("dB"), (d_out, r), od, X.device, "dB")
    dX = _out(outs.get("dX"), (T, d_in), od, X.device, "dX")
    dH = _out(outs.get("dH"), (T, r), torch.float32, X.device, "dH") if (want_dH or "dH" in outs) else None
    din = _DT[X.dtype]
    wp, wn, keep = _workspace(TG_OP_LORA_GRAD, (T, d_in, d_out, r), din, _DT[od], ws, X.device)
    _check(lib().tg_lora_grad(_ptr(X), _ptr(A), _ptr(B), _ptr(H), _ptr(dY), _ptr(dA), _ptr(dB), _ptr(dX),
                              _ptr(dH), T, d_in, d_out, r, din, _DT[od], wp, wn, _stream(stream)), "tg_lora_grad")
    _keep(keep, stream)
    res = {"dA": dA, "dB": dB, "dX": dX}
    if dH is not None:
        res["dH"] = dH
    return res


def tg_lora_grad_add(X, A, B, H, dY, dX, scale, want_dH=False, outs=None, ws=None, stream=None):
    """Gradients of Y = X W^T + scale (X A^T) B^T with the LoRA part added into
    dX (the base layer's dgrad on entry): returns dict dA, dB (scaled), dX (the
    same tensor, updated) and dH (FP32, unscaled) when asked.  dA and dB take
    dX's dtype."""
    for t, n in ((X, "X"), (A, "A"), (B, "B"), (H, "H"), (dY, "dY")):
        _need(t, n, 2)
    T, d_in = X.shape
    r = A.shape[0]
    d_out = B.shape[0]
    if A.shape[1] != d_in or B.shape[1] != r or H.shape != (T, r) or dY.shape != (T, d_out):
        raise ValueError("inconsistent LoRA shapes")
    if dX is None or tuple(dX.shape) != (T, d_in) or not dX.is_contiguous():
        raise ValueError("dX must be a contiguous [T, d_in] tensor")
    od = dX.dtype
    outs = dict(outs or {})
    dA = _out(outs.get("dA"), (r, d_in), od, X.device, "dA")
    dB = _out(outs.get("dB"), (d_out, r), od, X.device, "dB")
    dH = _out(outs.get("dH"), (T, r), torch.float32, X.device, "dH") if (want_dH or "dH" in outs) else None
    din = _DT[X.dtype]
    wp, wn, keep = _workspace(TG_OP_LORA_GRAD, (T, d_in, d_out, r), din, _DT[od], ws, X.device)
    _check(lib().tg_lora_grad_add(_ptr(X), _ptr(A), _ptr(B), _ptr(H), _ptr(dY), _ptr(dA), _ptr(dB), _ptr(dX),
                                  _ptr(dH), T, d_in, d_out, r, float(scale), din, _DT[od], wp, wn, _stream(stream)),
           "tg_lora_grad_add")
    _keep(keep, stream)
    res = {"dA": dA, "dB": dB, "dX": dX}
    if dH is not None:
        res["dH"] = dH
    return res


def _need_f32(t, name, shape):
    _need(t, name, len(shape))
    if t.dtype != torch.float32 or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be an FP32 {tuple(shape)} tensor, got {t.dtype} {tuple(t.shape)}")


def tg_lora_down_f32w(X, A, H=None, out_dtype=None, ws=None, stream=None):
    """H[T, r] = X[T, d_in] A[r, d_in]^T with an FP32 factor A and 16-bit X."""
    _need(X, "X", 2)
    T, d_in = X.shape
    r = A.shape[0]
    _need_f32(A, "A", (r, d_in))
    H = _out(H, (T, r), out_dtype or X.dtype, X.device, "H")
    wp, wn, keep = _workspace(TG_OP_LORA_DOWN_F32W, (T, d_in, r, 0), _DT[X.dtype], _DT[H.dtype], ws, X.device)
    _check(lib().tg_lora_down_f32w(_ptr(X), _ptr(A), _ptr(H), T, d_in, r, _DT[X.dtype], _DT[H.dtype], wp, wn,
                                   _stream(stream)), "tg_lora_down_f32w")
    _keep(keep, stream)
    return H


def tg_lora_up_f32w(H, B, Y=None, out_dtype=None, ws=None, stream=None):
    """Y[T, d_out] = H[T, r] B[d_out, r]^T with an FP32 factor B and 16-bit H."""
    _need(H, "H", 2)
    T, r = H.shape
    d_out = B.shape[0]
    _need_f32(B, "B", (d_out, r))
    Y = _out(Y, (T, d_out), out_dtype or H.dtype, H.device, "Y")
    wp, wn, keep = _workspace(TG_OP_LORA_UP_F32W, (T, d_out, r, 0), _DT[H.dtype], _DT[Y.dtype], ws, H.device)
    _check(lib().tg_lora_up_f32w(_ptr(H), _ptr(B), _ptr(Y), T, d_out, r, _DT[H.dtype], _DT[Y.dtype], wp, wn,
                                 _stream(stream)), "tg_lora_up_f32w")
    _keep(keep, stream)
    return Y


def tg_lora_grad_f32w(X, A, B, H, dY, out_dtype=None, want_dH=False, outs=None, ws=None, stream=None):
    """Gradients of Y = (X A^T) B^T with FP32 factors A, B and 16-bit X, H, dY:
    dict dA, dB (FP32), dX (out_dtype, default X's) and dH (FP32) when asked."""
    for t, n in ((X, "X"), (H, "H"), (dY, "dY")):
        _need(t, n, 2)
    T, d_in = X.shape
    r = A.shape[0]
    d_out = B.shape[0]
    _need_f32(A, "A", (r, d_in))
    _need_f32(B, "B", (d_out, r))
    if H.shape != (T, r) or dY.shape != (T, d_out):
        raise ValueError("inconsistent LoRA shapes")
    od = out_dtype or X.dtype
    outs = dict(outs or {})
    dA = _out(outs.get("dA"), (r, d_in), torch.float32, X.device, "dA")
    dB = _out(outs.get("dB"), (d_out, r), torch.float32, X.device, "dB")
    dX = _out(outs.get("dX"), (T, d_in), od, X.device, "dX")
    dH = _out(outs.get("dH"), (T, r), torch.float32, X.device, "dH") if (want_dH or "dH" in outs) else None
    din = _DT[X.dtype]
    wp, wn, keep = _workspace(TG_OP_LORA_GRAD_F32W, (T, d_in, d_out, r), din, _DT[od], ws, X.device)
    _check(lib().tg_lora_grad_f32w(_ptr(X), _ptr(A), _ptr(B), _ptr(H), _ptr(dY), _ptr(dA), _ptr(dB), _ptr(dX),
                                   _ptr(dH), T, d_in, d_out, r, din, _DT[od], wp, wn, _stream(stream)),
           "tg_lora_grad_f32w")
    _keep(keep, stream)
    res = {"dA": dA, "dB": dB, "dX": dX}
    if dH is not None:
        res["dH"] = dH
    return res


def tg_attn_fwd(Q, K, V, O=None, scale=None, out_dtype=None, stream=None):
    """Fused attention forward: O = softmax(scale Q K^T) V per head; Q, K, V [heads, s, 64]."""
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, n, 3)
    heads, s, d = Q.shape
    if tuple(K.shape) != (heads, s, d) or tuple(V.shape) != (heads, s, d) or K.dtype != Q.dtype or V.dtype != Q.dtype:
        raise ValueError("K and V must match Q")
    O = _out(O, (heads, s, d), out_dtype or Q.dtype, Q.device, "O")
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    _check(lib().tg_attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), heads, s, d, sc, _DT[Q.dtype], _DT[O.dtype],
                             _stream(stream)), "tg_attn_fwd")
    return O


def tg_attn_bwd(Q, K, V, dO, scale=None, out_dtype=None, outs=None, ws=None, stream=None):
    """Fused attention backward: {"dQ", "dK", "dV"} of the forward of tg_attn_fwd given dO; all [heads, s, 64]."""
    for t, n in ((Q, "Q"), (K, "K"), (V, "V"), (dO, "dO")):
        _need(t, n, 3)
    heads, s, d = Q.shape
    for t in (K, V, dO):
        if tuple(t.shape) != (heads, s, d) or t.dtype != Q.dtype:
            raise ValueError("K, V and dO must match Q")
    outs = dict(outs or {})
    dt = out_dtype or (next(iter(outs.values())).dtype if outs else Q.dtype)
    res = {k: _out(outs.get(k), (heads, s, d), dt, Q.device, k) for k in ("dQ", "dK", "dV")}
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    wptr, wbytes, buf = _workspace(TG_OP_ATTN_BWD, (heads, s, d, 0), _DT[Q.dtype], _DT[dt], ws, Q.device)
    _check(lib().tg_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(res["dQ"]), _ptr(res["dK"]), _ptr(res["dV"]),
                             heads, s, d, sc, _DT[Q.dtype], _DT[dt], wptr, wbytes, _stream(stream)), "tg_attn_bwd")
    if buf is not ws:
        _keep(buf, stream)
    return res


def tg_bmm_attn(op, A, B, C=None, out_dtype=None, ws=None, stream=None):
    """One of the attention products (see include/tg.h); op is a name or a tg_attn_op value."""
    code = ATTN_OPS[op] if isinstance(op, str) else int(op)
    _need(A, "A", 3), _need(B, "B", 3)
    batch, s, d = B.shape
    ss_out = code in (0, 2)
    if code in (0, 2):
        if tuple(A.shape) != (batch, s, d):
            raise ValueError("A must be [batch, s, d]")
    elif tuple(A.shape) != (batch, s, s):
        raise ValueError("A must be [batch, s, s]")
    C = _out(C, (batch, s, s if ss_out else d), out_dtype or A.dtype, A.device, "C")
    wp, wn, keep = _workspace(TG_OP_BMM_ATTN, (code, batch, s, d), _DT[A.dtype], _DT[C.dtype], ws, A.device)
    _check(lib().tg_bmm_attn(code, _ptr(A), _ptr(B), _ptr(C), batch, s, d, _DT[A.dtype], _DT[C.dtype], wp, wn,
                             _stream(stream)), "tg_bmm_attn")
    _keep(keep, stream)
    return C


def tg_workspace_size(op, d0, d1, d2, d3, din, dout) -> int:
    return lib().tg_workspace_size(op, d0, d1, d2, d3, _DT.get(din, din), _DT.get(dout, dout))


def tg_stream_status(stream=None) -> int:
    return lib().tg_stream_status(_stream(stream))


def tg_status_string(status: int) -> str:
    return lib().tg_status_string(status).decode()


def tg_load_table(path) -> int:
    return lib().tg_load_table(None if path is None else str(path).encode())


def tg_version() -> int:
    return lib().tg_version()


def tg_plan_describe(op, M, N, K, batch, din, dout, sms) -> str:
    """The plan the tensor-core path would use (host only; see include/tg.h)."""
    buf = ctypes.create_string_buffer(512)
    n = lib().tg_plan_describe(op, M, N, K, batch, _DT[din], _DT[dout], sms, buf, 512)
    return buf.value.decode() if n else ""


def tg_last_call() -> str:
    buf = ctypes.create_string_buffer(512)
    lib().tg_last_call(buf, 512)
    return buf.value.decode()


def tg_wait_probe(timeout_us: int, stream=None) -> int:
    return lib().tg_wait_probe(timeout_us, _stream(stream))
