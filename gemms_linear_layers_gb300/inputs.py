"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no arithmetic of the products themselves: it only draws
random tensors.  Every tensor is drawn in fp32 from a seeded generator, scaled,
and rounded to its 16-bit type with round-to-nearest-even (``Tensor.to``).  The
rounded tensor is the single source of truth: the GPU receives a copy of it and
the oracle decodes it exactly.

Value distributions follow the layer shapes the page tunes for ("Twice the
training speed on a BC-250 from tuned matrix kernels", section "Tuning the
kernels": every layer of a 135M-class and a 2B-class decoder, the rank-16 LoRA
matrices and the batched products inside attention):

* activations X ~ N(0, 1), weights W ~ N(0, 0.02), output gradients
  dY ~ N(0, 0.01); the second parameter is a standard deviation;
* LoRA factors A, B ~ N(0, 0.02); the LoRA activation H (an input of the up
  product and of the gradients) is drawn on its own, N(0, 0.02 * sqrt(d_in)),
  the spread X A^T has for these X and A;
* attention Q, K, V ~ N(0, 1); P = U(0, 1) with each row divided by its sum
  (in fp32, before rounding); dO, dS ~ N(0, 0.01).
"""
from __future__ import annotations

import math
import zlib

import torch

STD_X, STD_W, STD_G = 1.0, 0.02, 0.01
STD_LORA = 0.02


def seed_for(*parts) -> int:
    """Stable 32-bit seed from a description of the tensor."""
    return zlib.crc32("/".join(str(p) for p in parts).encode())


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std, dtype, seed, device="cpu") -> torch.Tensor:
    """N(0, std^2) drawn in fp32, then rounded to ``dtype``."""
    g = _gen(seed, device)
    t = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def rownorm_uniform(shape, dtype, seed, device="cpu") -> torch.Tensor:
    """U(0,1) with every row (last dim) divided by its fp32 sum, then rounded."""
    g = _gen(seed, device)
    t = torch.rand(tuple(shape), generator=g, dtype=torch.float32, device=device)
    t.div_(t.sum(dim=-1, keepdim=True))
    return t.to(dtype)


def small_int(shape, lo, hi, dtype, seed, device="cpu") -> torch.Tensor:
    """Integers in [lo, hi], exact in every 16-bit type for |v| <= 256."""
    g = _gen(seed, device)
    t = torch.randint(lo, hi + 1, tuple(shape), generator=g, dtype=torch.int32, device=device)
    return t.to(dtype)


def layer_inputs(T, d_in, d_out, dtype, tag="layer", device="cpu"):
    """(X [T, d_in], W [d_out, d_in], dY [T, d_out]) for one linear layer."""
    name = str(dtype).replace("torch.", "")
    X = normal((T, d_in), STD_X, dtype, seed_for(tag, T, d_in, d_out, name, "X"), device)
    W = normal((d_out, d_in), STD_W, dtype, seed_for(tag, T, d_in, d_out, name, "W"), device)
    dY = normal((T, d_out), STD_G, dtype, seed_for(tag, T, d_in, d_out, name, "dY"), device)
    return X, W, dY


def lora_inputs(T, d_in, d_out, r, dtype, tag="lora", device="cpu"):
    """(X, A, B, H, dY) for a rank-r LoRA branch on a d_in -> d_out projection."""
    name = str(dtype).replace("torch.", "")
    key = (tag, T, d_in, d_out, r, name)
    X = normal((T, d_in), STD_X, dtype, seed_for(*key, "X"), device)
    A = normal((r, d_in), STD_LORA, dtype, seed_for(*key, "A"), device)
    B = normal((d_out, r), STD_LORA, dtype, seed_for(*key, "B"), device)
    H = normal((T, r), STD_LORA * math.sqrt(d_in), dtype, seed_for(*key, "H"), device)
    dY = normal((T, d_out), STD_G, dtype, seed_for(*key, "dY"), device)
    return X, A, B, H, dY


def attn_inputs(heads, s, d, dtype, tag="attn", device="cpu"):
    """Dict of Q, K, V, P, dO, dS for the batched attention products."""
    name = str(dtype).replace("torch.", "")
    key = (tag, heads, s, d, name)
    return {
        "Q": normal((heads, s, d), STD_X, dtype, seed_for(*key, "Q"), device),
        "K": normal((heads, s, d), STD_X, dtype, seed_for(*key, "K"), device),
        "V": normal((heads, s, d), STD_X, dtype, seed_for(*key, "V"), device),
        "P": rownorm_uniform((heads, s, s), dtype, seed_for(*key, "P"), device),
        "dO": normal((heads, s, d), STD_G, dtype, seed_for(*key, "dO"), device),
        "dS": normal((heads, s, s), STD_G, dtype, seed_for(*key, "dS"), device),
    }


# which inputs each attention product takes, in (A, B) order
ATTN_OPERANDS = {
    "qk": ("Q", "K"),
    "pv": ("P", "V"),
    "do_vt": ("dO", "V"),
    "pt_do": ("P", "dO"),
    "ds_k": ("dS", "K"),
    "dst_q": ("dS", "Q"),
}
