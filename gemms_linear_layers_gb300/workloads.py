"""The product sets the library is measured and checked on (shapes only).

Page "Twice the training speed on a BC-250 from tuned matrix kernels", section
"Tuning the kernels": every layer of a 135M-class and a 2B-class decoder at
1,024, 2,048 and 4,096 tokens, the rank-16 LoRA matrices and the batched
products inside attention, in bf16 and fp16 with FP32 accumulation.

Each layer is (name, d_in, d_out); its three products at T tokens are
forward T x d_out x d_in, input gradient T x d_in x d_out and weight gradient
d_out x d_in x T (rows x columns x reduction).
"""
from __future__ import annotations

import torch

DTYPES = (torch.bfloat16, torch.float16)

# one linear layer, 576 -> 1536 at 1,024 tokens (the small case)
SINGLE_LAYER = {"T": 1024, "layers": [("proj", 576, 1536)], "dtypes": (torch.bfloat16,)}

# 135M-class decoder, hidden 576, at 2,048 tokens
LAYERS_135M = [
    ("q", 576, 576), ("k", 576, 192), ("v", 576, 192), ("o", 576, 576),
    ("gate", 576, 1536), ("up", 576, 1536), ("down", 1536, 576), ("head", 576, 49152),
]
DECODER_135M = {"T": 2048, "layers": LAYERS_135M, "dtypes": DTYPES}

# 2B-class decoder, hidden 2304, at 1,024 / 2,048 / 4,096 tokens
LAYERS_2B = [
    ("q", 2304, 2304), ("k", 2304, 2304), ("v", 2304, 2304), ("o", 2304, 2304),
    ("gate", 2304, 5760), ("up", 2304, 5760), ("down", 5760, 2304),
]
DECODER_2B = {"T": (1024, 2048, 4096), "layers": LAYERS_2B, "dtypes": DTYPES}

# rank-16 LoRA on every projection of the 2B-class layer set, 4,096 tokens, bf16
LORA_2B = {"T": 4096, "r": 16, "layers": LAYERS_2B, "dtypes": (torch.bfloat16,)}

# batched attention products: 36 heads, head_dim 64, batch 1
ATTENTION = {"heads": 36, "d": 64, "s": (1024, 2048, 4096), "dtypes": DTYPES,
             "ops": ("qk", "pv", "do_vt", "pt_do", "ds_k", "dst_q")}


def layer_products(T, layers):
    """[(layer, op, M, N, K)] with M x N the output and K the reduction length."""
    out = []
    for name, d_in, d_out in layers:
        out.append((name, "fwd", T, d_out, d_in))
        out.append((name, "dgrad", T, d_in, d_out))
        out.append((name, "wgrad", d_out, d_in, T))
    return out


def flops(M, N, K, batch=1) -> int:
    """Multiply-adds counted as two operations: 2 M N K per product."""
    return 2 * M * N * K * batch
