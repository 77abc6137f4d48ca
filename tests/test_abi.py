"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every symbol include/tg.h declares, and rejects bad arguments before
any device work.  The tile-table reader is host logic and is checked here too."""
import ctypes
import os
import re

import pytest

from gemms_linear_layers_gb300 import _binding as B
from gemms_linear_layers_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tg.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tg_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("tg_gemm_fwd", "tg_gemm_dgrad", "tg_gemm_wgrad", "tg_lora_down", "tg_lora_up",
              "tg_lora_grad", "tg_bmm_attn", "tg_workspace_size", "tg_stream_status"):
        assert n in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert n in B.SIGNATURES, n
    assert lib.tg_version() == 10000


def test_package_exports_every_entry_point():
    """The package's public names are the binding's, and every C entry point
    that computes something is among them."""
    import gemms_linear_layers_gb300 as pkg
    for n in pkg.__all__:
        assert hasattr(B, n), n
    for n in declared_functions():
        if n.startswith(("tg_gemm", "tg_lora", "tg_bmm", "tg_attn")):
            assert n in pkg.__all__, n


def test_status_strings(lib):
    for code in range(9):
        s = lib.tg_status_string(code)
        assert s and s != b"unknown status"
    assert lib.tg_status_string(99) == b"unknown status"


NULL = ctypes.c_void_p(0)
ODD = ctypes.c_void_p(0x1001)   # never dereferenced: checks fail first
EVEN = ctypes.c_void_p(0x1000)


@pytest.mark.parametrize("fn", ["tg_gemm_fwd", "tg_gemm_dgrad", "tg_gemm_wgrad"])
def test_layer_products_reject_bad_arguments(lib, fn):
    f = getattr(lib, fn)
    # negative size
    assert f(EVEN, EVEN, EVEN, -1, 8, 8, B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 1
    assert f(EVEN, EVEN, EVEN, 8, 8, 1 << 31, B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 1
    # unsupported dtypes: a 16-bit output of FP32 inputs or of the other 16-bit type
    assert f(EVEN, EVEN, EVEN, 8, 8, 8, B.TG_F32, B.TG_BF16, NULL, 0, NULL) == 2
    assert f(EVEN, EVEN, EVEN, 8, 8, 8, B.TG_BF16, B.TG_F16, NULL, 0, NULL) == 2
    # FP32 operands are 4-byte elements
    assert f(ctypes.c_void_p(0x1002), EVEN, EVEN, 8, 8, 8, B.TG_F32, B.TG_F32, NULL, 0, NULL) == 3
    assert f(EVEN, EVEN, EVEN, 8, 8, 8, 7, B.TG_F32, NULL, 0, NULL) == 2
    # NULL operand with a non-empty tensor
    assert f(NULL, EVEN, EVEN, 8, 8, 8, B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 1
    # pointer not aligned to its element
    assert f(ODD, EVEN, EVEN, 8, 8, 8, B.TG_F16, B.TG_F16, NULL, 0, NULL) == 3
    assert f(EVEN, EVEN, ctypes.c_void_p(0x1002), 8, 8, 8, B.TG_F16, B.TG_F32, NULL, 0, NULL) == 3


def test_lora_and_attention_reject_bad_arguments(lib):
    assert lib.tg_lora_down(EVEN, EVEN, EVEN, 8, -8, 16, B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 1
    assert lib.tg_lora_up(EVEN, EVEN, EVEN, 8, 8, 16, B.TG_F32, B.TG_F32, NULL, 0, NULL) == 2
    assert lib.tg_lora_grad(EVEN, EVEN, EVEN, EVEN, NULL, EVEN, EVEN, EVEN, NULL, 8, 8, 8, 16,
                            B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 1
    assert lib.tg_bmm_attn(0, EVEN, EVEN, EVEN, 2, -4, 8, B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 1
    assert lib.tg_bmm_attn(9, EVEN, EVEN, EVEN, 2, 4, 8, B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 1
    assert lib.tg_wait_probe(0, NULL) == 1
    assert lib.tg_wait_probe(10 ** 8, NULL) == 1
    assert lib.tg_workspace_size(B.TG_OP_LORA_UP, 8, 8, 8, 0, B.TG_F32, B.TG_F32) == B.SIZE_MAX  # FP32: layers only
    assert lib.tg_workspace_size(B.TG_OP_GEMM_FWD, 8, 8, 8, 0, B.TG_F32, B.TG_BF16) == B.SIZE_MAX
    assert lib.tg_workspace_size(0, -8, 8, 8, 0, B.TG_BF16, B.TG_F32) == B.SIZE_MAX


def test_accumulating_entry_points_reject_bad_arguments(lib):
    """All are checked before any device work: the accumulating weight
    gradient takes 16-bit operands and an aligned FP32 buffer; the LoRA
    up-add and gradient-add take a finite scale."""
    f = lib.tg_gemm_wgrad_accumulate
    assert f(EVEN, EVEN, EVEN, 8, -8, 8, B.TG_BF16, NULL, 0, NULL) == 1
    assert f(EVEN, EVEN, EVEN, 8, 8, 8, 7, NULL, 0, NULL) == 2
    assert f(ctypes.c_void_p(0x1002), EVEN, EVEN, 8, 8, 8, B.TG_F32, NULL, 0, NULL) == 3  # FP32 dY not 4-aligned
    assert f(EVEN, EVEN, ctypes.c_void_p(0x1002), 8, 8, 8, B.TG_BF16, NULL, 0, NULL) == 3  # dW not 4-aligned
    g = lib.tg_lora_up_add
    assert g(EVEN, EVEN, EVEN, 8, 8, 16, float("nan"), B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 1
    assert g(EVEN, EVEN, EVEN, 8, 8, 16, float("inf"), B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 1
    assert g(EVEN, EVEN, EVEN, 8, 8, 16, 2.0, B.TG_BF16, B.TG_F16, NULL, 0, NULL) == 2
    h = lib.tg_lora_grad_add
    for bad in (float("nan"), float("-inf")):
        assert h(EVEN, EVEN, EVEN, EVEN, EVEN, EVEN, EVEN, EVEN, NULL, 8, 8, 8, 16, bad,
                 B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 1
    assert h(EVEN, EVEN, EVEN, EVEN, EVEN, EVEN, EVEN, EVEN, NULL, 8, -8, 8, 16, 1.0,
             B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 1
    assert h(EVEN, EVEN, EVEN, EVEN, EVEN, EVEN, EVEN, EVEN, NULL, 8, 8, 8, 16, 1.0,
             B.TG_F32, B.TG_F32, NULL, 0, NULL) == 2


def test_fp32_factor_lora_rejects_bad_arguments(lib):
    """The FP32 factors are 4-byte elements; the activations stay 16-bit."""
    A2 = ctypes.c_void_p(0x1002)  # aligned for 16-bit, not for FP32
    assert lib.tg_lora_down_f32w(EVEN, A2, EVEN, 8, 8, 16, B.TG_BF16, B.TG_BF16, NULL, 0, NULL) == 3
    assert lib.tg_lora_down_f32w(EVEN, EVEN, EVEN, 8, 8, 16, B.TG_F32, B.TG_F32, NULL, 0, NULL) == 2
    assert lib.tg_lora_up_f32w(EVEN, A2, EVEN, 8, 8, 16, B.TG_F16, B.TG_F32, NULL, 0, NULL) == 3
    assert lib.tg_lora_up_f32w(EVEN, EVEN, EVEN, -8, 8, 16, B.TG_F16, B.TG_F32, NULL, 0, NULL) == 1
    f = lib.tg_lora_grad_f32w
    assert f(EVEN, EVEN, A2, EVEN, EVEN, EVEN, EVEN, EVEN, NULL, 8, 8, 8, 16, B.TG_BF16, B.TG_BF16,
             NULL, 0, NULL) == 3  # B
    assert f(EVEN, EVEN, EVEN, EVEN, EVEN, A2, EVEN, EVEN, NULL, 8, 8, 8, 16, B.TG_BF16, B.TG_BF16,
             NULL, 0, NULL) == 3  # dA is FP32
    assert f(EVEN, EVEN, EVEN, EVEN, NULL, EVEN, EVEN, EVEN, NULL, 8, 8, 8, 16, B.TG_BF16, B.TG_BF16,
             NULL, 0, NULL) == 1  # no dY


def test_fused_attention_rejects_bad_arguments(lib):
    f = lib.tg_attn_fwd
    assert f(EVEN, EVEN, EVEN, EVEN, 2, 64, 32, 0.125, B.TG_BF16, B.TG_BF16, NULL) == 1  # head dim must be 64
    assert f(EVEN, EVEN, EVEN, EVEN, 2, 64, 64, float("nan"), B.TG_BF16, B.TG_BF16, NULL) == 1
    assert f(EVEN, EVEN, EVEN, EVEN, 2, -1, 64, 0.125, B.TG_BF16, B.TG_BF16, NULL) == 1
    assert f(EVEN, EVEN, EVEN, EVEN, 2, 64, 64, 0.125, B.TG_F32, B.TG_F32, NULL) == 2
    assert f(EVEN, ctypes.c_void_p(0x1008), EVEN, EVEN, 2, 64, 64, 0.125, B.TG_BF16, B.TG_BF16, NULL) == 3  # 16 B


def test_tile_table_reader(lib, tmp_path):
    good = tmp_path / "t.txt"
    good.write_text("# op in out M N K batch bn splits\n"
                    "fwd bf16 bf16 2048 576 576 1 192 1\n"
                    "tn f16 f32 2304 2304 4096 1 256 2   # trailing comment\n\n")
    assert lib.tg_load_table(str(good).encode()) == 0
    bad = tmp_path / "bad.txt"
    bad.write_text("fwd bf16 bf16 2048 576\n")
    assert lib.tg_load_table(str(bad).encode()) == 7
    bad.write_text("fwd bf16 bf16 2048 576 576 1 100 1\n")  # tile width not offered
    assert lib.tg_load_table(str(bad).encode()) == 7
    bad.write_text("xyz bf16 bf16 2048 576 576 1 128 1\n")
    assert lib.tg_load_table(str(bad).encode()) == 7
    assert lib.tg_load_table(str(tmp_path / "missing.txt").encode()) == 7
    assert lib.tg_load_table(None) == 0
    # the committed table parses
    committed = os.path.join(ROOT, "gemms_linear_layers_gb300", "tables", "gb300.txt")
    if os.path.exists(committed):
        assert lib.tg_load_table(committed.encode()) == 0
        assert lib.tg_load_table(None) == 0


def test_last_call_buffer(lib):
    buf = ctypes.create_string_buffer(4)
    n = lib.tg_last_call(buf, 4)
    assert n >= 0 and len(buf.value) <= 3


def test_tile_table_schedules(lib, tmp_path):
    """Table tokens for the schedules: stream-K (sk) and tail split (tN) need
    64-column multiples; 144-wide tiles take plain split counts; CTA pairs
    ("p" after the width) take widths 128, 192 and 256 with every schedule;
    the cluster split-K (cN, 2 <= N <= 8) takes single-CTA widths 64..256."""
    t = tmp_path / "s.txt"
    t.write_text("tn bf16 bf16 2304 2304 2048 1 256 sk n\n"
                 "tn bf16 bf16 2304 2304 4096 1 256 t4 m\n"
                 "nt bf16 f32 1024 2304 2304 1 144 1 n\n"
                 "nn f16 f16 1024 2304 5760 1 144 2\n"
                 "nt bf16 bf16 2048 49152 576 1 256p 1 m\n"
                 "nn bf16 bf16 2048 576 49152 1 192p 3\n"
                 "tn f16 f32 576 576 2048 1 128p 2 n\n"
                 "tn bf16 bf16 2304 2304 2048 1 256p sk m\n"
                 "tn bf16 bf16 2304 2304 4096 1 256p t13 m\n"
                 "nt bf16 bf16 2048 576 1536 1 192 c3 m\n"
                 "tn f16 f32 576 576 2048 1 64 c8\n")
    assert lib.tg_load_table(str(t).encode()) == 0
    for bad in ("tn bf16 bf16 2304 2304 2048 1 144 sk\n", "tn bf16 bf16 2304 2304 2048 1 144 t2\n",
                "tn bf16 bf16 2304 2304 2048 1 256 t1\n", "tn bf16 bf16 2304 2304 2048 1 256 tx\n",
                "tn bf16 bf16 2304 2304 2048 1 160 1\n", "tn bf16 bf16 2304 2304 2048 1 64p 1\n",
                "tn bf16 bf16 2304 2304 2048 1 144p 1\n",
                "tn bf16 bf16 2304 2304 2048 1 256q 1\n", "nt bf16 bf16 2048 576 1536 1 192p c3\n",
                "nt bf16 bf16 2048 576 1536 1 144 c3\n", "nt bf16 bf16 2048 576 1536 1 192 c1\n",
                "nt bf16 bf16 2048 576 1536 1 192 c9\n", "nt bf16 bf16 2048 576 1536 1 192 cx\n",
                "tn bf16 bf16 2304 2304 2048 1 256pp 1\n"):
        t.write_text(bad)
        assert lib.tg_load_table(str(t).encode()) == 7, bad
    assert lib.tg_load_table(None) == 0


def _plan(op, M, N, K, batch=1, sms=152):
    import torch
    return B.tg_plan_describe(op, M, N, K, batch, torch.bfloat16, torch.bfloat16, sms)


def test_plan_describe_reports_table_entries_and_the_cuda_core_path(lib):
    import torch
    """tg_plan_describe (host only) gives the plan a call would use: a shipped
    table entry is reported as a hit; sizes the tensor-core path cannot
    address go to the CUDA-core path; bad arguments give an empty answer."""
    assert lib.tg_load_table(B.DEFAULT_TABLE.encode()) == 0
    try:
        p = _plan(B.TG_OP_GEMM_FWD, 2048, 49152, 576)
        assert p.startswith("tc nt M=2048 N=49152 K=576 batch=1 bn=") and "table=hit" in p, p
        assert _plan(B.TG_OP_GEMM_FWD, 3000, 1000, 700) == "simt nt"  # K = 700: rows of 1,400 bytes
        assert _plan(B.TG_OP_GEMM_WGRAD, 0, 576, 2048) == ""
        assert _plan(B.TG_OP_LORA_DOWN, 2048, 576, 16) == ""
        # FP32 operands: three bf16 parts each on the tensor cores (a reduction six
        # times as long) when the pitches allow TMA, else the FFMA kernel, split
        # along K when few tiles would occupy the SMs
        f32 = lambda op, M, N, K: B.tg_plan_describe(op, M, N, K, 1, torch.float32, torch.float32, 152)
        assert f32(B.TG_OP_GEMM_FWD, 4096, 5760, 2304).startswith("tc3 nt M=4096 N=5760 K=13824 batch=1 bn=")
        assert f32(B.TG_OP_GEMM_DGRAD, 2048, 576, 49152).startswith("tc3 nn M=2048 N=576 K=294912 ")
        assert " cs " not in f32(B.TG_OP_GEMM_WGRAD, 576, 576, 2048)  # no cluster split for the parts
        assert f32(B.TG_OP_GEMM_FWD, 1000, 1001, 999) == "ffma nt splits=1"  # rows of 999 floats
        assert f32(B.TG_OP_GEMM_DGRAD, 2048, 578, 49152) == "ffma nn splits=3"
        assert B.tg_plan_describe(B.TG_OP_GEMM_FWD, 64, 64, 64, 1, torch.float32, torch.bfloat16, 152) == ""
    finally:
        assert lib.tg_load_table(None) == 0


@pytest.mark.parametrize("case", [
    # (op, M, N, K, batch, must contain, must not contain): choices measured to matter
    (2, 2304, 2304, 4096, 1, " pair", " bn=144"),   # square weight gradient: pairs, not 144-wide single CTAs
    (0, 2048, 49152, 576, 1, "bn=256 pair", None),   # the vocabulary head forward
    (1, 2048, 576, 1536, 1, "bn=64 splits=1", " cs"),  # a cluster split of 3 x 48 tiles would not fit at once
    (2, 576, 576, 2048, 1, " cs ", " sk"),           # small weight gradient: cluster split, not stream-K
    (1, 1024, 64, 1024, 36, "bn=64", None),          # 64-wide attention products: no wider tile
    (0, 2048, 2048, 64, 36, "bn=256 splits=1", " sk"),  # one K block per tile: no stream-K
])
def test_cost_model_choices_without_a_table(lib, case):
    """With no table entry, the cost model must avoid the plans measured to be
    2x slower than the best (see the sweep's 'heuristic' column)."""
    op, M, N, K, batch, want, avoid = case
    assert lib.tg_load_table(b"") == 0
    try:
        p = _plan(op, M, N, K, batch)
        assert "table=miss" in p and want in p, p
        if avoid:
            assert avoid not in p, p
    finally:
        assert lib.tg_load_table(None) == 0


def _plan_fields(p):
    f = p.split()
    kv = dict(x.split("=", 1) for x in f if "=" in x)
    return f, kv


@pytest.mark.parametrize("seed", range(4))
def test_cost_model_plans_are_well_formed(lib, seed):
    """Over random shapes (no table), every plan the cost model makes is one
    the kernels can run: a tile width they offer, CTA pairs only over more
    than 128 rows, no more K splits than 64-deep K blocks, cluster splits of
    2-8 CTAs whose clusters all fit on the 152 SMs at once, never stream-K
    (whose waits need the whole grid resident), and the CUDA-core path exactly when
    a row pitch is not a multiple of 16 bytes."""
    import random
    import torch
    rng = random.Random(seed)
    assert lib.tg_load_table(None) == 0
    sizes = [1, 7, 16, 64, 100, 128, 129, 192, 256, 576, 1000, 1536, 2048, 2304, 4096, 5760, 49152]
    for _ in range(150):
        op = rng.randrange(3)
        M, N, K = (rng.choice(sizes) for _ in range(3))
        batch = rng.choice([1, 1, 1, 4, 36])
        dout = rng.choice([torch.bfloat16, torch.float32])
        p = B.tg_plan_describe(op, M, N, K, batch, torch.bfloat16, dout, 152)
        layout = ("nt", "nn", "tn")[op]
        lda, ldb = (M if layout == "tn" else K), (K if layout == "nt" else N)
        ob = 4 if dout == torch.float32 else 2
        misaligned = (lda * 2) % 16 or (ldb * 2) % 16 or (N * ob) % 16
        if misaligned:
            assert p == f"simt {layout}", (op, M, N, K, batch, p)
            continue
        f, kv = _plan_fields(p)
        assert f[0] == "tc" and f[1] == layout, p
        bn = int(kv["bn"])
        assert bn in (64, 128, 144, 192, 256), p
        kb = -(-K // 64)
        if "pair" in f:
            assert M > 128 and bn in (128, 192, 256), p
        # stream-K needs its whole grid resident; only a table entry may pick it
        assert "sk" not in f, p
        assert 1 <= int(kv["splits"]) <= kb, p
        if "cs" in f:
            cs = int(kv["cluster"])
            tiles = batch * -(-M // 128) * -(-N // bn)
            assert 2 <= cs <= 8 and cs <= kb and tiles * cs <= 152, p
        if "tail" in kv:  # the tiles of the last partial wave, each cut into K pieces
            tail_tiles, pieces = (int(x) for x in kv["tail"].split("x"))
            tiles = batch * -(-M // (256 if "pair" in f else 128)) * -(-N // bn)
            assert 1 <= tail_tiles < tiles and 2 <= pieces <= kb, p
