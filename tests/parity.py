"""Comparison helpers: GPU results against the fp64 oracle.

Tolerances (the pages fix none; they follow from the arithmetic of an FP32
accumulation over exactly represented 16-bit inputs):
  FP32 output:   |C - C*| <= 1e-5 * S*             elementwise
  16-bit output: |C - C*| <= ulp(C*) + 1e-5 * S*   (the FP32 tolerance plus
                 one unit of the output grid for the final rounding)
where C* is the exact product and S* = sum_k |a_ik b_kj| (both from the oracle).
"""
import numpy as np
import torch

import oracle

REL = 1e-5


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_close(got, ref, scale, what, out_dtype=None, rel=REL):
    """got: GPU tensor (any shape) or float64 array; ref/scale: float64 arrays."""
    g = to_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64).reshape(g.shape)
    scale = np.asarray(scale, dtype=np.float64).reshape(g.shape)
    bound = rel * scale
    if out_dtype in (torch.bfloat16, torch.float16):
        bound = bound + oracle.ulp16(ref, out_dtype)
    err = np.abs(g - ref)
    bad = ~(err <= bound)  # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.nanmax(np.where(bound > 0, err / np.maximum(bound, 1e-300), np.inf))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance "
                             f"(worst err/bound {worst:.3g}); first at {idx.tolist()}: "
                             f"got {g[tuple(idx[0])]} want {ref[tuple(idx[0])]} scale {scale[tuple(idx[0])]}")


def exact_rne_fraction(got16, ref, dtype) -> float:
    """Share of 16-bit outputs equal to the correctly rounded exact product."""
    want = oracle.round16(np.asarray(ref, dtype=np.float64), dtype)
    have = got16.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16).reshape(want.shape)
    return float(np.mean(have == want))


def sample_coords(M, N, batch=1, rows=128, cols=128, rand=8192, seed=0):
    """Coordinates of `rows` full rows, `cols` full columns and `rand` random
    elements (spread over the batch), for products too large for a full check."""
    rng = np.random.default_rng(seed)
    bi, ii, jj = [], [], []
    rsel = rng.choice(M, size=min(rows, M), replace=False)
    rb = rng.integers(0, batch, len(rsel))
    for b, i in zip(rb, rsel):
        bi.append(np.full(N, b))
        ii.append(np.full(N, i))
        jj.append(np.arange(N))
    csel = rng.choice(N, size=min(cols, N), replace=False)
    cb = rng.integers(0, batch, len(csel))
    for b, j in zip(cb, csel):
        bi.append(np.full(M, b))
        ii.append(np.arange(M))
        jj.append(np.full(M, j))
    bi.append(rng.integers(0, batch, rand))
    ii.append(rng.integers(0, M, rand))
    jj.append(rng.integers(0, N, rand))
    # the four corners: tile tails
    for b in (0, batch - 1):
        for i in (0, M - 1):
            for j in (0, N - 1):
                bi.append([b]); ii.append([i]); jj.append([j])
    return (np.concatenate(bi).astype(np.int64), np.concatenate(ii).astype(np.int64),
            np.concatenate(jj).astype(np.int64))


def sample_coords_every_batch(M, N, batch, rows=128, cols=128, rand=8192, seed=0):
    """Like sample_coords, but the full rows and columns are dealt to the
    batch entries in turn, so every entry (every attention head) has at least
    one full row and one full column checked when rows, cols >= batch."""
    rng = np.random.default_rng(seed)
    bi, ii, jj = [], [], []
    for t in range(rows):
        b, i = t % batch, int(rng.integers(0, M))
        bi.append(np.full(N, b)); ii.append(np.full(N, i)); jj.append(np.arange(N))
    for t in range(cols):
        b, j = t % batch, int(rng.integers(0, N))
        bi.append(np.full(M, b)); ii.append(np.arange(M)); jj.append(np.full(M, j))
    bi.append(rng.integers(0, batch, rand))
    ii.append(rng.integers(0, M, rand))
    jj.append(rng.integers(0, N, rand))
    for b in (0, batch - 1):
        for i in (0, M - 1):
            for j in (0, N - 1):
                bi.append([b]); ii.append([i]); jj.append([j])
    return (np.concatenate(bi).astype(np.int64), np.concatenate(ii).astype(np.int64),
            np.concatenate(jj).astype(np.int64))


def gather(t: torch.Tensor, coords):
    """Values of a GPU tensor ([M,N] or [batch,M,N]) at sampled coordinates, as float64."""
    bi, ii, jj = (torch.from_numpy(c).to(t.device) for c in coords)
    if t.dim() == 2:
        v = t[ii, jj]
    else:
        v = t[bi, ii, jj]
    return to_f64(v)
