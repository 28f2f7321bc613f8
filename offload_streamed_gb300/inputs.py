"""Seeded synthetic inputs for the streamed tiled linear operator.

This module holds no arithmetic of the method: it only draws random numbers
and writes bf16 bit patterns.  The tests feed the SAME host bytes to the CPU
oracle and to the GPU library, so neither side depends on how the numbers were
drawn.

Distributions (the workloads are FFN projections, X [T,K] activations, W
[K,M] weights, dY [T,M] output gradients):
    X  ~ N(0, 1)        bf16 (round-to-nearest-even from fp32)
    W  ~ N(0, 1/K)      bf16, drawn tile by tile: tile i = columns
                        [i*Mi, (i+1)*Mi) comes from its own generator stream,
                        so the logical W does not depend on the host layout
    dY ~ N(0, 1)        bf16
    ternary:            values in {-1, 0, +1} (exact-arithmetic cases)

Generators: ``torch.Generator(device).manual_seed(stream_seed(seed, j, i))``
with j = 0 (X), 1 (W, i = tile), 2 (dY).  Large tensors may be drawn on the
GPU (``device="cuda"``) purely for speed; their values then differ from a CPU
draw with the same seed, which is harmless because both sides read one copy.
"""
from __future__ import annotations

import math

import numpy as np
import torch

X_STREAM, W_STREAM, DY_STREAM = 0, 1, 2


def stream_seed(seed: int, stream: int, index: int = 0) -> int:
    """A distinct 63-bit seed per (seed, tensor, tile)."""
    return (seed * 1_000_003 + stream * 7_919 + index * 104_729 + 17) & ((1 << 63) - 1)


def _gen(device, s: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """fp32 N(0, std^2) draw rounded to bf16 on ``device``."""
    g = _gen(device, seed)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def ternary_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """Uniform over {-1, 0, +1}, as bf16 (exact)."""
    g = _gen(device, seed)
    t = torch.randint(-1, 2, tuple(shape), generator=g, device=device, dtype=torch.int32)
    return t.to(torch.bfloat16)


def make_x(T: int, K: int, seed: int, device="cpu", kind="normal") -> torch.Tensor:
    s = stream_seed(seed, X_STREAM)
    return ternary_bf16((T, K), s, device) if kind == "ternary" else normal_bf16((T, K), 1.0, s, device)


def make_dy(T: int, M: int, seed: int, device="cpu", kind="normal") -> torch.Tensor:
    s = stream_seed(seed, DY_STREAM)
    return ternary_bf16((T, M), s, device) if kind == "ternary" else normal_bf16((T, M), 1.0, s, device)


def make_w_tile(K: int, Mi: int, i: int, seed: int, device="cpu", kind="normal") -> torch.Tensor:
    """Tile i of W: [K, Mi] with std 1/sqrt(K)."""
    s = stream_seed(seed, W_STREAM, i)
    if kind == "ternary":
        return ternary_bf16((K, Mi), s, device)
    if kind == "identity":
        raise ValueError("identity W is built by make_w_identity")
    return normal_bf16((K, Mi), 1.0 / math.sqrt(K), s, device)


def fill_w_host(w_host: torch.Tensor, K: int, M: int, N: int, tile_major: bool,
                seed: int, device="cpu", kind="normal") -> None:
    """Write W into a host bf16 buffer of K*M elements.

    tile_major: buffer is [N][K][Mi] (each tile contiguous); else [K][M]."""
    Mi = M // N
    flat = w_host.view(-1)
    if tile_major:
        view = flat.view(N, K, Mi)
    else:
        view = flat.view(K, M)
    for i in range(N):
        tile = make_w_tile(K, Mi, i, seed, device, kind)
        if tile_major:
            view[i].copy_(tile)
        else:
            view[:, i * Mi:(i + 1) * Mi].copy_(tile)


def w_logical(w_host: torch.Tensor, K: int, M: int, N: int, tile_major: bool) -> torch.Tensor:
    """The logical [K, M] view/copy of a host W buffer (small sizes only)."""
    Mi = M // N
    flat = w_host.view(-1)
    if not tile_major:
        return flat.view(K, M)
    return flat.view(N, K, Mi).permute(1, 0, 2).reshape(K, M)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (CPU) -> numpy uint16 view of its bit patterns (no copy
    when contiguous)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_indices(nrows: int, ncols: int, n: int, seed: int, tensor_id: int,
                   col_block: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """n uniformly drawn (row, col) pairs plus the edge entries: rows 0 and
    nrows-1 crossed with the first and last column of every column block of
    width ``col_block`` (the whole width if None)."""
    rng = np.random.default_rng(seed + 100 + tensor_id)
    r = rng.integers(0, nrows, n, dtype=np.int64)
    c = rng.integers(0, ncols, n, dtype=np.int64)
    blk = col_block or ncols
    edge_cols = sorted({x for b in range(0, ncols, blk) for x in (b, min(b + blk, ncols) - 1)})
    edge_rows = sorted({0, nrows - 1})
    er = np.array([a for a in edge_rows for _ in edge_cols], np.int64)
    ec = np.array([b for _ in edge_rows for b in edge_cols], np.int64)
    return np.concatenate([r, er]), np.concatenate([c, ec])
