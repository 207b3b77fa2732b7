"""Seeded synthetic inputs for the masked attention forward.

This module is the only thing the oracle side and the CUDA side have in
common: it draws the inputs (Q, K, V, window assignments, sink logits,
block-selection matrices, token orders) and describes the workloads.  It
holds none of the method's arithmetic: no score, mask predicate, softmax,
tile enumeration or pair count lives here.

The workloads stand in for the pages' data, which are not available here:
ViT layers on COCO / Cambrian images at 448^2..1792^2 (SHS slides, the
cost slide: 1,024 / 4,096 / 16,384 tokens; Qwen2.5-VL-style 14-px patches),
a 1B LM at 4096 tokens with head-wise causal windows (Asymmetric Attention
Heads, Table 2) and 128K-token prefill with a ~50% block-sparse pattern
(RRAttention, section 4, HELMET / Video-MME contexts).  Values are i.i.d.
normal, drawn with ``torch.Generator`` seeded per tensor in the order
q, k, v; mask-side randomness (window shuffle, sinks, Bernoulli blocks)
comes from ``numpy.random.default_rng(seed)``.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np


@dataclasses.dataclass
class MaskSpec:
    """Mask description consumed by both the oracle and the library binding.

    kind:       "full" | "chunk" | "sliding" | "causal_window" | "block"
    head_param: per head, C (chunk), w (half-width), W (causal window) or the
                block size B (block); ignored for "full".
    perm:       per head, None (identity) or an int array with
                perm[p] = caller token index at sequence position p.
    perm_grid:  per head, None, (rows, cols) when perm is the column-major
                order of a rows x cols raster grid, or (rows, cols, kind) with
                kind "column_major", "block2x2_row" or "block2x2_col" (a plain
                description of the same perm, so that a caller can name the
                order instead of passing the array).
    block:      bool [H, Nb, Nb] block-selection matrices (kind "block").
    sink:       float [H] sink logits, or None.
    sink_tokens: kind "causal_window": the first sink_tokens positions stay
                visible to every query at or after them (0 = none).
    """

    kind: str
    head_param: List[int]
    perm: Optional[List[Optional[np.ndarray]]] = None
    perm_grid: Optional[List[Optional[tuple]]] = None
    block: Optional[np.ndarray] = None
    sink: Optional[np.ndarray] = None
    name: str = ""
    sink_tokens: int = 0


def column_major_order(rows: int, cols: int) -> np.ndarray:
    """perm[p] for the column-major walk of a rows x cols raster-numbered grid.

    Raster token t = r * cols + c; walking columns first puts position
    p = c * rows + r on token r * cols + c.
    """
    c, r = np.divmod(np.arange(rows * cols, dtype=np.int64), rows)
    return (r * cols + c).astype(np.int64)


def block2x2_order(rows: int, cols: int, by_columns: bool = False) -> np.ndarray:
    """perm[p] for the walk over the 2x2 patch blocks of a rows x cols
    raster-numbered grid (SHS slides, Factor 2: Qwen2.5-VL merges 2x2 patches
    into one block; order (c) takes the blocks left to right then top to
    bottom, order (d) top to bottom then left to right).  Inside a block the
    four patches go in raster order (the figure is not in the text; read).
    Position p = 4 * block + 2 * dr + dc."""
    if rows % 2 or cols % 2:
        raise ValueError("2x2-block orders need an even grid")
    p = np.arange(rows * cols, dtype=np.int64)
    blk, dr, dc = p // 4, (p // 2) % 2, p % 2
    if by_columns:
        C, R = np.divmod(blk, rows // 2)
    else:
        R, C = np.divmod(blk, cols // 2)
    return ((2 * R + dr) * cols + 2 * C + dc).astype(np.int64)


def chunk2d_order(rows: int, cols: int, win: int) -> np.ndarray:
    """perm[p] for the chunk-window walk of a rows x cols raster-numbered
    grid (SHS slides, Factor 2 background, order (b): Qwen2.5-VL's chunk
    windows, every block of window 0 walked before window 1).  The grid is
    cut into win x win-patch windows, taken left to right then top to
    bottom; inside a window its 2x2 patch blocks go left to right then top to
    bottom, and inside a block the four patches in raster order (the figure
    is not in the text: the walk inside a window is our reading, the window
    by window part is the slide's).  win must be even and divide rows and
    cols."""
    if win % 2 or rows % win or cols % win:
        raise ValueError("win must be even and divide the grid")
    out = []
    for wr in range(rows // win):
        for wc in range(cols // win):
            for br in range(win // 2):
                for bc in range(win // 2):
                    for dr in range(2):
                        for dc in range(2):
                            r = wr * win + 2 * br + dr
                            c = wc * win + 2 * bc + dc
                            out.append(r * cols + c)
    return np.array(out, dtype=np.int64)


def random_order(n: int, seed: int) -> np.ndarray:
    return np.random.default_rng(seed).permutation(n).astype(np.int64)


def bernoulli_causal_blocks(n_heads: int, nb: int, seed: int, keep_prob: float = 0.5,
                            keep_diagonal: bool = True, keep_first_column: bool = True) -> np.ndarray:
    """bool [H, nb, nb]: lower-triangle blocks kept with probability keep_prob.

    Per head h an independent generator ``default_rng([seed, h])``; the
    diagonal and the first block column are always kept when asked (the
    "sink & recent blocks" kept by the block-sparse baselines of RRAttention,
    Table 5).  Upper-triangle entries are left False.
    """
    out = np.zeros((n_heads, nb, nb), dtype=bool)
    tri = np.tril(np.ones((nb, nb), dtype=bool))
    for h in range(n_heads):
        rng = np.random.default_rng([seed, h])
        out[h] = (rng.random((nb, nb)) < keep_prob) & tri
        if keep_diagonal:
            out[h][np.arange(nb), np.arange(nb)] = True
        if keep_first_column:
            out[h][:, 0] = True
    return out


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str          # "f32" | "bf16"
    value_scale: float
    grid: Optional[tuple]
    masks: Sequence[str]
    description: str
    kv_heads: Optional[int] = None  # grouped-query attention: K / V heads (None = H)


WORKLOADS = {
    "vit256_tiny": Workload(
        "vit256_tiny", 1, 2, 256, 64, "f32", 1.0, (16, 16),
        ("full", "chunk64", "sliding32"),
        "16x16 patch grid raster order, B1 H2 N256 d64, fp32 N(0,1); no sink"),
    "vit4096": Workload(
        "vit4096", 1, 16, 4096, 80, "bf16", 0.5, (64, 64),
        ("full", "chunk256", "sliding128"),
        "896^2 ViT layer: 64x64 grid raster order, B1 H16 N4096 d80, bf16 0.5*N(0,1)"),
    "vit16384": Workload(
        "vit16384", 1, 16, 16384, 80, "bf16", 0.5, (128, 128),
        ("sliding256_rowcol", "full", "chunk512", "sliding256_blocks"),
        "1792^2 ViT layer: 128x128 grid, B1 H16 N16384 d80, bf16 0.5*N(0,1); "
        "sliding window 256 on raster order for heads 0-7 and column-major order for heads 8-15"),
    "causal4096": Workload(
        "causal4096", 1, 16, 4096, 128, "bf16", 1.0, None,
        ("causal_window_sink",),
        "LM layer L4096 B1 H16 d128 bf16 N(0,1); per-head causal window from "
        "{512,1024,2048,4096} (4 heads each, seeded shuffle); sink ~ N(0,1)"),
    "bsparse128k": Workload(
        "bsparse128k", 1, 32, 131072, 128, "bf16", 1.0, None,
        ("block128",),
        "128K prefill B1 H32 d128 bf16 N(0,1); block 128 (Nb 1024): diagonal and "
        "first column kept, other causal blocks Bernoulli(0.5), per head"),
    "gqa32k": Workload(
        "gqa32k", 1, 32, 32768, 128, "bf16", 1.0, None,
        ("swa572_sinktok4", "swa576_sink"),
        "LM prefill with grouped-query attention (Qwen3-4B layout: 32 query heads "
        "sharing 8 K/V heads, d128), B1 N32768 bf16 N(0,1); causal window 572 plus "
        "the first 4 tokens (StreamingLLM sink tokens), or window 576 with a "
        "learned sink logit ~ N(0,1) per head", kv_heads=8),
    "prefill_d256": Workload(
        "prefill_d256", 1, 16, 16384, 256, "bf16", 1.0, None,
        ("causal", "swa576_sink"),
        "LM prefill of a 16K-token prompt in the speed-test layout (16 query heads "
        "sharing 4 K/V heads of dimension 256), B1 bf16 N(0,1); causal, or causal "
        "window 576 with a learned sink logit ~ N(0,1) per head", kv_heads=4),
    "decode128k": Workload(
        "decode128k", 1, 16, 131072, 256, "bf16", 1.0, None,
        ("full", "swa576_sink", "swa572_sinktok4"),
        "decode step after a 128K-token prompt (the speed-test layout: 16 query heads "
        "sharing 4 K/V heads, d256), B1, one new query per sequence against a full "
        "bf16 N(0,1) cache of 131072 tokens; full, window 576 with a learned sink "
        "logit, or window 572 plus 4 sink tokens", kv_heads=4),
}


def make_mask(wl: Workload, mask: str, seed: int = 0, n: Optional[int] = None,
              heads: Optional[int] = None) -> MaskSpec:
    """The MaskSpec of workload ``wl``'s mask named ``mask``.

    ``n`` / ``heads`` shrink the workload (same recipe at a smaller size);
    grid-based orders then need ``n`` to be a square of a power of two.
    """
    n = wl.N if n is None else n
    nh = wl.H if heads is None else heads
    if mask == "full":
        return MaskSpec("full", [0] * nh, name=mask)
    if mask.startswith("chunk"):
        return MaskSpec("chunk", [int(mask[5:])] * nh, name=mask)
    if mask.startswith("sliding") and mask.endswith("_blocks"):
        # SWA-1D over the 2x2 patch blocks: row order (c) on the first half of
        # the heads, column order (d) on the second (SHS slides, Factor 2)
        w = int(mask[len("sliding"):-len("_blocks")])
        side = int(round(n ** 0.5))
        if side * side != n:
            raise ValueError("2x2-block orders need a square grid here")
        perm, grid = [None] * nh, [None] * nh
        for h in range(nh):
            by_cols = h >= nh // 2
            perm[h] = block2x2_order(side, side, by_cols)
            grid[h] = (side, side, "block2x2_col" if by_cols else "block2x2_row")
        return MaskSpec("sliding", [w] * nh, perm=perm, perm_grid=grid, name=mask)
    if mask.startswith("sliding") and mask.endswith("_rowcol"):
        w = int(mask[len("sliding"):-len("_rowcol")])
        side = int(round(n ** 0.5))
        if side * side != n:
            raise ValueError("row/column orders need a square grid")
        col = column_major_order(side, side)
        perm = [None] * nh
        grid = [None] * nh
        for h in range(nh // 2, nh):
            perm[h] = col
            grid[h] = (side, side)
        return MaskSpec("sliding", [w] * nh, perm=perm, perm_grid=grid, name=mask)
    if mask.startswith("sliding"):
        return MaskSpec("sliding", [int(mask[7:])] * nh, name=mask)
    if mask == "causal_window_sink":
        rng = np.random.default_rng(seed)
        sizes = np.array([512, 1024, 2048, 4096] * ((nh + 3) // 4))[:nh]
        windows = rng.permutation(sizes)
        sink = rng.standard_normal(nh)
        return MaskSpec("causal_window", [int(x) for x in windows], sink=sink, name=mask)
    if mask == "causal":
        return MaskSpec("causal_window", [n] * nh, name=mask)
    if mask.startswith("swa") and "_sinktok" in mask:
        w, s = mask[3:].split("_sinktok")
        return MaskSpec("causal_window", [int(w)] * nh, sink_tokens=int(s), name=mask)
    if mask.startswith("swa") and mask.endswith("_sink"):
        rng = np.random.default_rng(seed)
        return MaskSpec("causal_window", [int(mask[3:-5])] * nh, sink=rng.standard_normal(nh), name=mask)
    if mask.startswith("block"):
        bs = int(mask[5:])
        nb = (n + bs - 1) // bs
        blk = bernoulli_causal_blocks(nh, nb, seed)
        return MaskSpec("block", [bs] * nh, block=blk, name=mask)
    raise ValueError(f"unknown mask {mask!r}")


def make_qkv(B: int, H: int, N: int, d: int, dtype: str = "bf16", value_scale: float = 1.0,
             seed: int = 0, device: str = "cpu", kv_heads: Optional[int] = None):
    """Seeded q [B, H, N, d] and k, v [B, kv_heads, N, d] tensors (torch;
    kv_heads defaults to H), drawn in the order q, k, v.

    fp32 draws from N(0,1), multiplied by ``value_scale``, then cast to the
    dtype.  On a CUDA device the CUDA generator is used (different stream of
    numbers than on the CPU, same recipe); tests hand the very same tensors
    to both sides.
    """
    import torch

    g = torch.Generator(device=device).manual_seed(seed)
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    out = []
    for i in range(3):
        nh = H if (i == 0 or kv_heads is None) else kv_heads
        x = torch.randn((B, nh, N, d), generator=g, device=device, dtype=torch.float32)
        if value_scale != 1.0:
            x.mul_(value_scale)
        out.append(x.to(tdt))
    return tuple(out)


def make_decode_inputs(wl: Workload, seed: int = 0, device: str = "cpu"):
    """Seeded decode inputs (torch): q [B, H, d] (the new tokens' queries),
    then the caches k, v [B, kv_heads, N, d], drawn in that order."""
    import torch

    g = torch.Generator(device=device).manual_seed(seed)
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32}[wl.dtype]
    kv = wl.kv_heads or wl.H
    q = torch.randn((wl.B, wl.H, wl.d), generator=g, device=device) * wl.value_scale
    k = torch.randn((wl.B, kv, wl.N, wl.d), generator=g, device=device) * wl.value_scale
    v = torch.randn((wl.B, kv, wl.N, wl.d), generator=g, device=device) * wl.value_scale
    return q.to(tdt), k.to(tdt), v.to(tdt)


def make_workload_inputs(wl: Workload, seed: int = 0, device: str = "cpu",
                         n: Optional[int] = None, heads: Optional[int] = None):
    n = wl.N if n is None else n
    nh = wl.H if heads is None else heads
    kv = None if wl.kv_heads is None else max(1, wl.kv_heads * nh // wl.H)
    return make_qkv(wl.B, nh, n, wl.d, wl.dtype, wl.value_scale, seed, device, kv_heads=kv)
