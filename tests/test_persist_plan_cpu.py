"""Host-side work plan of the persistent kernel, on the CPU (no GPU): the
paired items of an interval mask, the long ones split into one item per
query tile, assigned to CTAs longest first.

Checked against the host tile plan (itself checked bit for bit against the
oracle's dense enumeration in test_abi_cpu.py):
- every query tile of every (batch, head) is taken by exactly one item, as
  a sub-tile of a paired item or as a split item;
- each item's key-tile list is the union of its query tiles' key tiles (a
  split item: exactly its query tile's), and each sub-tile's first / last
  entries are the ones it multiplies (a split item: entry j to sub-tile
  j % 2);
- items above a CTA's fair share are split, the others are not (the rule),
  none / all are split under the test hook's modes;
- the CTA ranges partition the items, and no CTA's load exceeds the fair
  share by more than one item's load (the longest-first bound).
"""

import ctypes
import os

import numpy as np
import pytest

from workloads import MaskSpec, WORKLOADS, make_mask

mattn = pytest.importorskip("block_sparse_attention_masked_gb300")

I4 = 6          # int4 per item descriptor
OVERHEAD = 4    # tile products of an item's set-up and output in its load


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(mattn.LIB_PATH):
        from block_sparse_attention_masked_gb300 import build

        build.build()
    lib = mattn.lib()
    lib.mattn_internal_persist_plan.argtypes = [
        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t,
        ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_int)]
    lib.mattn_internal_set_persist_split.argtypes = [ctypes.c_int]
    yield lib
    lib.mattn_internal_set_persist_split(0)


def _plan(L, spec, B, H, N, d, grid, mode):
    assert L.mattn_internal_set_persist_split(mode) == 0
    mask = mattn.PreparedMask(spec, H, N, host_side=True)
    cap = 4 * B * H * ((N + 127) // 128) + 8
    items = np.zeros(cap * I4 * 4, dtype=np.int32)
    off = np.zeros(grid + 1, dtype=np.int32)
    n, g = ctypes.c_size_t(), ctypes.c_int()
    rc = L.mattn_internal_persist_plan(ctypes.byref(mask.desc), B, H, N, d, grid, items.ctypes.data, cap,
                                       off.ctypes.data, grid + 1, ctypes.byref(n), ctypes.byref(g))
    assert rc == mattn.OK, L.mattn_last_error()
    return items[: n.value * I4 * 4].reshape(n.value, I4, 4), off[: g.value + 1]


def _kt(item, j):
    n, lo, na = item[1][0], item[1][1], item[1][2]
    assert 0 <= j < n
    return j if j < na else lo + j - na


def _load(item):
    if (item[4][2] >> 16) & 1:
        return item[1][0] + OVERHEAD
    f0, l0, f1, l1 = item[5]
    return (l0 - f0 + 1 if f0 >= 0 else 0) + (l1 - f1 + 1 if f1 >= 0 else 0) + OVERHEAD


def _check_plan(items, off, spec, B, H, N, mode, grid):
    nt = (N + 127) // 128
    tiles = mattn.plan_tiles(spec, H, N)  # rows (h, qt, kt, class)
    want = {}
    for h, qt, kt, _ in tiles:
        want.setdefault((int(h), int(qt)), set()).add(int(kt))
    seen = {}
    split_count = 0
    for i, it in enumerate(items):
        bh, h, b, qt0 = (int(x) for x in it[0])
        assert bh == b * H + h and 0 <= h < H and 0 <= b < B
        split = bool((it[4][2] >> 16) & 1)
        n = int(it[1][0])
        lst = [_kt(it, j) for j in range(n)]
        assert lst == sorted(set(lst)), f"item {i}: list not ascending"
        if split:
            split_count += 1
            assert want[(h, qt0)] == set(lst), f"item {i}: split list"
            f0, l0, f1, l1 = (int(x) for x in it[5])
            assert (f0, l0) == (0, (n - 1) & ~1)
            assert (f1, l1) == ((1, n - 1 if (n - 1) % 2 else n - 2) if n >= 2 else (-1, -1))
            tqs = [qt0]
        else:
            tqs = [q for q in (qt0, qt0 + 1) if q < nt]
            union = set()
            for s, q in enumerate((qt0, qt0 + 1)):
                f, l = int(it[5][2 * s]), int(it[5][2 * s + 1])
                mine = want.get((h, q), set()) if q < nt else set()
                if not mine:
                    assert f == -1 and l == -1
                    continue
                used = [j for j in range(n) if lst[j] in mine]
                assert (f, l) == (used[0], used[-1]), f"item {i} sub-tile {s}: first / last"
                union |= mine
            assert union == set(lst), f"item {i}: pair list"
        for q in tqs:
            assert (b, h, q) not in seen, f"query tile {(b, h, q)} taken twice"
            seen[(b, h, q)] = i
    assert len(seen) == B * H * nt, "a query tile is missing"
    # the split rule, and the test hook's modes
    if mode < 0:
        assert split_count == 0
    # CTA ranges partition the items; longest-first balance
    g = len(off) - 1
    assert off[0] == 0 and off[-1] == len(items) and np.all(np.diff(off) >= 0)
    loads = [sum(_load(items[k]) for k in range(off[c], off[c + 1])) for c in range(g)]
    total = sum(_load(it) for it in items)
    assert max(loads) <= total / g + max(_load(it) for it in items)
    return split_count


def test_causal_windows_split_the_long_items(L):
    """The head-wise causal-window layer (windows 512..4096): the pairs of
    the 4096-key heads whose load passes the fair share become split
    items; under the rule no remaining paired item is above it."""
    wl = WORKLOADS["causal4096"]
    spec = make_mask(wl, "causal_window_sink", seed=0)
    items, off = _plan(L, spec, wl.B, wl.H, wl.N, wl.d, 152, 0)
    n_split = _check_plan(items, off, spec, wl.B, wl.H, wl.N, 0, 152)
    assert n_split > 0
    pairs = [it for it in items if not ((it[4][2] >> 16) & 1)]
    loads = [_load(it) for it in pairs]
    # the fair share the rule used: the total load of the unsplit plan over the grid
    plain, _ = _plan(L, spec, wl.B, wl.H, wl.N, wl.d, 152, -1)
    fair = sum(_load(it) for it in plain) // min(152, len(plain))
    assert max(loads) <= fair
    big = [it for it in plain if _load(it) > fair]
    assert n_split == sum(sum(1 for s in (0, 1) if it[5][2 * s] >= 0) for it in big)


@pytest.mark.parametrize("mode", [-1, 0, 1])
@pytest.mark.parametrize("case", ["sliding_ragged", "chunk", "causal_sink_tokens", "full_small", "vit16384"])
def test_plans_cover_every_query_tile(L, mode, case):
    """Coverage, lists and balance on ragged and per-head parameters, with no
    item split, the rule, and every item split."""
    if case == "vit16384":
        wl = WORKLOADS["vit16384"]
        B, H, N, d = wl.B, wl.H, wl.N, wl.d
        spec = make_mask(wl, "sliding256_rowcol", seed=0)
    else:
        B, H, N, d = 2, 5, 1000, 64
        spec = {
            "sliding_ragged": MaskSpec("sliding", [1, 37, 128, 200, 256]),
            "chunk": MaskSpec("chunk", [64, 100, 128, 256, 512]),
            "causal_sink_tokens": MaskSpec("causal_window", [60, 128, 300, 572, 1000], sink_tokens=4),
            "full_small": MaskSpec("full", [0] * H),
        }[case]
    for grid in (152, 7):
        items, off = _plan(L, spec, B, H, N, d, grid, mode)
        n_split = _check_plan(items, off, spec, B, H, N, mode, grid)
        if mode > 0:
            assert n_split > 0
