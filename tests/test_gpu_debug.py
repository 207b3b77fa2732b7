"""The debug library (libmattn_debug.so: every source compiled with
MATTN_DEBUG=1) on the GPU.

Its kernels check, before each use, every coordinate handed to a TMA or
bulk copy, every work item and key-tile list entry, every explicit-order
value and every decode ring slot; a failed check records MATTN_ERR_BOUNDS
and the site in the device error word, skips the access, and the CTA
returns.  Two kinds of test:

- clean runs: small cases of every kernel and schedule (paired, split,
  single pipeline, persistent, the reorder pre-pass, grouped-query heads,
  decode, block selection, received attention, the no-allocation entry
  point) pass every check (status MATTN_OK) and give the product library's
  results bit for bit -- the checks change no arithmetic;
- planted defects, each caught by its check before it addresses memory:
  an explicit order holding a token past N (a caller input the product
  library does not check), and, through the debug library's test hook, a
  work item naming a head row past the last (paired and persistent
  schedules), a persistent item whose key tiles run past the sequence, and
  a column-major grid the kernel is told has half its rows (tile
  coordinates outside the TMA view).  Each reports MATTN_ERR_BOUNDS with
  the expected site bit, and the device stays usable: a clean call
  afterwards passes.
"""

import ctypes
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from workloads import (MaskSpec, bernoulli_causal_blocks, block2x2_order, column_major_order,  # noqa: E402
                       make_qkv, random_order)

pytestmark = pytest.mark.gpu

mattn = pytest.importorskip("block_sparse_attention_masked_gb300")

from test_gpu_parity import check  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not (os.path.exists(mattn.LIB_PATH) and os.path.exists(mattn.DEBUG_LIB_PATH)):
        from block_sparse_attention_masked_gb300 import build

        build.build()
    mattn.use_debug_library(True)
    assert mattn.lib().mattn_debug_checks() == 1
    mattn.use_debug_library(False)
    assert mattn.lib().mattn_debug_checks() == 0
    yield
    mattn.use_debug_library(False)


def _on(debug, fn):
    """fn() with every call routed to the debug (or product) library; the
    device error word of that library read and cleared afterwards."""
    mattn.use_debug_library(debug)
    try:
        out = fn()
        torch.cuda.synchronize()
        rc, word = mattn.device_status()
    finally:
        mattn.use_debug_library(False)
    return out, rc, word


def _same_both(fn, tag):
    """The debug library passes every check and matches the product library bit for bit."""
    ref, rc0, w0 = _on(False, fn)
    got, rc1, w1 = _on(True, fn)
    assert rc0 == 0, f"{tag}: product library error word {w0:#x}"
    assert rc1 == 0, f"{tag}: debug library error word {w1:#x}"
    for a, b in zip(ref, got):
        if a is None:
            assert b is None
            continue
        assert torch.equal(a, b), f"{tag}: debug library result differs"


def _qkv(B, H, N, d, seed, dtype="bf16"):
    return make_qkv(B, H, N, d, dtype, 1.0, seed, device="cuda")


def _fwd(q, k, v, spec, schedule=None):
    B, H, N, d = q.shape
    return lambda: mattn.attention(q, k, v, mattn.prepare(spec, H, N, schedule=schedule))


@pytest.mark.parametrize("schedule", ["paired", "persistent"])
@pytest.mark.parametrize("d", [64, 80, 128])
def test_clean_interval_masks(schedule, d):
    n, H = 1000, 4
    q, k, v = _qkv(2, H, n, d, seed=d)
    rng = np.random.default_rng(d)
    for spec in (MaskSpec("sliding", [37, 128, 200, 256], sink=rng.standard_normal(H)),
                 MaskSpec("chunk", [64, 100, 256, 512]),
                 MaskSpec("causal_window", [60, 128, 572, 1000], sink_tokens=4),
                 MaskSpec("full", [0] * H)):
        _same_both(_fwd(q, k, v, spec, schedule), f"{spec.kind} d{d} {schedule}")


@pytest.mark.parametrize("schedule", ["paired", "persistent"])
def test_clean_token_orders(schedule):
    """Column-major and 2x2-block heads read through TMA views (and, for the
    persistent kernel at d <= 96, O stored through them); an explicit order
    and fp32 inputs through the reorder pre-pass."""
    rows = cols = 64
    n, d = rows * cols, 80
    q, k, v = _qkv(1, 4, n, d, seed=3)
    cm = column_major_order(rows, cols)
    spec = MaskSpec("sliding", [128, 90, 64, 300],
                    perm=[None, cm, block2x2_order(rows, cols), block2x2_order(rows, cols, by_columns=True)],
                    perm_grid=[None, (rows, cols), (rows, cols, "block2x2_row"), (rows, cols, "block2x2_col")])
    _same_both(_fwd(q, k, v, spec, schedule), f"grid orders {schedule}")
    spec2 = MaskSpec("chunk", [256, 100, 256, 64], perm=[random_order(n, 3), None, cm, None])
    _same_both(_fwd(q, k, v, spec2, schedule), f"explicit order {schedule}")
    qf, kf, vf = _qkv(1, 2, 1000, 64, seed=6, dtype="f32")
    _same_both(_fwd(qf, kf, vf, MaskSpec("sliding", [32, 100]), schedule), f"fp32 {schedule}")


@pytest.mark.parametrize("schedule", ["split", "paired"])
def test_clean_block_sparse(schedule):
    n, d = 2000, 64
    nb = -(-n // 128)
    q, k, v = _qkv(1, 2, n, d, seed=5)
    spec = MaskSpec("block", [128, 128], block=bernoulli_causal_blocks(2, nb, 11), sink=np.array([0.2, -0.4]))
    _same_both(_fwd(q, k, v, spec, schedule), f"block {schedule}")
    blk = bernoulli_causal_blocks(1, -(-n // 256), 4)
    spec256 = MaskSpec("block", [256, 256], block=np.repeat(blk, 2, axis=0))
    _same_both(_fwd(q, k, v, spec256, schedule), f"block256 {schedule}")


def test_clean_single_pipeline_and_gqa():
    q, k, v = _qkv(1, 2, 700, 256, seed=8)
    _same_both(_fwd(q, k, v, MaskSpec("causal_window", [100, 700], sink=np.array([0.5, -1.0]))), "d256 window")
    nb = -(-700 // 128)
    _same_both(_fwd(q, k, v, MaskSpec("block", [128, 128], block=bernoulli_causal_blocks(2, nb, 2))), "d256 block")
    q2, k2, v2 = _qkv(1, 2, 1000, 128, seed=9)
    spec = MaskSpec("sliding", [100, 40], perm=[random_order(1000, 5), None])
    _same_both(_fwd(q2, k2, v2, spec, "single"), "d128 single, explicit order")
    g = torch.Generator(device="cuda").manual_seed(12)
    qg = torch.randn((1, 8, 1500, 128), generator=g, device="cuda").to(torch.bfloat16)
    kg = torch.randn((1, 2, 1500, 128), generator=g, device="cuda").to(torch.bfloat16)
    vg = torch.randn((1, 2, 1500, 128), generator=g, device="cuda").to(torch.bfloat16)
    gqa = MaskSpec("causal_window", [576] * 8, sink=np.linspace(-1, 1, 8))
    for sched in ("paired", "persistent"):
        _same_both(lambda: mattn.attention(qg, kg, vg, mattn.prepare(gqa, 8, 1500, schedule=sched)), f"gqa {sched}")


def test_clean_decode_selection_received_noalloc():
    g = torch.Generator(device="cuda").manual_seed(3)
    B, H, Hkv, L, d = 2, 16, 4, 3000, 256
    q = torch.randn((B, H, d), generator=g, device="cuda").to(torch.bfloat16)
    kc = torch.randn((B, Hkv, L, d), generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn((B, Hkv, L, d), generator=g, device="cuda").to(torch.bfloat16)
    sl = torch.tensor([3000, 1234], dtype=torch.int32, device="cuda")
    for spec in (MaskSpec("full", [0] * H), MaskSpec("causal_window", [572] * H, sink_tokens=4)):
        _same_both(lambda: mattn.decode(q, kc, vc, mattn.prepare(spec, H, L), seq_lens=sl), f"decode {spec.kind}")
    qs, ks, _ = _qkv(1, 2, 4096, 128, seed=4)
    _same_both(lambda: mattn.rr_select(qs, ks, 8, 128, 0.9, want_scores=True), "block selection")
    qr, kr, vr = _qkv(1, 2, 1000, 64, seed=7)
    for spec in (MaskSpec("sliding", [50, 200]), MaskSpec("causal_window", [128, 300])):
        def recv(spec=spec):
            mask = mattn.prepare(spec, 2, 1000)
            _, lse = mattn.attention(qr, kr, vr, mask)
            return (mattn.received(qr, kr, lse, mask),)
        _same_both(recv, f"received {spec.kind}")

    def noalloc():
        out = torch.empty_like(qr)
        lse = torch.empty((1, 2, 1000), dtype=torch.float32, device="cuda")
        return mattn.attention_noalloc(qr, kr, vr, mattn.prepare(MaskSpec("chunk", [256, 100]), 2, 1000), out, lse)
    _same_both(noalloc, "no-allocation entry point")


def test_clean_against_the_oracle():
    """Debug results stand on their own against the fp64 oracle too."""
    mattn.use_debug_library(True)
    try:
        q, k, v = _qkv(1, 3, 1000, 80, seed=21)
        check(q, k, v, MaskSpec("sliding", [40, 128, 300], sink=np.array([0.1, 0.0, -0.3])), tag="debug sliding",
              schedule="persistent")
        check(q, k, v, MaskSpec("chunk", [96, 128, 256], perm=[random_order(1000, 1), None, None]),
              tag="debug explicit order")
    finally:
        mattn.use_debug_library(False)


# ---------------------------------------------------------------- planted defects

def _plant(what):
    L = mattn.lib()
    L.mattn_internal_debug_corrupt.argtypes = [ctypes.c_int]
    L.mattn_internal_debug_corrupt.restype = ctypes.c_int
    assert L.mattn_internal_debug_corrupt(what) == 0


def _caught(fn, site, tag):
    """fn() on the debug library reports MATTN_ERR_BOUNDS with `site`; a
    clean call afterwards passes its checks and matches the oracle."""
    _, rc, word = _on(True, fn)
    assert rc == mattn.ERR_BOUNDS, f"{tag}: status {rc}, word {word:#x}"
    assert word & mattn.ERRW_BOUNDS and word & mattn.ERRW_SITE[site], f"{tag}: word {word:#x}"
    mattn.use_debug_library(True)
    try:
        q, k, v = _qkv(1, 2, 700, 64, seed=1)
        check(q, k, v, MaskSpec("sliding", [64, 200]), tag=f"clean call after {tag}")
    finally:
        mattn.use_debug_library(False)


@pytest.mark.parametrize("schedule", ["paired", "persistent", "single"])
def test_explicit_order_past_n_is_caught(schedule):
    """An explicit order holding token N + 5 and token -3: the reorder
    pre-pass does not read those rows and the epilogue does not store them."""
    n, d = 1000, 128
    q, k, v = _qkv(1, 2, n, d, seed=2)
    bad = random_order(n, 7).astype(np.int64)
    bad[17] = n + 5
    bad[901] = -3
    spec = MaskSpec("sliding", [64, 64], perm=[bad, None])
    _caught(_fwd(q, k, v, spec, schedule), "order", f"explicit order {schedule}")


def test_explicit_order_past_n_is_caught_by_received_attention():
    n = 1000
    q, k, v = _qkv(1, 2, n, 64, seed=3)
    bad = random_order(n, 8).astype(np.int64)
    bad[0] = n
    mask = mattn.prepare(MaskSpec("chunk", [128, 128], perm=[bad, None]), 2, n)
    lse = torch.zeros((1, 2, n), dtype=torch.float32, device="cuda")
    _caught(lambda: mattn.received(q, k, lse, mask), "order", "received attention")


@pytest.mark.parametrize("schedule", ["paired", "persistent", "split"])
def test_work_item_head_past_the_last_is_caught(schedule):
    n, d = 1000, 64
    q, k, v = _qkv(1, 2, n, d, seed=4)
    if schedule == "split":
        spec = MaskSpec("block", [128, 128], block=bernoulli_causal_blocks(2, -(-n // 128), 3))
    else:
        spec = MaskSpec("sliding", [100, 300])
    mask = mattn.prepare(spec, 2, n, schedule=schedule)

    def run():
        _plant(1)
        return mattn.attention(q, k, v, mask)
    _caught(run, "item", f"item head {schedule}")


def test_persistent_key_tiles_past_the_sequence_are_caught():
    n, d = 3000, 80
    q, k, v = _qkv(1, 2, n, d, seed=5)
    mask = mattn.prepare(MaskSpec("chunk", [256, 512]), 2, n, schedule="persistent")

    def run():
        _plant(2)
        return mattn.attention(q, k, v, mask)
    _caught(run, "key_tile", "persistent key tiles")


@pytest.mark.parametrize("schedule", ["paired", "persistent"])
def test_tile_coordinates_outside_the_view_are_caught(schedule):
    """A 256 x 16 grid walked column by column (read through the 4D TMA
    view): told it has 128 rows, the kernel computes grid columns 16..31
    for the second half of the sequence, outside the view."""
    rows, cols = 256, 16
    n, d = rows * cols, 64
    q, k, v = _qkv(1, 2, n, d, seed=6)
    spec = MaskSpec("sliding", [64, 64], perm=[column_major_order(rows, cols), None],
                    perm_grid=[(rows, cols), None])
    mask = mattn.prepare(spec, 2, n, schedule=schedule)

    def run():
        _plant(3)
        return mattn.attention(q, k, v, mask)
    _caught(run, "load", f"tile coordinates {schedule}")
