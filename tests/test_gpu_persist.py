"""GPU parity of the persistent schedule (MATTN_FLAG_SCHEDULE_PERSISTENT) for
the interval masks: one CTA per SM walking paired work items back to back.

Each case is checked twice:
- against the fp64 oracle with the tolerances of the other parity tests
  (max abs 2e-2, rel L2 5e-3 on O; LSE 1e-3, plus the bf16-rounding bound
  for fp32 inputs);
- against the one-item-per-CTA paired kernel, bit for bit: a work item's
  arithmetic (products, softmax, accumulation order, epilogue) is the same
  in both kernels, only the schedule differs.

Small problems have fewer work items than SMs, so most cases also run with
the grid capped at a few CTAs (a test hook), which gives every CTA many
items: Q slots wrap several times, the K/V rings run across item
boundaries, and O accumulators are reused item after item.
"""

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from workloads import (MaskSpec, WORKLOADS, block2x2_order, column_major_order,  # noqa: E402
                       make_mask, make_qkv, make_workload_inputs, random_order)

pytestmark = pytest.mark.gpu

mattn = pytest.importorskip("block_sparse_attention_masked_gb300")

from test_gpu_parity import check  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os

    if not os.path.exists(mattn.LIB_PATH):
        from block_sparse_attention_masked_gb300 import build

        build.build()
    mattn.lib()


@pytest.fixture
def grid_cap():
    """Sets the persistent grid cap for one test and restores one CTA per SM."""
    L = mattn.lib()
    L.mattn_internal_set_persist_grid.argtypes = [ctypes.c_int]

    def set_cap(n):
        assert L.mattn_internal_set_persist_grid(n) == 0

    yield set_cap
    L.mattn_internal_set_persist_grid(0)


SCHEDULES = ["persistent"]


@pytest.fixture
def split_mode():
    """Sets which persistent items are split (test hook: -1 none, 0 the load
    rule, 1 every item whose query tiles see two or more key tiles) for one
    test and restores the rule."""
    L = mattn.lib()
    L.mattn_internal_set_persist_split.argtypes = [ctypes.c_int]

    def set_mode(m):
        assert L.mattn_internal_set_persist_split(m) == 0

    yield set_mode
    L.mattn_internal_set_persist_split(0)


def _same_as_paired(q, k, v, spec, tag, schedule="persistent", exact=True):
    """Without split items the persistent kernel does a paired item's
    arithmetic exactly: equal bits.  A split item deals a query tile's key
    tiles to the two sub-tiles and merges their partial sums at the end, so
    its sums are added in another order: O within one bf16 (or 2^-20 fp32)
    rounding step of the paired result, LSE within 1e-5."""
    B, H, N, d = q.shape
    o_p, l_p = mattn.attention(q, k, v, mattn.prepare(spec, H, N, schedule=schedule))
    o_r, l_r = mattn.attention(q, k, v, mattn.prepare(spec, H, N, schedule="paired"))
    torch.cuda.synchronize()
    rc, word = mattn.device_status()
    assert rc == 0, f"{tag}: device error word {word:#x}"
    if exact:
        assert torch.equal(o_p, o_r), f"{tag}: O differs from the paired kernel"
        assert torch.equal(l_p, l_r), f"{tag}: LSE differs from the paired kernel"
        return
    step = 2.0 ** -7 if o_p.dtype == torch.bfloat16 else 2.0 ** -20
    a, r = o_p.float(), o_r.float()
    assert ((a - r).abs() <= step * r.abs() + 1e-6).all(), f"{tag}: O differs from the paired kernel"
    fin = torch.isfinite(l_r)
    assert torch.equal(fin, torch.isfinite(l_p)), f"{tag}: LSE -inf pattern differs"
    assert (l_p[fin] - l_r[fin]).abs().max().item() <= 1e-5, f"{tag}: LSE differs from the paired kernel"


def _specs(H, n):
    rng = np.random.default_rng(n + H)
    return [
        MaskSpec("full", [0] * H),
        MaskSpec("chunk", [int(x) for x in rng.choice([64, 100, 128, 256, 512], H)]),
        MaskSpec("sliding", [int(x) for x in rng.choice([1, 37, 128, 200, 256], H)], sink=rng.standard_normal(H)),
        MaskSpec("causal_window", [int(x) for x in rng.choice([1, 64, 300, 512, 1024], H)], sink=rng.standard_normal(H)),
        MaskSpec("causal_window", [int(x) for x in rng.choice([60, 128, 572], H)], sink_tokens=4),
    ]


@pytest.mark.parametrize("sched", SCHEDULES)
@pytest.mark.parametrize("split", [-1, 1])
@pytest.mark.parametrize("cap", [0, 3])
@pytest.mark.parametrize("d", [32, 64, 80, 96, 128])
@pytest.mark.parametrize("n", [256, 1000, 2200])
def test_interval_kinds(d, n, cap, split, sched, grid_cap, split_mode):
    """Every interval kind with per-head parameters, ragged N (a partial last
    query tile, and at 1000 / 2200 an odd tile count whose last pair has one
    empty sub-tile), with and without a capped grid, with no item split and
    with every item split (each query tile's key tiles dealt to the two
    sub-tiles, merged at its end)."""
    grid_cap(cap)
    split_mode(split)
    H = 3
    q, k, v = make_qkv(2, H, n, d, "bf16", 1.0, seed=d * 7 + n, device="cuda")
    for spec in _specs(H, n):
        tag = f"{spec.kind} d{d} n{n} cap{cap} split{split} {sched}"
        check(q, k, v, spec, tag=tag, schedule=sched)
        _same_as_paired(q, k, v, spec, tag, sched, exact=split < 0)


@pytest.mark.parametrize("sched", SCHEDULES)
@pytest.mark.parametrize("split", [-1, 1])
@pytest.mark.parametrize("cap", [0, 2])
def test_token_orders(cap, split, sched, grid_cap, split_mode):
    """Column-major heads (strided TMA views), the two 2x2-block orders (5D
    views), an explicit order and fp32 inputs (both through the reorder
    pre-pass, the kernel then launched as its programmatic dependent)."""
    grid_cap(cap)
    split_mode(split)
    ex = split < 0
    rows, cols = 64, 64
    n, d = rows * cols, 80
    q, k, v = make_qkv(1, 4, n, d, "bf16", 0.5, seed=5, device="cuda")
    cm = column_major_order(rows, cols)
    spec = MaskSpec("sliding", [128, 128, 90, 300],
                    perm=[None, cm, block2x2_order(rows, cols), block2x2_order(rows, cols, by_columns=True)],
                    perm_grid=[None, (rows, cols), (rows, cols, "block2x2_row"), (rows, cols, "block2x2_col")])
    check(q, k, v, spec, tag="grid orders", schedule=sched)
    _same_as_paired(q, k, v, spec, "grid orders", sched, exact=ex)
    rng = np.random.default_rng(9)
    spec2 = MaskSpec("chunk", [256, 100, 256, 64], perm=[random_order(n, 3), None, cm, None],
                     sink=rng.standard_normal(4))
    check(q, k, v, spec2, tag="explicit order", schedule=sched)
    _same_as_paired(q, k, v, spec2, "explicit order", sched, exact=ex)
    qf, kf, vf = make_qkv(1, 2, 1000, 64, "f32", 1.0, seed=6, device="cuda")
    spec3 = MaskSpec("sliding", [32, 100])
    check(qf, kf, vf, spec3, tag="fp32", schedule=sched)
    _same_as_paired(qf, kf, vf, spec3, "fp32", sched, exact=ex)


@pytest.mark.parametrize("sched", SCHEDULES)
@pytest.mark.parametrize("split", [-1, 1])
@pytest.mark.parametrize("cap", [0, 5])
def test_grouped_query_heads(cap, split, sched, grid_cap, split_mode):
    """Grouped-query attention: 8 query heads sharing 2 K/V heads."""
    grid_cap(cap)
    split_mode(split)
    from oracle import dense

    B, H, Hkv, n, d = 1, 8, 2, 3000, 128
    g = torch.Generator(device="cuda").manual_seed(11)
    q = torch.randn((B, H, n, d), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((B, Hkv, n, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, Hkv, n, d), generator=g, device="cuda").to(torch.bfloat16)
    spec = MaskSpec("causal_window", [576] * H, sink=np.linspace(-1, 1, H))
    o, lse = mattn.attention(q, k, v, mattn.prepare(spec, H, n, schedule=sched))
    torch.cuda.synchronize()
    assert mattn.device_status()[0] == 0
    _same_as_paired(q, k, v, spec, f"gqa {sched}", sched, exact=split < 0)
    rows = np.unique(np.r_[0, 127, 128, 575, 576, n - 1, np.random.default_rng(0).choice(n, 40, replace=False)])
    f = lambda t: t.float().cpu().numpy()  # noqa: E731
    ref_o, ref_l = dense.attention(f(q), f(k), f(v), spec, rows=rows)
    got = f(o)[0][:, rows]
    assert np.abs(got - ref_o).max() <= 2e-2
    assert np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o) <= 5e-3
    assert np.abs(f(lse)[0][:, rows] - ref_l).max() <= 1e-3


@pytest.mark.parametrize("sched", SCHEDULES)
@pytest.mark.parametrize("mask", ["sliding256_rowcol", "chunk512", "sliding256_blocks"])
def test_vit16384_full_size(mask, sched):
    """The 16,384-token ViT layer (B1 H16 d80) at full size, in the launch
    configuration the benchmark times: sampled heads (raster, column-major
    and 2x2-block heads) against the oracle on sampled rows, all heads equal
    to the paired kernel bit for bit."""
    wl = WORKLOADS["vit16384"]
    q, k, v = make_workload_inputs(wl, seed=0, device="cuda")
    spec = make_mask(wl, mask, seed=0)
    rng = np.random.default_rng(1)
    rows = np.unique(np.r_[0, 255, 256, 8191, wl.N - 1, rng.choice(wl.N, 48, replace=False)])
    check(q, k, v, spec, rows=rows, heads=[(0, 0), (0, 5), (0, 8), (0, 15)], tag=mask, schedule=sched)
    _same_as_paired(q, k, v, spec, mask, sched, exact=False)


@pytest.mark.parametrize("sched", SCHEDULES)
def test_causal_windows_with_sink_full_size(sched):
    """The head-wise causal-window LM layer (B1 H16 L4096 d128, windows
    512..4096, sink logits) at full size."""
    wl = WORKLOADS["causal4096"]
    q, k, v = make_workload_inputs(wl, seed=0, device="cuda")
    spec = make_mask(wl, "causal_window_sink", seed=0)
    rows = np.unique(np.r_[0, 511, 512, 2047, 2048, 4095, np.random.default_rng(2).choice(4096, 64, replace=False)])
    check(q, k, v, spec, rows=rows, tag="causal4096", schedule=sched)
    _same_as_paired(q, k, v, spec, "causal4096", sched, exact=False)


@pytest.mark.parametrize("sched", SCHEDULES)
def test_rejects_block_sparse(sched):
    from workloads import bernoulli_causal_blocks

    spec = MaskSpec("block", [128, 128], block=bernoulli_causal_blocks(2, 4, 0))
    q, k, v = make_qkv(1, 2, 512, 64, "bf16", 1.0, seed=0, device="cuda")
    with pytest.raises(RuntimeError, match="persistent"):
        mattn.attention(q, k, v, mattn.prepare(spec, 2, 512, schedule=sched))
