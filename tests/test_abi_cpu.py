"""CPU checks of the C ABI: the library loads, exports every declared symbol,
validates arguments, and its host planner / pair counter agree bit-exactly
with the oracle's dense enumeration.  No compute call touches a GPU here."""

import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT
from oracle import dense
from workloads import MaskSpec, WORKLOADS, bernoulli_causal_blocks, column_major_order, make_mask

mattn = pytest.importorskip("block_sparse_attention_masked_gb300")


@pytest.fixture(scope="session")
def L():
    if not os.path.exists(mattn.LIB_PATH):
        from block_sparse_attention_masked_gb300 import build

        build.build()
    return mattn.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "mattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mattn_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert "mattn_fwd" in names and "mattn_count_pairs" in names
    for name in names:
        assert hasattr(L, name), name
    assert set(mattn.EXPORTS) == set(names)


def test_status_strings_and_version(L):
    assert L.mattn_status_string(0) == b"MATTN_OK"
    assert L.mattn_status_string(-4) == b"MATTN_ERR_TIMEOUT"
    assert L.mattn_version() >= 100


def test_struct_layout_matches_header():
    # x86-64 / aarch64 LP64: 4+4 + 8 + 8 + 4+4 + 8 + 4(+4) + 8 + 4(+4) + 8 + 4 + 4 + 4(+4)
    assert ctypes.sizeof(mattn.MaskDesc) == 88
    assert mattn.MaskDesc.block_bits.offset == 48
    assert mattn.MaskDesc.sink.offset == 64
    assert mattn.MaskDesc.sink_tokens.offset == 80


def _desc(kind, param, **kw):
    d = mattn.MaskDesc()
    d.kind = kind
    d.param = param
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_invalid_arguments_rejected_on_host(L):
    out = ctypes.c_uint64(0)
    assert L.mattn_count_pairs(None, 1, 1, 16, ctypes.byref(out)) == mattn.ERR_INVALID_ARG
    assert L.mattn_count_pairs(ctypes.byref(_desc(9, 1)), 1, 1, 16, ctypes.byref(out)) == mattn.ERR_INVALID_ARG
    assert L.mattn_count_pairs(ctypes.byref(_desc(2, 0)), 1, 1, 16, ctypes.byref(out)) == mattn.ERR_INVALID_ARG
    assert L.mattn_count_pairs(ctypes.byref(_desc(2, 3)), 1, 0, 16, ctypes.byref(out)) == mattn.ERR_INVALID_ARG
    assert L.mattn_count_pairs(ctypes.byref(_desc(4, 64)), 1, 1, 256, ctypes.byref(out)) == mattn.ERR_UNSUPPORTED
    assert L.mattn_count_pairs(ctypes.byref(_desc(4, 128)), 1, 1, 256, ctypes.byref(out)) == mattn.ERR_INVALID_ARG
    # block-sparse N is capped by the per-CTA key-tile list (4096 tiles of 128)
    bits = np.zeros(4097 * 65, dtype=np.uint64)
    big = _desc(4, 128, block_bits=bits.ctypes.data, block_heads=1)
    assert L.mattn_count_pairs(ctypes.byref(big), 1, 1, 128 * 4096 + 1, ctypes.byref(out)) == mattn.ERR_UNSUPPORTED
    assert b"524288" in L.mattn_last_error()
    bad_scale = _desc(0, 0, softmax_scale=-1.0)
    assert L.mattn_count_pairs(ctypes.byref(bad_scale), 1, 1, 16, ctypes.byref(out)) == mattn.ERR_INVALID_ARG
    for ok_flags in (mattn.FLAG_SCHEDULE_PAIRED, mattn.FLAG_SCHEDULE_SPLIT, mattn.FLAG_SCHEDULE_SINGLE,
                     mattn.FLAG_SCHEDULE_PERSISTENT):
        assert L.mattn_count_pairs(ctypes.byref(_desc(0, 0, flags=ok_flags)), 1, 1, 16, ctypes.byref(out)) == mattn.OK
    # one schedule flag at most; the persistent schedule takes the interval masks only
    for bad_flags in (3, 5, 9, 12, 16, 0x80000000):
        flags = _desc(0, 0, flags=bad_flags)
        assert L.mattn_count_pairs(ctypes.byref(flags), 1, 1, 16, ctypes.byref(out)) == mattn.ERR_INVALID_ARG
    blk_bits = np.ones(1, dtype=np.uint64)
    persist_blk = _desc(4, 128, block_bits=blk_bits.ctypes.data, block_heads=1, flags=mattn.FLAG_SCHEDULE_PERSISTENT)
    assert L.mattn_count_pairs(ctypes.byref(persist_blk), 1, 1, 128, ctypes.byref(out)) == mattn.ERR_UNSUPPORTED
    assert b"persistent" in L.mattn_last_error()
    order = (ctypes.c_int32 * 1)(mattn.ORDER_COLUMN_MAJOR)
    cm = _desc(2, 3, head_order=order, grid_rows=3, grid_cols=5)
    assert L.mattn_count_pairs(ctypes.byref(cm), 1, 1, 16, ctypes.byref(out)) == mattn.ERR_INVALID_ARG
    assert b"grid_rows" in L.mattn_last_error()
    # sink tokens: causal windows only, never negative
    assert L.mattn_count_pairs(ctypes.byref(_desc(2, 3, sink_tokens=4)), 1, 1, 16, ctypes.byref(out)) == \
        mattn.ERR_INVALID_ARG
    assert L.mattn_count_pairs(ctypes.byref(_desc(3, 3, sink_tokens=-1)), 1, 1, 16, ctypes.byref(out)) == \
        mattn.ERR_INVALID_ARG
    assert L.mattn_count_pairs(ctypes.byref(_desc(3, 3, sink_tokens=4)), 1, 1, 16, ctypes.byref(out)) == mattn.OK
    # mattn_fwd validates before touching a device
    d = _desc(2, 3)
    x16 = ctypes.c_void_p(16)
    # grouped-query attention: H must be a multiple of H_kv
    assert L.mattn_fwd_gqa(x16, x16, x16, x16, None, 1, 6, 4, 16, 64, 0, ctypes.byref(d), None) == \
        mattn.ERR_INVALID_ARG
    assert L.mattn_fwd_gqa(x16, x16, x16, x16, None, 1, 6, 0, 16, 64, 0, ctypes.byref(d), None) == \
        mattn.ERR_INVALID_ARG
    x = ctypes.c_void_p(16)
    assert L.mattn_fwd(x, x, x, x, None, 1, 1, 16, 72, 0, ctypes.byref(d), None) == mattn.ERR_UNSUPPORTED
    assert L.mattn_fwd(None, x, x, x, None, 1, 1, 16, 64, 0, ctypes.byref(d), None) == mattn.ERR_INVALID_ARG
    assert L.mattn_fwd(ctypes.c_void_p(8), x, x, x, None, 1, 1, 16, 64, 0, ctypes.byref(d), None) == \
        mattn.ERR_UNSUPPORTED
    assert L.mattn_fwd(x, x, x, x, None, 1, 1, 16, 64, 7, ctypes.byref(d), None) == mattn.ERR_UNSUPPORTED
    # the single-pipeline schedule takes head dim 128 or 256
    single = _desc(2, 3, flags=mattn.FLAG_SCHEDULE_SINGLE)
    assert L.mattn_fwd(x, x, x, x, None, 1, 1, 16, 64, 0, ctypes.byref(single), None) == mattn.ERR_UNSUPPORTED


@pytest.mark.parametrize("rows,cols,orders,copy", [
    (64, 64, "rc-r", False),   # both 2x2-block orders through 5D TMA views
    (16, 64, "r-r-", False),   # order (c): cols % 64 == 0
    (128, 16, "c-cc", False),  # order (d): rows % 64 == 0
    (16, 64, "rc-r", True),    # order (d) with rows % 64 != 0: all heads through the copy
    (128, 16, "rc--", True),   # order (c) with cols % 64 != 0
    (64, 64, "rcc-", False),
])
def test_block2x2_orders_pick_tma_views(L, rows, cols, orders, copy):
    """Which 2x2-block orders are read in place through TMA views and which
    send the call through the reorder copy, told apart on the host: the
    no-allocation entry point refuses a call that needs the copy before it
    checks its head capacity, so with H above that capacity the first case
    returns UNSUPPORTED (the copy) and the second CAPACITY.  Neither touches
    a device."""
    H = 4097  # MATTN_NOALLOC_MAX_HEADS + 1
    code = {"r": mattn.ORDER_BLOCK2X2_ROW, "c": mattn.ORDER_BLOCK2X2_COL, "-": mattn.ORDER_RASTER}
    arr = (ctypes.c_int32 * H)(*[code[orders[h % len(orders)]] for h in range(H)])
    d = _desc(2, 40, head_order=arr, grid_rows=rows, grid_cols=cols)
    x = ctypes.c_void_p(16)
    rc = L.mattn_fwd_noalloc(x, x, x, x, None, 1, H, rows * cols, 64, 0, ctypes.byref(d), None, None)
    if copy:
        assert rc == mattn.ERR_UNSUPPORTED and b"reorder" in L.mattn_last_error()
    else:
        assert rc == mattn.ERR_CAPACITY, L.mattn_last_error()


def test_capacity_error_reports_count(L):
    spec = MaskSpec("full", [0])
    m = mattn.PreparedMask(spec, 1, 512, host_side=True)
    d = m.host_desc()
    n = ctypes.c_size_t(0)
    buf = np.zeros((3, 4), dtype=np.int32)
    rc = L.mattn_plan_tiles(ctypes.byref(d), 1, 512, buf.ctypes.data, 3, ctypes.byref(n))
    assert rc == mattn.ERR_CAPACITY and n.value == 16


def test_pack_block_bits_roundtrip():
    blk = bernoulli_causal_blocks(3, 70, 5)
    words = mattn.pack_block_bits(blk)
    assert words.shape == (3, 70, 2) and words.dtype == np.uint64
    for h in range(3):
        for m in range(70):
            for nb in range(70):
                bit = (int(words[h, m, nb // 64]) >> (nb % 64)) & 1
                assert bit == int(blk[h, m, nb])


def _spec_cases(n):
    rng = np.random.default_rng(7)
    yield "full", MaskSpec("full", [0, 0])
    yield "chunk", MaskSpec("chunk", [64, 200])
    yield "sliding", MaskSpec("sliding", [32, 300])
    yield "causal", MaskSpec("causal_window", [128, 77])
    # causal windows with sink tokens: 4 sinks (one partial tile), sinks over
    # more than one tile, a window that reaches back into the sinks
    yield "causal_sink4", MaskSpec("causal_window", [128, 77], sink_tokens=4)
    yield "causal_sink130", MaskSpec("causal_window", [572, 300], sink_tokens=130)
    yield "causal_sink128", MaskSpec("causal_window", [40, 200], sink_tokens=128)
    for bs in (128, 256):
        nb = -(-n // bs)
        yield f"block{bs}", MaskSpec("block", [bs, bs], block=bernoulli_causal_blocks(2, nb, bs))
    # upper-triangle bits present in the input must be ignored
    nb = -(-n // 128)
    blk = rng.random((2, nb, nb)) < 0.5
    yield "block_upper", MaskSpec("block", [128, 128], block=blk)


@pytest.mark.parametrize("n", [1000, 1024, 129])
def test_host_plan_matches_oracle_tiles(L, n):
    for name, spec in _spec_cases(n):
        tiles = mattn.plan_tiles(spec, 2, n)
        for h in range(2):
            got = [tuple(int(x) for x in t[1:]) for t in tiles if t[0] == h]
            assert got == dense.tile_list(spec, h, n, 128), (name, h)


def test_host_plan_matches_oracle_at_workload_sizes(L):
    for wl_name, mask in (("vit4096", "chunk256"), ("vit4096", "sliding128"), ("vit16384", "sliding256_rowcol"),
                          ("vit16384", "chunk512"), ("causal4096", "causal_window_sink")):
        wl = WORKLOADS[wl_name]
        spec = make_mask(wl, mask)
        tiles = mattn.plan_tiles(spec, wl.H, wl.N)
        for h in (0, wl.H - 1):
            got = [tuple(int(x) for x in t[1:]) for t in tiles if t[0] == h]
            assert got == dense.tile_list(spec, h, wl.N, 128), (wl_name, mask, h)


@pytest.mark.parametrize("n", [257, 1000, 4096])
def test_pair_count_matches_oracle(L, n):
    for name, spec in _spec_cases(n):
        assert mattn.count_pairs(spec, 3, 2, n) == 3 * dense.pair_count(spec, n, n_heads=2), name


def test_pair_count_workloads(L):
    """Exact unmasked pairs of the workloads (the unit of the metric)."""
    wl = WORKLOADS["vit16384"]
    assert mattn.count_pairs(make_mask(wl, "full"), 1, 16, 16384) == 16 * 16384 ** 2
    assert mattn.count_pairs(make_mask(wl, "sliding256_rowcol"), 1, 16, 16384) == 16 * 8339200
    assert mattn.count_pairs(make_mask(wl, "chunk512"), 1, 16, 16384) == 16 * 8388608
    wl4 = WORKLOADS["causal4096"]
    spec = make_mask(wl4, "causal_window_sink")
    per = {512: 1966336, 1024: 3670528, 2048: 6292480, 4096: 8390656}
    assert mattn.count_pairs(spec, 1, 16, 4096) == sum(per[w] for w in spec.head_param)
    assert sorted(spec.head_param) == sorted([512, 1024, 2048, 4096] * 4)


def test_column_major_grid_description_matches_explicit_order(L):
    n = 256
    perm = column_major_order(16, 16)
    grid = MaskSpec("sliding", [20], perm=[perm], perm_grid=[(16, 16)])
    explicit = MaskSpec("sliding", [20], perm=[perm])
    a = mattn.PreparedMask(grid, 1, n, host_side=True).host_desc()
    b = mattn.PreparedMask(explicit, 1, n, host_side=True).host_desc()
    assert a.head_order[0] == mattn.ORDER_COLUMN_MAJOR and (a.grid_rows, a.grid_cols) == (16, 16)
    assert b.head_order[0] == 0 and b.n_perm == 1


def test_plan_schedule_follows_the_stated_rules(L):
    """The schedule mattn_fwd runs, on the host: a flag wins; otherwise SPLIT
    for 128-blocks, SINGLE at head dim 256, PERSISTENT for interval masks
    whose query tiles see about 40 key tiles or fewer, PAIRED for the rest."""
    from workloads import WORKLOADS, make_mask

    def sched(wl_name, mask, d=None, flags=None):
        wl = WORKLOADS[wl_name]
        spec = make_mask(wl, mask, seed=0)
        pm = mattn.prepare(spec, wl.H, wl.N, device="cpu")
        if flags is not None:
            pm.desc.flags = flags
        return mattn.plan_schedule(pm, wl.B, wl.N, d or wl.d, mattn.F32 if wl.dtype == "f32" else mattn.BF16)

    assert sched("vit16384", "sliding256_rowcol") == "persistent"
    assert sched("vit16384", "chunk512") == "persistent"
    assert sched("vit16384", "full") == "paired"
    assert sched("vit4096", "sliding128") == "persistent"
    assert sched("causal4096", "causal_window_sink") == "persistent"  # windows up to 4096: ~16 tiles on average
    assert sched("vit4096", "full") == "persistent"  # 32 tiles
    assert sched("gqa32k", "swa572_sinktok4") == "persistent"
    assert sched("bsparse128k", "block128") == "split"
    assert sched("prefill_d256", "swa576_sink") == "single"
    assert sched("vit16384", "sliding256_rowcol", flags=mattn.FLAG_SCHEDULE_PAIRED) == "paired"
    assert sched("vit16384", "full", flags=mattn.FLAG_SCHEDULE_PERSISTENT) == "persistent"
    out = ctypes.c_uint32(0)
    assert L.mattn_plan_schedule(None, 1, 1, 128, 64, mattn.BF16, ctypes.byref(out)) == mattn.ERR_INVALID_ARG


def test_bench_pair_count_matches_the_oracle():
    """The reference arm's closed-form pair count of a block mask (kept
    blocks below the diagonal Bs^2 each, kept diagonal blocks Bs(Bs+1)/2)
    equals the oracle's count from the dense mask."""
    import bench
    from oracle import dense
    from workloads import MaskSpec, bernoulli_causal_blocks

    n, H = 1024, 3
    spec = MaskSpec("block", [128] * H, block=bernoulli_causal_blocks(H, n // 128, 5))
    assert bench.block_mask_pairs(spec, n) == dense.pair_count(spec, n, n_heads=H)
    assert bench.block_mask_pairs(spec, n, B=2) == 2 * dense.pair_count(spec, n, n_heads=H)
    one = bench.spec_head(spec, 2)
    assert one.head_param == [128] and np.array_equal(np.asarray(one.block)[0], np.asarray(spec.block)[2])
