"""GPU parity of the LLM variants: grouped-query attention and a causal
window with StreamingLLM sink tokens (the Bifocal page: Qwen3-4B's 32 query
heads sharing 8 key/value heads; a 572-token window plus the first 4
tokens), through the C ABI against the fp64 oracle.

Tolerances as for the other parity tests: max |dO| <= 2e-2, rel-L2 <= 5e-3,
|dLSE| <= 1e-3 (bf16 inputs, fp32 accumulation on both sides of the
comparison; fp32 inputs add the bound of their bf16 rounding to the LSE).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import dense  # noqa: E402
from workloads import MaskSpec, WORKLOADS, bernoulli_causal_blocks, make_mask, make_qkv  # noqa: E402
from workloads import make_workload_inputs  # noqa: E402

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3

mattn = pytest.importorskip("block_sparse_attention_masked_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import os

    if not os.path.exists(mattn.LIB_PATH):
        from block_sparse_attention_masked_gb300 import build

        build.build()
    mattn.lib()


def _host(t):
    return t.detach().float().cpu().numpy()


def check_gqa(q, k, v, spec, rows=None, groups=None, tag=""):
    """Run the library on q [B, H, N, d], k, v [B, H_kv, N, d] and compare the
    query heads of key/value groups ``groups`` (all by default) with the
    oracle on the same group slices (the oracle maps query heads to their
    key/value head itself)."""
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    G = H // Hkv
    mask = mattn.prepare(spec, H, N)
    o, lse = mattn.attention(q, k, v, mask)
    torch.cuda.synchronize()
    rc, word = mattn.device_status()
    assert rc == 0, f"device error word {word:#x}"
    groups = list(range(Hkv)) if groups is None else list(groups)
    rows_arr = np.arange(N) if rows is None else np.asarray(rows)
    for g in groups:
        hs = list(range(g * G, (g + 1) * G))
        sub = MaskSpec(spec.kind, [spec.head_param[h] for h in hs],
                       sink=None if spec.sink is None else np.asarray(spec.sink)[hs],
                       block=None if spec.block is None else np.asarray(spec.block)[hs],
                       sink_tokens=spec.sink_tokens,
                       perm=None if spec.perm is None else [spec.perm[h] for h in hs],
                       perm_grid=None if spec.perm_grid is None else [spec.perm_grid[h] for h in hs])
        qs = _host(q[:, g * G:(g + 1) * G])
        ks, vs = _host(k[:, g:g + 1]), _host(v[:, g:g + 1])
        ref_o, ref_lse = dense.attention(qs, ks, vs, sub, rows=rows_arr)
        got_o = np.stack([_host(o[b, h])[rows_arr] for b in range(B) for h in hs]).astype(np.float64)
        got_lse = np.stack([_host(lse[b, h])[rows_arr] for b in range(B) for h in hs]).astype(np.float64)
        err = np.abs(got_o - ref_o)
        rel = np.linalg.norm(got_o - ref_o) / max(np.linalg.norm(ref_o), 1e-30)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(got_lse)), f"{tag} group {g}: LSE -inf pattern differs"
        lse_tol = LSE_ABS
        if q.dtype == torch.float32:
            scale = 1.0 / np.sqrt(d)
            qa, ka = np.abs(qs[0]), np.abs(ks[0, 0])
            bound = np.stack([(qa[i][rows_arr] @ ka.T).max(axis=1) for i in range(G)])
            lse_tol = np.maximum(LSE_ABS, scale * 2.0 ** -8 * bound + 1e-4)
        lse_err = np.abs(np.where(fin, got_lse, 0.0) - np.where(fin, ref_lse, 0.0))
        assert err.max() <= MAX_ABS, f"{tag} group {g}: max abs {err.max():.3e}"
        assert rel <= REL_L2, f"{tag} group {g}: rel L2 {rel:.3e}"
        assert (lse_err <= lse_tol).all(), f"{tag} group {g}: lse err {lse_err.max():.3e}"
    return o, lse


@pytest.mark.parametrize("H,Hkv", [(8, 2), (4, 1), (6, 3)])
@pytest.mark.parametrize("d,n", [(64, 1000), (128, 700)])
def test_gqa_kinds(H, Hkv, d, n):
    """Every mask kind with query heads sharing key/value heads; several
    tiles and a ragged last tile."""
    q, k, v = make_qkv(1, H, n, d, "bf16", 1.0, seed=H * n + d, device="cuda", kv_heads=Hkv)
    nb = -(-n // 128)
    sink = np.linspace(-1.0, 1.0, H)
    specs = [
        MaskSpec("full", [0] * H),
        MaskSpec("chunk", [256] * H),
        MaskSpec("sliding", [100] * H),
        MaskSpec("causal_window", [300] * H, sink=sink),
        MaskSpec("causal_window", [200] * H, sink_tokens=4),
        MaskSpec("block", [128] * H, block=bernoulli_causal_blocks(H, nb, n)),
    ]
    for spec in specs:
        check_gqa(q, k, v, spec, tag=f"{spec.kind} H{H}/{Hkv} d{d} n{n} sinktok{spec.sink_tokens}")


@pytest.mark.parametrize("w,s,n", [(128, 4, 1000), (572, 4, 1300), (40, 130, 900), (300, 128, 1024),
                                   (1, 1, 260), (2000, 4, 700)])
def test_sink_tokens(w, s, n):
    """Causal windows with sink tokens: sinks inside one tile, sinks over
    more than one tile, a window that reaches back into the sinks, a
    one-key window, a window longer than the sequence; with a learned sink
    logit as well on odd heads."""
    H = 2
    q, k, v = make_qkv(1, H, n, 128, "bf16", 1.0, seed=w + s + n, device="cuda")
    for sink in (None, np.array([0.0, 1.5])):
        spec = MaskSpec("causal_window", [w, w + 17], sink=sink, sink_tokens=s)
        check_gqa(q, k, v, spec, tag=f"W{w} S{s} n{n} sink{sink is not None}")


def test_gqa_fp32_inputs_and_column_major():
    """fp32 inputs (rounded to bf16 in the pre-pass, which copies each
    key/value head once per query head) and column-major query heads read
    in place."""
    n, H, Hkv = 1024, 4, 2
    q, k, v = make_qkv(1, H, n, 64, "f32", 1.0, seed=5, device="cuda", kv_heads=Hkv)
    check_gqa(q, k, v, MaskSpec("causal_window", [200] * H, sink_tokens=4), tag="fp32")
    qb, kb, vb = make_qkv(1, H, n, 64, "bf16", 0.5, seed=6, device="cuda", kv_heads=Hkv)
    from workloads import column_major_order

    col = column_major_order(128, 8)
    spec = MaskSpec("sliding", [64] * H, perm=[None, col, None, col], perm_grid=[None, (128, 8), None, (128, 8)])
    mask = mattn.prepare(spec, H, n)
    o, lse = mattn.attention(qb, kb, vb, mask)
    torch.cuda.synchronize()
    ref_o, ref_lse = dense.attention(_host(qb), _host(kb), _host(vb), spec)
    got = np.stack([_host(o[0, h]) for h in range(H)]).astype(np.float64)
    assert np.abs(got - ref_o).max() <= MAX_ABS
    assert np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o) <= REL_L2
    assert np.abs(np.stack([_host(lse[0, h]) for h in range(H)]) - ref_lse).max() <= LSE_ABS


def test_gqa_with_2x2_block_orders():
    """Query heads sharing key/value heads, each query head with its own
    grid order (both 2x2-block orders and raster over a 64 x 64 grid, read
    in place through 5D tensor maps): a work item reads its K/V head's rows
    in its query head's order."""
    from workloads import block2x2_order

    side, H, Hkv = 64, 4, 2
    n = side * side
    q, k, v = make_qkv(1, H, n, 128, "bf16", 1.0, seed=9, device="cuda", kv_heads=Hkv)
    row, col = block2x2_order(side, side), block2x2_order(side, side, by_columns=True)
    spec = MaskSpec("sliding", [70, 70, 200, 33], perm=[row, col, None, row],
                    perm_grid=[(side, side, "block2x2_row"), (side, side, "block2x2_col"), None,
                               (side, side, "block2x2_row")])
    check_gqa(q, k, v, spec, tag="gqa 2x2-block orders")


def test_device_tile_walk_with_sink_tokens():
    n = 4096
    spec = MaskSpec("causal_window", [572, 300, 40], sink_tokens=4)
    tiles = mattn.plan_tiles_device(mattn.prepare(spec, 3, n), 3, n)
    for h in range(3):
        got = [tuple(int(x) for x in t[1:]) for t in tiles if t[0] == h]
        assert got == dense.tile_list(spec, h, n, 128)
    spec = MaskSpec("causal_window", [130], sink_tokens=300)
    tiles = mattn.plan_tiles_device(mattn.prepare(spec, 1, n), 1, n)
    assert [tuple(int(x) for x in t[1:]) for t in tiles] == dense.tile_list(spec, 0, n, 128)


@pytest.mark.parametrize("mask", ["swa572_sinktok4", "swa576_sink"])
def test_gqa32k_full_size_sampled(mask):
    """The 32K-token grouped-query prefill the bench times (32 query heads,
    8 key/value heads, d128), full size, on sampled rows of the first and the
    last key/value group: the sink tokens, the window edges, tile edges and
    the last row."""
    wl = WORKLOADS["gqa32k"]
    q, k, v = make_workload_inputs(wl, seed=0, device="cuda")
    spec = make_mask(wl, mask)
    rng = np.random.default_rng(3)
    rows = sorted({0, 1, 3, 4, 5, 127, 128, 571, 572, 575, 576, 577, 4095, 4096, wl.N - 129, wl.N - 128,
                   wl.N - 1} | set(int(x) for x in rng.integers(0, wl.N, 40)))
    check_gqa(q, k, v, spec, rows=rows, groups=[0, wl.kv_heads - 1], tag=f"gqa32k {mask}")


# ---------------------------------------------------------------- head dim 256

@pytest.mark.parametrize("H,Hkv,n", [(4, 1, 1000), (16, 4, 700), (2, 2, 300)])
def test_d256_kinds(H, Hkv, n):
    """Head dim 256 (the speed-test layout) on every interval mask, with a
    sink logit and sink tokens, several tiles and a ragged last tile."""
    q, k, v = make_qkv(1, H, n, 256, "bf16", 1.0, seed=7 * n + H, device="cuda", kv_heads=Hkv)
    sink = np.linspace(-1.0, 1.0, H)
    specs = [
        MaskSpec("full", [0] * H),
        MaskSpec("causal_window", [n] * H),
        MaskSpec("chunk", [256] * H),
        MaskSpec("sliding", [100] * H, sink=sink),
        MaskSpec("causal_window", [300] * H, sink=sink),
        MaskSpec("causal_window", [200] * H, sink_tokens=4),
        MaskSpec("causal_window", [64] * H, sink_tokens=130),
    ]
    for spec in specs:
        check_gqa(q, k, v, spec, tag=f"d256 {spec.kind} {spec.head_param[0]} H{H}/{Hkv} n{n} st{spec.sink_tokens}")


def test_d256_fp32_and_orders():
    """fp32 inputs and column-major / explicit orders go through the reorder
    copy; outputs come back in caller order."""
    n, H = 512, 2
    q, k, v = make_qkv(1, H, n, 256, "f32", 1.0, seed=9, device="cuda")
    check_gqa(q, k, v, MaskSpec("causal_window", [200, 333], sink=np.array([0.3, -0.3])), tag="d256 fp32")
    from workloads import column_major_order, random_order

    qb, kb, vb = make_qkv(1, H, n, 256, "bf16", 0.5, seed=10, device="cuda")
    spec = MaskSpec("sliding", [40, 40], perm=[column_major_order(128, 4), random_order(n, 3)],
                    perm_grid=[(128, 4), None])
    mask = mattn.prepare(spec, H, n)
    o, lse = mattn.attention(qb, kb, vb, mask)
    torch.cuda.synchronize()
    ref_o, ref_lse = dense.attention(_host(qb), _host(kb), _host(vb), spec)
    got = np.stack([_host(o[0, h]) for h in range(H)]).astype(np.float64)
    assert np.abs(got - ref_o).max() <= MAX_ABS
    assert np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o) <= REL_L2
    assert np.abs(np.stack([_host(lse[0, h]) for h in range(H)]) - ref_lse).max() <= LSE_ABS


@pytest.mark.parametrize("bs,n", [(128, 1000), (256, 1300)])
def test_d256_block_sparse(bs, n):
    """Block-sparse masks at head dim 256 (the CTA's key-tile list from the
    bitmap, causal diagonal tiles masked), with GQA and a sink logit."""
    H, Hkv = 4, 2
    q, k, v = make_qkv(1, H, n, 256, "bf16", 1.0, seed=bs + n, device="cuda", kv_heads=Hkv)
    spec = MaskSpec("block", [bs] * H, block=bernoulli_causal_blocks(H, -(-n // bs), n + bs),
                    sink=np.linspace(-0.5, 0.5, H))
    check_gqa(q, k, v, spec, tag=f"d256 block{bs} n{n}")


@pytest.mark.parametrize("n", [1000, 4096])
def test_single_schedule_d128(n):
    """Head dim 128 in the single-pipeline schedule (one query tile per CTA,
    S double-buffered): block-sparse, causal window with sink tokens, full."""
    H, Hkv = 4, 2
    q, k, v = make_qkv(1, H, n, 128, "bf16", 1.0, seed=n + 3, device="cuda", kv_heads=Hkv)
    nb = -(-n // 128)
    specs = [MaskSpec("block", [128] * H, block=bernoulli_causal_blocks(H, nb, n)),
             MaskSpec("causal_window", [300] * H, sink_tokens=4, sink=np.linspace(-1, 1, H)),
             MaskSpec("full", [0] * H)]
    for spec in specs:
        B, Hq, N, d = q.shape
        mask = mattn.prepare(spec, Hq, N, schedule="single")
        o, lse = mattn.attention(q, k, v, mask)
        torch.cuda.synchronize()
        ref = mattn.attention(q, k, v, mattn.prepare(spec, Hq, N))
        torch.cuda.synchronize()
        # the same result as the two-sub-tile kernel up to rounding order
        assert (o.float() - ref[0].float()).abs().max().item() <= 2e-2
        assert (lse - ref[1]).abs().max().item() <= 1e-3
        if n <= 1000:
            sub = [0, Hkv - 1]
            for g in sub:
                hs = list(range(g * 2, g * 2 + 2))
                qs = _host(q[:, hs[0]:hs[-1] + 1])
                ks, vs = _host(k[:, g:g + 1]), _host(v[:, g:g + 1])
                ss = MaskSpec(spec.kind, [spec.head_param[h] for h in hs],
                              sink=None if spec.sink is None else np.asarray(spec.sink)[hs],
                              block=None if spec.block is None else np.asarray(spec.block)[hs],
                              sink_tokens=spec.sink_tokens)
                ref_o, _ = dense.attention(qs, ks, vs, ss)
                got = np.stack([_host(o[0, h]) for h in hs]).astype(np.float64)
                assert np.abs(got - ref_o[:]).max() <= MAX_ABS
                assert np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o) <= REL_L2


@pytest.mark.parametrize("mask", ["causal", "swa576_sink"])
def test_prefill_d256_full_size_sampled(mask):
    """The 16K-token d256 prefill the bench times (16 query heads, 4 K/V
    heads), sampled rows of the first and last groups."""
    wl = WORKLOADS["prefill_d256"]
    q, k, v = make_workload_inputs(wl, seed=0, device="cuda")
    spec = make_mask(wl, mask)
    rng = np.random.default_rng(5)
    rows = sorted({0, 1, 63, 64, 127, 128, 575, 576, 577, wl.N - 65, wl.N - 64, wl.N - 1}
                  | set(int(x) for x in rng.integers(0, wl.N, 24)))
    check_gqa(q, k, v, spec, rows=rows, groups=[0, wl.kv_heads - 1], tag=f"prefill_d256 {mask}")
