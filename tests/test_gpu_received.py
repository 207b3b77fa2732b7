"""GPU parity of the received attention (``mattn_received``, the column sums
of the masked attention matrix) against the fp64 oracle
``oracle.dense.received_attention``.

Tolerance.  r_j = sum_i exp(s_ij - lse_i); the GPU uses the forward's fp32
log-sum-exp, which the forward parity tests hold within 1e-3 of the oracle's
(observed ~1e-6), so every term moves by at most a factor e^(1e-3): |dr_j| <=
2e-3 r_j, plus 1e-5 for fp32 accumulation.  With fp32 inputs the device
rounds q and k to bf16, which moves each score by at most delta_i =
scale * 2^-8 * max_j sum_c |q_ic||k_jc| and each term by a factor e^(2 delta_i),
so that factor is added for those cases.  Properties checked at full size:
the columns add up to N minus the sink's share of every row.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import dense  # noqa: E402
from workloads import (MaskSpec, WORKLOADS, bernoulli_causal_blocks, column_major_order,  # noqa: E402
                       make_mask, make_qkv, make_workload_inputs, random_order)

pytestmark = pytest.mark.gpu

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


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _run(q, k, v, spec, heads=None):
    B, H, N, d = q.shape
    mask = mattn.prepare(spec, H, N)
    _, lse = mattn.attention(q, k, v, mask)
    r = mattn.received(q, k, lse, mask)
    torch.cuda.synchronize()
    rc, word = mattn.device_status()
    assert rc == 0, f"device error word {word:#x}"
    return r, lse


def _check(q, k, v, spec, tag, heads=None, cols=None):
    B, H, N, d = q.shape
    r, _ = _run(q, k, v, spec)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    ref = dense.received_attention(_np(q), _np(k), spec, heads=heads, cols=cols)
    got = np.stack([_np(r[b, h]) for b, h in heads])
    if cols is not None:
        got = got[:, cols]
    rtol = np.full(len(heads), 2e-3)
    if q.dtype == torch.float32:
        scale = 1.0 / math.sqrt(d)
        for i, (b, h) in enumerate(heads):
            qa, ka = np.abs(_np(q[b, h])), np.abs(_np(k[b, h]))
            delta = scale * 2.0 ** -8 * (qa @ ka.T).max()
            rtol[i] += math.exp(2 * delta) - 1
    err = np.abs(got - ref)
    bad = err > rtol[:, None] * ref + 1e-5
    assert not bad.any(), f"{tag}: max rel err {(err / np.maximum(ref, 1e-12)).max():.3e}"


@pytest.mark.parametrize("d", [64, 80, 128])
@pytest.mark.parametrize("n", [256, 1000])
def test_kinds(d, n):
    q, k, v = make_qkv(1, 2, n, d, "bf16", 1.0, seed=d + n + 1, device="cuda")
    nb = -(-n // 128)
    specs = [
        MaskSpec("full", [0, 0]),
        MaskSpec("chunk", [100, 128]),
        MaskSpec("sliding", [70, 200]),
        MaskSpec("causal_window", [300, 64], sink=np.array([0.5, -1.0])),
        MaskSpec("block", [128, 128], block=bernoulli_causal_blocks(2, nb, n), sink=np.array([1.5, 0.0])),
    ]
    for spec in specs:
        _check(q, k, v, spec, f"{spec.kind} d{d} n{n}")


def test_orders_batch_and_fp32():
    """Column-major heads read through strided views, an explicit order and
    fp32 inputs (both through the reorder pass), two batch entries."""
    n, d = 1024, 64
    grid = (128, 8)
    cm = column_major_order(*grid)
    q, k, v = make_qkv(2, 3, n, d, "bf16", 1.0, seed=3, device="cuda")
    spec = MaskSpec("sliding", [40, 90, 300], perm=[None, cm, None], perm_grid=[None, grid, None],
                    sink=np.array([0.2, -0.3, 0.9]))
    _check(q, k, v, spec, "column-major")
    spec = MaskSpec("chunk", [64, 200, 128], perm=[random_order(n, 5), None, cm])
    _check(q, k, v, spec, "explicit orders")
    q32, k32, v32 = make_qkv(1, 2, 256, 64, "f32", 1.0, seed=4, device="cuda")
    _check(q32, k32, v32, MaskSpec("sliding", [32, 32]), "fp32")


@pytest.mark.parametrize("name,mask", [("vit16384", "sliding256_rowcol"), ("causal4096", "causal_window_sink")])
def test_workload_sizes(name, mask):
    """Full workload sizes: every head's columns add up to N minus the sink's
    share of the rows (from the forward's LSE), and on one raster and one
    column-major / windowed head, sampled columns match the oracle."""
    wl = WORKLOADS[name]
    q, k, v = make_workload_inputs(wl, seed=0, device="cuda")
    spec = make_mask(wl, mask, seed=0)
    r, lse = _run(q, k, v, spec)
    rn, ln = _np(r), _np(lse)
    for b in range(wl.B):
        for h in range(wl.H):
            share = 0.0
            if spec.sink is not None:
                share = np.exp(float(spec.sink[h]) - ln[b, h]).sum()
            assert rn[b, h].sum() == pytest.approx(wl.N - share, rel=1e-3)
    rng = np.random.default_rng(1)
    cols = np.unique(np.concatenate([[0, wl.N - 1], rng.choice(wl.N, 62, replace=False)]))
    heads = [(0, 0), (0, wl.H - 1)]
    _check(q, k, v, spec, f"{name}/{mask}", heads=heads, cols=cols)


def test_block_sparse_128k_conserves_mass():
    """The 128K-token, 32-head block-sparse recipe: each head's columns add
    up to N (every row keeps its diagonal block, no sink)."""
    wl = WORKLOADS["bsparse128k"]
    q, k, v = make_workload_inputs(wl, seed=0, device="cuda")
    spec = make_mask(wl, "block128", seed=0)
    r, _ = _run(q, k, v, spec)
    sums = _np(r).sum(axis=-1)
    np.testing.assert_allclose(sums, wl.N, rtol=1e-3)
