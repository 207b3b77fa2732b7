"""GPU parity of decode-shaped attention (one new query per sequence against
its key/value cache; the Bifocal page's speed-test shapes: 16 query heads
sharing 4 key/value heads of dimension 256, prompts up to 128K tokens)
through the C ABI against the fp64 oracle.  Tolerances as for the forward:
max |dO| <= 2e-2, rel-L2 <= 5e-3, |dLSE| <= 1e-3."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import dense  # noqa: E402
from workloads import MaskSpec, WORKLOADS, make_decode_inputs, make_mask  # noqa: E402

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


def check_decode(q, k, v, spec, lens=None, tag=""):
    B, H, d = q.shape
    L = k.shape[2]
    mask = mattn.prepare(spec, H, L)
    sl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = mattn.decode(q, k, v, mask, seq_lens=sl)
    torch.cuda.synchronize()
    ref_o, ref_lse = dense.decode(_host(q), _host(k), _host(v), lens, spec)
    got_o = _host(o).astype(np.float64)
    got_lse = _host(lse).astype(np.float64)
    err = np.abs(got_o - ref_o)
    rel = np.linalg.norm(got_o - ref_o) / max(np.linalg.norm(ref_o), 1e-30)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(fin, np.isfinite(got_lse)), f"{tag}: LSE -inf pattern differs"
    lse_err = np.abs(np.where(fin, got_lse, 0.0) - np.where(fin, ref_lse, 0.0))
    assert err.max() <= MAX_ABS, f"{tag}: max abs {err.max():.3e}"
    assert rel <= REL_L2 or np.linalg.norm(ref_o) == 0, f"{tag}: rel L2 {rel:.3e}"
    assert lse_err.max() <= LSE_ABS, f"{tag}: lse err {lse_err.max():.3e}"
    return o, lse


def _inputs(B, H, Hkv, L, d, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn((B, H, d), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((B, Hkv, L, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, Hkv, L, d), generator=g, device="cuda").to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("H,Hkv", [(8, 2), (3, 1), (8, 1), (4, 4)])
def test_decode_masks(d, H, Hkv):
    """Full and windowed decode (per-head windows that differ inside a
    key/value group, a learned sink logit, sink tokens) on sequences of
    different lengths in one batch: a full cache, one token, a ragged one."""
    L = 1000
    q, k, v = _inputs(3, H, Hkv, L, d, seed=d * 7 + H + Hkv)
    lens = [L, 1, 517]
    wins = [64, 300, 128, 999, 1, 500, 1000, 77][:H]
    sink = np.linspace(-1.0, 1.5, H)
    specs = [
        MaskSpec("full", [0] * H),
        MaskSpec("full", [0] * H, sink=sink),
        MaskSpec("causal_window", wins, sink=sink),
        MaskSpec("causal_window", [572] * H, sink_tokens=4),
        MaskSpec("causal_window", wins, sink_tokens=130),
    ]
    for spec in specs:
        check_decode(q, k, v, spec, lens=lens, tag=f"{spec.kind} d{d} H{H}/{Hkv} W{spec.head_param[:2]}")


def test_decode_edge_lengths():
    """len = L for every sequence (seq_lens omitted), len = 0 (no key:
    O = 0 and LSE = -inf, or the sink logit alone), lengths past L clamped."""
    q, k, v = _inputs(2, 4, 2, 300, 128, seed=3)
    check_decode(q, k, v, MaskSpec("causal_window", [100] * 4), lens=None, tag="no seq_lens")
    spec = MaskSpec("full", [0] * 4, sink=np.array([0.5, -0.5, 1.0, 0.0]))
    o, lse = check_decode(q, k, v, spec, lens=[0, 300], tag="len 0 with sink")
    assert float(o[0].abs().max()) == 0.0
    np.testing.assert_allclose(_host(lse[0]), [0.5, -0.5, 1.0, 0.0], atol=1e-6)
    sl = torch.tensor([1000, 5], dtype=torch.int32, device="cuda")
    o2, lse2 = mattn.decode(q, k, v, mattn.prepare(MaskSpec("full", [0] * 4), 4, 300), seq_lens=sl)
    ref_o, ref_lse = dense.decode(_host(q), _host(k), _host(v), [300, 5], MaskSpec("full", [0] * 4))
    assert np.abs(_host(o2) - ref_o).max() <= MAX_ABS
    assert np.abs(_host(lse2) - ref_lse).max() <= LSE_ABS


@pytest.mark.parametrize("mask", ["full", "swa576_sink", "swa572_sinktok4"])
def test_decode128k_full_size(mask):
    """The 128K-token decode step the bench times (B1, 16 query heads, 4
    key/value heads, d256, full cache), every head against the oracle."""
    wl = WORKLOADS["decode128k"]
    q, k, v = make_decode_inputs(wl, seed=0, device="cuda")
    spec = make_mask(wl, mask)
    check_decode(q, k, v, spec, lens=None, tag=f"decode128k {mask}")
