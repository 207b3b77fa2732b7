"""GPU parity of RRAttention's dynamic block selection (``mattn_rr_select``)
against the fp64 oracle ``oracle.rr_select``.

What is compared, and how closely:

- Block scores S (Eq. 10).  The GPU sums each stride's keys in fp32 and
  rounds the sum to bf16 before the tensor-core product, so every importance
  I_ij moves by at most delta_i = scale * sum_c |q_ic| |Ksum_jc| * 2^-8
  (relative bf16 rounding 2^-9, doubled for margin); a softmax moves by at
  most a factor exp(+-2 delta) under such a change, so
  |S_gpu - S| <= S * (exp(2 delta_m) - 1) with delta_m the largest delta_i of
  query block m, plus 1e-5 per stride pair for fp32 accumulation and the
  exp2 approximation.
- The selection (Eq. 11) is an integer result decided by floating point.
  The GPU's bits are compared with the fp64 Eq. 11 rule (``top_tau``)
  applied to the GPU's own scores.  They must be equal on every row except
  one whose sorted running sum passes tau times the row total within
  2^-18 of the total: there the kernel's own precision decides (it sums
  scores quantised to 2^-30 of the row maximum over at most 1024 blocks,
  < 2^-19 of the total in all, and rounds tau to a multiple of 2^-20), so
  either side of the crossing is correct.  On such a row the GPU's set
  must still be valid: apart from the crossing block, the blocks in which
  the two sets differ add up to less than that 2^-18 of the total, and no
  dropped block scores above a kept one (beyond 2^-28 of the row maximum).  On inputs with a planted pattern, whose decisions have a wide
  margin, the GPU's bits must equal the oracle's bits from its own fp64
  scores exactly.
- Eq. 12 and Eq. 5 (last query block full, nothing above the diagonal) are
  checked exactly everywhere, also at the 128K-token, 32-head size on every
  row, with scores compared on sampled rows there.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import dense, rr_select as orr  # noqa: E402
from workloads import MaskSpec, make_qkv  # noqa: E402

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


# A crossing of tau * total closer than this share of the total is decided
# by the kernel's precision (see the module docstring).
NEAR_CROSSING = 2.0 ** -18
SCORE_SLACK = 2.0 ** -28


def _check_decision(row_scores, gpu_row, tau, m, sink_recent, tag):
    """Eq. 11 on one query block m: GPU bits vs the fp64 rule on the GPU's
    own (fp32) scores, with the near-crossing allowance."""
    x = np.maximum(np.asarray(row_scores, dtype=np.float64), 0.0)
    nb = x.size
    causal = np.arange(nb) <= m
    want = orr.top_tau(x, tau) & causal
    if sink_recent:
        want[0] = True
        want[m] = True
    if (want == gpu_row).all():
        return
    order = np.lexsort((np.arange(nb), -x))
    csum = np.cumsum(x[order])
    total = x.sum()
    gap = np.abs(csum - tau * total).min()
    assert gap <= NEAR_CROSSING * total, f"{tag}: selection differs away from a near-crossing (gap {gap / total:.3e})"
    pinned = np.zeros(nb, dtype=bool)
    if sink_recent:
        pinned[0] = pinned[m] = True
    free = causal & ~pinned
    kept, dropped = x[free & gpu_row], x[free & ~gpu_row]
    # both sets are prefixes of the same descending order whose sums sit on
    # either side of the ambiguous crossing: apart from the crossing block
    # itself, the blocks in one set only add up to less than the ambiguity
    diff = x[free & (gpu_row != want)]
    assert diff.sum() - diff.max() <= NEAR_CROSSING * total, f"{tag}: the sets differ beyond the crossing block"
    if kept.size and dropped.size:
        assert dropped.max() <= kept.min() + SCORE_SLACK * x.max(), f"{tag}: a dropped block outscores a kept one"


def _check_scores(q, k, S, Bs, tau, sink_recent, scores_gpu, bits_gpu, exact_bits):
    B, H, L, d = q.shape
    nb = -(-(L // S) // (Bs // S))
    qn, kn = _np(q), _np(k)
    bits = mattn.unpack_block_bits(bits_gpu.cpu().numpy(), nb).reshape(B, H, nb, nb)
    sc = scores_gpu.cpu().numpy().astype(np.float64).reshape(B, H, nb, nb)
    g = Bs // S
    for b in range(B):
        for h in range(H):
            B_or, S_or = orr.select_head(qn[b, h], kn[b, h], S, Bs, tau, h, sink_recent)
            # score tolerance per query block
            scale = 1.0 / (S * math.sqrt(d))
            ks = np.abs(orr.stride_key_sums(kn[b, h], S))
            qs = np.abs(qn[b, h][orr.sampled_positions(L, S, h)])
            delta = scale * 2.0 ** -8 * (qs @ ks.T).max(axis=1)      # per sampled query
            dm = np.array([delta[m * g:(m + 1) * g].max() for m in range(nb)])
            tol = S_or * (np.exp(2 * dm) - 1)[:, None] + 1e-5 * g * g
            err = np.abs(sc[b, h] - S_or)
            assert (err <= tol).all(), f"b{b} h{h}: score err {err.max():.3e} (tol {tol[err.argmax() // nb].max():.3e})"
            # Eq. 12 and Eq. 5
            assert bits[b, h, nb - 1].all()
            assert not np.triu(bits[b, h], 1).any()
            # Eq. 11 on the GPU's own scores (fp64 rule, near-crossing allowance)
            for m in range(nb - 1):
                _check_decision(sc[b, h, m], bits[b, h, m], tau, m, sink_recent, f"b{b} h{h} m{m}")
            if exact_bits:
                assert (bits[b, h] == B_or).all(), f"b{b} h{h}: bits differ from the oracle's"
    return bits


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S,Bs", [(8, 128), (4, 128), (16, 128), (8, 64)])
@pytest.mark.parametrize("L", [1024, 1536])
def test_random_inputs(d, S, Bs, L):
    """Random N(0,1) heads (flat, near-tied scores): scores within the derived
    tolerance, decisions consistent with the GPU's own scores; two sampling
    offsets per stride at least (H = 3), a ragged last query tile at L = 1536."""
    q, k, _ = make_qkv(1, 3, L, d, "bf16", 1.0, seed=L + d + S, device="cuda")
    for tau, sr in ((0.9, False), (0.95, True)):
        bits, scores = mattn.rr_select(q, k, S, Bs, tau, sink_recent=sr, want_scores=True)
        torch.cuda.synchronize()
        assert mattn.device_status()[0] == 0
        _check_scores(q, k, S, Bs, tau, sr, scores, bits, exact_bits=False)


def _planted(B, H, L, d, S, seed):
    """Heads whose attention concentrates on a few key strides per head: a
    shared direction e_0 carries large weight on the planted strides."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, L, d)) * 0.3
    k = rng.standard_normal((B, H, L, d)) * 0.3
    q[..., 0] = 2.0
    ns = L // S
    for b in range(B):
        for h in range(H):
            for j in rng.choice(ns, size=max(2, ns // 16), replace=False):
                k[b, h, j * S:(j + 1) * S, 0] = rng.uniform(6.0, 12.0)
    tq = torch.from_numpy(q).to(torch.bfloat16).cuda()
    tk = torch.from_numpy(k).to(torch.bfloat16).cuda()
    return tq, tk


@pytest.mark.parametrize("d,S,Bs,L", [(128, 8, 128, 2048), (64, 16, 128, 2048), (128, 4, 128, 1152)])
def test_planted_pattern_matches_oracle_bits(d, S, Bs, L):
    """With a planted pattern the decisions have margin: the GPU bitmap equals
    the oracle's bitmap from its own fp64 scores, for two batch entries."""
    q, k = _planted(2, 3, L, d, S, seed=L + S)
    bits, scores = mattn.rr_select(q, k, S, Bs, 0.9, want_scores=True)
    torch.cuda.synchronize()
    assert mattn.device_status()[0] == 0
    _check_scores(q, k, S, Bs, 0.9, False, scores, bits, exact_bits=True)


def test_selection_feeds_attention():
    """The bitmap is in the attention kernel's layout: attention with the GPU's
    bits equals the fp64 attention oracle with the same (oracle-equal) bits."""
    L, d, S, Bs, H = 2048, 128, 8, 128, 3
    q, k = _planted(1, H, L, d, S, seed=7)
    v = torch.randn((1, H, L, d), device="cuda").to(torch.bfloat16)
    bits, _ = mattn.rr_select(q, k, S, Bs, 0.9)
    mask = mattn.DeviceBlockMask(bits, H, L, Bs)
    o, lse = mattn.attention(q, k, v, mask)
    torch.cuda.synchronize()
    assert mattn.device_status()[0] == 0
    nb = L // Bs
    Bm = mattn.unpack_block_bits(bits.cpu().numpy(), nb)
    B_or, _ = orr.select(_np(q), _np(k), S, Bs, 0.9)
    assert (Bm == B_or[0]).all()
    spec = MaskSpec("block", [Bs] * H, block=B_or[0])
    ref_o, ref_lse = dense.attention(_np(q), _np(k), _np(v), spec)
    got = _np(o).reshape(ref_o.shape)
    assert np.abs(got - ref_o).max() <= 2e-2
    assert np.linalg.norm(got - ref_o) / np.linalg.norm(ref_o) <= 5e-3
    assert np.abs(_np(lse).reshape(ref_lse.shape) - ref_lse).max() <= 1e-3


def test_full_size_128k_sampled_rows():
    """The 128K-token, 32-head prefill recipe (d 128, stride 8, block 128,
    tau 0.95): the whole bitmap obeys Eq. 12 and Eq. 5; on sampled (head,
    query block) rows the scores match the fp64 oracle's row within the
    derived tolerance and the decision follows Eq. 11 on the GPU's own scores."""
    B, H, L, d, S, Bs, tau = 1, 32, 131072, 128, 8, 128, 0.95
    q, k, _ = make_qkv(B, H, L, d, "bf16", 1.0, seed=0, device="cuda")
    bits, scores = mattn.rr_select(q, k, S, Bs, tau, want_scores=True)
    torch.cuda.synchronize()
    assert mattn.device_status()[0] == 0
    nb = L // Bs
    allbits = mattn.unpack_block_bits(bits.cpu().numpy(), nb)
    assert allbits[:, nb - 1].all()
    assert not (allbits & np.triu(np.ones((nb, nb), dtype=bool), 1)).any()
    rng = np.random.default_rng(0)
    ns, g = L // S, Bs // S
    for h in rng.choice(H, size=3, replace=False):
        qh, kh = _np(q[0, h]), _np(k[0, h])
        ksum = orr.stride_key_sums(kh, S)
        pos = orr.sampled_positions(L, S, int(h))
        for m in [0, int(rng.integers(1, nb - 1)), nb - 2]:
            rows = pos[m * g:(m + 1) * g]
            I = (qh[rows] @ ksum.T) / (S * math.sqrt(d))
            P = orr.stride_softmax(I)
            S_row = P.reshape(g, nb, g).sum(axis=(0, 2))
            delta = (2.0 ** -8 / (S * math.sqrt(d))) * (np.abs(qh[rows]) @ np.abs(ksum).T).max()
            tol = S_row * (np.exp(2 * delta) - 1) + 1e-5 * g * g
            got = scores[int(h), m].cpu().numpy().astype(np.float64)
            assert (np.abs(got - S_row) <= tol).all(), (int(h), m)
            _check_decision(got, allbits[int(h), m], tau, m, False, f"h{int(h)} m{m}")
