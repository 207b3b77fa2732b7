"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks ``oracle.dense`` against something other than itself: a
worked example printed on the pages, a hand-computed closed form, a
structural special case, an invariant, or the independent pure-Python brute
force.  The comment on each test names the plausible oracle mistake it
catches.
"""

import math

import numpy as np
import pytest

from conftest import read_golden
from oracle import brute, dense
from workloads import MaskSpec, bernoulli_causal_blocks, column_major_order, random_order


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _one_head(kind, param, perm=None, block=None, sink=None):
    return MaskSpec(kind, [param], perm=[perm] if perm is not None else None,
                    block=None if block is None else block[None],
                    sink=None if sink is None else np.array([sink]))


# -- masks -------------------------------------------------------------------

def test_worked_example_sliding_window():
    """SHS slides, Factor 2: anchor 15 -> 7..23, anchor 23 -> 15..31 (catches
    an exclusive bound or a one-sided window)."""
    for n, w, anchor, lo, hi in read_golden("swa_worked_example.txt"):
        n, w, anchor, lo, hi = map(int, (n, w, anchor, lo, hi))
        spec = _one_head("sliding", w)
        row = dense.dense_mask_strip(spec, 0, n, anchor, anchor + 1)[0]
        assert list(np.nonzero(row)[0]) == list(range(lo, hi + 1))
        got = brute.neighbour_set("sliding", w, n, anchor, list(range(n)))
        assert got == list(range(lo, hi + 1))


def test_column_major_order_hand_written():
    """Column-major walk of a 4x4 grid written out by hand (pins the
    generator's order and the oracle's inverse permutation)."""
    (row,) = read_golden("column_major_4x4.txt")
    perm = np.array([int(x) for x in row])
    assert np.array_equal(column_major_order(4, 4), perm)
    pos = dense.inverse_permutation(perm, 16)
    # raster token 1 (row 0, column 1) is the 5th position of the column walk
    assert pos[1] == 4 and pos[4] == 1 and pos[15] == 15
    assert np.array_equal(perm[pos], np.arange(16))


def _mean_over(v, idx_lo, idx_hi):
    return v[idx_lo:idx_hi + 1].mean(axis=0)


@pytest.mark.parametrize("n", [37, 64])
def test_zero_query_closed_forms(n):
    """With q = 0 every allowed score is 0, so o_i is the plain mean of the
    values over an explicitly sliced key range and lse_i = ln |N(i)|.  The
    slices below are written from the mask definitions, not from the
    oracle's predicate (catches off-by-one bounds, a wrong chunk index or a
    non-causal window)."""
    d = 5
    q = np.zeros((1, 1, n, d))
    k = _rand((1, 1, n, d), 1)
    v = _rand((1, 1, n, d), 2)
    vh = v[0, 0]
    cases = {
        ("sliding", 6): lambda i: (max(0, i - 6), min(n - 1, i + 6)),
        ("chunk", 8): lambda i: (8 * (i // 8), min(n - 1, 8 * (i // 8) + 7)),
        ("causal_window", 5): lambda i: (max(0, i - 4), i),
        ("full", 0): lambda i: (0, n - 1),
    }
    for (kind, param), rng_of in cases.items():
        o, lse = dense.attention(q, k, v, _one_head(kind, param))
        for i in range(n):
            lo, hi = rng_of(i)
            np.testing.assert_allclose(o[0, i], _mean_over(vh, lo, hi), rtol=0, atol=1e-12)
            assert abs(lse[0, i] - math.log(hi - lo + 1)) < 1e-12


def test_zero_query_with_sink_closed_form():
    """q = 0 and a sink b: o_i = sum_{N(i)} v_j / (n_i + e^b), lse = ln(n_i + e^b),
    and the attention row sums to n_i / (n_i + e^b) (SHS slides, Eq. 1)."""
    n, d, w, b = 30, 3, 4, 0.7
    q = np.zeros((1, 1, n, d))
    k = _rand((1, 1, n, d), 3)
    v = _rand((1, 1, n, d), 4)
    spec = _one_head("sliding", w, sink=b)
    o, lse = dense.attention(q, k, v, spec)
    a = dense.attention_probabilities(q, k, spec, 0, 0)
    for i in range(n):
        lo, hi = max(0, i - w), min(n - 1, i + w)
        cnt = hi - lo + 1
        np.testing.assert_allclose(o[0, i], v[0, 0, lo:hi + 1].sum(0) / (cnt + math.exp(b)), atol=1e-12)
        assert abs(lse[0, i] - math.log(cnt + math.exp(b))) < 1e-12
        assert abs(a[i].sum() - cnt / (cnt + math.exp(b))) < 1e-12


def test_two_key_hand_example():
    """One query, two keys, worked by hand: pins the 1/sqrt(d) scale (1/d or
    no scale gives other numbers) and that the sink is compared with the
    scaled scores and carries no value."""
    q = np.zeros((1, 1, 2, 4)); q[0, 0, 0, 0] = 2.0
    k = np.zeros((1, 1, 2, 4)); k[0, 0, 0, 0] = 1.0
    v = np.zeros((1, 1, 2, 4)); v[0, 0, 0, 0] = 1.0; v[0, 0, 1, 1] = 1.0
    for sink, o0, o1, lse in read_golden("two_key_softmax.txt"):
        s = None if sink == "none" else float(sink)
        spec = _one_head("full", 0, sink=s)
        o, l = dense.attention(q, k, v, spec, rows=[0])
        np.testing.assert_allclose(o[0, 0], [float(o0), float(o1), 0, 0], rtol=0, atol=1e-15)
        assert abs(l[0, 0] - float(lse)) < 1e-14


# -- softmax invariants --------------------------------------------------------

@pytest.mark.parametrize("kind,param", [("full", 0), ("chunk", 7), ("sliding", 5),
                                        ("causal_window", 9), ("block", 4)])
def test_rows_sum_to_one(kind, param):
    """Every row of the attention matrix sums to 1 (SHS slides: the row sums
    of the N x N attention matrix; Vision transformers section 2)."""
    n, d = 40, 8
    q = _rand((1, 1, n, d), 5) * 2
    k = _rand((1, 1, n, d), 6) * 2
    blk = bernoulli_causal_blocks(1, (n + 3) // 4, 11)[0] if kind == "block" else None
    a = dense.attention_probabilities(q, k, _one_head(kind, param, block=blk), 0, 0)
    np.testing.assert_allclose(a.sum(1), 1.0, atol=1e-13)
    assert (a >= 0).all()


def test_sink_limits():
    """s_aux -> -inf recovers the plain softmax; s_aux -> +inf sends o -> 0
    (SHS slides, Eq. 1 and the slide after it)."""
    n, d = 24, 6
    q, k, v = (_rand((1, 1, n, d), s) for s in (7, 8, 9))
    o0, l0 = dense.attention(q, k, v, _one_head("sliding", 3))
    o1, l1 = dense.attention(q, k, v, _one_head("sliding", 3, sink=-800.0))
    np.testing.assert_allclose(o1, o0, atol=1e-14)
    np.testing.assert_allclose(l1, l0, atol=1e-14)
    o2, l2 = dense.attention(q, k, v, _one_head("sliding", 3, sink=200.0))
    assert np.abs(o2).max() < 1e-60
    np.testing.assert_allclose(l2, 200.0, atol=1e-12)


# -- structural special cases ----------------------------------------------------

def test_window_at_least_n_is_full_or_causal():
    """A window >= N reproduces full attention (sliding, chunk) or causal
    attention (causal window), and B all-ones with causality is causal
    attention (RRAttention Eq. 2)."""
    n, d = 33, 7
    q, k, v = (_rand((2, 1, n, d), s) for s in (10, 11, 12))
    full = dense.attention(q, k, v, _one_head("full", 0))
    for spec in (_one_head("sliding", n - 1), _one_head("sliding", 5 * n), _one_head("chunk", n)):
        got = dense.attention(q, k, v, spec)
        np.testing.assert_allclose(got[0], full[0], atol=1e-14)
        np.testing.assert_allclose(got[1], full[1], atol=1e-14)
    causal = dense.attention(q, k, v, _one_head("causal_window", n))
    ones = np.ones((9, 9), dtype=bool)
    blk = dense.attention(q, k, v, _one_head("block", 4, block=ones))
    np.testing.assert_allclose(blk[0], causal[0], atol=1e-14)
    # and causal attention row i is the full softmax over the prefix 0..i
    for i in (0, 5, n - 1):
        sub = dense.attention(q[:, :, :i + 1], k[:, :, :i + 1], v[:, :, :i + 1],
                              _one_head("full", 0), rows=[i])
        np.testing.assert_allclose(causal[0][:, i], sub[0][:, 0], atol=1e-14)


def test_chunk_is_independent_softmax_per_chunk():
    """A chunk mask equals a separate full softmax on every chunk (SHS slides,
    chunk window: chunks do not exchange information in the layer)."""
    n, d, c = 40, 5, 8
    q, k, v = (_rand((1, 2, n, d), s) for s in (13, 14, 15))
    o, lse = dense.attention(q, k, v, MaskSpec("chunk", [c, c]))
    for s0 in range(0, n, c):
        sl = slice(s0, s0 + c)
        so, sl_lse = dense.attention(q[:, :, sl], k[:, :, sl], v[:, :, sl], MaskSpec("full", [0, 0]))
        np.testing.assert_allclose(o[:, s0:s0 + c], so, atol=1e-14)
        np.testing.assert_allclose(lse[:, s0:s0 + c], sl_lse, atol=1e-14)


def test_identity_block_matrix_is_blockwise_causal():
    """B = identity keeps only the diagonal blocks: causal attention inside
    each block, independently (RRAttention Eq. 2)."""
    n, d, bs = 24, 4, 6
    q, k, v = (_rand((1, 1, n, d), s) for s in (16, 17, 18))
    o, _ = dense.attention(q, k, v, _one_head("block", bs, block=np.eye(n // bs, dtype=bool)))
    for s0 in range(0, n, bs):
        sl = slice(s0, s0 + bs)
        so, _ = dense.attention(q[:, :, sl], k[:, :, sl], v[:, :, sl], _one_head("causal_window", bs))
        np.testing.assert_allclose(o[:, s0:s0 + bs], so, atol=1e-14)


def test_upper_triangle_bits_contribute_nothing():
    """Bits above the diagonal of B never unmask a pair (Eq. 2 keeps j <= i)."""
    n, d, bs = 20, 3, 4
    q, k, v = (_rand((1, 1, n, d), s) for s in (19, 20, 21))
    low = bernoulli_causal_blocks(1, 5, 3)[0]
    full_bits = low | np.triu(np.ones((5, 5), dtype=bool), 1)
    a = dense.attention(q, k, v, _one_head("block", bs, block=low))
    b = dense.attention(q, k, v, _one_head("block", bs, block=full_bits))
    np.testing.assert_allclose(a[0], b[0], atol=0)


def test_permutation_relabels_tokens():
    """With a token order perm, the output equals un-permuted attention on the
    inputs laid out in sequence order, mapped back to caller order (SHS
    slides, Factor 2: the mask lives on the 1D serialisation)."""
    n, d = 36, 5
    q, k, v = (_rand((1, 1, n, d), s) for s in (22, 23, 24))
    perm = column_major_order(6, 6)
    for kind, param in (("sliding", 4), ("chunk", 6), ("causal_window", 7)):
        o, lse = dense.attention(q, k, v, _one_head(kind, param, perm=perm))
        o2, lse2 = dense.attention(q[:, :, perm], k[:, :, perm], v[:, :, perm], _one_head(kind, param))
        np.testing.assert_allclose(o[0][perm], o2[0], atol=1e-14)
        np.testing.assert_allclose(lse[0][perm], lse2[0], atol=1e-14)


# -- brute force ------------------------------------------------------------------

@pytest.mark.parametrize("n,d", [(5, 3), (12, 4), (16, 8)])
def test_dense_matches_brute_force(n, d):
    """Independent pure-Python enumeration of N(i) and of the softmax, all
    kinds, with and without a permutation and a sink."""
    q, k, v = (_rand((1, 1, n, d), s + 100 * n) for s in (1, 2, 3))
    bs = 3
    nb = (n + bs - 1) // bs
    blk = bernoulli_causal_blocks(1, nb, n)[0]
    perm = random_order(n, n)
    for kind, param in (("full", 0), ("chunk", 4), ("sliding", 2), ("causal_window", 3), ("block", bs)):
        for use_perm in (False, True):
            for sink in (None, 0.3):
                spec = _one_head(kind, param, perm=perm if use_perm else None,
                                 block=blk if kind == "block" else None, sink=sink)
                o, lse = dense.attention(q, k, v, spec)
                bo, blse = brute.attention_head(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(),
                                                kind, param, perm if use_perm else None,
                                                blk if kind == "block" else None, sink)
                np.testing.assert_allclose(o[0], np.array(bo), rtol=0, atol=1e-12)
                np.testing.assert_allclose(lse[0], np.array(blse), rtol=0, atol=1e-12)


def test_empty_rows_defined():
    """A row with no allowed key (a diagonal block left out of B) gets o = 0
    and lse = -inf, or lse = s_aux with a sink (the reading of an empty
    neighbour set)."""
    n, d = 8, 2
    q, k, v = (_rand((1, 1, n, d), s) for s in (31, 32, 33))
    blk = np.zeros((2, 2), dtype=bool); blk[1, 1] = True
    o, lse = dense.attention(q, k, v, _one_head("block", 4, block=blk))
    assert np.all(o[0, :4] == 0) and np.all(np.isneginf(lse[0, :4]))
    o, lse = dense.attention(q, k, v, _one_head("block", 4, block=blk, sink=0.25))
    assert np.all(o[0, :4] == 0) and np.allclose(lse[0, :4], 0.25)
    bo, blse = brute.attention_head(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(),
                                    "block", 4, None, blk, 0.25)
    np.testing.assert_allclose(o[0], np.array(bo), atol=1e-12)


# -- pair counts and tile enumeration -----------------------------------------------

@pytest.mark.parametrize("n", [64, 100, 1000])
def test_pair_count_closed_forms(n):
    """Allowed-pair counts against closed forms: full N^2; chunk C | N: N*C;
    sliding (N > 2w): N(2w+1) - w(w+1); causal window (N >= W):
    N*W - W(W-1)/2; B all-ones: N(N+1)/2."""
    assert dense.pair_count(MaskSpec("full", [0]), n) == n * n
    c = 4 if n % 8 else 8
    assert dense.pair_count(MaskSpec("chunk", [c]), n) == n * c
    w = 13
    assert dense.pair_count(MaskSpec("sliding", [w]), n) == n * (2 * w + 1) - w * (w + 1)
    wc = 17
    assert dense.pair_count(MaskSpec("causal_window", [wc]), n) == n * wc - wc * (wc - 1) // 2
    nb = (n + 15) // 16
    spec = MaskSpec("block", [16], block=np.ones((1, nb, nb), dtype=bool))
    assert dense.pair_count(spec, n) == n * (n + 1) // 2


def test_pair_count_reproduces_printed_attention_flops():
    """The SHS slides' attention-FLOP totals (0.69T / 11.0T / 175.9T full,
    1.68T for 4 full + 28 sliding layers with w = 64) follow from the pair
    counter under the pages' 16 * 1280 FLOPs-per-pair convention.  An
    exclusive or one-sided window gives 1.67T instead of 1.68T."""
    for tokens, n_full, n_swa, w, printed, decimals in read_golden("shs_attention_flops.txt"):
        tokens, n_full, n_swa, w, decimals = map(int, (tokens, n_full, n_swa, w, decimals))
        pairs = n_full * tokens * tokens
        if n_swa:
            pairs += n_swa * dense.pair_count(MaskSpec("sliding", [w]), tokens)
        assert round(16 * 1280 * pairs / 1e12, decimals) == float(printed)


def _brute_tiles(kind, param, n, tile, block=None):
    """Tile enumeration from brute.neighbour_set (pure Python)."""
    nt = (n + tile - 1) // tile
    allowed = [[False] * n for _ in range(n)]
    for p in range(n):
        for j in brute.neighbour_set(kind, param, n, p, list(range(n)), block):
            allowed[p][j] = True
    out = []
    for qt in range(nt):
        for kt in range(nt):
            cells = [allowed[p][j] for p in range(qt * tile, min(n, qt * tile + tile))
                     for j in range(kt * tile, min(n, kt * tile + tile))]
            if any(cells):
                full = len(cells) == tile * tile and all(cells)
                out.append((qt, kt, dense.FULL_TILE if full else dense.PARTIAL_TILE))
    return out


@pytest.mark.parametrize("n", [16, 23, 32])
def test_tile_list_matches_brute_force(n):
    tile = 4
    nb = (n + 2) // 3
    blk = bernoulli_causal_blocks(1, nb, n)[0]
    for kind, param in (("full", 0), ("chunk", 6), ("sliding", 5), ("causal_window", 7), ("block", 3)):
        spec = _one_head(kind, param, block=blk if kind == "block" else None)
        assert dense.tile_list(spec, 0, n, tile) == _brute_tiles(kind, param, n, tile,
                                                                 blk if kind == "block" else None)


def _tile_closed_form_sliding(nt, a):
    """Half-width w = a * T: query tile i visits key tiles i-a..i+a; the inner
    2a-1 of them are FULL, the outer two PARTIAL (clipped to the grid)."""
    full = sum(len(range(max(0, i - a + 1), min(nt - 1, i + a - 1) + 1)) for i in range(nt))
    part = sum((i - a >= 0) + (i + a <= nt - 1) for i in range(nt))
    return full, part


def _tile_closed_form_causal(nt, a):
    """Window W = a * T: query tile i visits i-a..i; i-a+1..i-1 are FULL, the
    diagonal tile and tile i-a (when it exists) PARTIAL."""
    full = sum(len(range(max(0, i - a + 1), i)) for i in range(nt))
    part = sum(1 + (i - a >= 0) for i in range(nt))
    return full, part


@pytest.mark.parametrize("n,kind,param", [(4096, "sliding", 128), (4096, "chunk", 256),
                                          (4096, "causal_window", 512), (4096, "causal_window", 1024),
                                          (4096, "causal_window", 2048), (4096, "causal_window", 4096),
                                          (16384, "sliding", 256), (16384, "chunk", 512)])
def test_tile_counts_closed_forms(n, kind, param):
    """FULL / PARTIAL tile counts (T = 128) at the workloads' sizes against
    the closed forms derived from the window geometry."""
    spec = MaskSpec(kind, [param])
    tiles = dense.tile_list(spec, 0, n, 128)
    nf = sum(1 for t in tiles if t[2] == dense.FULL_TILE)
    npart = len(tiles) - nf
    nt = n // 128
    if kind == "sliding":
        assert (nf, npart) == _tile_closed_form_sliding(nt, param // 128)
    elif kind == "causal_window":
        assert (nf, npart) == _tile_closed_form_causal(nt, param // 128)
    else:
        assert (nf, npart) == (nt * (param // 128), 0)


# -- received attention ------------------------------------------------------

@pytest.mark.parametrize("kind,param", [("full", 0), ("chunk", 8), ("sliding", 5), ("causal_window", 9)])
def test_received_attention_conserves_row_mass(kind, param):
    """Every row of the attention matrix sums to 1 (SHS slides), so the
    column sums add up to N (catches summing rows instead of columns, or a
    missing normalisation)."""
    n = 40
    q, k = _rand((1, 1, n, 6), 1), _rand((1, 1, n, 6), 2)
    r = dense.received_attention(q, k, _one_head(kind, param))[0]
    assert r.sum() == pytest.approx(n, rel=1e-12)
    assert (r >= 0).all()


def test_received_attention_chunks_keep_their_mass():
    """Chunk mask: queries only see their own chunk, so each chunk's columns
    receive exactly C (catches leakage across chunk borders)."""
    n, c = 48, 12
    q, k = _rand((1, 1, n, 5), 3), _rand((1, 1, n, 5), 4)
    r = dense.received_attention(q, k, _one_head("chunk", c))[0]
    np.testing.assert_allclose(r.reshape(n // c, c).sum(axis=1), c, rtol=1e-12)


def test_received_attention_zero_query_closed_forms():
    """q = 0 makes every visible score equal, so a_ij = 1/|N(i)| (plus the
    sink: 1/(|N(i)| + e^b)).  Causal (W >= N): r_j = sum_{i>=j} 1/(i+1) =
    H_N - H_j; sliding w: r_j = sum over |i-j| <= w of 1/|N(i)| with
    |N(i)| = min(n-1, i+w) - max(0, i-w) + 1 counted by hand; the sink share
    is what the columns no longer receive (catches a transposed mask or a
    sink that adds to the columns)."""
    n, w, b = 30, 4, 0.7
    q = np.zeros((1, 1, n, 3))
    k = _rand((1, 1, n, 3), 5)
    r = dense.received_attention(q, k, _one_head("causal_window", n + 5))[0]
    harm = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, n + 1))])
    np.testing.assert_allclose(r, harm[n] - harm[np.arange(n)], rtol=1e-12)
    size = np.array([min(n - 1, i + w) - max(0, i - w) + 1 for i in range(n)], dtype=float)
    want = np.array([sum(1.0 / size[i] for i in range(max(0, j - w), min(n - 1, j + w) + 1)) for j in range(n)])
    np.testing.assert_allclose(dense.received_attention(q, k, _one_head("sliding", w))[0], want, rtol=1e-12)
    want_sink = np.array([sum(1.0 / (size[i] + math.exp(b)) for i in range(max(0, j - w), min(n - 1, j + w) + 1))
                          for j in range(n)])
    np.testing.assert_allclose(dense.received_attention(q, k, _one_head("sliding", w, sink=b))[0], want_sink,
                               rtol=1e-12)


@pytest.mark.parametrize("kind,param", [("full", 0), ("chunk", 4), ("sliding", 3), ("causal_window", 5),
                                        ("block", 4)])
def test_received_attention_matches_brute_force(kind, param):
    """The fp64 column sums against the pure-Python loops, with a token
    order and a sink (catches an ordering slip between positions and tokens)."""
    n = 16
    q, k = _rand((1, 1, n, 4), 6), _rand((1, 1, n, 4), 7)
    perm = np.random.default_rng(8).permutation(n)
    block = None
    if kind == "block":
        block = np.random.default_rng(9).random((n // param, n // param)) < 0.6
        np.fill_diagonal(block, True)
    for pm, sink in ((None, None), (perm, -0.4)):
        spec = _one_head(kind, param, perm=pm, block=block, sink=sink)
        r = dense.received_attention(q, k, spec)[0]
        rb = brute.received_head(q[0, 0].tolist(), k[0, 0].tolist(), kind, param, perm=pm,
                                 block=None if block is None else block.tolist(), sink=sink)
        np.testing.assert_allclose(r, rb, rtol=1e-12, atol=1e-15)


# -- grouped-query attention --------------------------------------------------------

@pytest.mark.parametrize("kind,param", [("full", 0), ("causal_window", 5), ("sliding", 3)])
def test_gqa_equals_mha_with_repeated_kv(kind, param):
    """Grouped-query attention (the Bifocal page: 32 query heads sharing 8
    key/value heads) is multi-head attention whose key/value heads are
    repeated for the consecutive query heads of their group.  Catches a
    wrong head mapping (h % H_kv instead of h // group) or K and V taken
    from different heads."""
    B, H, Hkv, n, d = 2, 6, 2, 19, 4
    q = _rand((B, H, n, d), 1)
    k = _rand((B, Hkv, n, d), 2)
    v = _rand((B, Hkv, n, d), 3)
    spec = MaskSpec(kind, [param] * H, sink=np.linspace(-1.0, 1.0, H))
    o, lse = dense.attention(q, k, v, spec)
    kr, vr = np.repeat(k, H // Hkv, axis=1), np.repeat(v, H // Hkv, axis=1)
    o2, lse2 = dense.attention(q, kr, vr, spec)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    # and head by head against the brute force on the shared key/value head
    for b in range(B):
        for h in range(H):
            bo, blse = brute.attention_head(q[b, h].tolist(), kr[b, h].tolist(), vr[b, h].tolist(), kind, param,
                                            sink=spec.sink[h])
            np.testing.assert_allclose(o[b * H + h], np.array(bo), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b * H + h], np.array(blse), rtol=0, atol=1e-12)


# -- causal window with sink tokens (StreamingLLM) ------------------------------------

def test_sink_token_budget_worked_example():
    """The Bifocal page gives the SWA student with sink tokens a 572-token
    window plus the first 4 tokens, for the same 576 cached tokens per layer
    as the 576-token window of the other student: a query far from the
    start sees exactly 576 keys (catches a window of W + 1 keys, or sink
    tokens counted when the window already covers them)."""
    for n, w, s, p, count, first in read_golden("swa_sink_tokens_budget.txt"):
        n, w, s, p, count, first = map(int, (n, w, s, p, count, first))
        spec = MaskSpec("causal_window", [w], sink_tokens=s)
        row = dense.dense_mask_strip(spec, 0, n, p, p + 1)[0]
        assert int(row.sum()) == count
        keys = np.nonzero(row)[0]
        assert keys[0] == 0 and keys[-1] == p
        assert int(keys[min(s, len(keys) - 1)]) == first  # the first key after the sinks
        got = brute.neighbour_set("causal_window", w, n, p, list(range(n)), sink_tokens=s)
        assert got == list(keys)


@pytest.mark.parametrize("n,w,s", [(64, 9, 3), (200, 50, 4), (300, 128, 40)])
def test_sink_token_pair_count_closed_form(n, w, s):
    """Rows p >= W see W window keys plus min(S, p - W + 1) sink keys below
    the window; rows p < W see all p + 1 keys: pairs = N W - W (W - 1) / 2 +
    S (S + 1) / 2 + S (N - W - S) for N - W >= S."""
    spec = MaskSpec("causal_window", [w], sink_tokens=s)
    expect = n * w - w * (w - 1) // 2 + s * (s + 1) // 2 + s * (n - w - s)
    assert dense.pair_count(spec, n) == expect


def test_sink_tokens_change_nothing_when_the_window_covers_all():
    """W >= N already sees every earlier key (plain causal attention)."""
    n, d = 23, 4
    q, k, v = (_rand((1, 1, n, d), s) for s in (4, 5, 6))
    a = dense.attention(q, k, v, MaskSpec("causal_window", [n], sink_tokens=5))
    b = dense.attention(q, k, v, MaskSpec("causal_window", [n]))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("n,d", [(12, 4), (16, 3)])
def test_sink_tokens_match_brute_force(n, d):
    """Independent enumeration of the window-plus-sinks neighbour sets, with
    and without a permutation and a sink logit."""
    q, k, v = (_rand((1, 1, n, d), s + 7 * n) for s in (1, 2, 3))
    perm = random_order(n, n + 1)
    for w, s in ((3, 2), (4, 5), (1, 1)):
        for use_perm in (False, True):
            for sink in (None, -0.4):
                spec = _one_head("causal_window", w, perm=perm if use_perm else None, sink=sink)
                spec.sink_tokens = s
                o, lse = dense.attention(q, k, v, spec)
                bo, blse = brute.attention_head(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(),
                                                "causal_window", w, perm if use_perm else None, None, sink,
                                                sink_tokens=s)
                np.testing.assert_allclose(o[0], np.array(bo), rtol=0, atol=1e-12)
                np.testing.assert_allclose(lse[0], np.array(blse), rtol=0, atol=1e-12)


# -- decode ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind,param,s", [("full", 0, 0), ("causal_window", 7, 0), ("causal_window", 5, 3)])
def test_decode_is_the_last_row_of_the_forward(kind, param, s):
    """A decode step is the forward's row len - 1 over the first len cached
    tokens, with the new query in that row (catches an off-by-one in the
    query position, a window counted from the cache capacity instead of
    the sequence length, or the wrong key/value head)."""
    B, H, Hkv, L, d = 2, 4, 2, 30, 5
    k = _rand((B, Hkv, L, d), 11)
    v = _rand((B, Hkv, L, d), 12)
    qd = _rand((B, H, d), 13)
    lens = [L, 17]
    spec = MaskSpec(kind, [param] * H, sink=np.array([0.3, -0.2, 1.0, 0.0]), sink_tokens=s)
    o, lse = dense.decode(qd, k, v, lens, spec)
    for b in range(B):
        n = lens[b]
        qf = _rand((1, H, n, d), 14)
        qf[0, :, n - 1] = qd[b]
        fo, flse = dense.attention(qf, k[b:b + 1, :, :n], v[b:b + 1, :, :n], spec, rows=[n - 1])
        np.testing.assert_allclose(o[b], fo[:, 0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], flse[:, 0], rtol=0, atol=1e-13)


def test_decode_empty_sequence():
    """len = 0: no key; o = 0 and lse = -inf, or the sink logit alone."""
    k = _rand((1, 1, 8, 3), 1)
    q = _rand((1, 2, 3), 2)
    o, lse = dense.decode(q, k, k, [0], MaskSpec("full", [0, 0], sink=np.array([-np.inf, 0.7])))
    assert np.all(o == 0)
    assert lse[0, 0] == -np.inf and lse[0, 1] == pytest.approx(0.7)


def test_block2x2_orders_hand_written():
    """The 2x2-block orders (c) and (d) of a 4x4 grid written out by hand
    (pins the generator the tests feed both sides with, and the oracle's
    inverse permutation of it)."""
    from workloads import block2x2_order

    row, col = ([int(x) for x in r] for r in read_golden("block2x2_orders_4x4.txt"))
    assert list(block2x2_order(4, 4)) == row
    assert list(block2x2_order(4, 4, by_columns=True)) == col
    pos = dense.inverse_permutation(np.array(row), 16)
    assert pos[4] == 2 and pos[2] == 4 and pos[15] == 15
    # a sliding window over order (c) keeps the 2x2 block neighbours together
    spec = _one_head("sliding", 1, perm=np.array(row))
    q = np.zeros((1, 1, 16, 2))
    v = np.arange(32, dtype=np.float64).reshape(1, 1, 16, 2)
    o, _ = dense.attention(q, q, v, spec)
    # token 5 sits at position 3, its window holds positions 2..4 = tokens 4, 5, 2
    np.testing.assert_allclose(o[0, 5], v[0, 0, [4, 5, 2]].mean(axis=0))


def test_chunk2d_order_states_what_the_page_states():
    """Order (b), Qwen2.5-VL's chunk windows walked window by window, on the
    page's 4 x 8 grid: the window split, the anchor-15 window (positions
    7..23) and where positions 16-23 land, all as the slide states them; the
    walk inside a window is our reading, pinned only by the hand-written row
    of the golden file."""
    from workloads import chunk2d_order

    lines = {}
    for row in read_golden("chunk2d_order_4x8.txt"):
        lines.setdefault(row[0], []).append(row[1:])
    perm = chunk2d_order(4, 8, 4)
    rows, cols = perm // 8, perm % 8
    for w in lines["window"]:
        p0, p1, c0, c1 = int(w[2]), int(w[3]), int(w[5]), int(w[6])
        assert set(cols[p0:p1 + 1]) == set(range(c0, c1 + 1)) and set(rows[p0:p1 + 1]) == {0, 1, 2, 3}
    a, lo, hi = (int(x) for x in (lines["anchor"][0][0], lines["anchor"][0][2], lines["anchor"][0][3]))
    s0, s1 = (int(x) for x in lines["same_window"][0])
    assert (cols[s0:s1 + 1] < 4).all() and cols[a] < 4
    u = lines["upper_half"][0]
    p0, p1, r0, r1, c0, c1 = int(u[0]), int(u[1]), int(u[3]), int(u[4]), int(u[6]), int(u[7])
    assert set(rows[p0:p1 + 1]) == set(range(r0, r1 + 1)) and set(cols[p0:p1 + 1]) == set(range(c0, c1 + 1))
    assert list(perm) == [int(x) for x in lines["reading"][0]]
    # the oracle's sliding window over this order: the anchor's keys are the
    # tokens at positions 7..23 (q = 0: O is their plain mean)
    spec = _one_head("sliding", 8, perm=perm)
    q = np.zeros((1, 1, 32, 2))
    v = np.arange(64, dtype=np.float64).reshape(1, 1, 32, 2)
    o, lse = dense.attention(q, q, v, spec)
    anchor_token = int(perm[a])
    np.testing.assert_allclose(o[0, anchor_token], v[0, 0, perm[lo:hi + 1]].mean(axis=0))
    np.testing.assert_allclose(lse[0, anchor_token], np.log(hi - lo + 1))
    # and on a real grid the generator is a permutation in windows of win x win
    big = chunk2d_order(64, 64, 8)
    assert np.array_equal(np.sort(big), np.arange(64 * 64))
    assert set(big[:64] // 64) == set(range(8)) and set(big[:64] % 64) == set(range(8))
