"""Pins of the RRAttention block-selection oracle (``oracle.rr_select``).

Each test checks the oracle against something other than itself: positions
and selections worked by hand (golden files citing the page), closed forms of
special inputs, invariants the equations imply, and the independent
pure-Python loops of ``oracle.rr_brute``.  The docstring of each test names
the plausible oracle mistake it catches.
"""

import math

import numpy as np
import pytest

from conftest import GOLDEN, read_golden
from oracle import rr_brute, rr_select


def test_sampled_positions_worked_by_hand():
    """Eq. 6 (catches a reversed offset, h instead of h mod S, or a stride off by one)."""
    for L, S, h, *pos in read_golden("rr_sampled_positions.txt"):
        got = rr_select.sampled_positions(int(L), int(S), int(h))
        assert list(got) == [int(x) for x in pos]


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16])
def test_round_robin_covers_every_offset(S):
    """Section 3.1: over S consecutive heads every position of a stride is
    sampled exactly once (catches a sampling offset that ignores h)."""
    L = 8 * S
    for h0 in (0, 3):
        seen = np.concatenate([rr_select.sampled_positions(L, S, h) for h in range(h0, h0 + S)])
        assert sorted(seen) == list(range(L))


def test_importance_of_identical_keys_is_flat():
    """Eq. 8-9 closed form: when every key equals kappa, each stride sum is
    S kappa and I_ij = q_P(i) . kappa / sqrt(d) for every j, so P is uniform
    (catches a missing 1/S, a missing 1/sqrt(d) or a stride sum over the wrong rows)."""
    rng = np.random.default_rng(1)
    L, d, S = 64, 8, 4
    q = rng.standard_normal((L, d))
    kappa = rng.standard_normal(d)
    k = np.tile(kappa, (L, 1))
    for h in range(3):
        I = rr_select.stride_importance(q, k, S, h)
        pos = rr_select.sampled_positions(L, S, h)
        expect = (q[pos] @ kappa) / math.sqrt(d)
        np.testing.assert_allclose(I, np.repeat(expect[:, None], L // S, axis=1), rtol=1e-12, atol=1e-12)
        P = rr_select.stride_softmax(I)
        np.testing.assert_allclose(P, 1.0 / (L // S), rtol=1e-12)


def test_importance_single_stride_of_one_hot_keys():
    """Eq. 8 on a hand-sized case: d = 4, S = 2, the query sampled in stride 0
    of head 0 is row 1; keys are zero except k_2 = (2,0,0,0) and
    k_3 = (0,4,0,0), so stride 1 sums to (2,4,0,0).  With q_1 = (1,1,0,0):
    I_01 = (2 + 4) / (2 * 2) = 1.5 and I_00 = 0 (catches a dot product with a
    single key instead of the stride sum)."""
    L, d, S = 4, 4, 2
    q = np.zeros((L, d))
    q[1] = [1, 1, 0, 0]
    k = np.zeros((L, d))
    k[2] = [2, 0, 0, 0]
    k[3] = [0, 4, 0, 0]
    I = rr_select.stride_importance(q, k, S, 0)
    assert I[0, 0] == 0.0
    assert I[0, 1] == pytest.approx(1.5, abs=1e-15)


def test_stride_softmax_rows_and_shift():
    """Eq. 9: rows sum to 1 and adding a constant to a row changes nothing
    (catches a column-wise normalisation)."""
    rng = np.random.default_rng(2)
    I = rng.standard_normal((12, 12)) * 3
    P = rr_select.stride_softmax(I)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(rr_select.stride_softmax(I + rng.standard_normal((12, 1)) * 50), P, rtol=1e-12)


@pytest.mark.parametrize("L,S,Bs", [(64, 4, 16), (72, 4, 16), (64, 8, 8)])
def test_block_scores_mass(L, S, Bs):
    """Eq. 10: a row of block scores sums to the number of query strides in
    the block (each P row sums to 1) and a uniform P gives S_mn = g_m g_n / (L/S)
    (catches summing over the wrong axis or mis-assigning strides to blocks,
    also with a short last block when Bs does not divide L)."""
    ns, g = L // S, Bs // S
    P = np.full((ns, ns), 1.0 / ns)
    Sb = rr_select.block_scores(P, S, Bs)
    sizes = np.array([min(g, ns - m * g) for m in range(-(-ns // g))], dtype=float)
    np.testing.assert_allclose(Sb.sum(axis=1), sizes, rtol=1e-14)
    np.testing.assert_allclose(Sb, np.outer(sizes, sizes) / ns, rtol=1e-14)


def test_top_tau_worked_by_hand():
    """Eq. 11 on rows worked by hand (catches ascending order, an absolute
    threshold, keeping one block too many or too few, or ties by larger index)."""
    for line in open(GOLDEN + "/rr_top_tau.txt"):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        tau, scores, kept = (x.split() for x in line.split("|"))
        got = rr_select.top_tau(np.array([float(x) for x in scores]), float(tau[0]))
        assert list(np.nonzero(got)[0]) == [int(x) for x in kept]


@pytest.mark.parametrize("sink_recent", [False, True])
def test_static_and_causal_structure(sink_recent):
    """Eq. 12 and Eq. 5: the last query block keeps every key block at or
    below the diagonal, nothing above the diagonal survives; with the sink
    and recent option the first column and the diagonal are kept too."""
    rng = np.random.default_rng(3)
    L, d, S, Bs = 128, 8, 4, 16
    q, k = rng.standard_normal((L, d)), rng.standard_normal((L, d))
    B, _ = rr_select.select_head(q, k, S, Bs, 0.5, 2, sink_recent)
    nb = B.shape[0]
    assert B[nb - 1].all()
    assert not np.triu(B, 1).any()
    if sink_recent:
        assert B[:, 0].all() and np.diag(B).all()


def test_planted_key_stride_is_selected():
    """A key stride aligned with every query takes almost all the mass, so
    each query block keeps exactly that block when it lies at or below the
    diagonal, and only the diagonal-free remainder otherwise (catches a
    selection that ignores the scores)."""
    L, d, S, Bs = 256, 16, 8, 32
    rng = np.random.default_rng(4)
    q = rng.standard_normal((L, d)) * 0.1
    q[:, 0] = 1.0
    k = rng.standard_normal((L, d)) * 0.1
    j_star = 13                                  # stride 13 -> block 13 // 4 = 3
    k[j_star * S:(j_star + 1) * S, 0] = 40.0
    B, Sb = rr_select.select_head(q, k, S, Bs, 0.9, 1)
    n_star = j_star * S // Bs
    nb = B.shape[0]
    for m in range(nb - 1):
        expect = np.zeros(nb, dtype=bool)
        if n_star <= m:
            expect[n_star] = True
        assert (B[m] == expect).all(), m
    assert (Sb[:, n_star] > 0.99 * Sb.sum(axis=1)).all()


@pytest.mark.parametrize("tau,sink_recent", [(0.5, False), (0.9, False), (0.95, True)])
def test_matches_brute_force(tau, sink_recent):
    """The fp64 numpy oracle against the pure-Python loops on tiny heads,
    with a short last block (catches any indexing or ordering slip that the
    special cases above miss)."""
    rng = np.random.default_rng(int(tau * 100))
    L, d, S, Bs = 40, 4, 4, 8
    for h in range(3):
        q = rng.standard_normal((L, d))
        k = rng.standard_normal((L, d))
        B, Sb = rr_select.select_head(q, k, S, Bs, tau, h, sink_recent)
        Bb, Sbb = rr_brute.select_head(q.tolist(), k.tolist(), S, Bs, tau, h, sink_recent)
        np.testing.assert_allclose(Sb, np.array(Sbb), rtol=1e-12, atol=1e-14)
        assert (B == np.array(Bb)).all()


def test_batch_and_heads_are_independent():
    """select() over [B, H] equals select_head per (b, h) with the head's own
    round-robin offset (catches using the batch index as the head index)."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((2, 3, 64, 8))
    k = rng.standard_normal((2, 3, 64, 8))
    B, Sb = rr_select.select(q, k, 4, 16, 0.8)
    for b in range(2):
        for h in range(3):
            Bh, Sh = rr_select.select_head(q[b, h], k[b, h], 4, 16, 0.8, h)
            assert (B[b, h] == Bh).all()
            np.testing.assert_array_equal(Sb[b, h], Sh)
