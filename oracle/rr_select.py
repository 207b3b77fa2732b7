"""fp64 definition of RRAttention's dynamic block selection (oracle; test
infrastructure only -- see the package docstring).

What it computes ("RRAttention", section 3, Eq. 6-12, and Eq. 5 of
section 2.1), for one head h of a sequence of L tokens with queries Q and
keys K (rows = tokens, d columns), a stride S and a block size Bs:

    P(i, h)  = i S + (S - 1 - (h mod S))                       (Eq. 6)
               one sampled query per stride i = 0 .. L/S - 1   (Eq. 7)
    I_ij     = q_{P(i,h)} . (sum_{k = jS}^{jS+S-1} k_k) / (S sqrt(d))   (Eq. 8)
    P_ij     = exp(I_ij) / sum_{j'} exp(I_ij')                 (Eq. 9)
    S_mn     = sum_{i in block m} sum_{j in block n} P_ij      (Eq. 10)
    Bdyn_mn  = n is among the fewest largest S_m* whose running
               sum reaches tau                                 (Eq. 11)
    B        = Bdyn or Bstatic, Bstatic = all of the last query
               block row                                       (Eq. 12)
    B_mn     = 0 for n > m                                     (Eq. 5)

A stride i belongs to block m = floor(i S / Bs).  Readings of the points the
page leaves open or prints garbled:

1. Eq. 7 lets i run to floor(L/S) inclusive, one past the last stride when
   S divides L; the sampled query of that stride would lie beyond the
   sequence.  Read: i < L/S, one sampled query per stride; L must be a
   multiple of S.
2. Eq. 9's softmax runs over every key stride j' = 0 .. L/S - 1, as
   printed (no stride-level causal mask); causality enters through Eq. 5.
3. Eq. 11 compares the running sum with tau, but a row S_m* sums to the
   number of query strides in block m (Bs/S for a whole block), so an
   absolute tau below 1 would keep a single block.  Read: tau is a fraction
   of the row's total, the kept set is the shortest prefix of the row
   sorted in decreasing order whose sum reaches tau times the row total.
   Equal scores are ordered by the smaller block index first.
4. The round-robin head index is the head's index h in the layer, the same
   for every batch entry.
5. Optional "sink and recent" blocks (Table 5's ablation column: the first
   key block and the diagonal block of every query block) are off unless
   asked for; Table 2's RRAttention rows are the configuration without them.
"""

from __future__ import annotations

import math
from typing import Tuple

import numpy as np


def sampled_positions(L: int, S: int, h: int) -> np.ndarray:
    """Eq. 6-7: the query position sampled in each stride for head h."""
    if L % S:
        raise ValueError("L must be a multiple of the stride S")
    i = np.arange(L // S, dtype=np.int64)
    return i * S + (S - 1 - (h % S))


def stride_key_sums(k: np.ndarray, S: int) -> np.ndarray:
    """The key sum of every stride, sum_{k=jS}^{jS+S-1} K_k (Eq. 8), fp64 [L/S, d]."""
    k = np.asarray(k, dtype=np.float64)
    L, d = k.shape
    return k.reshape(L // S, S, d).sum(axis=1)


def stride_importance(q: np.ndarray, k: np.ndarray, S: int, h: int) -> np.ndarray:
    """Eq. 8: I [L/S, L/S] for one head (q, k: [L, d])."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[1]
    qs = q[sampled_positions(q.shape[0], S, h)]
    return (qs @ stride_key_sums(k, S).T) / (S * math.sqrt(d))


def stride_softmax(I: np.ndarray) -> np.ndarray:
    """Eq. 9: row softmax of I over every key stride."""
    I = np.asarray(I, dtype=np.float64)
    e = np.exp(I - I.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def block_scores(P: np.ndarray, S: int, Bs: int) -> np.ndarray:
    """Eq. 10: S_mn, the sum of P over the strides of query block m and key
    block n; [Nb, Nb] with Nb = ceil(L / Bs)."""
    if Bs % S:
        raise ValueError("the block size must be a multiple of the stride")
    ns = P.shape[0]
    g = Bs // S                       # strides per block
    nb = -(-ns // g)
    blk = np.arange(ns) // g          # block of every stride
    out = np.zeros((nb, nb), dtype=np.float64)
    np.add.at(out, (blk[:, None], blk[None, :]), P)
    return out


def top_tau(row: np.ndarray, tau: float) -> np.ndarray:
    """Eq. 11 for one query block: the shortest prefix of the row sorted in
    decreasing order (equal scores: smaller index first) whose sum reaches
    tau times the row total (reading 3).  Returns a bool mask."""
    row = np.asarray(row, dtype=np.float64)
    order = np.lexsort((np.arange(row.size), -row))   # by -value, then index
    csum = np.cumsum(row[order])
    target = tau * row.sum()
    k = int(np.searchsorted(csum, target, side="left"))  # first prefix reaching it
    k = min(k, row.size - 1)
    keep = np.zeros(row.size, dtype=bool)
    keep[order[:k + 1]] = True
    return keep


def select_head(q: np.ndarray, k: np.ndarray, S: int, Bs: int, tau: float, h: int,
                sink_recent: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """Block-selection matrix B [Nb, Nb] (bool) and block scores S [Nb, Nb]
    of one head (Eq. 6-12 and Eq. 5)."""
    Sblk = block_scores(stride_softmax(stride_importance(q, k, S, h)), S, Bs)
    nb = Sblk.shape[0]
    B = np.zeros((nb, nb), dtype=bool)
    for m in range(nb):
        B[m] = top_tau(Sblk[m], tau)                    # Eq. 11
    B[nb - 1, :] = True                                 # Eq. 12, B_static
    if sink_recent:
        B[:, 0] = True
        B[np.arange(nb), np.arange(nb)] = True
    B &= np.tril(np.ones((nb, nb), dtype=bool))         # Eq. 5
    return B, Sblk


def select(q: np.ndarray, k: np.ndarray, S: int, Bs: int, tau: float,
           sink_recent: bool = False) -> Tuple[np.ndarray, np.ndarray]:
    """All heads: q, k [B, H, L, d] -> (B bool [B, H, Nb, Nb], S fp64 [B, H, Nb, Nb])."""
    q = np.asarray(q)
    k = np.asarray(k)
    nbat, nh = q.shape[:2]
    outs_b, outs_s = [], []
    for b in range(nbat):
        rb, rs = [], []
        for h in range(nh):
            B, Sblk = select_head(q[b, h], k[b, h], S, Bs, tau, h, sink_recent)
            rb.append(B)
            rs.append(Sblk)
        outs_b.append(np.stack(rb))
        outs_s.append(np.stack(rs))
    return np.stack(outs_b), np.stack(outs_s)
