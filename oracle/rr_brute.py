"""Pure-Python loops for RRAttention's block selection, tiny sizes (oracle;
test infrastructure only).

Written independently of ``oracle.rr_select`` (no shared helper), straight
from "RRAttention" section 3: for every head, walk the strides, pick the
sampled query by Eq. 6, add up the stride's keys element by element (Eq. 8),
exponentiate and normalise each row (Eq. 9), add the stride probabilities
into their blocks (Eq. 10), and keep, per query block, the largest blocks
one at a time until the kept share of the row reaches tau (Eq. 11, with the
same readings as ``rr_select``: tau is a share of the row total, equal
scores go smaller index first).  The last query block keeps everything
(Eq. 12) and nothing above the diagonal survives (Eq. 5).
"""

from __future__ import annotations

import math


def select_head(q, k, S, Bs, tau, h, sink_recent=False):
    """q, k: lists of L rows of d floats.  Returns (B, scores) as lists of lists."""
    L = len(q)
    d = len(q[0])
    ns = L // S
    g = Bs // S
    nb = (ns + g - 1) // g
    # Eq. 8 and 9, one sampled query per stride
    prob = []
    for i in range(ns):
        pos = i * S + (S - 1 - (h % S))
        imp = []
        for j in range(ns):
            ksum = [0.0] * d
            for t in range(S):
                for c in range(d):
                    ksum[c] += float(k[j * S + t][c])
            dot = 0.0
            for c in range(d):
                dot += float(q[pos][c]) * ksum[c]
            imp.append(dot / (S * math.sqrt(d)))
        top = max(imp)
        ex = [math.exp(x - top) for x in imp]
        tot = sum(ex)
        prob.append([e / tot for e in ex])
    # Eq. 10
    scores = [[0.0] * nb for _ in range(nb)]
    for i in range(ns):
        for j in range(ns):
            scores[i // g][j // g] += prob[i][j]
    # Eq. 11 and 12, Eq. 5
    B = [[False] * nb for _ in range(nb)]
    for m in range(nb):
        row = scores[m]
        total = sum(row)
        left = list(range(nb))
        kept = 0.0
        while left:
            best = left[0]
            for n in left:
                if row[n] > row[best]:
                    best = n                      # strictly larger only: ties keep the smaller index
            left.remove(best)
            B[m][best] = True
            kept += row[best]
            if kept >= tau * total:
                break
    for n in range(nb):
        B[nb - 1][n] = True
    if sink_recent:
        for m in range(nb):
            B[m][0] = True
            B[m][m] = True
    for m in range(nb):
        for n in range(m + 1, nb):
            B[m][n] = False
    return B, scores
