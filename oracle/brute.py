"""Pure-Python brute force of the masked attention forward, N <= 16 (oracle).

TEST INFRASTRUCTURE ONLY.  Written independently of ``oracle.dense`` (no
shared helper) straight from the neighbour-set definitions, so that it can
pin the dense oracle: for each query it first builds the neighbour set N(i)
as an explicit Python list by walking the keys one by one, then evaluates
the softmax with the sink term over that list with ``math.exp`` (SHS slides:
recap slide for N(i), Eq. 1 for the sink; Vision transformers and hybrid
architectures section 2 for the score q.k / sqrt(d) and the weighted sum).
"""

from __future__ import annotations

import math


def neighbour_set(kind, param, n, pos_i, pos_of_token, block=None, sink_tokens=0):
    """List of caller token indices j that query position ``pos_i`` may see.

    ``sink_tokens`` (causal_window only): positions 0 .. sink_tokens - 1 stay
    visible to every query at or after them (the Bifocal page: a window
    plus the first 4 tokens of the sequence)."""
    out = []
    for j in range(n):
        pj = pos_of_token[j]
        if kind == "full":
            ok = True
        elif kind == "chunk":
            # same chunk of ``param`` consecutive positions
            ok = int(pos_i / param) == int(pj / param)
        elif kind == "sliding":
            # param neighbours to the left and param to the right, plus itself
            ok = pos_i - param <= pj <= pos_i + param
        elif kind == "causal_window":
            # itself and the param - 1 positions before it, and the first
            # sink_tokens positions when they are not after it
            ok = pos_i - param < pj <= pos_i or (pj < sink_tokens and pj <= pos_i)
        elif kind == "block":
            ok = bool(block[pos_i // param][pj // param]) and pj <= pos_i
        else:
            raise ValueError(kind)
        if ok:
            out.append(j)
    return out


def attention_head(q, k, v, kind, param=0, perm=None, block=None, sink=None, sink_tokens=0):
    """One head: q, k, v are lists of lists (n x d).  Returns (o, lse) lists."""
    n = len(q)
    d = len(q[0])
    pos_of_token = list(range(n))
    if perm is not None:
        for p, t in enumerate(perm):
            pos_of_token[int(t)] = p
    o_rows, lses = [], []
    for i in range(n):
        nb = neighbour_set(kind, param, n, pos_of_token[i], pos_of_token, block, sink_tokens)
        scores = []
        for j in nb:
            acc = 0.0
            for c in range(d):
                acc += float(q[i][c]) * float(k[j][c])
            scores.append(acc / math.sqrt(d))
        logits = list(scores) + ([float(sink)] if sink is not None else [])
        if not logits:
            o_rows.append([0.0] * d)
            lses.append(-math.inf)
            continue
        top = max(logits)
        weights = [math.exp(s - top) for s in scores]
        denom = sum(weights) + (math.exp(float(sink) - top) if sink is not None else 0.0)
        row = [0.0] * d
        for w, j in zip(weights, nb):
            for c in range(d):
                row[c] += w * float(v[j][c])
        o_rows.append([x / denom for x in row])
        lses.append(top + math.log(denom))
    return o_rows, lses


def received_head(q, k, kind, param=0, perm=None, block=None, sink=None):
    """Column sums of one head's attention matrix: for each key token j, the
    sum over query tokens i of the weight row i gives j (SHS slides, the
    received-attention slide).  The weights come from the same neighbour
    sets and sink as ``attention_head``; lists in, list out."""
    n = len(q)
    d = len(q[0])
    pos_of_token = list(range(n))
    if perm is not None:
        for p, t in enumerate(perm):
            pos_of_token[int(t)] = p
    received = [0.0] * n
    for i in range(n):
        nb = neighbour_set(kind, param, n, pos_of_token[i], pos_of_token, block)
        scores = []
        for j in nb:
            acc = 0.0
            for c in range(d):
                acc += float(q[i][c]) * float(k[j][c])
            scores.append(acc / math.sqrt(d))
        if not scores and sink is None:
            continue
        logits = list(scores) + ([float(sink)] if sink is not None else [])
        top = max(logits)
        denom = sum(math.exp(s - top) for s in logits)
        for s, j in zip(scores, nb):
            received[j] += math.exp(s - top) / denom
    return received
