"""fp64 definition of the masked attention forward (oracle; test infrastructure).

What it computes, in the pages' notation
----------------------------------------
For one head with queries Q, keys K, values V (rows = tokens, d columns):

    s_ij  = (q_i . k_j) / sqrt(d)                      (Vision transformers and
            hybrid architectures, section 2 "Self-attention from first
            principles": the score and the sqrt(d) scaling)
    a_ij  = exp(s_ij) / (sum_{j' in N(i)} exp(s_ij') + exp(s_aux))
                                                       (SHS slides, the sink
            slide, Eq. 1: one learned logit per head added to the denominator
            only, with no value vector; s_aux = -inf is the plain softmax)
    o_i   = sum_{j in N(i)} a_ij v_j
    lse_i = log(sum_{j in N(i)} exp(s_ij) + exp(s_aux))

N(i), the set of keys query i may see, is where the masks come in (SHS
slides, the local-attention recap slide: the softmax runs over N(i) only).
Every key is scored (step "s" above runs over all N keys) and the mask is
applied elementwise afterwards, as the plain definition reads.

Masks are evaluated on *sequence positions*.  A head may carry a token
permutation perm (perm[p] = caller token index at sequence position p, the
1D serialisation of the 2D patch grid of the SHS slides, "Factor 2"); then
token t sits at position pos(t) = perm^-1(t).  Outputs are returned in
caller (token) order.

Readings of points the pages leave open are listed with each function.
"""

from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

KINDS = ("full", "chunk", "sliding", "causal_window", "block")

FULL_TILE = 1
PARTIAL_TILE = 2


def allowed(kind: str, param: int, p: np.ndarray, q: np.ndarray,
            block_h: Optional[np.ndarray] = None, sink_tokens: int = 0) -> np.ndarray:
    """M(p, q): may the query at position p see the key at position q?

    ``p`` and ``q`` broadcast against each other (integer arrays).

    - full: every key (SHS slides, local-attention recap slide).
    - chunk, C = param: non-overlapping 1D chunks of C tokens, attention only
      inside one's own chunk, a block-diagonal mask (SHS slides, recap slide
      and the "two local attentions" slide).  Reading: bidirectional inside
      the chunk; a short last chunk when N is not a multiple of C.
    - sliding, w = param: each token sees w neighbours on each side, a
      diagonal band (same slides).  Reading: symmetric and inclusive,
      |p - q| <= w, as fixed by the Factor 2 worked example (a +-8 window
      around position 15 covers 7..23).
    - causal_window, W = param: a causal local window of W tokens (Asymmetric
      Attention Heads, "What was done", candidate windows 512..4096 of
      Table 2).  Reading: 0 <= p - q < W, i.e. W keys including the query
      itself, so W >= N is plain causal attention.  With ``sink_tokens`` S
      > 0 the first S positions stay visible as well (the Bifocal page,
      "Comparison at equal memory" and "Details": the SWA student with
      StreamingLLM sink tokens keeps a 572-token window plus the first 4
      tokens of the sequence): M(p, q) = window or (q < S and q <= p).
      Reading: the sink tokens obey causality like every other key.
    - block, B = param: the block-selection matrix expanded to tokens,
      M_B[p, q] = B[floor(p/B), floor(q/B)] and q <= p (RRAttention, section
      2.1, Eq. 1-2).  Reading: block indices are 0-based (Eq. 2 uses floor);
      ``block_h`` is this head's boolean B matrix.
    """
    p = np.asarray(p, dtype=np.int64)
    q = np.asarray(q, dtype=np.int64)
    if kind == "full":
        return np.ones(np.broadcast_shapes(p.shape, q.shape), dtype=bool)
    if kind == "chunk":
        return (p // param) == (q // param)
    if kind == "sliding":
        return np.abs(p - q) <= param
    if kind == "causal_window":
        win = (p - q >= 0) & (p - q < param)
        if sink_tokens > 0:
            win = win | ((q < sink_tokens) & (q <= p))
        return win
    if kind == "block":
        if block_h is None:
            raise ValueError("block mask needs the block-selection matrix")
        bp = p // param
        bq = q // param
        return np.asarray(block_h, dtype=bool)[bp, bq] & (q <= p)
    raise ValueError(f"unknown mask kind {kind!r}")


def inverse_permutation(perm: Optional[np.ndarray], n: int) -> np.ndarray:
    """pos[t] = sequence position of caller token t (identity when perm is None)."""
    if perm is None:
        return np.arange(n, dtype=np.int64)
    perm = np.asarray(perm, dtype=np.int64)
    if perm.shape != (n,) or not np.array_equal(np.sort(perm), np.arange(n)):
        raise ValueError("perm must be a permutation of 0..N-1")
    pos = np.empty(n, dtype=np.int64)
    pos[perm] = np.arange(n, dtype=np.int64)
    return pos


def _head_param(spec, h: int) -> int:
    return int(spec.head_param[h]) if spec.kind != "full" else 0


def _head_block(spec, h: int) -> Optional[np.ndarray]:
    if spec.kind != "block":
        return None
    blk = np.asarray(spec.block, dtype=bool)
    return blk[h] if blk.ndim == 3 else blk


def _head_perm(spec, h: int):
    perms = getattr(spec, "perm", None)
    if perms is None:
        return None
    return perms[h]


def _sink_tokens(spec) -> int:
    return int(getattr(spec, "sink_tokens", 0) or 0)


def _head_sink(spec, h: int) -> Optional[float]:
    sink = getattr(spec, "sink", None)
    if sink is None:
        return None
    return float(np.asarray(sink, dtype=np.float64)[h])


def attention(q, k, v, spec, rows: Optional[Sequence[int]] = None,
              heads: Optional[Iterable[Tuple[int, int]]] = None,
              scale: Optional[float] = None, row_block: int = 256):
    """Masked attention forward in fp64, the plain definition.

    q: array [B, H, N, d]; k, v: arrays [B, H_kv, N, d] with H a multiple
    of H_kv, of any float dtype (upcast exactly to fp64; bf16 and fp32
    values are exact in fp64).  H_kv < H is grouped-query attention (the
    Bifocal page, "Comparison at equal memory": 32 query heads sharing 8
    key/value heads): query head h reads key/value head h // (H / H_kv),
    consecutive query heads forming a group.  ``spec`` describes the mask
    (kind, head_param[h], perm[h], block, sink), per query head.

    ``heads``: iterable of (b, h) pairs to compute (default: all).
    ``rows``: caller token indices to compute for every selected head
    (default: all N).

    Returns (o, lse): o float64 [len(heads), len(rows), d], lse float64
    [len(heads), len(rows)], in the order of ``heads`` and ``rows``.

    Steps, for each head and query row i (SHS slides Eq. 1; RRAttention
    Eq. 1-2; Vision transformers section 2):
      1. s_ij = scale * sum_k Q_ik K_jk over every key j (scale = 1/sqrt(d)).
      2. keep j where M(pos(i), pos(j)) holds; the rest are excluded (the
         "(.) M" of RRAttention Eq. 1 read as exclusion: B = 0 means the
         pair is skipped, and the softmax runs over N(i) only).
      3. m_i = max over kept s_ij and, with a sink, s_aux (the sink is
         compared with the *scaled* scores: it is one more logit).
      4. Z_i = sum_kept exp(s_ij - m_i) + exp(s_aux - m_i).
      5. o_i = sum_kept exp(s_ij - m_i) v_j / Z_i;  lse_i = m_i + ln Z_i.
    A row with no kept key and no sink gets o_i = 0 and lse_i = -inf; with a
    sink only, o_i = 0 and lse_i = s_aux.
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    bsz, nh, n, d = q.shape
    nkv = k.shape[1]
    if nh % nkv or v.shape[1] != nkv:
        raise ValueError("the query head count must be a multiple of the key/value head count")
    group = nh // nkv
    if heads is None:
        heads = [(b, h) for b in range(bsz) for h in range(nh)]
    heads = list(heads)
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o_out = np.zeros((len(heads), len(rows), d), dtype=np.float64)
    lse_out = np.full((len(heads), len(rows)), -np.inf, dtype=np.float64)
    for hi, (b, h) in enumerate(heads):
        kh = np.asarray(k[b, h // group], dtype=np.float64)
        vh = np.asarray(v[b, h // group], dtype=np.float64)
        pos = inverse_permutation(_head_perm(spec, h), n)
        param = _head_param(spec, h)
        blk = _head_block(spec, h)
        sink = _head_sink(spec, h)
        for r0 in range(0, len(rows), row_block):
            r = rows[r0:r0 + row_block]
            qh = np.asarray(q[b, h][r], dtype=np.float64)
            s = scale * (qh @ kh.T)                          # step 1
            keep = allowed(spec.kind, param, pos[r][:, None],
                           pos[None, :], blk, _sink_tokens(spec))  # step 2
            s = np.where(keep, s, -np.inf)
            m = s.max(axis=1)                                # step 3
            if sink is not None:
                m = np.maximum(m, sink)
            finite = np.isfinite(m)
            m_safe = np.where(finite, m, 0.0)
            e = np.exp(s - m_safe[:, None])                  # exp(-inf) = 0
            z = e.sum(axis=1)                                # step 4
            if sink is not None:
                z = z + np.exp(sink - m_safe)
            num = e @ vh                                     # step 5
            with np.errstate(divide="ignore", invalid="ignore"):
                o = np.where(z[:, None] > 0, num / np.where(z > 0, z, 1.0)[:, None], 0.0)
                lse = np.where(z > 0, m_safe + np.log(np.where(z > 0, z, 1.0)), -np.inf)
            o_out[hi, r0:r0 + len(r)] = o
            lse_out[hi, r0:r0 + len(r)] = lse
    return o_out, lse_out


def attention_probabilities(q, k, spec, b: int, h: int,
                            scale: Optional[float] = None) -> np.ndarray:
    """The full N x N attention matrix a_ij of one head (small N only).

    Same steps as ``attention`` without the value product; row i sums to 1
    without a sink and to Z_i / (Z_i + exp(s_aux)) with one (SHS slides:
    every row of the attention matrix sums to 1; the sink absorbs mass).
    """
    q = np.asarray(q[b, h], dtype=np.float64)
    k = np.asarray(k[b, h], dtype=np.float64)
    n, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pos = inverse_permutation(_head_perm(spec, h), n)
    s = scale * (q @ k.T)
    keep = allowed(spec.kind, _head_param(spec, h), pos[:, None], pos[None, :],
                   _head_block(spec, h), _sink_tokens(spec))
    s = np.where(keep, s, -np.inf)
    sink = _head_sink(spec, h)
    m = s.max(axis=1)
    if sink is not None:
        m = np.maximum(m, sink)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m[:, None])
    z = e.sum(axis=1)
    if sink is not None:
        z = z + np.exp(sink - m)
    return np.where(z[:, None] > 0, e / np.where(z > 0, z, 1.0)[:, None], 0.0)


def received_attention(q, k, spec, heads: Optional[Iterable[Tuple[int, int]]] = None,
                       cols: Optional[Sequence[int]] = None,
                       scale: Optional[float] = None, row_block: int = 256):
    """Received attention r_h(j) = sum_i a_ij, the column sums of the
    attention matrix (SHS slides, the "received attention" slide: every row
    of the matrix sums to 1, a column sums to the votes token j receives
    from the queries that may see it).  a_ij is the weight the forward
    gives key j in row i, so with a sink the rows sum to Z_i/(Z_i + exp(s_aux))
    and the sink's share is not received by any token.

    Steps per head: the forward's log-sum-exp lse_i of every row (all N
    rows; ``attention`` above), then r_j = sum over rows i that may see j of
    exp(s_ij - lse_i).  ``cols``: caller token indices to return (default
    all).  Returns float64 [len(heads), len(cols)].
    """
    q = np.asarray(q)
    k = np.asarray(k)
    bsz, nh, n, d = q.shape
    if heads is None:
        heads = [(b, h) for b in range(bsz) for h in range(nh)]
    heads = list(heads)
    cols = np.arange(n) if cols is None else np.asarray(cols, dtype=np.int64)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((len(heads), len(cols)), dtype=np.float64)
    zeros_v = np.zeros((bsz, nh, n, 1))
    for hi, (b, h) in enumerate(heads):
        _, lse = attention(q, k, zeros_v, spec, heads=[(b, h)], scale=scale, row_block=row_block)
        lse = lse[0]
        kh = np.asarray(k[b, h][cols], dtype=np.float64)
        pos = inverse_permutation(_head_perm(spec, h), n)
        param = _head_param(spec, h)
        blk = _head_block(spec, h)
        for r0 in range(0, n, row_block):
            r = np.arange(r0, min(n, r0 + row_block))
            qh = np.asarray(q[b, h][r], dtype=np.float64)
            s = scale * (qh @ kh.T)
            keep = allowed(spec.kind, param, pos[r][:, None], pos[cols][None, :], blk, _sink_tokens(spec))
            fin = np.isfinite(lse[r])[:, None]
            a = np.where(keep & fin, np.exp(np.where(keep, s, 0.0) - np.where(fin, lse[r][:, None], 0.0)), 0.0)
            out[hi] += a.sum(axis=0)
    return out


def dense_mask_strip(spec, h: int, n: int, p0: int, p1: int) -> np.ndarray:
    """Rows p0..p1-1 of the mask M in *position* space, bool [p1-p0, n]."""
    p = np.arange(p0, p1, dtype=np.int64)[:, None]
    qq = np.arange(n, dtype=np.int64)[None, :]
    return allowed(spec.kind, _head_param(spec, h), p, qq, _head_block(spec, h), _sink_tokens(spec))


def tile_list(spec, h: int, n: int, tile: int = 128) -> List[Tuple[int, int, int]]:
    """Enumerate the (query tile, key tile) pairs the mask touches, from the dense mask.

    Tiles are ``tile`` x ``tile`` squares of *position* space.  A tile is
    listed when at least one of its (p, q) pairs with p, q < n is allowed
    (the block-sparse rule of RRAttention section 2.1: B = 0 means the pair
    of blocks is skipped; the same rule applied to any mask).  Its class is
    FULL_TILE (1) when every one of its tile x tile pairs exists (p, q < n)
    and is allowed, else PARTIAL_TILE (2).  Sorted by (query tile, key tile).
    """
    out = []
    nt = (n + tile - 1) // tile
    for qt in range(nt):
        p0, p1 = qt * tile, min(n, (qt + 1) * tile)
        strip = dense_mask_strip(spec, h, n, p0, p1)
        for kt in range(nt):
            sub = strip[:, kt * tile:min(n, (kt + 1) * tile)]
            if not sub.any():
                continue
            complete = (p1 - p0 == tile) and (sub.shape[1] == tile)
            out.append((qt, kt, FULL_TILE if (complete and sub.all()) else PARTIAL_TILE))
    return out


def pair_count(spec, n: int, batch: int = 1, n_heads: Optional[int] = None,
               strip_rows: int = 1024) -> int:
    """Exact number of allowed (query, key) pairs summed over batch and heads.

    This is the unit of the effective-FLOP count (4 d FLOPs per allowed
    pair: one multiply-add per element for q.k and one for a.v).  The count
    does not depend on the permutation (it only relabels tokens).
    """
    nh = n_heads if n_heads is not None else len(spec.head_param)
    total = 0
    for h in range(nh):
        for p0 in range(0, n, strip_rows):
            total += int(dense_mask_strip(spec, h, n, p0, min(n, p0 + strip_rows)).sum())
    return total * batch


def decode(q, k, v, seq_lens, spec, scale: Optional[float] = None):
    """Decode-shaped attention in fp64: one new query per sequence against
    its key/value cache (the Bifocal page, "Details": the speed test reads a
    prompt, then generates one token at a time; 16 query heads share 4
    key/value heads of dimension 256).

    q: [B, H, d], the query of sequence b's newest token, which sits at
    position len_b - 1; k, v: [B, H_kv, L, d] caches whose first len_b rows
    are valid (seq_lens[b] = len_b; None means L).  Query head h reads
    key/value head h // (H / H_kv).  The keys it may see are those of
    ``allowed`` for p = len_b - 1 (full: all len_b keys; causal window W:
    the last W, plus the first ``sink_tokens``), and the softmax with the
    optional sink logit is the one of ``attention``: m = max(kept scores,
    sink), Z = sum exp(s - m) + exp(sink - m), o = sum exp(s - m) v / Z,
    lse = m + ln Z; no kept key and no sink gives o = 0, lse = -inf.
    Returns (o [B, H, d], lse [B, H]) in float64.
    """
    q = np.asarray(q)
    k = np.asarray(k)
    v = np.asarray(v)
    bsz, nh, d = q.shape
    nkv, L = k.shape[1], k.shape[2]
    group = nh // nkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    lens = [L] * bsz if seq_lens is None else [int(x) for x in np.asarray(seq_lens)]
    o_out = np.zeros((bsz, nh, d), dtype=np.float64)
    lse_out = np.full((bsz, nh), -np.inf, dtype=np.float64)
    for b in range(bsz):
        n = max(0, min(L, lens[b]))
        for h in range(nh):
            kh = np.asarray(k[b, h // group, :n], dtype=np.float64)
            vh = np.asarray(v[b, h // group, :n], dtype=np.float64)
            s = scale * (kh @ np.asarray(q[b, h], dtype=np.float64))
            keep = allowed(spec.kind, _head_param(spec, h), np.int64(n - 1), np.arange(n, dtype=np.int64),
                           None, _sink_tokens(spec))
            s = np.where(keep, s, -np.inf)
            sink = _head_sink(spec, h)
            m = s.max() if n else -np.inf
            if sink is not None:
                m = max(m, sink)
            if not np.isfinite(m):
                continue
            e = np.exp(s - m)
            z = e.sum() + (math.exp(sink - m) if sink is not None else 0.0)
            o_out[b, h] = (e @ vh) / z
            lse_out[b, h] = m + math.log(z)
    return o_out, lse_out
