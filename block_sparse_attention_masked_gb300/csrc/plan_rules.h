// Tile-plan rules of the masked attention forward, shared by the host planner
// and the device kernels (so the device visits exactly the tiles the host
// plan lists).
//
// Every mask kind except the block-selection matrix gives each query
// position p one contiguous interval of visible key positions
// [lo(p), hi(p)], with lo and hi non-decreasing in p and p inside it:
//   full            [0, N-1]
//   chunk C         [C*floor(p/C), C*floor(p/C) + C - 1]   (SHS slides, chunk window)
//   sliding w       [p - w, p + w]                          (SHS slides, sliding window;
//                                                            inclusive, Factor 2 example)
//   causal window W [p - W + 1, p]                          (Asymmetric Attention Heads)
// so a 128-row query tile sees the contiguous key-tile range covering
// [lo(first row), hi(last row)], and a key tile is FULL (no masking) when it
// lies inside [lo(last row), hi(first row)] and both tiles are complete.
//
// The block-selection matrix (RRAttention section 2.1, Eq. 1-2) with block
// size Bs = 128*c keeps tile (qt, kt) when B[qt/c][kt/c] is set and kt <= qt
// (Eq. 5 causality); such a tile is FULL when kt < qt and both tiles are
// complete, PARTIAL on the diagonal (q <= p inside the tile).
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define MATTN_HD __host__ __device__ __forceinline__
#else
#define MATTN_HD inline
#endif

namespace mattn {

constexpr int kTile = 128;

enum Kind : int { kFull = 0, kChunk = 1, kSliding = 2, kCausalWindow = 3, kBlockSparse = 4 };
enum TileClass : int { kTileFull = 1, kTilePartial = 2 };

MATTN_HD int64_t floor_div(int64_t a, int64_t b) {
  int64_t q = a / b;
  return (q * b > a) ? q - 1 : q;
}
MATTN_HD int64_t ceil_div(int64_t a, int64_t b) { return -floor_div(-a, b); }
MATTN_HD int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }
MATTN_HD int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

// Visible key interval of query position p (unclipped); block kind: [-inf, p].
MATTN_HD void row_interval(int kind, int64_t param, int64_t n, int64_t p, int64_t* lo, int64_t* hi) {
  switch (kind) {
    case kChunk: {
      int64_t c0 = floor_div(p, param) * param;
      *lo = c0;
      *hi = c0 + param - 1;
      break;
    }
    case kSliding:
      *lo = p - param;
      *hi = p + param;
      break;
    case kCausalWindow:
      *lo = p - param + 1;
      *hi = p;
      break;
    case kBlockSparse:
      *lo = 0;
      *hi = p;
      break;
    default:  // full
      *lo = 0;
      *hi = n - 1;
      break;
  }
}

struct KRange {
  int lo, hi;    // visited key tiles [lo, hi]; empty when lo > hi
  int flo, fhi;  // FULL key tiles [flo, fhi] inside it; none when flo > fhi
};

// Key-tile range of query tile qt for the interval kinds (full, chunk,
// sliding, causal window).
MATTN_HD KRange interval_krange(int kind, int64_t param, int64_t n, int qt) {
  KRange r;
  int64_t p0 = (int64_t)qt * kTile;
  int64_t p1 = imin64(n, p0 + kTile) - 1;
  if (p0 > p1) {
    r.lo = 0; r.hi = -1; r.flo = 0; r.fhi = -1;
    return r;
  }
  int64_t lo0, hi0, lo1, hi1;
  row_interval(kind, param, n, p0, &lo0, &hi0);
  row_interval(kind, param, n, p1, &lo1, &hi1);
  int64_t vlo = imax64(0, lo0), vhi = imin64(n - 1, hi1);
  r.lo = (int)floor_div(vlo, kTile);
  r.hi = (int)floor_div(vhi, kTile);
  // FULL: both tiles complete and every key of the tile inside every row's interval
  bool rows_complete = (p1 - p0 + 1) == kTile;
  int64_t complete_kt_max = n / kTile - 1;  // key tiles with all kTile keys < n
  int64_t flo = ceil_div(imax64(0, lo1), kTile);
  int64_t fhi = floor_div(imin64(n - 1, hi0) + 1, kTile) - 1;
  fhi = imin64(fhi, complete_kt_max);
  flo = imax64(flo, r.lo);
  fhi = imin64(fhi, r.hi);
  if (!rows_complete || flo > fhi) {
    r.flo = 0; r.fhi = -1;
  } else {
    r.flo = (int)flo; r.fhi = (int)fhi;
  }
  return r;
}

// Causal window with sink tokens: a causal window of W keys plus the first
// S tokens of the sequence ("Sliding window attention vs. linear attention
// at equal memory" (Bifocal page), the StreamingLLM sink-token student: a
// 572-token window plus the first 4 tokens).  Row p sees [p - W + 1, p]
// and [0, min(S - 1, p)].  The window part is interval_krange's
// kCausalWindow range; the sink keys add the leading key tiles
// [0, sink_tiles) to a query tile's list.

// Last sink key visible to row p (-1: none).
MATTN_HD int64_t sink_last(int64_t s, int64_t p) { return s > 0 ? imin64(s - 1, p) : -1; }

// Leading key tiles holding sink keys that some row of query tile qt sees.
MATTN_HD int sink_tiles(int64_t s, int64_t n, int qt) {
  const int64_t p0 = (int64_t)qt * kTile;
  const int64_t p1 = imin64(n, p0 + kTile) - 1;
  if (s <= 0 || p0 > p1) return 0;
  const int64_t last = imin64(imin64(s - 1, p1), n - 1);  // the last row sees the most
  return (int)(last / kTile) + 1;
}

// Exact class of a visited key tile kt of query tile qt: FULL when every
// (p, q) of the two complete tiles is visible.  Every row must see the
// tile's last key (causality: p0 >= k1), and the last row's window must
// start at or before the first key of the tile that no sink covers (none
// when the whole tile is sink keys).
MATTN_HD int sink_window_tile_class(int64_t w, int64_t s, int64_t n, int qt, int kt) {
  const int64_t p0 = (int64_t)qt * kTile, k0 = (int64_t)kt * kTile;
  const int64_t p1 = p0 + kTile - 1, k1 = k0 + kTile - 1;
  if (p1 > n - 1 || k1 > n - 1) return kTilePartial;  // incomplete tile
  if (p0 < k1) return kTilePartial;
  if (k1 >= s) {
    const int64_t e = k0 >= s ? k0 : s;  // first key of the tile outside the sink
    if (p1 - w + 1 > e) return kTilePartial;
  }
  return kTileFull;
}

// Key-tile list of a CTA whose two query sub-tiles take the window ranges
// [lo0, hi0] and [lo1, hi1] (empty when lo > hi; the ranges of neighbouring
// query tiles overlap or touch) plus the sink tiles [0, ns0) and [0, ns1):
// entry j < na is sink tile j, entry j >= na is key tile lo + j - na, n
// entries in all.  The sink tiles form a segment before the window's tiles,
// or one segment with them when they meet.
MATTN_HD void pair_list_span(int lo0, int hi0, int lo1, int hi1, int ns0, int ns1, int* lo, int* n, int* na) {
  const bool e0 = lo0 <= hi0, e1 = lo1 <= hi1;
  *lo = e0 ? (e1 ? (lo0 < lo1 ? lo0 : lo1) : lo0) : lo1;
  int hi = e0 ? (e1 ? (hi0 > hi1 ? hi0 : hi1) : hi0) : hi1;
  *n = (e0 || e1) ? hi - *lo + 1 : 0;
  *na = 0;
  const int ns = ns0 > ns1 ? ns0 : ns1;
  if (ns > 0 && *n > 0) {
    if (ns >= *lo) {
      hi = hi > ns - 1 ? hi : ns - 1;
      *lo = 0;
      *n = hi + 1;
    } else {
      *na = ns;
      *n += ns;
    }
  }
}

// Block-selection bit B[m][nblk] of one head's bitmap (words per row = wpr).
MATTN_HD bool block_bit(const uint64_t* bits, int wpr, int m, int nblk) {
  return (bits[(int64_t)m * wpr + (nblk >> 6)] >> (nblk & 63)) & 1ull;
}

MATTN_HD bool block_row_bit(const uint64_t* row, int nblk) { return (row[nblk >> 6] >> (nblk & 63)) & 1ull; }

// Smallest kept key tile kt >= from with kt <= ktmax in one bitmap row of a
// block-sparse head (Bs = 128*c); returns INT32_MAX when there is none.
MATTN_HD int block_row_next_kt(const uint64_t* row, int c, int from, int ktmax) {
  if (from < 0) from = 0;
  if (from > ktmax) return 0x7fffffff;
  int nb0 = from / c;
  if ((row[nb0 >> 6] >> (nb0 & 63)) & 1ull) return from;
  int nb = nb0 + 1;
  int nbmax = ktmax / c;
  while (nb <= nbmax) {
    uint64_t w = row[nb >> 6] >> (nb & 63);
    if (w) {
#ifdef __CUDA_ARCH__
      nb += __ffsll((long long)w) - 1;
#else
      nb += __builtin_ctzll(w);
#endif
      break;
    }
    nb = (nb | 63) + 1;
  }
  if (nb > nbmax) return 0x7fffffff;
  int kt = nb * c;
  return kt <= ktmax ? kt : 0x7fffffff;
}

// The same for query tile qt of a head whose bitmap starts at `bits`.
MATTN_HD int block_next_kt(const uint64_t* bits, int wpr, int c, int qt, int from, int ktmax) {
  return block_row_next_kt(bits + (int64_t)(qt / c) * wpr, c, from, ktmax);
}

MATTN_HD int block_tile_class(int qt, int kt, int64_t n) {
  bool complete = ((int64_t)(qt + 1) * kTile <= n) && ((int64_t)(kt + 1) * kTile <= n);
  return (kt < qt && complete) ? kTileFull : kTilePartial;
}

MATTN_HD int interval_tile_class(const KRange& r, int kt) {
  return (kt >= r.flo && kt <= r.fhi) ? kTileFull : kTilePartial;
}

}  // namespace mattn
