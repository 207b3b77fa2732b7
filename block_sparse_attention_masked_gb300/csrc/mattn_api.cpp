// Host side of libmattn: argument validation, the tile planner and work
// list, per-device state, TMA descriptors and kernel launches behind the C
// ABI declared in include/mattn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <queue>
#include <string>
#include <vector>

#include "kernel_params.h"
#include "launch_prep.h"
#include "mattn.h"
#include "plan_rules.h"

namespace mattn {
namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MATTN_CUDA(call, what)                   \
  do {                                           \
    cudaError_t e_ = (call);                     \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

std::atomic<unsigned long long> g_timeout_ns{0};
// Test hook: an upper bound on the persistent kernel's grid (0 = one CTA per
// SM), so that small problems still give each CTA many work items.
std::atomic<int> g_persist_grid_cap{0};
// Test hook: which persistent items are split (0: the load rule of
// split_persist_items; 1: every item whose query tiles have two or more key
// tiles; -1: none).
std::atomic<int> g_persist_split{0};
// Debug library test hook: a defect planted in the next forward launch's
// plan (kCorrupt*), consumed by that launch.
enum DebugCorruption : int {
  kCorruptNone = 0,
  kCorruptItemHead = 1,     // the first work item names head row B*H (one past the last)
  kCorruptKeyTiles = 2,     // persistent: the first item's key-tile window starts past the last key tile
  kCorruptGridRows = 3,     // the kernel is told half the grid rows (column-major heads read through TMA)
};
std::atomic<int> g_debug_corrupt{kCorruptNone};

unsigned long long wait_timeout_ns() {
  unsigned long long t = g_timeout_ns.load();
  if (t) return t;
  const char* env = getenv("MATTN_WAIT_TIMEOUT_NS");
  unsigned long long v = env ? strtoull(env, nullptr, 10) : 0ull;
  if (!v) v = 2000000000ull;
  g_timeout_ns.store(v);
  return v;
}

// ------------------------------------------------------------ mask normalisation
struct HeadPlan {
  int param;
  int load;   // LoadMode
  int store;  // StoreMode
  int perm_row;
};

struct Normalized {
  int kind;
  int B, H, N, d, dtype;
  std::vector<HeadPlan> heads;
  bool need_copy;     // reorder / convert into a bf16 copy in position order
  bool any_colmajor_tma;
  bool any_block_tma;      // some head reads the 2x2-block row-major order through 5D TMA views
  bool any_block_col_tma;  // some head reads the 2x2-block column-major order through 5D TMA views
  int block_c, block_nb, block_wpr, block_heads;
  int sink_tokens;    // causal window: leading positions every later query sees
  float scale;
  bool split;         // schedule: one query tile per CTA, key tiles dealt to two pipelines
  bool single;        // the single-pipeline kernel (head dim 256, or 128 on request)
  bool persistent;    // the persistent kernel (interval masks, paired work items)
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Average key tiles per query tile up to which an interval mask runs on the
// persistent kernel by default.  Measured on GB300 with the items assigned
// longest first: windows of 3-7 tiles 1.2-1.6x faster persistent, head-wise
// windows of 5-33 tiles (17 on average) and 32-tile full masks 0-4% faster,
// 128-tile full masks 1.5% slower.
constexpr double kPersistMaxTiles = 40.0;

// allow_block_tma: the caller's kernel reads the 2x2-block row-major order
// through its 5D TMA views (the attention forward); otherwise such heads go
// through the reorder copy.
int normalize(const mattn_mask_desc* desc, int B, int H, int N, int d, int dtype, bool need_data, Normalized* out,
              bool allow_block_tma = true) {
  if (!desc) return fail(MATTN_ERR_INVALID_ARG, "mask descriptor is NULL");
  if (desc->flags != 0 && desc->flags != MATTN_FLAG_SCHEDULE_PAIRED && desc->flags != MATTN_FLAG_SCHEDULE_SPLIT &&
      desc->flags != MATTN_FLAG_SCHEDULE_SINGLE && desc->flags != MATTN_FLAG_SCHEDULE_PERSISTENT)
    return fail(MATTN_ERR_INVALID_ARG, "flags must be 0 or one MATTN_FLAG_SCHEDULE_* flag (got %u)",
                desc->flags);
  if (B < 1 || H < 1 || N < 1) return fail(MATTN_ERR_INVALID_ARG, "B, H, N must be >= 1 (got %d, %d, %d)", B, H, N);
  if (N > (1 << 30)) return fail(MATTN_ERR_UNSUPPORTED, "N = %d exceeds 2^30", N);
  if ((int64_t)B * H > (1 << 30)) return fail(MATTN_ERR_UNSUPPORTED, "B*H too large");
  if (need_data) {
    if (d != 32 && d != 64 && d != 80 && d != 96 && d != 128 && d != 256)
      return fail(MATTN_ERR_UNSUPPORTED, "head dim %d not supported (32, 64, 80, 96, 128, 256)", d);
    if (dtype != MATTN_BF16 && dtype != MATTN_F32) return fail(MATTN_ERR_UNSUPPORTED, "dtype %d not supported", dtype);
  }
  if (desc->kind < MATTN_FULL || desc->kind > MATTN_BLOCK_SPARSE)
    return fail(MATTN_ERR_INVALID_ARG, "unknown mask kind %d", desc->kind);
  if (!(desc->softmax_scale >= 0.f) || std::isinf(desc->softmax_scale))
    return fail(MATTN_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
  Normalized n;
  n.kind = desc->kind;
  n.B = B; n.H = H; n.N = N; n.d = d; n.dtype = dtype;
  n.scale = desc->softmax_scale > 0.f ? desc->softmax_scale : (d > 0 ? 1.0f / std::sqrt((float)d) : 1.0f);
  n.heads.resize(H);
  n.need_copy = need_data && dtype == MATTN_F32;
  n.any_colmajor_tma = false;
  n.block_c = n.block_nb = n.block_wpr = 0;
  n.block_heads = 1;
  if (desc->sink_tokens < 0) return fail(MATTN_ERR_INVALID_ARG, "sink_tokens must be >= 0 (got %d)", desc->sink_tokens);
  if (desc->sink_tokens > 0 && desc->kind != MATTN_CAUSAL_WINDOW)
    return fail(MATTN_ERR_INVALID_ARG, "sink_tokens applies to MATTN_CAUSAL_WINDOW masks only");
  n.sink_tokens = desc->sink_tokens;
  for (int h = 0; h < H; ++h) {
    int prm = desc->head_param ? desc->head_param[h] : desc->param;
    if (n.kind != MATTN_FULL && prm < 1)
      return fail(MATTN_ERR_INVALID_ARG, "mask parameter of head %d must be >= 1 (got %d)", h, prm);
    if (n.kind == MATTN_FULL) prm = 0;
    n.heads[h].param = prm;
    int order = desc->head_order ? desc->head_order[h] : MATTN_ORDER_RASTER;
    n.heads[h].perm_row = -1;
    if (order == MATTN_ORDER_RASTER) {
      n.heads[h].load = kLoadRaster;
      n.heads[h].store = kStoreIdentity;
    } else if (order == MATTN_ORDER_COLUMN_MAJOR) {
      if (desc->grid_rows < 1 || desc->grid_cols < 1 || (int64_t)desc->grid_rows * desc->grid_cols != N)
        return fail(MATTN_ERR_INVALID_ARG, "column-major order needs grid_rows * grid_cols == N (%d x %d vs %d)",
                    desc->grid_rows, desc->grid_cols, N);
      n.heads[h].store = kStoreColumnMajor;
      if (desc->grid_rows % kTile == 0) {
        n.heads[h].load = kLoadColumnMajor;
      } else {
        n.heads[h].load = kLoadRaster;
        n.need_copy = true;
      }
    } else if (order == MATTN_ORDER_BLOCK2X2_ROW || order == MATTN_ORDER_BLOCK2X2_COL) {
      if (desc->grid_rows < 2 || desc->grid_cols < 2 || (int64_t)desc->grid_rows * desc->grid_cols != N ||
          (desc->grid_rows & 1) || (desc->grid_cols & 1))
        return fail(MATTN_ERR_INVALID_ARG,
                    "2x2-block orders need an even grid with grid_rows * grid_cols == N (%d x %d vs %d)",
                    desc->grid_rows, desc->grid_cols, N);
      const bool row = order == MATTN_ORDER_BLOCK2X2_ROW;
      n.heads[h].store = row ? kStoreBlock2x2Row : kStoreBlock2x2Col;
      // a 128-position tile is 32 blocks of one block row when cols % 64 == 0
      // (row order), of one block column when rows % 64 == 0 (column order)
      if (allow_block_tma && (row ? desc->grid_cols : desc->grid_rows) % 64 == 0) {
        n.heads[h].load = row ? kLoadBlock2x2Row : kLoadBlock2x2Col;
      } else {
        n.heads[h].load = kLoadRaster;
        n.need_copy = true;
      }
    } else if (order >= 0) {
      if (!desc->perm || order >= desc->n_perm)
        return fail(MATTN_ERR_INVALID_ARG, "head %d selects explicit order %d but n_perm = %d", h, order, desc->n_perm);
      n.heads[h].load = kLoadRaster;
      n.heads[h].store = kStoreExplicit;
      n.heads[h].perm_row = order;
      n.need_copy = true;
    } else {
      return fail(MATTN_ERR_INVALID_ARG, "head %d has invalid order code %d", h, order);
    }
  }
  n.any_block_tma = false;
  n.any_block_col_tma = false;
  if (n.need_copy) {
    for (auto& hp : n.heads) hp.load = kLoadRaster;  // the copy is already in position order
  } else {
    for (auto& hp : n.heads) {
      n.any_colmajor_tma |= hp.load == kLoadColumnMajor;
      n.any_block_tma |= hp.load == kLoadBlock2x2Row;
      n.any_block_col_tma |= hp.load == kLoadBlock2x2Col;
    }
  }
  if (n.kind == MATTN_BLOCK_SPARSE) {
    const int bs = n.heads[0].param;
    for (int h = 1; h < H; ++h)
      if (n.heads[h].param != bs) return fail(MATTN_ERR_UNSUPPORTED, "block size must be the same for every head");
    if (bs % kTile != 0) return fail(MATTN_ERR_UNSUPPORTED, "block size %d is not a multiple of %d", bs, kTile);
    if ((N + kTile - 1) / kTile > kBlockListMax)
      return fail(MATTN_ERR_UNSUPPORTED, "block-sparse masks support N <= %d (got %d)", kBlockListMax * kTile, N);
    if (!desc->block_bits) return fail(MATTN_ERR_INVALID_ARG, "block-sparse mask without block_bits");
    if (desc->block_heads != 1 && desc->block_heads != H)
      return fail(MATTN_ERR_INVALID_ARG, "block_heads must be 1 or H (got %d)", desc->block_heads);
    n.block_c = bs / kTile;
    n.block_nb = (N + bs - 1) / bs;
    n.block_wpr = (n.block_nb + 63) / 64;
    n.block_heads = desc->block_heads;
  }
  // Schedule: SPLIT when neighbouring query tiles share few key tiles (block
  // rows of one tile: independent rows of the block matrix), else PAIRED.
  n.split = n.kind == kBlockSparse && n.block_c == 1;
  if (desc->flags == MATTN_FLAG_SCHEDULE_PAIRED) n.split = false;
  if (desc->flags == MATTN_FLAG_SCHEDULE_SPLIT) n.split = true;
  n.single = false;
  if (need_data && desc->flags == MATTN_FLAG_SCHEDULE_SINGLE && d != 128 && d != 256)
    return fail(MATTN_ERR_UNSUPPORTED, "the single-pipeline schedule takes head dim 128 or 256 (got %d)", d);
  if (need_data && (d == 256 || desc->flags == MATTN_FLAG_SCHEDULE_SINGLE)) {
    // the single-pipeline kernel: one query tile per work item, inputs in
    // raster order (other orders through the reorder copy)
    n.single = true;
    for (const auto& hp : n.heads)
      if (hp.store != kStoreIdentity) n.need_copy = true;
    for (auto& hp : n.heads) hp.load = kLoadRaster;
    n.any_colmajor_tma = false;
    n.any_block_tma = false;
    n.any_block_col_tma = false;
    n.split = true;
  }
  // The persistent kernel: interval masks at head dim <= 128 (paired work
  // items).  Without a schedule flag it is chosen when a query tile's
  // key-tile list is short on average (at most kPersistMaxTiles): there the
  // one-item-per-CTA kernel spends much of its time in per-CTA set-up and
  // epilogue, which the persistent kernel overlaps with neighbouring items;
  // on long lists the hardware's dynamic CTA scheduling balances better.
  n.persistent = false;
  if (need_data && desc->flags == 0 && n.kind != kBlockSparse && !n.single && d <= 128) {
    const int64_t nt = ((int64_t)N + kTile - 1) / kTile;
    double tiles = 0.0;
    for (const auto& hp : n.heads) {
      const double w = (double)std::min<int64_t>(hp.param, N);
      double t;
      switch (n.kind) {
        case kChunk: t = w / kTile + 1.0; break;
        case kSliding: t = (2.0 * w + kTile) / kTile + 1.0; break;
        case kCausalWindow: t = w / kTile + 1.0 + (n.sink_tokens > 0 ? 1.0 : 0.0); break;
        default: t = (double)nt; break;
      }
      tiles += std::min<double>(t, (double)nt);
    }
    n.persistent = tiles / H <= kPersistMaxTiles;
  }
  if (desc->flags == MATTN_FLAG_SCHEDULE_PERSISTENT) {
    if (n.kind == kBlockSparse)
      return fail(MATTN_ERR_UNSUPPORTED, "the persistent schedule takes the interval masks (not block-sparse)");
    if (need_data && d > 128)
      return fail(MATTN_ERR_UNSUPPORTED, "the persistent schedule takes head dim <= 128 (got %d)", d);
    n.persistent = need_data;
    n.split = false;
  }
  *out = std::move(n);
  return MATTN_OK;
}

// Whether no key tile of the launch is PARTIAL for any query tile: full
// masks, and chunks that are multiples of the tile (or cover the sequence),
// on a sequence length that is a multiple of the tile.  Every other kind has
// PARTIAL tiles (windows' edges, causal diagonals, sink columns).
bool launch_has_no_partial(const Normalized& n) {
  if (n.N % kTile != 0) return false;
  if (n.kind == kFull) return true;
  if (n.kind != kChunk) return false;
  for (const auto& hp : n.heads)
    if (hp.param % kTile != 0 && hp.param < n.N) return false;
  return true;
}

// ------------------------------------------------------------ planning (host)
template <typename Fn>
void walk_tiles_host(const Normalized& n, const uint64_t* host_bits, int h, int qt, Fn&& fn) {
  if (n.kind == kBlockSparse) {
    const uint64_t* bits = host_bits + (int64_t)((n.block_heads == 1) ? 0 : h) * n.block_nb * n.block_wpr;
    for (int kt = block_next_kt(bits, n.block_wpr, n.block_c, qt, 0, qt); kt != 0x7fffffff;
         kt = block_next_kt(bits, n.block_wpr, n.block_c, qt, kt + 1, qt))
      fn(kt, block_tile_class(qt, kt, n.N));
  } else if (n.sink_tokens > 0) {
    // the sink tiles below the window, then the window's tiles
    const int w = n.heads[h].param;
    KRange r = interval_krange(n.kind, w, n.N, qt);
    const int ns = sink_tiles(n.sink_tokens, n.N, qt);
    for (int kt = 0; kt < ns && kt < r.lo; ++kt) fn(kt, sink_window_tile_class(w, n.sink_tokens, n.N, qt, kt));
    for (int kt = r.lo; kt <= r.hi; ++kt) fn(kt, sink_window_tile_class(w, n.sink_tokens, n.N, qt, kt));
  } else {
    KRange r = interval_krange(n.kind, n.heads[h].param, n.N, qt);
    for (int kt = r.lo; kt <= r.hi; ++kt) fn(kt, interval_tile_class(r, kt));
  }
}

int interval_tiles(const Normalized& n, int h, int qt) {
  if (qt * (int64_t)kTile >= n.N) return 0;
  KRange r = interval_krange(n.kind, n.heads[h].param, n.N, qt);
  const int win = r.hi >= r.lo ? r.hi - r.lo + 1 : 0;
  const int ns = sink_tiles(n.sink_tokens, n.N, qt);
  return win + (ns < r.lo ? ns : r.lo);  // sink tiles below the window
}

// Work list: one item per (b*H + h, query-tile pair), or per (b*H + h,
// query tile) under the split schedule.
std::vector<int2> build_items(const Normalized& n) {
  const int nt = (n.N + kTile - 1) / kTile;
  const int npairs = n.split ? nt : (nt + 1) / 2;  // work units per (b, h)
  std::vector<int2> items;
  items.reserve((size_t)n.B * n.H * npairs);
  if (n.kind == kBlockSparse) {
    // Head by head, and inside a head the later query tiles (more key tiles
    // under causality) first.  The CTAs in flight then share one head's K
    // and V, which fit in L2, instead of streaming every head's at once; the
    // lightest tiles of the last head end the launch.
    for (int bh = 0; bh < n.B * n.H; ++bh)
      for (int pr = npairs - 1; pr >= 0; --pr) items.push_back(make_int2(bh, pr));
  } else {
    for (int bh = 0; bh < n.B * n.H; ++bh)
      for (int pr = 0; pr < npairs; ++pr) items.push_back(make_int2(bh, pr));
    std::vector<int> cost((size_t)n.H * npairs);
    for (int h = 0; h < n.H; ++h)
      for (int pr = 0; pr < npairs; ++pr)
        cost[(size_t)h * npairs + pr] = n.split ? interval_tiles(n, h, pr)
                                                : interval_tiles(n, h, 2 * pr) + interval_tiles(n, h, 2 * pr + 1);
    const int H = n.H;
    std::stable_sort(items.begin(), items.end(), [&](const int2& a, const int2& b) {
      return cost[(size_t)(a.x % H) * npairs + a.y] > cost[(size_t)(b.x % H) * npairs + b.y];
    });
  }
  return items;
}

// Descriptors of the persistent kernel's work items (paired items of an
// interval mask): each item's key-tile plan from plan_rules.h, in the
// layout kPersistItemInt4 documents, so that no role of the kernel divides.
std::vector<int4> build_persist_items(const Normalized& n, const std::vector<int2>& items) {
  const int nt = (n.N + kTile - 1) / kTile;
  std::vector<int4> out(items.size() * kPersistItemInt4);
  for (size_t i = 0; i < items.size(); ++i) {
    const int bh = items[i].x, h = bh % n.H, b = bh / n.H, qt0 = 2 * items[i].y;
    const HeadPlan& hp = n.heads[h];
    KRange r[2];
    int ns[2];
    for (int s = 0; s < 2; ++s) {
      const int qt = qt0 + s;
      if (qt < nt) {
        r[s] = interval_krange(n.kind, hp.param, n.N, qt);
        ns[s] = sink_tiles(n.sink_tokens, n.N, qt);
      } else {
        r[s].lo = 1; r[s].hi = 0; r[s].flo = 0; r[s].fhi = -1;  // no rows
        ns[s] = 0;
      }
    }
    int lo, cnt, na;
    pair_list_span(r[0].lo, r[0].hi, r[1].lo, r[1].hi, ns[0], ns[1], &lo, &cnt, &na);
    int first[2] = {-1, -1}, last[2] = {-1, -1};
    for (int j = 0; j < cnt; ++j) {
      const int kt = j < na ? j : lo + j - na;
      for (int s = 0; s < 2; ++s) {
        if ((kt >= r[s].lo && kt <= r[s].hi) || kt < ns[s]) {
          if (first[s] < 0) first[s] = j;
          last[s] = j;
        }
      }
    }
    int4* d = &out[i * kPersistItemInt4];
    d[0] = make_int4(bh, h, b, qt0);
    d[1] = make_int4(cnt, lo, na, hp.param);
    d[2] = make_int4(r[0].lo, r[0].hi, r[1].lo, r[1].hi);
    d[3] = make_int4(r[0].flo, r[0].fhi, r[1].flo, r[1].fhi);
    d[4] = make_int4(ns[0], ns[1], hp.load | (hp.store << 8), hp.perm_row);
    d[5] = make_int4(first[0], last[0], first[1], last[1]);
  }
  return out;
}

// The split item of query tile qt of row block bh (layout kPersistItemInt4):
// the query tile's own key tiles, entry j multiplied by sub-tile j % 2.
void make_split_item(const Normalized& n, int bh, int qt, int4* d) {
  const int h = bh % n.H, b = bh / n.H;
  const HeadPlan& hp = n.heads[h];
  const KRange r = interval_krange(n.kind, hp.param, n.N, qt);
  const int ns = sink_tiles(n.sink_tokens, n.N, qt);
  int lo, cnt, na;
  pair_list_span(r.lo, r.hi, r.lo, r.hi, ns, ns, &lo, &cnt, &na);
  d[0] = make_int4(bh, h, b, qt);
  d[1] = make_int4(cnt, lo, na, hp.param);
  d[2] = make_int4(r.lo, r.hi, r.lo, r.hi);
  d[3] = make_int4(r.flo, r.fhi, r.flo, r.fhi);
  d[4] = make_int4(ns, ns, hp.load | (hp.store << 8) | (1 << 16), hp.perm_row);
  const int last0 = cnt >= 1 ? ((cnt - 1) & ~1) : -1;
  const int last1 = cnt >= 2 ? ((cnt - 1) % 2 == 1 ? cnt - 1 : cnt - 2) : -1;
  d[5] = make_int4(cnt >= 1 ? 0 : -1, last0, cnt >= 2 ? 1 : -1, last1);
}

// Fixed share of an item's load for its set-up and output, in tile products.
constexpr int kItemOverheadTiles = 4;

// An item's load for the work assignment: the tile products its sub-tiles
// multiply plus kItemOverheadTiles.  Both sub-tiles run side by side, so a
// paired item takes about max(t0, t1) steps and a split item of t tiles
// about t / 2: both are about half the load.
int persist_item_load(const int4* d) {
  if ((d[4].z >> 16) & 1) return d[1].x + kItemOverheadTiles;
  const int4 u = d[5];  // first / last entries of each sub-tile
  return (u.x >= 0 ? u.y - u.x + 1 : 0) + (u.z >= 0 ? u.w - u.z + 1 : 0) + kItemOverheadTiles;
}

// Long paired items become split items.  The CTA that holds the longest
// item cannot finish before it, and a paired item's two query tiles run side
// by side, each over its whole key-tile list: head-wise causal windows of
// up to 32 key tiles made single items of ~60 tile products against ~35 per
// CTA on average.  An item whose load is above a CTA's fair share (the total
// over the grid) is replaced by one split item per query tile, whose key
// tiles the two sub-tiles take in turn (half the steps; no K / V shared
// between the two query tiles, which matters little for so few items).
void split_persist_items(const Normalized& n, int grid, std::vector<int4>* d) {
  const int mode = g_persist_split.load();
  if (mode < 0) return;
  const size_t cnt = d->size() / kPersistItemInt4;
  long total = 0;
  for (size_t i = 0; i < cnt; ++i) total += persist_item_load(&(*d)[i * kPersistItemInt4]);
  const long fair = total / std::max(1, grid);
  const int nt = (n.N + kTile - 1) / kTile;
  std::vector<int4> out;
  out.reserve(d->size());
  for (size_t i = 0; i < cnt; ++i) {
    const int4* it = &(*d)[i * kPersistItemInt4];
    const int4 u = it[5];
    const int t0 = u.x >= 0 ? u.y - u.x + 1 : 0, t1 = u.z >= 0 ? u.w - u.z + 1 : 0;
    const bool split = mode > 0 ? (t0 >= 2 || t1 >= 2) : persist_item_load(it) > fair;
    if (!split) {
      out.insert(out.end(), it, it + kPersistItemInt4);
      continue;
    }
    for (int s = 0; s < 2; ++s) {
      const int qt = it[0].w + s;
      if ((s ? t1 : t0) == 0 || qt >= nt) continue;
      int4 sd[kPersistItemInt4];
      make_split_item(n, it[0].x, qt, sd);
      out.insert(out.end(), sd, sd + kPersistItemInt4);
    }
  }
  d->swap(out);
}

// ------------------------------------------------------------ per-device state
struct Plan {
  std::vector<int2> items_host;
  std::vector<int32_t> head_info_host;
  std::vector<int4> pitems_host;  // persistent kernel: the items' descriptors, CTA by CTA
  std::vector<int> cta_off_host;  // persistent kernel: CTA c takes descriptors [off[c], off[c+1])
  int persist_grid = 0;           // persistent kernel: CTAs of the launch
  bool has_split = false;         // persistent kernel: some item is a split item
  int2* items = nullptr;
  int32_t* head_info = nullptr;
  int4* pitems = nullptr;
  int* cta_off = nullptr;
};

struct DeviceBuf {
  void* ptr = nullptr;
  size_t bytes = 0;
  int reserve(size_t need, const char* what) {
    if (need <= bytes) return MATTN_OK;
    if (ptr) cudaFree(ptr);
    ptr = nullptr;
    bytes = 0;
    cudaError_t e = cudaMalloc(&ptr, need);
    if (e != cudaSuccess) {
      ptr = nullptr;
      return cuda_fail(e, what);
    }
    bytes = need;
    return MATTN_OK;
  }
};

struct DeviceState {
  uint32_t* err = nullptr;
  int sm_count = 0;
  DeviceBuf copy;      // reordered / converted q, k, v
  DeviceBuf host_io;   // mattn_fwd_host staging
  DeviceBuf dump;      // plan dump
  DeviceBuf rr_ksum;   // block selection: stride key sums
  DeviceBuf rr_scores; // block selection: block scores when the caller passes none
  DeviceBuf recv_lse;  // received attention: the lse in position order
  DeviceBuf dec_part;  // decode: per-chunk softmax states
  std::map<std::string, std::unique_ptr<DeviceBuf>> dec_heads;  // decode: per-head tables by content
  std::map<std::string, std::unique_ptr<Plan>> plans;
  cudaStream_t io_stream = nullptr;      // mattn_fwd_host: copies in and out
  std::vector<cudaEvent_t> io_events;    // mattn_fwd_host: chunk hand-offs
};

std::mutex g_mutex;
std::map<int, std::unique_ptr<DeviceState>> g_devices;

int device_state(DeviceState** out) {
  int dev = -1;
  MATTN_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  auto it = g_devices.find(dev);
  if (it == g_devices.end()) {
    int major = 0, minor = 0;
    MATTN_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "compute capability");
    MATTN_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "compute capability");
    if (major != 10 || minor != 3)
      return fail(MATTN_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
    auto st = std::make_unique<DeviceState>();
    MATTN_CUDA(cudaDeviceGetAttribute(&st->sm_count, cudaDevAttrMultiProcessorCount, dev), "SM count");
    MATTN_CUDA(cudaMalloc(&st->err, sizeof(uint32_t)), "cudaMalloc(error word)");
    MATTN_CUDA(cudaMemset(st->err, 0, sizeof(uint32_t)), "cudaMemset(error word)");
    it = g_devices.emplace(dev, std::move(st)).first;
  }
  *out = it->second.get();
  return MATTN_OK;
}

// The persistent kernel's work items assigned to `grid` CTAs: longest first,
// each to the CTA with the least load so far (the longest-processing-time
// rule), then laid out CTA by CTA so that CTA c takes descriptors
// [off[c], off[c + 1]).  An item's load is persist_item_load.  Items of one
// mask kind with equal windows get equal loads and fall to the CTAs in turn;
// head-wise windows (a few key tiles next to tens) no longer leave the CTAs
// holding two long items to run while others idle.
void assign_persist_items(std::vector<int4>* d, int grid, std::vector<int>* off) {
  const size_t n = d->size() / kPersistItemInt4;
  std::vector<std::pair<int, int>> order(n);  // (load, item)
  for (size_t i = 0; i < n; ++i) order[i] = {persist_item_load(&(*d)[i * kPersistItemInt4]), (int)i};
  std::stable_sort(order.begin(), order.end(), [](const auto& a, const auto& b) { return a.first > b.first; });
  std::vector<std::vector<int>> per(grid);
  std::priority_queue<std::pair<long, int>, std::vector<std::pair<long, int>>, std::greater<>> heap;
  for (int c = 0; c < grid; ++c) heap.push({0, c});
  for (const auto& [load, i] : order) {
    auto [l, c] = heap.top();
    heap.pop();
    per[c].push_back(i);
    heap.push({l + load, c});
  }
  std::vector<int4> out;
  out.reserve(d->size());
  off->assign(grid + 1, 0);
  for (int c = 0; c < grid; ++c) {
    (*off)[c] = (int)(out.size() / kPersistItemInt4);
    for (int i : per[c])
      for (int w = 0; w < kPersistItemInt4; ++w) out.push_back((*d)[(size_t)i * kPersistItemInt4 + w]);
  }
  (*off)[grid] = (int)(out.size() / kPersistItemInt4);
  d->swap(out);
}

std::string plan_key(const Normalized& n, int persist_grid) {
  std::string k;
  char buf[96];
  snprintf(buf, sizeof(buf), "%d|%d|%d|%d|%d|%d|%d|%d|%d|%d|", n.kind, n.B, n.H, n.N, n.need_copy ? 1 : 0,
           n.split ? 1 : 0, n.sink_tokens, n.single ? 1 : 0, n.persistent ? persist_grid : 0,
           n.persistent ? g_persist_split.load() : 0);
  k += buf;
  for (const auto& hp : n.heads) {
    snprintf(buf, sizeof(buf), "%d,%d,%d,%d;", hp.param, hp.load, hp.store, hp.perm_row);
    k += buf;
  }
  return k;
}

// persist_grid: the persistent kernel's CTAs before clamping to the item
// count (one per SM, or the test hook's cap); ignored for other schedules.
int get_plan(DeviceState* st, const Normalized& n, cudaStream_t stream, Plan** out, int persist_grid = 0) {
  std::string key = plan_key(n, persist_grid);
  auto it = st->plans.find(key);
  if (it != st->plans.end()) {
    *out = it->second.get();
    return MATTN_OK;
  }
  auto pl = std::make_unique<Plan>();
  pl->items_host = build_items(n);
  pl->head_info_host.resize((size_t)n.H * 4);
  for (int h = 0; h < n.H; ++h) {
    pl->head_info_host[h * 4 + kHeadParam] = n.heads[h].param;
    pl->head_info_host[h * 4 + kHeadLoad] = n.heads[h].load;
    pl->head_info_host[h * 4 + kHeadStore] = n.heads[h].store;
    pl->head_info_host[h * 4 + kHeadPermRow] = n.heads[h].perm_row;
  }
  if (n.persistent) {
    pl->pitems_host = build_persist_items(n, pl->items_host);
    pl->persist_grid = std::max(1, std::min<int>(persist_grid, (int)pl->items_host.size()));
    split_persist_items(n, pl->persist_grid, &pl->pitems_host);
    pl->persist_grid = std::max(1, std::min<int>(persist_grid, (int)(pl->pitems_host.size() / kPersistItemInt4)));
    assign_persist_items(&pl->pitems_host, pl->persist_grid, &pl->cta_off_host);
    for (size_t i = 0; i < pl->pitems_host.size(); i += kPersistItemInt4)
      pl->has_split = pl->has_split || ((pl->pitems_host[i + 4].z >> 16) & 1);
    MATTN_CUDA(cudaMalloc(&pl->pitems, std::max<size_t>(1, pl->pitems_host.size()) * sizeof(int4)),
               "cudaMalloc(item descriptors)");
    MATTN_CUDA(cudaMemcpyAsync(pl->pitems, pl->pitems_host.data(), pl->pitems_host.size() * sizeof(int4),
                               cudaMemcpyHostToDevice, stream),
               "upload item descriptors");
    MATTN_CUDA(cudaMalloc(&pl->cta_off, pl->cta_off_host.size() * sizeof(int)), "cudaMalloc(CTA item ranges)");
    MATTN_CUDA(cudaMemcpyAsync(pl->cta_off, pl->cta_off_host.data(), pl->cta_off_host.size() * sizeof(int),
                               cudaMemcpyHostToDevice, stream),
               "upload CTA item ranges");
  }
  MATTN_CUDA(cudaMalloc(&pl->items, std::max<size_t>(1, pl->items_host.size()) * sizeof(int2)), "cudaMalloc(items)");
  MATTN_CUDA(cudaMalloc(&pl->head_info, pl->head_info_host.size() * sizeof(int32_t)), "cudaMalloc(head table)");
  MATTN_CUDA(cudaMemcpyAsync(pl->items, pl->items_host.data(), pl->items_host.size() * sizeof(int2),
                             cudaMemcpyHostToDevice, stream),
             "upload items");
  MATTN_CUDA(cudaMemcpyAsync(pl->head_info, pl->head_info_host.data(), pl->head_info_host.size() * sizeof(int32_t),
                             cudaMemcpyHostToDevice, stream),
             "upload head table");
  MATTN_CUDA(cudaStreamSynchronize(stream), "plan upload");
  *out = pl.get();
  st->plans.emplace(key, std::move(pl));
  return MATTN_OK;
}

// ------------------------------------------------------------ TMA descriptors
// The driver's tensor-map encoder, looked up once per process.  Entry points
// that hold different locks (mattn_fwd under g_mutex, mattn_fwd_noalloc under
// its own) reach it, so the lookup runs under std::call_once.
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && fn)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(MATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  return MATTN_OK;
}

int encode(CUtensorMap* tm, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
           const cuuint32_t* box, CUtensorMapSwizzle sw) {
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MATTN_OK;
}

// Raster views [heads][N][d] and, when asked, column-major views
// [heads][rows][cols][d] of one bf16 tensor (heads = B * its head count):
// map [0] covers 64-column chunks (128-byte swizzle), map [1] the 16- or
// 32-column rest.
int make_maps(const Normalized& n, const void* base, CUtensorMap raster[2], CUtensorMap colmaj[2], int rows, int cols,
              int64_t heads, int box_rows = kTile) {
  const int d = n.d;
  const int chunks = d / 64, rem = d % 64;
  const cuuint64_t bh = (cuuint64_t)heads;
  const CUtensorMapSwizzle rem_sw = rem == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B;
  memset(raster, 0, 2 * sizeof(CUtensorMap));
  memset(colmaj, 0, 2 * sizeof(CUtensorMap));
  const char* rem_base = static_cast<const char*>(base) + (size_t)chunks * 64 * 2;
  {
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)n.N * d * 2};
    if (chunks) {
      cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n.N, bh};
      cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
      int rc = encode(&raster[0], base, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc) return rc;
    }
    if (rem) {
      cuuint64_t dims[3] = {(cuuint64_t)rem, (cuuint64_t)n.N, bh};
      cuuint32_t box[3] = {(cuuint32_t)rem, (cuuint32_t)kTile, 1};
      int rc = encode(&raster[1], rem_base, 3, dims, strides, box, rem_sw);
      if (rc) return rc;
    }
  }
  if (rows > 0) {
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)cols * d * 2, (cuuint64_t)n.N * d * 2};
    if (chunks) {
      cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)cols, (cuuint64_t)rows, bh};
      cuuint32_t box[4] = {64, 1, (cuuint32_t)kTile, 1};
      int rc = encode(&colmaj[0], base, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc) return rc;
    }
    if (rem) {
      cuuint64_t dims[4] = {(cuuint64_t)rem, (cuuint64_t)cols, (cuuint64_t)rows, bh};
      cuuint32_t box[4] = {(cuuint32_t)rem, 1, (cuuint32_t)kTile, 1};
      int rc = encode(&colmaj[1], rem_base, 4, dims, strides, box, rem_sw);
      if (rc) return rc;
    }
  }
  return MATTN_OK;
}

// Views of V in one uniform swizzle (map [0] only): boxes of vw columns,
// vw = 64 when d % 64 == 0, else 32 when d % 32 == 0, else 16; the kernel's
// P V product reads all d columns as one MN-major operand.
int make_v_maps(const Normalized& n, const void* base, CUtensorMap raster[2], CUtensorMap colmaj[2], int rows,
                int cols, int64_t heads) {
  const int d = n.d;
  const int vw = d % 64 == 0 ? 64 : (d % 32 == 0 ? 32 : 16);
  const CUtensorMapSwizzle sw =
      vw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : (vw == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  const cuuint64_t bh = (cuuint64_t)heads;
  memset(raster, 0, 2 * sizeof(CUtensorMap));
  memset(colmaj, 0, 2 * sizeof(CUtensorMap));
  {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n.N, bh};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)n.N * d * 2};
    cuuint32_t box[3] = {(cuuint32_t)vw, (cuuint32_t)kTile, 1};
    int rc = encode(&raster[0], base, 3, dims, strides, box, sw);
    if (rc) return rc;
  }
  if (rows > 0) {
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)cols, (cuuint64_t)rows, bh};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)cols * d * 2, (cuuint64_t)n.N * d * 2};
    cuuint32_t box[4] = {(cuuint32_t)vw, 1, (cuuint32_t)kTile, 1};
    int rc = encode(&colmaj[0], base, 4, dims, strides, box, sw);
    if (rc) return rc;
  }
  return MATTN_OK;
}

// 5D views of one bf16 [heads][rows][cols][d] raster tensor in the 2x2-block
// orders, so that a box (d chunk, dc 2, dr 2, 32 blocks, 1) lands in
// sequence-position order.  Row-major blocks (by_cols false): dims (d, dc,
// dr, C, R + head * rows/2); column-major blocks: (d, dc, dr, R + head *
// rows/2, C).  K-major tiles (Q, K): map [0] covers 64-column chunks
// (128-byte swizzle), map [1] the 16- or 32-column rest; V (v_layout): map
// [0] with the uniform kVW-column boxes.
int make_block_maps(const Normalized& n, const void* base, CUtensorMap maps[2], int rows, int cols, int64_t heads,
                    bool v_layout, bool by_cols) {
  const int d = n.d;
  memset(maps, 0, 2 * sizeof(CUtensorMap));
  const cuuint64_t es = 2;
  const cuuint64_t s_c = 2 * (cuuint64_t)d * es, s_r = 2 * (cuuint64_t)cols * d * es;
  const cuuint64_t n_c = (cuuint64_t)cols / 2, n_r = (cuuint64_t)(rows / 2) * heads;
  cuuint64_t strides[4] = {(cuuint64_t)d * es, (cuuint64_t)cols * d * es, by_cols ? s_r : s_c, by_cols ? s_c : s_r};
  auto one = [&](CUtensorMap* m, const void* b, int width, int box_w, CUtensorMapSwizzle sw) {
    cuuint64_t dims[5] = {(cuuint64_t)width, 2, 2, by_cols ? n_r : n_c, by_cols ? n_c : n_r};
    cuuint32_t box[5] = {(cuuint32_t)box_w, 2, 2, 32, 1};
    return encode(m, b, 5, dims, strides, box, sw);
  };
  if (v_layout) {
    const int vw = d % 64 == 0 ? 64 : (d % 32 == 0 ? 32 : 16);
    const CUtensorMapSwizzle sw =
        vw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : (vw == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
    return one(&maps[0], base, d, vw, sw);
  }
  const int chunks = d / 64, rem = d % 64;
  if (chunks) {
    int rc = one(&maps[0], base, d, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  if (rem) {
    const char* rem_base = static_cast<const char*>(base) + (size_t)chunks * 64 * 2;
    int rc = one(&maps[1], rem_base, rem, rem, rem == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B);
    if (rc) return rc;
  }
  return MATTN_OK;
}

// The 2x2-block views that the heads' load modes need.
int make_all_block_maps(const Normalized& n, const void* q, const void* k, const void* v, FwdParams* p, int rows,
                        int cols, int64_t heads_q, int64_t heads_kv) {
  int rc;
  for (int by_cols = 0; by_cols < 2; ++by_cols) {
    if (!(by_cols ? n.any_block_col_tma : n.any_block_tma)) continue;
    if ((rc = make_block_maps(n, q, by_cols ? p->bcq : p->bq, rows, cols, heads_q, false, by_cols))) return rc;
    if ((rc = make_block_maps(n, k, by_cols ? p->bck : p->bk, rows, cols, heads_kv, false, by_cols))) return rc;
    if ((rc = make_block_maps(n, v, by_cols ? p->bcv : p->bv, rows, cols, heads_kv, true, by_cols))) return rc;
  }
  return MATTN_OK;
}

int check_device_ptrs(const void* q, const void* k, const void* v, const void* o, const float* lse) {
  if (!q || !k || !v || !o) return fail(MATTN_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(MATTN_ERR_UNSUPPORTED, "q, k, v and o must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(MATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  return MATTN_OK;
}

// Debug library test hook: writes the launch's work list with defect `what`
// planted into `buf` and points the launch at it.  The checks of the debug
// kernels must catch each defect before it is used to address memory.
int plant_defect(int what, const Normalized& n, const Plan& plan, cudaStream_t stream, DeviceBuf* buf,
                 FwdParams* p) {
  const int nt = (n.N + kTile - 1) / kTile;
  if (what == kCorruptGridRows) {
    p->grid_rows /= 2;
    return MATTN_OK;
  }
  if (n.persistent) {
    std::vector<int4> d = plan.pitems_host;
    if (d.empty()) return fail(MATTN_ERR_INVALID_ARG, "no work items to corrupt");
    if (what == kCorruptItemHead) d[0].x = n.B * n.H;
    else if (what == kCorruptKeyTiles) d[1].y = nt + 3;
    else return fail(MATTN_ERR_INVALID_ARG, "unknown defect %d", what);
    int rc = buf->reserve(d.size() * sizeof(int4), "cudaMalloc(corrupted items)");
    if (rc) return rc;
    MATTN_CUDA(cudaMemcpyAsync(buf->ptr, d.data(), d.size() * sizeof(int4), cudaMemcpyHostToDevice, stream),
               "upload corrupted items");
    p->pitems = static_cast<const int4*>(buf->ptr);
    return MATTN_OK;
  }
  if (what != kCorruptItemHead)
    return fail(MATTN_ERR_INVALID_ARG, "defect %d needs the persistent schedule", what);
  std::vector<int2> items = plan.items_host;
  if (items.empty()) return fail(MATTN_ERR_INVALID_ARG, "no work items to corrupt");
  items[0].x = n.B * n.H;
  int rc = buf->reserve(items.size() * sizeof(int2), "cudaMalloc(corrupted items)");
  if (rc) return rc;
  MATTN_CUDA(cudaMemcpyAsync(buf->ptr, items.data(), items.size() * sizeof(int2), cudaMemcpyHostToDevice, stream),
             "upload corrupted items");
  p->items = static_cast<const int2*>(buf->ptr);
  return MATTN_OK;
}

int fwd_locked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N, int d,
               int dtype, const mattn_mask_desc* desc, cudaStream_t stream, int self_test) {
  if (H_kv < 1 || H % H_kv != 0)
    return fail(MATTN_ERR_INVALID_ARG, "the query head count %d must be a multiple of the K/V head count %d", H, H_kv);
  Normalized n;
  int rc = normalize(desc, B, H, N, d, dtype, true, &n);
  if (rc) return rc;
  rc = check_device_ptrs(q, k, v, o, lse);
  if (rc) return rc;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc) return rc;
  rc = get_encoder();
  if (rc) return rc;
  Plan* plan = nullptr;
  const int cap = g_persist_grid_cap.load();
  rc = get_plan(st, n, stream, &plan, (cap > 0 && cap < st->sm_count) ? cap : st->sm_count);
  if (rc) return rc;

  const size_t elems = (size_t)B * H * N * d;
  const void* src[3] = {q, k, v};
  const void* use[3] = {q, k, v};
  if (n.need_copy) {
    rc = st->copy.reserve(3 * elems * 2, "cudaMalloc(reorder workspace)");
    if (rc) return rc;
    GatherParams gp;
    memset(&gp, 0, sizeof(gp));
    for (int t = 0; t < 3; ++t) {
      gp.src[t] = src[t];
      gp.dst[t] = static_cast<char*>(st->copy.ptr) + (size_t)t * elems * 2;
      use[t] = gp.dst[t];
    }
    gp.head_info = plan->head_info;
    gp.perm = desc->perm;
    gp.B = B; gp.H = H; gp.N = N; gp.d = d;
    gp.kv_group = H / H_kv;
    gp.src_f32 = dtype == MATTN_F32;
    gp.grid_rows = desc->grid_rows;
    gp.grid_cols = desc->grid_cols;
    gp.n_perm = desc->perm ? desc->n_perm : 0;
    gp.err = st->err;
    MATTN_CUDA(launch_gather(gp, stream), "gather launch");
  }
  // the copies hold one K / V head per query head
  const int kv_heads = n.need_copy ? H : H_kv;

  FwdParams p;
  memset(&p, 0, sizeof(p));
  const int rows = n.any_colmajor_tma ? desc->grid_rows : 0;
  const int cols = n.any_colmajor_tma ? desc->grid_cols : 0;
  if (n.single) {
    // 64-column chunks with 128-byte swizzle for Q (128-row boxes) and for K
    // and V (key-tile boxes; V's MN-major atoms have the same layout)
    const int kt = attention_sp_key_tile(d);
    if ((rc = make_maps(n, use[0], p.tq, p.cq, 0, 0, (int64_t)B * H, kTile))) return rc;
    if ((rc = make_maps(n, use[1], p.tk, p.ck, 0, 0, (int64_t)B * kv_heads, kt))) return rc;
    if ((rc = make_maps(n, use[2], p.tv, p.cv, 0, 0, (int64_t)B * kv_heads, kt))) return rc;
  } else {
    if ((rc = make_maps(n, use[0], p.tq, p.cq, rows, cols, (int64_t)B * H))) return rc;
    if ((rc = make_maps(n, use[1], p.tk, p.ck, rows, cols, (int64_t)B * kv_heads))) return rc;
    if ((rc = make_v_maps(n, use[2], p.tv, p.cv, rows, cols, (int64_t)B * kv_heads))) return rc;
    if ((rc = make_all_block_maps(n, use[0], use[1], use[2], &p, desc->grid_rows, desc->grid_cols, (int64_t)B * H,
                                  (int64_t)B * kv_heads)))
      return rc;
  }
  if (n.persistent && dtype == MATTN_BF16 && !n.need_copy && d <= 96) {
    // the persistent kernel stores bf16 output tiles with TMA through views of
    // O in each head's order (the same views as Q's)
    if ((rc = make_maps(n, o, p.o_raster, p.o_colmaj, rows, cols, (int64_t)B * H))) return rc;
    for (int by_cols = 0; by_cols < 2; ++by_cols) {
      if (!(by_cols ? n.any_block_col_tma : n.any_block_tma)) continue;
      if ((rc = make_block_maps(n, o, by_cols ? p.o_blkc : p.o_blk, desc->grid_rows, desc->grid_cols, (int64_t)B * H,
                                false, by_cols)))
        return rc;
    }
    p.o_tma = 1;
  }
  p.H_kv = kv_heads;
  p.kv_group = H / kv_heads;
  p.o = o;
  p.lse = lse;
  p.items = plan->items;
  p.pitems = plan->pitems;
  p.cta_off = plan->cta_off;
  p.after_prepass = (n.need_copy && !n.single) ? 1 : 0;
  p.no_partial = launch_has_no_partial(n) ? 1 : 0;
  // work items of the launch: the persistent kernel's descriptors (long
  // paired items may have become two split items), else the work list
  p.n_items = n.persistent ? (int)(plan->pitems_host.size() / kPersistItemInt4) : (int)plan->items_host.size();
  p.has_split = n.persistent && plan->has_split ? 1 : 0;
  p.head_info = plan->head_info;
  p.perm = desc->perm;
  p.n_perm = desc->perm ? desc->n_perm : 0;
  p.block_bits = n.kind == kBlockSparse ? desc->block_bits : nullptr;
  p.sink = desc->sink;
  p.err = st->err;
  p.timeout_ns = wait_timeout_ns();
  p.B = B; p.H = H; p.N = N;
  p.kind = n.kind;
  p.sink_tokens = n.sink_tokens;
  p.block_heads = n.block_heads;
  p.block_wpr = n.block_wpr;
  p.block_c = n.block_c;
  p.block_nb = n.block_nb;
  p.grid_rows = desc->grid_rows;
  p.grid_cols = desc->grid_cols;
  p.scale_log2 = n.scale * 1.4426950408889634f;
  p.self_test_timeout = self_test;
  p.split = n.split ? 1 : 0;
  p.out_f32 = dtype == MATTN_F32 ? 1 : 0;
  // the launch's corrupted work list (debug library test hook), freed on return
  struct Planted {
    DeviceBuf b;
    ~Planted() {
      if (b.ptr) cudaFree(b.ptr);
    }
  } planted;
  if (kDebugChecks) {
    const int what = g_debug_corrupt.exchange(kCorruptNone);
    if (what != kCorruptNone && (rc = plant_defect(what, n, *plan, stream, &planted.b, &p))) return rc;
  }
  if (n.single)
    MATTN_CUDA(launch_attention_sp(p, d, stream), "attention launch (single pipeline)");
  else if (n.persistent) {
    MATTN_CUDA(launch_attention_persist(p, d, dtype == MATTN_F32, plan->persist_grid, stream),
               "attention launch (persistent)");
  } else
    MATTN_CUDA(launch_attention(p, d, dtype == MATTN_F32, stream), "attention launch");
  if (planted.b.ptr) MATTN_CUDA(cudaStreamSynchronize(stream), "corrupted launch");  // before the list is freed
  return MATTN_OK;
}

}  // namespace

int report_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int prepare_in_place_launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                            int d, int dtype, const mattn_mask_desc* desc, int max_heads, size_t max_items,
                            InPlaceLaunch* out) {
  Normalized n;
  int rc = normalize(desc, B, H, N, d, dtype, true, &n);
  if (rc) return rc;
  rc = check_device_ptrs(q, k, v, o, lse);
  if (rc) return rc;
  if (n.single)
    return fail(MATTN_ERR_UNSUPPORTED, "the no-allocation entry point runs the two-sub-tile kernel (head dim <= 128)");
  if (n.need_copy)
    return fail(MATTN_ERR_UNSUPPORTED,
                "inputs need the reorder / convert pre-pass (fp32 inputs, explicit orders, or a column-major grid "
                "whose row count is not a multiple of %d); only bf16 inputs read in place are supported here",
                kTile);
  if (H > max_heads) return fail(MATTN_ERR_CAPACITY, "H = %d heads exceeds the limit of %d", H, max_heads);
  std::vector<int2> items = build_items(n);
  if (items.size() > max_items)
    return fail(MATTN_ERR_CAPACITY, "the launch has %zu work items, more than the limit of %zu", items.size(),
                max_items);
  int dev = -1, major = 0, minor = 0;
  MATTN_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  MATTN_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "compute capability");
  MATTN_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "compute capability");
  if (major != 10 || minor != 3)
    return fail(MATTN_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
  if ((rc = get_encoder())) return rc;

  FwdParams& p = out->p;
  memset(&p, 0, sizeof(p));
  const int rows = n.any_colmajor_tma ? desc->grid_rows : 0;
  const int cols = n.any_colmajor_tma ? desc->grid_cols : 0;
  if ((rc = make_maps(n, q, p.tq, p.cq, rows, cols, (int64_t)B * H))) return rc;
  if ((rc = make_maps(n, k, p.tk, p.ck, rows, cols, (int64_t)B * H))) return rc;
  if ((rc = make_v_maps(n, v, p.tv, p.cv, rows, cols, (int64_t)B * H))) return rc;
  if ((rc = make_all_block_maps(n, q, k, v, &p, desc->grid_rows, desc->grid_cols, (int64_t)B * H, (int64_t)B * H)))
    return rc;
  p.H_kv = H;
  p.kv_group = 1;
  p.o = o;
  p.lse = lse;
  p.items = nullptr;
  p.n_items = (int)items.size();
  p.head_info = nullptr;
  p.perm = nullptr;
  p.block_bits = n.kind == kBlockSparse ? desc->block_bits : nullptr;
  p.sink = desc->sink;
  p.err = nullptr;
  p.timeout_ns = wait_timeout_ns();
  p.B = B; p.H = H; p.N = N;
  p.kind = n.kind;
  p.sink_tokens = n.sink_tokens;
  p.block_heads = n.block_heads;
  p.block_wpr = n.block_wpr;
  p.block_c = n.block_c;
  p.block_nb = n.block_nb;
  p.grid_rows = desc->grid_rows;
  p.grid_cols = desc->grid_cols;
  p.scale_log2 = n.scale * 1.4426950408889634f;
  p.self_test_timeout = 0;
  p.split = n.split ? 1 : 0;
  p.no_partial = launch_has_no_partial(n) ? 1 : 0;
  out->items = std::move(items);
  out->head_info.assign((size_t)H * 4, 0);
  for (int h = 0; h < H; ++h) {
    out->head_info[h * 4 + kHeadParam] = n.heads[h].param;
    out->head_info[h * 4 + kHeadLoad] = n.heads[h].load;
    out->head_info[h * 4 + kHeadStore] = n.heads[h].store;
    out->head_info[h * 4 + kHeadPermRow] = n.heads[h].perm_row;
  }
  return MATTN_OK;
}

}  // namespace mattn

using namespace mattn;

extern "C" {

int mattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d, int dtype,
              const mattn_mask_desc* desc, void* stream) {
  std::lock_guard<std::mutex> lk(g_mutex);
  return fwd_locked(q, k, v, o, lse, B, H, H, N, d, dtype, desc, static_cast<cudaStream_t>(stream), 0);
}

int mattn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                  int d, int dtype, const mattn_mask_desc* desc, void* stream) {
  std::lock_guard<std::mutex> lk(g_mutex);
  return fwd_locked(q, k, v, o, lse, B, H, H_kv, N, d, dtype, desc, static_cast<cudaStream_t>(stream), 0);
}

// Test hook (not in the public header): the same launch, with the MMA warp
// first waiting on a barrier that nothing ever arrives on, so that the
// bounded-wait / error-word path can be exercised without a hang.
int mattn_internal_fwd_wait_selftest(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                     int N, int d, int dtype, const mattn_mask_desc* desc, void* stream) {
  std::lock_guard<std::mutex> lk(g_mutex);
  return fwd_locked(q, k, v, o, lse, B, H, H, N, d, dtype, desc, static_cast<cudaStream_t>(stream), 1);
}

// Test hook (not in the public header), debug library only: plants defect
// `what` (1: a work item's head row past the last; 2: a persistent item's
// key tiles past the last; 3: half the grid rows for column-major heads)
// into the next forward launch, whose device checks must report it as
// MATTN_ERR_BOUNDS.  The product library refuses (MATTN_ERR_UNSUPPORTED).
int mattn_internal_debug_corrupt(int what) {
  if (!kDebugChecks) return fail(MATTN_ERR_UNSUPPORTED, "defects are planted only in the debug library");
  if (what < kCorruptNone || what > kCorruptGridRows) return fail(MATTN_ERR_INVALID_ARG, "unknown defect %d", what);
  g_debug_corrupt.store(what);
  return MATTN_OK;
}

// Test hook (not in the public header): caps the persistent kernel's grid
// at `ctas` CTAs (0 restores one per SM).
int mattn_internal_set_persist_grid(int ctas) {
  if (ctas < 0) return fail(MATTN_ERR_INVALID_ARG, "ctas must be >= 0");
  g_persist_grid_cap.store(ctas);
  return MATTN_OK;
}

// Test hook (not in the public header), host only: the persistent kernel's
// work items for these arguments on a grid of `grid` CTAs, as the launch
// would build them (paired items, the long ones split, assigned longest
// first): kPersistItemInt4 x 4 int32 per item into items_out (capacity
// cap_items items), the CTA ranges (grid' + 1 ints, grid' = the CTAs the
// launch would use) into off_out (capacity cap_off), their counts into
// *n_items_out and *grid_out.  MATTN_ERR_UNSUPPORTED when the arguments do
// not run the persistent schedule.
int mattn_internal_persist_plan(const mattn_mask_desc* desc, int B, int H, int N, int d, int grid, int32_t* items_out,
                                size_t cap_items, int32_t* off_out, size_t cap_off, size_t* n_items_out,
                                int* grid_out) {
  if (!n_items_out || !grid_out) return fail(MATTN_ERR_INVALID_ARG, "n_items_out / grid_out is NULL");
  if (grid < 1) return fail(MATTN_ERR_INVALID_ARG, "grid must be >= 1");
  Normalized n;
  int rc = normalize(desc, B, H, N, d, MATTN_BF16, true, &n);
  if (rc) return rc;
  if (!n.persistent) return fail(MATTN_ERR_UNSUPPORTED, "these arguments do not run the persistent schedule");
  const std::vector<int2> items = build_items(n);
  std::vector<int4> d4 = build_persist_items(n, items);
  int g = std::max(1, std::min<int>(grid, (int)items.size()));
  split_persist_items(n, g, &d4);
  g = std::max(1, std::min<int>(grid, (int)(d4.size() / kPersistItemInt4)));
  std::vector<int> off;
  assign_persist_items(&d4, g, &off);
  const size_t cnt = d4.size() / kPersistItemInt4;
  *n_items_out = cnt;
  *grid_out = g;
  if (cnt > cap_items || (size_t)g + 1 > cap_off || (cnt && !items_out) || !off_out)
    return fail(MATTN_ERR_CAPACITY, "plan has %zu items and %d CTAs", cnt, g);
  for (size_t i = 0; i < d4.size(); ++i) {
    items_out[4 * i + 0] = d4[i].x;
    items_out[4 * i + 1] = d4[i].y;
    items_out[4 * i + 2] = d4[i].z;
    items_out[4 * i + 3] = d4[i].w;
  }
  for (int c = 0; c <= g; ++c) off_out[c] = off[c];
  return MATTN_OK;
}

// Test hook (not in the public header): which persistent items are split
// (0: the load rule; 1: every item whose query tiles see two or more key
// tiles; -1: none).
int mattn_internal_set_persist_split(int mode) {
  if (mode < -1 || mode > 1) return fail(MATTN_ERR_INVALID_ARG, "mode must be -1, 0 or 1");
  g_persist_split.store(mode);
  return MATTN_OK;
}

int mattn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   int dtype, const mattn_mask_desc* desc, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  std::lock_guard<std::mutex> lk(g_mutex);
  Normalized n;
  int rc = normalize(desc, B, H, N, d, dtype, true, &n);
  if (rc) return rc;
  if (!q || !k || !v || !o) return fail(MATTN_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
  DeviceState* st = nullptr;
  if ((rc = device_state(&st))) return rc;
  if (!st->io_stream) MATTN_CUDA(cudaStreamCreateWithFlags(&st->io_stream, cudaStreamNonBlocking), "copy stream");
  const size_t esz = dtype == MATTN_F32 ? 4 : 2;
  const size_t head_elems = (size_t)N * d;  // one head of one batch entry
  const size_t tensor = (size_t)B * H * head_elems * esz;
  const size_t lse_bytes = (size_t)B * H * N * 4;
  const size_t sink_bytes = desc->sink ? (size_t)H * 4 : 0;
  const size_t bits_bytes =
      n.kind == kBlockSparse ? (size_t)n.block_heads * n.block_nb * n.block_wpr * sizeof(uint64_t) : 0;
  const size_t perm_bytes = (desc->perm && desc->n_perm > 0) ? (size_t)desc->n_perm * N * sizeof(int32_t) : 0;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t total = 4 * up(tensor) + up(lse_bytes) + up(sink_bytes) + up(bits_bytes) + up(perm_bytes);
  if ((rc = st->host_io.reserve(total, "cudaMalloc(host staging)"))) return rc;
  char* base = static_cast<char*>(st->host_io.ptr);
  char* dq = base;
  char* dk = dq + up(tensor);
  char* dv = dk + up(tensor);
  char* dout = dv + up(tensor);
  float* dlse = reinterpret_cast<float*>(dout + up(tensor));
  char* dsink = reinterpret_cast<char*>(dlse) + up(lse_bytes);
  char* dbits = dsink + up(sink_bytes);
  char* dperm = dbits + up(bits_bytes);
  cudaStream_t io = st->io_stream;
  // the mask's device copies first, on the copy stream
  mattn_mask_desc dd = *desc;
  if (desc->sink) {
    MATTN_CUDA(cudaMemcpyAsync(dsink, desc->sink, sink_bytes, cudaMemcpyHostToDevice, io), "copy sink");
    dd.sink = reinterpret_cast<const float*>(dsink);
  }
  if (bits_bytes) {
    MATTN_CUDA(cudaMemcpyAsync(dbits, desc->block_bits, bits_bytes, cudaMemcpyHostToDevice, io), "copy bits");
    dd.block_bits = reinterpret_cast<const uint64_t*>(dbits);
  }
  if (perm_bytes) {
    MATTN_CUDA(cudaMemcpyAsync(dperm, desc->perm, perm_bytes, cudaMemcpyHostToDevice, io), "copy perm");
    dd.perm = reinterpret_cast<const int32_t*>(dperm);
  }
  // Pipeline over chunks of heads (about six per call, whole heads of one
  // batch entry each): the compute stream starts on a chunk as soon as its
  // inputs are in, while the copy stream brings the next ones.
  const int per_b = std::max(1, std::min(H, (6 + B - 1) / B));
  const int hc = (H + per_b - 1) / per_b;
  struct Chunk { int b, h0, h1; };
  std::vector<Chunk> chunks;
  for (int b = 0; b < B; ++b)
    for (int h0 = 0; h0 < H; h0 += hc) chunks.push_back({b, h0, std::min(H, h0 + hc)});
  while (st->io_events.size() < 2 * chunks.size()) {
    cudaEvent_t e;
    MATTN_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "cudaEventCreate");
    st->io_events.push_back(e);
  }
  // the compute stream's earlier work comes first
  cudaEvent_t* ev = st->io_events.data();
  MATTN_CUDA(cudaEventRecord(ev[0], stream), "event record");
  MATTN_CUDA(cudaStreamWaitEvent(io, ev[0], 0), "stream wait");
  // the copy stream takes every chunk's inputs first (each a set of
  // contiguous copies), so that they stream in at full bandwidth while the
  // compute stream starts on the first chunks; the outputs follow it back,
  // chunk by chunk, each after its own compute
  auto chunk_off = [&](const Chunk& ch) { return ((size_t)ch.b * H + ch.h0) * head_elems * esz; };
  auto chunk_bytes = [&](const Chunk& ch) { return (size_t)(ch.h1 - ch.h0) * head_elems * esz; };
  for (size_t c = 0; c < chunks.size(); ++c) {
    const size_t off = chunk_off(chunks[c]), bytes = chunk_bytes(chunks[c]);
    MATTN_CUDA(cudaMemcpyAsync(dq + off, static_cast<const char*>(q) + off, bytes, cudaMemcpyHostToDevice, io),
               "copy q");
    MATTN_CUDA(cudaMemcpyAsync(dk + off, static_cast<const char*>(k) + off, bytes, cudaMemcpyHostToDevice, io),
               "copy k");
    MATTN_CUDA(cudaMemcpyAsync(dv + off, static_cast<const char*>(v) + off, bytes, cudaMemcpyHostToDevice, io),
               "copy v");
    MATTN_CUDA(cudaEventRecord(ev[2 * c], io), "event record");
  }
  for (size_t c = 0; c < chunks.size(); ++c) {
    const Chunk& ch = chunks[c];
    const size_t off = chunk_off(ch);
    MATTN_CUDA(cudaStreamWaitEvent(stream, ev[2 * c], 0), "stream wait");
    // the chunk's heads as a call of their own
    mattn_mask_desc cd = dd;
    if (desc->head_param) cd.head_param = desc->head_param + ch.h0;
    if (desc->head_order) cd.head_order = desc->head_order + ch.h0;
    if (dd.sink) cd.sink = dd.sink + ch.h0;
    if (bits_bytes && n.block_heads == H) {
      cd.block_bits = dd.block_bits + (size_t)ch.h0 * n.block_nb * n.block_wpr;
      cd.block_heads = ch.h1 - ch.h0;
    }
    const size_t lse_off = ((size_t)ch.b * H + ch.h0) * N;
    rc = fwd_locked(dq + off, dk + off, dv + off, dout + off, lse ? dlse + lse_off : nullptr, 1, ch.h1 - ch.h0,
                    ch.h1 - ch.h0, N, d, dtype, &cd, stream, 0);
    if (rc) {
      cudaStreamSynchronize(io);
      return rc;
    }
    MATTN_CUDA(cudaEventRecord(ev[2 * c + 1], stream), "event record");
  }
  for (size_t c = 0; c < chunks.size(); ++c) {
    const Chunk& ch = chunks[c];
    const size_t off = chunk_off(ch), bytes = chunk_bytes(ch);
    const size_t lse_off = ((size_t)ch.b * H + ch.h0) * N;
    MATTN_CUDA(cudaStreamWaitEvent(io, ev[2 * c + 1], 0), "stream wait");
    MATTN_CUDA(cudaMemcpyAsync(static_cast<char*>(o) + off, dout + off, bytes, cudaMemcpyDeviceToHost, io), "copy o");
    if (lse)
      MATTN_CUDA(cudaMemcpyAsync(lse + lse_off, dlse + lse_off, (size_t)(ch.h1 - ch.h0) * N * 4,
                                 cudaMemcpyDeviceToHost, io),
                 "copy lse");
  }
  MATTN_CUDA(cudaStreamSynchronize(io), "copy stream sync");
  MATTN_CUDA(cudaStreamSynchronize(stream), "stream sync");
  return MATTN_OK;
}

int mattn_decode(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* seq_lens, int B,
                 int H, int H_kv, int L, int d, int dtype, const mattn_mask_desc* desc, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  std::lock_guard<std::mutex> lk(g_mutex);
  if (!desc) return fail(MATTN_ERR_INVALID_ARG, "mask descriptor is NULL");
  if (!q || !k || !v || !o) return fail(MATTN_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
  if (B < 1 || H < 1 || H_kv < 1 || L < 1) return fail(MATTN_ERR_INVALID_ARG, "B, H, H_kv, L must be >= 1");
  if (H % H_kv) return fail(MATTN_ERR_INVALID_ARG, "H = %d is not a multiple of H_kv = %d", H, H_kv);
  if (H / H_kv > 8) return fail(MATTN_ERR_UNSUPPORTED, "decode supports up to 8 query heads per key/value head");
  if (d != 64 && d != 128 && d != 256) return fail(MATTN_ERR_UNSUPPORTED, "decode head dim %d (64, 128, 256)", d);
  if (dtype != MATTN_BF16) return fail(MATTN_ERR_UNSUPPORTED, "decode takes bf16 q, k, v");
  if (desc->kind != MATTN_FULL && desc->kind != MATTN_CAUSAL_WINDOW)
    return fail(MATTN_ERR_UNSUPPORTED, "decode masks: MATTN_FULL or MATTN_CAUSAL_WINDOW (got kind %d)", desc->kind);
  if (desc->head_order)
    for (int h = 0; h < H; ++h)
      if (desc->head_order[h] != MATTN_ORDER_RASTER)
        return fail(MATTN_ERR_UNSUPPORTED, "decode reads the cache in sequence order (head_order must be raster)");
  if (desc->sink_tokens < 0) return fail(MATTN_ERR_INVALID_ARG, "sink_tokens must be >= 0");
  if (desc->sink_tokens > 0 && desc->kind != MATTN_CAUSAL_WINDOW)
    return fail(MATTN_ERR_INVALID_ARG, "sink_tokens applies to MATTN_CAUSAL_WINDOW masks only");
  if (!(desc->softmax_scale >= 0.f) || std::isinf(desc->softmax_scale))
    return fail(MATTN_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(MATTN_ERR_UNSUPPORTED, "q, k, v and o must be 16-byte aligned");
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(MATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  if (seq_lens && (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return fail(MATTN_ERR_INVALID_ARG, "seq_lens must be 4-byte aligned");
  std::vector<int32_t> head((size_t)H * 4, 0);
  for (int h = 0; h < H; ++h) {
    const int w = desc->head_param ? desc->head_param[h] : desc->param;
    if (desc->kind == MATTN_CAUSAL_WINDOW && w < 1)
      return fail(MATTN_ERR_INVALID_ARG, "window of head %d must be >= 1 (got %d)", h, w);
    head[(size_t)h * 4 + kHeadParam] = desc->kind == MATTN_CAUSAL_WINDOW ? w : 0;
  }
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  int dev = 0, sms = 0;
  MATTN_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  MATTN_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
  // chunks of the keys a key/value head's query heads may see (every
  // cached key, or at most the widest window plus the sink tokens), in
  // 64-key multiples, at most kDecodeMaxSplits per group.  A CTA holds its
  // SM (its ring fills the shared memory), so the launch runs in waves of
  // `sms` CTAs: the number of chunks per group is the one of up to four
  // waves that fills them best, each extra wave charged 2% for its CTAs'
  // start-up (the first copies' latency before the stream flows).
  int64_t nvis = L;
  if (desc->kind == MATTN_CAUSAL_WINDOW) {
    int64_t wmax = 1;
    for (int h = 0; h < H; ++h) wmax = std::max<int64_t>(wmax, head[(size_t)h * 4 + kHeadParam]);
    nvis = std::min<int64_t>(L, wmax + desc->sink_tokens);
  }
  const int64_t groups = (int64_t)B * H_kv;
  int64_t want = 1;
  double best = -1.0;
  for (int64_t waves = 1; waves <= 4; ++waves) {
    const int64_t ns = std::max<int64_t>(1, waves * sms / groups);
    const int64_t ctas = groups * ns;
    const int64_t used = (ctas + sms - 1) / sms;
    const double fill = (double)ctas / (double)(used * sms) - 0.02 * (double)(used - 1);
    if (fill > best + 1e-9) {
      best = fill;
      want = ns;
    }
  }
  int64_t chunk = ((nvis + want - 1) / want + 63) / 64 * 64;
  const int64_t min_chunk = ((nvis + kDecodeMaxSplits - 1) / kDecodeMaxSplits + 63) / 64 * 64;
  chunk = std::max<int64_t>(std::max<int64_t>(chunk, 64), min_chunk);
  const int n_split = (int)((nvis + chunk - 1) / chunk);
  const size_t part_floats = (size_t)B * H * n_split * ((size_t)d + 2);
  if ((rc = st->dec_part.reserve(part_floats * sizeof(float), "cudaMalloc(decode chunk states)"))) return rc;
  // the per-head table, uploaded once per distinct content
  std::string hkey(reinterpret_cast<const char*>(head.data()), head.size() * sizeof(int32_t));
  auto hit = st->dec_heads.find(hkey);
  if (hit == st->dec_heads.end()) {
    auto buf = std::make_unique<DeviceBuf>();
    if ((rc = buf->reserve(head.size() * sizeof(int32_t), "cudaMalloc(decode head table)"))) return rc;
    MATTN_CUDA(cudaMemcpy(buf->ptr, head.data(), head.size() * sizeof(int32_t), cudaMemcpyHostToDevice),
               "upload decode head table");
    hit = st->dec_heads.emplace(hkey, std::move(buf)).first;
  }
  DecodeParams p;
  memset(&p, 0, sizeof(p));
  p.q = q; p.k = k; p.v = v;
  p.seq_lens = seq_lens;
  p.head_info = static_cast<const int32_t*>(hit->second->ptr);
  p.sink = desc->sink;
  p.part_o = static_cast<float*>(st->dec_part.ptr);
  p.part_ml = p.part_o + (size_t)B * H * n_split * d;
  p.o = o;
  p.lse = lse;
  p.B = B; p.H = H; p.H_kv = H_kv; p.L = L;
  p.n_split = n_split;
  p.chunk = (int)chunk;
  p.kind = desc->kind == MATTN_CAUSAL_WINDOW ? kCausalWindow : kFull;
  p.sink_tokens = desc->sink_tokens;
  const float scale = desc->softmax_scale > 0.f ? desc->softmax_scale : 1.0f / std::sqrt((float)d);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out_f32 = 0;
  p.err = st->err;
  p.timeout_ns = wait_timeout_ns();
  MATTN_CUDA(launch_decode(p, d, stream), "decode launch");
  return MATTN_OK;
}

int mattn_received(const void* q, const void* k, const float* lse, float* r, int B, int H, int N, int d, int dtype,
                   const mattn_mask_desc* desc, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  std::lock_guard<std::mutex> lk(g_mutex);
  Normalized n;
  int rc = normalize(desc, B, H, N, d, dtype, true, &n, false);
  if (rc) return rc;
  if (n.sink_tokens > 0) return fail(MATTN_ERR_UNSUPPORTED, "received attention does not take sink tokens");
  if (d == 256) return fail(MATTN_ERR_UNSUPPORTED, "received attention supports head dims up to 128");
  if (!q || !k || !lse || !r) return fail(MATTN_ERR_INVALID_ARG, "q, k, lse and r must be non-NULL");
  if (!aligned16(q) || !aligned16(k)) return fail(MATTN_ERR_UNSUPPORTED, "q and k must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(r) & 3u))
    return fail(MATTN_ERR_INVALID_ARG, "lse and r must be 4-byte aligned");
  DeviceState* st = nullptr;
  if ((rc = device_state(&st))) return rc;
  if ((rc = get_encoder())) return rc;
  Plan* plan = nullptr;
  if ((rc = get_plan(st, n, stream, &plan))) return rc;
  const size_t elems = (size_t)B * H * N * d;
  const void* use[2] = {q, k};
  if (n.need_copy) {
    if ((rc = st->copy.reserve(3 * elems * 2, "cudaMalloc(reorder workspace)"))) return rc;
    GatherParams gp;
    memset(&gp, 0, sizeof(gp));
    const void* src[3] = {q, k, k};
    for (int t = 0; t < 3; ++t) {
      gp.src[t] = src[t];
      gp.dst[t] = static_cast<char*>(st->copy.ptr) + (size_t)t * elems * 2;
    }
    use[0] = gp.dst[0];
    use[1] = gp.dst[1];
    gp.head_info = plan->head_info;
    gp.perm = desc->perm;
    gp.B = B; gp.H = H; gp.N = N; gp.d = d;
    gp.kv_group = 1;
    gp.src_f32 = dtype == MATTN_F32;
    gp.grid_rows = desc->grid_rows;
    gp.grid_cols = desc->grid_cols;
    gp.n_perm = desc->perm ? desc->n_perm : 0;
    gp.err = st->err;
    MATTN_CUDA(launch_gather(gp, stream), "gather launch");
  }
  RecvParams p;
  memset(&p, 0, sizeof(p));
  const int rows = n.any_colmajor_tma ? desc->grid_rows : 0;
  const int cols = n.any_colmajor_tma ? desc->grid_cols : 0;
  if ((rc = make_maps(n, use[0], p.tq, p.cq, rows, cols, (int64_t)B * H))) return rc;
  if ((rc = make_maps(n, use[1], p.tk, p.ck, rows, cols, (int64_t)B * H))) return rc;
  p.lse_pitch = ((int64_t)N + 127) / 128 * 128;
  if ((rc = st->recv_lse.reserve((size_t)B * H * p.lse_pitch * sizeof(float), "cudaMalloc(received lse)"))) return rc;
  p.lse2p = static_cast<float*>(st->recv_lse.ptr);
  p.r = r;
  p.head_info = plan->head_info;
  p.perm = desc->perm;
  p.n_perm = desc->perm ? desc->n_perm : 0;
  p.block_bits = n.kind == kBlockSparse ? desc->block_bits : nullptr;
  p.err = st->err;
  p.timeout_ns = wait_timeout_ns();
  p.B = B; p.H = H; p.N = N;
  p.kind = n.kind;
  p.block_heads = n.block_heads;
  p.block_wpr = n.block_wpr;
  p.block_c = n.block_c;
  p.block_nb = n.block_nb;
  p.grid_rows = desc->grid_rows;
  p.grid_cols = desc->grid_cols;
  p.scale_log2 = n.scale * 1.4426950408889634f;
  MATTN_CUDA(launch_received(p, lse, d, stream), "received attention launch");
  return MATTN_OK;
}

int mattn_rr_select(const void* q, const void* k, int B, int H, int N, int d, int dtype, int stride, int block,
                    float tau, uint32_t flags, uint64_t* block_bits, float* block_scores, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  std::lock_guard<std::mutex> lk(g_mutex);
  if (!q || !k || !block_bits) return fail(MATTN_ERR_INVALID_ARG, "q, k and block_bits must be non-NULL");
  if (B < 1 || H < 1 || N < 1) return fail(MATTN_ERR_INVALID_ARG, "B, H, N must be >= 1 (got %d, %d, %d)", B, H, N);
  if ((int64_t)B * H > (1 << 20)) return fail(MATTN_ERR_UNSUPPORTED, "B*H too large");
  if (dtype != MATTN_BF16) return fail(MATTN_ERR_UNSUPPORTED, "block selection takes bf16 inputs only");
  if (d != 64 && d != 128) return fail(MATTN_ERR_UNSUPPORTED, "block selection supports head dim 64 or 128 (got %d)", d);
  if (!aligned16(q) || !aligned16(k)) return fail(MATTN_ERR_UNSUPPORTED, "q and k must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_bits) & 7u) || (reinterpret_cast<uintptr_t>(block_scores) & 3u))
    return fail(MATTN_ERR_INVALID_ARG, "block_bits must be 8-byte and block_scores 4-byte aligned");
  if (stride < 1 || N % stride != 0)
    return fail(MATTN_ERR_INVALID_ARG, "the stride must be >= 1 and divide N (stride %d, N %d)", stride, N);
  if (block < stride || block % stride != 0)
    return fail(MATTN_ERR_INVALID_ARG, "the block size must be a multiple of the stride (block %d, stride %d)", block,
                stride);
  const int g = block / stride;
  if (g != 4 && g != 8 && g != 16 && g != 32)
    return fail(MATTN_ERR_UNSUPPORTED, "block / stride must be 4, 8, 16 or 32 (got %d)", g);
  if (!(tau > 0.f && tau <= 1.f)) return fail(MATTN_ERR_INVALID_ARG, "tau must lie in (0, 1] (got %g)", (double)tau);
  if (flags & ~MATTN_RR_SINK_RECENT) return fail(MATTN_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  const int n_s = N / stride;
  const int nb = (n_s + g - 1) / g;
  if (nb > 8192) return fail(MATTN_ERR_UNSUPPORTED, "more than 8192 blocks per row (%d)", nb);
  const int wpr = (nb + 63) / 64;
  const int BH = B * H;
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  if ((rc = get_encoder())) return rc;
  if ((rc = st->rr_ksum.reserve((size_t)BH * n_s * d * 2, "cudaMalloc(stride key sums)"))) return rc;
  if (!block_scores) {
    if ((rc = st->rr_scores.reserve((size_t)BH * nb * nb * sizeof(float), "cudaMalloc(block scores)"))) return rc;
    block_scores = static_cast<float*>(st->rr_scores.ptr);
  }
  RrSumParams sp;
  sp.k = static_cast<const __nv_bfloat16*>(k);
  sp.ksum = static_cast<__nv_bfloat16*>(st->rr_ksum.ptr);
  sp.BH = BH; sp.N = N; sp.n_s = n_s; sp.d = d; sp.S = stride;
  MATTN_CUDA(launch_rr_stride_sum(sp, stream), "stride sum launch");

  RrParams rp;
  memset(&rp, 0, sizeof(rp));
  {
    // sampled queries: element (c, o, i, bh) = Q[bh][i*stride + o][c] (Eq. 6-7)
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)stride, (cuuint64_t)n_s, (cuuint64_t)BH};
    cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)stride * d * 2, (cuuint64_t)N * d * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)kTile, 1};
    if ((rc = encode(&rp.tq[0], q, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))) return rc;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n_s, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)n_s * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
    if ((rc = encode(&rp.tk[0], st->rr_ksum.ptr, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))) return rc;
  }
  rp.block_scores = block_scores;
  rp.err = st->err;
  rp.timeout_ns = wait_timeout_ns();
  rp.BH = BH; rp.H = H; rp.n_s = n_s; rp.S = stride; rp.g = g; rp.nb = nb;
  rp.scale_log2 = (float)(1.4426950408889634 / (stride * std::sqrt((double)d)));
  MATTN_CUDA(launch_rr_scores(rp, d, stream), "block score launch");

  RrTopParams tp;
  tp.scores = block_scores;
  tp.bits = block_bits;
  tp.BH = BH; tp.nb = nb; tp.wpr = wpr;
  tp.tau = tau;
  tp.sink_recent = (flags & MATTN_RR_SINK_RECENT) ? 1 : 0;
  MATTN_CUDA(launch_rr_topk(tp, stream), "top-tau launch");
  return MATTN_OK;
}

int mattn_plan_schedule(const mattn_mask_desc* desc, int B, int H, int N, int d, int dtype,
                        uint32_t* schedule_out) {
  if (!schedule_out) return fail(MATTN_ERR_INVALID_ARG, "schedule_out is NULL");
  Normalized n;
  int rc = normalize(desc, B, H, N, d, dtype, true, &n);
  if (rc) return rc;
  *schedule_out = n.single       ? MATTN_FLAG_SCHEDULE_SINGLE
                  : n.persistent ? MATTN_FLAG_SCHEDULE_PERSISTENT
                  : n.split      ? MATTN_FLAG_SCHEDULE_SPLIT
                                 : MATTN_FLAG_SCHEDULE_PAIRED;
  return MATTN_OK;
}

int mattn_count_pairs(const mattn_mask_desc* desc, int B, int H, int N, uint64_t* pairs_out) {
  if (!pairs_out) return fail(MATTN_ERR_INVALID_ARG, "pairs_out is NULL");
  Normalized n;
  int rc = normalize(desc, B, H, N, 0, MATTN_BF16, false, &n);
  if (rc) return rc;
  uint64_t total = 0;
  for (int h = 0; h < H; ++h) {
    if (n.kind == kBlockSparse) {
      const uint64_t* bits =
          desc->block_bits + (int64_t)((n.block_heads == 1) ? 0 : h) * n.block_nb * n.block_wpr;
      const int64_t bs = n.heads[h].param;
      for (int m = 0; m < n.block_nb; ++m) {
        const int64_t r0 = m * bs, r1 = std::min<int64_t>(N, r0 + bs);  // rows [r0, r1)
        for (int nb = 0; nb <= m; ++nb) {
          if (!block_bit(bits, n.block_wpr, m, nb)) continue;
          if (nb < m) {
            total += (uint64_t)(r1 - r0) * (uint64_t)bs;
          } else {
            // diagonal block: row p sees keys r0 .. p
            const int64_t len = r1 - r0;
            total += (uint64_t)(len * (len + 1) / 2);
          }
        }
      }
    } else {
      for (int64_t p = 0; p < N; ++p) {
        int64_t lo, hi;
        row_interval(n.kind, n.heads[h].param, N, p, &lo, &hi);
        lo = std::max<int64_t>(0, lo);
        hi = std::min<int64_t>(N - 1, hi);
        if (hi >= lo) total += (uint64_t)(hi - lo + 1);
        // sink keys below the window: [0, min(S - 1, p, lo - 1)]
        const int64_t sl = std::min<int64_t>(sink_last(n.sink_tokens, p), lo - 1);
        if (sl >= 0) total += (uint64_t)(sl + 1);
      }
    }
  }
  *pairs_out = total * (uint64_t)B;
  return MATTN_OK;
}

int mattn_plan_tiles(const mattn_mask_desc* desc, int H, int N, int32_t* out, size_t cap, size_t* n_out) {
  if (!n_out) return fail(MATTN_ERR_INVALID_ARG, "n_out is NULL");
  if (cap && !out) return fail(MATTN_ERR_INVALID_ARG, "out is NULL with cap > 0");
  Normalized n;
  int rc = normalize(desc, 1, H, N, 0, MATTN_BF16, false, &n);
  if (rc) return rc;
  const int nt = (N + kTile - 1) / kTile;
  size_t cnt = 0;
  for (int h = 0; h < H; ++h)
    for (int qt = 0; qt < nt; ++qt)
      walk_tiles_host(n, desc->block_bits, h, qt, [&](int kt, int cls) {
        if (cnt < cap) {
          out[4 * cnt + 0] = h;
          out[4 * cnt + 1] = qt;
          out[4 * cnt + 2] = kt;
          out[4 * cnt + 3] = cls;
        }
        ++cnt;
      });
  *n_out = cnt;
  if (cnt > cap) return fail(MATTN_ERR_CAPACITY, "plan has %zu tiles, buffer holds %zu", cnt, cap);
  return MATTN_OK;
}

int mattn_plan_tiles_device(const mattn_mask_desc* desc, int H, int N, int32_t* out, size_t cap, size_t* n_out,
                            void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!n_out) return fail(MATTN_ERR_INVALID_ARG, "n_out is NULL");
  if (cap && !out) return fail(MATTN_ERR_INVALID_ARG, "out is NULL with cap > 0");
  std::lock_guard<std::mutex> lk(g_mutex);
  Normalized n;
  int rc = normalize(desc, 1, H, N, 0, MATTN_BF16, false, &n);
  if (rc) return rc;
  DeviceState* st = nullptr;
  if ((rc = device_state(&st))) return rc;
  Plan* plan = nullptr;
  if ((rc = get_plan(st, n, stream, &plan))) return rc;
  const int nt = (N + kTile - 1) / kTile;
  const size_t slots = (size_t)H * nt * nt * 4;
  if (slots > ((size_t)1 << 31)) return fail(MATTN_ERR_UNSUPPORTED, "plan dump too large (H * nt^2 = %zu)", slots / 4);
  if ((rc = st->dump.reserve((slots + (size_t)H * nt) * sizeof(int32_t), "cudaMalloc(plan dump)"))) return rc;
  PlanDumpParams pp;
  pp.head_info = plan->head_info;
  pp.block_bits = n.kind == kBlockSparse ? desc->block_bits : nullptr;
  pp.H = H; pp.N = N; pp.kind = n.kind;
  pp.sink_tokens = n.sink_tokens;
  pp.block_heads = n.block_heads; pp.block_wpr = n.block_wpr; pp.block_c = n.block_c; pp.block_nb = n.block_nb;
  pp.out = static_cast<int32_t*>(st->dump.ptr);
  pp.counts = pp.out + slots;
  MATTN_CUDA(launch_plan_dump(pp, stream), "plan dump launch");
  std::vector<int32_t> host(slots + (size_t)H * nt);
  MATTN_CUDA(cudaMemcpyAsync(host.data(), st->dump.ptr, host.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, stream),
             "plan dump copy");
  MATTN_CUDA(cudaStreamSynchronize(stream), "plan dump sync");
  size_t cnt = 0;
  for (int h = 0; h < H; ++h)
    for (int qt = 0; qt < nt; ++qt) {
      const int c = host[slots + (size_t)h * nt + qt];
      const int32_t* src = host.data() + ((size_t)h * nt + qt) * nt * 4;
      for (int i = 0; i < c; ++i, ++cnt)
        if (cnt < cap) memcpy(out + 4 * cnt, src + 4 * i, 4 * sizeof(int32_t));
    }
  *n_out = cnt;
  if (cnt > cap) return fail(MATTN_ERR_CAPACITY, "plan has %zu tiles, buffer holds %zu", cnt, cap);
  return MATTN_OK;
}

int mattn_device_status(void* stream, uint32_t* detail_out) {
  std::lock_guard<std::mutex> lk(g_mutex);
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  MATTN_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream sync");
  uint32_t word = 0;
  MATTN_CUDA(cudaMemcpy(&word, st->err, sizeof(word), cudaMemcpyDeviceToHost), "read error word");
  MATTN_CUDA(cudaMemset(st->err, 0, sizeof(word)), "clear error word");
  if (detail_out) *detail_out = word;
  if (word & kErrBounds) return fail(MATTN_ERR_BOUNDS, "a device bounds check failed (error word 0x%x)", word);
  if (word) return fail(MATTN_ERR_TIMEOUT, "a device wait gave up (error word 0x%x)", word);
  return MATTN_OK;
}

int mattn_debug_checks(void) { return kDebugChecks ? 1 : 0; }

int mattn_set_wait_timeout_ns(uint64_t ns) {
  g_timeout_ns.store(ns);
  if (!ns) wait_timeout_ns();
  return MATTN_OK;
}

const char* mattn_status_string(int status) {
  switch (status) {
    case MATTN_OK: return "MATTN_OK";
    case MATTN_ERR_INVALID_ARG: return "MATTN_ERR_INVALID_ARG";
    case MATTN_ERR_UNSUPPORTED: return "MATTN_ERR_UNSUPPORTED";
    case MATTN_ERR_CUDA: return "MATTN_ERR_CUDA";
    case MATTN_ERR_TIMEOUT: return "MATTN_ERR_TIMEOUT";
    case MATTN_ERR_NO_DEVICE: return "MATTN_ERR_NO_DEVICE";
    case MATTN_ERR_CAPACITY: return "MATTN_ERR_CAPACITY";
    case MATTN_ERR_BOUNDS: return "MATTN_ERR_BOUNDS";
    default: return "MATTN_ERR_UNKNOWN";
  }
}

const char* mattn_last_error(void) { return g_last_error; }

int mattn_version(void) { return 101; }

}  // extern "C"
