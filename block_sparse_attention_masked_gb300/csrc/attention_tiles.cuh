// Device pieces shared by the two forward kernels that stage 128-row
// tiles with TMA and run tcgen05 MMAs (attention_fwd.cu: one work item per
// CTA; attention_persist.cu: a persistent CTA walking work items): the
// per-item key-tile plan, tile loads through the raster / column-major /
// 2x2-block views, the P V product, the softmax row pass and the MMA issue
// order.  A work item is (b*H + h, query-tile pair) -- or (b*H + h, query
// tile) under the split schedule -- and every role of a CTA derives the same
// plan from it.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernel_params.h"
#include "plan_rules.h"
#include "ptx.cuh"
#include "tile_mma.cuh"

namespace mattn {

namespace {

constexpr int kNoTile = 0x7fffffff;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// The running row maximum m only guards against overflow: numerator and
// denominator share it, so any m gives the same result.  A tile is
// exponentiated against the stale m as long as its row sum of P stays below
// 2^40 (no overflow in fp32 or bf16, nor in O's fp32 accumulation); a tile
// above it is redone against the tile's true maximum.
constexpr float kMaxTileSum = 1099511627776.0f;  // 2^40
// Before a row has a running maximum, its first tile is exponentiated
// against 0 and kept when the row sum lands in [2^-64, 2^40]: every P is
// then finite and the row's largest is at least 2^-71, so whatever flushes
// to zero is below 2^-55 of it (the standard algorithm, exponentiating
// against the true maximum, drops the same terms below 2^-126 of it).  A
// row that sees scores in the tile but sums below 2^-64 (all scores far
// below 0), or above 2^40, is redone against the tile's own maximum.
constexpr float kMinTileSum = 5.421010862427522e-20f;  // 2^-64

// The CTA's key-tile list: entry j (0 <= j < n) is key tile kt(j).  Paired,
// sub-tile s multiplies entry j when uses(j, s); split, entry j belongs to
// pipeline j % 2.  Interval kinds: the entries are the key tiles lo .. lo +
// n - 1 (the union of the sub-tiles' ranges, which overlap or touch), each
// sub-tile using its own range.  Block kind: the entries sit in shared
// memory as kt | use0 << 30 | use1 << 31, built once per CTA.  Reading an
// entry is one add or one shared load, which keeps the loops of the
// copy and MMA warps short.
struct TileList {
  int n, lo;
  int na;              // interval kinds: leading entries 0 .. na - 1 are sink tiles below lo
  int lo0, hi0, lo1, hi1;
  int ns0, ns1;        // sink tiles of each sub-tile (causal window with sink tokens)
  int use_n0, use_n1;  // block kind: entries sub-tile 0 / 1 uses
  const uint32_t* e;
  bool block;
};

// Capacity of the per-CTA key-tile list of block-sparse masks (a query
// tile sees at most N/128 key tiles, so N <= 128 * kMaxList).
constexpr int kMaxList = kBlockListMax;

// Key-tile plan of one 128-row query sub-tile.
struct SubPlan {
  int qt;
  bool rows;                 // the sub-tile has query rows (< N)
  KRange r;                  // interval kinds (causal window with sink tokens: the window part)
  int ns;                    // sink tiles [0, ns) (causal window with sink tokens)
  int param;                 // the head's mask parameter
  int ktmax;                 // block kind: last admissible key tile (causality)
};

// Work description of one CTA, computed identically by every thread.
struct ItemPlan {
  int bh, h, b;
  int bh_kv;  // K / V head row of (b, h): b * H_kv + h / kv_group
  SubPlan sp0, sp1;
};

// Query tile of sub-tile s of work item `it`.
__device__ __forceinline__ int item_qt(const FwdParams& p, int2 it, int s) { return p.split ? it.y : 2 * it.y + s; }

// Global bitmap row of sub-tile s of work item `it` (block kind).
__device__ __forceinline__ const uint64_t* global_row(const FwdParams& p, int2 it, int s) {
  const int h = it.x % p.H;
  const int hb = (p.block_heads == 1) ? 0 : h;
  const int qt = item_qt(p, it, s);
  return p.block_bits + ((int64_t)hb * p.block_nb + qt / p.block_c) * p.block_wpr;
}

__device__ __forceinline__ SubPlan make_subplan(const FwdParams& p, int2 it, int s, int param) {
  SubPlan sp;
  const int nt = (p.N + kTile - 1) / kTile;
  sp.qt = item_qt(p, it, s);
  sp.rows = sp.qt < nt;
  sp.ktmax = sp.qt < nt ? sp.qt : nt - 1;
  sp.param = param;
  sp.ns = 0;
  if (p.kind != kBlockSparse && sp.rows) {
    sp.r = interval_krange(p.kind, param, p.N, sp.qt);
    sp.ns = sink_tiles(p.sink_tokens, p.N, sp.qt);
  } else {
    sp.r.lo = 1; sp.r.hi = 0; sp.r.flo = 0; sp.r.fhi = -1;  // empty
  }
  return sp;
}

__device__ __forceinline__ ItemPlan make_plan(const FwdParams& p, int2 it, int param) {
  ItemPlan ip;
  ip.bh = it.x;
  ip.h = it.x % p.H;
  ip.b = it.x / p.H;
  ip.bh_kv = ip.b * p.H_kv + ip.h / p.kv_group;
  ip.sp0 = make_subplan(p, it, 0, param);
  ip.sp1 = make_subplan(p, it, 1, param);
  return ip;
}

__device__ __forceinline__ int list_kt(const TileList& L, int j) {
  return L.block ? (int)(L.e[j] & 0x3fffffffu) : (j < L.na ? j : L.lo + j - L.na);
}

__device__ __forceinline__ bool list_uses(const TileList& L, int j, int s) {
  if (L.block) return (L.e[j] >> (30 + s)) & 1u;
  const int kt = list_kt(L, j);
  return s ? ((kt >= L.lo1 && kt <= L.hi1) || kt < L.ns1) : ((kt >= L.lo0 && kt <= L.hi0) || kt < L.ns0);
}

// Whether sub-tile s (split: pipeline s, which shares the one query tile)
// has any key tile: its Q tile is loaded and waited for only then.
__device__ __forceinline__ bool list_has(const TileList& L, int s, bool split) {
  if (split) return L.n > 0;
  if (L.block) return (s ? L.use_n1 : L.use_n0) > 0;
  return s ? L.lo1 <= L.hi1 : L.lo0 <= L.hi0;
}

__device__ __forceinline__ TileList make_list(const FwdParams& p, const ItemPlan& ip, const uint32_t* entries,
                                              const int* block_counts) {
  TileList L;
  L.block = p.kind == kBlockSparse;
  L.e = entries;
  L.use_n0 = L.block ? block_counts[1] : 0;
  L.use_n1 = L.block ? block_counts[2] : 0;
  L.lo0 = ip.sp0.r.lo; L.hi0 = ip.sp0.r.hi;
  L.lo1 = ip.sp1.r.lo; L.hi1 = ip.sp1.r.hi;
  L.ns0 = ip.sp0.ns; L.ns1 = ip.sp1.ns;
  L.na = 0;
  if (L.block) {
    L.n = block_counts[0];
    L.lo = 0;
  } else {
    pair_list_span(L.lo0, L.hi0, L.lo1, L.hi1, L.ns0, L.ns1, &L.lo, &L.n, &L.na);
  }
  return L;
}

__device__ __forceinline__ bool sub_partial(const FwdParams& p, const SubPlan& sp, int kt) {
  if (p.kind == kBlockSparse) return block_tile_class(sp.qt, kt, p.N) == kTilePartial;
  if (p.sink_tokens > 0) return sink_window_tile_class(sp.param, p.sink_tokens, p.N, sp.qt, kt) == kTilePartial;
  return interval_tile_class(sp.r, kt) == kTilePartial;
}

// Issue order of the MMA groups (a shared-memory word): the group with
// ticket t is pushed once mma_turn == t, and its issuer then passes the turn
// on.  Paired: entry j's group of sub-tile s has ticket 2j + s; split: entry
// j's group has ticket j.  A plain load / store pair: far cheaper on the
// critical path than an atomic lock.  The bounded spin gives up on abort or
// timeout like any wait.
template <typename Bar>
__device__ __forceinline__ bool mma_turn_wait(Bar* bar, uint32_t ticket, uint64_t timeout_ns,
                                              volatile int* abort_flag) {
  const uint32_t a = ptx::smem_addr(&bar->mma_turn);
  if (ptx::ld_shared_acquire(a) == ticket) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1; it < 0x80000000u; ++it) {
    if (ptx::ld_shared_acquire(a) == ticket) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > timeout_ns) return false;
    }
  }
  return false;
}

template <typename Bar>
__device__ __forceinline__ void mma_turn_pass(Bar* bar, uint32_t ticket) {
  ptx::st_release_shared(ptx::smem_addr(&bar->mma_turn), ticket + 1u);
}

template <typename Bar>
__device__ __forceinline__ void raise_error(const FwdParams& p, Bar* bar, uint32_t bit) {
  *reinterpret_cast<volatile int*>(&bar->abort_flag) = 1;
  atomicOr(p.err, bit);
}

// Debug checks (debug_check in kernel_params.h).  A failed check also
// raises the CTA's abort flag, so that every role leaves as after a
// timed-out wait; always true in the product build.
template <typename Bar>
__device__ __forceinline__ bool check_or_abort(const FwdParams& p, Bar* bar, bool ok, uint32_t site) {
  if (debug_check(p.err, ok, site)) return true;
  *reinterpret_cast<volatile int*>(&bar->abort_flag) = 1;
  return false;
}

// The abort flag after a failed check that recorded itself (load_tile,
// store_tile).
template <typename Bar>
__device__ __forceinline__ void abort_cta(Bar* bar) {
  *reinterpret_cast<volatile int*>(&bar->abort_flag) = 1;
}

// Debug builds: whether the CTA has been aborted, so that the copy threads
// stop issuing; always false in the product build.
__device__ __forceinline__ bool debug_aborted(volatile int* abort_flag) { return kDebugChecks && *abort_flag; }

// A key tile of the sequence (debug checks of key-tile list entries).
__device__ __forceinline__ bool key_tile_ok(const FwdParams& p, int kt) {
  return kt >= 0 && (int64_t)kt * kTile < p.N;
}

// A work item of this launch: its index, its head row and its query tile
// (pair) inside the sequence (debug checks).
__device__ __forceinline__ bool item_in_range(const FwdParams& p, int index, int2 it) {
  const int nt = (p.N + kTile - 1) / kTile;
  const int ny = p.split ? nt : (nt + 1) / 2;
  return index >= 0 && index < p.n_items && it.x >= 0 && it.x < p.B * p.H && it.y >= 0 && it.y < ny;
}

// 2x2-block orders: the 5D view's coordinates (c3, c4) of the tile at
// position p0 (32 consecutive blocks).  Row-major view (d, dc, dr, C,
// R + bh * rows/2): 32 blocks of one block row (cols % 64 == 0).
// Column-major view (d, dc, dr, R + bh * rows/2, C): 32 blocks of one block
// column (rows % 64 == 0).
__device__ __forceinline__ void block2x2_coords(const FwdParams& p, int mode, int p0, int bh, int* c3, int* c4) {
  const int blk = p0 >> 2;
  const int half_rows = p.grid_rows >> 1;
  if (mode == kLoadBlock2x2Row) {
    const int half_cols = p.grid_cols >> 1;
    const int R = blk / half_cols;
    *c3 = blk - R * half_cols;
    *c4 = R + bh * half_rows;
  } else {
    const int C = blk / half_rows;
    *c3 = blk - C * half_rows + bh * half_rows;
    *c4 = C;
  }
}

// Whether the 128-position tile at position p0 of view row bh (nbh rows)
// lies inside the view that `mode` selects, on the coordinates load_tile
// computes (debug checks).
__device__ __forceinline__ bool tile_in_view(const FwdParams& p, int mode, int p0, int bh, int nbh) {
  if (p0 < 0 || p0 >= p.N || (p0 & (kTile - 1)) || bh < 0 || bh >= nbh) return false;
  if (mode == kLoadRaster) return true;
  if (mode == kLoadColumnMajor) {
    if (p.grid_rows <= 0 || p.grid_cols <= 0) return false;
    const int col = p0 / p.grid_rows, r0 = p0 - col * p.grid_rows;
    return col < p.grid_cols && r0 + kTile <= p.grid_rows;
  }
  if (mode != kLoadBlock2x2Row && mode != kLoadBlock2x2Col) return false;
  const int half_rows = p.grid_rows >> 1, half_cols = p.grid_cols >> 1;
  if (half_rows <= 0 || half_cols <= 0) return false;
  int c3, c4;
  block2x2_coords(p, mode, p0, bh, &c3, &c4);
  const int64_t block_rows = (int64_t)nbh * half_rows;  // the view's block-row extent
  if (mode == kLoadBlock2x2Row) return c3 >= 0 && c3 + 32 <= half_cols && c4 >= 0 && c4 < block_rows;
  return c3 >= 0 && c3 + 32 <= block_rows && c4 >= 0 && c4 < half_cols;
}

// TMA load of one 128-row Q (is_k false) or K tile (all d columns) starting
// at sequence position p0, through the raster view, the column-major view or
// a 2x2-block view (`mode`, a LoadMode).  `policy` is the L2 eviction
// priority of the tile's lines.  Debug builds: false, and nothing loaded,
// when the tile is outside the view.
template <int D>
__device__ __forceinline__ bool load_tile(const FwdParams& p, bool is_k, int mode, uint8_t* dst, uint64_t* bar, int p0,
                                          int bh, uint64_t policy) {
  using G = Geo<D>;
  if (!debug_check(p.err, tile_in_view(p, mode, p0, bh, p.B * (is_k ? p.H_kv : p.H)), kSiteLoad)) return false;
  if (mode == kLoadRaster) {
    const CUtensorMap* raster = is_k ? p.tk : p.tq;
#pragma unroll
    for (int c = 0; c < G::kChunks; ++c)
      ptx::tma_load_3d_hint(dst + c * G::kChunkBytes, &raster[0], bar, c * 64, p0, bh, policy);
    if (G::kRem) ptx::tma_load_3d_hint(dst + G::kChunks * G::kChunkBytes, &raster[1], bar, 0, p0, bh, policy);
  } else if (mode == kLoadBlock2x2Row || mode == kLoadBlock2x2Col) {
    // the box (d chunk, dc 2, dr 2, 32 blocks) lands in position order:
    // row 4 * block + 2 * dr + dc of the tile
    const CUtensorMap* blocks =
        mode == kLoadBlock2x2Row ? (is_k ? p.bk : p.bq) : (is_k ? p.bck : p.bcq);
    int c3, c4;
    block2x2_coords(p, mode, p0, bh, &c3, &c4);
#pragma unroll
    for (int c = 0; c < G::kChunks; ++c)
      ptx::tma_load_5d_hint(dst + c * G::kChunkBytes, &blocks[0], bar, c * 64, 0, 0, c3, c4, policy);
    if (G::kRem)
      ptx::tma_load_5d_hint(dst + G::kChunks * G::kChunkBytes, &blocks[1], bar, 0, 0, 0, c3, c4, policy);
  } else {
    // position p = c * rows + r holds token r * cols + c; a 128-position tile is
    // one grid column c, rows r0 .. r0 + 127 (rows % 128 == 0 is required).
    const CUtensorMap* colmaj = is_k ? p.ck : p.cq;
    const int col = p0 / p.grid_rows;
    const int r0 = p0 - col * p.grid_rows;
#pragma unroll
    for (int c = 0; c < G::kChunks; ++c)
      ptx::tma_load_4d_hint(dst + c * G::kChunkBytes, &colmaj[0], bar, c * 64, col, r0, bh, policy);
    if (G::kRem)
      ptx::tma_load_4d_hint(dst + G::kChunks * G::kChunkBytes, &colmaj[1], bar, 0, col, r0, bh, policy);
  }
  return true;
}

// TMA load of one 128-row V tile in its uniform-swizzle layout (map [0] of
// the V views has a kVW-column box); false as load_tile.
template <int D>
__device__ __forceinline__ bool load_v_tile(const FwdParams& p, int mode, uint8_t* dst, uint64_t* bar, int p0,
                                            int bh, uint64_t policy) {
  using G = Geo<D>;
  if (!debug_check(p.err, tile_in_view(p, mode, p0, bh, p.B * p.H_kv), kSiteLoad)) return false;
  if (mode == kLoadRaster) {
#pragma unroll
    for (int c = 0; c < G::kVChunks; ++c)
      ptx::tma_load_3d_hint(dst + c * G::kVChunkBytes, &p.tv[0], bar, c * G::kVW, p0, bh, policy);
  } else if (mode == kLoadBlock2x2Row || mode == kLoadBlock2x2Col) {
    const CUtensorMap* blocks = mode == kLoadBlock2x2Row ? p.bv : p.bcv;
    int c3, c4;
    block2x2_coords(p, mode, p0, bh, &c3, &c4);
#pragma unroll
    for (int c = 0; c < G::kVChunks; ++c)
      ptx::tma_load_5d_hint(dst + c * G::kVChunkBytes, &blocks[0], bar, c * G::kVW, 0, 0, c3, c4, policy);
  } else {
    const int col = p0 / p.grid_rows;
    const int r0 = p0 - col * p.grid_rows;
#pragma unroll
    for (int c = 0; c < G::kVChunks; ++c)
      ptx::tma_load_4d_hint(dst + c * G::kVChunkBytes, &p.cv[0], bar, c * G::kVW, col, r0, bh, policy);
  }
  return true;
}

// TMA store of one 128-row O tile from shared memory (laid out as
// load_tile writes a Q tile) to the output rows at sequence positions
// [p0, p0 + 128) of row block bh, through the O view of the head's order
// (`mode`, a LoadMode; requires p.o_tma).  Rows past N are clipped.  O is
// written once and not re-read: its lines go first out of L2 (`policy`,
// evict-first), ahead of the K / V tiles other query tiles still read.
// Debug builds: false, and nothing stored, when the tile is outside the view.
template <int D>
__device__ __forceinline__ bool store_tile(const FwdParams& p, int mode, const uint8_t* src, int p0, int bh,
                                           uint64_t policy) {
  using G = Geo<D>;
  if (!debug_check(p.err, tile_in_view(p, mode, p0, bh, p.B * p.H), kSiteStore)) return false;
  if (mode == kLoadRaster) {
#pragma unroll
    for (int c = 0; c < G::kChunks; ++c)
      ptx::tma_store_3d_hint(&p.o_raster[0], src + c * G::kChunkBytes, c * 64, p0, bh, policy);
    if (G::kRem) ptx::tma_store_3d_hint(&p.o_raster[1], src + G::kChunks * G::kChunkBytes, 0, p0, bh, policy);
  } else if (mode == kLoadBlock2x2Row || mode == kLoadBlock2x2Col) {
    const CUtensorMap* blocks = mode == kLoadBlock2x2Row ? p.o_blk : p.o_blkc;
    int c3, c4;
    block2x2_coords(p, mode, p0, bh, &c3, &c4);
#pragma unroll
    for (int c = 0; c < G::kChunks; ++c)
      ptx::tma_store_5d_hint(&blocks[0], src + c * G::kChunkBytes, c * 64, 0, 0, c3, c4, policy);
    if (G::kRem) ptx::tma_store_5d_hint(&blocks[1], src + G::kChunks * G::kChunkBytes, 0, 0, 0, c3, c4, policy);
  } else {
    const int col = p0 / p.grid_rows;
    const int r0 = p0 - col * p.grid_rows;
#pragma unroll
    for (int c = 0; c < G::kChunks; ++c)
      ptx::tma_store_4d_hint(&p.o_colmaj[0], src + c * G::kChunkBytes, c * 64, col, r0, bh, policy);
    if (G::kRem)
      ptx::tma_store_4d_hint(&p.o_colmaj[1], src + G::kChunks * G::kChunkBytes, 0, col, r0, bh, policy);
  }
  return true;
}

// Writes 8 bf16 values (one 16-byte unit u of the d columns) of row `row`
// into a tile laid out as load_tile writes it: 64-column chunks of 128-byte
// rows in the 128-byte swizzle (unit index XOR row % 8), then the 16- or
// 32-column rest in the 32- or 64-byte swizzle.
template <int D>
__device__ __forceinline__ void tile_put16(uint8_t* tile, int row, int u, uint4 v) {
  using G = Geo<D>;
  const int c = u >> 3;  // 64-column chunk
  uint8_t* dst;
  if (c < G::kChunks) {
    dst = tile + c * G::kChunkBytes + row * 128 + (((u & 7) ^ (row & 7)) << 4);
  } else {
    const int ur = u - 8 * G::kChunks;  // unit inside the rest
    const int sw = G::kRem == 16 ? ((row >> 2) & 1) : ((row >> 1) & 3);
    dst = tile + G::kChunks * G::kChunkBytes + row * G::kRemRowBytes + ((ur ^ sw) << 4);
  }
  *reinterpret_cast<uint4*>(dst) = v;
}

// O += P V for one sub-tile: P (128 x 128 keys, bf16 pairs in TMEM) is the
// A operand; V (keys x d, d contiguous) is an MN-major B operand whose
// kVW-column atoms lie kVChunkBytes apart (leading byte offset) and whose
// 8-key groups lie 8 rows apart (stride byte offset).  One N = D MMA per
// 16 keys, issued by one thread.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_addr4, bool accumulate) {
  using G = Geo<D>;
  constexpr uint32_t idesc = ptx::idesc_bf16(128, D, 1);
  constexpr uint32_t row_bytes = G::kVW * 2;
  constexpr uint32_t lbo = (uint32_t)(G::kVChunkBytes >> 4) << 16;
  constexpr uint32_t hi = ptx::smem_desc_hi(8 * row_bytes, G::kVSwizzle);
  uint32_t acc = accumulate ? 1u : 0u;
#pragma unroll 1
  for (int k = 0; k < kTile / 16; ++k) {
    // 16 bf16 keys = 8 tensor-memory columns of P; 16 rows of V
    ptx::mma_ts(o_tmem, p_tmem + k * 8, desc_of(v_addr4 + ((k * 16 * row_bytes) >> 4) + lbo, hi), idesc, acc);
    acc = 1;
  }
}

// P = exp2(x * sl2 - mref) for the 128 scores of this thread's row, stored
// to tensor memory at p_tmem as bf16 pairs (64 columns, round to nearest);
// returns the row sum of the fp32 values.  All exponentials use MUFU ex2:
// moving a share of them to an FMA-pipe polynomial measured slower at every
// share tried, as did a truncating pack with a second sum over the
// truncated values (one more add and two integer ops per pair).  Masked
// scores are -inf (mask_row) and give exactly 0.  `none` may flag 32-column
// groups (bit g) to be exponentiated against -inf as a whole; every caller
// passes 0, and the per-group reference is kept in this form because the
// unmasked pass measured slower with the reference hoisted out of the group
// loop (16384-token ViT full 1.09 -> 1.12 ms).
// (NC = 128 for a whole row; a thread holding half a row passes its 64
// scores and the tensor-memory address of its half of P.)
template <int NC>
__device__ __forceinline__ float exp_to_tmem(const float (&x)[NC], float sl2, float mref, uint32_t p_tmem,
                                             uint32_t none = 0u) {
  static_assert(NC % 32 == 0, "whole 32-column groups");
  const float2 sl2v = make_float2(sl2, sl2);
  float2 acc[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
  for (int c0 = 0; c0 < NC; c0 += 32) {
    const float nm = ((none >> (c0 / 32)) & 1u) ? -INFINITY : -mref;
    const float2 negm = make_float2(nm, nm);
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 t = ptx::ffma2(make_float2(x[c0 + 2 * i], x[c0 + 2 * i + 1]), sl2v, negm);
      const float2 pp = make_float2(ptx::ex2(t.x), ptx::ex2(t.y));
      pk[i] = ptx::pack_bf16x2(pp.x, pp.y);
      acc[i & 1] = ptx::fadd2(acc[i & 1], pp);
    }
    ptx::tmem_st16(p_tmem + c0 / 2, pk);
  }
  const float2 a = ptx::fadd2(acc[0], acc[1]);
  return a.x + a.y;
}

// Bits of the 32 columns [32g, 32g + 31] inside [lo, hi] (column indices of
// a 128-column tile; lo > hi: none).
__device__ __forceinline__ uint32_t range_bits(int g, int lo, int hi) {
  const int a = lo - 32 * g, b = hi - 32 * g;
  if (b < 0 || a > 31 || a > b) return 0u;
  const int a0 = a < 0 ? 0 : a, b0 = b > 31 ? 31 : b;
  return (0xffffffffu >> (31 - b0)) & (0xffffffffu << a0);
}

// Boundary mask of one row of a PARTIAL tile: x[c] = -inf for the key
// columns c of the 128-key tile outside this row's visible interval
// [c_lo, c_hi] and outside its sink columns [0, c_s] (c_s < 0: none), one
// select per column from its 32-column group's bit mask, with no branch
// per group (measured faster than selecting only in the groups some lane
// of the warp sees in part and flagging the empty ones: 16384-token ViT
// sliding window 92.9 -> 89.2 us, head-wise causal windows 64.2 -> 60.1
// us).  Returns whether the row sees any column of the tile.
// (x may hold NC < 128 columns of the row, starting at tile column col0, a
// multiple of 32.)
template <int NC>
__device__ __forceinline__ bool mask_row(float (&x)[NC], int c_lo, int c_hi, int c_s, int col0 = 0) {
#pragma unroll
  for (int g = 0; g < NC / 32; ++g) {
    const int gt = g + col0 / 32;  // 32-column group of the tile
    const uint32_t vis = range_bits(gt, c_lo, c_hi) | range_bits(gt, 0, c_s);
#pragma unroll
    for (int j = 0; j < 32; ++j) x[32 * g + j] = ((vis >> j) & 1u) ? x[32 * g + j] : -INFINITY;
  }
  const int a = max(c_lo, col0), b = min(c_hi, col0 + NC - 1);
  return a <= b || c_s >= col0;
}

// Maximum of the 128 raw scores of this thread's row (8 independent chains;
// measured faster here than three-input maxima).
template <int NC>
__device__ __forceinline__ float row_max(const float (&x)[NC]) {
  float r = -INFINITY;
#pragma unroll
  for (int c = 0; c < NC; c += 32) {
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = x[c + i];
#pragma unroll
    for (int u = 8; u < 32; u += 8)
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = fmaxf(a[i], x[c + u + i]);
    const float g = fmaxf(fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])), fmaxf(fmaxf(a[4], a[5]), fmaxf(a[6], a[7])));
    r = fmaxf(r, g);
  }
  return r;
}

// O row *= alpha in tensor memory (warp-collective; alpha is per lane), for
// the 16-column chunks of O in [c_begin, c_end).
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t o_tmem, float alpha, int c_begin = 0, int c_end = D) {
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 16) {
    if (c0 < c_begin || c0 >= c_end) continue;  // warp-uniform: a column range of O
    float ov[16];
    ptx::tmem_ld16(o_tmem + c0, ov);
    ptx::tmem_wait_ld();
    uint32_t ou[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) ou[i] = __float_as_uint(ov[i] * alpha);
    ptx::tmem_st16(o_tmem + c0, ou);
  }
}

__device__ __forceinline__ int64_t token_of(const FwdParams& p, int store_mode, int perm_row, int64_t pos) {
  return token_at(store_mode, p.grid_rows, p.grid_cols,
                  store_mode == kStoreExplicit ? p.perm + (int64_t)perm_row * p.N : nullptr, pos);
}

// token_of for an output row at position pos < N.  Debug builds check the
// head's explicit-order row against the orders passed (kSiteItem) and the
// token against [0, N) (kSiteOrder: the device does not otherwise check
// that an explicit order is a permutation), and return -1 after a failed
// check: the row is then not stored.
__device__ __forceinline__ int64_t out_token(const FwdParams& p, int store_mode, int perm_row, int64_t pos) {
  if (!debug_check(p.err, store_mode != kStoreExplicit || (perm_row >= 0 && perm_row < p.n_perm), kSiteItem))
    return -1;
  const int64_t tok = token_of(p, store_mode, perm_row, pos);
  if (!debug_check(p.err, tok >= 0 && tok < p.N, kSiteOrder)) return -1;
  return tok;
}

// Final normalisation of one query row: O = (O_a e_a + O_b e_b) /
// (l_a e_a + l_b e_b + exp(sink)) with e_x = exp2(m_x - M) against the
// common maximum M (a second state (m_b, l_b) is the split schedule's other
// pipeline; -inf and 0 when there is none), and the natural-log LSE of the
// same normaliser.  All values in the log2 domain; b2 = the sink logit
// times log2(e), -inf for no sink.  Rows with nothing visible get scales 0
// and LSE -inf (or the sink logit).
__device__ __forceinline__ void finalize_row(float m, float l, float m_o, float l_o, float b2, float* o_scale,
                                             float* oo_scale, float* lse) {
  const float M = fmaxf(fmaxf(m, m_o), b2);
  *o_scale = 0.f;
  *oo_scale = 0.f;
  *lse = -INFINITY;
  if (M != -INFINITY) {
    const float em = (m == -INFINITY) ? 0.f : ptx::ex2(m - M);
    const float eo = (m_o == -INFINITY) ? 0.f : ptx::ex2(m_o - M);
    const float lf = l * em + l_o * eo + ((b2 == -INFINITY) ? 0.f : ptx::ex2(b2 - M));
    if (lf > 0.f) {
      *o_scale = em / lf;
      *oo_scale = eo / lf;
      *lse = (M + ptx::lg2(lf)) * kLn2;
    }
  }
}

}  // namespace

}  // namespace mattn
