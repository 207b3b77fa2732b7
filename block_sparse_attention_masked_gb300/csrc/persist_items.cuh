// Work items of the persistent attention kernel (attention_persist.cu) and
// its two TMA producer loops.  A work item is a query-tile pair of one
// (batch, head) whose key-tile plan the host worked out (plan_rules.h;
// layout kPersistItemInt4 in kernel_params.h); each CTA takes the items the
// host assigned it (cta_items) and walks their key-tile lists as one stream.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attention_tiles.cuh"
#include "kernel_params.h"
#include "plan_rules.h"
#include "ptx.cuh"
#include "tile_mma.cuh"

namespace mattn {

namespace {

// A work item as every role reads it: the plan the host worked out for it
// (the layout of kPersistItemInt4 in kernel_params.h), no division needed.
struct PItem {
  ItemPlan ip;
  TileList L;
  int load, store, perm_row;
  int first0, last0, first1, last1;  // first and last entries each sub-tile uses (-1: none)
  bool split;                        // one query tile, entries dealt to the sub-tiles in turn
  __device__ __forceinline__ int first(int s) const { return s ? first1 : first0; }
  __device__ __forceinline__ int last(int s) const { return s ? last1 : last0; }
  // whether sub-tile s multiplies list entry j (SPLIT: builds that take split items)
  template <bool SPLIT>
  __device__ __forceinline__ bool uses(int j, int s) const {
    return (SPLIT && split) ? (j & 1) == s : list_uses(L, j, s);
  }
};

__device__ __forceinline__ const int4* pitem_ptr(const FwdParams& p, int it) {
  return p.pitems + (size_t)it * kPersistItemInt4;
}

// Pulls work item `it`'s descriptor into this SM's L1 ahead of its use.
__device__ __forceinline__ void prefetch_pitem(const FwdParams& p, int it) {
  if (it < p.n_items) {
    ptx::prefetch_l1(pitem_ptr(p, it));
    ptx::prefetch_l1(pitem_ptr(p, it) + kPersistItemInt4 - 1);
  }
}

__device__ __forceinline__ PItem load_pitem(const FwdParams& p, int it) {
  const int4* d = pitem_ptr(p, it);
  const int4 a = __ldg(d + 0), b = __ldg(d + 1), c = __ldg(d + 2);
  const int4 f = __ldg(d + 3), g = __ldg(d + 4), u = __ldg(d + 5);
  PItem r;
  r.ip.bh = a.x;
  r.ip.h = a.y;
  r.ip.b = a.z;
  r.ip.bh_kv = a.z * p.H_kv + a.y / p.kv_group;
  r.ip.sp0.qt = a.w;
  r.ip.sp1.qt = a.w + 1;
  r.ip.sp0.rows = (int64_t)a.w * kTile < p.N;
  r.ip.sp1.rows = (int64_t)(a.w + 1) * kTile < p.N;
  r.ip.sp0.r.lo = c.x; r.ip.sp0.r.hi = c.y; r.ip.sp0.r.flo = f.x; r.ip.sp0.r.fhi = f.y;
  r.ip.sp1.r.lo = c.z; r.ip.sp1.r.hi = c.w; r.ip.sp1.r.flo = f.z; r.ip.sp1.r.fhi = f.w;
  r.ip.sp0.ns = g.x;
  r.ip.sp1.ns = g.y;
  r.ip.sp0.param = r.ip.sp1.param = b.w;
  r.ip.sp0.ktmax = r.ip.sp1.ktmax = 0;  // block kind only
  r.L.n = b.x;
  r.L.lo = b.y;
  r.L.na = b.z;
  r.L.lo0 = c.x; r.L.hi0 = c.y; r.L.lo1 = c.z; r.L.hi1 = c.w;
  r.L.ns0 = g.x; r.L.ns1 = g.y;
  r.L.use_n0 = r.L.use_n1 = 0;
  r.L.e = nullptr;
  r.L.block = false;
  r.load = g.z & 0xff;
  r.store = (g.z >> 8) & 0xff;
  r.split = ((g.z >> 16) & 1) != 0;
  if (r.split) {  // both sub-tiles take the one query tile
    r.ip.sp1.qt = a.w;
    r.ip.sp1.rows = r.ip.sp0.rows;
  }
  r.perm_row = g.w;
  r.first0 = u.x; r.last0 = u.y;
  r.first1 = u.z; r.last1 = u.w;
  return r;
}

// A descriptor whose fields index inside the launch (debug checks): the
// head row and its batch entry and head, the first query tile, the list
// counts and the entries each sub-tile uses, the load and store modes.  The
// key tiles its list names are checked where they are loaded.
__device__ __forceinline__ bool pitem_ok(const FwdParams& p, const PItem& r) {
  const int nt = (p.N + kTile - 1) / kTile;
  const int n = r.L.n;
  auto uses_ok = [n](int first, int last) {
    return (first == -1 && last == -1) || (first >= 0 && first <= last && last < n);
  };
  return r.ip.h >= 0 && r.ip.h < p.H && r.ip.b >= 0 && r.ip.b < p.B && r.ip.bh == r.ip.b * p.H + r.ip.h &&
         r.ip.sp0.qt >= 0 && r.ip.sp0.qt < nt && n >= 0 && n <= nt && r.L.na >= 0 && r.L.na <= n &&
         uses_ok(r.first0, r.last0) && uses_ok(r.first1, r.last1) && r.load >= kLoadRaster &&
         r.load <= kLoadBlock2x2Col && r.store >= kStoreIdentity && r.store <= kStoreBlock2x2Col;
}

// Visible key interval [lo, hi] of query position pos in 32-bit arithmetic
// (N <= 2^30): the rule of plan_rules.h's row_interval with the parameter
// clamped to N, which leaves the interval clipped to [0, N - 1] unchanged.
__device__ __forceinline__ void row_interval32(int kind, int param, int n, int pos, int* lo, int* hi) {
  const int w = param < n ? param : n;
  if (kind == kChunk) {
    const int c0 = (pos / w) * w;
    *lo = c0;
    *hi = c0 + w - 1;
  } else if (kind == kSliding) {
    *lo = pos - w;
    *hi = pos + w;
  } else if (kind == kCausalWindow) {
    *lo = pos - w + 1;
    *hi = pos;
  } else {
    *lo = 0;
    *hi = n - 1;
  }
}

// The CTA's work items: descriptors [first, end) of p.pitems (the host
// assigns items to CTAs and lays them out CTA by CTA).  Thread 0 reads the
// range at the start of the kernel (read_cta_items) and leaves it in
// shared memory for every role.  Debug builds: an empty range, after
// recording the failure, when the range is not inside the launch's items.
struct CtaItems {
  int first, end;
};

__device__ __forceinline__ CtaItems read_cta_items(const FwdParams& p) {
  CtaItems r{__ldg(p.cta_off + blockIdx.x), __ldg(p.cta_off + blockIdx.x + 1)};
  if (!debug_check(p.err, r.first >= 0 && r.first <= r.end && r.end <= p.n_items, kSiteItem)) r.end = r.first;
  return r;
}

template <typename Bar>
__device__ __forceinline__ CtaItems cta_items(const Bar* bar) {
  return CtaItems{bar->item_first, bar->item_end};
}

// Q and K producer (one thread): Q tile t = 2 i + s (i = the CTA's i-th
// item, s its sub-tile) goes to slot t % NQ, K tiles of the concatenated
// key-tile lists to ring slot e % KS.  `Bar` has q_full / q_empty [NQ],
// k_full / k_empty [KS] and abort_flag.  Returns on completion, on abort or
// after a wait that ran past the limit (recorded as kErrProducer).
template <int D, int NQ, int KS, typename Bar>
__device__ __forceinline__ void produce_q_k(const FwdParams& p, Bar* bar, uint8_t* sq, uint8_t* sk,
                                            volatile int* abort_flag) {
  using G = Geo<D>;
  // Two streams served in turn by one thread: the Q tiles (slot t % NQ,
  // free once the S products of Q tile t - NQ are done) and the K tiles of
  // the concatenated key-tile lists (ring slot e % KS).  Neither blocks the
  // other: each is advanced whenever its next slot is free, polled with the
  // non-blocking test_wait (a try_wait would suspend the thread on a slot
  // that stays busy while the other stream's slot frees up).
  const uint64_t keep = ptx::l2_policy_evict_last();
  const uint64_t once = ptx::l2_policy_evict_first();
  const CtaItems items = cta_items(bar);
  const int iend = items.end;
  int qit = items.first, kit = items.first;  // items of the Q and K streams
  PItem qi, ki;
  if (qit < iend) qi = load_pitem(p, qit);
  if (kit < iend) ki = load_pitem(p, kit);
  prefetch_pitem(p, qit + 1);
  int qs = 0;      // sub-tile of the next Q tile
  int t = 0;       // next Q tile
  int kj = 0;      // next entry of the current K item
  int e = 0;       // next entry of the K stream
  while (kit < iend && ki.L.n == 0) {  // (no item has an empty list; kept for safety)
    ++kit;
    if (kit < iend) ki = load_pitem(p, kit);
  }
  uint64_t t_idle = 0;  // start of the current stretch without progress
  uint32_t idle = 0;
  bool failed = false;
  while (qit < iend || kit < iend) {
    bool moved = false;
    if (kit < iend) {
      const int slot = e % KS;
      if (ptx::mbar_test_wait(&bar->k_empty[slot], ((e / KS) & 1) ^ 1)) {
        const int kt = list_kt(ki.L, kj);
        if (!check_or_abort(p, bar, pitem_ok(p, ki), kSiteItem) ||
            !check_or_abort(p, bar, key_tile_ok(p, kt), kSiteKeyTile))
          break;
        ptx::mbar_arrive_expect_tx(&bar->k_full[slot], G::kTileBytes);
        if (!load_tile<D>(p, true, ki.load, sk + slot * G::kTileBytes, &bar->k_full[slot], kt * kTile,
                          ki.ip.bh_kv, keep)) {
          abort_cta(bar);
          break;
        }
        ++e;
        if (++kj == ki.L.n) {
          kj = 0;
          do {
            ++kit;
            if (kit < iend) ki = load_pitem(p, kit);
          } while (kit < iend && ki.L.n == 0);
        }
        moved = true;
      }
    }
    if (qit < iend) {
      const int slot = t % NQ;
      if (ptx::mbar_test_wait(&bar->q_empty[slot], ((t / NQ) & 1) ^ 1)) {
        if (!check_or_abort(p, bar, pitem_ok(p, qi), kSiteItem)) break;
        if (qi.first(qs) >= 0) {
          const SubPlan& sp = qs ? qi.ip.sp1 : qi.ip.sp0;
          ptx::mbar_arrive_expect_tx(&bar->q_full[slot], G::kTileBytes);
          if (!load_tile<D>(p, false, qi.load, sq + slot * G::kTileBytes, &bar->q_full[slot], sp.qt * kTile,
                            qi.ip.bh, once)) {
            abort_cta(bar);
            break;
          }
        } else {
          ptx::mbar_arrive(&bar->q_full[slot]);  // no rows: an empty fill keeps the slot's phases in step
        }
        ++t;
        if (++qs == 2) {
          qs = 0;
          ++qit;
          if (qit < iend) qi = load_pitem(p, qit);
          prefetch_pitem(p, qit + 1);
        }
        moved = true;
      }
    }
    if (moved) {
      idle = 0;
    } else if ((++idle & 63u) == 0) {
      // bounded like every wait: give up after timeout_ns without progress
      if (*abort_flag) break;
      const uint64_t now = ptx::globaltimer_ns();
      if (idle == 64) {
        t_idle = now;
      } else if (now - t_idle > p.timeout_ns) {
        failed = true;
        break;
      }
    }
  }
  if (failed) raise_error(p, bar, kErrProducer);
  if (*abort_flag) {
    uint64_t w0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - w0 < 2000000ull) { }
  }
}

// V producer (one thread): the V tiles of the concatenated key-tile lists
// into ring slot e % VS.  Same exits as produce_q_k.
template <int D, int VS, typename Bar>
__device__ __forceinline__ void produce_v(const FwdParams& p, Bar* bar, uint8_t* sv, volatile int* abort_flag) {
  using G = Geo<D>;
  const uint64_t keep = ptx::l2_policy_evict_last();
  int e = 0;
  bool ok = true;
  const CtaItems items = cta_items(bar);
  for (int it = items.first; ok && it < items.end; ++it) {
    const PItem pi = load_pitem(p, it);
    prefetch_pitem(p, it + 1);
    if (!check_or_abort(p, bar, pitem_ok(p, pi), kSiteItem)) break;
    for (int j = 0; j < pi.L.n; ++j, ++e) {
      const int slot = e % VS;
      const int kt = list_kt(pi.L, j);
      if (debug_aborted(abort_flag) || !check_or_abort(p, bar, key_tile_ok(p, kt), kSiteKeyTile)) {
        ok = false;
        break;
      }
      if (!ptx::mbar_wait(&bar->v_empty[slot], ((e / VS) & 1) ^ 1, p.timeout_ns, abort_flag)) {
        raise_error(p, bar, kErrProducer);
        ok = false;
        break;
      }
      ptx::mbar_arrive_expect_tx(&bar->v_full[slot], G::kTileBytes);
      if (!load_v_tile<D>(p, pi.load, sv + slot * G::kTileBytes, &bar->v_full[slot], kt * kTile, pi.ip.bh_kv,
                          keep)) {
        abort_cta(bar);
        ok = false;
        break;
      }
    }
  }
  if (*abort_flag) {
    uint64_t w0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - w0 < 2000000ull) { }
  }
}

}  // namespace

}  // namespace mattn
