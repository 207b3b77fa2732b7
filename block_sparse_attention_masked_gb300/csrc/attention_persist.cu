// Persistent masked attention forward for the interval masks (full, chunk,
// sliding window, causal window with or without sink tokens) on sm_103a.
//
// The computation of a work item is that of attention_fwd.cu's paired
// schedule: query rows [256*pair, 256*pair + 256) of one (batch, head) as
// two 128-row sub-tiles s = 0, 1 sharing the staged K/V tiles, for every
// key tile kt of the item's list
//     S_s  = Q_s K_kt^T                        (tcgen05.mma, smem x smem -> TMEM)
//     P_s  = exp2(S_s * scale*log2e - m_s)     (softmax warps, online max m_s)
//     O_s += P_s V_kt                          (tcgen05.mma, P from TMEM, V from smem)
// and O_s / (l_s + exp(sink)) with the log-sum-exp at the end (SHS slides
// Eq. 1 for the sink; the FlashAttention idea of the Vision transformers
// lesson).  What differs is the schedule: the grid has one CTA per SM and
// each CTA takes the work items the host assigned it (longest first, each
// to the least-loaded CTA).  Its key-tile lists are walked as one stream, so
// the K/V rings, the MMA issue order and the softmax never drain between
// items: the next item's Q tiles are loaded while the current one runs (Q
// slots rotate) and its first Q K^T goes to the tensor core in the same
// group as the current item's last P V.  The softmax warps of a sub-tile
// write the item's output while that product runs: they wait for the last
// P V, read O_s, normalise and store it, then take the next item's first
// S, which is ready by then.  Masks whose items are short (a window of a
// few key tiles) spend most of a one-item-per-CTA launch in set-up and
// epilogue; here those overlap the neighbouring items' work.
//
// A split item (built when a plan holds one: SPLIT) is one query tile whose
// key tiles alternate between the two sub-tiles; each keeps its own (m, l,
// O) and at the item's end the two are merged (the split schedule of
// attention_fwd.cu, per item): long query tiles then take half the steps.
//
// Roles (384 threads):
//   warp 0        TMA producer: Q tiles into their slots and K tiles into their ring
//   warp 1        tensor-memory allocator; MMA issuer of sub-tile 0
//   warp 2        MMA issuer of sub-tile 1
//   warp 3        TMA producer of the V ring
//   warps 4..7    softmax and epilogue of sub-tile 0 (one query row per thread)
//   warps 8..11   softmax and epilogue of sub-tile 1
// Tensor memory (512 columns x 128 lanes, fp32): S_0 [0,128), S_1
// [128,256) (P_s as bf16 pairs in the first 64 columns of S_s), O_0
// [256,384), O_1 [384,512).  O_s of an item is read once its last P V is
// done (o_full); the next item's first P V, which overwrites it, is issued
// only after that item's first P, which the same threads write after
// reading O_s.
// Every wait is bounded in time and gives up by raising a CTA-wide abort
// flag and a device error bit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attention_tiles.cuh"
#include "kernel_params.h"
#include "persist_items.cuh"
#include "plan_rules.h"
#include "ptx.cuh"
#include "tile_mma.cuh"

namespace mattn {

namespace {

constexpr int kPThreads = 384;
// Registers per thread after setmaxnreg: producer / MMA-issuer warpgroup and
// the two softmax warpgroups (their sum times 128 equals the launch budget).
constexpr uint32_t kPRegsControl = 56;
constexpr uint32_t kPRegsSoftmax = 224;
static_assert(kPRegsControl + 2 * kPRegsSoftmax == 3 * 168, "register split must match the launch budget");

// Q slots: Q tile t = 2 i + s (i = the CTA's i-th item) goes to slot
// t % kQSlots, free again once the S products of Q tile t - kQSlots are done.
// Output staging: one tile per sub-tile, written by the softmax warps and
// stored with TMA (bf16 output at head dim <= 96; at 128 the shared memory
// is full and rows are stored directly).
template <int D, bool OUT_F32>
struct PGeo {
  static constexpr int kQSlots = 3;
  static constexpr bool kStage = (D <= 96) && !OUT_F32;
  static constexpr int kStageTiles = kStage ? 2 : 0;
};

struct PBarriers {
  uint64_t q_full[3], q_empty[3];
  uint64_t k_full[3], k_empty[3];
  uint64_t v_full[3], v_empty[3];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];      // the item's last P V of sub-tile s is done
  uint64_t drain[2];       // MMA drain on abort, one per issuer
  uint64_t stage_sync[2];  // per sub-tile: barrier of its 128 softmax threads (output staging)
  uint64_t split_sync;     // the 256 softmax threads (merge of a split item)
  uint64_t never;          // self-test: nothing ever arrives here
  uint32_t tmem_base;
  int abort_flag;
  uint32_t mma_turn;       // ticket of the MMA group that may be issued next
  int item_first, item_end;  // the CTA's work items (read_cta_items)
  float2 xch[kTile];         // split items: sub-tile 1's (m, l) per row, then the two scales
};

template <int D, bool OUT_F32, bool MASK, bool SPLIT>
__global__ void __launch_bounds__(kPThreads, 1) attention_persist_kernel(const __grid_constant__ FwdParams p) {
  using G = Geo<D>;
  constexpr int KS = G::kStages;
  constexpr int VS = G::kStages;
  using PG = PGeo<D, OUT_F32>;
  constexpr int NQ = PG::kQSlots;
  static_assert(KS == VS, "one ring depth for K and V");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = base;
  uint8_t* sk = sq + NQ * G::kTileBytes;
  uint8_t* sv = sk + KS * G::kTileBytes;
  uint8_t* sstage = sv + VS * G::kTileBytes;  // PG::kStageTiles output tiles
  PBarriers* bar = reinterpret_cast<PBarriers*>(sstage + PG::kStageTiles * G::kTileBytes);
  volatile int* abort_flag = &bar->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    // after the reorder pre-pass: no wait of this CTA may start while its
    // copies are still being written
    if (p.after_prepass) asm volatile("griddepcontrol.wait;" ::: "memory");
    // the CTA's item range, the raster maps' descriptors and (below) its
    // first item's descriptor are fetched while the barriers are set up
    const CtaItems items = read_cta_items(p);
    ptx::prefetch_tmap(&p.tq[0]);
    ptx::prefetch_tmap(&p.tk[0]);
    ptx::prefetch_tmap(&p.tv[0]);
    for (int i = 0; i < NQ; ++i) {
      ptx::mbar_init(&bar->q_full[i], 1);
      ptx::mbar_init(&bar->q_empty[i], 1);
    }
    for (int i = 0; i < KS; ++i) {
      ptx::mbar_init(&bar->k_full[i], 1);
      ptx::mbar_init(&bar->k_empty[i], 2);  // one commit from each issuer
      ptx::mbar_init(&bar->v_full[i], 1);
      ptx::mbar_init(&bar->v_empty[i], 2);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bar->s_full[s], 1);
      ptx::mbar_init(&bar->p_full[s], kTile);
      ptx::mbar_init(&bar->o_full[s], 1);
      ptx::mbar_init(&bar->drain[s], 1);
      ptx::mbar_init(&bar->stage_sync[s], kTile);
    }
    ptx::mbar_init(&bar->split_sync, 2 * kTile);
    ptx::mbar_init(&bar->never, 1);
    bar->abort_flag = 0;
    bar->mma_turn = 0;
    bar->item_first = items.first;
    bar->item_end = items.end;
    prefetch_pitem(p, items.first);
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bar->tmem_base, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bar->tmem_base;

  if (warp == 0) {
    ptx::setmaxnreg_dec<kPRegsControl>();
    if (lane == 0) produce_q_k<D, NQ, KS>(p, bar, sq, sk, abort_flag);
  } else if (warp == 3) {
    ptx::setmaxnreg_dec<kPRegsControl>();
    if (lane == 0) produce_v<D, VS>(p, bar, sv, abort_flag);
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Issuer s walks every entry e of the CTA's stream (both issuers release
    // every K / V slot, the empty barriers counting 2) and, in ticket order
    // 2e + s, issues the group P V(e-1) + S(e): the pending product of the
    // previous entry (when s used it) and this entry's S (when s uses it).
    // At an item boundary the group is the last P V of one item and the
    // first S of the next.  The next item's first P V (accumulate = 0) needs
    // that item's first P, which the softmax warps write only after reading
    // O_s: waiting for P is waiting for O_s to be free.
    ptx::setmaxnreg_dec<kPRegsControl>();
    const int s = warp - 1;
    auto wait_all = [&](uint64_t* b, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(b, parity, p.timeout_ns, abort_flag));
    };
    constexpr uint32_t tile4 = G::kTileBytes >> 4;  // descriptor start-address units
    const uint32_t q4 = ptx::smem_addr(sq) >> 4;
    const uint32_t k4 = ptx::smem_addr(sk) >> 4;
    const uint32_t v4 = ptx::smem_addr(sv) >> 4;
    const uint32_t s_tm = tmem + s * 128;
    const uint32_t o_tm = tmem + 256 + s * 128;
    bool ok = true, issued_any = false;
    if (p.self_test_timeout && s == 0) {
      // nothing ever arrives on this barrier: exercises the bounded-wait path
      if (!wait_all(&bar->never, 0)) {
        if (lane == 0) raise_error(p, bar, kErrSelfTest);
        ok = false;
      }
    }
    bool pend = false, pend_first = false, pend_last = false;
    uint32_t pcount = 0;  // P tiles consumed
    int e = 0;
    int i = 0;  // the CTA's item count so far
    const CtaItems items = cta_items(bar);
    for (int it = items.first; ok && it < items.end; ++it, ++i) {
      const PItem pi = load_pitem(p, it);
      prefetch_pitem(p, it + 1);
      if (!check_or_abort(p, bar, pitem_ok(p, pi), kSiteItem)) {
        ok = false;
        break;
      }
      const TileList& L = pi.L;
      const int first_use = pi.first(s), last_use = pi.last(s);
      const int t = 2 * i + s;
      const int qslot = t % NQ;
      const uint32_t qpar = (t / NQ) & 1;
      if (first_use < 0) {
        // no rows in this sub-tile: take the slot's empty fill and hand it back
        if (!wait_all(&bar->q_full[qslot], qpar)) {
          ok = false;
          break;
        }
        if (lane == 0) ptx::mbar_arrive(&bar->q_empty[qslot]);
      }
      for (int j = 0; j < L.n; ++j, ++e) {
        const bool use = pi.uses<SPLIT>(j, s);
        const int ks = e % KS;
        const bool rel_v = e >= 1;
        const int ve = e - 1;
        if (rel_v && !wait_all(&bar->v_full[ve % VS], (ve / VS) & 1)) { ok = false; break; }
        if (!wait_all(&bar->k_full[ks], (e / KS) & 1)) { ok = false; break; }
        if (pend) {
          if (!wait_all(&bar->p_full[s], pcount & 1)) { ok = false; break; }
          ++pcount;
          ptx::tc_fence_after();
        }
        if (use && j == first_use && !wait_all(&bar->q_full[qslot], qpar)) { ok = false; break; }
        const uint32_t ticket = (uint32_t)(2 * e + s);
        if (!__all_sync(0xffffffffu, mma_turn_wait(bar, ticket, p.timeout_ns, abort_flag))) { ok = false; break; }
        if (ptx::elect_one()) {
          if (pend) issue_pv<D>(o_tm, s_tm, v4 + (ve % VS) * tile4, !pend_first);
          if (use) issue_qk<D>(s_tm, q4 + qslot * tile4, k4 + ks * tile4);
        }
        __syncwarp();
        if (lane == 0) mma_turn_pass(bar, ticket);
        if (use) {
          ptx::mma_commit_elect(&bar->s_full[s]);
          issued_any = true;
        }
        if (rel_v) ptx::mma_commit_elect(&bar->v_empty[ve % VS]);
        ptx::mma_commit_elect(&bar->k_empty[ks]);
        if (pend && pend_last) ptx::mma_commit_elect(&bar->o_full[s]);
        if (use && j == last_use) ptx::mma_commit_elect(&bar->q_empty[qslot]);
        pend = use;
        pend_first = use && j == first_use;
        pend_last = use && j == last_use;
      }
    }
    if (ok && e >= 1) {
      // the last entry: its V slot and this sub-tile's pending P V
      const int ve = e - 1;
      if (!wait_all(&bar->v_full[ve % VS], (ve / VS) & 1)) ok = false;
      if (ok && pend) {
        if (!wait_all(&bar->p_full[s], pcount & 1)) {
          ok = false;
        } else {
          ++pcount;
          ptx::tc_fence_after();
          if (ptx::elect_one()) issue_pv<D>(o_tm, s_tm, v4 + (ve % VS) * tile4, !pend_first);
          __syncwarp();
          ptx::mma_commit_elect(&bar->o_full[s]);
        }
      }
      if (ok) ptx::mma_commit_elect(&bar->v_empty[ve % VS]);
    }
    if (!ok) {
      if (lane == 0) raise_error(p, bar, kErrMma);
      if (issued_any) {
        // wait (bounded) for the MMAs already issued before tensor memory is freed
        ptx::mma_commit_elect(&bar->drain[s]);
        ptx::mbar_wait_time_only(&bar->drain[s], 0, p.timeout_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    ptx::setmaxnreg_inc<kPRegsSoftmax>();
    const int s = (warp - 4) >> 2;
    const int quarter = warp & 3;  // tensor-memory lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + s * 128;
    const uint32_t o_tmem = tmem + lane_off + 256 + s * 128;
    const float sl2 = p.scale_log2;
    uint32_t count = 0;  // S tiles of this sub-tile so far (all items)
    int o_items = 0;     // items whose O_s has been read
    uint32_t sync_seq = 0;  // uses of stage_sync[s]
    uint32_t split_seq = 0;  // uses of split_sync
    bool ok = true;
    const CtaItems items = cta_items(bar);
    for (int it = items.first; ok && it < items.end; ++it) {
      const PItem pi = load_pitem(p, it);
      prefetch_pitem(p, it + 1);
      if (!check_or_abort(p, bar, pitem_ok(p, pi), kSiteItem)) {
        ok = false;
        break;
      }
      const TileList& L = pi.L;
      const SubPlan& sp = s ? pi.ip.sp1 : pi.ip.sp0;
      const int pos = sp.qt * kTile + row;
      int lo, hi;
      row_interval32(p.kind, sp.param, p.N, pos, &lo, &hi);
      if (hi > p.N - 1) hi = p.N - 1;
      const int sink_hi = (int)sink_last(p.sink_tokens, pos);  // sink keys [0, sink_hi]
      float m = -INFINITY;  // running (stale) max of scaled scores, log2 domain
      float l = 0.f;        // running sum of exp2(x - m)
      for (int jj = 0; jj < L.n; ++jj) {
        if (!pi.uses<SPLIT>(jj, s)) continue;
        const int kt = list_kt(L, jj);
        bool got = ptx::mbar_wait(&bar->s_full[s], count & 1, p.timeout_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) raise_error(p, bar, kErrSoftmax);
          ok = false;
          break;
        }
        ++count;
        ptx::tc_fence_after();
        float x[128];
        ptx::tmem_ld32(s_tmem + 0, *reinterpret_cast<float(*)[32]>(&x[0]));
        ptx::tmem_ld32(s_tmem + 32, *reinterpret_cast<float(*)[32]>(&x[32]));
        ptx::tmem_ld32(s_tmem + 64, *reinterpret_cast<float(*)[32]>(&x[64]));
        ptx::tmem_ld32(s_tmem + 96, *reinterpret_cast<float(*)[32]>(&x[96]));
        ptx::tmem_wait_ld();
        bool sees = true;  // this row sees a key of the tile
        if (MASK && sub_partial(p, sp, kt)) {
          // visible key columns of this row inside the tile: [c_lo, c_hi],
          // and the sink keys of the tile: columns [0, c_s]
          const int k0 = kt * kTile;
          const int c_lo = min(max(lo - k0, -1), 128);
          const int c_hi = min(max(hi - k0, -1), 128);
          const int c_s = min(max(sink_hi - k0, -1), 128);
          sees = mask_row(x, c_lo, c_hi, c_s);
        }
        // P = exp2(s * scale * log2e - m) into tensor memory (the stale-max
        // rule of attention_fwd.cu: m only guards against overflow)
        float ts;
        // Exponentiate against the running maximum, or against 0 for a row's
        // first visible scores (kMinTileSum).  It only guards against overflow
        // (the final normalisation uses the same m for numerator and
        // denominator), so it is kept while every P stays below 2^40; a tile that
        // breaks this, or a first tile whose visible scores all came out below
        // 2^-64, is redone below against the tile's own maximum (rare).
        const bool first = m == -INFINITY;
        ts = exp_to_tmem(x, sl2, first ? 0.f : m, s_tmem);
        bool slow = __any_sync(0xffffffffu, !(ts <= kMaxTileSum) || (first && sees && !(ts >= kMinTileSum)));
        if (slow) {
          ptx::tmem_wait_st();  // let these stores land before they are overwritten
        } else if (first && sees) {
          m = 0.f;  // the row's reference from here on
        }
        if (slow) {
          const float m_new = fmaxf(m, row_max(x) * sl2);
          const bool need_rescale = (m != -INFINITY) && (m_new > m);
          if (m == -INFINITY) m = m_new;
          if (__any_sync(0xffffffffu, need_rescale)) {
            // O_s holds this item's products so far (its P V for the
            // previous tile is done: S of this tile was committed after it)
            const float alpha = need_rescale ? ptx::ex2(m - m_new) : 1.f;
            rescale_o<D>(o_tmem, alpha);
            if (need_rescale) {
              l *= alpha;
              m = m_new;
            }
          }
          ts = exp_to_tmem(x, sl2, (m == -INFINITY) ? 0.f : m, s_tmem);
        }
        l += ts;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bar->p_full[s]);
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      // While the tensor core runs this item's last P V and the next item's
      // first S: wait for the P V, read O_s, write O / (l + exp(sink)) and
      // the LSE in caller token order.
      const bool has_o = pi.first(s) >= 0;
      const bool has_oo = pi.first(s ^ 1) >= 0;  // the other sub-tile's O of this item
      const float b2 = p.sink ? __ldg(p.sink + pi.ip.h) * kLog2e : -INFINITY;
      if (SPLIT && pi.split) {
        // Both sub-tiles hold partial (m, l, O) of the same rows: merged as
        // O = (O_0 e_0 + O_1 e_1) / (l_0 e_0 + l_1 e_1 + exp(sink)), e_s =
        // exp2(m_s - M) against the common maximum M; sub-tile 1 hands its
        // (m, l) to sub-tile 0, which forms both scales (and the LSE), and
        // each writes half of the O columns.
        bool valid = pos < p.N;
        const int64_t tok = valid ? out_token(p, pi.store, pi.perm_row, pos) : 0;
        if (kDebugChecks && tok < 0) valid = false;
        const int64_t orow = ((int64_t)pi.ip.bh * p.N + tok) * D;
        auto sync_all = [&]() {
          if (__all_sync(0xffffffffu, ptx::mbar_sync(&bar->split_sync, split_seq, p.timeout_ns, abort_flag)))
            return true;
          if (lane == 0) raise_error(p, bar, kErrEpilogue);
          return false;
        };
        // this sub-tile's O is complete; after the first barrier so is the
        // other's (its threads waited for it before arriving)
        if (has_o) {
          const bool got = ptx::mbar_wait(&bar->o_full[s], o_items & 1, p.timeout_ns, abort_flag);
          if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) raise_error(p, bar, kErrEpilogue);
            ok = false;
            break;
          }
          ++o_items;
        }
        if (s == 1) bar->xch[row] = make_float2(m, l);
        if (!sync_all()) {
          ok = false;
          break;
        }
        float2 sc;
        if (s == 0) {
          const float2 o1 = bar->xch[row];
          float lse_v;
          finalize_row(m, l, o1.x, o1.y, b2, &sc.x, &sc.y, &lse_v);
          if (valid && p.lse) p.lse[(int64_t)pi.ip.bh * p.N + tok] = lse_v;
          bar->xch[row] = sc;
        }
        if (!sync_all()) {
          ok = false;
          break;
        }
        if (s == 1) sc = bar->xch[row];
        ptx::tc_fence_after();
        const float sc_self = s ? sc.y : sc.x, sc_other = s ? sc.x : sc.y;
        const uint32_t oo_tmem = tmem + lane_off + 256 + (s ^ 1) * 128;
        constexpr int kHalf = 16 * ((D + 31) / 32);  // columns [0, kHalf) by sub-tile 0, the rest by 1
        const uint64_t o_policy = ptx::l2_policy_evict_first();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          if (s ? c0 < kHalf : c0 >= kHalf) continue;  // warp-uniform
          float ov[16];
          if (has_o) {
            ptx::tmem_ld16(o_tmem + c0, ov);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] *= sc_self;
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = 0.f;
          }
          if (has_oo) {
            float ow[16];
            ptx::tmem_ld16(oo_tmem + c0, ow);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = fmaf(ow[i], sc_other, ov[i]);
          }
          if (valid) {
            if (OUT_F32) {
              float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.o) + orow + c0);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
            } else {
              uint32_t pk[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) pk[i] = ptx::pack_bf16x2(ov[2 * i], ov[2 * i + 1]);
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + orow + c0);
              ptx::st_global_v4_hint(dst, make_uint4(pk[0], pk[1], pk[2], pk[3]), o_policy);
              ptx::st_global_v4_hint(dst + 1, make_uint4(pk[4], pk[5], pk[6], pk[7]), o_policy);
            }
          }
        }
        // neither sub-tile writes its next item's first P (which lets the
        // next P V overwrite its O) before both have read both O's
        ptx::tc_fence_before();
        if (!sync_all()) {
          ok = false;
          break;
        }
        continue;
      }
      // What does not need O comes first, while the last P V runs: the
      // row's scale, its LSE (stored) and output row, and (staged output)
      // the staging tile, free once its previous store has read it.
      float o_scale, unused, lse_v;
      finalize_row(m, l, -INFINITY, 0.f, b2, &o_scale, &unused, &lse_v);
      bool valid = pos < p.N;
      const int64_t tok = valid ? out_token(p, pi.store, pi.perm_row, pos) : 0;
      if (kDebugChecks && tok < 0) valid = false;
      const int64_t orow = ((int64_t)pi.ip.bh * p.N + tok) * D;
      if (valid && p.lse) p.lse[(int64_t)pi.ip.bh * p.N + tok] = lse_v;
      const bool staged = PG::kStage && p.o_tma;
      uint8_t* stage = sstage + s * G::kTileBytes;
      const bool leader = quarter == 0 && lane == 0;
      if (staged && has_o) {
        if (leader) ptx::bulk_wait_read_all();  // the previous store has read the tile
        if (!__all_sync(0xffffffffu, ptx::mbar_sync(&bar->stage_sync[s], sync_seq, p.timeout_ns, abort_flag))) {
          if (lane == 0) raise_error(p, bar, kErrEpilogue);
          ok = false;
          break;
        }
      }
      if (has_o) {
        bool got = ptx::mbar_wait(&bar->o_full[s], o_items & 1, p.timeout_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) raise_error(p, bar, kErrEpilogue);
          ok = false;
          break;
        }
        ++o_items;
        ptx::tc_fence_after();
      }
      if (staged) {
        // Through shared memory: each thread writes its row into this
        // sub-tile's staging tile, one thread stores the tile with TMA.
        if (has_o) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16) {
            float ov[16];
            ptx::tmem_ld16(o_tmem + c0, ov);
            ptx::tmem_wait_ld();
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) pk[i] = ptx::pack_bf16x2(ov[2 * i] * o_scale, ov[2 * i + 1] * o_scale);
            tile_put16<D>(stage, row, c0 / 8, make_uint4(pk[0], pk[1], pk[2], pk[3]));
            tile_put16<D>(stage, row, c0 / 8 + 1, make_uint4(pk[4], pk[5], pk[6], pk[7]));
          }
          ptx::fence_proxy_async_shared();  // the tile's generic writes, before the async-proxy read
          if (!__all_sync(0xffffffffu, ptx::mbar_sync(&bar->stage_sync[s], sync_seq, p.timeout_ns, abort_flag))) {
            if (lane == 0) raise_error(p, bar, kErrEpilogue);
            ok = false;
            break;
          }
          if (leader) {
            if (!store_tile<D>(p, pi.load, stage, sp.qt * kTile, pi.ip.bh, ptx::l2_policy_evict_first()))
              abort_cta(bar);
            ptx::bulk_commit_group();
          }
        }
      } else {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          float ov[16];
          if (has_o) {
            ptx::tmem_ld16(o_tmem + c0, ov);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] *= o_scale;
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = 0.f;
          }
          if (valid) {
            if (OUT_F32) {
              float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.o) + orow + c0);
#pragma unroll
              for (int i = 0; i < 4; ++i) dst[i] = make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
            } else {
              // written once, not re-read: evicted from L2 first
              const uint64_t o_policy = ptx::l2_policy_evict_first();
              uint32_t pk[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) pk[i] = ptx::pack_bf16x2(ov[2 * i], ov[2 * i + 1]);
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + orow + c0);
              ptx::st_global_v4_hint(dst, make_uint4(pk[0], pk[1], pk[2], pk[3]), o_policy);
              ptx::st_global_v4_hint(dst + 1, make_uint4(pk[4], pk[5], pk[6], pk[7]), o_policy);
            }
          }
        }
      }
    }
  }

  // the output tiles' TMA stores (issued by one thread per sub-tile) have
  // completed before the CTA and its shared memory go away
  if (PGeo<D, OUT_F32>::kStage && p.o_tma && warp >= 4 && (warp & 3) == 0 && lane == 0) ptx::bulk_wait_all();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int D, bool F32>
size_t persist_smem_for() {
  using G = Geo<D>;
  using PG = PGeo<D, F32>;
  return (size_t)(PG::kQSlots + 2 * G::kStages + PG::kStageTiles) * G::kTileBytes + sizeof(PBarriers) + 1024;
}

template <int D, bool F32, bool MASK, bool SPLIT = false>
cudaError_t launch_persist_one(const FwdParams& p, int grid, cudaStream_t stream) {
  const size_t smem = persist_smem_for<D, F32>();
  auto kern = attention_persist_kernel<D, F32, MASK, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.after_prepass ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

size_t attention_persist_smem_bytes(int d) {
  switch (d) {
    case 32: return persist_smem_for<32, false>();
    case 64: return persist_smem_for<64, false>();
    case 80: return persist_smem_for<80, false>();
    case 96: return persist_smem_for<96, false>();
    case 128: return persist_smem_for<128, false>();
    default: return 0;
  }
}

cudaError_t launch_attention_persist(const FwdParams& p, int d, bool out_f32, int grid, cudaStream_t stream) {
  if (p.n_items <= 0) return cudaSuccess;
  if (grid > p.n_items) grid = p.n_items;
  // bf16 launches without PARTIAL tiles run the build without the boundary
  // mask; launches with split items the build with their merge (masked)
#define MATTN_CASE(DD)                                                                           \
  case DD:                                                                                       \
    if (p.has_split)                                                                             \
      return out_f32 ? launch_persist_one<DD, true, true, true>(p, grid, stream)                 \
                     : launch_persist_one<DD, false, true, true>(p, grid, stream);               \
    return out_f32 ? launch_persist_one<DD, true, true>(p, grid, stream)                         \
                   : (p.no_partial ? launch_persist_one<DD, false, false>(p, grid, stream)       \
                                   : launch_persist_one<DD, false, true>(p, grid, stream));
  switch (d) {
    MATTN_CASE(32)
    MATTN_CASE(64)
    MATTN_CASE(80)
    MATTN_CASE(96)
    MATTN_CASE(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef MATTN_CASE
}

}  // namespace mattn
