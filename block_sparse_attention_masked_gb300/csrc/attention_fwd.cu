// Masked attention forward for sm_103a: TMA-staged tiles, tcgen05 MMAs with
// tensor-memory accumulators, warp-specialised online softmax.
//
// What one CTA computes, in one of two schedules:
//   paired: query rows [256*pair, 256*pair + 256) of one (batch, head), as
//     two 128-row query sub-tiles s = 0, 1 that share the staged K/V tiles
//     (for masks whose neighbouring query tiles see mostly the same keys);
//   split: query rows [128*qt, 128*qt + 128), its key tiles dealt out
//     alternately to two sub-tile pipelines s = 0, 1 that keep separate
//     running (m, l, O) and are merged at the end (for masks whose
//     neighbouring query tiles share few key tiles, e.g. 128-blocks).
// For every key tile kt a sub-tile takes (plan_rules.h),
//     S_s  = Q_s K_kt^T                        (tcgen05.mma, smem x smem -> TMEM)
//     P_s  = exp2(S_s * scale*log2e - m_s)     (softmax warps, online max m_s)
//     O_s += P_s V_kt                          (tcgen05.mma, P from TMEM, V from smem)
// with the running sum l_s; at the end O_s / (l_s + exp(sink)) and the
// log-sum-exp are written out (SHS slides Eq. 1 for the sink; RRAttention
// Eq. 1-2 for the skipped block pairs; the FlashAttention idea of the Vision
// transformers lesson -- tile, fuse the softmax, never materialise N x N).
//
// Roles (384 threads):
//   warp 0        TMA producer: Q once, then K tiles into their ring
//   warp 1        tensor-memory allocator; MMA issuer of sub-tile 0
//   warp 2        MMA issuer of sub-tile 1
//   warp 3        TMA producer of the V ring
//   warps 4..7    softmax + epilogue of sub-tile 0 (one query row per thread)
//   warps 8..11   softmax + epilogue of sub-tile 1
// Tensor memory (512 columns x 128 lanes, fp32):
//   [  0,128) S_0 (P_0 as bf16 pairs in its first 64 columns)
//   [128,256) S_1 / P_1
//   [256,384) O_0      [384,512) O_1
// Synchronisation is by mbarriers only; every wait is bounded in time and
// gives up by raising a CTA-wide abort flag and a device error bit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attention_tiles.cuh"
#include "kernel_params.h"
#include "plan_rules.h"
#include "ptx.cuh"
#include "tile_mma.cuh"

namespace mattn {

namespace {

constexpr int kThreads = 384;
// Registers per thread after setmaxnreg: producer / MMA-issuer warpgroup and the
// two softmax warpgroups (their sum times 128 equals the launch budget).
constexpr uint32_t kRegsControl = 72;
constexpr uint32_t kRegsSoftmax = 216;
static_assert(kRegsControl + 2 * kRegsSoftmax == 3 * 168, "register split must match the launch budget");

struct Barriers {
  uint64_t q_full[2];
  uint64_t k_full[3], k_empty[3];
  uint64_t v_full[3], v_empty[3];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_final[2];
  uint64_t never;       // self-test: nothing ever arrives here
  uint64_t drain[2];    // MMA drain on abort, one per issuer
  uint32_t tmem_base;
  int abort_flag;
  uint32_t mma_turn;    // ticket of the MMA group that may be issued next
  int head_store, head_perm_row;  // the head's store mode and explicit-order row, for the epilogue
  float sink_log2;                // the head's sink logit in the log2 domain (-inf: none)
  int list_n[3];        // block kind: entries of the CTA's key-tile list, and per sub-tile
  TileList tl;          // the CTA's key-tile list (read by every role from shared memory)
  float xch[2][3][kTile];  // split schedule: per sub-tile (m, l, tile count) of each row
};

// Block kind: one warp writes the CTA's entries to `list` (ascending key
// tiles; the union of the sub-tiles' kept tiles at or below their
// diagonals) and counts[0..2] = their number and the entries sub-tile 0 and
// sub-tile 1 use.
// Lanes take 64-bit words of the bitmap rows, a warp prefix sum of their
// tile counts gives each lane its first output slot, and each lane then
// writes its own words' tiles.
__device__ __forceinline__ void build_block_list(const FwdParams& p, int2 item, const ItemPlan& ip, uint32_t* list,
                                                 int* counts, int lane) {
  const int c = p.block_c;
  int used0 = 0, used1 = 0;
  const int km0 = ip.sp0.rows ? ip.sp0.ktmax : -1;
  const int km1 = ip.sp1.rows ? ip.sp1.ktmax : -1;
  const int km = km0 > km1 ? km0 : km1;
  int base = 0;
  if (km >= 0) {
    const uint64_t* row0 = km0 >= 0 ? global_row(p, item, 0) : nullptr;
    const uint64_t* row1 = km1 >= 0 ? global_row(p, item, 1) : nullptr;
    const int nb0 = km0 >= 0 ? km0 / c : -1, nb1 = km1 >= 0 ? km1 / c : -1;  // last block of each sub-tile
    const int nbm = km / c;
    const int nwords = nbm / 64 + 1;
    auto keep_upto = [](int w, int nbl) -> uint64_t {  // bits n <= nbl of word w
      const int hi = nbl - w * 64;
      return hi < 0 ? 0ull : (hi >= 63 ? ~0ull : ((2ull << hi) - 1ull));
    };
    for (int w0 = 0; w0 < nwords; w0 += 32) {
      const int w = w0 + lane;
      uint64_t u0 = 0, u1 = 0;
      if (w < nwords) {
        if (row0) u0 = row0[w] & keep_upto(w, nb0);
        if (row1) u1 = row1[w] & keep_upto(w, nb1);
      }
      const uint64_t U = u0 | u1;
      // tiles from this word: c per kept block, fewer for the block holding km
      int cnt = __popcll(U) * c;
      if (w == nbm / 64 && ((U >> (nbm % 64)) & 1ull)) cnt -= c - (km - nbm * c + 1);
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      int pos = base + incl - cnt;
      uint64_t bits = U;
      while (bits) {
        const int bpos = __ffsll((long long)bits) - 1;
        bits &= bits - 1ull;
        const int n = w * 64 + bpos;
        for (int i = 0; i < c; ++i) {
          const int kt = n * c + i;
          if (kt > km) break;
          const uint32_t use0 = (((u0 >> bpos) & 1ull) && kt <= km0) ? 1u : 0u;
          const uint32_t use1 = (((u1 >> bpos) & 1ull) && kt <= km1) ? 1u : 0u;
          // (debug builds: never past the list's capacity; the kernel checks the count)
          if (!kDebugChecks || pos < kMaxList) list[pos] = (uint32_t)kt | (use0 << 30) | (use1 << 31);
          ++pos;
          used0 += (int)use0;
          used1 += (int)use1;
        }
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    used0 += __shfl_xor_sync(0xffffffffu, used0, off);
    used1 += __shfl_xor_sync(0xffffffffu, used1, off);
  }
  if (lane == 0) {
    counts[0] = base;
    counts[1] = used0;
    counts[2] = used1;
  }
}

// Split schedule: O columns [0, kOHalf) are written by sub-tile 0's threads,
// [kOHalf, D) by sub-tile 1's (whole 16-column loads).
template <int D>
__host__ __device__ constexpr int kOHalf() {
  return 16 * ((D + 31) / 32);
}

// The CTA's Q tiles: one per sub-tile that has key tiles (split: the one
// query tile both pipelines share).  Issued by the K producer thread.
template <int D>
__device__ __forceinline__ void issue_q_loads(const FwdParams& p, const ItemPlan& ip, const TileList& L, int load_mode,
                                              uint8_t* sq, Barriers* bar) {
  using G = Geo<D>;
  const CUtensorMap* mq = load_mode == kLoadColumnMajor   ? p.cq
                          : load_mode == kLoadBlock2x2Row ? p.bq
                          : load_mode == kLoadBlock2x2Col ? p.bcq
                                                          : p.tq;
  ptx::prefetch_tmap(&mq[0]);
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const SubPlan& sp = s ? ip.sp1 : ip.sp0;
    if (!list_has(L, s, p.split) || (p.split && s == 1)) continue;  // split: one Q tile for both pipelines
    ptx::mbar_arrive_expect_tx(&bar->q_full[s], G::kTileBytes);
    if (!load_tile<D>(p, false, load_mode, sq + s * G::kTileBytes, &bar->q_full[s], sp.qt * kTile, ip.bh,
                      ptx::l2_policy_evict_first()))
      abort_cta(bar);
  }
}

template <int D, bool OUT_F32, bool MASK>
__global__ void __launch_bounds__(kThreads, 1) attention_fwd_kernel(const __grid_constant__ FwdParams p) {
  using G = Geo<D>;
  constexpr int KS = G::kStages;
  constexpr int VS = G::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = base;
  uint8_t* sk = sq + 2 * G::kTileBytes;
  uint8_t* sv = sk + KS * G::kTileBytes;
  Barriers* bar = reinterpret_cast<Barriers*>(sv + VS * G::kTileBytes);
  uint32_t* list_e = reinterpret_cast<uint32_t*>(bar + 1);  // block kind: [kMaxList] key-tile entries
  volatile int* abort_flag = &bar->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int2 item = p.items[blockIdx.x];
  // debug builds: a work item outside the launch's heads and query tiles
  // ends the CTA here, before any barrier or allocation
  if (!item_in_range(p, blockIdx.x, item)) {
    if (threadIdx.x == 0) debug_check(p.err, false, kSiteItem);
    if (kDebugChecks) return;
  }
  // the head's row of the per-head table (param, load, store, perm_row) in
  // one load
  const int4 head_row = __ldg(reinterpret_cast<const int4*>(p.head_info) + item.x % p.H);
  const ItemPlan ip = make_plan(p, item, head_row.x);
  const int load_mode = head_row.y;
  if (p.kind == kBlockSparse && warp == 2) build_block_list(p, item, ip, list_e, bar->list_n, lane);
  // Q tiles and the first ring's K tiles requested before the set-up below
  // (interval kinds, whose key-tile list needs no shared state), so that
  // their DRAM latency overlaps it; the K producer continues from k_early
  int k_early = 0;
  bool q_early = false;
  if (threadIdx.x == 96) bar->sink_log2 = p.sink ? __ldg(p.sink + item.x % p.H) * kLog2e : -INFINITY;

  if (threadIdx.x == 0) {
    // After the reorder pre-pass: the CTA's bounded waits below must not run
    // while the pre-pass is still copying, so every thread is held at the
    // first CTA barrier until its copies are complete.
    if (p.after_prepass) asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bar->q_full[s], 1);
      ptx::mbar_init(&bar->s_full[s], 1);
      ptx::mbar_init(&bar->p_full[s], 128);
      ptx::mbar_init(&bar->o_final[s], 1);
    }
    for (int i = 0; i < 3; ++i) {
      ptx::mbar_init(&bar->k_full[i], 1);
      // released by a commit from each MMA issuer (paired) or from the one
      // issuer the entry is dealt to (split)
      ptx::mbar_init(&bar->k_empty[i], p.split ? 1 : 2);
      ptx::mbar_init(&bar->v_full[i], 1);
      ptx::mbar_init(&bar->v_empty[i], p.split ? 1 : 2);
    }
    ptx::mbar_init(&bar->never, 1);
    ptx::mbar_init(&bar->drain[0], 1);
    ptx::mbar_init(&bar->drain[1], 1);
    bar->abort_flag = 0;
    bar->mma_turn = 0;
    bar->head_store = head_row.z;
    bar->head_perm_row = head_row.w;
    ptx::fence_barrier_init();
    if (p.kind != kBlockSparse) {
      ptx::fence_proxy_async_shared();
      const TileList L0 = make_list(p, ip, nullptr, nullptr);
      issue_q_loads<D>(p, ip, L0, load_mode, sq, bar);
      q_early = true;
      k_early = L0.n < KS ? L0.n : KS;
      const uint64_t keep = ptx::l2_policy_evict_last();
      for (int j = 0; j < k_early; ++j) {  // fresh ring slots: nothing to wait for
        const int kt = list_kt(L0, j);
        if (!check_or_abort(p, bar, key_tile_ok(p, kt), kSiteKeyTile)) break;
        ptx::mbar_arrive_expect_tx(&bar->k_full[j], G::kTileBytes);
        if (!load_tile<D>(p, true, load_mode, sk + j * G::kTileBytes, &bar->k_full[j], kt * kTile, ip.bh_kv, keep)) {
          abort_cta(bar);
          break;
        }
      }
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bar->tmem_base, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bar->tmem_base;

  if (threadIdx.x == 0) {
    bar->tl = make_list(p, ip, list_e, bar->list_n);
    // debug builds: a block list past its capacity is dropped (nothing read
    // beyond the entries written)
    if (p.kind == kBlockSparse && !check_or_abort(p, bar, bar->list_n[0] <= kMaxList, kSiteKeyTile)) {
      bar->tl.n = 0;
      bar->tl.use_n0 = bar->tl.use_n1 = 0;
    }
  }
  __syncthreads();
  const TileList& L = bar->tl;

  // Registers: 384 threads launched at 168 each; the producer / MMA
  // warpgroup gives up to kRegsControl so that each softmax warpgroup can hold
  // a full 128-column score row (kRegsControl + 2 * kRegsSoftmax = 3 * 168).  Each
  // role branch starts with its own budget change.
  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ producers
    // Warp 0 loads Q and the K ring, warp 3 the V ring, each walking the
    // CTA's key-tile list in order: a K load never queues behind a V slot
    // that is still being read (V is released only after P V, K already
    // after S).
    ptx::setmaxnreg_dec<kRegsControl>();
    if (lane == 0) {
      const bool is_k = warp == 0;
      // K and V tiles are re-read by the other query tiles of the head (keep
      // them in L2); a Q tile is read by this CTA alone
      const uint64_t keep = ptx::l2_policy_evict_last();
      if (is_k && !q_early) issue_q_loads<D>(p, ip, L, load_mode, sq, bar);
      uint64_t* empty = is_k ? bar->k_empty : bar->v_empty;
      uint64_t* full = is_k ? bar->k_full : bar->v_full;
      uint8_t* ring = is_k ? sk : sv;
      constexpr int S = KS;
      static_assert(KS == VS, "one ring depth for K and V");
      for (int j = is_k ? k_early : 0; j < L.n; ++j) {
        const int kt = list_kt(L, j);
        const int slot = j % S;
        if (debug_aborted(abort_flag) || !check_or_abort(p, bar, key_tile_ok(p, kt), kSiteKeyTile)) break;
        if (!ptx::mbar_wait(&empty[slot], ((j / S) & 1) ^ 1, p.timeout_ns, abort_flag)) {
          raise_error(p, bar, kErrProducer);
          break;
        }
        ptx::mbar_arrive_expect_tx(&full[slot], G::kTileBytes);
        const bool issued =
            is_k ? load_tile<D>(p, true, load_mode, ring + slot * G::kTileBytes, &full[slot], kt * kTile, ip.bh_kv,
                                keep)
                 : load_v_tile<D>(p, load_mode, ring + slot * G::kTileBytes, &full[slot], kt * kTile, ip.bh_kv, keep);
        if (!issued) {
          abort_cta(bar);
          break;
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA's shared memory goes away
        uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 2000000ull) { }
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues the MMAs of sub-tile 0, warp 2 those of sub-tile 1, so
    // that neither waits behind the other's softmax.  Both walk the CTA's
    // key-tile list in order.  Paired: every K / V ring slot is released by
    // one commit from each issuer (the empty barriers count 2); an issuer
    // that skips an entry still waits for the slot to be filled before
    // releasing it, which keeps the two issuers' arrivals in phase order.
    // Split: entry j belongs to issuer j % 2 alone, which releases it; the
    // other issuer never touches it.  The whole warp runs the loop
    // (warp-uniform control flow and operand arithmetic, which the compiler
    // keeps in uniform registers); one elected lane issues each tcgen05
    // instruction.
    ptx::setmaxnreg_dec<kRegsControl>();
    const int s = warp - 1;
    auto wait_all = [&](uint64_t* b, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(b, parity, p.timeout_ns, abort_flag));
    };
    auto fail = [&]() {
      if (lane == 0) raise_error(p, bar, kErrMma);
    };
    bool ok = true;
    if (p.self_test_timeout && s == 0) {
      // nothing ever arrives on this barrier: exercises the bounded-wait path
      if (!wait_all(&bar->never, 0)) {
        if (lane == 0) raise_error(p, bar, kErrSelfTest);
        ok = false;
      }
    }
    const int qs = p.split ? 0 : s;  // Q tile this sub-tile multiplies
    if (ok && list_has(L, s, p.split) && !wait_all(&bar->q_full[qs], 0)) {
      fail();
      ok = false;
    }
    ptx::tc_fence_after();
    constexpr uint32_t tile4 = G::kTileBytes >> 4;  // descriptor start-address units
    const uint32_t q4 = (ptx::smem_addr(sq) >> 4) + qs * tile4;
    const uint32_t k4 = ptx::smem_addr(sk) >> 4;
    const uint32_t v4 = ptx::smem_addr(sv) >> 4;
    const uint32_t s_tm = tmem + s * 128;
    const uint32_t o_tm = tmem + 256 + s * 128;
    bool pend = false, first = true, issued_any = false;
    int pe = 0;  // entry whose P V is pending
    uint32_t pcount = 0;
    int j = 0;
    if (ok) {
      // split: this issuer's entries are j = s, s + 2, ...
      for (j = p.split ? s : 0; j < L.n; j += p.split ? 2 : 1) {
        const bool use = p.split || list_uses(L, j, s);
        const int ks = j % KS;
        // the V slot read and released at this step: the previous entry
        // (paired), the pending product's entry (split)
        const bool rel_v = p.split ? pend : (j >= 1);
        const int ve = p.split ? pe : j - 1;
        // every input of this step first: V and K (both arrive through the
        // async proxy the MMA reads, so no tcgen05 fence), then -- last, as
        // it is the one that arrives last -- this sub-tile's pending P
        if (rel_v && !wait_all(&bar->v_full[ve % VS], (ve / VS) & 1)) {
          fail(); ok = false; break;
        }
        if (!wait_all(&bar->k_full[ks], (j / KS) & 1)) {
          fail(); ok = false; break;
        }
        if (pend) {
          if (!wait_all(&bar->p_full[s], pcount & 1)) {
            fail(); ok = false; break;
          }
          ++pcount;
          ptx::tc_fence_after();
        }
        // then the group P V(pe) + S(j), in ticket order so that the two
        // sub-tiles' groups run back to back instead of interleaving
        // (interleaved groups finish together and the two softmaxes then run
        // in lockstep while the tensor core idles)
        const uint32_t ticket = p.split ? (uint32_t)j : (uint32_t)(2 * j + s);
        if (!__all_sync(0xffffffffu, mma_turn_wait(bar, ticket, p.timeout_ns, abort_flag))) {
          fail(); ok = false; break;
        }
        if (ptx::elect_one()) {
          if (pend) issue_pv<D>(o_tm, s_tm, v4 + (ve % VS) * tile4, !first);
          if (use) issue_qk<D>(s_tm, q4, k4 + ks * tile4);
        }
        __syncwarp();
        if (pend) {
          first = false;
          pend = false;
        }
        if (lane == 0) mma_turn_pass(bar, ticket);
        // commits after the turn has passed: each tracks this thread's own
        // MMAs only, so the other issuer need not wait for them
        if (use) {
          ptx::mma_commit_elect(&bar->s_full[s]);
          pend = true;
          pe = j;
          issued_any = true;
        }
        if (rel_v) ptx::mma_commit_elect(&bar->v_empty[ve % VS]);
        ptx::mma_commit_elect(&bar->k_empty[ks]);
      }
    }
    if (ok && (p.split ? pend : j >= 1)) {
      const int ve = p.split ? pe : j - 1;
      if (!wait_all(&bar->v_full[ve % VS], (ve / VS) & 1)) {
        fail(); ok = false;
      }
      if (ok && pend) {
        if (!wait_all(&bar->p_full[s], pcount & 1)) {
          fail(); ok = false;
        } else {
          ++pcount;
          ptx::tc_fence_after();
          if (ptx::elect_one()) issue_pv<D>(o_tm, s_tm, v4 + (ve % VS) * tile4, !first);
          __syncwarp();
          first = false;
          pend = false;
        }
      }
      if (ok) ptx::mma_commit_elect(&bar->v_empty[ve % VS]);
    }
    if (ok && issued_any) ptx::mma_commit_elect(&bar->o_final[s]);
    if (!ok && issued_any) {
      // wait (bounded) for the MMAs already issued before tensor memory is freed
      ptx::mma_commit_elect(&bar->drain[s]);
      ptx::mbar_wait_time_only(&bar->drain[s], 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    ptx::setmaxnreg_inc<kRegsSoftmax>();
    const int s = (warp - 4) >> 2;
    const int quarter = warp & 3;  // tensor-memory lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + s * 128;
    const uint32_t o_tmem = tmem + lane_off + 256 + s * 128;
    const SubPlan sp = s ? ip.sp1 : ip.sp0;
    const int64_t pos = (int64_t)sp.qt * kTile + row;
    const int param = head_row.x;
    int64_t lo, hi;
    row_interval(p.kind, param, p.N, pos, &lo, &hi);
    if (hi > p.N - 1) hi = p.N - 1;
    const int64_t sink_hi = sink_last(p.sink_tokens, pos);  // sink keys [0, sink_hi]
    const float sl2 = p.scale_log2;

    float m = -INFINITY;  // running (stale) max of scaled scores, log2 domain
    float l = 0.f;        // running sum of exp2(x - m) in fp32
    int count = 0;  // key tiles this sub-tile has processed
    bool ok = true;
    // entries of the CTA's list this sub-tile (split: pipeline) multiplies
    for (int jj = p.split ? s : 0; jj < L.n; jj += p.split ? 2 : 1) {
      if (!p.split && !list_uses(L, jj, s)) continue;
      const int kt = list_kt(L, jj);
      bool got = ptx::mbar_wait(&bar->s_full[s], count & 1, p.timeout_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) raise_error(p, bar, kErrSoftmax);
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      float x[128];
      ptx::tmem_ld32(s_tmem + 0, *reinterpret_cast<float(*)[32]>(&x[0]));
      ptx::tmem_ld32(s_tmem + 32, *reinterpret_cast<float(*)[32]>(&x[32]));
      ptx::tmem_ld32(s_tmem + 64, *reinterpret_cast<float(*)[32]>(&x[64]));
      ptx::tmem_ld32(s_tmem + 96, *reinterpret_cast<float(*)[32]>(&x[96]));
      ptx::tmem_wait_ld();
      bool sees = true;  // this row sees a key of the tile
      const bool partial = MASK && sub_partial(p, sp, kt);
      if (partial) {
        // visible key columns of this row inside the tile: [c_lo, c_hi]
        const int64_t k0 = (int64_t)kt * kTile;
        const int c_lo = (int)(lo - k0 < -1 ? -1 : (lo - k0 > 128 ? 128 : lo - k0));
        const int c_hi = (int)(hi - k0 < -1 ? -1 : (hi - k0 > 128 ? 128 : hi - k0));
        // and the sink keys of the tile: columns [0, c_s]
        const int c_s = (int)(sink_hi - k0 < -1 ? -1 : (sink_hi - k0 > 128 ? 128 : sink_hi - k0));
        sees = mask_row(x, c_lo, c_hi, c_s);
      }
      // P = exp2(s * scale * log2e - m) into tensor memory.  tcgen05.ld / st
      // are warp-collective, so every branch below is taken by whole warps
      // (each lane applying its own factors).
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
        // tile maximum first (also the first tile of a row)
        const float m_new = fmaxf(m, row_max(x) * sl2);
        const bool need_rescale = (m != -INFINITY) && (m_new > m);
        if (m == -INFINITY) m = m_new;  // nothing accumulated yet (all earlier P were zero)
        if (__any_sync(0xffffffffu, need_rescale)) {
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
      ++count;
    }

    // ---------------------------------------------------------- epilogue
    // Paired: each sub-tile writes its own rows.  Split: both sub-tiles hold
    // partial (m, l, O) of the same rows; they exchange (m, l, count) and
    // each writes half of the O columns, O = (O_0 e_0 + O_1 e_1) / (l_0 e_0 +
    // l_1 e_1 + exp(sink)) with e_s = exp2(m_s - M) against the common
    // maximum M (the merge of two online-softmax states).
    float m_o = -INFINITY, l_o = 0.f;
    int count_o = 0;
    if (p.split) {
      bar->xch[s][0][row] = m;
      bar->xch[s][1][row] = l;
      bar->xch[s][2][row] = (float)count;
      asm volatile("bar.sync 1, 256;" ::: "memory");  // the eight softmax warps
      m_o = bar->xch[s ^ 1][0][row];
      l_o = bar->xch[s ^ 1][1][row];
      count_o = (int)bar->xch[s ^ 1][2][row];
    }
    if (ok && sp.rows) {
      // O accumulators this thread reads: its own; when split, also the other's
      bool have_o = false, have_oo = false;
      auto wait_final = [&](int t) {
        bool got = ptx::mbar_wait(&bar->o_final[t], 0, p.timeout_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) raise_error(p, bar, kErrEpilogue);
          return false;
        }
        ptx::tc_fence_after();
        return true;
      };
      if (count > 0) {
        have_o = wait_final(s);
        ok = have_o;
      }
      if (ok && p.split && count_o > 0) {
        have_oo = wait_final(s ^ 1);
        ok = have_oo;
      }
      if (ok) {
        // O = sum of P V / (l + exp(sink)) with every term taken against
        // the common maximum; the LSE from the same normaliser
        float o_scale, oo_scale, lse_v;
        finalize_row(m, l, m_o, l_o, bar->sink_log2, &o_scale, &oo_scale, &lse_v);
        bool valid = pos < p.N;
        const int store_mode = bar->head_store;
        const int perm_row = bar->head_perm_row;
        const int64_t tok = valid ? out_token(p, store_mode, perm_row, pos) : 0;
        if (kDebugChecks && tok < 0) valid = false;
        const int64_t orow = ((int64_t)ip.bh * p.N + tok) * D;
        // columns written: all (paired); this sub-tile's half (split)
        const int c_begin = (p.split && s == 1) ? kOHalf<D>() : 0;
        const int c_end = (p.split && s == 0) ? kOHalf<D>() : D;
        const uint32_t oo_tmem = tmem + lane_off + 256 + (s ^ 1) * 128;
        const uint64_t o_policy = ptx::l2_policy_evict_first();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          if (c0 < c_begin || c0 >= c_end) continue;  // warp-uniform
          float ov[16];
          if (have_o) {
            ptx::tmem_ld16(o_tmem + c0, ov);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] *= o_scale;
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = 0.f;
          }
          if (have_oo) {
            float ow[16];
            ptx::tmem_ld16(oo_tmem + c0, ow);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = fmaf(ow[i], oo_scale, ov[i]);
          }
          if (valid) {
            // O is written once and never re-read here: evict it from L2
            // first, so that it does not push out the K / V tiles other
            // query tiles of the head still read
            if (OUT_F32) {
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<float*>(p.o) + orow + c0);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                ptx::st_global_v4_hint(dst + i,
                                       make_uint4(__float_as_uint(ov[4 * i]), __float_as_uint(ov[4 * i + 1]),
                                                  __float_as_uint(ov[4 * i + 2]), __float_as_uint(ov[4 * i + 3])),
                                       o_policy);
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
        if (valid && p.lse && (!p.split || s == 0)) p.lse[(int64_t)ip.bh * p.N + tok] = lse_v;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// Tile-plan dump: one thread per (head, query tile) walks the same rules the
// attention kernel walks and writes (h, qt, kt, class) quadruples.
__global__ void plan_dump_kernel(const PlanDumpParams p) {
  const int nt = (p.N + kTile - 1) / kTile;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.H * nt) return;
  const int h = idx / nt, qt = idx % nt;
  const int param = p.head_info[h * 4 + kHeadParam];
  int32_t* out = p.out + ((int64_t)h * nt + qt) * nt * 4;
  int n = 0;
  if (p.kind == kBlockSparse) {
    const uint64_t* bits = p.block_bits + (int64_t)((p.block_heads == 1) ? 0 : h) * p.block_nb * p.block_wpr;
    for (int kt = block_next_kt(bits, p.block_wpr, p.block_c, qt, 0, qt); kt != kNoTile;
         kt = block_next_kt(bits, p.block_wpr, p.block_c, qt, kt + 1, qt)) {
      out[4 * n + 0] = h; out[4 * n + 1] = qt; out[4 * n + 2] = kt;
      out[4 * n + 3] = block_tile_class(qt, kt, p.N);
      ++n;
    }
  } else {
    KRange r = interval_krange(p.kind, param, p.N, qt);
    const int ns = sink_tiles(p.sink_tokens, p.N, qt);
    for (int kt = 0; kt < ns && kt < r.lo; ++kt) {  // sink tiles below the window
      out[4 * n + 0] = h; out[4 * n + 1] = qt; out[4 * n + 2] = kt;
      out[4 * n + 3] = sink_window_tile_class(param, p.sink_tokens, p.N, qt, kt);
      ++n;
    }
    for (int kt = r.lo; kt <= r.hi; ++kt) {
      out[4 * n + 0] = h; out[4 * n + 1] = qt; out[4 * n + 2] = kt;
      out[4 * n + 3] = p.sink_tokens > 0 ? sink_window_tile_class(param, p.sink_tokens, p.N, qt, kt)
                                         : interval_tile_class(r, kt);
      ++n;
    }
  }
  p.counts[idx] = n;
}

// Reorder to sequence positions (and round fp32 to bf16): one thread per 8
// elements of one destination row, for q, k and v (blockIdx.y).  K and V
// rows of query head h are read from K / V head h / kv_group, so that the
// copies have one head per query head.
__global__ void gather_kernel(const GatherParams p) {
  // the attention grid that reads these copies may be scheduled now
  asm volatile("griddepcontrol.launch_dependents;");
  const int t = blockIdx.y;
  const int64_t vec_per_row = p.d / 8;
  const int64_t total = (int64_t)p.B * p.H * p.N * vec_per_row;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int64_t row = i / vec_per_row;  // (b*H + h)*N + pos
  const int c8 = (int)(i - row * vec_per_row) * 8;
  const int64_t pos = row % p.N;
  const int64_t bh = row / p.N;
  const int h = (int)(bh % p.H);
  const int store_mode = p.head_info[h * 4 + kHeadStore];
  const int perm_row = p.head_info[h * 4 + kHeadPermRow];
  // debug builds: the head's explicit-order row and the token it holds
  if (!debug_check(p.err, store_mode != kStoreExplicit || (perm_row >= 0 && perm_row < p.n_perm), kSiteItem)) return;
  const int64_t tok = token_at(store_mode, p.grid_rows, p.grid_cols,
                               store_mode == kStoreExplicit ? p.perm + (int64_t)perm_row * p.N : nullptr, pos);
  if (!debug_check(p.err, tok >= 0 && tok < p.N, kSiteOrder)) return;
  const int64_t src_bh = t == 0 ? bh : (bh / p.H) * (p.H / p.kv_group) + h / p.kv_group;
  const int64_t src_off = (src_bh * p.N + tok) * p.d + c8;
  uint4 out;
  if (p.src_f32) {
    const float4* s = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.src[t]) + src_off);
    float4 a = s[0], b = s[1];
    out.x = ptx::pack_bf16x2(a.x, a.y);
    out.y = ptx::pack_bf16x2(a.z, a.w);
    out.z = ptx::pack_bf16x2(b.x, b.y);
    out.w = ptx::pack_bf16x2(b.z, b.w);
  } else {
    out = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.src[t]) + src_off);
  }
  *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.dst[t]) + row * p.d + c8) = out;
}

template <int D, bool F32, bool MASK>
cudaError_t launch_one(const FwdParams& p, cudaStream_t stream) {
  const size_t smem = attention_smem_bytes(D);
  auto kern = attention_fwd_kernel<D, F32, MASK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (!p.after_prepass) {
    kern<<<p.n_items, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
  }
  // After the reorder pre-pass: a programmatic dependent launch, so that the
  // CTAs are resident when the copies are done (thread 0 waits in
  // griddepcontrol.wait for them before the CTA's first barrier).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_items);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int D>
size_t smem_for() {
  using G = Geo<D>;
  size_t bytes = (size_t)(2 + 2 * G::kStages) * G::kTileBytes + sizeof(Barriers) +
                 kMaxList * sizeof(uint32_t) + 1024;
  // at least ~120 KiB so that one CTA owns an SM (and all of its tensor memory)
  return bytes < 120 * 1024 ? 120 * 1024 : bytes;
}

}  // namespace

size_t attention_smem_bytes(int d) {
  switch (d) {
    case 32: return smem_for<32>();
    case 64: return smem_for<64>();
    case 80: return smem_for<80>();
    case 96: return smem_for<96>();
    case 128: return smem_for<128>();
    default: return 0;
  }
}

cudaError_t launch_attention(const FwdParams& p, int d, bool out_f32, cudaStream_t stream) {
  if (p.n_items <= 0) return cudaSuccess;
  // bf16 launches without PARTIAL tiles run the build without the boundary
  // mask: its code, even when never taken, slows the exponential pass
#define MATTN_CASE(DD)                                                                                 \
  case DD:                                                                                             \
    return out_f32 ? launch_one<DD, true, true>(p, stream)                                             \
                   : (p.no_partial ? launch_one<DD, false, false>(p, stream) : launch_one<DD, false, true>(p, stream));
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

cudaError_t launch_plan_dump(const PlanDumpParams& p, cudaStream_t stream) {
  const int nt = (p.N + kTile - 1) / kTile;
  const int total = p.H * nt;
  if (total == 0) return cudaSuccess;
  plan_dump_kernel<<<(total + 127) / 128, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream) {
  const int64_t total = (int64_t)p.B * p.H * p.N * (p.d / 8);
  if (total == 0) return cudaSuccess;
  dim3 grid((unsigned)((total + 255) / 256), 3);
  gather_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mattn
