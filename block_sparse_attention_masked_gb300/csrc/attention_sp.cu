// Single-pipeline masked attention forward for sm_103a: one 128-row query
// tile per CTA, S double-buffered in tensor memory.  It serves head dim 256
// (the speed-test layout of the Bifocal page, "Details": query and
// key/value heads of dimension 256), where an O accumulator takes 256 of the
// 512 tensor-memory columns so that the two-sub-tile kernel does not fit,
// and, on request, head dim 128.  With KT keys per key tile:
//   S_j  = Q K_j^T        M128 N=KT K=D   (D/16 MMAs of K16, smem x smem -> TMEM)
//   P_j  = exp2(S_j * scale*log2e - m)    (softmax warps, one row per thread)
//   O   += P_j V_j        M128 N=D  K=KT  (KT/16 MMAs of K16, P from TMEM)
// (D, KT) = (256, 64) or (128, 128).  S is double-buffered, so the product
// of tile j + 1 runs while the softmax works on tile j:
//   issue order  S_0, S_1, [P_0] PV_0, S_2, [P_1] PV_1, S_3, ...
// Tensor memory: S_0 [0, KT), S_1 [KT, 2 KT) (P as bf16 pairs in the first
// KT/2 columns of its S), O [256, 256 + D).  Shared memory: Q (D/4 KB), K
// and V rings of two KT x D tiles each, and for block-sparse masks the
// CTA's key-tile list.
//
// The key tiles are the 128-key tiles of the plan (plan_rules.h: interval
// masks incl. sink tokens, or the block-selection matrix), each taken as
// 128 / KT pieces; the mask is applied on the pieces of PARTIAL tiles.
// Inputs are read in raster order (the host reorders other orders into a
// position-order copy first).
//
// Roles (256 threads): warp 0 TMA producer; warp 1 tensor-memory allocator
// and MMA issuer; warps 4..7 softmax and epilogue (one query row per
// thread); warps 2, 3 idle.  Every wait is bounded in time and gives up by
// raising a CTA-wide abort flag and a device error bit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attention_tiles.cuh"
#include "kernel_params.h"
#include "plan_rules.h"
#include "ptx.cuh"

namespace mattn {
namespace {

constexpr int kThreadsD256 = 256;
constexpr int kStagesD256 = 2;

// Shared-memory geometry: Q and K / V tiles as 64-column chunks of 128-byte
// rows (128-byte swizzle), as TMA writes them.
template <int D, int KT>
struct SpGeo {
  static_assert(D % 64 == 0 && D <= 256 && (KT == 64 || KT == 128), "single-pipeline geometry");
  static constexpr int kQChunk = kTile * 64 * 2;  // 16 KB
  static constexpr int kQBytes = (D / 64) * kQChunk;
  static constexpr int kKVChunk = KT * 64 * 2;
  static constexpr int kKVBytes = (D / 64) * kKVChunk;
  static constexpr int kSub = kTile / KT;         // key tiles per 128-key plan tile
};

constexpr float kLog2eX = 1.4426950408889634f;
constexpr float kLn2X = 0.6931471805599453f;
constexpr float kMaxTileSumX = 1099511627776.0f;  // 2^40, as in the d <= 128 kernel
constexpr float kMinTileSumX = 5.421010862427522e-20f;  // 2^-64: a row's first tile against 0, as there

struct BarD256 {
  uint64_t q_full;
  uint64_t k_full[kStagesD256], k_empty[kStagesD256];
  uint64_t v_full[kStagesD256], v_empty[kStagesD256];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done;  // one phase per P V product
  uint64_t o_final;
  uint64_t drain;
  uint64_t never;    // self-test: nothing ever arrives here
  uint32_t tmem_base;
  int abort_flag;
  int list_n;        // block kind: entries of the CTA's key-tile list
};

__device__ __forceinline__ uint64_t dsc(uint32_t lo, uint32_t hi) { return ((uint64_t)hi << 32) | lo; }

// The CTA's 128-key tiles: interval masks, the sink tiles below the window
// then the window; block masks, a list in shared memory.
struct ListD256 {
  int n, na, lo;
  KRange r;
  int param;
  const uint32_t* e;  // block kind: the entries
};

__device__ __forceinline__ int list_kt_d256(const ListD256& L, int j) {
  return L.e ? (int)L.e[j] : (j < L.na ? j : L.lo + (j - L.na));
}

// Block kind: one warp writes the key tiles of query tile qt (ascending; kept
// blocks at or below the diagonal, tiles up to qt) to `list`, their number
// to *count.  Lanes take 64-bit words of the bitmap row; a warp prefix sum
// of their tile counts gives each lane its first output slot.
__device__ __forceinline__ void build_list_sp(const FwdParams& p, int h, int qt, uint32_t* list, int* count,
                                              int lane) {
  const int c = p.block_c;
  const int hb = (p.block_heads == 1) ? 0 : h;
  const uint64_t* row = p.block_bits + ((int64_t)hb * p.block_nb + qt / c) * p.block_wpr;
  const int nbl = qt / c;  // last admissible block
  const int nwords = nbl / 64 + 1;
  int base = 0;
  for (int w0 = 0; w0 < nwords; w0 += 32) {
    const int w = w0 + lane;
    uint64_t u = 0;
    if (w < nwords) {
      const int top = nbl - w * 64;
      u = row[w] & (top >= 63 ? ~0ull : ((2ull << top) - 1ull));
    }
    int cnt = __popcll(u) * c;
    if (w == nbl / 64 && ((u >> (nbl % 64)) & 1ull)) cnt -= c - (qt - nbl * c + 1);
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    int pos = base + incl - cnt;
    uint64_t bits = u;
    while (bits) {
      const int bpos = __ffsll((long long)bits) - 1;
      bits &= bits - 1ull;
      const int n = w * 64 + bpos;
      for (int i = 0; i < c; ++i) {
        const int kt = n * c + i;
        if (kt > qt) break;
        // (debug builds: never past the list's capacity; the kernel checks the count)
        if (!kDebugChecks || pos < kBlockListMax) list[pos] = (uint32_t)kt;
        ++pos;
      }
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) *count = base;
}

__device__ __forceinline__ void fail_d256(const FwdParams& p, BarD256* bar, uint32_t bit) {
  *reinterpret_cast<volatile int*>(&bar->abort_flag) = 1;
  atomicOr(p.err, bit);
}

// Debug checks (debug_check in kernel_params.h): a failed one also raises
// the CTA's abort flag; always true in the product build.
__device__ __forceinline__ bool check_d256(const FwdParams& p, BarD256* bar, bool ok, uint32_t site) {
  if (debug_check(p.err, ok, site)) return true;
  *reinterpret_cast<volatile int*>(&bar->abort_flag) = 1;
  return false;
}

template <int D, int KT>
__global__ void __launch_bounds__(kThreadsD256, 1) attention_sp_kernel(const __grid_constant__ FwdParams p) {
  using SG = SpGeo<D, KT>;
  constexpr int kD = D, kKT = KT;
  constexpr int kQBytes = SG::kQBytes, kQChunk = SG::kQChunk;
  constexpr int kKVBytes = SG::kKVBytes, kKVChunk = SG::kKVChunk;
  constexpr int kSub = SG::kSub;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = base;
  uint8_t* sk = sq + kQBytes;
  uint8_t* sv = sk + kStagesD256 * kKVBytes;
  BarD256* bar = reinterpret_cast<BarD256*>(sv + kStagesD256 * kKVBytes);
  uint32_t* list_e = reinterpret_cast<uint32_t*>(bar + 1);  // block kind: [kBlockListMax] key tiles
  volatile int* abort_flag = &bar->abort_flag;
  const bool block = p.kind == kBlockSparse;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int2 item = p.items[blockIdx.x];  // (b * H + h, query tile)
  // debug builds: a work item outside the launch's heads and query tiles
  // ends the CTA here, before any barrier or allocation
  if (!((int)blockIdx.x < p.n_items && item.x >= 0 && item.x < p.B * p.H && item.y >= 0 &&
        (int64_t)item.y * kTile < p.N)) {
    if (threadIdx.x == 0) debug_check(p.err, false, kSiteItem);
    if (kDebugChecks) return;
  }
  const int bh = item.x, qt = item.y;
  const int h = bh % p.H, b = bh / p.H;
  const int bh_kv = b * p.H_kv + h / p.kv_group;
  const int param = p.head_info[h * 4 + kHeadParam];
  if (block && warp == 2) build_list_sp(p, h, qt, list_e, &bar->list_n, lane);
  // key-tile list (128-key tiles) of this query tile
  ListD256 L;
  L.param = param;
  L.e = nullptr;
  L.r.lo = 1; L.r.hi = 0; L.r.flo = 0; L.r.fhi = -1;
  if (!block) L.r = interval_krange(p.kind, param, p.N, qt);
  L.lo = L.r.lo;
  L.n = L.r.hi >= L.r.lo ? L.r.hi - L.r.lo + 1 : 0;
  L.na = 0;
  const int ns = block ? 0 : sink_tiles(p.sink_tokens, p.N, qt);
  if (ns > 0 && L.n > 0) {
    if (ns >= L.lo) {
      const int hi = L.r.hi > ns - 1 ? L.r.hi : ns - 1;
      L.lo = 0;
      L.n = hi + 1;
    } else {
      L.na = ns;
      L.n += ns;
    }
  }

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar->q_full, 1);
    for (int i = 0; i < kStagesD256; ++i) {
      ptx::mbar_init(&bar->k_full[i], 1);
      ptx::mbar_init(&bar->k_empty[i], 1);
      ptx::mbar_init(&bar->v_full[i], 1);
      ptx::mbar_init(&bar->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bar->s_full[i], 1);
      ptx::mbar_init(&bar->p_full[i], 128);
    }
    ptx::mbar_init(&bar->pv_done, 1);
    ptx::mbar_init(&bar->o_final, 1);
    ptx::mbar_init(&bar->drain, 1);
    ptx::mbar_init(&bar->never, 1);
    bar->abort_flag = 0;
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
  if (block) {
    L.e = list_e;
    L.n = bar->list_n;
    if (kDebugChecks && L.n > kBlockListMax) {  // debug builds: a list past its capacity is dropped
      if (threadIdx.x == 0) check_d256(p, bar, false, kSiteKeyTile);
      L.n = 0;
    }
  }
  // key tiles of KT keys: plan tile j gives pieces kSub j .. kSub j + kSub - 1
  // (the last ones only when they hold keys < N)
  auto half_key0 = [&](int t) { return list_kt_d256(L, t / kSub) * kTile + (t % kSub) * kKT; };
  int n_half = 0;
  if (L.n > 0) {
    const int last_kt = list_kt_d256(L, L.n - 1);
    n_half = kSub * L.n - ((kSub == 2 && last_kt * kTile + kKT >= p.N) ? 1 : 0);
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_half > 0) {
      const uint64_t keep = ptx::l2_policy_evict_last();
      const uint64_t once = ptx::l2_policy_evict_first();
      ptx::mbar_arrive_expect_tx(&bar->q_full, kQBytes);
      // (debug builds: tile coordinates inside the [B*H][N][d] and [B*H_kv][N][d] views)
      if (check_d256(p, bar, (int64_t)qt * kTile < p.N && bh >= 0 && bh < p.B * p.H, kSiteLoad)) {
#pragma unroll
        for (int c = 0; c < kD / 64; ++c)
          ptx::tma_load_3d_hint(sq + c * kQChunk, &p.tq[0], &bar->q_full, c * 64, qt * kTile, bh, once);
      }
      // K and V halves in list order, interleaved so that neither ring
      // waits behind the other
      for (int t = 0; t < n_half; ++t) {
        const int slot = t % kStagesD256;
        const uint32_t par = ((t / kStagesD256) & 1) ^ 1;
        const int k0 = half_key0(t);
        if (kDebugChecks) {
          const int kt = list_kt_d256(L, t / kSub);
          if (*abort_flag || !check_d256(p, bar, kt >= 0 && (int64_t)kt * kTile < p.N, kSiteKeyTile) ||
              !check_d256(p, bar, k0 >= 0 && k0 < p.N && bh_kv >= 0 && bh_kv < p.B * p.H_kv, kSiteLoad))
            break;
        }
        if (!ptx::mbar_wait(&bar->k_empty[slot], par, p.timeout_ns, abort_flag)) {
          fail_d256(p, bar, kErrProducer);
          break;
        }
        ptx::mbar_arrive_expect_tx(&bar->k_full[slot], kKVBytes);
#pragma unroll
        for (int c = 0; c < kD / 64; ++c)
          ptx::tma_load_3d_hint(sk + slot * kKVBytes + c * kKVChunk, &p.tk[0], &bar->k_full[slot], c * 64, k0,
                                bh_kv, keep);
        if (!ptx::mbar_wait(&bar->v_empty[slot], par, p.timeout_ns, abort_flag)) {
          fail_d256(p, bar, kErrProducer);
          break;
        }
        ptx::mbar_arrive_expect_tx(&bar->v_full[slot], kKVBytes);
#pragma unroll
        for (int c = 0; c < kD / 64; ++c)
          ptx::tma_load_3d_hint(sv + slot * kKVBytes + c * kKVChunk, &p.tv[0], &bar->v_full[slot], c * 64, k0,
                                bh_kv, keep);
      }
      if (*abort_flag) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 2000000ull) { }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    auto wait_all = [&](uint64_t* b, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(b, parity, p.timeout_ns, abort_flag));
    };
    bool ok = n_half > 0;
    bool issued = false;
    if (p.self_test_timeout && ok && !wait_all(&bar->never, 0)) {  // nothing arrives here: exercises the abort path
      if (lane == 0) fail_d256(p, bar, kErrSelfTest);
      ok = false;
    }
    if (ok && !wait_all(&bar->q_full, 0)) {
      if (lane == 0) fail_d256(p, bar, kErrMma);
      ok = false;
    }
    ptx::tc_fence_after();
    const uint32_t q4 = ptx::smem_addr(sq) >> 4;
    const uint32_t k4 = ptx::smem_addr(sk) >> 4;
    const uint32_t v4 = ptx::smem_addr(sv) >> 4;
    constexpr uint32_t hi128 = ptx::smem_desc_hi(1024, ptx::kSw128);
    constexpr uint32_t lbo_k = 1u << 16;  // unused for swizzled K-major operands
    constexpr uint32_t idesc_qk = ptx::idesc_bf16(128, kKT, 0);
    constexpr uint32_t idesc_pv = ptx::idesc_bf16(128, kD, 1);
    constexpr uint32_t lbo_v = (uint32_t)(kKVChunk >> 4) << 16;  // 64-column atoms of V lie a chunk apart
    auto issue_s = [&](int t) {  // S_{t % 2} = Q K_t^T
      const int slot = t % kStagesD256;
      const uint32_t s_tm = tmem + (t & 1) * kKT;
      if (ptx::elect_one()) {
        uint32_t acc = 0;
#pragma unroll 1
        for (int step = 0; step < kD / 16; ++step) {
          const uint32_t qo = (uint32_t)(((step >> 2) * kQChunk + (step & 3) * 32) >> 4) + lbo_k;
          const uint32_t ko = (uint32_t)((slot * kKVBytes + (step >> 2) * kKVChunk + (step & 3) * 32) >> 4) + lbo_k;
          ptx::mma_ss(s_tm, dsc(q4 + qo, hi128), dsc(k4 + ko, hi128), idesc_qk, acc);
          acc = 1;
        }
      }
      __syncwarp();
      ptx::mma_commit_elect(&bar->s_full[t & 1]);
      ptx::mma_commit_elect(&bar->k_empty[slot]);
    };
    auto take_k = [&](int t) {
      return wait_all(&bar->k_full[t % kStagesD256], (t / kStagesD256) & 1);
    };
    if (ok) {
      for (int t = 0; t < 2 && t < n_half; ++t) {
        if (!take_k(t)) { ok = false; break; }
        issue_s(t);
        issued = true;
      }
    }
    for (int t = 0; ok && t < n_half; ++t) {
      // P_t ready, V_t landed: O += P_t V_t
      if (!wait_all(&bar->p_full[t & 1], (t >> 1) & 1) ||
          !wait_all(&bar->v_full[t % kStagesD256], (t / kStagesD256) & 1)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const int slot = t % kStagesD256;
      if (ptx::elect_one()) {
        const uint32_t p_tm = tmem + (t & 1) * kKT;
        const uint32_t hiv = ptx::smem_desc_hi(8 * 128, ptx::kSw128);
#pragma unroll 1
        for (int k = 0; k < kKT / 16; ++k) {
          // 16 keys: 8 tensor-memory columns of P, 16 rows (2 KB) of V
          const uint32_t vo = (uint32_t)((slot * kKVBytes + k * 16 * 128) >> 4) + lbo_v;
          ptx::mma_ts(tmem + 256, p_tm + k * 8, dsc(v4 + vo, hiv), idesc_pv, (t > 0 || k > 0) ? 1u : 0u);
        }
      }
      __syncwarp();
      ptx::mma_commit_elect(&bar->pv_done);
      ptx::mma_commit_elect(&bar->v_empty[slot]);
      // the next product into the S buffer this P V has read
      if (t + 2 < n_half) {
        if (!take_k(t + 2)) { ok = false; break; }
        issue_s(t + 2);
      }
    }
    if (!ok && n_half > 0 && lane == 0) fail_d256(p, bar, kErrMma);
    if (ok && n_half > 0) ptx::mma_commit_elect(&bar->o_final);
    if (!ok && issued) {
      ptx::mma_commit_elect(&bar->drain);
      ptx::mbar_wait_time_only(&bar->drain, 0, p.timeout_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t o_tmem = tmem + lane_off + 256;
    const int64_t pos = (int64_t)qt * kTile + row;
    int64_t lo, hi;
    row_interval(p.kind, param, p.N, pos, &lo, &hi);
    if (hi > p.N - 1) hi = p.N - 1;
    const int64_t sink_hi = sink_last(p.sink_tokens, pos);
    const float sl2 = p.scale_log2;
    const float b2 = p.sink ? p.sink[h] * kLog2eX : -INFINITY;
    float m = -INFINITY, l = 0.f;
    bool ok = n_half > 0;
    for (int t = 0; ok && t < n_half; ++t) {
      const uint32_t s_tmem = tmem + lane_off + (t & 1) * kKT;
      const bool got = ptx::mbar_wait(&bar->s_full[t & 1], (t >> 1) & 1, p.timeout_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) fail_d256(p, bar, kErrSoftmax);
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      float x[kKT];
#pragma unroll
      for (int c0 = 0; c0 < kKT; c0 += 32) ptx::tmem_ld32(s_tmem + c0, *reinterpret_cast<float(*)[32]>(&x[c0]));
      ptx::tmem_wait_ld();
      const int kt = list_kt_d256(L, t / kSub);
      const int64_t k0 = (int64_t)half_key0(t);
      const bool partial = block ? block_tile_class(qt, kt, p.N) == kTilePartial
                           : p.sink_tokens > 0 ? sink_window_tile_class(param, p.sink_tokens, p.N, qt, kt) == kTilePartial
                                               : interval_tile_class(L.r, kt) == kTilePartial;
      bool sees = true;  // this row sees a key of the tile
      if (partial || k0 + kKT > p.N) {
        const int c_lo = (int)(lo - k0 < -1 ? -1 : (lo - k0 > kKT ? kKT : lo - k0));
        const int c_hi = (int)(hi - k0 < -1 ? -1 : (hi - k0 > kKT ? kKT : hi - k0));
        const int c_s = (int)(sink_hi - k0 < -1 ? -1 : (sink_hi - k0 > kKT ? kKT : sink_hi - k0));
        sees = mask_row(x, c_lo, c_hi, c_s);
      }
      // exponentiate against the running (stale) maximum, or against 0 for a
      // row's first visible scores; a tile whose row sum passes 2^40, or a
      // first tile whose visible scores sum below 2^-64, is redone against
      // its own maximum, rescaling O once the previous P V (which adds into
      // O) is done
      auto exp_pass = [&](float mref, float& sum) {
        const float2 sl2v = make_float2(sl2, sl2);
        const float2 negm = make_float2(-mref, -mref);
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c0 = 0; c0 < kKT; c0 += 64) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float2 tt = ptx::ffma2(make_float2(x[c0 + 2 * i], x[c0 + 2 * i + 1]), sl2v, negm);
            const float2 pp = make_float2(ptx::ex2(tt.x), ptx::ex2(tt.y));
            pk[i] = ptx::pack_bf16x2(pp.x, pp.y);
            acc[i & 1] = ptx::fadd2(acc[i & 1], pp);
          }
          ptx::tmem_st32(s_tmem + c0 / 2, pk);
        }
        const float2 a = ptx::fadd2(acc[0], acc[1]);
        sum = a.x + a.y;
      };
      float ts = 0.f;
      const bool first = m == -INFINITY;
      exp_pass(first ? 0.f : m, ts);
      bool slow = __any_sync(0xffffffffu, !(ts <= kMaxTileSumX) || (first && sees && !(ts >= kMinTileSumX)));
      if (slow) {
        ptx::tmem_wait_st();
      } else if (first && sees) {
        m = 0.f;  // the row's reference from here on
      }
      if (slow) {
        float mx = x[0];
#pragma unroll
        for (int c = 1; c < kKT; ++c) mx = fmaxf(mx, x[c]);
        const float m_new = fmaxf(m, mx * sl2);
        const bool need_rescale = (m != -INFINITY) && (m_new > m);
        if (m == -INFINITY) m = m_new;
        if (__any_sync(0xffffffffu, need_rescale)) {
          // P_{t-1} V_{t-1} adds into O: wait for it (the (t-1)-th phase of
          // pv_done; S_t being ready means P_{t-2} V_{t-2} is done, so the
          // barrier is at most one phase ahead of the one waited for)
          const bool pv = ptx::mbar_wait(&bar->pv_done, (t - 1) & 1, p.timeout_ns, abort_flag);
          if (!__all_sync(0xffffffffu, pv)) {
            if (lane == 0) fail_d256(p, bar, kErrSoftmax);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const float alpha = need_rescale ? ptx::ex2(m - m_new) : 1.f;
#pragma unroll 1
          for (int c0 = 0; c0 < kD; c0 += 32) {
            float ov[32];
            ptx::tmem_ld32(o_tmem + c0, ov);
            ptx::tmem_wait_ld();
            uint32_t ou[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) ou[i] = __float_as_uint(ov[i] * alpha);
            ptx::tmem_st32(o_tmem + c0, ou);
          }
          if (need_rescale) {
            l *= alpha;
            m = m_new;
          }
        }
        exp_pass(m == -INFINITY ? 0.f : m, ts);
      }
      l += ts;
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bar->p_full[t & 1]);
    }
    // ---------------------------------------------------------- epilogue
    const bool valid = pos < p.N;
    if (ok && n_half > 0) {
      const bool got = ptx::mbar_wait(&bar->o_final, 0, p.timeout_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) fail_d256(p, bar, kErrEpilogue);
        ok = false;
      }
      ptx::tc_fence_after();
    }
    if (ok || n_half == 0) {
      const float M = fmaxf(m, b2);
      float o_scale = 0.f, lse_v = -INFINITY;
      if (M != -INFINITY) {
        const float em = (m == -INFINITY) ? 0.f : ptx::ex2(m - M);
        const float lf = l * em + ((b2 == -INFINITY) ? 0.f : ptx::ex2(b2 - M));
        if (lf > 0.f) {
          o_scale = em / lf;
          lse_v = (M + ptx::lg2(lf)) * kLn2X;
        }
      }
      // caller token of this position (the inputs were reordered to
      // positions; the output goes back to token order)
      const int store_mode = p.head_info[h * 4 + kHeadStore];
      const int perm_row = p.head_info[h * 4 + kHeadPermRow];
      // debug builds: the head's explicit-order row and the token it holds
      // are checked; a row that fails is not stored
      bool store = valid &&
                   debug_check(p.err, store_mode != kStoreExplicit || (perm_row >= 0 && perm_row < p.n_perm), kSiteItem);
      const int64_t tok = !store ? pos
                                 : token_at(store_mode, p.grid_rows, p.grid_cols,
                                            store_mode == kStoreExplicit ? p.perm + (int64_t)perm_row * p.N : nullptr,
                                            pos);
      store = store && debug_check(p.err, tok >= 0 && tok < p.N, kSiteOrder);
      const int64_t orow = ((int64_t)bh * p.N + tok) * kD;
#pragma unroll 1
      for (int c0 = 0; c0 < kD; c0 += 32) {
        float ov[32];
        if (n_half > 0) {
          ptx::tmem_ld32(o_tmem + c0, ov);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0.f;
        }
        if (store) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.o) + orow + c0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(ov[4 * i] * o_scale, ov[4 * i + 1] * o_scale, ov[4 * i + 2] * o_scale,
                                   ov[4 * i + 3] * o_scale);
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = ptx::pack_bf16x2(ov[2 * i] * o_scale, ov[2 * i + 1] * o_scale);
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + orow + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      }
      if (store && p.lse) p.lse[(int64_t)bh * p.N + tok] = lse_v;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int D, int KT>
size_t sp_smem_bytes() {
  return 1024 + (size_t)SpGeo<D, KT>::kQBytes + 2 * kStagesD256 * (size_t)SpGeo<D, KT>::kKVBytes + sizeof(BarD256) +
         kBlockListMax * sizeof(uint32_t);
}

template <int D, int KT>
cudaError_t launch_sp(const FwdParams& p, cudaStream_t stream) {
  const size_t smem = sp_smem_bytes<D, KT>();
  auto kern = attention_sp_kernel<D, KT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<p.n_items, kThreadsD256, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int attention_sp_key_tile(int d) { return d == 256 ? 64 : 128; }

cudaError_t launch_attention_sp(const FwdParams& p, int d, cudaStream_t stream) {
  if (p.n_items <= 0) return cudaSuccess;
  switch (d) {
    case 128: return launch_sp<128, 128>(p, stream);
    case 256: return launch_sp<256, 64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mattn
