// Masked attention forward for sm_103a: TMA-staged tiles, tcgen05 MMAs with
// tensor-memory accumulators, warp-specialised online softmax.
//
// What one CTA computes: query rows [256*pair, 256*pair + 256) of one
// (batch, head), as two 128-row query sub-tiles s = 0, 1 that share the
// staged K/V tiles.  For every key tile kt the mask touches (plan_rules.h),
//     S_s  = Q_s K_kt^T                        (tcgen05.mma, smem x smem -> TMEM)
//     P_s  = exp2(S_s * scale*log2e - m_s)     (softmax warps, online max m_s)
//     O_s += P_s V_kt                          (tcgen05.mma, P from TMEM, V from smem)
// with the running sum l_s; at the end O_s / (l_s + exp(sink)) and the
// log-sum-exp are written out (SHS slides Eq. 1 for the sink; RRAttention
// Eq. 1-2 for the skipped block pairs; the FlashAttention idea of the Vision
// transformers lesson -- tile, fuse the softmax, never materialise N x N).
//
// Roles (384 threads):
//   warp 0        TMA producer: Q_0, Q_1 once, then K/V tiles into rings
//   warp 1        tensor-memory allocator and single-thread MMA issuer
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

#include "kernel_params.h"
#include "plan_rules.h"
#include "ptx.cuh"

namespace mattn {

namespace {

constexpr int kThreads = 384;
constexpr int kNoTile = 0x7fffffff;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// A new row maximum replaces the running one only when it exceeds it by more
// than 2^8 (log2 domain); below that the stale maximum is kept, which is
// exact because O and l share it, and P stays <= 256 (fine in bf16 / fp32).
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct Geo {
  static_assert(D == 32 || D == 64 || D == 80 || D == 96 || D == 128, "unsupported head dim");
  static constexpr int kChunks = D / 64;                  // 64-column chunks, 128-byte swizzle
  static constexpr int kRem = D % 64;                     // 0, 16 or 32 trailing columns
  static constexpr int kChunkBytes = kTile * 64 * 2;      // 16 KiB
  static constexpr int kRemBytes = kTile * kRem * 2;
  static constexpr int kTileBytes = kChunks * kChunkBytes + kRemBytes;
  static constexpr int kStages = (D >= 96) ? 2 : 3;       // K ring and V ring depth
  static constexpr uint32_t kRemSwizzle = (kRem == 16) ? ptx::kSw32 : ptx::kSw64;
  static constexpr int kRemRowBytes = kRem * 2;           // 32 or 64
  static_assert(kTileBytes % 1024 == 0, "tiles must keep 1 KiB alignment");
};

struct Barriers {
  uint64_t q_full[2];
  uint64_t k_full[3], k_empty[3];
  uint64_t v_full[3], v_empty[3];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_final[2];
  uint64_t never;       // self-test: nothing ever arrives here
  uint64_t drain;       // MMA drain on abort
  uint32_t tmem_base;
  int abort_flag;
};

// Work description of one CTA, computed identically by every thread.
struct ItemPlan {
  int bh, h, b;
  int qt[2];
  bool rows[2];         // sub-tile has query rows (< N)
  bool has_tiles[2];    // and at least one key tile
  KRange r[2];          // interval kinds
  int ktmax[2];         // block kind: last admissible key tile
  const uint64_t* bits; // block kind: this head's bitmap
};

__device__ __forceinline__ int sub_next(const FwdParams& p, const ItemPlan& ip, int s, int from) {
  if (!ip.rows[s]) return kNoTile;
  if (p.kind == kBlockSparse) {
    return block_next_kt(ip.bits, p.block_wpr, p.block_c, ip.qt[s], from, ip.ktmax[s]);
  }
  int kt = from > ip.r[s].lo ? from : ip.r[s].lo;
  return kt <= ip.r[s].hi ? kt : kNoTile;
}

__device__ __forceinline__ bool sub_uses(const FwdParams& p, const ItemPlan& ip, int s, int kt) {
  if (!ip.rows[s]) return false;
  if (p.kind == kBlockSparse) {
    return kt <= ip.ktmax[s] && block_bit(ip.bits, p.block_wpr, ip.qt[s] / p.block_c, kt / p.block_c);
  }
  return kt >= ip.r[s].lo && kt <= ip.r[s].hi;
}

__device__ __forceinline__ bool sub_partial(const FwdParams& p, const ItemPlan& ip, int s, int kt) {
  if (p.kind == kBlockSparse) return block_tile_class(ip.qt[s], kt, p.N) == kTilePartial;
  return interval_tile_class(ip.r[s], kt) == kTilePartial;
}

__device__ __forceinline__ int union_next(const FwdParams& p, const ItemPlan& ip, int from) {
  int a = sub_next(p, ip, 0, from);
  int c = sub_next(p, ip, 1, from);
  return a < c ? a : c;
}

__device__ __forceinline__ ItemPlan make_plan(const FwdParams& p, int item) {
  ItemPlan ip;
  int2 it = p.items[item];
  ip.bh = it.x;
  ip.h = it.x % p.H;
  ip.b = it.x / p.H;
  const int nt = (p.N + kTile - 1) / kTile;
  const int param = p.head_info[ip.h * 4 + kHeadParam];
  ip.bits = nullptr;
  if (p.kind == kBlockSparse) {
    int hb = (p.block_heads == 1) ? 0 : ip.h;
    ip.bits = p.block_bits + (int64_t)hb * p.block_nb * p.block_wpr;
  }
  for (int s = 0; s < 2; ++s) {
    ip.qt[s] = 2 * it.y + s;
    ip.rows[s] = ip.qt[s] < nt;
    ip.ktmax[s] = ip.qt[s] < nt ? ip.qt[s] : nt - 1;
    if (p.kind != kBlockSparse) ip.r[s] = interval_krange(p.kind, param, p.N, ip.qt[s]);
    else { ip.r[s].lo = 0; ip.r[s].hi = -1; ip.r[s].flo = 0; ip.r[s].fhi = -1; }
  }
  for (int s = 0; s < 2; ++s) ip.has_tiles[s] = sub_next(p, ip, s, 0) != kNoTile;
  return ip;
}

__device__ __forceinline__ void raise_error(const FwdParams& p, Barriers* bar, uint32_t bit) {
  *reinterpret_cast<volatile int*>(&bar->abort_flag) = 1;
  atomicOr(p.err, bit);
}

// TMA load of one 128-row tile (all d columns) starting at sequence position p0.
template <int D>
__device__ __forceinline__ void load_tile(const FwdParams& p, const CUtensorMap* raster, const CUtensorMap* colmaj,
                                          bool column_major, uint8_t* dst, uint64_t* bar, int p0, int bh) {
  using G = Geo<D>;
  if (!column_major) {
#pragma unroll
    for (int c = 0; c < G::kChunks; ++c) ptx::tma_load_3d(dst + c * G::kChunkBytes, &raster[0], bar, c * 64, p0, bh);
    if (G::kRem) ptx::tma_load_3d(dst + G::kChunks * G::kChunkBytes, &raster[1], bar, 0, p0, bh);
  } else {
    // position p = c * rows + r holds token r * cols + c; a 128-position tile is
    // one grid column c, rows r0 .. r0 + 127 (rows % 128 == 0 is required).
    const int col = p0 / p.grid_rows;
    const int r0 = p0 - col * p.grid_rows;
#pragma unroll
    for (int c = 0; c < G::kChunks; ++c)
      ptx::tma_load_4d(dst + c * G::kChunkBytes, &colmaj[0], bar, c * 64, col, r0, bh);
    if (G::kRem) ptx::tma_load_4d(dst + G::kChunks * G::kChunkBytes, &colmaj[1], bar, 0, col, r0, bh);
  }
}

// S = Q K^T for one sub-tile: D/16 MMAs of M128 N128 K16, both operands K-major.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint32_t q_smem, uint32_t k_smem) {
  using G = Geo<D>;
  constexpr uint32_t idesc = ptx::idesc_bf16(128, 128, 0);
  int step = 0;
#pragma unroll
  for (int c = 0; c < G::kChunks; ++c) {
#pragma unroll
    for (int k = 0; k < 4; ++k, ++step) {
      uint32_t off = c * G::kChunkBytes + k * 32;
      uint64_t a = ptx::smem_desc(q_smem + off, 16, 1024, ptx::kSw128);
      uint64_t b = ptx::smem_desc(k_smem + off, 16, 1024, ptx::kSw128);
      ptx::mma_ss(s_tmem, a, b, idesc, step > 0);
    }
  }
  if (G::kRem) {
#pragma unroll
    for (int k = 0; k < G::kRem / 16; ++k, ++step) {
      uint32_t off = G::kChunks * G::kChunkBytes + k * 32;
      uint64_t a = ptx::smem_desc(q_smem + off, 16, 8 * G::kRemRowBytes, G::kRemSwizzle);
      uint64_t b = ptx::smem_desc(k_smem + off, 16, 8 * G::kRemRowBytes, G::kRemSwizzle);
      ptx::mma_ss(s_tmem, a, b, idesc, step > 0);
    }
  }
}

// O += P V for one sub-tile: P (128 x 128 keys, bf16 pairs in TMEM) is the
// A operand; V (keys x d, d contiguous) is an MN-major B operand.  One MMA
// per 16 keys and per column chunk.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem, bool accumulate) {
  using G = Geo<D>;
  constexpr uint32_t idesc64 = ptx::idesc_bf16(128, 64, 1);
  constexpr uint32_t idescR = ptx::idesc_bf16(128, G::kRem ? G::kRem : 16, 1);
#pragma unroll
  for (int k = 0; k < kTile / 16; ++k) {
    const uint32_t acc = (accumulate || k > 0) ? 1u : 0u;
    const uint32_t a = p_tmem + k * 8;  // 16 bf16 keys = 8 columns
#pragma unroll
    for (int c = 0; c < G::kChunks; ++c) {
      uint64_t bdesc = ptx::smem_desc(v_smem + c * G::kChunkBytes + k * 16 * 128, G::kChunkBytes, 1024, ptx::kSw128);
      ptx::mma_ts(o_tmem + c * 64, a, bdesc, idesc64, acc);
    }
    if (G::kRem) {
      uint64_t bdesc = ptx::smem_desc(v_smem + G::kChunks * G::kChunkBytes + k * 16 * G::kRemRowBytes,
                                      G::kRemBytes, 8 * G::kRemRowBytes, G::kRemSwizzle);
      ptx::mma_ts(o_tmem + G::kChunks * 64, a, bdesc, idescR, acc);
    }
  }
}

__device__ __forceinline__ int64_t token_of(const FwdParams& p, int store_mode, int perm_row, int64_t pos) {
  if (store_mode == kStoreColumnMajor) {
    int64_t c = pos / p.grid_rows;
    int64_t r = pos - c * p.grid_rows;
    return r * p.grid_cols + c;
  }
  if (store_mode == kStoreExplicit) return p.perm[(int64_t)perm_row * p.N + pos];
  return pos;
}

template <int D, bool OUT_F32>
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
  volatile int* abort_flag = &bar->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bar->q_full[s], 1);
      ptx::mbar_init(&bar->s_full[s], 1);
      ptx::mbar_init(&bar->p_full[s], 128);
      ptx::mbar_init(&bar->o_final[s], 1);
    }
    for (int i = 0; i < 3; ++i) {
      ptx::mbar_init(&bar->k_full[i], 1);
      ptx::mbar_init(&bar->k_empty[i], 1);
      ptx::mbar_init(&bar->v_full[i], 1);
      ptx::mbar_init(&bar->v_empty[i], 1);
    }
    ptx::mbar_init(&bar->never, 1);
    ptx::mbar_init(&bar->drain, 1);
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

  const ItemPlan ip = make_plan(p, blockIdx.x);
  const int load_mode = p.head_info[ip.h * 4 + kHeadLoad];
  const bool colmaj = load_mode == kLoadColumnMajor;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const CUtensorMap* mq = colmaj ? p.cq : p.tq;
      ptx::prefetch_tmap(&mq[0]);
      for (int s = 0; s < 2; ++s) {
        if (!ip.has_tiles[s]) continue;
        ptx::mbar_arrive_expect_tx(&bar->q_full[s], G::kTileBytes);
        load_tile<D>(p, p.tq, p.cq, colmaj, sq + s * G::kTileBytes, &bar->q_full[s], ip.qt[s] * kTile, ip.bh);
      }
      int j = 0;
      for (int kt = union_next(p, ip, 0); kt != kNoTile; kt = union_next(p, ip, kt + 1), ++j) {
        const int ks = j % KS, vs = j % VS;
        if (!ptx::mbar_wait(&bar->k_empty[ks], ((j / KS) & 1) ^ 1, p.timeout_ns, abort_flag)) {
          raise_error(p, bar, kErrProducer);
          break;
        }
        ptx::mbar_arrive_expect_tx(&bar->k_full[ks], G::kTileBytes);
        load_tile<D>(p, p.tk, p.ck, colmaj, sk + ks * G::kTileBytes, &bar->k_full[ks], kt * kTile, ip.bh);
        if (!ptx::mbar_wait(&bar->v_empty[vs], ((j / VS) & 1) ^ 1, p.timeout_ns, abort_flag)) {
          raise_error(p, bar, kErrProducer);
          break;
        }
        ptx::mbar_arrive_expect_tx(&bar->v_full[vs], G::kTileBytes);
        load_tile<D>(p, p.tv, p.cv, colmaj, sv + vs * G::kTileBytes, &bar->v_full[vs], kt * kTile, ip.bh);
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA's shared memory goes away
        uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 2000000ull) { }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      if (p.self_test_timeout) {
        // nothing ever arrives on this barrier: exercises the bounded-wait path
        if (!ptx::mbar_wait(&bar->never, 0, p.timeout_ns, abort_flag)) {
          raise_error(p, bar, kErrSelfTest);
          ok = false;
        }
      }
      for (int s = 0; s < 2 && ok; ++s) {
        if (!ip.has_tiles[s]) continue;
        if (!ptx::mbar_wait(&bar->q_full[s], 0, p.timeout_ns, abort_flag)) {
          raise_error(p, bar, kErrMma);
          ok = false;
        }
      }
      ptx::tc_fence_after();
      const uint32_t q_smem = ptx::smem_addr(sq);
      const uint32_t k_smem = ptx::smem_addr(sk);
      const uint32_t v_smem = ptx::smem_addr(sv);
      bool pend[2] = {false, false};
      bool first[2] = {true, true};
      uint32_t pcount[2] = {0, 0};
      int j = 0;
      bool issued_any = false;
      if (ok) {
        for (int kt = union_next(p, ip, 0); kt != kNoTile; kt = union_next(p, ip, kt + 1), ++j) {
          const int ks = j % KS;
          if (j >= 1) {
            const int e = j - 1;
            if (!ptx::mbar_wait(&bar->v_full[e % VS], (e / VS) & 1, p.timeout_ns, abort_flag)) {
              raise_error(p, bar, kErrMma); ok = false; break;
            }
          }
          bool k_ready = false;
          for (int s = 0; s < 2 && ok; ++s) {
            if (pend[s]) {
              if (!ptx::mbar_wait(&bar->p_full[s], pcount[s] & 1, p.timeout_ns, abort_flag)) {
                raise_error(p, bar, kErrMma); ok = false; break;
              }
              ++pcount[s];
              ptx::tc_fence_after();
              issue_pv<D>(tmem + 256 + s * 128, tmem + s * 128, v_smem + ((j - 1) % VS) * G::kTileBytes, !first[s]);
              first[s] = false;
              pend[s] = false;
            }
            if (sub_uses(p, ip, s, kt)) {
              if (!k_ready) {
                if (!ptx::mbar_wait(&bar->k_full[ks], (j / KS) & 1, p.timeout_ns, abort_flag)) {
                  raise_error(p, bar, kErrMma); ok = false; break;
                }
                ptx::tc_fence_after();
                k_ready = true;
              }
              issue_qk<D>(tmem + s * 128, q_smem + s * G::kTileBytes, k_smem + ks * G::kTileBytes);
              ptx::mma_commit(&bar->s_full[s]);
              pend[s] = true;
              issued_any = true;
            }
          }
          if (!ok) break;
          ptx::mma_commit(&bar->k_empty[ks]);
          if (j >= 1) ptx::mma_commit(&bar->v_empty[(j - 1) % VS]);
        }
      }
      if (ok && j >= 1) {
        const int e = j - 1;
        if (!ptx::mbar_wait(&bar->v_full[e % VS], (e / VS) & 1, p.timeout_ns, abort_flag)) {
          raise_error(p, bar, kErrMma); ok = false;
        }
        for (int s = 0; s < 2 && ok; ++s) {
          if (!pend[s]) continue;
          if (!ptx::mbar_wait(&bar->p_full[s], pcount[s] & 1, p.timeout_ns, abort_flag)) {
            raise_error(p, bar, kErrMma); ok = false; break;
          }
          ++pcount[s];
          ptx::tc_fence_after();
          issue_pv<D>(tmem + 256 + s * 128, tmem + s * 128, v_smem + (e % VS) * G::kTileBytes, !first[s]);
          first[s] = false;
          pend[s] = false;
        }
        if (ok) {
          ptx::mma_commit(&bar->v_empty[e % VS]);
          for (int s = 0; s < 2; ++s)
            if (ip.has_tiles[s]) ptx::mma_commit(&bar->o_final[s]);
        }
      }
      if (!ok && issued_any) {
        // wait (bounded) for the MMAs already issued before tensor memory is freed
        ptx::mma_commit(&bar->drain);
        ptx::mbar_wait_time_only(&bar->drain, 0, p.timeout_ns);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    const int s = (warp - 4) >> 2;
    const int quarter = warp & 3;  // tensor-memory lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + s * 128;
    const uint32_t o_tmem = tmem + lane_off + 256 + s * 128;
    const int64_t pos = (int64_t)ip.qt[s] * kTile + row;
    const int h = ip.h;
    const int param = p.head_info[h * 4 + kHeadParam];
    int64_t lo, hi;
    row_interval(p.kind, param, p.N, pos, &lo, &hi);
    if (hi > p.N - 1) hi = p.N - 1;
    const float sl2 = p.scale_log2;

    float m = -INFINITY;  // running max of scaled scores, log2 domain
    float l = 0.f;        // running sum of exp2(x - m)
    int count = 0;
    bool ok = true;
    for (int kt = sub_next(p, ip, s, 0); kt != kNoTile; kt = sub_next(p, ip, s, kt + 1), ++count) {
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
      if (sub_partial(p, ip, s, kt)) {
        const int64_t k0 = (int64_t)kt * kTile;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int64_t q = k0 + c;
          if (q < lo || q > hi) x[c] = -INFINITY;
        }
      }
      float mx = x[0];
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, x[c]);
      mx *= sl2;
      const float m_new = fmaxf(m, mx);
      const bool need_rescale = (m != -INFINITY) && (m_new - m > kRescaleThreshold);
      if (m == -INFINITY) m = m_new;  // nothing accumulated yet (all earlier P were zero)
      // tcgen05.ld / st are warp-collective: the whole warp rescales when any
      // of its rows must, each lane with its own factor (1 when not needed)
      if (__any_sync(0xffffffffu, need_rescale)) {
        const float alpha = need_rescale ? ptx::ex2(m - m_new) : 1.f;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          float ov[16];
          ptx::tmem_ld16(o_tmem + c0, ov);
          ptx::tmem_wait_ld();
          uint32_t ou[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) ou[i] = __float_as_uint(ov[i] * alpha);
          ptx::tmem_st16(o_tmem + c0, ou);
        }
        if (need_rescale) {
          l *= alpha;
          m = m_new;
        }
      }
      const float mref = (m == -INFINITY) ? 0.f : m;
      float sum = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ptx::ex2(fmaf(x[c0 + 2 * i], sl2, -mref));
          const float p1 = ptx::ex2(fmaf(x[c0 + 2 * i + 1], sl2, -mref));
          sum += p0 + p1;
          pk[i] = ptx::pack_bf16x2(p0, p1);
        }
        ptx::tmem_st16(s_tmem + c0 / 2, pk);
      }
      l += sum;
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bar->p_full[s]);
    }

    // ---------------------------------------------------------- epilogue
    if (ok && ip.rows[s]) {
      bool have_o = false;
      if (count > 0) {
        bool got = ptx::mbar_wait(&bar->o_final[s], 0, p.timeout_ns, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) raise_error(p, bar, kErrEpilogue);
          ok = false;
        } else {
          ptx::tc_fence_after();
          have_o = true;
        }
      }
      if (ok) {
        const float b2 = p.sink ? p.sink[h] * kLog2e : -INFINITY;
        const float M = fmaxf(m, b2);
        float o_scale = 0.f;
        float lse_v = -INFINITY;
        if (M != -INFINITY) {
          const float em = (m == -INFINITY) ? 0.f : ptx::ex2(m - M);
          const float lf = l * em + ((b2 == -INFINITY) ? 0.f : ptx::ex2(b2 - M));
          if (lf > 0.f) {
            o_scale = em / lf;
            lse_v = (M + ptx::lg2(lf)) * kLn2;
          }
        }
        const bool valid = pos < p.N;
        const int store_mode = p.head_info[h * 4 + kHeadStore];
        const int perm_row = p.head_info[h * 4 + kHeadPermRow];
        const int64_t tok = valid ? token_of(p, store_mode, perm_row, pos) : 0;
        const int64_t orow = ((int64_t)ip.bh * p.N + tok) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          float ov[16];
          if (have_o) {
            ptx::tmem_ld16(o_tmem + c0, ov);
            ptx::tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = 0.f;
          }
          if (valid) {
            if (OUT_F32) {
              float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.o) + orow + c0);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_float4(ov[4 * i] * o_scale, ov[4 * i + 1] * o_scale, ov[4 * i + 2] * o_scale,
                                     ov[4 * i + 3] * o_scale);
            } else {
              uint32_t pk[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) pk[i] = ptx::pack_bf16x2(ov[2 * i] * o_scale, ov[2 * i + 1] * o_scale);
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + orow + c0);
              dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
          }
        }
        if (valid && p.lse) p.lse[(int64_t)ip.bh * p.N + tok] = lse_v;
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
    for (int kt = r.lo; kt <= r.hi; ++kt) {
      out[4 * n + 0] = h; out[4 * n + 1] = qt; out[4 * n + 2] = kt;
      out[4 * n + 3] = interval_tile_class(r, kt);
      ++n;
    }
  }
  p.counts[idx] = n;
}

// Reorder to sequence positions (and round fp32 to bf16): one thread per 8
// elements of one destination row, for q, k and v (blockIdx.y).
__global__ void gather_kernel(const GatherParams p) {
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
  int64_t tok = pos;
  if (store_mode == kStoreColumnMajor) {
    int64_t c = pos / p.grid_rows;
    tok = (pos - c * p.grid_rows) * p.grid_cols + c;
  } else if (store_mode == kStoreExplicit) {
    tok = p.perm[(int64_t)p.head_info[h * 4 + kHeadPermRow] * p.N + pos];
  }
  const int64_t src_off = (bh * p.N + tok) * p.d + c8;
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

template <int D, bool F32>
cudaError_t launch_one(const FwdParams& p, cudaStream_t stream) {
  const size_t smem = attention_smem_bytes(D);
  auto kern = attention_fwd_kernel<D, F32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<p.n_items, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
size_t smem_for() {
  using G = Geo<D>;
  size_t bytes = (size_t)(2 + 2 * G::kStages) * G::kTileBytes + sizeof(Barriers) + 1024;
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
#define MATTN_CASE(DD)                                                              \
  case DD:                                                                          \
    return out_f32 ? launch_one<DD, true>(p, stream) : launch_one<DD, false>(p, stream);
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
