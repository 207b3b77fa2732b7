// Received attention on sm_103a: r_h(j) = sum_i a_ij, the column sums of the
// masked attention matrix (SHS slides, the received-attention slide), from
// the log-sum-exp the forward wrote (a_ij = exp(s_ij - lse_i), so the sink's
// share of each row is received by no token).
//
// The transpose of the forward: one CTA holds two 128-key tiles of one
// (batch, head) and streams the 128-query tiles that may see either of them
// (the forward's tile plan read column-wise), computing S^T = K Q^T on the
// tensor cores into tensor memory; one thread per key row adds
// exp2(s * scale * log2e - lse_i * log2e) over the visible query columns.
// Roles (384 threads): warp 0 loads (TMA: the two key tiles once, a ring of
// query tiles), warp 1 allocates tensor memory and issues the MMAs, warps
// 4..7 / 8..11 own key tile 0 / 1.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernel_params.h"
#include "plan_rules.h"
#include "ptx.cuh"
#include "tile_mma.cuh"

namespace mattn {
namespace {

constexpr int kRcThreads = 384;
constexpr int kRcStages = 3;

// The CTA's query-tile list: entry j is query tile qt(j); key tile s of the
// CTA multiplies it when uses(j, s).  Interval kinds: qt(j) = lo + j, the
// union of the two key tiles' query ranges (adjacent key tiles have
// overlapping or touching ranges), each key tile using its own range.
// Block kind: entries qt | use0 << 30 | use1 << 31 in shared memory, built
// once per CTA by one warp walking the bitmap column of each key tile.
struct QList {
  int n, lo, lo0, hi0, lo1, hi1;
  const uint32_t* e;
  int block;
};

struct RcBarriers {
  uint64_t k_full;
  uint64_t q_full[kRcStages], q_empty[kRcStages];
  uint64_t s_full[2][2], s_empty[2][2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int list_n;
  QList ql;
};

__device__ __forceinline__ int ql_qt(const QList& Q, int j) { return Q.block ? (int)(Q.e[j] & 0x3fffffffu) : Q.lo + j; }
__device__ __forceinline__ bool ql_uses(const QList& Q, int j, int s) {
  if (Q.block) return (Q.e[j] >> (30 + s)) & 1u;
  const int qt = Q.lo + j;
  return s ? (qt >= Q.lo1 && qt <= Q.hi1) : (qt >= Q.lo0 && qt <= Q.hi0);
}

__device__ __forceinline__ void rc_raise(const RecvParams& p, RcBarriers* bar, uint32_t bit) {
  *reinterpret_cast<volatile int*>(&bar->abort_flag) = 1;
  atomicOr(p.err, bit);
}

// Query positions that may see key position t (the masks are symmetric
// except the causal window, whose queries lie at or after the key).
__device__ __forceinline__ void col_interval(int kind, int64_t param, int64_t n, int64_t t, int64_t* lo,
                                             int64_t* hi) {
  if (kind == kCausalWindow) {
    *lo = t;
    *hi = t + param - 1;
  } else if (kind == kBlockSparse) {
    *lo = t;  // causality; the block bits are checked per tile
    *hi = n - 1;
  } else {
    row_interval(kind, param, n, t, lo, hi);
  }
}

// Interval kinds: the query tiles [*qlo, *qhi] that see key tile kt (empty: qlo > qhi).
__device__ __forceinline__ void q_range(const RecvParams& p, int param, int kt, int* qlo, int* qhi) {
  const int nt = (p.N + kTile - 1) / kTile;
  if (kt >= nt) {
    *qlo = 1; *qhi = 0;
    return;
  }
  const int64_t t0 = (int64_t)kt * kTile;
  const int64_t t1 = (t0 + kTile < p.N ? t0 + kTile : p.N) - 1;
  int64_t lo0, hi0, lo1, hi1;
  col_interval(p.kind, param, p.N, t0, &lo0, &hi0);
  col_interval(p.kind, param, p.N, t1, &lo1, &hi1);
  *qlo = (int)(lo0 < 0 ? 0 : lo0 / kTile);
  *qhi = (int)((hi1 > p.N - 1 ? p.N - 1 : hi1) / kTile);
}

// Block kind: one warp lists, in increasing order, the query tiles qt >=
// kt0 whose bitmap row keeps key tile kt0 or kt0 + 1 (and qt >= that key
// tile), 32 rows per step: a ballot per key tile, the union's ballot gives
// every lane its output slot.
__device__ __forceinline__ void build_q_list(const RecvParams& p, const uint64_t* bits, int kt0, int nk, uint32_t* list,
                                             int* n_out, int lane) {
  const int nt = (p.N + kTile - 1) / kTile;
  const int c = p.block_c;
  const int nb0 = kt0 / c, nb1 = (kt0 + 1) / c;
  int base = 0;
  for (int q0 = kt0; q0 < nt; q0 += 32) {
    const int qt = q0 + lane;
    bool u0 = false, u1 = false;
    if (qt < nt) {
      const uint64_t* row = bits + (int64_t)(qt / c) * p.block_wpr;
      u0 = (row[nb0 >> 6] >> (nb0 & 63)) & 1ull;
      u1 = nk > 1 && qt >= kt0 + 1 && ((row[nb1 >> 6] >> (nb1 & 63)) & 1ull);
    }
    const uint32_t any = __ballot_sync(0xffffffffu, u0 || u1);
    if (u0 || u1) {
      const int pos = base + __popc(any & ((1u << lane) - 1u));
      if (!kDebugChecks || pos < kBlockListMax) list[pos] = (uint32_t)qt | ((u0 ? 1u : 0u) << 30) | ((u1 ? 1u : 0u) << 31);
    }
    base += __popc(any);
  }
  if (lane == 0) *n_out = base;
}

// Caller token at position pos.  Debug builds check the head's
// explicit-order row and the token (debug_check) and return -1 after a
// failed check: the value is then neither read nor stored.
__device__ __forceinline__ int64_t rc_token_of(const RecvParams& p, int store_mode, int perm_row, int64_t pos) {
  if (!debug_check(p.err, store_mode != kStoreExplicit || (perm_row >= 0 && perm_row < p.n_perm), kSiteItem))
    return -1;
  const int64_t tok = token_at(store_mode, p.grid_rows, p.grid_cols,
                               store_mode == kStoreExplicit ? p.perm + (int64_t)perm_row * p.N : nullptr, pos);
  if (!debug_check(p.err, tok >= 0 && tok < p.N, kSiteOrder)) return -1;
  return tok;
}

// A 128-position tile of view row bh inside the raster or column-major
// view, on the coordinates rc_load computes (debug checks).
__device__ __forceinline__ bool rc_tile_ok(const RecvParams& p, bool column_major, int p0, int bh) {
  if (p0 < 0 || p0 >= p.N || (p0 & (kTile - 1)) || bh < 0 || bh >= p.B * p.H) return false;
  if (!column_major) return true;
  if (p.grid_rows <= 0) return false;
  const int col = p0 / p.grid_rows, r0 = p0 - col * p.grid_rows;
  return col < p.grid_cols && r0 + kTile <= p.grid_rows;
}

// TMA load of one 128-row tile at sequence position p0 (raster view, or the
// column-major 4D view when the head walks its grid column by column).
template <int D>
__device__ __forceinline__ void rc_load(const CUtensorMap* raster, const CUtensorMap* colmaj, bool column_major,
                                        int grid_rows, uint8_t* dst, uint64_t* bar, int p0, int bh) {
  using T = Geo<D>;
  if (!column_major) {
#pragma unroll
    for (int c = 0; c < T::kChunks; ++c) ptx::tma_load_3d(dst + c * T::kChunkBytes, &raster[0], bar, c * 64, p0, bh);
    if (T::kRem) ptx::tma_load_3d(dst + T::kChunks * T::kChunkBytes, &raster[1], bar, 0, p0, bh);
  } else {
    const int col = p0 / grid_rows;
    const int r0 = p0 - col * grid_rows;
#pragma unroll
    for (int c = 0; c < T::kChunks; ++c)
      ptx::tma_load_4d(dst + c * T::kChunkBytes, &colmaj[0], bar, c * 64, col, r0, bh);
    if (T::kRem) ptx::tma_load_4d(dst + T::kChunks * T::kChunkBytes, &colmaj[1], bar, 0, col, r0, bh);
  }
}

template <int D>
__global__ void __launch_bounds__(kRcThreads, 1) received_kernel(const __grid_constant__ RecvParams p) {
  using T = Geo<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sk = base;                         // two key tiles
  uint8_t* sq = sk + 2 * T::kTileBytes;       // query ring
  RcBarriers* bar = reinterpret_cast<RcBarriers*>(sq + kRcStages * T::kTileBytes);
  volatile int* abort_flag = &bar->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int h = bh % p.H;
  const int nt = (p.N + kTile - 1) / kTile;
  const int kt0 = 2 * blockIdx.x;
  const int nk = (kt0 + 1 < nt) ? 2 : 1;   // key tiles of this CTA
  const int param = p.head_info[h * 4 + kHeadParam];
  const bool colmaj = p.head_info[h * 4 + kHeadLoad] == kLoadColumnMajor;
  const uint64_t* bits =
      p.kind == kBlockSparse ? p.block_bits + (int64_t)((p.block_heads == 1) ? 0 : h) * p.block_nb * p.block_wpr
                             : nullptr;
  uint32_t* list_e = reinterpret_cast<uint32_t*>(bar + 1);  // block kind: [kBlockListMax] entries
  if (p.kind == kBlockSparse && warp == 2) build_q_list(p, bits, kt0, nk, list_e, &bar->list_n, lane);

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar->k_full, 1);
    for (int i = 0; i < kRcStages; ++i) {
      ptx::mbar_init(&bar->q_full[i], 1);
      ptx::mbar_init(&bar->q_empty[i], 1);
    }
    for (int s = 0; s < 2; ++s)
      for (int b = 0; b < 2; ++b) {
        ptx::mbar_init(&bar->s_full[s][b], 1);
        ptx::mbar_init(&bar->s_empty[s][b], 128);
      }
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
  if (threadIdx.x == 0) {
    QList Q;
    Q.block = p.kind == kBlockSparse;
    Q.e = list_e;
    q_range(p, param, kt0, &Q.lo0, &Q.hi0);
    if (nk > 1) q_range(p, param, kt0 + 1, &Q.lo1, &Q.hi1);
    else { Q.lo1 = 1; Q.hi1 = 0; }
    if (Q.block) {
      Q.n = bar->list_n;
      Q.lo = 0;
      if (kDebugChecks && !debug_check(p.err, Q.n <= kBlockListMax, kSiteKeyTile)) {
        *abort_flag = 1;  // debug builds: a list past its capacity is dropped
        Q.n = 0;
      }
    } else {
      const bool e0 = Q.lo0 <= Q.hi0, e1 = Q.lo1 <= Q.hi1;
      Q.lo = e0 ? (e1 ? min(Q.lo0, Q.lo1) : Q.lo0) : Q.lo1;
      const int hi = e0 ? (e1 ? max(Q.hi0, Q.hi1) : Q.hi0) : Q.hi1;
      Q.n = (e0 || e1) ? hi - Q.lo + 1 : 0;
    }
    bar->ql = Q;
  }
  __syncthreads();
  const QList& QL = bar->ql;

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(&bar->k_full, nk * T::kTileBytes);
      for (int s = 0; s < nk; ++s) {
        // (debug builds: tile coordinates inside the view, else no load and the CTA aborts)
        if (!debug_check(p.err, rc_tile_ok(p, colmaj, (kt0 + s) * kTile, bh), kSiteLoad)) {
          *abort_flag = 1;
          break;
        }
        rc_load<D>(p.tk, p.ck, colmaj, p.grid_rows, sk + s * T::kTileBytes, &bar->k_full, (kt0 + s) * kTile, bh);
      }
      for (int j = 0; j < QL.n; ++j) {
        const int qt = ql_qt(QL, j);
        const int slot = j % kRcStages;
        if (kDebugChecks && (*abort_flag || !debug_check(p.err, rc_tile_ok(p, colmaj, qt * kTile, bh), kSiteLoad))) {
          *abort_flag = 1;
          break;
        }
        if (!ptx::mbar_wait(&bar->q_empty[slot], ((j / kRcStages) & 1) ^ 1, p.timeout_ns, abort_flag)) {
          rc_raise(p, bar, kErrProducer);
          break;
        }
        ptx::mbar_arrive_expect_tx(&bar->q_full[slot], T::kTileBytes);
        rc_load<D>(p.tq, p.cq, colmaj, p.grid_rows, sq + slot * T::kTileBytes, &bar->q_full[slot], qt * kTile, bh);
      }
      if (*abort_flag) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 2000000ull) { }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    auto wait_all = [&](uint64_t* b, uint32_t parity) {
      return __all_sync(0xffffffffu, ptx::mbar_wait(b, parity, p.timeout_ns, abort_flag));
    };
    bool ok = wait_all(&bar->k_full, 0);
    bool issued = false;
    constexpr uint32_t tile4 = T::kTileBytes >> 4;
    const uint32_t k4 = ptx::smem_addr(sk) >> 4;
    const uint32_t q4 = ptx::smem_addr(sq) >> 4;
    int used[2] = {0, 0};
    for (int j = 0; ok && j < QL.n; ++j) {
      const int slot = j % kRcStages;
      ok = wait_all(&bar->q_full[slot], (j / kRcStages) & 1);
      for (int s = 0; ok && s < nk; ++s) {
        if (!ql_uses(QL, j, s)) continue;
        const int b = used[s] & 1;
        ok = wait_all(&bar->s_empty[s][b], ((used[s] >> 1) & 1) ^ 1);
        if (!ok) break;
        ptx::tc_fence_after();
        // S^T (keys x queries) = K_s Q^T: A = the key tile, B = the query tile
        if (ptx::elect_one()) issue_qk<D>(tmem + (s * 2 + b) * 128, k4 + s * tile4, q4 + slot * tile4);
        __syncwarp();
        ptx::mma_commit_elect(&bar->s_full[s][b]);
        ++used[s];
        issued = true;
      }
      if (ok) ptx::mma_commit_elect(&bar->q_empty[slot]);
    }
    if (!ok) {
      if (lane == 0) rc_raise(p, bar, kErrMma);
      if (issued) {
        ptx::mma_commit_elect(&bar->drain);
        ptx::mbar_wait_time_only(&bar->drain, 0, p.timeout_ns);
      }
    }
  } else if (warp >= 4 && (warp - 4) / 4 < nk) {
    // ------------------------------------------------------------ column sums
    const int s = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int64_t t = (int64_t)(kt0 + s) * kTile + row;  // key position of this thread
    int64_t vlo, vhi;                                   // query positions that see it
    col_interval(p.kind, param, p.N, t, &vlo, &vhi);
    if (vhi > p.N - 1) vhi = p.N - 1;
    const float sl2 = p.scale_log2;
    const float* lse2 = p.lse2p + (int64_t)bh * p.lse_pitch;  // log2-domain lse in position order
    float racc = 0.f;
    int cnt = 0;
    for (int j = 0; j < QL.n; ++j) {
      if (!ql_uses(QL, j, s)) continue;
      const int qt = ql_qt(QL, j);
      const int b = cnt & 1;
      const bool got = ptx::mbar_wait(&bar->s_full[s][b], (cnt >> 1) & 1, p.timeout_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) rc_raise(p, bar, kErrSoftmax);
        break;
      }
      ptx::tc_fence_after();
      float x[128];
      const uint32_t sa = tmem + lane_off + (s * 2 + b) * 128;
      ptx::tmem_ld32(sa + 0, *reinterpret_cast<float(*)[32]>(&x[0]));
      ptx::tmem_ld32(sa + 32, *reinterpret_cast<float(*)[32]>(&x[32]));
      ptx::tmem_ld32(sa + 64, *reinterpret_cast<float(*)[32]>(&x[64]));
      ptx::tmem_ld32(sa + 96, *reinterpret_cast<float(*)[32]>(&x[96]));
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bar->s_empty[s][b]);
      ++cnt;
      const int64_t q0 = (int64_t)qt * kTile;
      // visible query columns of this key row in the tile: [c_lo, c_hi]
      const int c_lo = (int)(vlo - q0 < 0 ? 0 : (vlo - q0 > 128 ? 128 : vlo - q0));
      const int c_hi = (int)(vhi - q0 > 127 ? 127 : (vhi - q0 < -1 ? -1 : vhi - q0));
      const float4* l4 = reinterpret_cast<const float4*>(lse2 + q0);  // 16-byte aligned: pitch % 128 == 0
      const bool whole = __all_sync(0xffffffffu, c_lo == 0 && c_hi == 127) && q0 + kTile <= p.N;
      float acc0 = 0.f, acc1 = 0.f;
      if (whole) {
#pragma unroll
        for (int c4 = 0; c4 < 32; ++c4) {
          const float4 lv = __ldg(l4 + c4);  // the same 16 bytes for every lane
          acc0 += ptx::ex2(fmaf(x[4 * c4 + 0], sl2, -lv.x));
          acc1 += ptx::ex2(fmaf(x[4 * c4 + 1], sl2, -lv.y));
          acc0 += ptx::ex2(fmaf(x[4 * c4 + 2], sl2, -lv.z));
          acc1 += ptx::ex2(fmaf(x[4 * c4 + 3], sl2, -lv.w));
        }
      } else {
        const int cmax = (int)(p.N - q0 < 128 ? p.N - q0 : 128);  // query columns present
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const float lv = c < cmax ? lse2[q0 + c] : INFINITY;
          const float e = ptx::ex2(fmaf(x[c], sl2, -lv));
          if (c >= c_lo && c <= c_hi) {
            if (c & 1) acc1 += e;
            else acc0 += e;
          }
        }
      }
      racc += acc0 + acc1;
    }
    if (t < p.N) {
      const int store_mode = p.head_info[h * 4 + kHeadStore];
      const int perm_row = p.head_info[h * 4 + kHeadPermRow];
      const int64_t tok = rc_token_of(p, store_mode, perm_row, t);
      if (!kDebugChecks || tok >= 0) p.r[(int64_t)bh * p.N + tok] = racc;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// lse2p[bh][p] = lse[bh][token at position p] * log2(e): the forward's
// log-sum-exp in sequence-position order and the log2 domain.
__global__ void lse_positions_kernel(const RecvParams p, const float* lse) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)p.B * p.H * p.N;
  if (i >= total) return;
  const int64_t bh = i / p.N;
  const int64_t pos = i - bh * p.N;
  const int h = (int)(bh % p.H);
  const int64_t tok = rc_token_of(p, p.head_info[h * 4 + kHeadStore], p.head_info[h * 4 + kHeadPermRow], pos);
  if (kDebugChecks && tok < 0) return;
  p.lse2p[bh * p.lse_pitch + pos] = lse[bh * p.N + tok] * 1.4426950408889634f;
}

template <int D>
cudaError_t launch_recv_one(const RecvParams& p, cudaStream_t stream) {
  const size_t smem = received_smem_bytes(D);
  auto kern = received_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int nt = (p.N + kTile - 1) / kTile;
  dim3 grid((unsigned)((nt + 1) / 2), (unsigned)(p.B * p.H));
  kern<<<grid, kRcThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t received_smem_bytes(int d) {
  size_t tile;
  switch (d) {
    case 32: tile = Geo<32>::kTileBytes; break;
    case 64: tile = Geo<64>::kTileBytes; break;
    case 80: tile = Geo<80>::kTileBytes; break;
    case 96: tile = Geo<96>::kTileBytes; break;
    case 128: tile = Geo<128>::kTileBytes; break;
    default: return 0;
  }
  return (2 + kRcStages) * tile + sizeof(RcBarriers) + kBlockListMax * sizeof(uint32_t) + 1024;
}

cudaError_t launch_received(const RecvParams& p, const float* lse, int d, cudaStream_t stream) {
  const int64_t total = (int64_t)p.B * p.H * p.N;
  if (total == 0) return cudaSuccess;
  lse_positions_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(p, lse);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  switch (d) {
    case 32: return launch_recv_one<32>(p, stream);
    case 64: return launch_recv_one<64>(p, stream);
    case 80: return launch_recv_one<80>(p, stream);
    case 96: return launch_recv_one<96>(p, stream);
    case 128: return launch_recv_one<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mattn
