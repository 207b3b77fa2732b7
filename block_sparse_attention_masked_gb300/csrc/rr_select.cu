// RRAttention's dynamic block selection on sm_103a ("RRAttention", section 3,
// Eq. 6-12; Eq. 5 of section 2.1): from Q and K of every head, the
// block-selection bitmap the attention kernel consumes.
//
// Three launches:
//   rr_stride_sum_kernel  Ksum_j = sum of the S keys of stride j (Eq. 8's key
//                         aggregation), bf16 [B*H][L/S][d].  HBM-bound.
//   rr_scores_kernel      per (head, 2 x 128 sampled query strides): the
//                         sampled queries (Eq. 6-7, read through a strided
//                         TMA view, no gather) times Ksum^T on the tensor
//                         cores (Eq. 8), the row softmax over every key stride
//                         (Eq. 9) and its sum into blocks (Eq. 10).  Two
//                         passes over the key strides: the first finds each
//                         row's log-sum-exp, the second exponentiates and adds
//                         the probabilities of each g x g (query, key) stride
//                         square, g = Bs/S, into one block score, so the
//                         L/S x L/S importance matrix never reaches memory.
//   rr_topk_kernel        per (head, query block): keep the key blocks that
//                         the scores sorted in decreasing order need for
//                         their share of the row to reach tau (Eq. 11; found
//                         by a bitwise threshold search with exact integer
//                         sums, no sort), add the last query block (Eq. 12),
//                         drop blocks above the diagonal (Eq. 5), write the
//                         bitmap row.
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

constexpr int kRrThreads = 256;      // top-k kernel
constexpr int kRrScoreThreads = 384; // score kernel: 4 control warps + 2 x 4 row warps
constexpr int kRrStages = 4;         // Ksum ring depth
constexpr int kRrQTiles = 2;         // sampled-query tiles per CTA, sharing every Ksum tile

struct RrBarriers {
  uint64_t q_full;
  uint64_t k_full[kRrStages], k_empty[kRrStages];
  uint64_t s_full[kRrQTiles][2], s_empty[kRrQTiles][2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void rr_raise(const RrParams& p, RrBarriers* bar, uint32_t bit) {
  *reinterpret_cast<volatile int*>(&bar->abort_flag) = 1;
  atomicOr(p.err, bit);
}

// Pass 0 over one 128-column tile of a row: running maximum m and sum l of
// exp2(x * sl2 - m) (Eq. 9's denominator, log2 domain); columns >= ncols
// are absent.
template <bool RAGGED>
__device__ __forceinline__ void rr_pass0(const float (&x)[128], float sl2, int ncols, float& m, float& l) {
  float cm = -INFINITY;
#pragma unroll
  for (int c = 0; c < 128; ++c)
    if (!RAGGED || c < ncols) cm = fmaxf(cm, x[c]);
  const float m_new = fmaxf(m, cm * sl2);
  if (m_new == -INFINITY) return;
  const float2 sl2v = make_float2(sl2, sl2);
  const float2 negm = make_float2(-m_new, -m_new);
  float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int c = 0; c < 128; c += 2) {
    const float2 t = ptx::ffma2(make_float2(x[c], x[c + 1]), sl2v, negm);
    float2 e = make_float2(ptx::ex2(t.x), ptx::ex2(t.y));
    if (RAGGED) {
      if (c >= ncols) e.x = 0.f;
      if (c + 1 >= ncols) e.y = 0.f;
    }
    acc[(c >> 1) & 1] = ptx::fadd2(acc[(c >> 1) & 1], e);
  }
  const float2 a = ptx::fadd2(acc[0], acc[1]);
  l = (m == -INFINITY ? 0.f : l * ptx::ex2(m - m_new)) + (a.x + a.y);
  m = m_new;
}

// Pass 1 over one tile: P_ij = exp2(x * sl2 - lse2) (Eq. 9) summed over
// groups of G key strides (Eq. 10, the key side of a block).
template <int G, bool RAGGED>
__device__ __forceinline__ void rr_pass1(const float (&x)[128], float sl2, float lse2, int ncols,
                                         float (&gs)[128 / G]) {
  const float2 sl2v = make_float2(sl2, sl2);
  const float2 negl = make_float2(-lse2, -lse2);
#pragma unroll
  for (int i = 0; i < 128 / G; ++i) gs[i] = 0.f;
#pragma unroll
  for (int c = 0; c < 128; c += 2) {
    const float2 t = ptx::ffma2(make_float2(x[c], x[c + 1]), sl2v, negl);
    float2 e = make_float2(ptx::ex2(t.x), ptx::ex2(t.y));
    if (RAGGED) {
      if (c >= ncols) e.x = 0.f;
      if (c + 1 >= ncols) e.y = 0.f;
    }
    gs[c / G] += e.x + e.y;
  }
}

// Grid (ceil(n_s / 256), B*H); 384 threads: warp 0 loads (TMA), warp 1
// allocates tensor memory and issues the MMAs, warps 4..7 and 8..11 each
// hold one 128-row tile of sampled query strides, one row per thread.
// Tensor memory: per query tile two 128-column S buffers, so the products
// of the next key tile run while this one is exponentiated.
template <int D, int G>
__global__ void __launch_bounds__(kRrScoreThreads, 1) rr_scores_kernel(const __grid_constant__ RrParams p) {
  using T = Geo<D>;
  static_assert(D % 64 == 0, "sampled-query views use 64-column boxes");
  static_assert(G >= 4 && G <= 32 && (G & (G - 1)) == 0, "strides per block: 4, 8, 16 or 32");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = base;
  uint8_t* sk = sq + kRrQTiles * T::kTileBytes;
  RrBarriers* bar = reinterpret_cast<RrBarriers*>(sk + kRrStages * T::kTileBytes);
  volatile int* abort_flag = &bar->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int h = bh % p.H;
  const int q0 = blockIdx.x * kRrQTiles * kTile;                 // first sampled stride of the CTA
  const int nq = (q0 + kTile < p.n_s) ? kRrQTiles : 1;           // query tiles with rows
  const int n_kt = (p.n_s + kTile - 1) / kTile;
  const int steps = 2 * n_kt;  // pass 0 then pass 1 over the key-stride tiles

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar->q_full, 1);
    for (int i = 0; i < kRrStages; ++i) {
      ptx::mbar_init(&bar->k_full[i], 1);
      ptx::mbar_init(&bar->k_empty[i], 1);
    }
    for (int s = 0; s < kRrQTiles; ++s)
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

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      // Eq. 6: head h samples offset S - 1 - (h mod S) of every stride; the
      // view [B*H][L/S][S][d] turns that into one 128-row box per tile.
      const int off = p.S - 1 - (h % p.S);
      ptx::mbar_arrive_expect_tx(&bar->q_full, nq * T::kTileBytes);
      for (int s = 0; s < nq; ++s) {
        // (debug builds: coordinates inside the [B*H][L/S][S][d] view, else no load and the CTA aborts)
        if (!debug_check(p.err, off >= 0 && off < p.S && q0 + s * kTile < p.n_s && bh < p.BH, kSiteLoad)) {
          *abort_flag = 1;
          break;
        }
#pragma unroll
        for (int c = 0; c < T::kChunks; ++c)
          ptx::tma_load_4d(sq + s * T::kTileBytes + c * T::kChunkBytes, &p.tq[0], &bar->q_full, c * 64, off,
                           q0 + s * kTile, bh);
      }
      const uint64_t keep = ptx::l2_policy_evict_last();  // every query tile of the head re-reads Ksum
      for (int t = 0; t < steps; ++t) {
        const int slot = t % kRrStages;
        if (!ptx::mbar_wait(&bar->k_empty[slot], ((t / kRrStages) & 1) ^ 1, p.timeout_ns, abort_flag)) {
          rr_raise(p, bar, kErrProducer);
          break;
        }
        const int kt = t % n_kt;
        if (kDebugChecks && (*abort_flag || !debug_check(p.err, kt * kTile < p.n_s && bh < p.BH, kSiteLoad))) {
          *abort_flag = 1;
          break;
        }
        ptx::mbar_arrive_expect_tx(&bar->k_full[slot], T::kTileBytes);
#pragma unroll
        for (int c = 0; c < T::kChunks; ++c)
          ptx::tma_load_3d_hint(sk + slot * T::kTileBytes + c * T::kChunkBytes, &p.tk[0], &bar->k_full[slot], c * 64,
                                kt * kTile, bh, keep);
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
    bool ok = wait_all(&bar->q_full, 0);
    bool issued = false;
    constexpr uint32_t tile4 = T::kTileBytes >> 4;
    const uint32_t q4 = ptx::smem_addr(sq) >> 4;
    const uint32_t k4 = ptx::smem_addr(sk) >> 4;
    for (int t = 0; ok && t < steps; ++t) {
      const int slot = t % kRrStages;
      const int b = t & 1;
      ok = wait_all(&bar->k_full[slot], (t / kRrStages) & 1);
      for (int s = 0; ok && s < nq; ++s) {
        ok = wait_all(&bar->s_empty[s][b], ((t >> 1) & 1) ^ 1);
        if (!ok) break;
        ptx::tc_fence_after();
        if (ptx::elect_one()) issue_qk<D>(tmem + (s * 2 + b) * 128, q4 + s * tile4, k4 + slot * tile4);
        __syncwarp();
        ptx::mma_commit_elect(&bar->s_full[s][b]);
        issued = true;
      }
      if (ok) ptx::mma_commit_elect(&bar->k_empty[slot]);
    }
    if (!ok) {
      if (lane == 0) rr_raise(p, bar, kErrMma);
      if (issued) {
        ptx::mma_commit_elect(&bar->drain);
        ptx::mbar_wait_time_only(&bar->drain, 0, p.timeout_ns);
      }
    }
  } else if (warp >= 4 && (warp - 4) / 4 < nq) {
    // ------------------------------------------------------------ softmax and block sums
    const int s = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + s * 256;
    const int grow = q0 + s * kTile + row;  // sampled query stride of this thread
    const float sl2 = p.scale_log2;         // log2(e) / (S sqrt(d)), Eq. 8's scale
    float m = -INFINITY, l = 0.f, lse2 = 0.f;
    for (int t = 0; t < steps; ++t) {
      const int b = t & 1;
      const bool got = ptx::mbar_wait(&bar->s_full[s][b], (t >> 1) & 1, p.timeout_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) rr_raise(p, bar, kErrSoftmax);
        break;
      }
      ptx::tc_fence_after();
      float x[128];
      ptx::tmem_ld32(s_tmem + b * 128 + 0, *reinterpret_cast<float(*)[32]>(&x[0]));
      ptx::tmem_ld32(s_tmem + b * 128 + 32, *reinterpret_cast<float(*)[32]>(&x[32]));
      ptx::tmem_ld32(s_tmem + b * 128 + 64, *reinterpret_cast<float(*)[32]>(&x[64]));
      ptx::tmem_ld32(s_tmem + b * 128 + 96, *reinterpret_cast<float(*)[32]>(&x[96]));
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bar->s_empty[s][b]);  // the row is in registers: buffer b may be overwritten
      const int kt = t % n_kt;
      const int ncols = min(kTile, p.n_s - kt * kTile);  // key strides present in this tile
      if (t < n_kt) {
        if (ncols == kTile) rr_pass0<false>(x, sl2, ncols, m, l);
        else rr_pass0<true>(x, sl2, ncols, m, l);
        if (t == n_kt - 1) lse2 = grow < p.n_s ? m + ptx::lg2(l) : INFINITY;  // absent rows add nothing
      } else {
        float gs[128 / G];
        if (ncols == kTile) rr_pass1<G, false>(x, sl2, lse2, ncols, gs);
        else rr_pass1<G, true>(x, sl2, lse2, ncols, gs);
        // Eq. 10, the query side: sum over the G rows (lanes) of the block
#pragma unroll
        for (int off = 1; off < G; off <<= 1)
#pragma unroll
          for (int i = 0; i < 128 / G; ++i) gs[i] += __shfl_xor_sync(0xffffffffu, gs[i], off);
        if ((lane & (G - 1)) == 0) {
          const int mb = grow / G;          // query block
          const int nb0 = kt * (kTile / G);  // first key block of this tile
          if (mb < p.nb) {
            float* dst = p.block_scores + ((int64_t)bh * p.nb + mb) * p.nb;
#pragma unroll
            for (int i = 0; i < 128 / G; ++i)
              if (nb0 + i < p.nb) dst[nb0 + i] = gs[i];
          }
        }
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

// Ksum[bh][j][:] = sum_{t < S} K[bh][j*S + t][:] in fp32, stored as bf16:
// one thread per 8 output columns.
__global__ void rr_stride_sum_kernel(const RrSumParams p) {
  const int64_t vpr = p.d / 8;
  const int64_t total = (int64_t)p.BH * p.n_s * vpr;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int64_t orow = i / vpr;  // bh * n_s + j
  const int c8 = (int)(i - orow * vpr) * 8;
  const int64_t bh = orow / p.n_s;
  const int64_t j = orow - bh * p.n_s;
  const __nv_bfloat16* src = p.k + ((bh * p.N + j * p.S) * p.d + c8);
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int t = 0; t < p.S; ++t) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + (int64_t)t * p.d);
    const __nv_bfloat162* pr = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(pr[e]);
      acc[2 * e] += f.x;
      acc[2 * e + 1] += f.y;
    }
  }
  uint4 out;
  out.x = ptx::pack_bf16x2(acc[0], acc[1]);
  out.y = ptx::pack_bf16x2(acc[2], acc[3]);
  out.z = ptx::pack_bf16x2(acc[4], acc[5]);
  out.w = ptx::pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(p.ksum + orow * p.d + c8) = out;
}

// One warp per (head, query block) row of block scores: the top-tau choice
// of Eq. 11 without sorting.  The decision is taken on the scores quantised
// to integers, q_n = floor(s_n 2^(30 - e)) with 2^(e-1) <= max_n s_n < 2^e,
// so every sum below is exact and independent of the order it is formed in:
//   T  = ceil(tau_q total / 2^20), tau_q = round(tau 2^20), total = sum q_n;
//   v* = the largest score (as its bit pattern; scores are >= 0, so the
//        pattern orders like the value) with sum_{s_n >= v*} q_n >= T,
//        found bit by bit from the top;
//   kept = every block with s_n > v*, and the first blocks (by index) with
//          s_n == v* until the kept sum reaches T.
// That is the shortest prefix of the scores sorted in decreasing order
// (equal scores by increasing index) whose sum reaches tau times the total.
// Then the last query block keeps everything (Eq. 12) and blocks above the
// diagonal go (Eq. 5).  8 warps (rows) per CTA; the row is re-read from L1.
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__global__ void __launch_bounds__(kRrThreads) rr_topk_kernel(const RrTopParams p) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * (kRrThreads / 32) + warp;  // query block of this warp
  const int64_t bh = blockIdx.y;
  if (m >= p.nb) return;
  const float* row = p.scores + (bh * p.nb + m) * p.nb;
  const int nb = p.nb;
  // row maximum -> quantisation scale
  float mx = 0.f;
  for (int n = lane; n < nb; n += 32) mx = fmaxf(mx, row[n]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  int e = 0;
  frexpf(mx, &e);  // 2^(e-1) <= mx < 2^e (mx > 0: a row of softmax mass)
  const int sh = 30 - e;
  auto quant = [&](float x) -> unsigned long long {
    return (unsigned long long)__float2uint_rz(scalbnf(fmaxf(x, 0.f), sh));
  };
  unsigned long long tot = 0;
  for (int n = lane; n < nb; n += 32) tot += quant(row[n]);
  tot = warp_sum_u64(tot);
  const unsigned long long tau_q = (unsigned long long)llrintf(p.tau * 1048576.0f);
  const unsigned long long T = (tau_q * tot + ((1ull << 20) - 1)) >> 20;
  // v*: bit by bit from the top (bit 31 is the sign, always clear)
  uint32_t vstar = 0;
  for (int bit = 30; bit >= 0; --bit) {
    const uint32_t cand = vstar | (1u << bit);
    unsigned long long a = 0;
    for (int n = lane; n < nb; n += 32) {
      const float x = row[n];
      if (__float_as_uint(fmaxf(x, 0.f)) >= cand) a += quant(x);
    }
    if (warp_sum_u64(a) >= T) vstar = cand;
  }
  unsigned long long agt = 0;
  for (int n = lane; n < nb; n += 32) {
    const float x = row[n];
    if (__float_as_uint(fmaxf(x, 0.f)) > vstar) agt += quant(x);
  }
  agt = warp_sum_u64(agt);
  const unsigned long long qv = quant(__uint_as_float(vstar));
  // ties at v*: the first c_eq by index (T > agt here, and qv > 0)
  const unsigned long long c_eq = (T > agt && qv > 0) ? (T - agt + qv - 1) / qv : 0ull;
  uint64_t* out = p.bits + (bh * p.nb + m) * p.wpr;
  unsigned long long ties_before = 0;
  for (int w = 0; w < p.wpr; ++w) {
    uint64_t word = 0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int n = w * 64 + half * 32 + lane;
      const float x = n < nb ? row[n] : -1.f;
      const uint32_t kx = __float_as_uint(fmaxf(x, 0.f));
      const bool tie = n < nb && kx == vstar;
      const uint32_t tie_mask = __ballot_sync(0xffffffffu, tie);
      const unsigned long long rank = ties_before + __popc(tie_mask & ((1u << lane) - 1u));
      const bool keep = n < nb && (kx > vstar || (tie && rank < c_eq));
      const uint32_t keep_mask = __ballot_sync(0xffffffffu, keep);
      word |= (uint64_t)keep_mask << (32 * half);
      ties_before += __popc(tie_mask);
    }
    if (m == nb - 1) word = ~0ull;                     // Eq. 12, the last query block
    if (p.sink_recent) {
      if (w == 0) word |= 1ull;                        // first key block
      if (w == (m >> 6)) word |= 1ull << (m & 63);     // diagonal block
    }
    // Eq. 5: nothing above the diagonal (n <= m)
    const int hi_keep = m - w * 64;                    // highest kept bit in this word
    if (hi_keep < 0) word = 0ull;
    else if (hi_keep < 63) word &= (2ull << hi_keep) - 1ull;
    if (lane == 0) out[w] = word;
  }
}

template <int D, int G>
cudaError_t launch_scores_one(const RrParams& p, cudaStream_t stream) {
  const size_t smem = rr_scores_smem_bytes(D);
  auto kern = rr_scores_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((p.n_s + kRrQTiles * kTile - 1) / (kRrQTiles * kTile)), (unsigned)p.BH);
  kern<<<grid, kRrScoreThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t rr_scores_smem_bytes(int d) {
  if (d != 64 && d != 128) return 0;
  const size_t tile = (size_t)kTile * d * 2;
  return (kRrQTiles + kRrStages) * tile + sizeof(RrBarriers) + 1024;
}


cudaError_t launch_rr_stride_sum(const RrSumParams& p, cudaStream_t stream) {
  const int64_t total = (int64_t)p.BH * p.n_s * (p.d / 8);
  if (total == 0) return cudaSuccess;
  rr_stride_sum_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_rr_scores(const RrParams& p, int d, cudaStream_t stream) {
#define MATTN_RR_CASE(DD, GG) \
  if (d == DD && p.g == GG) return launch_scores_one<DD, GG>(p, stream);
  MATTN_RR_CASE(64, 4) MATTN_RR_CASE(64, 8) MATTN_RR_CASE(64, 16) MATTN_RR_CASE(64, 32)
  MATTN_RR_CASE(128, 4) MATTN_RR_CASE(128, 8) MATTN_RR_CASE(128, 16) MATTN_RR_CASE(128, 32)
#undef MATTN_RR_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_rr_topk(const RrTopParams& p, cudaStream_t stream) {
  const int rows_per_cta = kRrThreads / 32;
  dim3 grid((unsigned)((p.nb + rows_per_cta - 1) / rows_per_cta), (unsigned)p.BH);
  rr_topk_kernel<<<grid, kRrThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mattn
