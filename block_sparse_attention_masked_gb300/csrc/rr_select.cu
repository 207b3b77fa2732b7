// RRAttention's dynamic block selection on sm_103a ("RRAttention", section 3,
// Eq. 6-12; Eq. 5 of section 2.1): from Q and K of every head, the
// block-selection bitmap the attention kernel consumes.
//
// Three launches:
//   rr_stride_sum_kernel  Ksum_j = sum of the S keys of stride j (Eq. 8's key
//                         aggregation), bf16 [B*H][L/S][d].  HBM-bound.
//   rr_scores_kernel      per (head, 128 sampled query strides): the
//                         sampled queries (Eq. 6-7, read through a strided
//                         TMA view, no gather) times Ksum^T on the tensor
//                         cores (Eq. 8), the row softmax over every key stride
//                         (Eq. 9) and its sum into blocks (Eq. 10).  Two
//                         passes over the key strides: the first finds each
//                         row's log-sum-exp, the second exponentiates and adds
//                         the probabilities of each g x g (query, key) stride
//                         square, g = Bs/S, into one block score, so the
//                         L/S x L/S importance matrix never reaches memory.
//   rr_topk_kernel        per (head, query block): sort the block scores in
//                         decreasing order, keep the shortest prefix whose
//                         share of the row reaches tau (Eq. 11), add the last
//                         query block (Eq. 12), drop blocks above the diagonal
//                         (Eq. 5), write the bitmap row.
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

constexpr int kRrThreads = 256;
constexpr int kRrStages = 2;  // Ksum ring; two CTAs share an SM

struct RrBarriers {
  uint64_t q_full;
  uint64_t k_full[kRrStages], k_empty[kRrStages];
  uint64_t s_full[2], s_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void rr_raise(const RrParams& p, RrBarriers* bar, uint32_t bit) {
  *reinterpret_cast<volatile int*>(&bar->abort_flag) = 1;
  atomicOr(p.err, bit);
}

// Grid (ceil(n_s / 128), B*H); 256 threads: warp 0 loads (TMA), warp 1
// allocates tensor memory and issues the MMAs, warps 4..7 hold one sampled
// query stride (a row of S) per thread.  Tensor memory: two 128-column S
// buffers, so the product of the next key tile runs while this one is
// exponentiated.
template <int D, int G>
__global__ void __launch_bounds__(kRrThreads, 2) rr_scores_kernel(const __grid_constant__ RrParams p) {
  using T = Geo<D>;
  static_assert(D % 64 == 0, "sampled-query views use 64-column boxes");
  static_assert(G >= 4 && G <= 32 && (G & (G - 1)) == 0, "strides per block: 4, 8, 16 or 32");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = base;
  uint8_t* sk = sq + T::kTileBytes;
  RrBarriers* bar = reinterpret_cast<RrBarriers*>(sk + kRrStages * T::kTileBytes);
  volatile int* abort_flag = &bar->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qt = blockIdx.x;
  const int bh = blockIdx.y;
  const int h = bh % p.H;
  const int n_kt = (p.n_s + kTile - 1) / kTile;
  const int steps = 2 * n_kt;  // pass 0 then pass 1 over the key-stride tiles

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar->q_full, 1);
    for (int i = 0; i < kRrStages; ++i) {
      ptx::mbar_init(&bar->k_full[i], 1);
      ptx::mbar_init(&bar->k_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&bar->s_full[b], 1);
      ptx::mbar_init(&bar->s_empty[b], 128);
    }
    ptx::mbar_init(&bar->drain, 1);
    bar->abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&bar->tmem_base, 256);
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
      ptx::mbar_arrive_expect_tx(&bar->q_full, T::kTileBytes);
#pragma unroll
      for (int c = 0; c < T::kChunks; ++c)
        ptx::tma_load_4d(sq + c * T::kChunkBytes, &p.tq[0], &bar->q_full, c * 64, off, qt * kTile, bh);
      const uint64_t keep = ptx::l2_policy_evict_last();  // every query tile of the head re-reads Ksum
      for (int t = 0; t < steps; ++t) {
        const int slot = t % kRrStages;
        if (!ptx::mbar_wait(&bar->k_empty[slot], ((t / kRrStages) & 1) ^ 1, p.timeout_ns, abort_flag)) {
          rr_raise(p, bar, kErrProducer);
          break;
        }
        const int kt = t % n_kt;
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
      ok = wait_all(&bar->k_full[slot], (t / kRrStages) & 1) && wait_all(&bar->s_empty[b], ((t >> 1) & 1) ^ 1);
      if (!ok) break;
      ptx::tc_fence_after();
      if (ptx::elect_one()) issue_qk<D>(tmem + b * 128, q4, k4 + slot * tile4);
      __syncwarp();
      ptx::mma_commit_elect(&bar->s_full[b]);
      ptx::mma_commit_elect(&bar->k_empty[slot]);
      issued = true;
    }
    if (!ok) {
      if (lane == 0) rr_raise(p, bar, kErrMma);
      if (issued) {
        ptx::mma_commit_elect(&bar->drain);
        ptx::mbar_wait_time_only(&bar->drain, 0, p.timeout_ns);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax and block sums
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int grow = qt * kTile + row;  // sampled query stride of this thread
    const bool row_ok = grow < p.n_s;
    const float sl2 = p.scale_log2;     // log2(e) / (S sqrt(d)), Eq. 8's scale
    float m = -INFINITY, l = 0.f, lse2 = 0.f;
    for (int t = 0; t < steps; ++t) {
      const int b = t & 1;
      const bool got = ptx::mbar_wait(&bar->s_full[b], (t >> 1) & 1, p.timeout_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) rr_raise(p, bar, kErrSoftmax);
        break;
      }
      ptx::tc_fence_after();
      const int kt = t % n_kt;
      const bool second = t >= n_kt;
      const int ncols = min(kTile, p.n_s - kt * kTile);  // key strides present in this tile
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float x[32];
        ptx::tmem_ld32(tmem + lane_off + b * 128 + c * 32, x);
        ptx::tmem_wait_ld();
        if (c == 3) {
          ptx::tc_fence_before();
          ptx::mbar_arrive(&bar->s_empty[b]);  // S buffer b may be overwritten
        }
        const int col0 = c * 32;
        if (!second) {
          // pass 0 (Eq. 9's denominator): running max and sum, log2 domain
          float cm = -INFINITY;
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (col0 + k < ncols) cm = fmaxf(cm, x[k]);
          const float m_new = fmaxf(m, cm * sl2);
          if (m_new != -INFINITY) {
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < 32; ++k) s += (col0 + k < ncols) ? ptx::ex2(fmaf(x[k], sl2, -m_new)) : 0.f;
            l = (m == -INFINITY ? 0.f : l * ptx::ex2(m - m_new)) + s;
            m = m_new;
          }
        } else {
          // pass 1: P_ij (Eq. 9) summed over g key strides, then over the g
          // query strides (lanes) of the block (Eq. 10)
          float gs[32 / G];
#pragma unroll
          for (int i = 0; i < 32 / G; ++i) gs[i] = 0.f;
#pragma unroll
          for (int k = 0; k < 32; ++k)
            gs[k / G] += (row_ok && col0 + k < ncols) ? ptx::ex2(fmaf(x[k], sl2, -lse2)) : 0.f;
#pragma unroll
          for (int off = 1; off < G; off <<= 1)
#pragma unroll
            for (int i = 0; i < 32 / G; ++i) gs[i] += __shfl_xor_sync(0xffffffffu, gs[i], off);
          if ((lane & (G - 1)) == 0) {
            const int mb = grow / G;                    // query block
            const int nb0 = (kt * kTile + col0) / G;    // first key block of this chunk
            if (mb < p.nb) {
              float* dst = p.block_scores + ((int64_t)bh * p.nb + mb) * p.nb;
#pragma unroll
              for (int i = 0; i < 32 / G; ++i)
                if (nb0 + i < p.nb) dst[nb0 + i] = gs[i];
            }
          }
        }
      }
      if (t == n_kt - 1) lse2 = m + ptx::lg2(l);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 256);
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

// One CTA per (query block m, head bh).  Dynamic shared memory:
// part[kRrThreads] (double), bits[wpr] (uint64), key[p2] (float), idx[p2] (int).
__global__ void __launch_bounds__(kRrThreads) rr_topk_kernel(const RrTopParams p) {
  extern __shared__ uint8_t smem_raw[];
  const int p2 = p.p2;
  double* part = reinterpret_cast<double*>(smem_raw);
  unsigned long long* bits = reinterpret_cast<unsigned long long*>(part + kRrThreads);
  float* key = reinterpret_cast<float*>(bits + p.wpr);
  int* idx = reinterpret_cast<int*>(key + p2);
  __shared__ int cut;
  __shared__ double s_total;
  const int m = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int tid = threadIdx.x;
  const float* row = p.scores + (bh * p.nb + m) * p.nb;
  for (int i = tid; i < p2; i += kRrThreads) {
    key[i] = i < p.nb ? row[i] : -INFINITY;
    idx[i] = i;
  }
  for (int w = tid; w < p.wpr; w += kRrThreads) bits[w] = 0ull;
  if (tid == 0) cut = p.nb - 1;
  // bitonic sort: decreasing score, equal scores by increasing block index
  for (int k = 2; k <= p2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      __syncthreads();
      for (int i = tid; i < p2; i += kRrThreads) {
        const int ixj = i ^ j;
        if (ixj <= i) continue;
        const float ka = key[i], kb = key[ixj];
        const int ia = idx[i], ib = idx[ixj];
        const bool a_first = (ka > kb) || (ka == kb && ia < ib);
        const bool ascending_block = (i & k) != 0;  // this half runs the other way
        if (ascending_block ? a_first : !a_first) {
          key[i] = kb; key[ixj] = ka;
          idx[i] = ib; idx[ixj] = ia;
        }
      }
    }
  }
  __syncthreads();
  // running sums over the sorted scores in fp64 (Eq. 11): each thread owns
  // a contiguous run of per = p2 / kRrThreads entries
  const int per = p2 / kRrThreads;
  const int i0 = tid * per;
  double mine = 0.0;
  for (int e = 0; e < per; ++e) {
    const float v = key[i0 + e];
    if (v != -INFINITY) mine += (double)v;
  }
  part[tid] = mine;
  __syncthreads();
  if (tid == 0) {  // exclusive prefix of the per-thread sums, and the row total
    double run = 0.0;
    for (int t = 0; t < kRrThreads; ++t) {
      const double x = part[t];
      part[t] = run;
      run += x;
    }
    s_total = run;
  }
  __syncthreads();
  const double total = s_total;
  const double target = (double)p.tau * total;
  double run = part[tid];
  for (int e = 0; e < per; ++e) {
    const float v = key[i0 + e];
    if (v == -INFINITY) break;
    run += (double)v;
    if (run >= target) {
      atomicMin(&cut, i0 + e);
      break;
    }
  }
  __syncthreads();
  for (int i = tid; i <= cut; i += kRrThreads) {
    const int n = idx[i];
    atomicOr(&bits[n >> 6], 1ull << (n & 63));
  }
  __syncthreads();
  uint64_t* out = p.bits + (bh * p.nb + m) * p.wpr;
  for (int w = tid; w < p.wpr; w += kRrThreads) {
    uint64_t word = bits[w];
    if (m == p.nb - 1) word = ~0ull;                       // Eq. 12, the last query block
    if (p.sink_recent) {
      if (w == 0) word |= 1ull;                            // first key block
      if (w == (m >> 6)) word |= 1ull << (m & 63);         // diagonal block
    }
    // Eq. 5: nothing above the diagonal (n <= m), nothing past the last block
    const int lo = w * 64;
    const int hi_keep = min(m, p.nb - 1) - lo;             // highest kept bit in this word
    if (hi_keep < 0) word = 0ull;
    else if (hi_keep < 63) word &= (2ull << hi_keep) - 1ull;
    out[w] = word;
  }
}

template <int D, int G>
cudaError_t launch_scores_one(const RrParams& p, cudaStream_t stream) {
  const size_t smem = rr_scores_smem_bytes(D);
  auto kern = rr_scores_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((p.n_s + kTile - 1) / kTile), (unsigned)p.BH);
  kern<<<grid, kRrThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t rr_scores_smem_bytes(int d) {
  if (d != 64 && d != 128) return 0;
  const size_t tile = (size_t)kTile * d * 2;
  return (1 + kRrStages) * tile + sizeof(RrBarriers) + 1024;
}

size_t rr_topk_smem_bytes(int p2, int wpr) {
  return (size_t)kRrThreads * sizeof(double) + (size_t)wpr * sizeof(uint64_t) + (size_t)p2 * (sizeof(float) + sizeof(int));
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
  const size_t smem = rr_topk_smem_bytes(p.p2, p.wpr);
  cudaError_t e = cudaFuncSetAttribute(rr_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.nb, (unsigned)p.BH);
  rr_topk_kernel<<<grid, kRrThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mattn
