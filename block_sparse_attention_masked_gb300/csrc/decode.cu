// Decode-shaped masked attention for sm_103a: one new query token per
// sequence against its key/value cache, split over the cache (the decode
// launches of the Bifocal page's speed test: a 1K..128K-token prompt, then
// one token at a time, with 16 query heads sharing 4 key/value heads of
// dimension 256).
//
// The work is a stream of the cache through the SMs: per key one row of K
// and one of V (4 d bytes in bf16) against 4 d FLOPs for each of the G query
// heads that share the key/value head, so for G <= 8 it is HBM-bound and
// runs on the CUDA cores (a tensor-core tile would sit almost empty at
// G rows).  Two kernels:
//
//   decode_split_kernel<D, GP>: grid (n_split, B * H_kv).  A CTA takes a
//     chunk of the keys one key/value head's query heads may see, for all
//     of those heads.  Its producer warp streams the chunk's K and V rows
//     into a ring of shared-memory slots with bulk async copies (keys of a
//     cache are contiguous rows, so a slot is one or two copies per tensor),
//     keeping up to 192 KB in flight per SM; a slot holds 32 keys, in groups of
//     KPG = 32 / GP keys, and each (slot, group) pair of the ring has one
//     owner among up to twelve consumer warps.  In a group: lane l holds dims
//     [l*VPL, (l+1)*VPL) of every query (VPL = D / 32) and of each row, forms
//     the KPG x GP partial dot products, and a reduce-scatter across the
//     lanes leaves lane j with the score of pair j = (key j / GP, head
//     j % GP).  Online softmax per head (running max in the log2 domain,
//     rescaled sums), then P V with the pair weights broadcast through shared
//     memory.  The CTA's warps are merged in shared memory and the chunk's
//     (m, l, O) written out.
//   decode_combine_kernel<D>: one CTA per (b, h) merges the chunks' states
//     with the sink logit into O and the log-sum-exp.
//
// Visible keys of the query at position len - 1 (len = cached tokens of the
// sequence, the new token included): every key (MATTN_FULL), or the last W
// keys and the first S sink tokens (MATTN_CAUSAL_WINDOW), W per query head.
// A key/value head's chunks cover the union of its query heads' visible
// keys (the sink keys below the windows, then the windows' span), so a
// windowed decode launches only the chunks of ~W + S keys, whatever len is.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernel_params.h"
#include "plan_rules.h"
#include "ptx.cuh"

namespace mattn {
namespace {

constexpr float kLog2eD = 1.4426950408889634f;
constexpr float kLn2D = 0.6931471805599453f;
constexpr int kDecRingBytes = 192 * 1024;  // at d = 256: six 32-key slots, groups for twelve warps

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

template <int D, int GP>
struct DecGeo {
  static constexpr int VPL = D / 32;                  // dims per lane
  static constexpr int KPG = 32 / GP;                 // keys per group (one score per lane)
  static constexpr int U = 32;                        // keys per ring slot (one bulk copy per tensor)
  static constexpr int GPS = U / KPG;                 // groups per slot (= GP), each taken by one warp
  static constexpr int kRow = D * 2;                  // bytes of a bf16 row
  static constexpr int kSlot = 2 * U * kRow;          // K rows, then V rows
  static constexpr int NS0 = kDecRingBytes / kSlot;
  static constexpr int NS = NS0 > 32 ? 32 : NS0;      // ring slots
  // consumer warps: twelve (three per SM sub-partition), eight when the
  // queries and accumulators of G = 8 heads at d = 256 need more registers
  static constexpr int kConsW = (D * GP >= 2048) ? 8 : 12;
  static constexpr int kThreads = 32 * (kConsW + 1);  // consumers, then the producer warp
  // consumer warps that take groups: the largest divisor of NS * GPS up to
  // kConsW, so that every (ring slot, group) pair has one fixed owner warp
  static constexpr int largest_divisor(int n, int cap) {
    int best = 1;
    for (int k = 1; k <= cap; ++k)
      if (n % k == 0) best = k;
    return best;
  }
  static constexpr int kCons = largest_divisor(NS * GPS, kConsW);
  static_assert(VPL == 2 || VPL == 4 || VPL == 8, "D must be 64, 128 or 256");
  static_assert(NS >= 2, "ring too small");
};

// VPL bf16 values of one row, as VPL / 2 packed words, from shared memory.
template <int VPL>
__device__ __forceinline__ void load_row_s(const uint8_t* src, uint32_t (&w)[VPL / 2]) {
  if constexpr (VPL == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
  } else if constexpr (VPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    w[0] = u.x; w[1] = u.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(src);
  }
}

// Window start of the query at position qpos for window w (causal window
// kind) or 0 (full); sink keys are handled separately.
__device__ __forceinline__ int window_lo(const DecodeParams& p, int w, int qpos) {
  if (p.kind != kCausalWindow) return 0;
  const int lo = qpos - w + 1;
  return lo > 0 ? lo : 0;
}

struct DecBar {
  uint64_t full[32], empty[32];
  int abort_flag;
};

template <int D, int GP>
__global__ void __launch_bounds__(DecGeo<D, GP>::kThreads, 1) decode_split_kernel(const DecodeParams p) {
  using Geo = DecGeo<D, GP>;
  constexpr int kDecConsumers = Geo::kConsW;
  constexpr int kDecThreads = Geo::kThreads;
  constexpr int VPL = Geo::VPL, KPG = Geo::KPG, U = Geo::U, NS = Geo::NS;
  extern __shared__ __align__(128) uint8_t dsm[];
  uint8_t* ring = dsm;                                               // [NS][2][U][D] bf16
  DecBar* bar = reinterpret_cast<DecBar*>(dsm + NS * Geo::kSlot);
  float* wp = reinterpret_cast<float*>(bar + 1);                     // [kDecConsumers][32]
  float* wml = wp + kDecConsumers * 32;                              // [kDecConsumers][GP][2]
  float* wo = reinterpret_cast<float*>(ring);                        // [kDecConsumers][GP][D], after the loop
  volatile int* abort_flag = &bar->abort_flag;

  // the combine grid may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int bkv = blockIdx.y;
  const int b = bkv / p.H_kv, kvh = bkv % p.H_kv;
  const int G = p.H / p.H_kv;
  int len = p.seq_lens ? p.seq_lens[b] : p.L;
  len = len < 0 ? 0 : (len > p.L ? p.L : len);
  const int qpos = len - 1;

  // the group's visible keys as one list: range A = the sink keys below the
  // windows [0, na), then range B = [lo_u, len), lo_u the smallest window start
  int lo_u = len;
  for (int j = 0; j < G; ++j) {
    const int lo = window_lo(p, p.head_info[(kvh * G + j) * 4 + kHeadParam], qpos);
    lo_u = lo < lo_u ? lo : lo_u;
  }
  const int S = p.sink_tokens < len ? p.sink_tokens : len;
  const int na = S < lo_u ? S : lo_u;
  const int nk = na + (len - lo_u);
  auto key_at = [&](int i) { return i < na ? i : lo_u + (i - na); };
  // this CTA's share of the list
  const int i_begin = split * p.chunk;
  const int i_end = (i_begin + p.chunk < nk) ? i_begin + p.chunk : nk;

  const int64_t bh0 = (int64_t)b * p.H + kvh * G;  // first query head row of the group
  float* part_ml = p.part_ml + (bh0 * p.n_split + split) * 2;
  if (i_begin >= i_end) {
    // nothing visible in this chunk: an empty state for every head
    if (threadIdx.x < G) {
      part_ml[(int64_t)threadIdx.x * p.n_split * 2 + 0] = -INFINITY;
      part_ml[(int64_t)threadIdx.x * p.n_split * 2 + 1] = 0.f;
    }
    return;
  }
  const int nslots = (i_end - i_begin + U - 1) / U;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      ptx::mbar_init(&bar->full[i], 1);
      ptx::mbar_init(&bar->empty[i], Geo::GPS);  // one arrival per group of the slot
    }
    bar->abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();

  float m = -INFINITY;  // consumers: running max of head gl (same on every lane of gl)
  float l = 0.f;        // consumers: this lane's share of head gl's running sum
  // O of every head, this lane's dims as pairs (packed f32x2 arithmetic)
  float2 o[GP][VPL / 2];
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int i = 0; i < VPL / 2; ++i) o[g][i] = make_float2(0.f, 0.f);
  const int gl = lane % GP, kl = lane / GP;

  if (warp == kDecConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint8_t* kb = reinterpret_cast<const uint8_t*>(p.k) + (int64_t)bkv * p.L * Geo::kRow;
      const uint8_t* vb = reinterpret_cast<const uint8_t*>(p.v) + (int64_t)bkv * p.L * Geo::kRow;
      for (int s = 0; s < nslots; ++s) {
        const int slot = s % NS;
        if (!ptx::mbar_wait(&bar->empty[slot], ((s / NS) & 1) ^ 1, p.timeout_ns, abort_flag)) {
          *abort_flag = 1;
          atomicOr(p.err, 1u);
          break;
        }
        const int j0 = i_begin + s * U;
        const int j1 = (j0 + U < i_end) ? j0 + U : i_end;
        // debug builds: the ring slot and the keys it takes (at most U, inside
        // this CTA's share); else nothing is copied and the CTA aborts
        if (!debug_check(p.err, slot >= 0 && slot < NS && j0 >= i_begin && j0 < j1 && j1 - j0 <= U && j1 <= i_end,
                         kSiteRing)) {
          *abort_flag = 1;
          break;
        }
        ptx::mbar_arrive_expect_tx(&bar->full[slot], (uint32_t)((j1 - j0) * Geo::kRow * 2));
        uint8_t* sk = ring + slot * Geo::kSlot;
        uint8_t* sv = sk + U * Geo::kRow;
        // the slot's keys: at most two contiguous runs (a range boundary)
        int j = j0;
        bool copied = true;
        while (j < j1) {
          const int run_end = (j < na && j1 > na) ? na : j1;
          const int k0 = key_at(j);
          // debug builds: the run's cache rows inside the sequence's cached keys
          if (!debug_check(p.err, k0 >= 0 && run_end > j && k0 + (run_end - j) <= len && len <= p.L, kSiteLoad)) {
            copied = false;
            break;
          }
          const uint32_t bytes = (uint32_t)((run_end - j) * Geo::kRow);
          ptx::bulk_load_g2s(sk + (j - j0) * Geo::kRow, kb + (int64_t)k0 * Geo::kRow, bytes, &bar->full[slot]);
          ptx::bulk_load_g2s(sv + (j - j0) * Geo::kRow, vb + (int64_t)k0 * Geo::kRow, bytes, &bar->full[slot]);
          j = run_end;
        }
        if (kDebugChecks && !copied) {
          *abort_flag = 1;
          break;
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the shared memory goes away
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 2000000ull) { }
      }
    }
  } else if (warp < Geo::kCons) {
    // ------------------------------------------------------------ consumers
    // queries of the group, scaled into the log2 domain, this lane's dims
    // as pairs
    float2 q[GP][VPL / 2];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      if (g < G) {
        const uint32_t* src =
            reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + (bh0 + g) * D + lane * VPL);
#pragma unroll
        for (int i = 0; i < VPL / 2; ++i) {
          const uint32_t w = __ldg(src + i);
          q[g][i] = make_float2(bf_lo(w) * p.scale_log2, bf_hi(w) * p.scale_log2);
        }
      } else {
#pragma unroll
        for (int i = 0; i < VPL / 2; ++i) q[g][i] = make_float2(0.f, 0.f);
      }
    }
    const int wlo = gl < G ? window_lo(p, p.head_info[(kvh * G + gl) * 4 + kHeadParam], qpos) : len;
    float* wpw = wp + warp * 32;
    // Group gi of the chunk's slot s sits in ring slot s % NS.  Each (ring
    // slot, group) pair has one owner warp, (slot * GPS + gi) % kCons, which
    // takes that pair's groups in order, round after round: a warp waits for
    // round r of a ring slot only after it consumed round r - 1 itself, so
    // the parity of its wait always names the right round (copies land out
    // of order, so a warp that skipped rounds could mistake an older
    // round's completed phase for the one it waits for).
    for (int gid = 0; gid < nslots * Geo::GPS; ++gid) {
      const int s = gid / Geo::GPS, gi = gid % Geo::GPS;
      const int slot = s % NS;
      if ((slot * Geo::GPS + gi) % Geo::kCons != warp) continue;  // warp-uniform
      // debug builds: the (ring slot, group) pair read inside the ring
      if (kDebugChecks && !__all_sync(0xffffffffu, debug_check(lane == 0 ? p.err : nullptr,
                                                               slot >= 0 && slot < NS && gi >= 0 && gi < Geo::GPS,
                                                               kSiteRing))) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      const bool got = ptx::mbar_wait(&bar->full[slot], (s / NS) & 1, p.timeout_ns, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          *abort_flag = 1;
          atomicOr(p.err, 2u);
        }
        break;
      }
      const uint8_t* sk = ring + slot * Geo::kSlot + lane * VPL * 2;
      const uint8_t* sv = sk + U * Geo::kRow;
      {
        const int i0 = i_begin + s * U + gi * KPG;  // list index of the group's first key
        // partial dot products of the group's KPG keys with the GP queries
        float part[32];
#pragma unroll
        for (int kk = 0; kk < KPG; ++kk) {
          uint32_t kw[VPL / 2];
          load_row_s<VPL>(sk + (gi * KPG + kk) * Geo::kRow, kw);
          float2 kf[VPL / 2];
#pragma unroll
          for (int w = 0; w < VPL / 2; ++w) kf[w] = make_float2(bf_lo(kw[w]), bf_hi(kw[w]));
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            float2 acc = ptx::fmul2(q[g][0], kf[0]);
#pragma unroll
            for (int w = 1; w < VPL / 2; ++w) acc = ptx::ffma2(q[g][w], kf[w], acc);
            part[kk * GP + g] = acc.x + acc.y;
          }
        }
        // reduce-scatter over the lanes: lane j ends with the sum of pair j
#pragma unroll
        for (int off = 16, n = 32; off >= 1; off >>= 1, n >>= 1) {
          const bool upper = (lane & off) != 0;
#pragma unroll
          for (int t = 0; t < n / 2; ++t) {
            const float send = upper ? part[t] : part[t + n / 2];
            const float keep = upper ? part[t + n / 2] : part[t];
            part[t] = keep + __shfl_xor_sync(0xffffffffu, send, off);
          }
        }
        // mask: the pair's key must be in this chunk and visible to head gl
        // (rows of a slot's tail past the chunk hold stale data)
        const int ip = i0 + kl;
        const int key = key_at(ip < i_end ? ip : i_end - 1);
        const bool vis = ip < i_end && gl < G && (key >= wlo || key < S);
        const float x = vis ? part[0] : -INFINITY;
        // online softmax of head gl over the lanes that hold it
        float mx = x;
#pragma unroll
        for (int off = GP; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m, mx);
        const float alpha = (m_new == -INFINITY || m == m_new) ? 1.f : exp2f(m - m_new);
        const float pw = (x == -INFINITY) ? 0.f : exp2f(x - m_new);
        l = l * alpha + pw;
        m = m_new;
        wpw[lane] = pw;
        __syncwarp();
        // O of every head: rescale, then add the group's weighted value rows
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float a = __shfl_sync(0xffffffffu, alpha, g);
          const float2 a2 = make_float2(a, a);
#pragma unroll
          for (int i = 0; i < VPL / 2; ++i) o[g][i] = ptx::fmul2(o[g][i], a2);
        }
#pragma unroll
        for (int kk = 0; kk < KPG; ++kk) {
          if (i0 + kk >= i_end) break;  // warp-uniform: rows past the chunk hold stale data
          uint32_t vw[VPL / 2];
          load_row_s<VPL>(sv + (gi * KPG + kk) * Geo::kRow, vw);
          float2 vf[VPL / 2];
#pragma unroll
          for (int w = 0; w < VPL / 2; ++w) vf[w] = make_float2(bf_lo(vw[w]), bf_hi(vw[w]));
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const float pg = wpw[kk * GP + g];
            const float2 pg2 = make_float2(pg, pg);
#pragma unroll
            for (int t = 0; t < VPL / 2; ++t) o[g][t] = ptx::ffma2(pg2, vf[t], o[g][t]);
          }
        }
        __syncwarp();
      }
      if (lane == 0) ptx::mbar_arrive(&bar->empty[slot]);
    }
  }

  // per head: each consumer warp's sum over the lanes holding it
#pragma unroll
  for (int off = GP; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  __syncthreads();  // every slot consumed: the ring's memory takes the warps' O
  if (warp < kDecConsumers) {
    if (lane < GP) {
      wml[(warp * GP + lane) * 2 + 0] = m;
      wml[(warp * GP + lane) * 2 + 1] = l;
    }
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
      for (int i = 0; i < VPL / 2; ++i) {
        wo[((warp * GP) + g) * D + lane * VPL + 2 * i] = o[g][i].x;
        wo[((warp * GP) + g) * D + lane * VPL + 2 * i + 1] = o[g][i].y;
      }
  }
  __syncthreads();
  if (*abort_flag) return;
  // merge the warps: one thread per (head, dim)
  for (int t = threadIdx.x; t < G * D; t += kDecThreads) {
    const int g = t / D, c = t % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecConsumers; ++w) M = fmaxf(M, wml[(w * GP + g) * 2]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecConsumers; ++w) {
        const float mw = wml[(w * GP + g) * 2];
        if (mw == -INFINITY) continue;
        const float e = exp2f(mw - M);
        L = fmaf(wml[(w * GP + g) * 2 + 1], e, L);
        O = fmaf(wo[((w * GP) + g) * D + c], e, O);
      }
    }
    p.part_o[((bh0 + g) * p.n_split + split) * D + c] = O;
    if (c == 0) {
      part_ml[(int64_t)g * p.n_split * 2 + 0] = M;
      part_ml[(int64_t)g * p.n_split * 2 + 1] = L;
    }
  }
}

// One CTA of D threads per (b, h): O = sum_s O_s 2^(m_s - M) / (sum_s l_s
// 2^(m_s - M) + exp(sink - M')), LSE = ln of the same normaliser.  The
// chunks' weights 2^(m_s - M) are formed once, in shared memory.
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeParams p) {
  __shared__ float es[kDecodeMaxSplits];
  __shared__ float red[D / 32];
  // launched as a programmatic dependent of the split grid: its chunk
  // states are complete and visible past this point
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t bh = blockIdx.x;
  const int h = (int)(bh % p.H);
  const int c = threadIdx.x, warp = c >> 5, lane = c & 31;
  const float* ml = p.part_ml + bh * p.n_split * 2;
  float M = -INFINITY;
  for (int s = c; s < p.n_split; s += D) M = fmaxf(M, ml[2 * s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = -INFINITY;
#pragma unroll
  for (int w = 0; w < D / 32; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  const float b2 = p.sink ? p.sink[h] * kLog2eD : -INFINITY;
  const float Mt = fmaxf(M, b2);
  float L = 0.f;
  for (int s = c; s < p.n_split; s += D) {
    const float ms = ml[2 * s];
    const float e = (ms == -INFINITY) ? 0.f : exp2f(ms - Mt);
    es[s] = e;
    L = fmaf(ml[2 * s + 1], e, L);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  if (lane == 0) red[warp] = L;
  __syncthreads();
  L = 0.f;
#pragma unroll
  for (int w = 0; w < D / 32; ++w) L += red[w];
  float O = 0.f;
  for (int s = 0; s < p.n_split; ++s) {
    const float e = es[s];
    if (e != 0.f) O = fmaf(p.part_o[(bh * p.n_split + s) * D + c], e, O);
  }
  if (b2 != -INFINITY) L += exp2f(b2 - Mt);
  const float out = L > 0.f ? O / L : 0.f;
  if (p.out_f32)
    reinterpret_cast<float*>(p.o)[bh * D + c] = out;
  else
    reinterpret_cast<__nv_bfloat16*>(p.o)[bh * D + c] = __float2bfloat16_rn(out);
  if (c == 0 && p.lse) p.lse[bh] = L > 0.f ? (Mt + __log2f(L)) * kLn2D : -INFINITY;
}

template <int D, int GP>
cudaError_t launch_split(const DecodeParams& p, cudaStream_t stream) {
  using Geo = DecGeo<D, GP>;
  static_assert(Geo::kConsW * GP * D * 4 <= Geo::NS * Geo::kSlot, "the warps' O must fit in the ring");
  const size_t smem = (size_t)Geo::NS * Geo::kSlot + sizeof(DecBar) + Geo::kConsW * 32 * sizeof(float) +
                      Geo::kConsW * GP * 2 * sizeof(float);
  auto kern = decode_split_kernel<D, GP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(p.n_split, p.B * p.H_kv), Geo::kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeParams& p, int gp, cudaStream_t stream) {
  cudaError_t e;
  switch (gp) {
    case 1: e = launch_split<D, 1>(p, stream); break;
    case 2: e = launch_split<D, 2>(p, stream); break;
    case 4: e = launch_split<D, 4>(p, stream); break;
    case 8: e = launch_split<D, 8>(p, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: the combine grid is scheduled while the
  // split grid still runs (each split CTA allows it at its start) and waits
  // in griddepcontrol.wait until the split grid has completed and its
  // writes are visible, so the second launch's latency is hidden.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.B * p.H);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, p);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t stream) {
  const int g = p.H / p.H_kv;
  const int gp = g <= 1 ? 1 : (g <= 2 ? 2 : (g <= 4 ? 4 : 8));
  switch (d) {
    case 64: return launch_d<64>(p, gp, stream);
    case 128: return launch_d<128>(p, gp, stream);
    case 256: return launch_d<256>(p, gp, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mattn
