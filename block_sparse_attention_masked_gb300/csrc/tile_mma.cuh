// Tile geometry and the Q K^T tensor-core product shared by the kernels that
// stage 128-row bf16 tiles of d columns with TMA (attention_fwd.cu and
// rr_select.cu): shared-memory layout of a tile and one M128 N128 MMA chain.
#pragma once

#include <stdint.h>

#include "plan_rules.h"
#include "ptx.cuh"

namespace mattn {

// Shared-memory layout of one 128-row tile of d bf16 columns as TMA writes it.
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
  // V is the MN-major B operand of one N = D MMA per 16 keys (an MMA costs
  // the same ~64 cycles for any N <= 128), so it needs one swizzle across
  // all D columns: atoms of kVW columns (64 -> 128-byte swizzle, 32 -> 64,
  // 16 -> 32), one TMA box per atom column.
  static constexpr int kVW = (D % 64 == 0) ? 64 : ((D % 32 == 0) ? 32 : 16);
  static constexpr int kVChunks = D / kVW;
  static constexpr int kVChunkBytes = kTile * kVW * 2;
  static constexpr uint32_t kVSwizzle = kVW == 64 ? ptx::kSw128 : (kVW == 32 ? ptx::kSw64 : ptx::kSw32);
  static_assert(kVChunks * kVChunkBytes == kTileBytes, "V tile size");
};

__device__ __forceinline__ uint64_t desc_of(uint32_t lo, uint32_t hi) { return ((uint64_t)hi << 32) | lo; }

// S = Q K^T for one sub-tile: D/16 MMAs of M128 N128 K16, both operands K-major.
// Operand addresses are passed pre-shifted (shared address >> 4, the
// descriptor's start-address field): the issuing thread then spends one add
// per operand per MMA, the high descriptor words being compile-time constants.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint32_t q_addr4, uint32_t k_addr4) {
  using G = Geo<D>;
  constexpr uint32_t idesc = ptx::idesc_bf16(128, 128, 0);
  constexpr uint32_t lbo = 1u << 16;  // unused for swizzled K-major operands
  constexpr uint32_t hi128 = ptx::smem_desc_hi(1024, ptx::kSw128);
  constexpr uint32_t hiR = ptx::smem_desc_hi(8 * G::kRemRowBytes, G::kRemSwizzle);
  // Runtime loops (one thread issues): the tensor pipe takes an MMA every
  // ~64 cycles, so unrolling buys nothing and only lengthens the code the
  // issuing warp has to fetch.
  uint32_t acc = 0;
#pragma unroll 1
  for (int step = 0; step < G::kChunks * 4; ++step) {
    const uint32_t off4 = (uint32_t)(((step >> 2) * G::kChunkBytes + (step & 3) * 32) >> 4) + lbo;
    ptx::mma_ss(s_tmem, desc_of(q_addr4 + off4, hi128), desc_of(k_addr4 + off4, hi128), idesc, acc);
    acc = 1;
  }
  if (G::kRem) {
#pragma unroll 1
    for (int k = 0; k < G::kRem / 16; ++k) {
      const uint32_t off4 = (uint32_t)((G::kChunks * G::kChunkBytes + k * 32) >> 4) + lbo;
      ptx::mma_ss(s_tmem, desc_of(q_addr4 + off4, hiR), desc_of(k_addr4 + off4, hiR), idesc, acc);
      acc = 1;
    }
  }
}

}  // namespace mattn
