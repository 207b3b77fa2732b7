// Launch parameters shared by the host API and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mattn {

// Block-sparse masks: capacity of a CTA's key-tile list, so N <= 128 * this.
constexpr int kBlockListMax = 4096;

// Per-head table (device int32 [H][4]).
enum HeadField : int { kHeadParam = 0, kHeadLoad = 1, kHeadStore = 2, kHeadPermRow = 3 };
enum LoadMode : int { kLoadRaster = 0, kLoadColumnMajor = 1, kLoadBlock2x2Row = 2, kLoadBlock2x2Col = 3 };
enum StoreMode : int {
  kStoreIdentity = 0,
  kStoreColumnMajor = 1,
  kStoreExplicit = 2,
  kStoreBlock2x2Row = 3,
  kStoreBlock2x2Col = 4,
};

// Caller token at sequence position pos of a head in store mode `mode` on a
// rows x cols raster grid (perm_row: the head's explicit order, or null).
//   column-major      p = c * rows + r                        -> r * cols + c
//   2x2 blocks, rows  blocks left to right, then top to bottom, each block's
//                     four patches in raster order            -> (2R + dr) * cols + 2C + dc
//   2x2 blocks, cols  blocks top to bottom, then left to right
// (SHS slides, "Factor 2": orders (c) and (d) over the 2x2 patch blocks that
// Qwen2.5-VL merges; the walk inside a block is not given and is read as
// raster).
__host__ __device__ __forceinline__ int64_t token_at(int mode, int64_t rows, int64_t cols, const int32_t* perm_row,
                                                     int64_t pos) {
  if (mode == kStoreColumnMajor) {
    const int64_t c = pos / rows;
    return (pos - c * rows) * cols + c;
  }
  if (mode == kStoreBlock2x2Row || mode == kStoreBlock2x2Col) {
    const int64_t blk = pos >> 2, dr = (pos >> 1) & 1, dc = pos & 1;
    int64_t R, C;
    if (mode == kStoreBlock2x2Row) {
      R = blk / (cols / 2);
      C = blk - R * (cols / 2);
    } else {
      C = blk / (rows / 2);
      R = blk - C * (rows / 2);
    }
    return (2 * R + dr) * cols + 2 * C + dc;
  }
  if (mode == kStoreExplicit) return perm_row[pos];
  return pos;
}

// Device error-word bits: which wait gave up, or which debug check failed.
enum ErrBits : uint32_t {
  kErrProducer = 1u << 0,
  kErrMma = 1u << 1,
  kErrSoftmax = 1u << 2,
  kErrEpilogue = 1u << 3,
  kErrSelfTest = 1u << 4,
  kErrBounds = 1u << 5,    // a debug bounds check failed; the site bits say where
  kSiteItem = 1u << 8,     // a work item: its index or a field of its descriptor
  kSiteKeyTile = 1u << 9,  // a key-tile list entry, or the list's capacity
  kSiteLoad = 1u << 10,    // the coordinates of a TMA or bulk load
  kSiteStore = 1u << 11,   // the row of an O / LSE / output store, or TMA store coordinates
  kSiteOrder = 1u << 12,   // an explicit-order value outside [0, N)
  kSiteRing = 1u << 13,    // a decode ring slot or the key range copied into it
};

// Debug configuration (libmattn_debug.so, compiled with -DMATTN_DEBUG=1):
// before each use, the kernels check every coordinate handed to a TMA or
// bulk copy, every work item and key-tile list entry, every explicit-order
// value and every decode ring slot against the extent it indexes.  A failed
// check ORs kErrBounds and the site's bit into the device error word, raises
// the CTA's abort flag where the CTA has one, and skips the access; the CTA
// then leaves the way it leaves after a timed-out wait.  Nothing traps.  The
// product build compiles every check out.
#ifndef MATTN_DEBUG
#define MATTN_DEBUG 0
#endif
constexpr bool kDebugChecks = MATTN_DEBUG != 0;

#ifdef __CUDACC__
// True when `ok` holds or the checks are compiled out; otherwise records
// the failure (kErrBounds | site) in the error word and returns false.
__device__ __forceinline__ bool debug_check(uint32_t* err, bool ok, uint32_t site) {
  if (!kDebugChecks || ok) return true;
  if (err) atomicOr(err, kErrBounds | site);
  return false;
}
#endif

// A work item of the persistent kernel with its key-tile plan worked out on
// the host (plan_rules.h), six int4 per item:
//   [0] b*H + h, h, b, first query tile qt0 (the item's sub-tiles are qt0, qt0 + 1)
//   [1] list entries n, window start lo, sink entries na, the head's mask parameter
//   [2] window key tiles lo0, hi0, lo1, hi1 of the two sub-tiles (empty: lo > hi)
//   [3] FULL key tiles flo0, fhi0, flo1, fhi1 inside them
//   [4] sink tiles ns0, ns1, load mode | store mode << 8 | split << 16, explicit-order row
//   [5] first and last entries used by sub-tile 0 and by sub-tile 1 (-1: none)
// A split item (bit 16 of [4].z) is one query tile qt0 whose list entries
// alternate between the sub-tiles (entry j to sub-tile j % 2), both with the
// query tile's own plan in [2]-[4]; the sub-tiles' partial results are
// merged at its end.  The host makes long items split so that no CTA waits
// on one item longer than its share of the launch.
constexpr int kPersistItemInt4 = 6;

struct FwdParams {
  // [0]: 64-column chunks (128-byte swizzle); [1]: the 16- or 32-column rest.
  CUtensorMap tq[2], tk[2], tv[2];  // [B*H][N][d] views
  CUtensorMap cq[2], ck[2], cv[2];  // column-major views [B*H][rows][cols][d]
  CUtensorMap bq[2], bk[2], bv[2];  // 2x2-block row-major views [B*H*rows/2][cols/2][2][2][d]
  CUtensorMap bcq[2], bck[2], bcv[2];  // 2x2-block column-major views [cols/2][B*H*rows/2][2][2][d]
  // Views of O matching tq, cq, bq, bcq (bf16 output written with TMA stores
  // when o_tma is set: the persistent kernel at head dim <= 96)
  CUtensorMap o_raster[2], o_colmaj[2], o_blk[2], o_blkc[2];
  void* o;                          // [B][H][N][d], bf16 or fp32
  float* lse;                       // [B][H][N] or null
  const int2* items;                // (b*H + h, query-tile pair), or (b*H + h, query tile) when split
  const int4* pitems;               // persistent kernel: kPersistItemInt4 int4 per work item
  const int* cta_off;               // persistent kernel: CTA c takes pitems [cta_off[c], cta_off[c+1])
  int has_split;                    // persistent kernel: some item is a split item
  const int32_t* head_info;         // [H][4], HeadField
  const int32_t* perm;              // explicit orders [n_perm][N]
  int n_perm;
  const uint64_t* block_bits;       // [block_heads][Nb][wpr]
  const float* sink;                // [H] or null
  uint32_t* err;                    // device error word
  unsigned long long timeout_ns;
  int n_items;
  int B, H, N;
  int H_kv, kv_group;               // K / V heads (tk, ck, tv, cv are [B*H_kv] views);
                                    // query head h reads K / V head h / kv_group
  int kind;
  int sink_tokens;                  // kCausalWindow: first positions every later query sees
  int block_heads, block_wpr, block_c, block_nb;
  int grid_rows, grid_cols;
  float scale_log2;                 // softmax scale * log2(e)
  int self_test_timeout;            // 1: wait on a barrier nothing arrives on (tests)
  int split;                        // 0: a CTA takes two query tiles that share each key tile;
                                    // 1: a CTA takes one query tile, its key tiles dealt
                                    //    alternately to two sub-tile pipelines
                                    //    (head dim 256: one query tile per CTA, one pipeline)
  int out_f32;                      // head dim 256 kernel: O in fp32 (else bf16)
  int o_tma;                        // 1: the O views above are set (bf16 output, every head
                                    // stored in its load order: raster, column-major or 2x2 blocks)
  int after_prepass;                // 1: launched as a programmatic dependent of the reorder
                                    // pre-pass, whose copies its loads read
  int no_partial;                   // 1: no key tile of the launch is PARTIAL for any query
                                    // tile (full or chunk masks on 128-aligned sizes), so the
                                    // kernels run their build without the boundary mask
                                    // (0, the zeroed default: the build with it)
};

struct PlanDumpParams {
  const int32_t* head_info;
  const uint64_t* block_bits;
  int H, N, kind, block_heads, block_wpr, block_c, block_nb;
  int sink_tokens;
  int32_t* out;     // [H][nt][nt][4]
  int32_t* counts;  // [H][nt]
};

struct GatherParams {
  const void* src[3];               // q [B][H][N][d]; k, v [B][H / kv_group][N][d]
  void* dst[3];                     // [B][H][N][d] each (k, v repeated per query head)
  const int32_t* head_info;
  const int32_t* perm;
  int B, H, N, d;
  int kv_group;
  int src_f32;
  int grid_rows, grid_cols;
  int n_perm;
  uint32_t* err;                    // device error word (debug checks)
};

// RRAttention block selection (rr_select.cu).
struct RrParams {
  CUtensorMap tq[2];      // sampled queries: view [B*H][L/S][S][d], 64-column boxes (map [0])
  CUtensorMap tk[2];      // stride key sums [B*H][L/S][d], 64-column boxes (map [0])
  float* block_scores;    // out: [B*H][nb][nb]
  uint32_t* err;          // device error word
  unsigned long long timeout_ns;
  int BH, H, n_s, S, g, nb;  // n_s = L/S strides, g = strides per block, nb blocks
  float scale_log2;       // log2(e) / (S sqrt(d))
};

struct RrSumParams {
  const __nv_bfloat16* k;  // [B*H][N][d]
  __nv_bfloat16* ksum;     // [B*H][N/S][d]
  int BH, N, n_s, d, S;
};

struct RrTopParams {
  const float* scores;  // [B*H][nb][nb]
  uint64_t* bits;       // out: [B*H][nb][wpr]
  int BH, nb, wpr;
  float tau;
  int sink_recent;
};

cudaError_t launch_rr_stride_sum(const RrSumParams& p, cudaStream_t stream);
cudaError_t launch_rr_scores(const RrParams& p, int d, cudaStream_t stream);
cudaError_t launch_rr_topk(const RrTopParams& p, cudaStream_t stream);
size_t rr_scores_smem_bytes(int d);

// Received attention (received.cu).
struct RecvParams {
  CUtensorMap tq[2], tk[2];   // [B*H][N][d] views (map [1]: the 16/32-column rest)
  CUtensorMap cq[2], ck[2];   // column-major views [B*H][rows][cols][d]
  float* lse2p;               // workspace [B*H][lse_pitch]: lse in position order, log2 domain
  float* r;                   // out: [B][H][N] received attention, caller token order
  const int32_t* head_info;   // [H][4], HeadField
  const int32_t* perm;        // explicit orders [n_perm][N]
  int n_perm;
  const uint64_t* block_bits; // [block_heads][Nb][wpr]
  uint32_t* err;
  unsigned long long timeout_ns;
  int64_t lse_pitch;          // a multiple of 128 >= N
  int B, H, N;
  int kind;
  int block_heads, block_wpr, block_c, block_nb;
  int grid_rows, grid_cols;
  float scale_log2;
};

cudaError_t launch_received(const RecvParams& p, const float* lse, int d, cudaStream_t stream);
size_t received_smem_bytes(int d);

// Decode-shaped attention (decode.cu): one query per sequence against its
// key/value cache, split over the cache into chunks.
struct DecodeParams {
  const void* q;              // [B][H][D] bf16
  const void* k;              // [B][H_kv][L][D] bf16
  const void* v;              // [B][H_kv][L][D] bf16
  const int32_t* seq_lens;    // [B] cached tokens per sequence (new token included), or null: L
  const int32_t* head_info;   // [H][4], HeadField (kHeadParam: the window W)
  const float* sink;          // [H] or null
  float* part_o;              // [B*H][n_split][D] chunk states: unnormalised O
  float* part_ml;             // [B*H][n_split][2] chunk states: max (log2 domain), sum
  void* o;                    // [B][H][D] bf16 or fp32
  float* lse;                 // [B][H] or null
  int B, H, H_kv, L;
  int n_split, chunk;         // chunks per sequence, keys per chunk
  int kind;                   // kFull or kCausalWindow
  int sink_tokens;
  float scale_log2;
  int out_f32;
  uint32_t* err;              // device error word (a ring wait that gave up)
  unsigned long long timeout_ns;
};

// Most chunks per sequence a decode launch uses.
constexpr int kDecodeMaxSplits = 1024;

cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t stream);

// Single-pipeline kernel (attention_sp.cu), head dim 256, or 128 on request:
// one query tile per work item, inputs in raster order; tq is a
// [B*H][N][d] view with 64 x 128 boxes, tk and tv [B*H_kv][N][d] views with
// 64 x attention_sp_key_tile(d) boxes (128-byte swizzle).
cudaError_t launch_attention_sp(const FwdParams& p, int d, cudaStream_t stream);
int attention_sp_key_tile(int d);

// Persistent kernel for the interval masks (attention_persist.cu): `grid`
// CTAs (one per SM), CTA c taking work items c, c + grid, ...; the work
// items and parameters are those of launch_attention's paired schedule.
cudaError_t launch_attention_persist(const FwdParams& p, int d, bool out_f32, int grid, cudaStream_t stream);
size_t attention_persist_smem_bytes(int d);

// Launchers (attention_fwd.cu).
cudaError_t launch_attention(const FwdParams& p, int d, bool out_f32, cudaStream_t stream);
size_t attention_smem_bytes(int d);
cudaError_t launch_plan_dump(const PlanDumpParams& p, cudaStream_t stream);
cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream);

}  // namespace mattn
