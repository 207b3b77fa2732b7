/*
 * mattn.h -- C ABI of libmattn, the masked attention forward for GB300 (sm_103a).
 *
 * The operation (one call computes it for every batch entry b and head h):
 *
 *   O[b,h,i,:] = sum_{j in N_h(i)} a_ij V[b,h,j,:]
 *   a_ij       = exp(s_ij) / ( sum_{j' in N_h(i)} exp(s_ij') + exp(sink_h) )
 *   s_ij       = scale * <Q[b,h,i,:], K[b,h,j,:]>,   scale = 1/sqrt(d) by default
 *   LSE[b,h,i] = log( sum_{j in N_h(i)} exp(s_ij) + exp(sink_h) )   (natural log)
 *
 * Sources: the score and its 1/sqrt(d) scaling -- "Vision transformers and
 * hybrid architectures", section 2 (self-attention from first principles);
 * the per-head sink logit that enters only the denominator -- "Semantic Head
 * Specialization Guides Hybrid ViT Attention for Multimodal LLMs" (SHS
 * slides), the sink slide, Eq. 1; the neighbour set N(i) the softmax runs
 * over -- SHS slides, local-attention recap slide; the block-selection
 * matrix expanded to tokens, M_B[i,j] = B[floor(i/Bs), floor(j/Bs)] and
 * j <= i -- "RRAttention" section 2.1, Eq. 1-2; head-wise causal windows --
 * "Asymmetric Attention Heads", section "What was done" and Table 2.
 *
 * N_h(i) is defined on SEQUENCE POSITIONS.  Each head may read its tokens in
 * a different order (the 1D serialisation of a 2D patch grid, SHS slides
 * "Factor 2"): position p of head h holds caller token t = order_h(p).  The
 * mask is evaluated on positions; O and LSE are returned in caller token
 * order, so one call is a drop-in attention layer.
 *
 * Memory layout: q, k, v and o are dense row-major [B][H][N][d] tensors of
 * one element type (bf16, or fp32 for q/k/v/o with MATTN_F32), base address
 * 16-byte aligned; lse is fp32 [B][H][N].  Supported head dims: 32, 64, 80,
 * 96, 128 and 256 (the head dim of the Bifocal page's speed-test layout;
 * other token orders go through the reorder copy at d = 256).  fp32 inputs are rounded to bf16 on the device before the
 * tensor-core products (accumulation is fp32 throughout); O is written in
 * the input element type.
 *
 * Ownership: the caller owns every buffer and the stream.  The library keeps
 * per-device internal state (work lists, converted or reordered copies of
 * inputs, an error word) that it allocates on first use and reuses; it never
 * synchronises the caller's stream on the normal path (mattn_fwd returns
 * after the launches are queued).
 *
 * Errors: every entry point returns MATTN_OK (0) or a negative mattn_status.
 * Arguments are validated on the host before anything is launched; on error
 * nothing is launched and mattn_last_error() describes the cause.  A device
 * wait that exceeds its time limit (a broken pipeline; it should never
 * happen) makes the kernel record MATTN_ERR_TIMEOUT in the device error word
 * and return early instead of hanging; mattn_device_status() reports it.
 * No entry point aborts or throws.
 *
 * Debug library: libmattn_debug.so is the same library built with
 * MATTN_DEBUG=1.  Its kernels check, before each use, every coordinate
 * handed to a TMA or bulk copy, every work item and key-tile list entry,
 * every explicit-order value (which the product library does not check:
 * an order that is no permutation of 0..N-1 is undefined behaviour there)
 * and every decode ring slot.  A failed check records MATTN_ERR_BOUNDS in
 * the device error word, skips the access, and the CTA returns; nothing
 * traps.  mattn_device_status() then returns MATTN_ERR_BOUNDS with the
 * failed sites in its detail word (bit 5 set; bits 8..13: work item,
 * key-tile entry, load coordinates, store row, explicit-order value, ring
 * slot).  Results are those of the product library otherwise.
 */
#ifndef MATTN_H_
#define MATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MATTN_OK = 0,
  MATTN_ERR_INVALID_ARG = -1,  /* null pointer, bad size, bad mask parameter */
  MATTN_ERR_UNSUPPORTED = -2,  /* valid request outside what is implemented  */
  MATTN_ERR_CUDA = -3,         /* a CUDA runtime / driver call failed         */
  MATTN_ERR_TIMEOUT = -4,      /* a device wait ran past its limit            */
  MATTN_ERR_NO_DEVICE = -5,    /* no sm_103 device is current                 */
  MATTN_ERR_CAPACITY = -6,     /* more than a fixed-size buffer can hold      */
  MATTN_ERR_BOUNDS = -7        /* debug library: a device bounds check failed */
} mattn_status;

/* Mask kinds; all heads of one call share the kind (per-head parameters). */
typedef enum {
  MATTN_FULL = 0,          /* every key                                            */
  MATTN_CHUNK = 1,         /* same chunk: floor(p/C) == floor(q/C)                  */
  MATTN_SLIDING = 2,       /* bidirectional band: |p - q| <= w (w keys per side)    */
  MATTN_CAUSAL_WINDOW = 3, /* causal window of W keys: 0 <= p - q < W               */
  MATTN_BLOCK_SPARSE = 4   /* B[floor(p/Bs)][floor(q/Bs)] and q <= p                */
} mattn_kind;

typedef enum { MATTN_BF16 = 0, MATTN_F32 = 1 } mattn_dtype;

/* Per-head token order codes for mattn_mask_desc.head_order. */
#define MATTN_ORDER_RASTER (-1)       /* identity: position p holds token p             */
#define MATTN_ORDER_COLUMN_MAJOR (-2) /* grid_rows x grid_cols raster grid walked       */
                                      /* column by column: position p = c*rows + r      */
                                      /* holds token r*cols + c                         */
#define MATTN_ORDER_BLOCK2X2_ROW (-3) /* 2x2 patch blocks of the grid, blocks left to right  */
                                      /* then top to bottom, each block's patches in raster */
                                      /* order: position 4*(R*cols/2 + C) + 2*dr + dc holds */
                                      /* token (2R+dr)*cols + 2C+dc (SHS slides, Factor 2,  */
                                      /* order (c); read through TMA when cols % 64 == 0)   */
#define MATTN_ORDER_BLOCK2X2_COL (-4) /* the same blocks top to bottom then left to right:  */
                                      /* position 4*(C*rows/2 + R) + 2*dr + dc (order (d);  */
                                      /* read through TMA when rows % 64 == 0).  Both need  */
                                      /* even grid_rows and grid_cols; a call in which some */
                                      /* head's order is not read through TMA reorders all  */
                                      /* heads through a position-order copy first.         */
/* A value k >= 0 selects explicit order k: perm[k*N + p] = token at position p. */

#define MATTN_TILE 128 /* query / key tile edge of the tile plan */

/* Schedule flags for mattn_mask_desc.flags (results are the same either way,
 * up to floating-point rounding order).  A CTA either takes two neighbouring
 * 128-row query tiles that share each loaded key tile (PAIRED), or one query
 * tile whose key tiles are dealt alternately to two pipelines merged at the
 * end (SPLIT).  With neither flag set the library picks: SPLIT for
 * MATTN_BLOCK_SPARSE with Bs == 128 (neighbouring query tiles then fall in
 * different block rows and share few key tiles), PERSISTENT for the
 * interval masks whose query tiles see about 12 key tiles or fewer on
 * average (short windows and chunks), PAIRED otherwise. */
#define MATTN_FLAG_SCHEDULE_PAIRED 1u
#define MATTN_FLAG_SCHEDULE_SPLIT 2u
/* Head dim 128 only (head dim 256 always runs this way): one 128-row query
 * tile per CTA in a single pipeline whose S is double-buffered in tensor
 * memory, so that the next key tile's Q K^T runs during the softmax of
 * this one.  Other token orders go through the reorder copy. */
#define MATTN_FLAG_SCHEDULE_SINGLE 4u
/* Interval masks (not MATTN_BLOCK_SPARSE), head dim <= 128: the PAIRED work
 * items run on a persistent grid of one CTA per SM, each CTA walking its
 * items back to back: the next item's Q tiles load and its first Q K^T runs
 * while the current item's output is written, instead of every CTA paying
 * its own set-up and epilogue.  A paired item longer than a CTA's share of
 * the launch becomes one item per query tile whose key tiles the two
 * pipelines take in turn, merged at its end (the SPLIT schedule's
 * arithmetic for that query tile: the same result up to rounding order). */
#define MATTN_FLAG_SCHEDULE_PERSISTENT 8u

typedef struct {
  int32_t kind;              /* mattn_kind                                                */
  int32_t param;             /* C, w, W or Bs for every head (ignored for MATTN_FULL);     */
                             /* must be >= 1; MATTN_BLOCK_SPARSE needs Bs % 128 == 0      */
  const int32_t* head_param; /* optional HOST [H]: per-head override of param             */
  const int32_t* head_order; /* optional HOST [H]: MATTN_ORDER_* or explicit order index  */
                             /* (NULL = every head raster)                                */
  int32_t grid_rows;         /* grid of MATTN_ORDER_COLUMN_MAJOR: rows * cols == N         */
  int32_t grid_cols;
  const int32_t* perm;       /* explicit orders, DEVICE int32 [n_perm][N]; each row must   */
  int32_t n_perm;            /* be a permutation of 0..N-1 (not checked on the device)     */
  const uint64_t* block_bits;/* MATTN_BLOCK_SPARSE: DEVICE (mattn_fwd) or HOST (planning    */
                             /* and counting calls) bitmaps [block_heads][Nb][words],      */
                             /* Nb = ceil(N/Bs), words = ceil(Nb/64); bit n of row m is    */
                             /* word[n/64] >> (n%64) & 1 = B[m][n]; bits above the         */
                             /* diagonal are ignored (causality, RRAttention Eq. 5)        */
  int32_t block_heads;       /* 1 (one matrix for all heads) or H                          */
  const float* sink;         /* optional DEVICE fp32 [H] sink logits (NULL = no sink);     */
                             /* HOST for mattn_fwd_host                                    */
  float softmax_scale;       /* 0 => 1/sqrt(d)                                             */
  uint32_t flags;            /* 0 or one MATTN_FLAG_SCHEDULE_* flag                          */
  int32_t sink_tokens;       /* MATTN_CAUSAL_WINDOW only (else must be 0): S >= 0 sink      */
                             /* tokens, the first S positions, visible to every query at    */
                             /* or after them besides its window: query p sees             */
                             /* [p - W + 1, p] and [0, min(S - 1, p)] ("Sliding window      */
                             /* attention vs. linear attention at equal memory" (Bifocal    */
                             /* page): a 572-token window plus the first 4 tokens, the      */
                             /* StreamingLLM sink tokens).  Not to be confused with `sink`, */
                             /* the learned per-head logit.  mattn_received rejects S > 0.  */
} mattn_mask_desc;

/*
 * mattn_fwd -- masked attention forward on the current CUDA device.
 *   q, k, v  DEVICE [B][H][N][d] inputs (dtype: MATTN_BF16 or MATTN_F32).
 *   o        DEVICE [B][H][N][d] output, same dtype as the inputs.
 *   lse      DEVICE fp32 [B][H][N] log-sum-exp output, or NULL.
 *   stream   a cudaStream_t (NULL = legacy default stream).
 * Rows with no visible key and no sink get O = 0 and LSE = -inf.  Work is
 * done only on the 128 x 128 (query, key) tiles that hold at least one
 * visible pair (mattn_plan_tiles lists them); masking is applied only on
 * the PARTIAL ones.  Asynchronous: returns once the work is queued.
 */
int mattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int H, int N, int d, int dtype,
              const mattn_mask_desc* desc, void* stream);

/*
 * mattn_fwd_gqa -- mattn_fwd with grouped-query attention: the H query
 * heads share H_kv key/value heads, query head h reading K/V head
 * h / (H / H_kv) (consecutive query heads form a group).  Source: "Sliding
 * window attention vs. linear attention at equal memory" (Bifocal page),
 * section "Comparison at equal memory": the Qwen3-4B students keep the
 * teacher's grouped-query attention, 32 query heads sharing 8 key/value
 * heads; the speed test's configuration has 16 query heads and 4
 * key/value heads.  Everything else (masks, orders, sink) is per query
 * head, as for mattn_fwd.
 *   q, o     DEVICE [B][H][N][d];  k, v  DEVICE [B][H_kv][N][d];
 *   lse      DEVICE fp32 [B][H][N] or NULL.
 *   H_kv >= 1 and H % H_kv == 0, else MATTN_ERR_INVALID_ARG; H_kv == H is
 *   mattn_fwd.  Other arguments, ownership and errors as for mattn_fwd.
 */
int mattn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                  int B, int H, int H_kv, int N, int d, int dtype,
                  const mattn_mask_desc* desc, void* stream);

/*
 * mattn_decode -- decode-shaped attention: one new query token per
 * sequence against that sequence's key/value cache.  Source: "Sliding
 * window attention vs. linear attention at equal memory" (Bifocal page),
 * "Details", the speed test: each request reads a 1K..128K-token prompt,
 * then generates tokens one by one, with 16 query heads sharing 4
 * key/value heads of dimension 256; the SWA students keep the last 572 or
 * 576 tokens (plus 4 sink tokens, or a learned sink logit).  The query of
 * sequence b sits at position len_b - 1 and sees, per query head h:
 *   MATTN_FULL            every cached key 0 .. len_b - 1;
 *   MATTN_CAUSAL_WINDOW   the last W_h cached keys and the first
 *                         desc->sink_tokens ones;
 * with the optional learned sink logit in the denominator, as mattn_fwd.
 *   q        DEVICE bf16 [B][H][d];   o  DEVICE bf16 [B][H][d];
 *   k, v     DEVICE bf16 [B][H_kv][L][d], the caches (capacity L tokens);
 *            query head h reads key/value head h / (H / H_kv);
 *   lse      DEVICE fp32 [B][H] or NULL;
 *   seq_lens DEVICE int32 [B]: len_b, cached tokens of sequence b with the
 *            new one, or NULL for len_b = L.  Values outside 0..L are
 *            clamped to it; len_b = 0 gives O = 0 and LSE = -inf (or the
 *            sink logit).
 *   d in {64, 128, 256}; H % H_kv == 0 and H / H_kv <= 8; mask kinds
 *   MATTN_FULL or MATTN_CAUSAL_WINDOW, raster order (head_order NULL or all
 *   MATTN_ORDER_RASTER).  Other requests: MATTN_ERR_UNSUPPORTED or
 *   MATTN_ERR_INVALID_ARG, checked on the host before any launch.
 * The library splits each cache into chunks processed in parallel and
 * merges their softmax states (a per-device workspace of B*H*chunks*(d+2)
 * floats, allocated on first use and reused).  Asynchronous, like mattn_fwd.
 */
int mattn_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                 const int32_t* seq_lens, int B, int H, int H_kv, int L, int d, int dtype,
                 const mattn_mask_desc* desc, void* stream);

/*
 * mattn_fwd_host -- the same operation on HOST buffers: copies q, k, v (and
 * the sink and block bitmaps, which are then HOST pointers too) to device
 * memory owned by the library, runs the forward on `stream`, copies o and
 * lse back and synchronises.  The work is cut into chunks of whole heads
 * (about six per call): a second stream owned by the library copies chunk
 * c in and chunk c - 1's output back while `stream` computes, so the
 * copies overlap the kernels.  Pinned host memory gives full copy
 * bandwidth and the overlap; pageable memory works.  lse may be NULL.
 */
int mattn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int d, int dtype,
                   const mattn_mask_desc* desc, void* stream);

/*
 * mattn_fwd_noalloc -- mattn_fwd for callers that must not allocate device
 * memory.  The pages have no counterpart: this entry point serves the
 * library's callers, not the method.
 *
 * Who needs it: mattn_fwd allocates on first use (the work list, the
 * per-head table and the error word of each new mask, with cudaMalloc).
 * Some callers cannot allow that: a framework whose pooling allocator has
 * reserved the device memory up front, so that an allocation outside the
 * pool can fail or go unaccounted; a serving loop that forbids allocation
 * after start-up, because cudaMalloc and cudaFree may synchronise the
 * device and take unbounded time; a plug-in host that hands the operator
 * its buffers and gives it no allocator.  This entry point runs the same
 * attention kernel with that bookkeeping in a fixed static device array
 * inside the library instead, and calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 *   q, k, v, o, lse, B, H, N, d, dtype, desc, stream: as for mattn_fwd.
 *   wait_error_out  optional HOST pointer.  NULL: the call is asynchronous
 *                   like mattn_fwd (a device wait that gives up is then not
 *                   reported).  Non-NULL: the call synchronises `stream`,
 *                   stores the kernel's error word there (0 = none) and
 *                   returns MATTN_ERR_TIMEOUT if it is non-zero
 *                   (MATTN_ERR_BOUNDS if a debug check failed).
 *
 * Limits (the static array is sized for them, MATTN_NOALLOC_SCRATCH_BYTES
 * in all, held on every device that loads the library until the process
 * exits):
 *   - H <= MATTN_NOALLOC_MAX_HEADS;
 *   - at most MATTN_NOALLOC_MAX_ITEMS work items, where a launch has
 *     B*H*ceil(ceil(N/128)/2) items under the paired schedule and
 *     B*H*ceil(N/128) under the split one (the 128K-token, 32-head
 *     block-sparse prefill has 32768);
 *   - bf16 inputs read in place: every head raster, or column-major over a
 *     grid whose row count is a multiple of 128.  fp32 inputs and explicit
 *     orders need a reorder buffer and give MATTN_ERR_UNSUPPORTED.
 * Beyond a limit the call returns MATTN_ERR_CAPACITY (or UNSUPPORTED) with
 * a message in mattn_last_error() and launches nothing.
 *
 * Sharing: every call on a device uses the same static array and leaves
 * its work list there; each call rewrites what it reads and clears the
 * error word first, on `stream`.  Calls whose work overlaps on the GPU
 * (different streams, or several host threads) therefore race on the
 * array: order them, e.g. on one stream.  The first call on a device looks
 * up the array's device address (cudaGetSymbolAddress) with that device
 * current.
 *
 * Graph capture: the work list and the per-head table are uploaded with
 * cudaMemcpyAsync from host memory that lives only for the call, which a
 * captured graph could not replay.  On a stream under capture the call
 * therefore returns MATTN_ERR_UNSUPPORTED and records nothing.
 */
#define MATTN_NOALLOC_MAX_HEADS 4096
#define MATTN_NOALLOC_MAX_ITEMS 65536
#define MATTN_NOALLOC_SCRATCH_BYTES (256 + 16 * MATTN_NOALLOC_MAX_HEADS + 8 * MATTN_NOALLOC_MAX_ITEMS)
int mattn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H, int N, int d, int dtype,
                      const mattn_mask_desc* desc, void* stream, uint32_t* wait_error_out);

/*
 * mattn_received -- received attention, the column sums of the masked
 * attention matrix ("Semantic Head Specialization Guides Hybrid ViT
 * Attention for Multimodal LLMs" (SHS slides), the received-attention slide):
 *   r[b,h,j] = sum over the queries i that may see j of a_ij,
 *   a_ij     = exp(s_ij - lse[b,h,i]),
 * where lse is the log-sum-exp mattn_fwd wrote for the same q, k and mask
 * (so with a sink the rows sum to less than 1 and the sink's share is
 * received by no token; for the mass without the sink, pass the lse of a
 * forward without it).
 *   q, k      DEVICE [B][H][N][d] as for mattn_fwd (same dtypes and orders).
 *   lse       DEVICE fp32 [B][H][N], caller token order (mattn_fwd's output).
 *   r         DEVICE fp32 [B][H][N] output, caller token order.
 *   desc      the mask of the forward (the sink pointer is not read).
 * Asynchronous on `stream`; library workspace (the lse in sequence-position
 * order, reordered inputs when the forward needs them) is allocated on
 * first use.
 */
int mattn_received(const void* q, const void* k, const float* lse, float* r,
                   int B, int H, int N, int d, int dtype,
                   const mattn_mask_desc* desc, void* stream);

/*
 * mattn_rr_select -- RRAttention's dynamic block selection: the block-selection
 * bitmap B of every (batch entry, head), from Q and K ("RRAttention",
 * section 3, Eq. 6-12, with the causality of section 2.1, Eq. 5):
 *   - head h samples one query per stride of `stride` tokens, at offset
 *     stride - 1 - (h mod stride) inside the stride (Eq. 6-7);
 *   - the importance of key stride j for sampled query i is
 *     I_ij = q_i . (sum of the stride's keys) / (stride sqrt(d)) (Eq. 8),
 *     normalised by a softmax over every key stride (Eq. 9);
 *   - block score S_mn = sum of those probabilities over the strides of
 *     query block m and key block n, blocks of `block` tokens (Eq. 10);
 *   - per query block, the key blocks in decreasing score order are kept
 *     until their share of the row's total reaches tau (Eq. 11; equal
 *     scores: smaller block index first), the last query block keeps every
 *     block (Eq. 12), and blocks above the diagonal are dropped (Eq. 5).
 *   With MATTN_RR_SINK_RECENT the first key block and the diagonal block of
 *   every query block are kept too (the page's "sink and recent" option).
 *
 *   q, k         DEVICE bf16 [B][H][N][d], d = 64 or 128, 16-byte aligned.
 *   stride       tokens per stride; must divide N.
 *   block        block size, a multiple of stride with block/stride in
 *                {4, 8, 16, 32} (the page's configuration: stride 8,
 *                block 128).
 *   tau          threshold in (0, 1] (the page uses 0.9 and 0.95).
 *   block_bits   DEVICE output [B*H][Nb][ceil(Nb/64)] uint64, Nb =
 *                ceil(N / block), bit n of row m = B[m][n]: the layout of
 *                mattn_mask_desc.block_bits, one [H][Nb][..] slab per batch
 *                entry.
 *   block_scores optional DEVICE output fp32 [B*H][Nb][Nb], the scores S
 *                (NULL: kept in library memory).
 * Nb must not exceed 8192.  Asynchronous on `stream`; library workspace
 * (the stride key sums, and the scores when block_scores is NULL) is
 * allocated on first use and reused.  A device wait that gives up is
 * reported by mattn_device_status.
 */
#define MATTN_RR_SINK_RECENT 1u
int mattn_rr_select(const void* q, const void* k, int B, int H, int N, int d, int dtype,
                    int stride, int block, float tau, uint32_t flags,
                    uint64_t* block_bits, float* block_scores, void* stream);

/*
 * mattn_plan_schedule -- the schedule mattn_fwd would run for these
 * arguments: one of the MATTN_FLAG_SCHEDULE_* flags (PAIRED, SPLIT, SINGLE,
 * PERSISTENT), the descriptor's own flag if it sets one, else the
 * library's choice (see the schedule flags above).  Host only: validates
 * the arguments as mattn_fwd does (block_bits may be any non-NULL pointer,
 * it is not read) and launches nothing.  The choice follows the rules the
 * library states, not the pages: the pages have no counterpart.
 */
int mattn_plan_schedule(const mattn_mask_desc* desc, int B, int H, int N, int d, int dtype,
                        uint32_t* schedule_out);

/*
 * mattn_count_pairs -- exact number of visible (query, key) pairs summed over
 * B and H (the unit of the effective-FLOP count, 4*d FLOPs per pair).  Host
 * only; block_bits are read as HOST memory.
 */
int mattn_count_pairs(const mattn_mask_desc* desc, int B, int H, int N, uint64_t* pairs_out);

/*
 * mattn_plan_tiles -- the tile plan in position space: for every head h the
 * (query tile, key tile) pairs with at least one visible pair, as int32
 * quadruples (h, qt, kt, cls) sorted by (h, qt, kt); cls = 1 FULL (all
 * 128 x 128 pairs exist and are visible, no masking), 2 PARTIAL (masked
 * elementwise).  Host only, block_bits are HOST memory.  Writes at most
 * `cap` quadruples to `out` (HOST int32 [cap*4], may be NULL when cap == 0)
 * and the total count to *n_out; returns MATTN_ERR_CAPACITY when cap is too
 * small (after setting *n_out).
 */
int mattn_plan_tiles(const mattn_mask_desc* desc, int H, int N, int32_t* out, size_t cap,
                     size_t* n_out);

/*
 * mattn_plan_tiles_device -- the same quadruples, produced by the DEVICE tile
 * walker that mattn_fwd runs (block_bits DEVICE memory), copied back to the
 * HOST buffer `out`.  Synchronises `stream`.
 */
int mattn_plan_tiles_device(const mattn_mask_desc* desc, int H, int N, int32_t* out, size_t cap,
                            size_t* n_out, void* stream);

/*
 * mattn_device_status -- synchronises `stream`, then reads and clears the
 * current device's error word: MATTN_OK; MATTN_ERR_BOUNDS when a debug
 * check failed since the last call (debug library only); else
 * MATTN_ERR_TIMEOUT when a kernel gave up on a wait.  *detail_out (may be
 * NULL) receives the raw word (which wait gave up, which checks failed).
 */
int mattn_device_status(void* stream, uint32_t* detail_out);

/* 1 in the debug library (device bounds checks compiled in), else 0. */
int mattn_debug_checks(void);

/*
 * mattn_set_wait_timeout_ns -- limit for every device-side wait (default
 * 2e9 ns, i.e. 2 s; also read from the environment variable
 * MATTN_WAIT_TIMEOUT_NS at first use).  0 restores the default.
 */
int mattn_set_wait_timeout_ns(uint64_t ns);

/* Human-readable name of a status code (static string). */
const char* mattn_status_string(int status);

/* Message of the last error raised on the calling thread (static per thread). */
const char* mattn_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int mattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MATTN_H_ */
