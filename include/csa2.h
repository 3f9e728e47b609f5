/*
 * csa2.h -- C ABI of the CSA2 decode path over the FP4 global KV cache (sm_103a).
 *
 * Compressed Sparse Attention 2 as described in
 *   "DeepSeek-V4.1-Flash: pushing the limits of KV cache compression"
 *      section 2 (890 bytes/token), 4.1 (single-layer computation), 4.2 (Full /
 *      Reindex / Reuse), 4.3 (Hierarchical Sparse Indexer), 5 (FP4 Main KV Cache);
 *   "DeepSeek-V4.1-Flash course, 02 Architecture"
 *      2.2 Eq. (1), 2.3 CSA2, 2.3.1 cross-layer KV and index reuse, 2.3.2
 *      hierarchical sparse indexer (Fig. 5), 2.4.4 FP4 main KV cache;
 *   "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
 *      CSA step 2 (lightning indexer, top-k), step 3 (shared-KV MQA), the
 *      sliding-window branch.
 *
 * Conventions (all entry points):
 *  - Every pointer argument is DEVICE memory unless stated otherwise; the caller
 *    owns all memory and the stream.  The library allocates nothing and keeps no
 *    mutable global state; calls on different streams with different workspaces
 *    may run concurrently.
 *  - Tensors are dense and row-major.  bf16 tensors are passed as their 16-bit
 *    patterns.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Invalid arguments are reported synchronously and launch
 *    nothing.  A failed launch returns CSA2_ERR_CUDA.
 *  - Errors found on the device (an index out of range, a wait that timed out)
 *    are recorded in the first 16 bytes of the workspace `ws` and read by
 *    csa2_check().  Kernels never trap.
 *  - Workspaces must be 256-byte aligned and at least as large as the matching
 *    *_workspace_size() query; their contents need not be initialised.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- constants */
#define CSA2_D_MAIN 512          /* main-KV latent channels                    */
#define CSA2_D_IDX 128           /* indexer head dimension                     */
#define CSA2_H_IDX 32            /* indexer heads                              */
#define CSA2_H_ATT 64            /* attention query heads (MQA over the latent)*/
#define CSA2_MAIN_CODE_BYTES 256 /* 512 E2M1 codes, 2 per byte                 */
#define CSA2_MAIN_SCALE_BYTES 32 /* one E4M3 scale per 16 channels             */
#define CSA2_IDX_CODE_BYTES 64   /* 128 E2M1 codes                             */
#define CSA2_IDX_SCALE_BYTES 4   /* one E8M0 scale per 32 elements             */
#define CSA2_ENTRY_BYTES 356     /* 288 main + 68 indexer                      */
#define CSA2_MAX_TOPK 2048
#define CSA2_MAX_SWA 128
#define CSA2_MAX_DENSE 65536

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,   /* a pointer, size or alignment is not acceptable   */
  CSA2_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. an unusual m)    */
  CSA2_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small       */
  CSA2_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed             */
  CSA2_ERR_DEVICE_TIMEOUT = 5,/* a bounded device-side wait gave up               */
  CSA2_ERR_INDEX_RANGE = 6    /* a top-k / pool index outside the sequence slot   */
} csa2_status;

typedef void* csa2_stream; /* a cudaStream_t */

/* One Full layer's global KV: four structure-of-arrays planes, 356 B/entry.
 * Entry j of sequence slot s lives at flat index e = s * seq_stride + j.
 *   kv_codes  [e][256]  E2M1 codes of the 512 channels; channel 2i in the low
 *                       nibble of byte i, 2i+1 in the high nibble.
 *   kv_scales [e][32]   E4M3 scale of channels 16g..16g+15 in byte g.
 *   ix_codes  [e][64]   E2M1 codes of the 128-d indexer key, same nibble order.
 *   ix_scales [e][4]    E8M0 scale (2^(b-127)) of elements 32g..32g+31 in byte g.
 * ("DeepSeek-V4.1-Flash: pushing the limits of KV cache compression", section 2:
 *  288 + 68 = 356 bytes per entry.)  Base pointers must be 16-byte aligned, and
 *  ix_codes 32-byte aligned (the indexer reads it with packed 4-bit tensor
 *  loads; csa2_index_topk returns CSA2_ERR_INVALID_ARG otherwise). */
typedef struct {
  uint8_t* kv_codes;
  uint8_t* kv_scales;
  uint8_t* ix_codes;
  uint8_t* ix_scales;
  int64_t seq_stride; /* entries per sequence slot (capacity) */
} csa2_kv_planes;

typedef enum {
  CSA2_TOPK_FLAT = 0,       /* top-k over entries [0, n_entries)                    */
  CSA2_TOPK_HIER_BUILD = 1, /* also build the candidate pool: the n_blocks_keep     */
                            /* blocks of `block` entries with the largest block max */
  CSA2_TOPK_POOL = 2        /* top-k restricted to a given pool (Reindex layers)    */
} csa2_topk_mode;

/* ------------------------------------------------------------- cache format */

/* Quantize fp32 latents into cache entries (the cache format's codec alone).
 *   Cbar [n][512] fp32 -> kv planes; per 16-channel group g:
 *        s = E4M3_rne_satfinite(fp32(amax/6)), code_i = E2M1_rne_satfinite(fp32(x_i/s)),
 *        all-zero codes when s == 0.
 *   KI   [n][128] fp32 -> ix planes; per 32-element group (OCP MXFP4):
 *        X = 2^(floor(log2 amax) - 2) clamped to [2^-127, 2^127], byte = log2 X + 127,
 *        code_i = E2M1_rne_satfinite(x_i / X); amax == 0 gives byte 0, zero codes.
 *   A negative value that rounds to zero keeps its sign (code 8).
 * ("DeepSeek-V4.1-Flash: pushing the limits of KV cache compression", section 5;
 *  "DeepSeek-V4.1-Flash course, 02 Architecture", 2.4.4.)
 * Writes flat entries e0 .. e0+n-1 of `dst`.  Either input may be NULL to skip
 * that half.  Returns CSA2_ERR_INVALID_ARG for n < 0 or misaligned pointers. */
csa2_status csa2_quantize_entries(const float* Cbar, const float* KI, int64_t n,
                                  const csa2_kv_planes* dst, int64_t e0, csa2_stream stream);

/* MXFP4 indexer query ("DeepSeek-V4: Towards Highly Efficient Million-Token Context
 * Intelligence", lightning indexer: the indexer query is quantized to FP4 like its keys):
 * every group of 32 consecutive channels of q_bf16 [n_rows][128] (n_rows = B x 32 heads)
 * becomes E2M1 codes under one E8M0 scale by the indexer-key rule above, and q_out_bf16
 * receives the bf16 values the codes decode to (exact: two significant bits times a power
 * of two).  csa2_index_topk takes the result as its query.  q_out_bf16 may equal q_bf16;
 * both 16-byte aligned. */
csa2_status csa2_quantize_index_query(const void* q_bf16, int64_t n_rows, void* q_out_bf16,
                                      csa2_stream stream);

/* ----------------------------------------------------- in-layer RMSNorm/RoPE */

/* RMSNorm and partial RoPE of a 512-channel vector ("DeepSeek-V4: Towards Highly
 * Efficient Million-Token Context Intelligence", CSA, other details: RMSNorm of
 * every query head and compressed entry before the core attention; RoPE on the
 * last 64 channels of query, KV and output):
 *   y = norm_weight[c] * x[c] / sqrt(mean(x^2) + norm_eps)     when norm_weight != NULL;
 *   channels 448 + 2i, 449 + 2i (i < 32) turned counter-clockwise by
 *   pos * rope_base^(-i/32)                                    when rope != 0.
 * norm_weight is a device array of 512 fp32.  rope_base > 1, norm_eps >= 0. */
typedef struct {
  const float* norm_weight;
  float norm_eps;
  int32_t rope;
  float rope_base;
} csa2_norm_rope;

/* -------------------------------------------------------------- cache write */

/* Prefill cache write of one sequence slot (CED Eq. (1) and the CSA2 compressor):
 *   C = H W_KV, Z = H W_Z  (bf16 inputs, fp32 accumulation),
 *   Cbar_j[c] = sum_{i in B_j} softmax_i(Z_i[c]) C_i[c] over non-overlapping groups
 *   B_j of m consecutive tokens (aligned at token 0),
 *   K^I_j = Cbar_j W_IK  (from the fp32 Cbar, before quantization),
 *   then the codec of csa2_quantize_entries writes entries
 *   entry_offset .. entry_offset + T/m - 1 of slot `seq`.
 * ("DeepSeek-V4.1-Flash course, 02 Architecture", 2.2 Eq. (1) and 2.3;
 *  "DeepSeek-V4.1-Flash: pushing the limits of KV cache compression", 4.1.)
 *   H [T][d_model] bf16; W_KV, W_Z [d_model][512] bf16; W_IK [512][128] bf16.
 * Requires T % m == 0, 1 <= m <= 64 with 64 % m == 0, d_model % 64 == 0.
 * The projection runs on the tensor cores (bf16 operands, fp32 accumulation)
 * for m <= 32 and on the CUDA cores (fp32) for m = 64; the workspace also holds
 * a transposed copy of W_KV and W_Z (2 * d_model * 512 bf16).
 * kv_nr (or NULL): RMSNorm / RoPE of the main-KV copy before its quantization
 * ("DeepSeek-V4.1-Flash course, 02 Architecture", 2.4.4: quantized after RoPE);
 * entry j of the call sits at position pos_first + j * m.  The indexer key
 * keeps the pooled latent. */
csa2_status csa2_cache_write(const void* H_bf16, int64_t T, int32_t d_model, const void* Wkv_bf16,
                             const void* Wz_bf16, const void* Wik_bf16, int32_t m,
                             const csa2_kv_planes* dst, int32_t seq, int64_t entry_offset,
                             const csa2_norm_rope* kv_nr, int64_t pos_first, void* ws,
                             size_t ws_bytes, csa2_stream stream);
size_t csa2_cache_write_workspace_size(int64_t T, int32_t d_model, int32_t m);

/* Decode-time cache append: G groups of m consecutive tokens, each completing one
 * entry of its own sequence slot ("DeepSeek-V4.1-Flash course, 02 Architecture",
 * 3.1: during decode every new token projects its hidden state into a new global KV
 * entry; m = 1 in the decoder, a group completes every m-th token elsewhere).  Each
 * entry is computed exactly as csa2_cache_write computes one:
 *   H [G][m][d_model] bf16, the group's tokens in order;
 *   entry g goes to slot slot[g] (< n_slots), entry index entry[g] (< seq_stride) --
 *   a destination outside the planes is skipped and reported as CSA2_ERR_INDEX_RANGE
 *   through the workspace error word;
 *   kv_nr (or NULL) as in csa2_cache_write, entry g at position pos[g] (required with
 *   RoPE).  slot, entry, pos are device arrays. */
csa2_status csa2_cache_append(const void* H_bf16, int32_t G, int32_t d_model, const void* Wkv_bf16,
                              const void* Wz_bf16, const void* Wik_bf16, int32_t m,
                              const csa2_kv_planes* dst, int32_t n_slots, const int32_t* slot,
                              const int64_t* entry, const csa2_norm_rope* kv_nr, const int64_t* pos,
                              void* ws, size_t ws_bytes, csa2_stream stream);
size_t csa2_cache_append_workspace_size(int32_t G, int32_t d_model, int32_t m);

/* Sliding-window ring write ("DeepSeek-V4 ...", sliding-window branch: every query keeps
 * its last n_win uncompressed rows; "DeepSeek-V4.1-Flash course, 02 Architecture", 2.4.4:
 * they stay FP8): row r, the latent x [R][512] fp32 of a token at position pos[r] of
 * query query[r] (query == NULL: query r), optionally normalised / rotated by nr at
 * pos[r], is encoded as E4M3 (nearest even, saturating at +-448, no scale) into
 * ring[query][pos mod n_win][512] (ring: [n_queries][n_win][512] bytes).  Rows with a
 * negative position or a query outside [0, n_queries) are skipped.  The ring is the
 * swa_e4m3 input of csa2_sparse_attn_decode (n_swa = the rows written so far, at most
 * n_win): the attention does not depend on the order of its rows.  ring_pos (or NULL),
 * [n_queries][n_win] int64, receives each written row's position: the row positions of
 * csa2_window (initialise it to -1 for empty slots). */
csa2_status csa2_swa_append(const float* x, int32_t R, const int32_t* query, const int64_t* pos,
                            int32_t n_queries, const csa2_norm_rope* nr, uint8_t* ring, int64_t* ring_pos,
                            int32_t n_win, csa2_stream stream);

/* ------------------------------------------------------- V4 compressors */

/* The V4 compressors ("DeepSeek-V4: Towards Highly Efficient Million-Token Context
 * Intelligence", CSA step 1 and the HCA section), each writing the T/m compressed
 * latents as fp32 out [T/m][width] (quantize them into a cache with
 * csa2_quantize_entries).  The projections run on the tensor cores (bf16 operands,
 * fp32 sums); the pools take, per channel, one softmax over the scores of the rows
 * an entry draws from, position bias added.
 *
 * csa2_compress_overlap (CSA, two paths a and b, blocks overlapping):
 *   C^a = H W_aKV, C^b = H W_bKV, Z^a = H W_aZ, Z^b = H W_bZ;
 *   entry i draws from rows m i .. m i + m - 1 of path a (score Z^a + B^a[r]) and
 *   rows m (i-1) .. m i - 1 of path b (score Z^b + B^b[r]), 2m rows in all;
 *   entry 0 has no previous block and draws from its m path-a rows alone.
 * csa2_compress_hca (HCA, one path, no overlap): C = H W_KV, Z = H W_Z; entry i
 *   draws from rows m i .. m i + m - 1 (score Z + B[r]); m is m' (128 in V4).
 *
 *   width   output channels c: 512 for the main KV latents, 128 for V4's indexer keys
 *           ("the same compression, projected to c^I"; CSA step 2) -- a multiple of 128, <= 512
 *   H_bf16  [T][d_model] bf16;  W_* [d_model][width] bf16 (row-major, as in H W)
 *   B_*     [m][width] fp32 position biases (finite)
 *   out     [T/m][width] fp32, 16-byte aligned; H and the weights 16-byte aligned
 * T must be a multiple of m (CSA2_ERR_UNSUPPORTED otherwise), 1 <= m <= 1024,
 * d_model a multiple of 64 and >= 64, T < 2^30.  ws: 256-byte aligned, at least
 * csa2_compress_workspace_size(T, d_model) bytes (the unpooled projections; enough for any
 * width). */
csa2_status csa2_compress_overlap(const void* H_bf16, int64_t T, int32_t d_model, const void* Wa_kv,
                                  const void* Wb_kv, const void* Wa_z, const void* Wb_z, const float* Ba,
                                  const float* Bb, int32_t m, int32_t width, float* out, void* ws,
                                  size_t ws_bytes, csa2_stream stream);
csa2_status csa2_compress_hca(const void* H_bf16, int64_t T, int32_t d_model, const void* W_kv,
                              const void* W_z, const float* B, int32_t m, int32_t width, float* out,
                              void* ws, size_t ws_bytes, csa2_stream stream);
size_t csa2_compress_workspace_size(int64_t T, int32_t d_model);

/* ---------------------------------------------------------- indexer + top-k */

/* Lightning-indexer scores and top-k selection for B decode queries; query b
 * reads sequence slot b of `kv`:
 *   I_j = sum_h w[b,h] * ReLU(q[b,h,:] . K^I_j),  h over 32 heads of dim 128,
 *   K^I_j the dequantized MXFP4 key of entry j.
 * Selection order: score descending, then entry index ascending.
 *   FLAT:       the k best of entries [0, n_entries[b]).  For n_max >= 65,536 the call
 *               selects them through the 8-entry block maxima: the k best blocks hold the
 *               k best entries, so a pool of k blocks gives the same set exactly, from two
 *               small selections instead of one over every entry.
 *   HIER_BUILD: block score s_u = max of I_j over block u = [u*block, u*block+block)
 *               (partial last block allowed); the pool is the n_blocks_keep best
 *               blocks (ties to the lower block); topk = the k best entries of the
 *               pool, which equals the FLAT result when n_blocks_keep >= k.  The
 *               scan writes every entry's score (into scores_out, else the
 *               workspace) and the token top-k reads the pool's from there.
 *   POOL:       the k best entries of the blocks listed in pool_in[b] (ascending
 *               block ids, -1 padded), scored with this call's own q and w.
 * ("DeepSeek-V4.1-Flash: pushing the limits of KV cache compression", 4.1, 4.3;
 *  "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence",
 *  CSA step 2.)
 *   n_entries  [B] int32 (device)   visible entries per query, <= n_max
 *   n_max      host upper bound of n_entries, <= kv->seq_stride
 *   qidx_bf16  [B][32][128] bf16;   w [B][32] fp32
 *   topk_out   [B][k] int32: the chosen entry indices in ascending order, -1 padded
 *   pool_out   [B][n_blocks_keep] int32 (HIER_BUILD, optional): block ids ascending
 *   scores_out optional fp32: FLAT/HIER_BUILD [B][n_max] entry scores;
 *              POOL [B][n_blocks_keep*block] candidate scores in pool order
 * Limits: 1 <= k <= 2048; block == 8; n_blocks_keep*block <= 16384; n_max < 2^31. */
csa2_status csa2_index_topk(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries,
                            int64_t n_max, const void* qidx_bf16, const float* w, int32_t k,
                            csa2_topk_mode mode, int32_t block, int32_t n_blocks_keep,
                            const int32_t* pool_in, int32_t* topk_out, int32_t* pool_out,
                            float* scores_out, void* ws, size_t ws_bytes, csa2_stream stream);
size_t csa2_index_topk_workspace_size(int32_t B, int64_t n_max, int32_t k, int32_t block,
                                      int32_t n_blocks_keep);

/* The Reindex layers of one decode step re-score one shared candidate pool -- the
 * decoder Full layer's n_blocks_keep blocks -- over the same indexer keys, each with
 * its own query ("DeepSeek-V4.1-Flash: pushing the limits of KV cache compression",
 * 4.2 Full/Reindex/Reuse table and 4.3: the pool built once is shared by the Reindex
 * layers).  csa2_index_topk in POOL mode gathers the pool's keys on every call; these
 * two calls split that: csa2_pool_stage gathers them once, and every Reindex layer
 * calls csa2_index_topk_staged on the staged copy.  Results are identical to POOL mode.
 *
 * csa2_pool_stage: block u of pool[b] (entries u*8 .. u*8+7 of slot b) goes to staged
 * entries (b*n_blocks_keep + u)*8 .. +7 of
 *   stage_codes  [B][n_blocks_keep*block][64] bytes (MXFP4 codes), 32-byte aligned;
 *   stage_scales [B][n_blocks_keep*block][4] bytes (E8M0), 16-byte aligned;
 * caller-owned device buffers.  Padding (-1) and blocks starting at or beyond
 * n_entries[b] are not copied (their staged bytes stay as they were; the select
 * masks them by their ids).  n_entries, n_max, block, n_blocks_keep as for
 * csa2_index_topk; pool is the [B][n_blocks_keep] pool_out of a HIER_BUILD call.
 * The staged copy is valid while the pool and the slot's indexer keys stay unchanged. */
csa2_status csa2_pool_stage(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries, int64_t n_max,
                            int32_t block, int32_t n_blocks_keep, const int32_t* pool,
                            uint8_t* stage_codes, uint8_t* stage_scales, csa2_stream stream);

/* POOL-mode top-k over planes staged by csa2_pool_stage with the same pool_in,
 * n_entries, n_max, block and n_blocks_keep: the k best entries of the pool's blocks
 * under this call's q and w.  Arguments as for csa2_index_topk (scores_out, if given,
 * [B][n_blocks_keep*block] in pool order); ws: a workspace of
 * csa2_index_topk_workspace_size(B, n_max, k, block, n_blocks_keep) bytes is enough
 * (this call does not use that size's staging part, so less is accepted). */
csa2_status csa2_index_topk_staged(const uint8_t* stage_codes, const uint8_t* stage_scales, int32_t B,
                                   const int32_t* n_entries, int64_t n_max, const void* qidx_bf16,
                                   const float* w, int32_t k, int32_t block, int32_t n_blocks_keep,
                                   const int32_t* pool_in, int32_t* topk_out, float* scores_out, void* ws,
                                   size_t ws_bytes, csa2_stream stream);

/* Allocation-free form of csa2_index_topk (the design pages have no counterpart;
 * this exists for the library's users).  Some callers cannot allocate device
 * memory where they run the indexer -- a plugin handed only its input and output
 * buffers, a serving loop whose memory is partitioned once at start-up with no
 * allocator on the hot path.  This entry point takes the same inputs and outputs
 * (no scores_out, no workspace) and keeps its scratch in a file-scope device
 * array of CSA2_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds
 * until the process exits.  It never allocates or frees device memory.
 *  - Limit: the scratch needed is 256 B + 4*B*(round64(cand) + round64(nb)) +
 *    4*B*keep rounded to 256 B per part, with cand = n_max (FLAT) or
 *    n_blocks_keep*block (HIER_BUILD, POOL) and nb = ceil(n_max/8) (HIER_BUILD
 *    only, plus the pool when pool_out is NULL); a request beyond
 *    CSA2_NOALLOC_SCRATCH_BYTES returns CSA2_ERR_WORKSPACE before any launch.
 *    (Batch 32 at a 1,048,576-entry context in HIER_BUILD needs about 18 MB.)
 *  - The first call on a device looks up the array's device address with that
 *    device current; make that first call before any stream capture.  The
 *    address is cached per CUDA context: after a device reset the first call in
 *    the new context looks it up again (again: before any capture).
 *  - All calls share the one array and it keeps the last call's contents; the
 *    call clears the part that must start at zero.  Calls that overlap on the
 *    GPU (other streams, other threads) race on it and must be serialised.
 *  - Device-side error reports (an n_entries[b] above n_max, clamped, gives
 *    CSA2_ERR_INDEX_RANGE; a bounded wait that gave up, CSA2_ERR_DEVICE_TIMEOUT)
 *    go to the array's error word, which each call clears at its start and
 *    csa2_index_topk_noalloc_check reads; results equal csa2_index_topk's. */
#define CSA2_NOALLOC_SCRATCH_BYTES (32u << 20)

/* Prefill (encoder) indexer: Q queries of one sequence slot `seq` score its entries
 * with the same score and selection rules, query q seeing entries [0, n_visible[q])
 * (its causal bound: the caller counts the entries whose m tokens all precede it),
 * and each keeps its top-k ids (ascending, -1 padded).  This is the O(N^2) indexer
 * work of prefill ("DeepSeek-V4.1-Flash course, 04", decode-cost discussion: the
 * encoder's prefill indexer stays O(N^2), about 3072 N^2 multiply-adds over 3 Full
 * layers).  Every query streams the slot's keys (68 bytes per entry; after the
 * first query they come from L2 when the slot fits).  Queries run in batches whose
 * fp32 scores (with, for n_max >= 65,536, their 8-entry block maxima and a pool of k
 * blocks each, through which the top-k is then selected exactly as FLAT mode does)
 * take about 1.25 GiB of workspace.
 *   qidx [Q][32][128] bf16; w [Q][32] fp32; n_visible [Q] int32 (device);
 *   topk_out [Q][k] int32. */
csa2_status csa2_index_topk_prefill(const csa2_kv_planes* kv, int32_t seq, int32_t Q,
                                    const int32_t* n_visible, int64_t n_max, const void* qidx_bf16,
                                    const float* w, int32_t k, int32_t* topk_out, void* ws,
                                    size_t ws_bytes, csa2_stream stream);
size_t csa2_index_topk_prefill_workspace_size(int32_t Q, int64_t n_max, int32_t k);
csa2_status csa2_index_topk_noalloc(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries,
                                    int64_t n_max, const void* qidx_bf16, const float* w, int32_t k,
                                    csa2_topk_mode mode, int32_t block, int32_t n_blocks_keep,
                                    const int32_t* pool_in, int32_t* topk_out, int32_t* pool_out,
                                    csa2_stream stream);

/* Error word of csa2_index_topk_noalloc (no counterpart on the pages, like the entry point
 * itself): synchronises `stream`, returns the first device-side error recorded by the
 * allocation-free calls since the last call's start (CSA2_OK if none) and clears it, as
 * csa2_check does for a workspace.  *detail (host, may be NULL) receives the offending
 * value (the n_entries value for CSA2_ERR_INDEX_RANGE).  Allocates nothing. */
csa2_status csa2_index_topk_noalloc_check(csa2_stream stream, int64_t* detail);

/* ------------------------------------------------------- sparse attention */

/* Window bounds of an attention call (device arrays; see csa2_sparse_attn_decode). */
typedef struct {
  const int64_t* row_pos; /* [B][n_swa] position of each window row, < 0 = empty */
  const int64_t* lo;      /* [B] lowest visible position of each query */
} csa2_window;

/* Sparse MQA decode over the selected entries joined with the sliding window:
 *   X_b = [ dequant(main KV of topk[b][i], i < k, skipping -1) ; SWA rows of b ]
 *   out[b,h,:] = sum_s softmax_s(softmax_scale * q[b,h,:] . X_b[s]) X_b[s]
 *   lse[b,h]   = natural log of the softmax denominator, max included
 * with K = V = X (one 512-channel latent per entry), 64 heads sharing X.
 * ("DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence",
 *  CSA step 3 and the sliding-window branch; "DeepSeek-V4.1-Flash: pushing the
 *  limits of KV cache compression", 4.1.)
 *   topk      [B][k] int32 entry indices of slot b (-1 = skip)
 *   swa_e4m3  [B][n_swa][512] FP8 E4M3 bytes (no scale), 0 <= n_swa <= 128
 *   q_bf16    [B][64][512] bf16 (unscaled);  out [B][64][512] fp32;  lse_out [B][64] or NULL
 *   softmax_scale  positive and finite (CSA2_ERR_INVALID_ARG otherwise)
 * An index outside [0, seq_stride) is skipped and reported as CSA2_ERR_INDEX_RANGE
 * through the workspace error word.  With no rows, out = 0 and lse = -inf.
 * In-layer extras ("DeepSeek-V4 ...", CSA, other details), each off when NULL:
 *   q_nr      RMSNorm of every query head and/or RoPE of its last 64 channels at
 *             q_pos[b]; with RoPE the output's last 64 channels are turned back
 *             by -q_pos[b] (the cached entries and window rows carry their own);
 *   q_pos     [B] int64 query positions (required when q_nr->rope);
 *   sink      [64] fp32 per-head logits z'_h: exp(z'_h) joins every softmax
 *             denominator (and lse); with no rows out = 0 and lse = z'_h.
 *   win       window bounds (SWA bounded replay, "DeepSeek-V4.1-Flash: pushing the
 *             limits of KV cache compression", section 6: a replay from position s
 *             lets query i see the window [max(s, i - n_win + 1), i]): window row r
 *             of query b joins the softmax only if win->row_pos[b][r] >= max(win->lo[b], 0)
 *             (row_pos < 0 marks an empty row); NULL: every row given is seen.
 * The normalised / rotated q is rounded to f16 for the tensor cores. */
csa2_status csa2_sparse_attn_decode(const csa2_kv_planes* kv, int32_t B, const int32_t* topk,
                                    int32_t k, const uint8_t* swa_e4m3, int32_t n_swa,
                                    const void* q_bf16, float softmax_scale,
                                    const csa2_norm_rope* q_nr, const int64_t* q_pos,
                                    const float* sink, const csa2_window* win, float* out,
                                    float* lse_out, void* ws, size_t ws_bytes, csa2_stream stream);
size_t csa2_sparse_attn_workspace_size(int32_t B, int32_t k, int32_t n_swa);

/* Dense MQA decode over every compressed entry a query sees, joined with the
 * sliding window: HCA's core attention ("DeepSeek-V4: Towards Highly Efficient
 * Million-Token Context Intelligence", HCA section: no indexer and no top-k, the
 * attention reads all compressed entries).  Identical to csa2_sparse_attn_decode
 * with topk[b] = 0, 1, .., n_entries[b] - 1 (one pass, no index list):
 *   n_entries  [B] int32 (device): entries visible to query b (slot b of kv);
 *              values above n_max count as n_max, negative ones as 0
 *   n_max      host bound, 0 <= n_max <= min(CSA2_MAX_DENSE, kv->seq_stride)
 * Every other argument as in csa2_sparse_attn_decode; the workspace is
 * csa2_dense_attn_workspace_size(B, n_max, n_swa) bytes. */
csa2_status csa2_dense_attn_decode(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries,
                                   int64_t n_max, const uint8_t* swa_e4m3, int32_t n_swa,
                                   const void* q_bf16, float softmax_scale, const csa2_norm_rope* q_nr,
                                   const int64_t* q_pos, const float* sink, const csa2_window* win,
                                   float* out, float* lse_out, void* ws, size_t ws_bytes,
                                   csa2_stream stream);
size_t csa2_dense_attn_workspace_size(int32_t B, int64_t n_max, int32_t n_swa);

/* ---------------------------------------------------------------- schedule */

typedef enum { CSA2_LAYER_SWA = 0, CSA2_LAYER_FULL = 1, CSA2_LAYER_REINDEX = 2,
               CSA2_LAYER_REUSE = 3 } csa2_layer_mode;

/* The 40-layer V4.1-Flash layer table ("DeepSeek-V4.1-Flash: pushing the limits of
 * KV cache compression", section 2 layer layout and 4.2/4.3; "DeepSeek-V4.1-Flash
 * course, 02 Architecture", 2.1 and 2.3.1).  For layer l (0-based) it writes
 *   mode[l]      csa2_layer_mode
 *   m[l]         compression ratio of the KV the layer reads (0 for SWA-only)
 *   kv_src[l]    the Full layer p(l) whose main KV and indexer K the layer reads (-1: none)
 *   topk_src[l]  the layer p'(l) whose top-k the layer uses (itself for Full/Reindex, -1: none)
 *   pool_src[l]  for Reindex layers, the decoder Full layer that built the pool (-1: none)
 * Host pointers, n_layers entries each; returns CSA2_ERR_INVALID_ARG unless
 * n_layers == 40. */
csa2_status csa2_v41_layer_table(int32_t n_layers, int32_t* mode, int32_t* m, int32_t* kv_src,
                                 int32_t* topk_src, int32_t* pool_src);

/* ------------------------------------------------------------ kernel timing */

/* Device time per library kernel (instrumentation for users and benchmarks; the
 * design pages have no counterpart).  While enabled, every kernel the library
 * launches is bracketed by two CUDA events recorded on its launch stream (two
 * event records per launch; do not enable it around a stream capture).
 * csa2_timing_enable(on) first folds and then discards every total, and
 * switches recording on (on != 0) or off.  Off by default. */
typedef struct csa2_kernel_time {
  const char* name;  /* kernel name; valid until the next csa2_timing_enable */
  int64_t launches;  /* launches recorded since the last csa2_timing_enable    */
  double total_ms;   /* their summed device time                             */
} csa2_kernel_time;

csa2_status csa2_timing_enable(int32_t on);

/* Waits for the recorded launches, writes up to `max` totals (sorted by name)
 * to `out` (host; may be NULL to count) and returns how many kernels have
 * totals, or -1 if a CUDA event query failed. */
int32_t csa2_kernel_times(csa2_kernel_time* out, int32_t max);

/* ------------------------------------------------------------------ errors */

/* Synchronises `stream`, returns the first device-side error recorded in the
 * workspace `ws` since the last check (CSA2_OK if none) and clears it.
 * *detail (host, may be NULL) receives the offending value. */
csa2_status csa2_check(void* ws, csa2_stream stream, int64_t* detail);

const char* csa2_status_string(csa2_status s);

/* Self-test of the bounded device-side waits every kernel uses: one thread waits
 * on a barrier that nothing completes for `budget_cycles` (0 .. 2^32) clock
 * cycles, gives up and records CSA2_ERR_DEVICE_TIMEOUT in the workspace error
 * word (detail = cycles waited), which csa2_check then returns; the context stays
 * usable.  ws: at least 256 bytes, 256-byte aligned. */
csa2_status csa2_selftest_wait_timeout(long long budget_cycles, void* ws, size_t ws_bytes, csa2_stream stream);

/* Self-test of the main-KV codec's division x / s ("DeepSeek-V4.1-Flash: pushing the limits
 * of KV cache compression", section 5: E2M1(x / s_g)): the codec divides by the group's E4M3
 * scale with an FMA-corrected reciprocal product.  This runs it against the correctly
 * rounded fp32 division for every positive finite E4M3 scale and every fp32 significand of
 * x at the twelve binades where x / s lies in [2^-5, 2^7) (12,683,575,296 comparisons),
 * synchronises `stream`, and writes the number of differing quotients to *mismatches and
 * of comparisons to *compared (host pointers).  ws: device, 256-byte aligned, at least
 * 272 bytes (its counters sit after the 256-byte error header). */
csa2_status csa2_selftest_codec_division(void* ws, size_t ws_bytes, int64_t* mismatches, int64_t* compared,
                                         csa2_stream stream);

/* Self-test of the codec's two element encoders over all 2^32 fp32 bit patterns (the
 * cache format's E2M1 and E4M3 roundings: "DeepSeek-V4.1-Flash: pushing the limits of KV
 * cache compression", section 5; round to nearest even, saturating).  Chunk c
 * (chunk0 <= c < chunk0 + nchunks <= 4096) holds the patterns (c << 20) | i; for every
 * one that is not a NaN, the E2M1 code the codec gives it and the E4M3 byte are summed
 * with weight 2 i + 1 modulo 2^64 into sums[2 (c - chunk0)] and sums[2 (c - chunk0) + 1]
 * (host, 2 * nchunks values), so a reference encoder's sums, formed the same way, must
 * equal them chunk by chunk.  Synchronises `stream`.  ws: device, 256-byte aligned, at
 * least 256 + 16 * nchunks bytes. */
csa2_status csa2_selftest_encode_sweep(uint32_t chunk0, uint32_t nchunks, void* ws, size_t ws_bytes,
                                       uint64_t* sums, csa2_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA2_H */
