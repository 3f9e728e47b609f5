// Lightning indexer + top-k selection.
//   I_j = sum_h w_h ReLU(q_h . K^I_j)   ("DeepSeek-V4: Towards Highly Efficient
//   Million-Token Context Intelligence", CSA step 2; "DeepSeek-V4.1-Flash: pushing
//   the limits of KV cache compression", 4.1), the hierarchical pool of the first
//   decoder Full layer and the Reindex layers' pool-restricted top-k (4.3).
#include <cub/block/block_scan.cuh>

#include "common.cuh"
#include "index_scan.cuh"

namespace csa2 {

// ------------------------------------------------------------------ selection
// Radix select of the k largest keys of one query (one CTA per query), then an
// ordered collection pass: everything above the k-th key, plus the first
// (lowest-index) entries equal to it, written in ascending candidate order.
// Candidates are either entries [0, n) / blocks [0, ceil(n/block)) of the query,
// or the entries of the blocks listed in `pool` (ascending) -- in every case the
// candidate order is the entry (or block) order, so ties go to the lower index.
struct SelectArgs {
  const float* keys;    // [B][key_stride]
  int64_t key_stride;
  const int32_t* n_entries;
  const int32_t* pool;  // [B][keep] or nullptr
  int keep, block;
  int key_by_entry;     // key index = entry id (1) or candidate index (0)
  int count_blocks;     // candidates are the blocks of [0, n)
  int64_t ncand_fixed;  // candidate count when pool != nullptr
  int k;
  int32_t* out;         // [B][out_stride]
  int64_t out_stride;
  int64_t n_max;        // visible entries are clamped to this bound
};

template <int NT>
__device__ __forceinline__ void select_candidate(const SelectArgs& a, int b, int64_t c, int64_t ncand,
                                                 int64_t n, uint32_t& key, int64_t& id) {
  bool valid;
  if (a.pool) {
    int p = a.pool[(int64_t)b * a.keep + c / a.block];
    id = (int64_t)p * a.block + c % a.block;
    valid = c < ncand && p >= 0 && id < n;
  } else {
    id = c;
    valid = c < ncand;
  }
  key = 0u;
  if (valid) key = score_key(a.keys[(int64_t)b * a.key_stride + (a.key_by_entry ? id : c)]);
}

template <int NT>
__global__ void __launch_bounds__(NT) k_select(SelectArgs a) {
  using Scan = cub::BlockScan<int, NT>;
  __shared__ typename Scan::TempStorage scan_tmp;
  __shared__ unsigned hist[256];
  __shared__ unsigned s_valid;
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_need, s_gt;
  __shared__ int s_base_eq, s_base_out;

  const int b = blockIdx.x;
  const int64_t n = max((int64_t)0, min((int64_t)a.n_entries[b], a.n_max));
  const int64_t ncand = a.pool ? a.ncand_fixed : (a.count_blocks ? cdiv(n, a.block) : n);
  int32_t* out = a.out + (int64_t)b * a.out_stride;

  if (threadIdx.x == 0) {
    s_valid = 0;
    s_prefix = 0;
    s_mask = 0;
    s_gt = 0;
  }
  for (int d = threadIdx.x; d < 256; d += NT) hist[d] = 0;
  __syncthreads();

  // count the valid candidates
  unsigned myvalid = 0;
  for (int64_t c = threadIdx.x; c < ncand; c += NT) {
    uint32_t key;
    int64_t id;
    select_candidate<NT>(a, b, c, ncand, n, key, id);
    myvalid += key != 0u;
  }
  atomicAdd(&s_valid, myvalid);
  __syncthreads();
  if (threadIdx.x == 0) s_need = (int)min((int64_t)a.k, (int64_t)s_valid);
  __syncthreads();
  const int need_total = s_need;

  if (need_total > 0) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int d = threadIdx.x; d < 256; d += NT) hist[d] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix, mask = s_mask;
      for (int64_t c = threadIdx.x; c < ncand; c += NT) {
        uint32_t key;
        int64_t id;
        select_candidate<NT>(a, b, c, ncand, n, key, id);
        if (key != 0u && (key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int need = s_need;
        unsigned above = 0;
        int d = 255;
        for (; d > 0; --d) {
          if (above + hist[d] >= (unsigned)need) break;
          above += hist[d];
        }
        s_need = need - (int)above;
        s_gt += (int)above;
        s_prefix = prefix | ((uint32_t)d << shift);
        s_mask = mask | (255u << shift);
      }
      __syncthreads();
    }
  }
  const uint32_t T = s_prefix;
  const int take_eq = s_need;  // entries equal to T to take (lowest indices first)
  if (threadIdx.x == 0) {
    s_base_eq = 0;
    s_base_out = 0;
  }
  __syncthreads();

  if (need_total > 0) {
    for (int64_t c0 = 0; c0 < ncand; c0 += NT) {
      int64_t c = c0 + threadIdx.x;
      uint32_t key = 0u;
      int64_t id = -1;
      if (c < ncand) select_candidate<NT>(a, b, c, ncand, n, key, id);
      int is_eq = (key != 0u && key == T) ? 1 : 0;
      int eq_rank, eq_total;
      Scan(scan_tmp).ExclusiveSum(is_eq, eq_rank, eq_total);
      __syncthreads();
      int take = (key != 0u && key > T) || (is_eq && s_base_eq + eq_rank < take_eq);
      int pos, take_total;
      Scan(scan_tmp).ExclusiveSum(take, pos, take_total);
      if (take) out[s_base_out + pos] = (int32_t)id;
      __syncthreads();
      if (threadIdx.x == 0) {
        s_base_eq += eq_total;
        s_base_out += take_total;
      }
      __syncthreads();
    }
  }
  for (int i = (need_total > 0 ? s_base_out : 0) + threadIdx.x; i < a.k; i += NT) out[i] = -1;
}

// ------------------------------------------------------------------ workspace
struct IndexWs {
  float* scores;
  float* bmax;
  int32_t* pool;
  int64_t score_cols, bmax_cols;
  size_t bytes;
};

static IndexWs index_ws_layout(void* ws, int32_t B, int64_t n_max, int32_t block, int32_t keep) {
  IndexWs L;
  L.score_cols = (int64_t)align_up((size_t)std::max<int64_t>(n_max, (int64_t)keep * block), 64);
  L.bmax_cols = (int64_t)align_up((size_t)cdiv(n_max, block), 64);
  size_t off = kWsHeader;
  size_t s_bytes = (size_t)B * L.score_cols * 4;
  size_t b_bytes = (size_t)B * L.bmax_cols * 4;
  size_t p_bytes = align_up((size_t)B * keep * 4, 256);
  char* base = (char*)ws;
  L.scores = (float*)(base ? base + off : nullptr);
  off += align_up(s_bytes, 256);
  L.bmax = (float*)(base ? base + off : nullptr);
  off += align_up(b_bytes, 256);
  L.pool = (int32_t*)(base ? base + off : nullptr);
  off += p_bytes;
  L.bytes = off;
  return L;
}

}  // namespace csa2

extern "C" size_t csa2_index_topk_workspace_size(int32_t B, int64_t n_max, int32_t k, int32_t block,
                                                 int32_t n_blocks_keep) {
  (void)k;
  if (B <= 0 || n_max < 0 || block <= 0 || n_blocks_keep < 0) return 0;
  return csa2::index_ws_layout(nullptr, B, n_max, block, n_blocks_keep).bytes;
}

extern "C" csa2_status csa2_index_topk(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries,
                                       int64_t n_max, const void* qidx_bf16, const float* w, int32_t k,
                                       csa2_topk_mode mode, int32_t block, int32_t n_blocks_keep,
                                       const int32_t* pool_in, int32_t* topk_out, int32_t* pool_out,
                                       float* scores_out, void* ws, size_t ws_bytes,
                                       csa2_stream stream) {
  using namespace csa2;
  cudaStream_t st = (cudaStream_t)stream;
  if (!planes_ok(kv) || B <= 0 || !n_entries || !qidx_bf16 || !w || !topk_out) return CSA2_ERR_INVALID_ARG;
  if (k < 1 || k > CSA2_MAX_TOPK || n_max < 0 || n_max > kv->seq_stride || n_max >= ((int64_t)1 << 31))
    return CSA2_ERR_INVALID_ARG;
  if (mode != CSA2_TOPK_FLAT && mode != CSA2_TOPK_HIER_BUILD && mode != CSA2_TOPK_POOL)
    return CSA2_ERR_INVALID_ARG;
  if (mode != CSA2_TOPK_FLAT) {
    if (block != 8) return CSA2_ERR_UNSUPPORTED;
    if (n_blocks_keep < 1 || (int64_t)n_blocks_keep * block > 16384) return CSA2_ERR_INVALID_ARG;
    if (mode == CSA2_TOPK_POOL && !pool_in) return CSA2_ERR_INVALID_ARG;
  } else {
    block = 8;
    n_blocks_keep = 0;
  }
  if (!aligned(qidx_bf16, 16) || !aligned(w, 16)) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  IndexWs L = index_ws_layout(ws, B, n_max, block, n_blocks_keep);
  if (ws_bytes < L.bytes) return CSA2_ERR_WORKSPACE;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;

  const uint16_t* q = (const uint16_t*)qidx_bf16;
  const int64_t keep_c = (int64_t)n_blocks_keep * block;

  if (mode == CSA2_TOPK_POOL) {
    float* sc = scores_out ? scores_out : L.scores;
    int64_t sc_stride = scores_out ? keep_c : L.score_cols;
    csa2_status rs = launch_scan(kv, B, n_entries, n_max, keep_c, q, w, pool_in, n_blocks_keep, sc,
                                 sc_stride, nullptr, 0, ws, st);
    if (rs != CSA2_OK) return rs;
    SelectArgs a{sc, sc_stride, n_entries, pool_in, n_blocks_keep, block, 0, 0, keep_c, k,
                 topk_out, k, n_max};
    k_select<1024><<<B, 1024, 0, st>>>(a);
    return launch_status();
  }

  if (mode == CSA2_TOPK_FLAT) {
    float* sc = scores_out ? scores_out : L.scores;
    int64_t sc_stride = scores_out ? n_max : L.score_cols;
    csa2_status rs = launch_scan(kv, B, n_entries, n_max, n_max, q, w, nullptr, 0, sc, sc_stride,
                                 nullptr, 0, ws, st);
    if (rs != CSA2_OK) return rs;
    SelectArgs a{sc, sc_stride, n_entries, nullptr, 0, block, 1, 0, 0, k, topk_out, k, n_max};
    k_select<1024><<<B, 1024, 0, st>>>(a);
    return launch_status();
  }

  // HIER_BUILD: one full scan keeps only the block maxima (entry scores only when
  // asked for); the pool is selected from them; the token top-k re-scores the
  // pool's entries, which costs n_blocks_keep*block entries instead of a 4-byte
  // score per scanned entry.
  csa2_status rs = launch_scan(kv, B, n_entries, n_max, n_max, q, w, nullptr, 0, scores_out, n_max,
                               L.bmax, L.bmax_cols, ws, st);
  if (rs != CSA2_OK) return rs;
  int32_t* pool = pool_out ? pool_out : L.pool;
  SelectArgs pa{L.bmax, L.bmax_cols, n_entries, nullptr, 0, block, 1, 1, 0, n_blocks_keep, pool,
                n_blocks_keep, n_max};
  k_select<1024><<<B, 1024, 0, st>>>(pa);
  rs = launch_scan(kv, B, n_entries, n_max, keep_c, q, w, pool, n_blocks_keep, L.scores,
                   L.score_cols, nullptr, 0, ws, st);
  if (rs != CSA2_OK) return rs;
  SelectArgs ta{L.scores, L.score_cols, n_entries, pool, n_blocks_keep, block, 0, 0, keep_c, k,
                topk_out, k, n_max};
  k_select<1024><<<B, 1024, 0, st>>>(ta);
  return launch_status();
}
