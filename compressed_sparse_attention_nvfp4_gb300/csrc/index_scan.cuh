// Indexer scan launcher: scores every candidate of every query and, for the
// hierarchical build, the max of every 8-entry block.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace csa2 {

// cuTensorMapEncodeTiled from the driver (null if unavailable); shared by the
// kernels that build tensor maps.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn();

// Scores the candidates of B queries (query b reads sequence slot b).
// ncand_max: entries (pool == nullptr; n_entries[b] <= n_max are visible) or
// pool candidates keep*8 per query (pool blocks of 8 entries).
// scores[b*score_stride + c] (if non-null) receives the score of candidate c
// (-inf if invalid); bmax[b*bmax_stride + u] (if non-null) the max over entries
// 8u..8u+7.
csa2_status launch_scan(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries, int64_t n_max,
                        int64_t ncand_max, const uint16_t* q, const float* w, const int32_t* pool,
                        int keep, float* scores, int64_t score_stride, float* bmax, int64_t bmax_stride,
                        void* ws, cudaStream_t st, int shared_slot = -1);

// Prefill scores: Q queries over sequence slot `slot` (query b sees its first
// n_visible[b] <= n_max entries), four queries per key tile; scores[b][j] for
// j < n_visible[b] (the rest of each row is left as it was), and with bmax non-null
// bmax[b][u] = the maximum of the visible scores of block u = [8 u, 8 u + 8) for the
// blocks that start below n_visible[b].
csa2_status launch_scan_prefill(const csa2_kv_planes* kv, int32_t Q, const int32_t* n_visible, int64_t n_max,
                                const uint16_t* q, const float* w, float* scores, int64_t score_stride, float* bmax,
                                int64_t bmax_stride, void* ws, cudaStream_t st, int slot);

}  // namespace csa2
