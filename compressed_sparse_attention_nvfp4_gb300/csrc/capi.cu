// C-ABI odds and ends: error reporting and the V4.1-Flash layer table.
#include "common.cuh"

extern "C" const char* csa2_status_string(csa2_status s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported argument combination";
    case CSA2_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case CSA2_ERR_CUDA: return "CUDA runtime or launch error";
    case CSA2_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
    case CSA2_ERR_INDEX_RANGE: return "an index outside its sequence slot";
  }
  return "unknown status";
}

extern "C" csa2_status csa2_check(void* ws, csa2_stream stream, int64_t* detail) {
  using namespace csa2;
  if (!ws) return CSA2_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  ErrWord e;
  if (cudaMemcpyAsync(&e, ws, sizeof(e), cudaMemcpyDeviceToHost, st) != cudaSuccess) return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return CSA2_ERR_CUDA;
  if (detail) *detail = e.detail;
  if (e.code != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof(e), st) != cudaSuccess) return CSA2_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return CSA2_ERR_CUDA;
  }
  return (csa2_status)e.code;
}

// Layer layout of "DeepSeek-V4.1-Flash: pushing the limits of KV cache
// compression", section 2: layers 0-1 SWA only; encoder = 3 x (1 Full + 5 Reuse)
// at m = 2; decoder = (1 Full + 3 Reuse) + 4 x (1 Reindex + 3 Reuse) at m = 1.
// Sources per section 4.2: p(l) = the nearest Full layer at or before l,
// p'(l) = the nearest Full or Reindex layer at or before l; Reindex layers
// search the pool built by the first decoder Full layer (section 4.3).
extern "C" csa2_status csa2_v41_layer_table(int32_t n_layers, int32_t* mode, int32_t* m,
                                            int32_t* kv_src, int32_t* topk_src, int32_t* pool_src) {
  if (n_layers != 40 || !mode || !m || !kv_src || !topk_src || !pool_src) return CSA2_ERR_INVALID_ARG;
  int last_full = -1, last_index = -1, decoder_full = -1;
  for (int l = 0; l < 40; ++l) {
    int md, ratio;
    if (l < 2) {
      md = CSA2_LAYER_SWA;
      ratio = 0;
    } else if (l < 20) {
      md = ((l - 2) % 6 == 0) ? CSA2_LAYER_FULL : CSA2_LAYER_REUSE;
      ratio = 2;
    } else {
      const int r = (l - 20) % 4, grp = (l - 20) / 4;
      md = r != 0 ? CSA2_LAYER_REUSE : (grp == 0 ? CSA2_LAYER_FULL : CSA2_LAYER_REINDEX);
      ratio = 1;
    }
    if (md == CSA2_LAYER_FULL) {
      last_full = l;
      last_index = l;
      if (l >= 20 && decoder_full < 0) decoder_full = l;
    } else if (md == CSA2_LAYER_REINDEX) {
      last_index = l;
    }
    mode[l] = md;
    m[l] = ratio;
    kv_src[l] = md == CSA2_LAYER_SWA ? -1 : last_full;
    topk_src[l] = md == CSA2_LAYER_SWA ? -1 : last_index;
    pool_src[l] = md == CSA2_LAYER_REINDEX ? decoder_full : -1;
  }
  return CSA2_OK;
}
