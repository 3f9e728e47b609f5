// C-ABI odds and ends: error reporting, the wait self-test and the V4.1-Flash
// layer table.
#include "common.cuh"
#include "ptx.cuh"

// the self-test's barrier: initialised for one arrival that never comes
__device__ __forceinline__ void ptx_selftest_init(uint64_t* bar) {
  csa2::ptx::mbar_init(bar, 1);
  csa2::ptx::fence_mbar_init();
}
__device__ __forceinline__ bool ptx_selftest_wait(uint64_t* bar, volatile int* abort_flag, long long budget) {
  return csa2::ptx::mbar_wait(bar, 0, abort_flag, budget);
}

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

// The bounded-wait mechanism every kernel uses, on a barrier that nothing
// completes: one thread waits `budget` clock cycles, gives up and records
// CSA2_ERR_DEVICE_TIMEOUT (detail = the cycles it waited) in the workspace.
namespace csa2 {
namespace {
__global__ void k_wait_selftest(long long budget, void* ws) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  ptx_selftest_init(&bar);
  const long long t0 = clock64();
  int z = 0;
  volatile int* abort_flag = &z;
  if (!ptx_selftest_wait(&bar, abort_flag, budget)) report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, clock64() - t0);
}
}  // namespace
}  // namespace csa2

extern "C" csa2_status csa2_selftest_wait_timeout(long long budget_cycles, void* ws, size_t ws_bytes,
                                                  csa2_stream stream) {
  using namespace csa2;
  if (budget_cycles < 0 || budget_cycles > (1LL << 32)) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < kWsHeader) return CSA2_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;
  k_wait_selftest<<<1, 32, 0, st>>>(budget_cycles, ws);
  return launch_status();
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
