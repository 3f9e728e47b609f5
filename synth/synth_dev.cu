/*
 * Device build of the seeded input generator (see synth_core.h for the
 * definition).  Same element-wise results as synth_host.c, bit for bit; used to
 * synthesise the multi-gigabyte inputs of the long-context workloads directly
 * in device memory.  All pointers are device pointers; all calls are
 * asynchronous on the given stream and return the launch status.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth_core.h"

namespace {

enum { K_NORMAL_F32 = 0, K_NORMAL_BF16 = 1, K_UNIFORM_F32 = 2, K_E4M3 = 3, K_KEYS = 4 };

__global__ void fill_kernel(int kind, uint64_t key, uint64_t key2, uint64_t offset, int64_t n,
                            float scale, float hot_prob, const float* hotvec, int32_t dim,
                            void* out) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    uint64_t g = offset + (uint64_t)i;
    switch (kind) {
      case K_NORMAL_F32:
        ((float*)out)[i] = __fmul_rn(syn_normal(key, g), scale);
        break;
      case K_NORMAL_BF16:
        ((uint16_t*)out)[i] = syn_bf16_rne(__fmul_rn(syn_normal(key, g), scale));
        break;
      case K_UNIFORM_F32:
        ((float*)out)[i] = syn_uniform(key, g);
        break;
      case K_E4M3:
        ((uint8_t*)out)[i] = syn_e4m3_rne(__fmul_rn(syn_normal(key, g), scale));
        break;
      case K_KEYS: {
        uint64_t r = g / (uint64_t)dim;
        uint64_t d = g % (uint64_t)dim;
        float v = syn_normal(key, g);
        if (hotvec && syn_uniform(key2, r) < hot_prob) v = __fadd_rn(v, hotvec[d]);
        ((float*)out)[i] = v;
        break;
      }
    }
  }
}

int launch(int kind, uint64_t key, uint64_t key2, uint64_t offset, int64_t n, float scale,
           float hot_prob, const float* hotvec, int32_t dim, void* out, cudaStream_t st) {
  if (n <= 0) return 0;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  fill_kernel<<<(unsigned)blocks, 256, 0, st>>>(kind, key, key2, offset, n, scale, hot_prob, hotvec,
                                                dim, out);
  return (int)cudaGetLastError();
}

}  // namespace

extern "C" {

int syn_dev_normal_f32(uint64_t seed, uint64_t tid, uint64_t offset, int64_t n, float scale,
                       float* out, cudaStream_t st) {
  return launch(K_NORMAL_F32, syn_key(seed, tid), 0, offset, n, scale, 0.f, nullptr, 1, out, st);
}

int syn_dev_normal_bf16(uint64_t seed, uint64_t tid, uint64_t offset, int64_t n, float scale,
                        uint16_t* out, cudaStream_t st) {
  return launch(K_NORMAL_BF16, syn_key(seed, tid), 0, offset, n, scale, 0.f, nullptr, 1, out, st);
}

int syn_dev_uniform_f32(uint64_t seed, uint64_t tid, uint64_t offset, int64_t n, float* out,
                        cudaStream_t st) {
  return launch(K_UNIFORM_F32, syn_key(seed, tid), 0, offset, n, 1.f, 0.f, nullptr, 1, out, st);
}

int syn_dev_e4m3_normal(uint64_t seed, uint64_t tid, uint64_t offset, int64_t n, float scale,
                        uint8_t* out, cudaStream_t st) {
  return launch(K_E4M3, syn_key(seed, tid), 0, offset, n, scale, 0.f, nullptr, 1, out, st);
}

int syn_dev_keys(uint64_t seed, uint64_t tid, uint64_t tid_hot, uint64_t offset, int64_t n,
                 int32_t dim, float hot_prob, const float* hotvec, float* out, cudaStream_t st) {
  return launch(K_KEYS, syn_key(seed, tid), syn_key(seed, tid_hot), offset, n, 1.f, hot_prob,
                hotvec, dim, out, st);
}

}  // extern "C"
