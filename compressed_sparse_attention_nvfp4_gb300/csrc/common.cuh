// Device-side helpers shared by the CSA2 kernels: the FP4/FP8 codec on the
// hardware conversion instructions, the workspace error word, small utilities.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "csa2.h"

namespace csa2 {

constexpr int kDMain = CSA2_D_MAIN;
constexpr int kDIdx = CSA2_D_IDX;
constexpr int kHIdx = CSA2_H_IDX;
constexpr int kHAtt = CSA2_H_ATT;
constexpr size_t kWsHeader = 256;  // error word lives in the first 16 bytes

// ----------------------------------------------------------------------------
// Workspace error word: the first error of a call wins; csa2_check() reads it.
struct ErrWord {
  unsigned int code;
  unsigned int pad;
  long long detail;
};

__device__ __forceinline__ void report_error(void* ws, unsigned code, long long detail) {
  ErrWord* e = reinterpret_cast<ErrWord*>(ws);
  if (atomicCAS(&e->code, 0u, code) == 0u) e->detail = detail;
}

// ----------------------------------------------------------------------------
// Codec.  E2M1 and E4M3 values are exact in f16, so the hardware widening
// conversions decode without rounding.  Packing order of the cvt instructions:
// the first f32 source goes to the upper nibble/byte, the second to the lower.

// one byte of two E2M1 codes (element 2i low nibble) -> two floats (x = low)
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2)
      : "r"(byte));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// two E4M3 bytes (low byte first) -> two floats
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_bytes) {
  uint32_t h2;
  uint16_t v = (uint16_t)two_bytes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

__device__ __forceinline__ float e4m3_to_float(uint32_t b) { return e4m3x2_to_float2(b & 0xFFu).x; }

// E8M0 byte -> 2^(b-127) (exact; b = 0 gives the fp32 subnormal 2^-127)
__device__ __forceinline__ float e8m0_to_float(uint32_t b) {
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// fp32 -> E4M3 byte, round to nearest even, saturating to +-448
__device__ __forceinline__ uint32_t float_to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;
}

// two fp32 -> one byte of E2M1 codes (lo in the low nibble), nearest even, saturating
__device__ __forceinline__ uint32_t float2_to_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// order-preserving map of fp32 to u32 (larger score -> larger key); -inf -> 0
__device__ __forceinline__ uint32_t score_key(float s) {
  if (s == -INFINITY) return 0u;
  uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__host__ __device__ __forceinline__ int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace csa2

// Host helpers shared by the entry points.
namespace csa2 {
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
// Launches kernel k in stream order with programmatic dependent launch: its
// CTAs may be scheduled while the previous kernel of the stream drains, and
// every kernel launched this way starts with griddepcontrol.wait (nothing
// global is touched before the previous kernel has completed).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

// Status of the launches just issued.  With CSA2_DEBUG set in the environment the
// CUDA error string goes to stderr as well.
inline csa2_status launch_status() {
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return CSA2_OK;
  if (getenv("CSA2_DEBUG")) fprintf(stderr, "csa2: launch failed: %s\n", cudaGetErrorString(e));
  return CSA2_ERR_CUDA;
}
inline bool planes_ok(const csa2_kv_planes* kv) {
  return kv && kv->kv_codes && kv->kv_scales && kv->ix_codes && kv->ix_scales &&
         kv->seq_stride > 0 && aligned(kv->kv_codes, 16) && aligned(kv->kv_scales, 16) &&
         aligned(kv->ix_codes, 16) && aligned(kv->ix_scales, 16);
}
// RMSNorm / RoPE parameters: weight 16-byte aligned, eps >= 0, base > 1
inline bool norm_rope_ok(const csa2_norm_rope* nr) {
  if (nr->norm_weight && !aligned(nr->norm_weight, 16)) return false;
  if (!(nr->norm_eps >= 0.0f) || nr->norm_eps > 1.0e30f) return false;
  if (nr->rope && (!(nr->rope_base > 1.0f) || nr->rope_base > 1.0e30f)) return false;
  return true;
}
// clears the error word at the start of a call
inline csa2_status reset_error(void* ws, cudaStream_t st) {
  return cudaMemsetAsync(ws, 0, sizeof(ErrWord), st) == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}
}  // namespace csa2
