// Indexer scan on the CUDA cores: one thread per candidate entry, q^I held
// transposed in shared memory ([d][h], read as broadcast float4), 32 fp32
// accumulators per thread.  Exact dequantization (E2M1 via cvt, E8M0 as a power
// of two), fp32 accumulation.
#include "index_scan.cuh"

namespace csa2 {

namespace {

constexpr int kScanThreads = 256;

__device__ __forceinline__ float score_entry(const uint8_t* __restrict__ codes,
                                             const uint8_t* __restrict__ scales,
                                             const float (*__restrict__ qT)[kHIdx],
                                             const float* __restrict__ wv) {
  float acc[kHIdx];
#pragma unroll
  for (int h = 0; h < kHIdx; ++h) acc[h] = 0.0f;
  const uint32_t sc = *reinterpret_cast<const uint32_t*>(scales);
#pragma unroll 1
  for (int g = 0; g < 4; ++g) {
    const float s = e8m0_to_float((sc >> (8 * g)) & 0xFFu);
    const uint4 cv = reinterpret_cast<const uint4*>(codes)[g];
    const uint32_t words[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
      for (int bi = 0; bi < 4; ++bi) {
        float2 kv = e2m1x2_to_float2((words[wi] >> (8 * bi)) & 0xFFu);
        kv.x *= s;
        kv.y *= s;
        const int d = g * 32 + wi * 8 + bi * 2;
#pragma unroll
        for (int h4 = 0; h4 < kHIdx / 4; ++h4) {
          float4 q0 = reinterpret_cast<const float4*>(qT[d])[h4];
          float4 q1 = reinterpret_cast<const float4*>(qT[d + 1])[h4];
          acc[4 * h4 + 0] = fmaf(q1.x, kv.y, fmaf(q0.x, kv.x, acc[4 * h4 + 0]));
          acc[4 * h4 + 1] = fmaf(q1.y, kv.y, fmaf(q0.y, kv.x, acc[4 * h4 + 1]));
          acc[4 * h4 + 2] = fmaf(q1.z, kv.y, fmaf(q0.z, kv.x, acc[4 * h4 + 2]));
          acc[4 * h4 + 3] = fmaf(q1.w, kv.y, fmaf(q0.w, kv.x, acc[4 * h4 + 3]));
        }
      }
    }
  }
  float s = 0.0f;
#pragma unroll
  for (int h = 0; h < kHIdx; ++h) s = fmaf(wv[h], fmaxf(acc[h], 0.0f), s);
  return s;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_cuda_core(
    const uint8_t* __restrict__ ix_codes, const uint8_t* __restrict__ ix_scales, int64_t seq_stride,
    const int32_t* __restrict__ n_entries, int64_t ncand_max, const uint16_t* __restrict__ q,
    const float* __restrict__ w, const int32_t* __restrict__ pool, int keep, int block,
    float* __restrict__ scores, int64_t score_stride, float* __restrict__ bmax, int64_t bmax_stride) {
  __shared__ __align__(16) float qT[kDIdx][kHIdx];
  __shared__ float wv[kHIdx];
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < kHIdx * kDIdx; i += blockDim.x) {
    int h = i / kDIdx, d = i % kDIdx;
    qT[d][h] = bf16_bits_to_float(q[(int64_t)b * kHIdx * kDIdx + i]);
  }
  if (threadIdx.x < kHIdx) wv[threadIdx.x] = w[b * kHIdx + threadIdx.x];
  __syncthreads();

  const int64_t n = n_entries[b];
  const int64_t ncand = pool ? ncand_max : (n < ncand_max ? n : ncand_max);
  const int64_t bound = cdiv(ncand, kScanThreads) * kScanThreads;  // warp-uniform trip count
  const uint8_t* codes_b = ix_codes + (int64_t)b * seq_stride * 64;
  const uint8_t* scales_b = ix_scales + (int64_t)b * seq_stride * 4;
  for (int64_t c = (int64_t)blockIdx.x * kScanThreads + threadIdx.x; c < bound;
       c += (int64_t)gridDim.x * kScanThreads) {
    int64_t j = c;
    bool valid = c < ncand;
    if (pool && valid) {
      int p = pool[(int64_t)b * keep + c / block];
      j = (int64_t)p * block + c % block;
      valid = p >= 0 && j < n;
    }
    float s = -INFINITY;
    if (valid) s = score_entry(codes_b + j * 64, scales_b + j * 4, qT, wv);
    if (c < ncand) scores[(int64_t)b * score_stride + c] = s;
    if (bmax) {
      float m = s;
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      if ((c & 7) == 0 && c < ncand) bmax[(int64_t)b * bmax_stride + c / 8] = m;
    }
  }
}

}  // namespace

void launch_scan(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries, int64_t ncand_max,
                 const uint16_t* q, const float* w, const int32_t* pool, int keep, int block,
                 float* scores, int64_t score_stride, float* bmax, int64_t bmax_stride, void* ws,
                 cudaStream_t st) {
  (void)ws;
  if (ncand_max <= 0) return;
  int64_t gx = cdiv(ncand_max, kScanThreads);
  if (gx > 4096) gx = 4096;
  dim3 grid((unsigned)gx, (unsigned)B);
  k_scan_cuda_core<<<grid, kScanThreads, 0, st>>>(kv->ix_codes, kv->ix_scales, kv->seq_stride,
                                                  n_entries, ncand_max, q, w, pool, keep, block,
                                                  scores, score_stride, bmax, bmax_stride);
}

}  // namespace csa2
