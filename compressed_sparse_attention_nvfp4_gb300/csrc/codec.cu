// Cache-format codec: fp32 latents -> E2M1 codes with E4M3 (main KV) or E8M0
// (indexer key) group scales.  "DeepSeek-V4.1-Flash: pushing the limits of KV
// cache compression", section 5 (s_g = E4M3(max|x|/6), xhat = s_g E2M1(x/s_g));
// "DeepSeek-V4.1-Flash course, 02 Architecture", 2.4.4 (OCP MXFP4 indexer key).
#include "codec.cuh"
#include "timing.cuh"

namespace csa2 {

__global__ void k_quantize_main(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ codes,
                                uint8_t* __restrict__ scales, QDest d) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n * 32) return;
  const int64_t row = dest_row(d, t / 32);
  if (row < 0) return;
  quantize_main_group(x + t * 16, codes + row * 256 + (t % 32) * 8, scales + row * 32 + t % 32);
}

__global__ void k_quantize_index(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ codes,
                                 uint8_t* __restrict__ scales, QDest d) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n * 4) return;
  const int64_t row = dest_row(d, t / 4);
  if (row < 0) return;
  quantize_index_group(x + t * 32, codes + row * 64 + (t % 4) * 16, scales + row * 4 + t % 4);
}

// The main-KV quantizer with RMSNorm and RoPE first ("DeepSeek-V4: ...", CSA,
// other details; "DeepSeek-V4.1-Flash course, 02 Architecture", 2.4.4: the
// cache is quantized after RoPE): one warp per entry, lane l holds channels
// 16l .. 16l + 15 (its quantization group), the rotated pairs sit in lanes 28-31.
__global__ void k_quantize_main_nr(const float* __restrict__ x, int64_t n, const float* __restrict__ w,
                                   float eps, int rope, RopeTheta th, uint8_t* __restrict__ codes,
                                   uint8_t* __restrict__ scales, QDest d) {
  const int64_t e = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (e >= n) return;  // whole warps leave together
  const int64_t row = dest_row(d, e);
  if (row < 0) return;  // the same for the whole warp
  quantize_main_entry_warp(x + e * kDMain, w, eps, rope, th, rope ? (double)dest_pos(d, e) : 0.0,
                           codes + row * 256, scales + row * 32, lane);
}

// Self-test of div_by_e4m3: for positive E4M3 scale byte blockIdx.y + 1 and every fp32
// significand of x at the 12 binades around x / s in [2^-5, 2^7), the corrected quotient
// against __fdiv_rn; mismatches counted into *bad, comparisons into *n.
__global__ void __launch_bounds__(256) k_selftest_division(unsigned long long* bad, unsigned long long* n) {
  const int sb = blockIdx.y + 1;  // E4M3 bytes 1..126: the positive finite values
  const float s = e4m3_to_float((uint32_t)sb);
  const float r = __frcp_rn(s);
  const int es = ilogbf(s);
  unsigned long long nb = 0, nn = 0;
  for (uint32_t m = blockIdx.x * blockDim.x + threadIdx.x; m < (1u << 23); m += gridDim.x * blockDim.x) {
    const float sig = 1.0f + (float)m * 0x1p-23f;
    for (int e = -5; e < 7; ++e) {
      const float x = ldexpf(sig, es + e);
      nb += __float_as_uint(div_by_e4m3(x, s, r)) != __float_as_uint(__fdiv_rn(x, s)) ? 1u : 0u;
      ++nn;
    }
  }
  atomicAdd(bad, nb);
  atomicAdd(n, nn);
}

// Self-test of the codec's element encoders over every fp32 bit pattern: chunk c
// (blockIdx.y + chunk0) holds the 2^20 patterns (c << 20) | i.  For each pattern that is
// not a NaN, the E2M1 code (the codec's fp32 -> E2M1 conversion) and the E4M3 byte (its
// fp32 -> E4M3 scale conversion) are summed with weight 2 i + 1 modulo 2^64 into
// sums[c - chunk0][0] and [1]: any single differing code changes its chunk's sum.
constexpr int kSweepChunkBits = 20;
__global__ void __launch_bounds__(256) k_selftest_encode_sweep(uint32_t chunk0, unsigned long long* sums) {
  const uint32_t c = chunk0 + blockIdx.y;
  constexpr uint32_t per_cta = (1u << kSweepChunkBits) / 64;  // gridDim.x == 64
  unsigned long long s2 = 0, s4 = 0;
  for (uint32_t j = threadIdx.x; j < per_cta; j += blockDim.x) {
    const uint32_t i = blockIdx.x * per_cta + j;
    const uint32_t bits = (c << kSweepChunkBits) | i;
    if ((bits & 0x7F800000u) == 0x7F800000u && (bits & 0x007FFFFFu) != 0u) continue;  // NaN
    const float x = __uint_as_float(bits);
    const unsigned long long wgt = 2ull * i + 1ull;
    s2 += (unsigned long long)(float2_to_e2m1x2(x, 0.0f) & 0xFu) * wgt;
    s4 += (unsigned long long)float_to_e4m3(x) * wgt;
  }
  for (int o = 16; o > 0; o >>= 1) {
    s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    s4 += __shfl_xor_sync(0xffffffffu, s4, o);
  }
  if (threadIdx.x % 32 == 0) {
    atomicAdd(&sums[2 * blockIdx.y], s2);
    atomicAdd(&sums[2 * blockIdx.y + 1], s4);
  }
}

void launch_quantize(const float* Cbar, const float* KI, int64_t n, const csa2_kv_planes* dst, const QDest& d,
                     cudaStream_t st, const csa2_norm_rope* nr) {
  if (n <= 0) return;
  if (Cbar && nr && (nr->norm_weight || nr->rope)) {
    KernelTimer timer("k_quantize_main_nr", st);
    k_quantize_main_nr<<<(unsigned)cdiv(n * 32, 256), 256, 0, st>>>(
        Cbar, n, nr->norm_weight, nr->norm_eps, nr->rope, nr->rope ? make_rope_theta(nr->rope_base) : RopeTheta{},
        dst->kv_codes, dst->kv_scales, d);
  } else if (Cbar) {
    int64_t threads = n * 32;
    KernelTimer timer("k_quantize_main", st);
    k_quantize_main<<<(unsigned)cdiv(threads, 256), 256, 0, st>>>(Cbar, n, dst->kv_codes, dst->kv_scales, d);
  }
  if (KI) {
    int64_t threads = n * 4;
    KernelTimer timer("k_quantize_index", st);
    k_quantize_index<<<(unsigned)cdiv(threads, 256), 256, 0, st>>>(KI, n, dst->ix_codes, dst->ix_scales, d);
  }
}

// MXFP4 indexer query: one thread per group of 32 consecutive channels, quantized
// by the indexer-key rule and written back as the bf16 values the codes decode to
// (E2M1 times a power of two: exact in bf16, subnormal scales included).
__global__ void k_quantize_query_mxfp4(const uint16_t* __restrict__ q, int64_t ngroups, uint16_t* __restrict__ out) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= ngroups) return;
  const uint4* src = reinterpret_cast<const uint4*>(q + t * 32);
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 r = src[i];
    const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(w4[j] << 16);
      v[8 * i + 2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
    }
  }
  __align__(16) uint8_t codes[16];
  uint8_t sb;
  quantize_index_group_vals(v, codes, &sb);
  const float X = e8m0_to_float(sb);
  uint32_t o[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {  // byte i: elements 2i (low nibble), 2i + 1
    const float2 e = e2m1x2_to_float2(codes[i]);
    const uint32_t lo = __float_as_uint(e.x * X) >> 16, hi = __float_as_uint(e.y * X) >> 16;
    o[i] = lo | (hi << 16);
  }
  uint4* dst = reinterpret_cast<uint4*>(out + t * 32);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

// Window ring write: one warp per row; lane l holds channels 16l .. 16l + 15,
// optional RMSNorm and RoPE (pairs in lanes 28-31), then E4M3 (nearest even,
// saturating, no scale) into ring[query][pos mod n_win].  Rows with a negative
// position or a query outside [0, n_queries) are skipped.
__global__ void k_swa_append(const float* __restrict__ x, int32_t R, const int32_t* __restrict__ query,
                             const int64_t* __restrict__ pos, int32_t n_queries, const float* __restrict__ w,
                             float eps, int rope, RopeTheta th, uint8_t* __restrict__ ring,
                             int64_t* __restrict__ ring_pos, int32_t n_win) {
  const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (r >= R) return;
  const int64_t p = pos[r];
  const int32_t b = query ? query[r] : (int32_t)r;
  if (p < 0 || b < 0 || b >= n_queries) return;  // the same for the whole warp
  float v[16];
  const float4* src = reinterpret_cast<const float4*>(x + r * kDMain + lane * 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = src[i];
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
  if (w) {
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ss = fmaf(v[i], v[i], ss);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.0f / sqrtf(ss / (float)kDMain + eps);
    const float4* wv = reinterpret_cast<const float4*>(w + lane * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 g = wv[i];
      v[4 * i] = g.x * (v[4 * i] * inv);
      v[4 * i + 1] = g.y * (v[4 * i + 1] * inv);
      v[4 * i + 2] = g.z * (v[4 * i + 2] * inv);
      v[4 * i + 3] = g.w * (v[4 * i + 3] * inv);
    }
  }
  if (rope && lane * 16 >= kRopeFirst) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float c, sn;
      rope_cos_sin(th.t[(lane * 16 - kRopeFirst) / 2 + q], (double)p, c, sn);
      rope_pair(v[2 * q], v[2 * q + 1], c, sn);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = float_to_e4m3(v[4 * i]) | (float_to_e4m3(v[4 * i + 1]) << 8) | (float_to_e4m3(v[4 * i + 2]) << 16) |
           (float_to_e4m3(v[4 * i + 3]) << 24);
  uint8_t* dst = ring + ((int64_t)b * n_win + p % n_win) * kDMain + lane * 16;
  *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
  if (ring_pos && lane == 0) ring_pos[(int64_t)b * n_win + p % n_win] = p;
}

}  // namespace csa2

extern "C" csa2_status csa2_swa_append(const float* x, int32_t R, const int32_t* query, const int64_t* pos,
                                       int32_t n_queries, const csa2_norm_rope* nr, uint8_t* ring,
                                       int64_t* ring_pos, int32_t n_win, csa2_stream stream) {
  using namespace csa2;
  if (R < 0 || n_queries <= 0 || n_win <= 0) return CSA2_ERR_INVALID_ARG;
  if (R > 0 && (!x || !pos || !ring || !aligned(x, 16) || !aligned(pos, 8) || !aligned(ring, 16) ||
                (query && !aligned(query, 4)) || (ring_pos && !aligned(ring_pos, 8))))
    return CSA2_ERR_INVALID_ARG;
  if (nr && !norm_rope_ok(nr)) return CSA2_ERR_INVALID_ARG;
  if (R == 0) return CSA2_OK;
  cudaStream_t st = (cudaStream_t)stream;
  const bool rope = nr && nr->rope;
  KernelTimer timer("k_swa_append", st);
  k_swa_append<<<(unsigned)cdiv((int64_t)R * 32, 256), 256, 0, st>>>(
      x, R, query, pos, n_queries, nr ? nr->norm_weight : nullptr, nr ? nr->norm_eps : 0.0f, rope ? 1 : 0,
      rope ? make_rope_theta(nr->rope_base) : RopeTheta{}, ring, ring_pos, n_win);
  return launch_status();
}

extern "C" csa2_status csa2_quantize_index_query(const void* q_bf16, int64_t n_rows, void* q_out_bf16,
                                                 csa2_stream stream) {
  using namespace csa2;
  if (n_rows < 0 || (n_rows > 0 && (!q_bf16 || !q_out_bf16))) return CSA2_ERR_INVALID_ARG;
  if ((q_bf16 && !aligned(q_bf16, 16)) || (q_out_bf16 && !aligned(q_out_bf16, 16))) return CSA2_ERR_INVALID_ARG;
  if (n_rows == 0) return CSA2_OK;
  if (n_rows > (int64_t)1 << 34) return CSA2_ERR_UNSUPPORTED;
  const int64_t ngroups = n_rows * (kDIdx / 32);
  cudaStream_t st = (cudaStream_t)stream;
  KernelTimer timer("k_quantize_query_mxfp4", st);
  k_quantize_query_mxfp4<<<(unsigned)cdiv(ngroups, 256), 256, 0, st>>>((const uint16_t*)q_bf16, ngroups,
                                                                     (uint16_t*)q_out_bf16);
  return launch_status();
}

extern "C" csa2_status csa2_quantize_entries(const float* Cbar, const float* KI, int64_t n,
                                             const csa2_kv_planes* dst, int64_t e0,
                                             csa2_stream stream) {
  using namespace csa2;
  if (n < 0 || e0 < 0 || !planes_ok(dst)) return CSA2_ERR_INVALID_ARG;
  if ((Cbar && !aligned(Cbar, 16)) || (KI && !aligned(KI, 16))) return CSA2_ERR_INVALID_ARG;
  if (n == 0) return CSA2_OK;
  if (n > (int64_t)1 << 36) return CSA2_ERR_UNSUPPORTED;
  QDest d{};
  d.e0 = e0;
  launch_quantize(Cbar, KI, n, dst, d, (cudaStream_t)stream, nullptr);
  return launch_status();
}

extern "C" csa2_status csa2_selftest_codec_division(void* ws, size_t ws_bytes, int64_t* mismatches,
                                                    int64_t* compared, csa2_stream stream) {
  using namespace csa2;
  if (!mismatches || !compared) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < kWsHeader + 2 * sizeof(unsigned long long)) return CSA2_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned long long* d = reinterpret_cast<unsigned long long*>((char*)ws + kWsHeader);  // two counters
  if (cudaMemsetAsync(d, 0, 2 * sizeof(unsigned long long), st) != cudaSuccess) return CSA2_ERR_CUDA;
  k_selftest_division<<<dim3(512, 126), 256, 0, st>>>(d, d + 1);
  unsigned long long h[2] = {0, 0};
  if (cudaMemcpyAsync(h, d, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return CSA2_ERR_CUDA;
  *mismatches = (int64_t)h[0];
  *compared = (int64_t)h[1];
  return CSA2_OK;
}

extern "C" csa2_status csa2_selftest_encode_sweep(uint32_t chunk0, uint32_t nchunks, void* ws, size_t ws_bytes,
                                                  uint64_t* sums, csa2_stream stream) {
  using namespace csa2;
  constexpr uint32_t kChunks = 1u << (32 - kSweepChunkBits);
  if (!sums || nchunks == 0 || chunk0 >= kChunks || nchunks > kChunks - chunk0) return CSA2_ERR_INVALID_ARG;
  const size_t need = kWsHeader + (size_t)nchunks * 2 * sizeof(unsigned long long);
  if (!ws || !aligned(ws, 256) || ws_bytes < need) return CSA2_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned long long* d = reinterpret_cast<unsigned long long*>((char*)ws + kWsHeader);
  if (cudaMemsetAsync(d, 0, (size_t)nchunks * 2 * sizeof(unsigned long long), st) != cudaSuccess)
    return CSA2_ERR_CUDA;
  k_selftest_encode_sweep<<<dim3(64, nchunks), 256, 0, st>>>(chunk0, d);
  if (cudaGetLastError() != cudaSuccess) return CSA2_ERR_CUDA;
  if (cudaMemcpyAsync(sums, d, (size_t)nchunks * 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return CSA2_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return CSA2_ERR_CUDA;
  return CSA2_OK;
}
