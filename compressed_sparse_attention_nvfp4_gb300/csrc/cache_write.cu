// Prefill cache write: C = H W_KV, Z = H W_Z ("DeepSeek-V4.1-Flash course, 02
// Architecture", 2.2 Eq. (1)), per-channel softmax pooling of each group of m
// tokens and the indexer key K^I = Cbar W_IK ("DeepSeek-V4.1-Flash: pushing the
// limits of KV cache compression", 4.1), then the cache codec (section 5).
//
// First version on the CUDA cores: a 64-token x 64-channel fp32 tile GEMM that
// computes C and Z of the same channels, pools them in its epilogue and writes
// Cbar (fp32) to the workspace; a second kernel projects K^I in fp32; the codec
// kernels quantize both into the planes.
#include "codec.cuh"
#include "timing.cuh"

namespace csa2 {

namespace {

constexpr int kTM = 64, kTN = 64, kTK = 32, kCT = 256;

struct GemmSmem {
  float Hs[kTK][kTM + 4];
  float Wc[kTK][kTN + 4];
  float Wz[kTK][kTN + 4];
  float C[kTM][kTN + 1];
  float Z[kTM][kTN + 1];
};

__global__ void __launch_bounds__(kCT) k_cw_gemm_pool(const uint16_t* __restrict__ H, int64_t T,
                                                      int d_model,
                                                      const uint16_t* __restrict__ Wkv,
                                                      const uint16_t* __restrict__ Wz, int m,
                                                      float* __restrict__ cbar) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  GemmSmem& S = *reinterpret_cast<GemmSmem*>(smem_raw);
  const int64_t t0 = (int64_t)blockIdx.x * kTM;
  const int ch0 = blockIdx.y * kTN;
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  float ac[4][4] = {}, az[4][4] = {};
  for (int k0 = 0; k0 < d_model; k0 += kTK) {
    {  // H tile: 64 tokens x 32 -> Hs[kk][token]
      const int r = threadIdx.x / 4, c8 = (threadIdx.x % 4) * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (t0 + r < T) v = *reinterpret_cast<const uint4*>(H + (t0 + r) * d_model + k0 + c8);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        S.Hs[c8 + 2 * i][r] = __uint_as_float(w4[i] << 16);
        S.Hs[c8 + 2 * i + 1][r] = __uint_as_float(w4[i] & 0xFFFF0000u);
      }
    }
    {  // W tiles: 32 x 64 each
      const int kk = threadIdx.x / 8, c8 = (threadIdx.x % 8) * 8;
      const uint4 a = *reinterpret_cast<const uint4*>(Wkv + (int64_t)(k0 + kk) * kDMain + ch0 + c8);
      const uint4 z = *reinterpret_cast<const uint4*>(Wz + (int64_t)(k0 + kk) * kDMain + ch0 + c8);
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wz[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        S.Wc[kk][c8 + 2 * i] = __uint_as_float(wa[i] << 16);
        S.Wc[kk][c8 + 2 * i + 1] = __uint_as_float(wa[i] & 0xFFFF0000u);
        S.Wz[kk][c8 + 2 * i] = __uint_as_float(wz[i] << 16);
        S.Wz[kk][c8 + 2 * i + 1] = __uint_as_float(wz[i] & 0xFFFF0000u);
      }
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kTK; ++kk) {
      const float4 h = *reinterpret_cast<const float4*>(&S.Hs[kk][ty * 4]);
      const float4 wc = *reinterpret_cast<const float4*>(&S.Wc[kk][tx * 4]);
      const float4 wz = *reinterpret_cast<const float4*>(&S.Wz[kk][tx * 4]);
      const float hv[4] = {h.x, h.y, h.z, h.w}, cv[4] = {wc.x, wc.y, wc.z, wc.w},
                  zv[4] = {wz.x, wz.y, wz.z, wz.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ac[i][j] = fmaf(hv[i], cv[j], ac[i][j]);
          az[i][j] = fmaf(hv[i], zv[j], az[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      S.C[ty * 4 + i][tx * 4 + j] = ac[i][j];
      S.Z[ty * 4 + i][tx * 4 + j] = az[i][j];
    }
  __syncthreads();
  // pooling: group g of m tokens, channel c
  const int groups = kTM / m;
  const int64_t n = T / m;
  for (int o = threadIdx.x; o < groups * kTN; o += kCT) {
    const int g = o / kTN, c = o % kTN;
    if (t0 / m + g >= n) continue;
    float v;
    if (m == 1) {
      v = S.C[g][c];  // softmax over one token is exactly 1
    } else {
      float zmax = -INFINITY;
      for (int r = 0; r < m; ++r) zmax = fmaxf(zmax, S.Z[g * m + r][c]);
      float num = 0.0f, den = 0.0f;
      for (int r = 0; r < m; ++r) {
        const float e = expf(S.Z[g * m + r][c] - zmax);
        num = fmaf(e, S.C[g * m + r][c], num);
        den += e;
      }
      v = __fdiv_rn(num, den);
    }
    cbar[(t0 / m + g) * kDMain + ch0 + c] = v;
  }
}

// K^I[n][128] = Cbar[n][512] W_IK[512][128] in fp32; one CTA per 64 entries.
__global__ void __launch_bounds__(256) k_cw_ki(const float* __restrict__ cbar,
                                               const uint16_t* __restrict__ Wik, int64_t n,
                                               float* __restrict__ ki) {
  __shared__ float Ws[32][kDIdx];
  __shared__ float Cs[64][33];
  const int64_t e0 = (int64_t)blockIdx.x * 64;
  const int ty = threadIdx.x / 32, tx = threadIdx.x % 32;  // rows ty*8.., cols tx*4..
  float acc[8][4] = {};
  for (int k0 = 0; k0 < kDMain; k0 += 32) {
    for (int i = threadIdx.x; i < 32 * kDIdx; i += 256)
      Ws[i / kDIdx][i % kDIdx] = bf16_bits_to_float(Wik[(int64_t)(k0 + i / kDIdx) * kDIdx + i % kDIdx]);
    for (int i = threadIdx.x; i < 64 * 32; i += 256) {
      const int64_t e = e0 + i / 32;
      Cs[i / 32][i % 32] = e < n ? cbar[e * kDMain + k0 + i % 32] : 0.0f;
    }
    __syncthreads();
    for (int kk = 0; kk < 32; ++kk) {
      const float4 wv = *reinterpret_cast<const float4*>(&Ws[kk][tx * 4]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float c = Cs[ty * 8 + i][kk];
        acc[i][0] = fmaf(c, wv.x, acc[i][0]);
        acc[i][1] = fmaf(c, wv.y, acc[i][1]);
        acc[i][2] = fmaf(c, wv.z, acc[i][2]);
        acc[i][3] = fmaf(c, wv.w, acc[i][3]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t e = e0 + ty * 8 + i;
    if (e < n)
      *reinterpret_cast<float4*>(ki + e * kDIdx + tx * 4) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
}

struct CwWs {
  float* cbar;
  float* ki;
  size_t bytes;
};

CwWs cw_ws_layout(void* ws, int64_t n) {
  CwWs L;
  char* base = (char*)ws;
  size_t off = kWsHeader;
  L.cbar = (float*)(base ? base + off : nullptr);
  off += align_up((size_t)n * kDMain * 4, 256);
  L.ki = (float*)(base ? base + off : nullptr);
  off += align_up((size_t)n * kDIdx * 4, 256);
  L.bytes = off;
  return L;
}

}  // namespace

}  // namespace csa2

extern "C" size_t csa2_cache_write_workspace_size(int64_t T, int32_t m) {
  if (T < 0 || m < 1) return 0;
  return csa2::cw_ws_layout(nullptr, T / m).bytes;
}

extern "C" csa2_status csa2_cache_write(const void* H_bf16, int64_t T, int32_t d_model,
                                        const void* Wkv_bf16, const void* Wz_bf16, const void* Wik_bf16,
                                        int32_t m, const csa2_kv_planes* dst, int32_t seq,
                                        int64_t entry_offset, void* ws, size_t ws_bytes,
                                        csa2_stream stream) {
  using namespace csa2;
  cudaStream_t st = (cudaStream_t)stream;
  if (!planes_ok(dst) || !H_bf16 || !Wkv_bf16 || !Wz_bf16 || !Wik_bf16 || T < 0 || seq < 0 ||
      entry_offset < 0)
    return CSA2_ERR_INVALID_ARG;
  if (m < 1 || m > 64 || 64 % m != 0 || T % m != 0) return CSA2_ERR_UNSUPPORTED;
  if (d_model < kTK || d_model % 64 != 0) return CSA2_ERR_UNSUPPORTED;
  if (!aligned(H_bf16, 16) || !aligned(Wkv_bf16, 16) || !aligned(Wz_bf16, 16) || !aligned(Wik_bf16, 16))
    return CSA2_ERR_INVALID_ARG;
  const int64_t n = T / m;
  if (entry_offset + n > dst->seq_stride) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  CwWs L = cw_ws_layout(ws, n);
  if (ws_bytes < L.bytes) return CSA2_ERR_WORKSPACE;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;
  if (T == 0) return CSA2_OK;
  const int smem = (int)sizeof(GemmSmem);
  if (cudaFuncSetAttribute(k_cw_gemm_pool, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return CSA2_ERR_CUDA;
  {
    KernelTimer timer("k_cw_gemm_pool", st);
    k_cw_gemm_pool<<<dim3((unsigned)cdiv(T, kTM), kDMain / kTN), kCT, smem, st>>>(
        (const uint16_t*)H_bf16, T, d_model, (const uint16_t*)Wkv_bf16, (const uint16_t*)Wz_bf16, m, L.cbar);
  }
  {
    KernelTimer timer("k_cw_ki", st);
    k_cw_ki<<<(unsigned)cdiv(n, 64), 256, 0, st>>>(L.cbar, (const uint16_t*)Wik_bf16, n, L.ki);
  }
  launch_quantize(L.cbar, L.ki, n, dst, (int64_t)seq * dst->seq_stride + entry_offset, st);
  return launch_status();
}
