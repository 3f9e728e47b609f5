// Sparse MQA decode attention over the selected FP4 entries joined with the
// layer's FP8 sliding window, one softmax over both ("DeepSeek-V4: Towards
// Highly Efficient Million-Token Context Intelligence", CSA step 3 and the
// sliding-window branch; "DeepSeek-V4.1-Flash: pushing the limits of KV cache
// compression", 4.1).  K = V = the 512-channel latent; 64 heads share it.
//
// Each CTA takes a chunk of 64 rows of one query: it dequantizes them into
// shared memory (exact), computes the 64x64 logits, a chunk-local softmax
// (max m, sum l) and the unnormalised P X; a merge kernel combines the chunks
// with their log-sum-exp.
#include "common.cuh"

namespace csa2 {

namespace {

constexpr int kRows = 64;
constexpr int kAT = 256;
constexpr int kXPad = kDMain + 4;   // fp32 row pitch of X in shared memory
constexpr int kQPad = kDMain + 8;   // bf16 row pitch of q
constexpr int kPPad = kRows + 1;

struct AttnSmem {
  float X[kRows][kXPad];
  __nv_bfloat16 q[kHAtt][kQPad];
  float p[kHAtt][kPPad];
  int valid[kRows];
};

__global__ void __launch_bounds__(kAT) k_attn_chunk(
    const uint8_t* __restrict__ kv_codes, const uint8_t* __restrict__ kv_scales, int64_t seq_stride,
    const int32_t* __restrict__ topk, int k, const uint8_t* __restrict__ swa, int n_swa,
    const uint16_t* __restrict__ qg, float scale, int nchunks, float* __restrict__ part_o,
    float2* __restrict__ part_ml, void* ws) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AttnSmem& S = *reinterpret_cast<AttnSmem*>(smem_raw);
  const int b = blockIdx.y, chunk = blockIdx.x;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  // 1. rows -> fp32 in shared memory (each lane: one 16-channel group)
  for (int r = warp; r < kRows; r += kAT / 32) {
    const int gr = chunk * kRows + r;
    float* xr = S.X[r];
    bool ok = false;
    if (gr < k) {
      const int64_t idx = topk[(int64_t)b * k + gr];
      if (idx >= 0 && idx < seq_stride) {
        ok = true;
        const int64_t e = (int64_t)b * seq_stride + idx;
        const uint2 c = *reinterpret_cast<const uint2*>(kv_codes + e * 256 + lane * 8);
        const float s = e4m3_to_float(kv_scales[e * 32 + lane]);
        const uint32_t words[2] = {c.x, c.y};
#pragma unroll
        for (int wi = 0; wi < 2; ++wi)
#pragma unroll
          for (int bi = 0; bi < 4; ++bi) {
            float2 v = e2m1x2_to_float2((words[wi] >> (8 * bi)) & 0xFFu);
            xr[lane * 16 + wi * 8 + bi * 2] = v.x * s;
            xr[lane * 16 + wi * 8 + bi * 2 + 1] = v.y * s;
          }
      } else if (idx != -1 && lane == 0) {
        report_error(ws, CSA2_ERR_INDEX_RANGE, idx);
      }
    } else if (gr - k < n_swa) {
      ok = true;
      const uint8_t* srow = swa + ((int64_t)b * n_swa + (gr - k)) * kDMain + lane * 16;
      const uint4 c = *reinterpret_cast<const uint4*>(srow);
      const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        float2 v0 = e4m3x2_to_float2(words[wi] & 0xFFFFu);
        float2 v1 = e4m3x2_to_float2(words[wi] >> 16);
        xr[lane * 16 + wi * 4 + 0] = v0.x;
        xr[lane * 16 + wi * 4 + 1] = v0.y;
        xr[lane * 16 + wi * 4 + 2] = v1.x;
        xr[lane * 16 + wi * 4 + 3] = v1.y;
      }
    }
    if (!ok)
      for (int c = lane; c < kDMain; c += 32) xr[c] = 0.0f;
    if (lane == 0) S.valid[r] = ok ? 1 : 0;
  }
  // 2. q -> shared memory
  const uint4* qsrc = reinterpret_cast<const uint4*>(qg + (int64_t)b * kHAtt * kDMain);
  for (int i = threadIdx.x; i < kHAtt * kDMain / 8; i += kAT) {
    const int h = i / (kDMain / 8), c8 = i % (kDMain / 8);
    *reinterpret_cast<uint4*>(&S.q[h][c8 * 8]) = qsrc[i];
  }
  __syncthreads();

  // 3. logits: thread -> head h, rows r = j + 4 i (16 rows)
  const int h = threadIdx.x / 4, j = threadIdx.x % 4;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
  for (int c = 0; c < kDMain; c += 4) {
    const __nv_bfloat162 q01 = *reinterpret_cast<const __nv_bfloat162*>(&S.q[h][c]);
    const __nv_bfloat162 q23 = *reinterpret_cast<const __nv_bfloat162*>(&S.q[h][c + 2]);
    const float2 qa = __bfloat1622float2(q01), qb = __bfloat1622float2(q23);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float4 x = *reinterpret_cast<const float4*>(&S.X[j + 4 * i][c]);
      acc[i] = fmaf(qa.x, x.x, fmaf(qa.y, x.y, fmaf(qb.x, x.z, fmaf(qb.y, x.w, acc[i]))));
    }
  }
  float mloc = -INFINITY;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    acc[i] = S.valid[j + 4 * i] ? acc[i] * scale : -INFINITY;
    mloc = fmaxf(mloc, acc[i]);
  }
  mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
  mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
  float lsum = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float p = (mloc == -INFINITY || acc[i] == -INFINITY) ? 0.0f : expf(acc[i] - mloc);
    S.p[h][j + 4 * i] = p;
    lsum += p;
  }
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
  const int64_t pc = ((int64_t)b * nchunks + chunk) * kHAtt;
  if (j == 0) part_ml[pc + h] = make_float2(mloc, lsum);
  __syncthreads();

  // 4. O = P X : thread -> head h, columns 16 t + 4 j .. +3 for t = 0..31
  float4 o[32];
#pragma unroll
  for (int t = 0; t < 32; ++t) o[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r = 0; r < kRows; ++r) {
    const float p = S.p[h][r];
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const float4 x = *reinterpret_cast<const float4*>(&S.X[r][16 * t + 4 * j]);
      o[t].x = fmaf(p, x.x, o[t].x);
      o[t].y = fmaf(p, x.y, o[t].y);
      o[t].z = fmaf(p, x.z, o[t].z);
      o[t].w = fmaf(p, x.w, o[t].w);
    }
  }
  float* dst = part_o + (pc + h) * kDMain;
#pragma unroll
  for (int t = 0; t < 32; ++t) *reinterpret_cast<float4*>(dst + 16 * t + 4 * j) = o[t];
}

__global__ void __launch_bounds__(128) k_attn_merge(const float* __restrict__ part_o,
                                                    const float2* __restrict__ part_ml, int nchunks,
                                                    float* __restrict__ out, float* __restrict__ lse) {
  const int bh = blockIdx.x;  // b * 64 + h
  const int b = bh / kHAtt, h = bh % kHAtt;
  float M = -INFINITY;
  for (int c = 0; c < nchunks; ++c) M = fmaxf(M, part_ml[((int64_t)b * nchunks + c) * kHAtt + h].x);
  float L = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = 0; c < nchunks; ++c) {
    const int64_t pc = ((int64_t)b * nchunks + c) * kHAtt + h;
    const float2 ml = part_ml[pc];
    if (ml.y <= 0.0f) continue;
    const float f = expf(ml.x - M);
    L = fmaf(f, ml.y, L);
    const float4 v = reinterpret_cast<const float4*>(part_o + pc * kDMain)[threadIdx.x];
    acc.x = fmaf(f, v.x, acc.x);
    acc.y = fmaf(f, v.y, acc.y);
    acc.z = fmaf(f, v.z, acc.z);
    acc.w = fmaf(f, v.w, acc.w);
  }
  float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
  if (L > 0.0f) r = make_float4(acc.x / L, acc.y / L, acc.z / L, acc.w / L);
  reinterpret_cast<float4*>(out + (int64_t)bh * kDMain)[threadIdx.x] = r;
  if (lse && threadIdx.x == 0) lse[bh] = L > 0.0f ? M + logf(L) : -INFINITY;
}

struct AttnWs {
  float* part_o;
  float2* part_ml;
  size_t bytes;
};

AttnWs attn_ws_layout(void* ws, int32_t B, int nchunks) {
  AttnWs L;
  size_t off = kWsHeader;
  char* base = (char*)ws;
  L.part_o = (float*)(base ? base + off : nullptr);
  off += align_up((size_t)B * nchunks * kHAtt * kDMain * 4, 256);
  L.part_ml = (float2*)(base ? base + off : nullptr);
  off += align_up((size_t)B * nchunks * kHAtt * 8, 256);
  L.bytes = off;
  return L;
}

}  // namespace

}  // namespace csa2

extern "C" size_t csa2_sparse_attn_workspace_size(int32_t B, int32_t k, int32_t n_swa) {
  if (B <= 0 || k < 0 || n_swa < 0) return 0;
  int nchunks = (int)csa2::cdiv(k + n_swa, csa2::kRows);
  if (nchunks < 1) nchunks = 1;
  return csa2::attn_ws_layout(nullptr, B, nchunks).bytes;
}

extern "C" csa2_status csa2_sparse_attn_decode(const csa2_kv_planes* kv, int32_t B, const int32_t* topk,
                                               int32_t k, const uint8_t* swa_e4m3, int32_t n_swa,
                                               const void* q_bf16, float softmax_scale, float* out,
                                               float* lse_out, void* ws, size_t ws_bytes,
                                               csa2_stream stream) {
  using namespace csa2;
  cudaStream_t st = (cudaStream_t)stream;
  if (!planes_ok(kv) || B <= 0 || k < 0 || k > CSA2_MAX_TOPK || n_swa < 0 || n_swa > CSA2_MAX_SWA)
    return CSA2_ERR_INVALID_ARG;
  if ((k > 0 && !topk) || (n_swa > 0 && !swa_e4m3) || !q_bf16 || !out) return CSA2_ERR_INVALID_ARG;
  if (!aligned(q_bf16, 16) || !aligned(out, 16) || (swa_e4m3 && !aligned(swa_e4m3, 16)))
    return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  int nchunks = (int)cdiv(k + n_swa, kRows);
  if (nchunks < 1) nchunks = 1;
  AttnWs L = attn_ws_layout(ws, B, nchunks);
  if (ws_bytes < L.bytes) return CSA2_ERR_WORKSPACE;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;
  const int smem = (int)sizeof(AttnSmem);
  if (cudaFuncSetAttribute(k_attn_chunk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return CSA2_ERR_CUDA;
  k_attn_chunk<<<dim3(nchunks, B), kAT, smem, st>>>(kv->kv_codes, kv->kv_scales, kv->seq_stride, topk,
                                                    k, swa_e4m3, n_swa, (const uint16_t*)q_bf16,
                                                    softmax_scale, nchunks, L.part_o, L.part_ml, ws);
  k_attn_merge<<<B * kHAtt, 128, 0, st>>>(L.part_o, L.part_ml, nchunks, out, lse_out);
  return launch_status();
}
