// Sparse MQA decode attention over the selected FP4 entries joined with the
// layer's FP8 sliding window, one softmax over both ("DeepSeek-V4: Towards
// Highly Efficient Million-Token Context Intelligence", CSA step 3 and the
// sliding-window branch; "DeepSeek-V4.1-Flash: pushing the limits of KV cache
// compression", 4.1).  K = V = the 512-channel latent; 64 heads share it.
//
// Each CTA takes a chunk of 128 rows of one query and runs it on the tensor
// cores (tcgen05, kind::f16, fp32 accumulation in tensor memory):
//   1. gathers and dequantizes its rows into shared memory as f16 (exact:
//      E2M1 x E4M3 has at most 6 significant bits), in an interleaved layout
//      X[c/8][row][c%8] that is K-major for S and M-major for O;
//   2. stages q with a power-of-two prescale per head (exact for bf16 q);
//   3. S^T[128 rows x 64 heads] = X q'^T (one thread issues 32 MMAs);
//   4. chunk-local softmax per head over its rows (max m, sum l), P in f16;
//   5. O^T[512 x 64] = X^T P^T (four 128-channel M tiles), written unnormalised
//      with (m, l) per head; a merge kernel combines the chunks by log-sum-exp.
#include "codec.cuh"
#include "ptx.cuh"
#include "timing.cuh"

namespace csa2 {

namespace {

constexpr int kRows = 128;
constexpr int kAT = 128;
constexpr uint32_t kAttnTmemCols = 256;
constexpr long long kAttnWaitBudget = 1LL << 32;

struct __align__(1024) AttnSmem {
  uint16_t X[kDMain / 8][kRows * 8];  // f16, channel-chunk major: [c/8][row][c%8]
  union {
    uint16_t q[kDMain / 8][kHAtt * 8];  // f16 q': [c/8][head][c%8]
    float S[kRows][kHAtt + 1];          // logits, then probabilities (column reductions)
  } u;
  uint16_t P[kHAtt / 8][kRows * 8];     // f16 probabilities: [h/8][row][h%8]
  float colscale[kHAtt];                // softmax_scale * 2^s_h
  float red[2][kHAtt];
  float m[kHAtt], l[kHAtt];
  int valid[kRows];
  uint64_t bar;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void e2m1x8_to_f16(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\tmov.b32 {t0, t1, t2, t3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t0;\n\tcvt.rn.f16x2.e2m1x2 %1, t1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, t2;\n\tcvt.rn.f16x2.e2m1x2 %3, t3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h;
  uint16_t v = (uint16_t)two;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
  return h;
}

__global__ void __launch_bounds__(kAT, 1) k_attn_tc(
    const uint8_t* __restrict__ kv_codes, const uint8_t* __restrict__ kv_scales, int64_t seq_stride,
    const int32_t* __restrict__ topk, int k, const uint8_t* __restrict__ swa, int n_swa,
    const uint16_t* __restrict__ qg, float scale, int nchunks, float* __restrict__ part_o,
    float2* __restrict__ part_ml, void* ws) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  AttnSmem& S = *reinterpret_cast<AttnSmem*>(smem_raw);
  volatile int* abort_flag = &S.abort_flag;
  const int b = blockIdx.y, chunk = blockIdx.x;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  if (tid == 0) {
    ptx::mbar_init(&S.bar, 1);
    S.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) ptx::tmem_alloc(&S.tmem_base, kAttnTmemCols);

  // ---- q' = q 2^-s_h in f16 (two threads per head, 256 channels each)
  {
    const int h = tid / 2, half = tid % 2;
    const uint4* src = reinterpret_cast<const uint4*>(qg + ((int64_t)b * kHAtt + h) * kDMain + half * 256);
    uint4 raw[32];  // all of this thread's 256 channels in flight at once
#pragma unroll
    for (int i = 0; i < 32; ++i) raw[i] = src[i];
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w4[j] << 16)), fabsf(__uint_as_float(w4[j] & 0xFFFF0000u))));
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    // 2^sig brings the head's largest |q| to [2^14, 2^15); clamped so that both
    // 2^sig and 2^-sig are normal fp32 values (bf16 q keeps q' inside f16 range)
    const int sig = mx > 0.0f ? min(max(floor_log2_f32(mx) - 14, -126), 126) : 0;
    const float inv = exp2i_f32(-sig);  // exact power of two: q * 2^-sig rounds only in the f16 conversion
#pragma unroll
    for (int i = 0; i < 32; ++i) {  // 8 channels per uint4 -> one 16-byte chunk of q'
      const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 h2 = __floats2half2_rn(__uint_as_float(w4[j] << 16) * inv,
                                             __uint_as_float(w4[j] & 0xFFFF0000u) * inv);
        o[j] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      const int cc = half * 32 + i;  // channel chunk c/8
      *reinterpret_cast<uint4*>(&S.u.q[cc][h * 8]) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (half == 0) S.colscale[h] = scale * exp2i_f32(sig);
  }

  // ---- rows -> f16 X (thread r owns row r of the chunk)
  {
    const int r = tid;
    const int gr = chunk * kRows + r;
    bool ok = false;
    if (gr < k) {
      const int64_t idx = topk[(int64_t)b * k + gr];
      if (idx >= 0 && idx < seq_stride) {
        ok = true;
        const int64_t e = (int64_t)b * seq_stride + idx;
        const uint4* cs = reinterpret_cast<const uint4*>(kv_codes + e * 256);
        const uint4* ss = reinterpret_cast<const uint4*>(kv_scales + e * 32);
        uint4 c16[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) c16[i] = cs[i];
        const uint4 s0 = ss[0], s1 = ss[1];
        const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int g = 0; g < 32; ++g) {  // 16 channels: 8 code bytes, one E4M3 scale
          const uint32_t sb = (sw[g / 4] >> (8 * (g % 4))) & 0xFFu;
          const uint32_t s2 = e4m3x2_to_f16x2(sb | (sb << 8));
          const uint4 cw = c16[g / 2];
          const uint32_t w0 = (g & 1) ? cw.z : cw.x, w1 = (g & 1) ? cw.w : cw.y;
          uint32_t h0[4], h1[4];
          e2m1x8_to_f16(w0, h0);
          e2m1x8_to_f16(w1, h1);
          *reinterpret_cast<uint4*>(&S.X[2 * g][r * 8]) =
              make_uint4(hmul2_u32(h0[0], s2), hmul2_u32(h0[1], s2), hmul2_u32(h0[2], s2), hmul2_u32(h0[3], s2));
          *reinterpret_cast<uint4*>(&S.X[2 * g + 1][r * 8]) =
              make_uint4(hmul2_u32(h1[0], s2), hmul2_u32(h1[1], s2), hmul2_u32(h1[2], s2), hmul2_u32(h1[3], s2));
        }
      } else if (idx != -1) {
        report_error(ws, CSA2_ERR_INDEX_RANGE, idx);
      }
    } else if (gr - k < n_swa) {
      ok = true;
      const uint4* src = reinterpret_cast<const uint4*>(swa + ((int64_t)b * n_swa + (gr - k)) * kDMain);
      uint4 row[32];  // the whole 512-byte row in flight at once
#pragma unroll
      for (int i = 0; i < 32; ++i) row[i] = src[i];
#pragma unroll
      for (int i = 0; i < 32; ++i) {  // 16 channels per uint4 -> two chunks
        const uint4 v = row[i];
        *reinterpret_cast<uint4*>(&S.X[2 * i][r * 8]) =
            make_uint4(e4m3x2_to_f16x2(v.x), e4m3x2_to_f16x2(v.x >> 16), e4m3x2_to_f16x2(v.y),
                       e4m3x2_to_f16x2(v.y >> 16));
        *reinterpret_cast<uint4*>(&S.X[2 * i + 1][r * 8]) =
            make_uint4(e4m3x2_to_f16x2(v.z), e4m3x2_to_f16x2(v.z >> 16), e4m3x2_to_f16x2(v.w),
                       e4m3x2_to_f16x2(v.w >> 16));
      }
    }
    if (!ok)
#pragma unroll 8
      for (int cc = 0; cc < kDMain / 8; ++cc) *reinterpret_cast<uint4*>(&S.X[cc][r * 8]) = make_uint4(0, 0, 0, 0);
    S.valid[r] = ok ? 1 : 0;
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  // ---- S^T = X q'^T : M = 128 rows, N = 64 heads, K = 512
  if (tid == 0) {
    constexpr uint32_t idesc = ptx::idesc_f16(128, 64, 0);
#pragma unroll 4
    for (int ks = 0; ks < kDMain / 16; ++ks) {
      const uint64_t ad = ptx::smem_desc_noswizzle(&S.X[2 * ks][0], kRows * 16, 128);
      const uint64_t bd = ptx::smem_desc_noswizzle(&S.u.q[2 * ks][0], kHAtt * 16, 128);
      ptx::mma_f16_ss(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
    }
    ptx::mma_commit(&S.bar);
  }
  bool ok = ptx::mbar_wait_warp(&S.bar, 0, abort_flag, kAttnWaitBudget);
  if (!ok && lane == 0) {
    *abort_flag = 1;
    report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 21);
  }
  ptx::tc_fence_after();
  const int r = tid;
  const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
  float sv[kHAtt];
  {
    uint32_t a0[32], a1[32];
    ptx::tmem_ld_32x32b_x32(lane_addr, a0);
    ptx::tmem_ld_32x32b_x32(lane_addr + 32, a1);
    ptx::tmem_wait_ld();
    const bool v = S.valid[r] != 0;
#pragma unroll
    for (int h = 0; h < 32; ++h) {
      sv[h] = v ? __uint_as_float(a0[h]) * S.colscale[h] : -INFINITY;
      sv[32 + h] = v ? __uint_as_float(a1[h]) * S.colscale[32 + h] : -INFINITY;
    }
  }
  ptx::tc_fence_before();
  __syncthreads();  // D1 read by everyone; q' no longer needed (its MMAs completed)
#pragma unroll
  for (int h = 0; h < kHAtt; ++h) S.u.S[r][h] = sv[h];
  __syncthreads();
  {  // column max
    const int h = tid % kHAtt, half = tid / kHAtt;
    float mx = -INFINITY;
    for (int rr = half * 64; rr < half * 64 + 64; ++rr) mx = fmaxf(mx, S.u.S[rr][h]);
    S.red[half][h] = mx;
  }
  __syncthreads();
  if (tid < kHAtt) S.m[tid] = fmaxf(S.red[0][tid], S.red[1][tid]);
  __syncthreads();
#pragma unroll
  for (int hc = 0; hc < kHAtt / 8; ++hc) {  // probabilities, rounded to f16 once
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float pv[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int h = hc * 8 + 2 * j + t;
        const float mh = S.m[h];
        const float p = (sv[h] == -INFINITY || mh == -INFINITY) ? 0.0f : __expf(sv[h] - mh);
        const __half ph = __float2half_rn(p);
        pv[t] = __half2float(ph);
        S.u.S[r][h] = pv[t];
      }
      const __half2 h2 = __floats2half2_rn(pv[0], pv[1]);
      o[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(&S.P[hc][r * 8]) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  __syncthreads();
  {  // column sums of the (rounded) probabilities
    const int h = tid % kHAtt, half = tid / kHAtt;
    float sm = 0.0f;
    for (int rr = half * 64; rr < half * 64 + 64; ++rr) sm += S.u.S[rr][h];
    S.red[half][h] = sm;
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (tid < kHAtt) S.l[tid] = S.red[0][tid] + S.red[1][tid];

  // ---- O^T = X^T P^T : four M tiles of 128 channels, N = 64 heads, K = 128 rows
  if (tid == 0 && !*abort_flag) {
    constexpr uint32_t idesc = ptx::idesc_f16(128, 64, 0) | (1u << 15) | (1u << 16);  // both M/N-major
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int ks = 0; ks < kRows / 16; ++ks) {
        const uint64_t ad = ptx::smem_desc_noswizzle(&S.X[mt * 16][ks * 16 * 8], 128, kRows * 16);
        const uint64_t bd = ptx::smem_desc_noswizzle(&S.P[0][ks * 16 * 8], 128, kRows * 16);
        ptx::mma_f16_ss(tmem + (uint32_t)mt * 64u, ad, bd, idesc, ks > 0 ? 1u : 0u);
      }
    ptx::mma_commit(&S.bar);
  }
  ok = ok && ptx::mbar_wait_warp(&S.bar, 1, abort_flag, kAttnWaitBudget);
  if (!ok && lane == 0) {
    *abort_flag = 1;
    report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 22);
  }
  ptx::tc_fence_after();
  const int64_t pc = ((int64_t)b * nchunks + chunk) * kHAtt;
  if (ok) {
#pragma unroll 1
    for (int mt = 0; mt < 4; ++mt) {
      uint32_t a0[32], a1[32];
      ptx::tmem_ld_32x32b_x32(lane_addr + (uint32_t)mt * 64u, a0);
      ptx::tmem_ld_32x32b_x32(lane_addr + (uint32_t)mt * 64u + 32u, a1);
      ptx::tmem_wait_ld();
      const int c = mt * kRows + r;  // channel
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        part_o[(pc + h) * kDMain + c] = __uint_as_float(a0[h]);
        part_o[(pc + 32 + h) * kDMain + c] = __uint_as_float(a1[h]);
      }
    }
  }
  __syncthreads();
  if (tid < kHAtt) part_ml[pc + tid] = ok ? make_float2(S.m[tid], S.l[tid]) : make_float2(-INFINITY, 0.0f);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kAttnTmemCols);
  }
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
  if (cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return CSA2_ERR_CUDA;
  {
    KernelTimer timer("k_attn_tc", st);
    k_attn_tc<<<dim3(nchunks, B), kAT, smem, st>>>(kv->kv_codes, kv->kv_scales, kv->seq_stride, topk, k,
                                                   swa_e4m3, n_swa, (const uint16_t*)q_bf16, softmax_scale,
                                                   nchunks, L.part_o, L.part_ml, ws);
  }
  {
    KernelTimer timer("k_attn_merge", st);
    k_attn_merge<<<B * kHAtt, 128, 0, st>>>(L.part_o, L.part_ml, nchunks, out, lse_out);
  }
  return launch_status();
}
