// Sparse MQA decode attention over the selected FP4 entries joined with the
// layer's FP8 sliding window, one softmax over both ("DeepSeek-V4: Towards
// Highly Efficient Million-Token Context Intelligence", CSA step 3 and the
// sliding-window branch; "DeepSeek-V4.1-Flash: pushing the limits of KV cache
// compression", 4.1).  K = V = the 512-channel latent; 64 heads share it.
//
// k_attn_qprep stages q once per query: q' = q 2^-s_h in f16 with a
// power-of-two prescale per head (exact for bf16 q), already in the byte image
// of the S MMA's B operand.  Then each CTA of k_attn takes a chunk of 128 rows
// of one query and runs it on the tensor cores (tcgen05, kind::f16, fp32
// accumulation in tensor memory):
//   1. copies q' in with one bulk copy while its threads gather and dequantize
//      the rows into shared memory as f16 (exact: E2M1 x E4M3 has at most 6
//      significant bits), interleaved X[c/8][row][c%8]: K-major for S,
//      M-major for O;
//   2. S^T[128 rows x 64 heads] = X q'^T (one thread issues 32 MMAs);
//   3. per head, the maximum logit: over the chunk, then over the query;
//   4. P = exp(S - max) rounded to f16, with its column sums l;
//   5. O^T[512 x 64] = X^T P^T (four 128-channel M tiles).
// When a query's chunks fit one thread-block cluster (at most 8 chunks, 1024
// rows) the cluster exchanges the chunk maxima before step 4, so that every
// chunk's probabilities share one reference, and sums the chunks' O and l
// through distributed shared memory into the normalised output.  Longer
// selections write each chunk's unnormalised O with its (max, l) and a merge
// kernel combines the chunks by log-sum-exp.
#include <cooperative_groups.h>

#include "codec.cuh"
#include "ptx.cuh"
#include "timing.cuh"

namespace cg = cooperative_groups;

namespace csa2 {

namespace {

constexpr int kRows = 128;  // rows per CTA: the M of the S MMA
constexpr int kAT = 288;    // warps 0-7: two threads per row in the gather, the epilogues; warp 8: control
constexpr int kCtlWarp = 8;
constexpr int kMaxCluster = 8;
constexpr uint32_t kAttnTmemCols = 256;
constexpr long long kAttnWaitBudget = 1LL << 32;
constexpr uint32_t kQBytes = kDMain * kHAtt * 2;  // staged q' image per query

struct __align__(1024) AttnSmem {
  // f16 rows [c/8][row][c%8]; once the O MMA has completed, this CTA's O^T as
  // fp32 [head][channel] for the cluster's reduction
  uint16_t X[kDMain / 8][kRows * 8];
  uint16_t q[kDMain / 8][kHAtt * 8];  // f16 q' [c/8][head][c%8]
  uint16_t P[kHAtt / 8][kRows * 8];   // f16 probabilities [h/8][row][h%8]
  float colscale[kHAtt];              // softmax_scale * 2^s_h
  float red[4][kHAtt];                // per lane quarter partial column reductions
  float mloc[kHAtt];                  // chunk maximum (read by the cluster)
  float M[kHAtt];                     // reference maximum of this chunk's probabilities
  float lloc[kHAtt];                  // chunk sum of the rounded probabilities (read by the cluster)
  float invL[kHAtt];
  int valid[kRows];
  uint64_t qbar, bar;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(float) * kHAtt * kDMain == sizeof(uint16_t) * kDMain * kRows, "O^T fits the rows");

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

struct MaxOp {
  __device__ __forceinline__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct AddOp {
  __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};

// Reduce-scatter over a warp: every lane holds 32 values; afterwards lane l
// holds op over the 32 lanes of value l (31 shuffles; v is consumed).  The
// pairing is fixed, so sums are reproducible.
template <class Op>
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32], int lane, Op op) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;
#pragma unroll
    for (int j = 0; j < s; ++j) {
      const float keep = up ? v[j + s] : v[j];
      const float send = up ? v[j] : v[j + s];
      v[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, s));
    }
  }
  return v[0];
}

// q' = q_h 2^-s_h in f16 with 2^s_h bringing the head's largest |q| to
// [2^14, 2^15), clamped so that both 2^s_h and 2^-s_h are normal fp32 values;
// bf16 q keeps q' exact and inside the f16 range.  One warp per head: lane l
// converts channels 8l..8l+7 and 256+8l..256+8l+7, i.e. 16-byte chunks l and
// 32+l of the [c/8][head][c%8] image.
__global__ void __launch_bounds__(256) k_attn_qprep(const uint16_t* __restrict__ qg, float scale,
                                                    uint16_t* __restrict__ qs, float* __restrict__ colscale) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.y;
  const int h = blockIdx.x * 8 + threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint4* src = reinterpret_cast<const uint4*>(qg + ((int64_t)b * kHAtt + h) * kDMain);
  const uint4 raw[2] = {src[lane], src[32 + lane]};
  float mx = 0.0f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w4[j] << 16)), fabsf(__uint_as_float(w4[j] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const int sig = mx > 0.0f ? min(max(floor_log2_f32(mx) - 14, -126), 126) : 0;
  const float inv = exp2i_f32(-sig);  // exact power of two: q 2^-sig rounds only in the f16 conversion
  uint16_t* dst = qs + (int64_t)b * (kQBytes / 2);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h2 = __floats2half2_rn(__uint_as_float(w4[j] << 16) * inv,
                                           __uint_as_float(w4[j] & 0xFFFF0000u) * inv);
      o[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    const int cc = i * 32 + lane;
    *reinterpret_cast<uint4*>(dst + ((int64_t)cc * kHAtt + h) * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0) colscale[b * kHAtt + h] = scale * exp2i_f32(sig);
}

// Gathers and dequantizes half a row: channels [256 half, 256 half + 256).
__device__ __forceinline__ bool gather_half_row(AttnSmem& S, const uint8_t* __restrict__ kv_codes,
                                                const uint8_t* __restrict__ kv_scales, int64_t seq_stride,
                                                const int32_t* __restrict__ topk, int k,
                                                const uint8_t* __restrict__ swa, int n_swa, int b, int gr,
                                                int r, int half, void* ws) {
  if (gr < k) {
    const int64_t idx = topk[(int64_t)b * k + gr];
    if (idx >= 0 && idx < seq_stride) {
      const int64_t e = (int64_t)b * seq_stride + idx;
      const uint4* cs = reinterpret_cast<const uint4*>(kv_codes + e * 256 + half * 128);
      uint4 c8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) c8[i] = cs[i];
      const uint4 s4 = reinterpret_cast<const uint4*>(kv_scales + e * 32)[half];
      const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int g = 0; g < 16; ++g) {  // 16 channels: 8 code bytes, one E4M3 scale
        const uint32_t sb = (sw[g / 4] >> (8 * (g % 4))) & 0xFFu;
        const uint32_t s2 = e4m3x2_to_f16x2(sb | (sb << 8));
        const uint4 cw = c8[g / 2];
        const uint32_t w0 = (g & 1) ? cw.z : cw.x, w1 = (g & 1) ? cw.w : cw.y;
        uint32_t h0[4], h1[4];
        e2m1x8_to_f16(w0, h0);
        e2m1x8_to_f16(w1, h1);
        const int cc = half * 32 + 2 * g;
        *reinterpret_cast<uint4*>(&S.X[cc][r * 8]) =
            make_uint4(hmul2_u32(h0[0], s2), hmul2_u32(h0[1], s2), hmul2_u32(h0[2], s2), hmul2_u32(h0[3], s2));
        *reinterpret_cast<uint4*>(&S.X[cc + 1][r * 8]) =
            make_uint4(hmul2_u32(h1[0], s2), hmul2_u32(h1[1], s2), hmul2_u32(h1[2], s2), hmul2_u32(h1[3], s2));
      }
      return true;
    }
    if (idx != -1 && half == 0) report_error(ws, CSA2_ERR_INDEX_RANGE, idx);
    return false;
  }
  if (gr - k < n_swa) {
    const uint4* src = reinterpret_cast<const uint4*>(swa + ((int64_t)b * n_swa + (gr - k)) * kDMain + half * 256);
    uint4 row[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) row[i] = src[i];
#pragma unroll
    for (int i = 0; i < 16; ++i) {  // 16 channels per uint4 -> two chunks
      const uint4 v = row[i];
      const int cc = half * 32 + 2 * i;
      *reinterpret_cast<uint4*>(&S.X[cc][r * 8]) = make_uint4(
          e4m3x2_to_f16x2(v.x), e4m3x2_to_f16x2(v.x >> 16), e4m3x2_to_f16x2(v.y), e4m3x2_to_f16x2(v.y >> 16));
      *reinterpret_cast<uint4*>(&S.X[cc + 1][r * 8]) = make_uint4(
          e4m3x2_to_f16x2(v.z), e4m3x2_to_f16x2(v.z >> 16), e4m3x2_to_f16x2(v.w), e4m3x2_to_f16x2(v.w >> 16));
    }
    return true;
  }
  return false;
}

// kMerge: the grid's x dimension (the query's chunks) is one cluster and the
// kernel writes the normalised output; otherwise it writes per-chunk partials.
// Warps 0-7 gather the rows and run the epilogues (warp w reads tensor-memory
// lane quarter w % 4); warp 8 owns the barriers, the tensor memory, the q'
// copy and the MMA issue.
template <bool kMerge>
__global__ void __launch_bounds__(kAT, 1) k_attn(
    const uint8_t* __restrict__ kv_codes, const uint8_t* __restrict__ kv_scales, int64_t seq_stride,
    const int32_t* __restrict__ topk, int k, const uint8_t* __restrict__ swa, int n_swa,
    const uint16_t* __restrict__ qs, const float* __restrict__ qscale, int nchunks,
    float* __restrict__ out, float* __restrict__ lse, float* __restrict__ part_o,
    float2* __restrict__ part_ml, void* ws) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  AttnSmem& S = *reinterpret_cast<AttnSmem*>(smem_raw);
  volatile int* abort_flag = &S.abort_flag;
  const int b = blockIdx.y, chunk = blockIdx.x;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const bool ctl = warp == kCtlWarp;

  if (ctl) {
    if (lane == 0) {
      ptx::mbar_init(&S.qbar, 1);
      ptx::mbar_init(&S.bar, 1);
      S.abort_flag = 0;
      ptx::fence_mbar_init();
      // q' is written by the preceding staging kernel, which lets this grid
      // start early: wait for it here, then copy q' and its column scales in
      // while the other warps gather
      asm volatile("griddepcontrol.wait;" ::: "memory");
      ptx::mbar_arrive_expect_tx(&S.qbar, kQBytes + kHAtt * 4);
      ptx::bulk_g2s(&S.q[0][0], qs + (int64_t)b * (kQBytes / 2), kQBytes, &S.qbar);
      ptx::bulk_g2s(S.colscale, qscale + (int64_t)b * kHAtt, kHAtt * 4, &S.qbar);
    }
    __syncwarp();
    ptx::tmem_alloc(&S.tmem_base, kAttnTmemCols);
  } else {
    // ---- rows -> f16 X (threads r and r + 128 own the two halves of row r)
    const int r = tid % kRows, half = tid / kRows;
    const bool ok = gather_half_row(S, kv_codes, kv_scales, seq_stride, topk, k, swa, n_swa, b,
                                    chunk * kRows + r, r, half, ws);
    if (!ok)
#pragma unroll 8
      for (int cc = half * 32; cc < half * 32 + 32; ++cc)
        *reinterpret_cast<uint4*>(&S.X[cc][r * 8]) = make_uint4(0, 0, 0, 0);
    if (half == 0) S.valid[r] = ok ? 1 : 0;
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  // ---- S^T = X q'^T : M = 128 rows, N = 64 heads, K = 512
  if (ctl && lane == 0) {
    if (ptx::mbar_wait(&S.qbar, 0, abort_flag, kAttnWaitBudget)) {
      constexpr uint32_t idesc = ptx::idesc_f16(128, 64, 0);
#pragma unroll 4
      for (int ks = 0; ks < kDMain / 16; ++ks) {
        const uint64_t ad = ptx::smem_desc_noswizzle(&S.X[2 * ks][0], kRows * 16, 128);
        const uint64_t bd = ptx::smem_desc_noswizzle(&S.q[2 * ks][0], kHAtt * 16, 128);
        ptx::mma_f16_ss(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
      }
      ptx::mma_commit(&S.bar);
    } else {
      *abort_flag = 1;
      report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 20);
    }
  }
  bool ok = true;
  const int q4 = warp & 3, hh = (warp >> 2) & 1;
  const int r = q4 * 32 + lane;
  const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16);
  float sv[32];
  if (!ctl) {
    ok = ptx::mbar_wait_warp(&S.bar, 0, abort_flag, kAttnWaitBudget);
    if (!ok && lane == 0 && !*abort_flag) {
      *abort_flag = 1;
      report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 21);
    }
    ok = ok && ptx::mbar_wait_warp(&S.qbar, 0, abort_flag, kAttnWaitBudget);  // colscale landed (acquire)
    ptx::tc_fence_after();
    uint32_t a[32];
    ptx::tmem_ld_32x32b_x32(taddr + (uint32_t)hh * 32u, a);
    ptx::tmem_wait_ld();
    const bool v = ok && S.valid[r] != 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) sv[j] = v ? __uint_as_float(a[j]) * S.colscale[hh * 32 + j] : -INFINITY;
    float t[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) t[j] = sv[j];
    S.red[q4][hh * 32 + lane] = warp_reduce_scatter32(t, lane, MaxOp());
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (tid < kHAtt) {
    const float m = fmaxf(fmaxf(S.red[0][tid], S.red[1][tid]), fmaxf(S.red[2][tid], S.red[3][tid]));
    S.mloc[tid] = m;
    if (!kMerge) S.M[tid] = m;
  }
  if constexpr (kMerge) {
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // chunk maxima visible to the cluster
    if (tid < kHAtt) {
      float m = -INFINITY;
      for (int rr = 0; rr < nchunks; ++rr) m = fmaxf(m, cluster.map_shared_rank(S.mloc, rr)[tid]);
      S.M[tid] = m;
    }
  }
  __syncthreads();

  // ---- P = exp(S - M) rounded to f16 once; l = column sums of the rounded values
  if (!ctl) {
    float pr[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float mh = S.M[hh * 32 + j];
      const float p = (sv[j] == -INFINITY || mh == -INFINITY) ? 0.0f : __expf(sv[j] - mh);
      pr[j] = __half2float(__float2half_rn(p));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 h2 = __floats2half2_rn(pr[8 * i + 2 * j], pr[8 * i + 2 * j + 1]);
        o[j] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(&S.P[hh * 4 + i][r * 8]) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    S.red[q4][hh * 32 + lane] = warp_reduce_scatter32(pr, lane, AddOp());
    ptx::fence_proxy_async_smem();
  }
  __syncthreads();
  ptx::tc_fence_after();
  if (tid < kHAtt) S.lloc[tid] = ((S.red[0][tid] + S.red[1][tid]) + S.red[2][tid]) + S.red[3][tid];

  // ---- O^T = X^T P^T : four M tiles of 128 channels, N = 64 heads, K = 128 rows
  if (ctl && lane == 0 && !*abort_flag) {
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
  const int64_t pc = ((int64_t)b * nchunks + chunk) * kHAtt;
  float* obuf = reinterpret_cast<float*>(&S.X[0][0]);  // O^T as [head][channel]
  if (!ctl) {
    ok = ok && ptx::mbar_wait_warp(&S.bar, 1, abort_flag, kAttnWaitBudget);
    if (!ok && lane == 0 && !*abort_flag) {
      *abort_flag = 1;
      report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 22);
    }
    ptx::tc_fence_after();
    ptx::fence_proxy_async_smem();  // the MMAs' reads of X precede the writes below
#pragma unroll 1
    for (int mt = 0; mt < 4; mt += 2) {
      uint32_t a0[32], a1[32];
      ptx::tmem_ld_32x32b_x32(taddr + (uint32_t)mt * 64u + (uint32_t)hh * 32u, a0);
      ptx::tmem_ld_32x32b_x32(taddr + (uint32_t)(mt + 1) * 64u + (uint32_t)hh * 32u, a1);
      ptx::tmem_wait_ld();
      const int c0 = mt * kRows + r, c1 = c0 + kRows;  // channels
      if constexpr (kMerge) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          obuf[(hh * 32 + j) * kDMain + c0] = ok ? __uint_as_float(a0[j]) : 0.0f;
          obuf[(hh * 32 + j) * kDMain + c1] = ok ? __uint_as_float(a1[j]) : 0.0f;
        }
      } else if (ok) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          part_o[(pc + hh * 32 + j) * kDMain + c0] = __uint_as_float(a0[j]);
          part_o[(pc + hh * 32 + j) * kDMain + c1] = __uint_as_float(a1[j]);
        }
      }
    }
  }

  if constexpr (kMerge) {
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    cluster.sync();  // every chunk's O^T and l visible to the cluster
    if (tid < kHAtt) {
      float L = 0.0f;
      for (int rr = 0; rr < nchunks; ++rr) L += cluster.map_shared_rank(S.lloc, rr)[tid];
      S.invL[tid] = L > 0.0f ? 1.0f / L : 0.0f;
      if (lse && rank == 0) lse[b * kHAtt + tid] = L > 0.0f ? S.M[tid] + logf(L) : -INFINITY;
    }
    __syncthreads();
    // this CTA's share of the output: float4 slots [lo, hi) of the [64][512]
    // result, summed over the chunks in rank order with every load of a batch
    // in flight at once
    uint32_t peer[kMaxCluster];  // shared::cluster addresses of the chunks' O^T
#pragma unroll
    for (int rr = 0; rr < kMaxCluster; ++rr) peer[rr] = ptx::mapa_cluster(ptx::smem_u32(obuf), rr < nchunks ? rr : 0);
    constexpr int kF4 = kHAtt * kDMain / 4;
    constexpr int kU = 3;
    const int per = (kF4 + nchunks - 1) / nchunks;
    const int lo = rank * per, hi = min(kF4, lo + per);
    float4* ob = reinterpret_cast<float4*>(out + (int64_t)b * kHAtt * kDMain);
    for (int f0 = lo + tid; f0 < hi; f0 += kU * kAT) {
      float4 v[kMaxCluster][kU];
#pragma unroll
      for (int rr = 0; rr < kMaxCluster; ++rr)
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (rr < nchunks && f0 + u * kAT < hi) v[rr][u] = ptx::ld_cluster_f4(peer[rr] + (uint32_t)(f0 + u * kAT) * 16u);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int f = f0 + u * kAT;
        if (f < hi) {
          float4 acc = v[0][u];
#pragma unroll
          for (int rr = 1; rr < kMaxCluster; ++rr)
            if (rr < nchunks) {
              acc.x += v[rr][u].x;
              acc.y += v[rr][u].y;
              acc.z += v[rr][u].z;
              acc.w += v[rr][u].w;
            }
          const float il = S.invL[f / (kDMain / 4)];
          ob[f] = make_float4(acc.x * il, acc.y * il, acc.z * il, acc.w * il);
        }
      }
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
  } else {
    if (tid < kHAtt) part_ml[pc + tid] = ok ? make_float2(S.M[tid], S.lloc[tid]) : make_float2(-INFINITY, 0.0f);
  }
  if (ctl && lane == 0 && *abort_flag) {  // after a timeout: let the q' copy land before the CTA's memory is freed
    volatile int keep_waiting = 0;
    ptx::mbar_wait(&S.qbar, 0, &keep_waiting, kAttnWaitBudget);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (ctl) {
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
  uint16_t* qs;     // [B] staged q' images
  float* qscale;    // [B][64]
  float* part_o;    // [B][nchunks][64][512] (partials path only)
  float2* part_ml;  // [B][nchunks][64]
  size_t bytes;
};

AttnWs attn_ws_layout(void* ws, int32_t B, int nchunks) {
  AttnWs L{};
  size_t off = kWsHeader;
  char* base = (char*)ws;
  L.qs = (uint16_t*)(base ? base + off : nullptr);
  off += align_up((size_t)B * kQBytes, 256);
  L.qscale = (float*)(base ? base + off : nullptr);
  off += align_up((size_t)B * kHAtt * 4, 256);
  if (nchunks > kMaxCluster) {
    L.part_o = (float*)(base ? base + off : nullptr);
    off += align_up((size_t)B * nchunks * kHAtt * kDMain * 4, 256);
    L.part_ml = (float2*)(base ? base + off : nullptr);
    off += align_up((size_t)B * nchunks * kHAtt * 8, 256);
  }
  L.bytes = off;
  return L;
}

int attn_chunks(int32_t k, int32_t n_swa) {
  const int n = (int)cdiv(k + n_swa, kRows);
  return n < 1 ? 1 : n;
}

}  // namespace

}  // namespace csa2

extern "C" size_t csa2_sparse_attn_workspace_size(int32_t B, int32_t k, int32_t n_swa) {
  if (B <= 0 || k < 0 || n_swa < 0) return 0;
  return csa2::attn_ws_layout(nullptr, B, csa2::attn_chunks(k, n_swa)).bytes;
}

extern "C" csa2_status csa2_sparse_attn_decode(const csa2_kv_planes* kv, int32_t B, const int32_t* topk,
                                               int32_t k, const uint8_t* swa_e4m3, int32_t n_swa,
                                               const void* q_bf16, float softmax_scale, float* out,
                                               float* lse_out, void* ws, size_t ws_bytes,
                                               csa2_stream stream) {
  using namespace csa2;
  cudaStream_t st = (cudaStream_t)stream;
  if (!planes_ok(kv) || B <= 0 || B > 65535 || k < 0 || k > CSA2_MAX_TOPK || n_swa < 0 || n_swa > CSA2_MAX_SWA)
    return CSA2_ERR_INVALID_ARG;
  if ((k > 0 && !topk) || (n_swa > 0 && !swa_e4m3) || !q_bf16 || !out) return CSA2_ERR_INVALID_ARG;
  if (!aligned(q_bf16, 16) || !aligned(out, 16) || (swa_e4m3 && !aligned(swa_e4m3, 16)))
    return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  const int nchunks = attn_chunks(k, n_swa);
  AttnWs L = attn_ws_layout(ws, B, nchunks);
  if (ws_bytes < L.bytes) return CSA2_ERR_WORKSPACE;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;
  {
    KernelTimer timer("k_attn_qprep", st);
    k_attn_qprep<<<dim3(kHAtt / 8, B), 256, 0, st>>>((const uint16_t*)q_bf16, softmax_scale, L.qs, L.qscale);
  }
  const int smem = (int)sizeof(AttnSmem);
  if (nchunks <= kMaxCluster) {
    if (cudaFuncSetAttribute(k_attn<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return CSA2_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nchunks, B);
    cfg.blockDim = dim3(kAT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nchunks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap the q' staging kernel
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    KernelTimer timer("k_attn", st);
    if (cudaLaunchKernelEx(&cfg, k_attn<true>, kv->kv_codes, kv->kv_scales, kv->seq_stride, topk, k, swa_e4m3,
                           n_swa, (const uint16_t*)L.qs, (const float*)L.qscale, nchunks, out, lse_out,
                           (float*)nullptr, (float2*)nullptr, ws) != cudaSuccess)
      return CSA2_ERR_CUDA;
  } else {
    if (cudaFuncSetAttribute(k_attn<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return CSA2_ERR_CUDA;
    {
      KernelTimer timer("k_attn_part", st);
      k_attn<false><<<dim3(nchunks, B), kAT, smem, st>>>(kv->kv_codes, kv->kv_scales, kv->seq_stride, topk, k,
                                                          swa_e4m3, n_swa, L.qs, L.qscale, nchunks, out,
                                                          lse_out, L.part_o, L.part_ml, ws);
    }
    KernelTimer timer("k_attn_merge", st);
    k_attn_merge<<<B * kHAtt, 128, 0, st>>>(L.part_o, L.part_ml, nchunks, out, lse_out);
  }
  return launch_status();
}
