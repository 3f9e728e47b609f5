// Sparse MQA decode attention over the selected FP4 entries joined with the
// layer's FP8 sliding window, one softmax over both ("DeepSeek-V4: Towards
// Highly Efficient Million-Token Context Intelligence", CSA step 3 and the
// sliding-window branch; "DeepSeek-V4.1-Flash: pushing the limits of KV cache
// compression", 4.1).  K = V = the 512-channel latent; 64 heads share it.
//
// k_attn stages q in shared memory as q' = q 2^-s_h in f16 with a power-of-two
// prescale per head (exact for bf16 q), then runs the query's rows (selected
// entries, then window rows) in chunks of 128 on the tensor cores (tcgen05,
// kind::f16, fp32 accumulation in tensor memory):
//   1. the chunk's rows are dequantized into shared memory as f16 (exact:
//      E2M1 x E4M3 has at most 6 significant bits), interleaved
//      X[c/8][row][c%8]: K-major for S, M-major for O;
//   2. S^T[128 rows x 64 heads] = X q'^T;
//   3. online softmax per head, P rounded to f16 once, l = sums of the rounded P;
//   4. O^T[512 x 64] += X^T P^T (four 128-channel M tiles).
// One CTA per query keeps O in tensor memory across all its chunks, so no
// partial result leaves the SM.  When the batch is too small to fill the GPU
// a query's chunks are split over a few CTAs, which write (max, l, O) partials
// that a merge kernel combines by log-sum-exp.
#include "codec.cuh"
#include "ptx.cuh"
#include "timing.cuh"

namespace csa2 {

namespace {

constexpr int kRows = 128;  // rows per CTA: the M of the S MMA
constexpr int kAT = 288;    // warps 0-7: two threads per row in the gather, the epilogues; warp 8: control
constexpr int kCtlWarp = 8;
constexpr float kLog2e = 1.4426950408889634f;
// the softmax reference (log2 units) moves only when a chunk exceeds it by
// more than 8 nats, so probabilities stay below e^8 (inside f16)
constexpr float kTau2 = 8.0f * kLog2e;
// q' plane stride: 64 heads x 16 bytes plus 16 bytes of padding, so that the
// 16-byte stores of consecutive channel chunks fall in different banks
constexpr int kQPlane = kHAtt * 8 + 8;  // in f16 elements (1040 bytes)
constexpr uint32_t kAttnTmemCols = 512;  // O^T 256 columns, S^T 64
constexpr long long kAttnWaitBudget = 1LL << 32;

// In-layer extras ("DeepSeek-V4: ...", CSA, other details), each off when null /
// zero: RMSNorm weight of the query heads, RoPE of the query at qpos[b] with the
// output turned back by -qpos[b], per-head sink logits.
struct AttnExtras {
  const float* qnorm_w;
  float eps;
  int rope;
  const int64_t* qpos;
  const float* sink;
  const int64_t* win_pos;  // [B][n_swa] position of each window row (< 0: empty), or null: all visible
  const int64_t* win_lo;   // [B] lowest visible window position
  RopeTheta th;
};

struct __align__(1024) AttnSmem {
  uint16_t X[kDMain / 8][kRows * 8];  // f16 rows [c/8][row][c%8]; planes 0-31 / 32-63 = channel halves
  uint16_t q[kDMain / 8][kQPlane];    // f16 q' [c/8][head][c%8], planes padded
  uint16_t P[kHAtt / 8][kRows * 8];   // f16 probabilities [h/8][row][h%8]
  float c2[kHAtt];                    // log2(e) * softmax_scale * 2^s_h: logit (log2 units) per raw S
  float m2w[8][32];                   // per warp: the reference of its 32 heads (0 while none)
  float red[4][kHAtt];                // per lane quarter column maxima of the chunk
  float red2[4][kHAtt];               // per lane quarter column sums of the chunk's P
  int valid[kRows];
  uint64_t q_full;                    // q' and colscale written (8 warps)
  uint64_t x_full[2];                 // channel half of X written (4 warps each)
  uint64_t s_full;                    // S^T MMAs complete
  uint64_t red_full;                  // chunk maxima posted (8 warps)
  uint64_t p_full;                    // P written, O rescaled, sums posted (8 warps)
  uint64_t x_free[2];                 // O MMAs reading that channel half of X (and P) complete
  uint64_t drained;                   // every MMA issued complete
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
// bf16 q keeps q' exact and inside the f16 range (with RMSNorm or RoPE the
// fp32 result is rounded to f16 once).  Warp w converts heads 8w..8w+7: lane l
// holds channels 8l..8l+7 and 256+8l..256+8l+7 of each, i.e. chunks l and 32+l
// of the [c/8][head][c%8] image; the rotated pairs sit in lanes 24-31.
struct QFetch {
  uint4 raw[8][2];
};
__device__ __forceinline__ void fetch_q(QFetch& f, const uint16_t* __restrict__ qg, int b, int warp, int lane) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint4* src = reinterpret_cast<const uint4*>(qg + ((int64_t)b * kHAtt + warp * 8 + u) * kDMain);
    f.raw[u][0] = src[lane];
    f.raw[u][1] = src[32 + lane];
  }
}
template <bool kEx>
__device__ __forceinline__ void stage_q(AttnSmem& S, const QFetch& f, float scale, int warp, int lane,
                                        const AttnExtras& ex, int b) {
  // per lane: the RMSNorm weights of its 16 channels, the cos / sin of its 4 pairs
  float wq[16], rc[4], rs[4];
  const bool norm = kEx && ex.qnorm_w != nullptr;
  if (norm) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float4* wv = reinterpret_cast<const float4*>(ex.qnorm_w + i * 256 + lane * 8);
      const float4 a = wv[0], c = wv[1];
      wq[8 * i] = a.x, wq[8 * i + 1] = a.y, wq[8 * i + 2] = a.z, wq[8 * i + 3] = a.w;
      wq[8 * i + 4] = c.x, wq[8 * i + 5] = c.y, wq[8 * i + 6] = c.z, wq[8 * i + 7] = c.w;
    }
  }
  const bool rot = kEx && ex.rope && 256 + lane * 8 >= kRopeFirst;
  if (rot) {
    const double pos = (double)ex.qpos[b];
#pragma unroll
    for (int p = 0; p < 4; ++p) rope_cos_sin(ex.th.t[(256 + lane * 8 - kRopeFirst) / 2 + p], pos, rc[p], rs[p]);
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t w4[4] = {f.raw[u][i].x, f.raw[u][i].y, f.raw[u][i].z, f.raw[u][i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * i + 2 * j] = __uint_as_float(w4[j] << 16);
        v[8 * i + 2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
      }
    }
    if (norm) {
      float ss = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) ss = fmaf(v[i], v[i], ss);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float r = 1.0f / sqrtf(ss / (float)kDMain + ex.eps);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = wq[i] * (v[i] * r);
    }
    if (rot) {
#pragma unroll
      for (int p = 0; p < 4; ++p) rope_pair(v[8 + 2 * p], v[9 + 2 * p], rc[p], rs[p]);
    }
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(v[i]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const int sig = mx > 0.0f ? min(max(floor_log2_f32(mx) - 14, -126), 126) : 0;
    const float inv = exp2i_f32(-sig);  // exact power of two: q 2^-sig rounds only in the f16 conversion
    const int h = warp * 8 + u;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 h2 = __floats2half2_rn(v[8 * i + 2 * j] * inv, v[8 * i + 2 * j + 1] * inv);
        o[j] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(&S.q[i * 32 + lane][h * 8]) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (lane == 0) S.c2[h] = kLog2e * scale * exp2i_f32(sig);
  }
}

// One thread's half row of a chunk, fetched ahead of its dequantization.
struct RowFetch {
  uint4 raw[16];  // main entry: 8 x 16 code bytes + 16 scale bytes; window row: 256 bytes
  int kind;       // 0 = no row, 1 = main entry, 2 = window row
};

// entry of chunk row gr (rows gr >= k are window rows or padding): topk[b][gr],
// or, dense, entry gr itself while gr < dense_n[b]
__device__ __forceinline__ int64_t fetch_index(const int32_t* __restrict__ topk, const int32_t* __restrict__ dense_n,
                                               int k, int b, int gr) {
  if (gr >= k) return -1;
  if (dense_n) return gr < __ldg(dense_n + b) ? gr : -1;
  return (int64_t)topk[(int64_t)b * k + gr];
}

// Starts the loads of half a row: a selected entry (gr < k, index idx), a
// window row (k <= gr < k + n_swa) or nothing.
__device__ __forceinline__ void issue_row(RowFetch& f, int64_t idx, const uint8_t* __restrict__ kv_codes,
                                          const uint8_t* __restrict__ kv_scales, int64_t seq_stride,
                                          const uint8_t* __restrict__ swa, int n_swa, int k, int b, int gr,
                                          int half, void* ws, const int64_t* __restrict__ win_pos, int64_t win_lo) {
  f.kind = 0;
  if (gr < k) {
    if (idx >= 0 && idx < seq_stride) {
      const int64_t e = (int64_t)b * seq_stride + idx;
      const uint4* cs = reinterpret_cast<const uint4*>(kv_codes + e * 256 + half * 128);
#pragma unroll
      for (int i = 0; i < 8; ++i) f.raw[i] = cs[i];
      f.raw[8] = reinterpret_cast<const uint4*>(kv_scales + e * 32)[half];
      f.kind = 1;
    } else if (idx != -1 && half == 0) {
      report_error(ws, CSA2_ERR_INDEX_RANGE, idx);
    }
  } else if (gr - k < n_swa && (!win_pos || win_pos[(int64_t)b * n_swa + (gr - k)] >= win_lo)) {
    const uint4* src = reinterpret_cast<const uint4*>(swa + ((int64_t)b * n_swa + (gr - k)) * kDMain + half * 256);
#pragma unroll
    for (int i = 0; i < 16; ++i) f.raw[i] = src[i];
    f.kind = 2;
  }
}

// Writes the half row [256 half, 256 half + 256) of row r to X as f16 (zeros
// when there is no row), 64 channels at a time; returns whether the row exists.
__device__ __forceinline__ bool dequant_half_row(AttnSmem& S, const RowFetch& f, int r, int half) {
#pragma unroll
  for (int blk = 0; blk < 4; ++blk) {
    uint32_t w[32];  // channels 64 blk + 2j, 2j + 1 in w[j]
    if (f.kind == 1) {
      const uint32_t sw = blk == 0 ? f.raw[8].x : blk == 1 ? f.raw[8].y : blk == 2 ? f.raw[8].z : f.raw[8].w;
#pragma unroll
      for (int g = 0; g < 4; ++g) {  // 16 channels: 8 code bytes, one E4M3 scale
        const int G = blk * 4 + g;
        const uint32_t sb = (sw >> (8 * g)) & 0xFFu;
        const uint32_t s2 = e4m3x2_to_f16x2(sb | (sb << 8));
        const uint4 cw = f.raw[G / 2];
        const uint32_t w0 = (G & 1) ? cw.z : cw.x, w1 = (G & 1) ? cw.w : cw.y;
        uint32_t h0[4], h1[4];
        e2m1x8_to_f16(w0, h0);
        e2m1x8_to_f16(w1, h1);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          w[8 * g + j] = hmul2_u32(h0[j], s2);
          w[8 * g + 4 + j] = hmul2_u32(h1[j], s2);
        }
      }
    } else if (f.kind == 2) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {  // 16 channels per uint4
        const uint4 v = f.raw[blk * 4 + u];
        w[8 * u + 0] = e4m3x2_to_f16x2(v.x);
        w[8 * u + 1] = e4m3x2_to_f16x2(v.x >> 16);
        w[8 * u + 2] = e4m3x2_to_f16x2(v.y);
        w[8 * u + 3] = e4m3x2_to_f16x2(v.y >> 16);
        w[8 * u + 4] = e4m3x2_to_f16x2(v.z);
        w[8 * u + 5] = e4m3x2_to_f16x2(v.z >> 16);
        w[8 * u + 6] = e4m3x2_to_f16x2(v.w);
        w[8 * u + 7] = e4m3x2_to_f16x2(v.w >> 16);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) w[j] = 0u;
    }
#pragma unroll
    for (int pl = 0; pl < 8; ++pl)
      *reinterpret_cast<uint4*>(&S.X[half * 32 + blk * 8 + pl][r * 8]) =
          make_uint4(w[4 * pl], w[4 * pl + 1], w[4 * pl + 2], w[4 * pl + 3]);
  }
  return f.kind != 0;
}

// One CTA runs chunks [c0, c1) of query b's rows with an online softmax; the
// output accumulates in tensor memory across the chunks.
//   warps 0-3 / 4-7: dequantize channels 0-255 / 256-511 of each chunk into X,
//     fetching the next chunk's rows while the current one is on the tensor
//     cores; then all eight run the chunk's softmax (warp w reads tensor-memory
//     lane quarter w % 4, heads 32 (w / 4) .. +31);
//   warp 8: barriers, tensor memory, the q' copy and the MMA issue.
// Per chunk the MMA thread issues S over the first channel half as soon as it
// is written, then the second; after the softmax, O over the first channel
// half, whose completion frees that half of X for the next chunk, then the
// second.  The softmax keeps, per head, a reference m (the running maximum,
// raised only when a chunk exceeds it by more than kTau2, which then rescales
// O and l in place), so probabilities stay below e^8.  The softmax runs in
// log2 units: p = 2^(raw S * c2_h - m2_h).
// kPartial: write the unnormalised O with (m, l) for the merge kernel instead
// of the normalised output.
template <bool kPartial, bool kEx>
__global__ void __launch_bounds__(kAT, 1) k_attn(
    const uint8_t* __restrict__ kv_codes, const uint8_t* __restrict__ kv_scales, int64_t seq_stride,
    const int32_t* __restrict__ topk, const int32_t* __restrict__ dense_n, int k, const uint8_t* __restrict__ swa,
    int n_swa,
    const uint16_t* __restrict__ qg, float scale, AttnExtras ex, int nchunks, int cps,
    float* __restrict__ out, float* __restrict__ lse, float* __restrict__ part_o,
    float2* __restrict__ part_ml, void* ws) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  AttnSmem& S = *reinterpret_cast<AttnSmem*>(smem_raw);
  volatile int* abort_flag = &S.abort_flag;
  const int b = blockIdx.y, split = blockIdx.x;
  const int c0 = split * cps, nc = min(nchunks, c0 + cps) - c0;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

  if (warp == kCtlWarp) {
    if (lane == 0) {
      ptx::mbar_init(&S.q_full, 8);
      ptx::mbar_init(&S.x_full[0], 4);
      ptx::mbar_init(&S.x_full[1], 4);
      ptx::mbar_init(&S.s_full, 1);
      ptx::mbar_init(&S.red_full, 8);
      ptx::mbar_init(&S.p_full, 8);
      ptx::mbar_init(&S.x_free[0], 1);
      ptx::mbar_init(&S.x_free[1], 1);
      ptx::mbar_init(&S.drained, 1);
      S.abort_flag = 0;
      ptx::fence_mbar_init();
    }
    __syncwarp();
    ptx::tmem_alloc(&S.tmem_base, kAttnTmemCols);
  }
  ptx::griddep_wait();  // q, the indices and the rows may come from the previous kernel
  // q and the first chunk's indices load together; q is converted while the
  // indices arrive, then the rows are requested
  const int r = tid % kRows, half = (tid / kRows) & 1;
  RowFetch rf;
  const int64_t win_lo = ex.win_pos ? max(ex.win_lo[b], (int64_t)0) : 0;  // window rows below it are not seen
  if (warp < kCtlWarp) {
    const int gr = c0 * kRows + r;
    QFetch qf;
    fetch_q(qf, qg, b, warp, lane);
    const int64_t idx0 = fetch_index(topk, dense_n, k, b, gr);
    stage_q<kEx>(S, qf, scale, warp, lane, ex, b);
    ptx::fence_proxy_async_smem();
    issue_row(rf, idx0, kv_codes, kv_scales, seq_stride, swa, n_swa, k, b, gr, half, ws, ex.win_pos, win_lo);
  }
  ptx::tc_fence_before();
  __syncthreads();  // barriers initialised, tensor memory allocated
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const uint32_t tS = tmem + 256u;  // S^T: 64 columns after the 256 of O^T

  if (warp == kCtlWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issue
      bool good = ptx::mbar_wait(&S.q_full, 0, abort_flag, kAttnWaitBudget);
      constexpr uint32_t idesc_s = ptx::idesc_f16(128, 64, 0);
      constexpr uint32_t idesc_o = ptx::idesc_f16(128, 64, 0) | (1u << 15) | (1u << 16);  // M/N-major
      for (int i = 0; i < nc && good; ++i) {
        const uint32_t par = (uint32_t)(i & 1);
        // S^T = X q'^T : M = 128 rows, N = 64 heads, K = 512 in two channel halves
        for (int h2 = 0; h2 < 2 && good; ++h2) {
          good = ptx::mbar_wait(&S.x_full[h2], par, abort_flag, kAttnWaitBudget);
          if (!good) break;
          ptx::tc_fence_after();
#pragma unroll 4
          for (int ks = h2 * 16; ks < h2 * 16 + 16; ++ks) {
            const uint64_t ad = ptx::smem_desc_noswizzle(&S.X[2 * ks][0], kRows * 16, 128);
            const uint64_t bd = ptx::smem_desc_noswizzle(&S.q[2 * ks][0], kQPlane * 2, 128);
            ptx::mma_f16_ss(tS, ad, bd, idesc_s, ks > 0 ? 1u : 0u);
          }
        }
        if (!good) break;
        ptx::mma_commit(&S.s_full);
        // O^T += X^T P^T : four 128-channel M tiles, N = 64 heads, K = 128 rows
        good = ptx::mbar_wait(&S.p_full, par, abort_flag, kAttnWaitBudget);
        if (!good) break;
        ptx::tc_fence_after();
        for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
          for (int mt = 2 * h2; mt < 2 * h2 + 2; ++mt)
#pragma unroll
            for (int ks = 0; ks < kRows / 16; ++ks) {
              const uint64_t ad = ptx::smem_desc_noswizzle(&S.X[mt * 16][ks * 16 * 8], 128, kRows * 16);
              const uint64_t bd = ptx::smem_desc_noswizzle(&S.P[0][ks * 16 * 8], 128, kRows * 16);
              ptx::mma_f16_ss(tmem + (uint32_t)mt * 64u, ad, bd, idesc_o, (i > 0 || ks > 0) ? 1u : 0u);
            }
          ptx::mma_commit(&S.x_free[h2]);  // that channel half of X is no longer read
        }
      }
      if (!good && !*abort_flag) {
        *abort_flag = 1;
        report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 23);
      }
      // every MMA issued so far has completed before tensor memory is freed
      ptx::mma_commit(&S.drained);
      volatile int keep_waiting = 0;
      ptx::mbar_wait(&S.drained, 0, &keep_waiting, kAttnWaitBudget);
    }
  } else {
    // ------------------------------------------------------ rows and softmax
    const int q4 = warp & 3, hh = warp >> 2;
    const int rr = q4 * 32 + lane;  // row of this thread in the softmax (tensor-memory lane)
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    float m2 = -INFINITY, l_run = 0.0f;  // this lane's head hh * 32 + lane: reference (log2 units), sum
    S.m2w[warp][lane] = 0.0f;
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&S.q_full);
    bool good = true;
    for (int i = 0; i < nc && good; ++i) {
      const uint32_t par = (uint32_t)(i & 1);
      // the next chunk's index, in flight during the wait and the dequantization
      const int gr_next = (c0 + i + 1) * kRows + r;
      const int64_t idx_next = i + 1 < nc ? fetch_index(topk, dense_n, k, b, gr_next) : -1;
      if (i > 0) {
        good = ptx::mbar_wait_warp(&S.x_free[half], par ^ 1u, abort_flag, kAttnWaitBudget);
        if (!good) break;
      }
      const bool valid = dequant_half_row(S, rf, r, half);
      if (half == 0) S.valid[r] = valid ? 1 : 0;
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&S.x_full[half]);
      if (i + 1 < nc)
        issue_row(rf, idx_next, kv_codes, kv_scales, seq_stride, swa, n_swa, k, b, gr_next, half, ws, ex.win_pos,
                  win_lo);

      // ---- chunk softmax
      good = ptx::mbar_wait_warp(&S.s_full, par, abort_flag, kAttnWaitBudget) &&
             ptx::mbar_wait_warp(&S.x_full[0], par, abort_flag, kAttnWaitBudget) &&  // valid[] (acquire)
             ptx::mbar_wait_warp(&S.q_full, 0, abort_flag, kAttnWaitBudget);         // c2 (acquire)
      if (!good) break;
      ptx::tc_fence_after();
      float sv[32];
      {
        uint32_t a[32];
        ptx::tmem_ld_32x32b_x32(tS + lane_base + (uint32_t)hh * 32u, a);
        ptx::tmem_wait_ld();
        const bool v = S.valid[rr] != 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[j] = v ? __uint_as_float(a[j]) : -INFINITY;  // raw S
        float t[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) t[j] = sv[j];
        S.red[q4][hh * 32 + lane] = warp_reduce_scatter32(t, lane, MaxOp());
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&S.red_full);
      good = ptx::mbar_wait_warp(&S.red_full, par, abort_flag, kAttnWaitBudget);
      if (!good) break;
      const int h = hh * 32 + lane;
      const float cm = fmaxf(fmaxf(S.red[0][h], S.red[1][h]), fmaxf(S.red[2][h], S.red[3][h])) * S.c2[h];
      float alpha = 1.0f;
      if (cm > m2 + kTau2) {  // also the first chunk with a row of this head
        alpha = m2 == -INFINITY ? 0.0f : ptx::ex2(m2 - cm);
        m2 = cm;
      }
      const bool moved = __any_sync(0xffffffffu, alpha != 1.0f);
      const bool rescale = i > 0 && moved;
      if (moved) {  // this warp's copy of its heads' references
        S.m2w[warp][lane] = m2 == -INFINITY ? 0.0f : m2;
        __syncwarp();
      }
      if (i > 0) {  // P and O of the previous chunk are no longer read
        good = ptx::mbar_wait_warp(&S.x_free[1], par ^ 1u, abort_flag, kAttnWaitBudget);
        if (!good) break;
        ptx::tc_fence_after();
      }
      {
        float pr[32];  // the probabilities as rounded to f16, for the sums
        uint32_t ph[16];
        const float4* m2v = reinterpret_cast<const float4*>(S.m2w[warp]);
        const float4* c2v = reinterpret_cast<const float4*>(&S.c2[hh * 32]);
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float4 mq = m2v[j / 4], cq = c2v[j / 4];
          const float mm[4] = {mq.x, mq.y, mq.z, mq.w}, cc4[4] = {cq.x, cq.y, cq.z, cq.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) pr[j + t] = ptx::ex2(fmaf(sv[j + t], cc4[t], -mm[t]));  // -inf rows -> 0
        }
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const __half2 h2 = __floats2half2_rn(pr[j], pr[j + 1]);
          ph[j / 2] = *reinterpret_cast<const uint32_t*>(&h2);
          const float2 back = __half22float2(h2);
          pr[j] = back.x;
          pr[j + 1] = back.y;
        }
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4)
          *reinterpret_cast<uint4*>(&S.P[hh * 4 + i4][rr * 8]) =
              make_uint4(ph[4 * i4], ph[4 * i4 + 1], ph[4 * i4 + 2], ph[4 * i4 + 3]);
        S.red2[q4][h] = warp_reduce_scatter32(pr, lane, AddOp());
      }
      if (rescale) {  // O^T columns of this warp's heads, its lane quarter, all four M tiles
#pragma unroll 1
        for (int mt = 0; mt < 4; ++mt) {
          uint32_t a[32];
          const uint32_t ta = tmem + lane_base + (uint32_t)mt * 64u + (uint32_t)hh * 32u;
          ptx::tmem_ld_32x32b_x32(ta, a);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            a[j] = __float_as_uint(__uint_as_float(a[j]) * __shfl_sync(0xffffffffu, alpha, j));
          ptx::tmem_st_32x32b_x32(ta, a);
        }
        ptx::tmem_wait_st();
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&S.p_full);
      good = ptx::mbar_wait_warp(&S.p_full, par, abort_flag, kAttnWaitBudget);
      if (!good) break;
      l_run = fmaf(alpha, l_run, ((S.red2[0][h] + S.red2[1][h]) + S.red2[2][h]) + S.red2[3][h]);
    }
    if (good)
      good = ptx::mbar_wait_warp(&S.x_free[1], (uint32_t)((nc - 1) & 1), abort_flag, kAttnWaitBudget);
    if (!good && lane == 0 && !*abort_flag) {
      *abort_flag = 1;
      report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 24);
    }
    // ---- epilogue: O^T rows = channels of this lane quarter, 32 heads per warp;
    // for each head the warp stores 32 consecutive channels.  The sink joins
    // the denominator here (split queries: in the merge); with RoPE the last
    // 64 channels turn back by -qpos (pairs are adjacent lanes; the turn is
    // linear, so partials may take it before the merge).
    if (good) {
      ptx::tc_fence_after();
      const int h = hh * 32 + lane;
      const float m_nat = m2 / kLog2e;  // reference in natural units
      float den = l_run;
      if (!kPartial && kEx && ex.sink) den += ptx::ex2(ex.sink[h] * kLog2e - m2);  // 2^(z2 - m2); m2 = -inf -> inf
      const float inv = kPartial ? 1.0f : (den > 0.0f ? 1.0f / den : 0.0f);
      if (q4 == 0) {
        if (kPartial) {
          part_ml[((int64_t)b * gridDim.x + split) * kHAtt + h] = make_float2(m_nat, l_run);
        } else if (lse) {
          if (kEx && ex.sink) {
            const float z = ex.sink[h], mx = fmaxf(m_nat, z);
            lse[b * kHAtt + h] = mx + logf(l_run * expf(m_nat - mx) + expf(z - mx));
          } else {
            lse[b * kHAtt + h] = l_run > 0.0f ? m_nat + logf(l_run) : -INFINITY;
          }
        }
      }
      float* ob = kPartial ? part_o + ((int64_t)b * gridDim.x + split) * kHAtt * kDMain
                           : out + (int64_t)b * kHAtt * kDMain;
      float tc = 1.0f, ts = 0.0f;  // cos / sin of this lane's pair angle (channel c, c ^ 1)
      if (kEx && ex.rope && 3 * kRows + rr >= kRopeFirst)
        rope_cos_sin(ex.th.t[(3 * kRows + rr - kRopeFirst) / 2], (double)ex.qpos[b], tc, ts);
      if (lane & 1) ts = -ts;  // turning back by -t: x' = x c + y s, y' = y c - x s
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t a[32];
        ptx::tmem_ld_32x32b_x32(tmem + lane_base + (uint32_t)mt * 64u + (uint32_t)hh * 32u, a);
        ptx::tmem_wait_ld();
        const int c = mt * kRows + rr;
        const bool turn = kEx && ex.rope && mt == 3 && q4 >= 2;  // warp-uniform: channels 448..511
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float v = __uint_as_float(a[j]) * __shfl_sync(0xffffffffu, inv, j);
          if (turn) {
            const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
            v = fmaf(v, tc, partner * ts);
          }
          ob[(hh * 32 + j) * kDMain + c] = v;
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kCtlWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kAttnTmemCols);
  }
}

__global__ void __launch_bounds__(128) k_attn_merge(const float* __restrict__ part_o,
                                                    const float2* __restrict__ part_ml, int nchunks,
                                                    const float* __restrict__ sink, float* __restrict__ out,
                                                    float* __restrict__ lse) {
  const int bh = blockIdx.x;  // b * 64 + h
  const int b = bh / kHAtt, h = bh % kHAtt;
  ptx::griddep_wait();  // the partials come from the previous kernel
  float M = -INFINITY;
  for (int c = 0; c < nchunks; ++c) M = fmaxf(M, part_ml[((int64_t)b * nchunks + c) * kHAtt + h].x);
  const float z = sink ? sink[h] : -INFINITY;  // the sink joins the denominator once per query
  const float ref = fmaxf(M, z);
  float L = sink ? expf(z - ref) : 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = 0; c < nchunks; ++c) {
    const int64_t pc = ((int64_t)b * nchunks + c) * kHAtt + h;
    const float2 ml = part_ml[pc];
    if (ml.y <= 0.0f) continue;
    const float f = expf(ml.x - ref);
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
  if (lse && threadIdx.x == 0) lse[bh] = L > 0.0f ? ref + logf(L) : -INFINITY;
}

struct AttnWs {
  float* part_o;    // [B][nsplit][64][512] (split queries only)
  float2* part_ml;  // [B][nsplit][64]
  size_t bytes;
};

// Chunks per CTA and CTAs per query: one CTA per query once the batch fills the
// GPU; below that a query's chunks are spread over up to kFillCtas / B CTAs
// (then evened out) at the cost of a merge.  Depends only on the shapes, so the
// workspace size does too.
constexpr int kFillCtas = 148;
struct AttnPlan {
  int nchunks, cps, nsplit;
};
AttnPlan attn_plan(int32_t B, int32_t k, int32_t n_swa) {
  AttnPlan p;
  p.nchunks = (int)cdiv(k + n_swa, kRows);
  if (p.nchunks < 1) p.nchunks = 1;
  int want = B >= kFillCtas ? 1 : kFillCtas / B;
  want = want < 1 ? 1 : (want > p.nchunks ? p.nchunks : want);
  p.cps = (int)cdiv(p.nchunks, want);
  p.nsplit = (int)cdiv(p.nchunks, p.cps);
  return p;
}

AttnWs attn_ws_layout(void* ws, int32_t B, const AttnPlan& plan) {
  AttnWs L{};
  size_t off = kWsHeader;
  char* base = (char*)ws;
  if (plan.nsplit > 1) {
    L.part_o = (float*)(base ? base + off : nullptr);
    off += align_up((size_t)B * plan.nsplit * kHAtt * kDMain * 4, 256);
    L.part_ml = (float2*)(base ? base + off : nullptr);
    off += align_up((size_t)B * plan.nsplit * kHAtt * 8, 256);
  }
  L.bytes = off;
  return L;
}

}  // namespace

}  // namespace csa2

extern "C" size_t csa2_sparse_attn_workspace_size(int32_t B, int32_t k, int32_t n_swa) {
  if (B <= 0 || k < 0 || n_swa < 0) return 0;
  return csa2::attn_ws_layout(nullptr, B, csa2::attn_plan(B, k, n_swa)).bytes;
}

namespace csa2 {
namespace {

// One attention call over k rows per query named by topk (or, dense_n given,
// entries 0 .. dense_n[b] - 1) joined with n_swa window rows.
csa2_status attn_run(const csa2_kv_planes* kv, int32_t B, const int32_t* topk, const int32_t* dense_n, int32_t k,
                     const uint8_t* swa_e4m3, int32_t n_swa, const void* q_bf16, float softmax_scale,
                     const csa2_norm_rope* q_nr, const int64_t* q_pos, const float* sink, const csa2_window* win,
                     float* out, float* lse_out, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (win && (!win->row_pos || !win->lo || !aligned(win->row_pos, 8) || !aligned(win->lo, 8)))
    return CSA2_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || softmax_scale > 3.0e38f) return CSA2_ERR_INVALID_ARG;  // positive, finite
  if (q_nr && (!norm_rope_ok(q_nr) || (q_nr->rope && !q_pos))) return CSA2_ERR_INVALID_ARG;
  if ((q_pos && !aligned(q_pos, 8)) || (sink && !aligned(sink, 4))) return CSA2_ERR_INVALID_ARG;
  AttnExtras ex{};
  ex.qnorm_w = q_nr ? q_nr->norm_weight : nullptr;
  ex.eps = q_nr ? q_nr->norm_eps : 0.0f;
  ex.rope = q_nr ? q_nr->rope : 0;
  ex.qpos = ex.rope ? q_pos : nullptr;
  ex.sink = sink;
  ex.win_pos = win && n_swa > 0 ? win->row_pos : nullptr;
  ex.win_lo = win && n_swa > 0 ? win->lo : nullptr;
  if (ex.rope) ex.th = make_rope_theta(q_nr->rope_base);
  if (!aligned(q_bf16, 16) || !aligned(out, 16) || (swa_e4m3 && !aligned(swa_e4m3, 16)))
    return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  const AttnPlan plan = attn_plan(B, k, n_swa);
  AttnWs L = attn_ws_layout(ws, B, plan);
  if (ws_bytes < L.bytes) return CSA2_ERR_WORKSPACE;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;
  const int smem = (int)sizeof(AttnSmem);
  const bool partial = plan.nsplit > 1;
  const bool extras = ex.qnorm_w || ex.rope || ex.sink;
  auto kern = partial ? (extras ? k_attn<true, true> : k_attn<true, false>)
                      : (extras ? k_attn<false, true> : k_attn<false, false>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return CSA2_ERR_CUDA;
  {
    KernelTimer timer(partial ? "k_attn_part" : "k_attn", st);
    launch_pdl(kern, dim3(plan.nsplit, B), dim3(kAT), (size_t)smem, st, kv->kv_codes, kv->kv_scales, kv->seq_stride,
               topk, dense_n, k, swa_e4m3, n_swa, (const uint16_t*)q_bf16, softmax_scale, ex, plan.nchunks, plan.cps,
               out, lse_out, L.part_o, L.part_ml, ws);
  }
  if (partial) {
    KernelTimer timer("k_attn_merge", st);
    launch_pdl(k_attn_merge, dim3(B * kHAtt), dim3(128), 0, st, L.part_o, L.part_ml, plan.nsplit, sink, out, lse_out);
  }
  return launch_status();
}

}  // namespace
}  // namespace csa2

extern "C" csa2_status csa2_sparse_attn_decode(const csa2_kv_planes* kv, int32_t B, const int32_t* topk,
                                               int32_t k, const uint8_t* swa_e4m3, int32_t n_swa,
                                               const void* q_bf16, float softmax_scale,
                                               const csa2_norm_rope* q_nr, const int64_t* q_pos,
                                               const float* sink, const csa2_window* win, float* out,
                                               float* lse_out, void* ws, size_t ws_bytes, csa2_stream stream) {
  using namespace csa2;
  if (!planes_ok(kv) || B <= 0 || B > 65535 || k < 0 || k > CSA2_MAX_TOPK || n_swa < 0 || n_swa > CSA2_MAX_SWA)
    return CSA2_ERR_INVALID_ARG;
  if ((k > 0 && !topk) || (n_swa > 0 && !swa_e4m3) || !q_bf16 || !out) return CSA2_ERR_INVALID_ARG;
  return attn_run(kv, B, topk, nullptr, k, swa_e4m3, n_swa, q_bf16, softmax_scale, q_nr, q_pos, sink, win, out,
                  lse_out, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" size_t csa2_dense_attn_workspace_size(int32_t B, int64_t n_max, int32_t n_swa) {
  if (B <= 0 || n_max < 0 || n_max > CSA2_MAX_DENSE || n_swa < 0) return 0;
  return csa2::attn_ws_layout(nullptr, B, csa2::attn_plan(B, (int32_t)n_max, n_swa)).bytes;
}

extern "C" csa2_status csa2_dense_attn_decode(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries,
                                              int64_t n_max, const uint8_t* swa_e4m3, int32_t n_swa,
                                              const void* q_bf16, float softmax_scale,
                                              const csa2_norm_rope* q_nr, const int64_t* q_pos,
                                              const float* sink, const csa2_window* win, float* out,
                                              float* lse_out, void* ws, size_t ws_bytes, csa2_stream stream) {
  using namespace csa2;
  if (!planes_ok(kv) || B <= 0 || B > 65535 || n_max < 0 || n_max > CSA2_MAX_DENSE || n_max > kv->seq_stride ||
      n_swa < 0 || n_swa > CSA2_MAX_SWA)
    return CSA2_ERR_INVALID_ARG;
  if ((n_max > 0 && !n_entries) || (n_swa > 0 && !swa_e4m3) || !q_bf16 || !out) return CSA2_ERR_INVALID_ARG;
  if (n_entries && !aligned(n_entries, 4)) return CSA2_ERR_INVALID_ARG;
  return attn_run(kv, B, nullptr, n_entries, (int32_t)n_max, swa_e4m3, n_swa, q_bf16, softmax_scale, q_nr, q_pos,
                  sink, win, out, lse_out, ws, ws_bytes, (cudaStream_t)stream);
}
