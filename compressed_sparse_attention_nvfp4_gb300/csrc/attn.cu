// Sparse MQA decode attention over the selected FP4 entries joined with the
// layer's FP8 sliding window, one softmax over both ("DeepSeek-V4: Towards
// Highly Efficient Million-Token Context Intelligence", CSA step 3 and the
// sliding-window branch; "DeepSeek-V4.1-Flash: pushing the limits of KV cache
// compression", 4.1).  K = V = the 512-channel latent; 64 heads share it.
//
// k_attn stages q in shared memory as q' = q 2^-s_h in f16 with a power-of-two
// prescale per head (exact for bf16 q), then runs the query's rows (selected
// entries, then window rows) in chunks of 64 on the tensor cores (tcgen05,
// kind::f16, fp32 accumulation in tensor memory):
//   1. the chunk's rows are dequantized into shared memory as f16 (exact:
//      E2M1 x E4M3 has at most 6 significant bits), interleaved
//      X[c/8][row][c%8]: K-major for S, M-major for O;
//   2. S[64 heads x 64 rows] = q' X^T (heads as M, so each softmax thread owns
//      one head and its rows lie in its own registers), as two accumulators over
//      the channel halves that the softmax adds;
//   3. online softmax per head, P rounded to f16 once, l = sums of the rounded P;
//   4. O^T[512 x 64] += X^T P^T (four 128-channel M tiles).
// Two chunk slots (rows, S accumulators, probabilities) let the tensor cores
// compute S of one chunk while the softmax of the other runs.  Small MMAs are
// bound by their issue (one thread issues about one per 44 cycles, fewer when
// busy warps share its scheduler), so four warps, one per scheduler, issue them:
// the two S halves and the two channel halves of O.  One CTA per query keeps O in tensor memory across all
// its chunks, so no partial result leaves the SM.  When the batch is too small
// to fill the GPU a query's chunks are split over a few CTAs, which write
// (max, l, O) partials that a merge kernel combines by log-sum-exp.
#include "codec.cuh"
#include "ptx.cuh"
#include "timing.cuh"

namespace csa2 {

namespace {

constexpr int kRows = 64;   // rows per chunk: the N of the S MMA, the K of the O MMAs
// warps 0-7: a quarter row each in the gather and dequantization, then the epilogue;
// warps 8-11: the softmax (one warp per tensor-memory lane quarter); warps 12 and 13:
// the S MMAs over channels 0-255 / 256-511 (warp 12 also sets up the barriers, tensor
// memory and the q copy); warps 14 and 15: the O MMAs of channels 0-255 / 256-511
constexpr int kGatherWarps = 8;
constexpr int kCtlWarp = 12;
constexpr int kOWarp = 14;
constexpr int kAT = 16 * 32;
constexpr float kLog2e = 1.4426950408889634f;
// the softmax reference (log2 units) moves only when a chunk exceeds it by
// more than 8 nats, so probabilities stay below e^8 (inside f16)
constexpr float kTau2 = 8.0f * kLog2e;
// the reference of a head with no row yet: finite, so that 2^(S c2 - kNoRef) of a
// missing (-inf) row stays 0, and far below any logit, so that a row exceeds it
constexpr float kNoRef = -1.0e30f;
// q' plane stride: 64 heads x 16 bytes, unpadded, so that every core matrix the
// S MMAs read sits on a 128-byte line
constexpr int kQPlane = kHAtt * 8;       // in f16 elements (1024 bytes)
constexpr int kXPlane = kRows * 8;       // f16 elements per 8-channel plane of a slot (1024 bytes)
constexpr uint32_t kAttnTmemCols = 512;  // O^T 256 columns; per S half, two slots of 64
constexpr uint32_t kTmemS = 256;         // first column of S half 0, slot 0 (half h, slot s: + 128 h + 64 s)
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
  uint16_t X[2][kDMain / 8][kXPlane];  // per slot: f16 rows [c/8][row][c%8]; planes 0-31 / 32-63 = channel halves
  uint16_t q[kDMain / 8][kQPlane];     // f16 q' [c/8][head][c%8]
  uint16_t P[2][kRows / 8][kHAtt * 8]; // per slot: f16 probabilities [row/8][head][row%8] (P^T K-major)
  float c2[kHAtt];                     // log2(e) * softmax_scale * 2^s_h: logit (log2 units) per raw S
  float alpha[kHAtt];                  // factor of O and l when a head's reference moved
  float inv[kHAtt];                    // 1 / softmax denominator (or 1 for partials)
  uint32_t vmask[2][2];                // per slot and 32-row half: rows that exist
  uint64_t q_load;                     // the query's bf16 rows copied into slot 1 (bulk copy)
  uint64_t q_full;                     // q' and c2 written (the 8 softmax and MMA warps)
  uint64_t x_full[2][2];               // per slot, channel half of X written (8 row warps each)
  uint64_t s_full[2];                  // per slot: S MMAs complete (both halves)
  uint64_t p_full[2];                  // per slot: P written (4 softmax warps)
  uint64_t x_free[2][2];               // per slot, channel half: the O MMAs reading it complete
  uint64_t fin;                        // 1 / denominators posted (4 softmax warps)
  uint64_t drained;                    // every MMA issued complete (four MMA warps)
  uint32_t tmem_base;
  int abort_flag;
};

// fits the 227 KB of shared memory a CTA may have (and so every MMA operand sits
// below 256 KB, which the constant-stepped descriptors rely on)
static_assert(sizeof(AttnSmem) <= 232448, "attention shared memory");

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

// q' = q_h 2^-s_h in f16 with 2^s_h bringing the head's largest |q| to
// [2^14, 2^15), clamped so that both 2^s_h and 2^-s_h are normal fp32 values;
// bf16 q keeps q' exact and inside the f16 range (with RMSNorm or RoPE the
// fp32 result is rounded to f16 once).  One bulk copy brings the query's bf16
// rows ([64][512]) into row slot 1; the softmax and MMA warps, idle until the
// first chunk's rows are written, convert them from there while the row warps
// dequantize chunk 0 into slot 0.  Warp 8 + w takes heads 8w .. 8w + 7: lane
// l = 8g + t head 8w + t over the 8-channel planes (t + 4i + g) mod 64, i < 16.
// The eight lanes of a phase then read eight different banks of the bf16 rows
// (their planes differ mod 8) and write eight consecutive head slots of the
// [c/8][head][c%8] image, so neither side conflicts; the values are read again
// for each pass rather than held (a pass holding all 64 registers spills other
// warps' state), and the four lanes of a head combine its maximum (and sum of
// squares) with two shuffles.
template <bool kEx>
__device__ __forceinline__ void stage_q(AttnSmem& S, const uint16_t* qs, float scale, int w, int lane,
                                        const AttnExtras& ex, int b) {
  const int t = lane & 7, g = lane >> 3, h = 8 * w + t;
  const uint4* src = reinterpret_cast<const uint4*>(qs + h * kDMain);
  const bool norm = kEx && ex.qnorm_w != nullptr;
  const bool rot = kEx && ex.rope;
  float r = 1.0f;  // 1 / RMS of the head
  if (norm) {
    float ss = 0.0f;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const uint4 q4 = src[(t + 4 * i + g) & 63];
      const uint32_t w4[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float v0 = __uint_as_float(w4[j] << 16), v1 = __uint_as_float(w4[j] & 0xFFFF0000u);
        ss = fmaf(v0, v0, ss);
        ss = fmaf(v1, v1, ss);
      }
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 8);
    ss += __shfl_xor_sync(0xffffffffu, ss, 16);
    r = 1.0f / sqrtf(ss / (float)kDMain + ex.eps);
  }
  // RoPE turns planes 56 .. 63 (pairs 4 (p - 56) + pr); lane l keeps the cosine and
  // sine of pair l (every head turns by the same angles)
  float rcos = 1.0f, rsin = 0.0f;
  if (rot) rope_cos_sin(ex.th.t[lane], (double)ex.qpos[b], rcos, rsin);
  // the 8 channels of plane p after RMSNorm and RoPE
  auto plane = [&](int p, float (&v)[8]) {
    const uint4 q4 = src[p];
    const uint32_t w4[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w4[j] << 16);
      v[2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
    }
    if (norm) {
      const float4* wv = reinterpret_cast<const float4*>(ex.qnorm_w + 8 * p);
      const float4 a = __ldg(wv), c = __ldg(wv + 1);
      const float wq[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = wq[k] * (v[k] * r);
    }
    if (rot) {
#pragma unroll
      for (int pr = 0; pr < 4; ++pr) {  // every lane shuffles; only planes 56 .. 63 turn
        const int pair = (4 * (p - 56) + pr) & 31;
        const float c = __shfl_sync(0xffffffffu, rcos, pair), sn = __shfl_sync(0xffffffffu, rsin, pair);
        if (p >= 56) rope_pair(v[2 * pr], v[2 * pr + 1], c, sn);
      }
    }
  };
  float mx = 0.0f;
  if (kEx) {
#pragma unroll 2
    for (int i = 0; i < 16; ++i) {
      float v[8];
      plane((t + 4 * i + g) & 63, v);
#pragma unroll
      for (int k = 0; k < 8; ++k) mx = fmaxf(mx, fabsf(v[k]));
    }
  } else {  // |bf16| orders as its bit pattern: a packed 16-bit maximum over the raw words
    uint32_t m2 = 0;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const uint4 q4 = src[(t + 4 * i + g) & 63];
      const uint32_t w4[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) asm("max.u16x2 %0, %0, %1;" : "+r"(m2) : "r"(w4[j] & 0x7FFF7FFFu));
    }
    mx = __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16);
  }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
  const int sig = mx > 0.0f ? min(max(floor_log2_f32(mx) - 14, -126), 126) : 0;
  const float inv = exp2i_f32(-sig);  // exact power of two: q 2^-sig rounds only in the f16 conversion
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int p = (t + 4 * i + g) & 63;
    float v[8];
    plane(p, v);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h2 = __floats2half2_rn(v[2 * j] * inv, v[2 * j + 1] * inv);
      o[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(&S.q[p][h * 8]) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (g == 0) S.c2[h] = kLog2e * scale * exp2i_f32(sig);
}

// Whether some of the four softmax warps (named barrier 2, 128 threads) saw a
// logit above its head's reference (lane 0 of each warp posts `wover`) and
// whether one of them gave up waiting (lanes 1-8 post `wbad`): one barrier, the
// count of posted predicates below 8 for the first, at least 8 for the second.
// Every softmax warp passes it once per chunk, also after a failed wait, so no
// warp is left at the barrier.
__device__ __forceinline__ uint32_t softmax_vote(bool wover, bool wbad, int lane) {
  const uint32_t pred = lane == 0 ? (wover ? 1u : 0u) : (lane <= 8 && wbad ? 1u : 0u);
  uint32_t n;
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.popc.u32 %0, 2, 128, p;\n\t}"
      : "=r"(n)
      : "r"(pred)
      : "memory");
  return n;
}
// the four softmax warps (named barrier 2): shared-memory writes before it are seen after it
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// One thread's share of a chunk row, fetched two chunks ahead of its
// dequantization.  Gather warp w takes chunk rows 8w .. 8w + 7: lane l row
// 8w + l % 8 and column block cb = l / 8, so each load instruction reads 64
// contiguous bytes of eight rows (eight cache lines, not one line per lane).  A
// selected entry: 16-byte code chunks 4i + cb (i < 4; channels 32 (4i + cb) ..)
// and the entry's 32 scale bytes; a window row: 16-byte chunks 4i + cb (i < 8;
// channels 16 (4i + cb) ..).  Channels below 256 (channel half 0) come from i < 2
// (entries) or i < 4 (window rows).
struct RowFetch {
  uint4 raw[8];  // entry: raw[0..3] codes, raw[4..5] scales; window row: raw[0..7]
  int kind;      // 0 = no row, 1 = selected entry, 2 = window row
};

// entry of chunk row gr (rows gr >= k are window rows or padding): topk[b][gr],
// or, dense, entry gr itself while gr < dense_n[b]
__device__ __forceinline__ int64_t fetch_index(const int32_t* __restrict__ topk, const int32_t* __restrict__ dense_n,
                                               int k, int b, int gr) {
  if (gr >= k) return -1;
  if (dense_n) return gr < __ldg(dense_n + b) ? gr : -1;
  return (int64_t)topk[(int64_t)b * k + gr];
}

// Starts this lane's loads of chunk row gr: a selected entry (gr < k, index idx),
// a window row (k <= gr < k + n_swa, visible) or nothing.
__device__ __forceinline__ void issue_row(RowFetch& f, int64_t idx, const uint8_t* __restrict__ kv_codes,
                                          const uint8_t* __restrict__ kv_scales, int64_t seq_stride,
                                          const uint8_t* __restrict__ swa, int n_swa, int k, int b, int gr,
                                          int cb, void* ws, const int64_t* __restrict__ win_pos, int64_t win_lo) {
  f.kind = 0;
  if (gr < k) {
    if (idx >= 0 && idx < seq_stride) {
      const int64_t e = (int64_t)b * seq_stride + idx;
      const uint4* cs = reinterpret_cast<const uint4*>(kv_codes + e * 256);
#pragma unroll
      for (int i = 0; i < 4; ++i) f.raw[i] = cs[4 * i + cb];
      const uint4* sc = reinterpret_cast<const uint4*>(kv_scales + e * 32);
      f.raw[4] = sc[0];
      f.raw[5] = sc[1];
      f.kind = 1;
    } else if (idx != -1 && cb == 0) {
      report_error(ws, CSA2_ERR_INDEX_RANGE, idx);
    }
  } else if (gr - k < n_swa && (!win_pos || win_pos[(int64_t)b * n_swa + (gr - k)] >= win_lo)) {
    const uint4* src = reinterpret_cast<const uint4*>(swa + ((int64_t)b * n_swa + (gr - k)) * kDMain);
#pragma unroll
    for (int i = 0; i < 8; ++i) f.raw[i] = src[4 * i + cb];
    f.kind = 2;
  }
}

// Writes this lane's channels of channel half h of row r (see RowFetch) to slot
// `slot` of X as f16 (zeros when there is no row): 32 channels per code chunk of
// an entry (planes 4c .. 4c + 3), 16 per chunk of a window row (planes 2k, 2k + 1).
// The eight lanes of a store phase write eight rows of one plane: no bank conflict.
__device__ __forceinline__ void dequant_half_row(AttnSmem& S, const RowFetch& f, int slot, int r, int cb, int h) {
  if (f.kind == 1) {
#pragma unroll
    for (int i = 2 * h; i < 2 * h + 2; ++i) {
      const int c = 4 * i + cb;  // code chunk: channels 32c .., scale groups 2c, 2c + 1
      const uint32_t sw = i == 0 ? f.raw[4].x : i == 1 ? f.raw[4].z : i == 2 ? f.raw[5].x : f.raw[5].z;
      const uint32_t sw1 = i == 0 ? f.raw[4].y : i == 1 ? f.raw[4].w : i == 2 ? f.raw[5].y : f.raw[5].w;
      // scale bytes 2c, 2c + 1 = bytes 2 cb, 2 cb + 1 of the word pair covering bytes 8i .. 8i + 7
      const uint32_t pair = ((cb < 2 ? sw : sw1) >> (16 * (cb & 1))) & 0xFFFFu;
      const uint32_t s0 = e4m3x2_to_f16x2((pair & 0xFFu) * 0x0101u);
      const uint32_t s1 = e4m3x2_to_f16x2((pair >> 8) * 0x0101u);
      const uint4 cw = f.raw[i];
      const uint32_t wq[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 8 channels: plane 4c + q
        uint32_t hq[4];
        e2m1x8_to_f16(wq[q], hq);
        const uint32_t sq = q < 2 ? s0 : s1;
        *reinterpret_cast<uint4*>(&S.X[slot][4 * c + q][r * 8]) =
            make_uint4(hmul2_u32(hq[0], sq), hmul2_u32(hq[1], sq), hmul2_u32(hq[2], sq), hmul2_u32(hq[3], sq));
      }
    }
  } else if (f.kind == 2) {
#pragma unroll
    for (int i = 4 * h; i < 4 * h + 4; ++i) {
      const int kc = 4 * i + cb;  // channels 16 kc ..
      const uint4 v = f.raw[i];
      *reinterpret_cast<uint4*>(&S.X[slot][2 * kc][r * 8]) =
          make_uint4(e4m3x2_to_f16x2(v.x), e4m3x2_to_f16x2(v.x >> 16), e4m3x2_to_f16x2(v.y),
                     e4m3x2_to_f16x2(v.y >> 16));
      *reinterpret_cast<uint4*>(&S.X[slot][2 * kc + 1][r * 8]) =
          make_uint4(e4m3x2_to_f16x2(v.z), e4m3x2_to_f16x2(v.z >> 16), e4m3x2_to_f16x2(v.w),
                     e4m3x2_to_f16x2(v.w >> 16));
    }
  } else {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 2 * h; i < 2 * h + 2; ++i) {
      const int c = 4 * i + cb;
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(&S.X[slot][4 * c + q][r * 8]) = z;
    }
  }
}

// Raw S of this lane's head over its 32 rows of a chunk (lanes 0-15: rows 0-31, lanes
// 16-31: rows 32-63, the head's lane of the M = 64 accumulator): the two channel halves'
// accumulators (at taddr and taddr + 128) added, -inf for the rows the mask `vm` has not.
__device__ __forceinline__ void load_scores(uint32_t taddr, uint32_t vm, float (&sv)[32]) {
  uint32_t a[32], c[32];
  ptx::tmem_ld_16x32bx2_x32<32>(taddr, a);
  ptx::tmem_ld_16x32bx2_x32<32>(taddr + 128u, c);
  ptx::tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i)
    sv[i] = ((vm >> i) & 1u) ? __uint_as_float(a[i]) + __uint_as_float(c[i]) : -INFINITY;
}

// The probabilities of one head (this lane) over its 32 rows of a chunk:
// p = 2^(raw S * c2 - m2) rounded to f16, packed in pairs of rows into ph.
// Returns whether some logit exceeds the reference by more than kTau2 (a head
// with no reference yet, kNoRef, is exceeded by any row).
__device__ __forceinline__ bool head_probs(const float (&sv)[32], float c2h, float m2ref, uint32_t (&ph)[16]) {
  float tmax = -INFINITY;
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const float e0 = fmaf(sv[2 * u], c2h, -m2ref), e1 = fmaf(sv[2 * u + 1], c2h, -m2ref);  // -inf rows -> -inf
    tmax = fmaxf(tmax, fmaxf(e0, e1));
    const __half2 h2 = __floats2half2_rn(ptx::ex2(e0), ptx::ex2(e1));
    ph[u] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  return tmax > kTau2;
}

// P^T of slot `slot`: head hd, rows 32 ch .. 32 ch + 31 ([row/8][head][row%8]).
__device__ __forceinline__ void store_probs(AttnSmem& S, int slot, int ch, int hd, const uint32_t (&ph)[16]) {
#pragma unroll
  for (int i4 = 0; i4 < 4; ++i4)
    *reinterpret_cast<uint4*>(&S.P[slot][ch * 4 + i4][hd * 8]) =
        make_uint4(ph[4 * i4], ph[4 * i4 + 1], ph[4 * i4 + 2], ph[4 * i4 + 3]);
}

__device__ __forceinline__ float sum_probs(const uint32_t (&ph)[16]) {
  float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ph[u]));
    s0 += f.x;
    s1 += f.y;
  }
  return s0 + s1;
}

// One CTA runs chunks [c0, c0 + nc) of query b's rows (64 each) with an online
// softmax; the output accumulates in tensor memory across the chunks.
//   warps 0-7: thread t dequantizes channels 128 (t / 64) .. of chunk row t % 64
//     into the chunk's slot, fetching the rows of the chunk two ahead meanwhile;
//     afterwards, the epilogue;
//   warps 8-15 first stage q' (while warps 0-7 dequantize the first two chunks),
//     then take their roles:
//   warps 8-11: the softmax; warp 8 + q owns heads 16 q .. + 15 (lanes 0-15 of
//     lane quarter q, the rows of an M = 64 accumulator) over all of a chunk's rows;
//   warps 12-15: the MMA issue (S halves, O halves).
// The softmax keeps, per head, a reference m (the running maximum, raised only
// when a chunk exceeds it by more than kTau2, which then rescales O and l), so
// probabilities stay below e^8.  Each chunk first forms P with the references it
// has; one vote over the four softmax warps (a reducing named barrier) tells
// whether some head needs a new one, and only then are the chunk's exact maxima
// exchanged.  The softmax runs in
// log2 units: p = 2^(raw S * c2_h - m2_h).
// kPartial: write the unnormalised O with (m, l) for the merge kernel instead
// of the normalised output.
// 16 warps, four per scheduler, whose 16 K registers then allow 128 per thread.
template <bool kPartial, bool kEx>
__global__ void __launch_bounds__(512, 1) k_attn(
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
      ptx::mbar_init(&S.q_load, 1);
      ptx::mbar_init(&S.q_full, 8);
      for (int s = 0; s < 2; ++s) {
        ptx::mbar_init(&S.x_full[s][0], kGatherWarps);
        ptx::mbar_init(&S.x_full[s][1], kGatherWarps);
        ptx::mbar_init(&S.s_full[s], 2);
        ptx::mbar_init(&S.p_full[s], 4);
        ptx::mbar_init(&S.x_free[s][0], 1);
        ptx::mbar_init(&S.x_free[s][1], 1);
      }
      ptx::mbar_init(&S.fin, 4);
      ptx::mbar_init(&S.drained, 4);  // the four MMA warps
      S.abort_flag = 0;
      ptx::fence_mbar_init();
    }
    __syncwarp();
    ptx::tmem_alloc(&S.tmem_base, kAttnTmemCols);
  }
  ptx::griddep_wait();  // q, the indices and the rows may come from the previous kernel
  if (warp == kCtlWarp && lane == 0) {  // the query's bf16 rows into slot 1 (free until chunk 1)
    ptx::mbar_arrive_expect_tx(&S.q_load, kHAtt * kDMain * 2);
    ptx::bulk_g2s(&S.X[1][0][0], qg + (int64_t)b * kHAtt * kDMain, kHAtt * kDMain * 2, &S.q_load);
  }
  const int r = 8 * (warp & 7) + (lane & 7), cb = lane >> 3;  // gather: chunk row, column block
  const int64_t win_lo = ex.win_pos ? max(ex.win_lo[b], (int64_t)0) : 0;  // window rows below it are not seen
  int64_t idx0 = -1, idx1 = -1;
  if (warp < kGatherWarps) {
    const int gr0 = c0 * kRows + r, gr1 = gr0 + kRows;
    idx0 = fetch_index(topk, dense_n, k, b, gr0);
    idx1 = nc > 1 ? fetch_index(topk, dense_n, k, b, gr1) : -1;
  }
  ptx::tc_fence_before();
  __syncthreads();  // barriers initialised, tensor memory allocated
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  if (warp >= kGatherWarps) {  // q' and c2 from slot 1, while the row warps dequantize chunk 0
    if (ptx::mbar_wait_warp(&S.q_load, 0, abort_flag, kAttnWaitBudget)) {
      stage_q<kEx>(S, &S.X[1][0][0], scale, warp - kGatherWarps, lane, ex, b);
    } else if (lane == 0 && !*abort_flag) {
      *abort_flag = 1;
      report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 25);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&S.q_full);
  }

  if (warp >= kCtlWarp) {
    // ------------------------------------------------------------ MMA issue
    // One warp per scheduler, each running its loop with the whole warp (uniform control
    // flow and descriptors; one elected lane issues each MMA and commit).
    bool good = true;
    const int h2 = (warp - kCtlWarp) & 1;  // channel half
    if (warp < kOWarp) {
      // S half h2 over channels 256 h2 .. + 255: 16 K steps as soon as that half of X is written
      good = ptx::mbar_wait_warp(&S.q_full, 0, abort_flag, kAttnWaitBudget);
      constexpr uint32_t idesc_s = ptx::idesc_f16(64, 64, 0);  // S = q' X^T: heads x rows
      // descriptors of the half's first K step; later steps add their byte offset / 16 to
      // the start-address field (every operand lies below 256 KB, so the field cannot carry)
      const uint64_t dSa = ptx::smem_desc_noswizzle(&S.q[32 * h2][0], kQPlane * 2, 128);
      const uint64_t dSb0 = ptx::smem_desc_noswizzle(&S.X[0][32 * h2][0], kXPlane * 2, 128);  // K-major rows
      const uint64_t dSb1 = ptx::smem_desc_noswizzle(&S.X[1][32 * h2][0], kXPlane * 2, 128);
      for (int j = 0; j < nc && good; ++j) {  // S(j) half = q'[:, half] X[:, half]^T : M = 64, N = 64, K = 256
        const int s = j & 1;
        const uint32_t ph = (uint32_t)((j >> 1) & 1);
        const uint64_t dSb = s ? dSb1 : dSb0;
        const uint32_t dst = tmem + kTmemS + 128u * (uint32_t)h2 + 64u * (uint32_t)s;
        good = ptx::mbar_wait_warp(&S.x_full[s][h2], ph, abort_flag, kAttnWaitBudget);
        if (!good) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 16; ++ks)  // q'[2 ks], X[s][2 ks] of the half: ks * 2048 bytes on
          ptx::mma_f16_ss_elect(dst, dSa + (uint64_t)(ks * 128), dSb + (uint64_t)(ks * 128), idesc_s,
                                ks > 0 ? 1u : 0u);
        ptx::mma_commit_elect(&S.s_full[s]);
      }
    } else {
      // O^T tiles 2 h2, 2 h2 + 1 (channels 256 h2 .. + 255)
      constexpr uint32_t idesc_o = ptx::idesc_f16(128, 64, 0) | (1u << 15);  // O^T += X^T P^T: A M-major
      const uint64_t dOa0 = ptx::smem_desc_noswizzle(&S.X[0][32 * h2][0], 128, kXPlane * 2);  // M-major channels
      const uint64_t dOa1 = ptx::smem_desc_noswizzle(&S.X[1][32 * h2][0], 128, kXPlane * 2);
      const uint64_t dOb0 = ptx::smem_desc_noswizzle(&S.P[0][0][0], kHAtt * 16, 128);  // K-major P^T
      const uint64_t dOb1 = ptx::smem_desc_noswizzle(&S.P[1][0][0], kHAtt * 16, 128);
      const uint32_t dst = tmem + 128u * (uint32_t)h2;
      for (int j = 0; j < nc && good; ++j) {  // O^T += X^T P^T : two 128-channel M tiles, N = 64, K = 64 rows
        const int s = j & 1;
        const uint32_t ph = (uint32_t)((j >> 1) & 1);
        const uint64_t dOa = s ? dOa1 : dOa0, dOb = s ? dOb1 : dOb0;
        good = ptx::mbar_wait_warp(&S.p_full[s], ph, abort_flag, kAttnWaitBudget);
        if (!good) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int ks = 0; ks < kRows / 16; ++ks)  // X[s][16 mt][128 ks] of the half: mt * 16384 + ks * 256
                                                  // bytes on; P[s][2 ks]: ks * 2048 bytes on
            ptx::mma_f16_ss_elect(dst + (uint32_t)mt * 64u, dOa + (uint64_t)(mt * 1024 + ks * 16),
                                  dOb + (uint64_t)(ks * 128), idesc_o, (j > 0 || ks > 0) ? 1u : 0u);
        ptx::mma_commit_elect(&S.x_free[s][h2]);  // this half of the slot's X (and P) no longer read
      }
    }
    if (!good && lane == 0 && !*abort_flag) {
      *abort_flag = 1;
      report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 23);
    }
    // every MMA the four warps issued has completed before tensor memory is freed
    ptx::mma_commit_elect(&S.drained);
    volatile int keep_waiting = 0;
    ptx::mbar_wait_warp(&S.drained, 0, &keep_waiting, kAttnWaitBudget);
  } else if (warp < kGatherWarps) {
    // ------------------------------------------ rows (gather, dequantization), epilogue
    const int q4 = warp & 3, ch = warp >> 2;  // epilogue: lane quarter, heads 32 ch ..
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    RowFetch rf0, rf1;  // rows of the even / odd chunks
    const int gr0 = c0 * kRows + r;
    rf1.kind = 0;
    issue_row(rf0, idx0, kv_codes, kv_scales, seq_stride, swa, n_swa, k, b, gr0, cb, ws, ex.win_pos, win_lo);
    if (nc > 1)
      issue_row(rf1, idx1, kv_codes, kv_scales, seq_stride, swa, n_swa, k, b, gr0 + kRows, cb, ws, ex.win_pos,
                win_lo);
    // this lane's entries in chunks j + 2 (loaded after chunk j) and j + 3 (index read then)
    int64_t idx2 = nc > 2 ? fetch_index(topk, dense_n, k, b, gr0 + 2 * kRows) : -1;
    int64_t idx3 = nc > 3 ? fetch_index(topk, dense_n, k, b, gr0 + 3 * kRows) : -1;
    bool good = true;
    for (int p = 0; 2 * p < nc && good; ++p) {
      const uint32_t ph = (uint32_t)(p & 1);
      // ---- rows of chunks 2p and 2p + 1 into slots 0 and 1
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int j = 2 * p + s;
        if (j >= nc || !good) break;
        RowFetch& f = s ? rf1 : rf0;
        const int gr = (c0 + j) * kRows + r;
        // each channel half as soon as O(j - 2) no longer reads it; half 0 also posts the rows
        // that exist (lanes 0-7 hold this warp's eight rows)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (j >= 2)
            good = ptx::mbar_wait_warp(&S.x_free[s][h], ph ^ 1u, abort_flag, kAttnWaitBudget);
          else if (j == 1 && h == 0)  // slot 1 holds the bf16 query until q' is staged
            good = ptx::mbar_wait_warp(&S.q_full, 0, abort_flag, kAttnWaitBudget);
          if (!good) break;
          dequant_half_row(S, f, s, r, cb, h);
          if (h == 0) {
            const uint32_t vm = __ballot_sync(0xffffffffu, f.kind != 0) & 0xFFu;
            if (lane == 0) reinterpret_cast<uint8_t*>(&S.vmask[s][(warp & 7) >> 2])[warp & 3] = (uint8_t)vm;
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&S.x_full[s][h]);
        }
        if (!good) break;
        if (j + 2 < nc)
          issue_row(f, idx2, kv_codes, kv_scales, seq_stride, swa, n_swa, k, b, gr + 2 * kRows, cb, ws, ex.win_pos,
                    win_lo);
        idx2 = idx3;
        idx3 = j + 4 < nc ? fetch_index(topk, dense_n, k, b, gr + 4 * kRows) : -1;
      }
    }
    // ---- epilogue: O^T rows = channels of this lane quarter, 32 heads per warp; for each
    // head the warp stores 32 consecutive channels.  With RoPE the last 64 channels turn
    // back by -qpos (pairs are adjacent lanes; the turn is linear, so partials may take it
    // before the merge).  The softmax warps post 1 / denominator per head first.
    if (good)  // the last O MMAs of both halves (each commit covers its warp's earlier ones)
      good = ptx::mbar_wait_warp(&S.fin, 0, abort_flag, kAttnWaitBudget) &&
             ptx::mbar_wait_warp(&S.x_free[(nc - 1) & 1][0], (uint32_t)(((nc - 1) >> 1) & 1), abort_flag,
                                 kAttnWaitBudget) &&
             ptx::mbar_wait_warp(&S.x_free[(nc - 1) & 1][1], (uint32_t)(((nc - 1) >> 1) & 1), abort_flag,
                                 kAttnWaitBudget);
    if (!good && lane == 0 && !*abort_flag) {
      *abort_flag = 1;
      report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 24);
    }
    if (good) {
      ptx::tc_fence_after();
      const int rr = q4 * 32 + lane;  // channel of this lane within a 128-channel tile
      const float inv = S.inv[32 * ch + lane];  // head 32 ch + lane; broadcast per column below
      float* ob = kPartial ? part_o + ((int64_t)b * gridDim.x + split) * kHAtt * kDMain
                           : out + (int64_t)b * kHAtt * kDMain;
      float tc = 1.0f, ts = 0.0f;  // cos / sin of this lane's pair angle (channel c, c ^ 1)
      if (kEx && ex.rope && 3 * 128 + rr >= kRopeFirst)
        rope_cos_sin(ex.th.t[(3 * 128 + rr - kRopeFirst) / 2], (double)ex.qpos[b], tc, ts);
      if (lane & 1) ts = -ts;  // turning back by -t: x' = x c + y s, y' = y c - x s
#pragma unroll 1
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t a[32];
        ptx::tmem_ld_32x32b_x32(tmem + lane_base + (uint32_t)mt * 64u + 32u * (uint32_t)ch, a);
        ptx::tmem_wait_ld();
        const int c = mt * 128 + rr;
        const bool turn = kEx && ex.rope && mt == 3 && q4 >= 2;  // warp-uniform: channels 448..511
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          float v = __uint_as_float(a[jj]) * __shfl_sync(0xffffffffu, inv, jj);
          if (turn) {
            const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
            v = fmaf(v, tc, partner * ts);
          }
          ob[(32 * ch + jj) * kDMain + c] = v;
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax
    // Warp 8 + q reads lane quarter q of tensor memory: heads 16q .. 16q + 15 of each S
    // accumulator in lanes 0-15.  Lane l takes head 16q + l % 16 over the chunk rows
    // 32 (l / 16) .. + 31, so the two lanes of a head share its exponentials; its maximum
    // and sum are combined across the pair (lanes l and l ^ 16).
    const int q4 = warp & 3, rh = lane >> 4;
    const bool owner = lane < 16;
    const int hd = 16 * q4 + (lane & 15);  // this lane's head
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    float m2 = -INFINITY;  // this head's reference (log2 units; the same in both lanes)
    float lsum = 0.0f;     // rounded probabilities of this lane's rows, summed over every chunk
    bool good = ptx::mbar_wait_warp(&S.q_full, 0, abort_flag, kAttnWaitBudget);  // c2 (acquire)
    const float c2h = S.c2[hd];
    // Every softmax warp runs every chunk up to its vote, also after a failed wait: the
    // vote tells all four of them at once to stop.
    for (int j = 0; j < nc; ++j) {
      const int s = j & 1;
      const uint32_t ph = (uint32_t)((j >> 1) & 1);
      // x_full of both halves: the row warps wrote X(j) after O(j - 2) released the slot, so
      // the P^T slot is free too; half 0 also posts the row mask
      good = good && ptx::mbar_wait_warp(&S.s_full[s], ph, abort_flag, kAttnWaitBudget) &&
             ptx::mbar_wait_warp(&S.x_full[s][0], ph, abort_flag, kAttnWaitBudget) &&
             ptx::mbar_wait_warp(&S.x_full[s][1], ph, abort_flag, kAttnWaitBudget);
      const uint32_t taS = tmem + lane_base + kTmemS + 64u * (uint32_t)s;  // half 0; half 1 at + 128
      uint32_t vm = 0;  // this lane's rows that exist
      // P with the reference so far: stands unless some head needs a new one
      uint32_t pp[16];  // this lane's 32 rows, f16 pairs
      bool over = false;
      if (good) {
        ptx::tc_fence_after();
        vm = S.vmask[s][rh];
        const float ref = m2 == -INFINITY ? kNoRef : m2;
        float sv[32];
        load_scores(taS, vm, sv);
        over = head_probs(sv, c2h, ref, pp);
        store_probs(S, s, rh, hd, pp);
        ptx::fence_proxy_async_smem();  // before the vote: its latency overlaps the other warps'
      }
      const uint32_t nv = softmax_vote(__any_sync(0xffffffffu, over), !good || *abort_flag != 0, lane);
      if (nv >= 8) {
        good = false;
        break;
      }
      float alpha = 1.0f;  // this head's factor for its sum and O
      if (nv != 0) {
        // the chunk's exact maximum of this head (both lanes' rows; S stays in tensor memory
        // until P is handed over)
        float sv[32], cm = -INFINITY;
        load_scores(taS, vm, sv);
#pragma unroll
        for (int i = 0; i < 32; ++i) cm = fmaxf(cm, sv[i]);
        cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
        cm *= c2h;  // -inf stays -inf (c2 > 0)
        if (cm > m2 + kTau2) {  // also the first chunk with a row of this head
          alpha = m2 == -INFINITY ? 0.0f : ptx::ex2(m2 - cm);
          m2 = cm;
        }
        const float ref = m2 == -INFINITY ? kNoRef : m2;
        (void)head_probs(sv, c2h, ref, pp);
        store_probs(S, s, rh, hd, pp);
        ptx::fence_proxy_async_smem();
        if (j > 0) {  // O^T holds earlier chunks: scale the columns of the heads that moved
          if (owner) S.alpha[hd] = alpha;
          softmax_sync();
          // O(j - 1) complete; a wait that gives up stops the loop at the next vote
          good = ptx::mbar_wait_warp(&S.x_free[s ^ 1][0], (uint32_t)(((j - 1) >> 1) & 1), abort_flag,
                                     kAttnWaitBudget) &&
                 ptx::mbar_wait_warp(&S.x_free[s ^ 1][1], (uint32_t)(((j - 1) >> 1) & 1), abort_flag,
                                     kAttnWaitBudget);
          if (good) {
            ptx::tc_fence_after();
            // this warp's share: O^T lanes of quarter q4 (channels), the columns of all 64 heads
#pragma unroll 1
            for (int c32 = 0; c32 < 2; ++c32) {
              const float a32 = S.alpha[32 * c32 + lane];
              if (!__any_sync(0xffffffffu, a32 != 1.0f)) continue;
#pragma unroll 1
              for (int mt = 0; mt < 4; ++mt) {
                uint32_t a[32];
                const uint32_t ta = tmem + lane_base + (uint32_t)mt * 64u + 32u * (uint32_t)c32;
                ptx::tmem_ld_32x32b_x32(ta, a);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                  a[jj] = __float_as_uint(__uint_as_float(a[jj]) * __shfl_sync(0xffffffffu, a32, jj));
                ptx::tmem_st_32x32b_x32(ta, a);
              }
              ptx::tmem_wait_st();
            }
          }
        }
      }
      if (good) {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.p_full[s]);  // the MMA warps wait; the softmax goes on
      }
      lsum = fmaf(alpha, lsum, sum_probs(pp));
    }
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);  // the head's two lanes: every row
    if (!good && lane == 0 && !*abort_flag) {
      *abort_flag = 1;
      report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 26);
    }
    // ---- this head's denominator, the lse / partials, 1 / denominator for the epilogue.
    // The sink joins the denominator here (split queries: in the merge).
    if (good && owner) {
      const float m_nat = m2 / kLog2e;  // reference in natural units
      float den = lsum;
      if (!kPartial && kEx && ex.sink) den += ptx::ex2(ex.sink[hd] * kLog2e - m2);  // 2^(z2 - m2); m2 = -inf -> inf
      S.inv[hd] = kPartial ? 1.0f : (den > 0.0f ? 1.0f / den : 0.0f);
      if (kPartial) {
        part_ml[((int64_t)b * gridDim.x + split) * kHAtt + hd] = make_float2(m_nat, lsum);
      } else if (lse) {
        if (kEx && ex.sink) {
          const float z = ex.sink[hd], mxv = fmaxf(m_nat, z);
          lse[b * kHAtt + hd] = mxv + logf(lsum * expf(m_nat - mxv) + expf(z - mxv));
        } else {
          lse[b * kHAtt + hd] = lsum > 0.0f ? m_nat + logf(lsum) : -INFINITY;
        }
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&S.fin);  // also on failure: the row warps then see the abort flag
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
    return launch_status();
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
