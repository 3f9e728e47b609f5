// Lightning-indexer scan on the 5th-generation tensor cores.
//
//   I_j = sum_h w_h ReLU(q_h . K^I_j)   ("DeepSeek-V4: Towards Highly Efficient
//   Million-Token Context Intelligence", CSA step 2; "DeepSeek-V4.1-Flash:
//   pushing the limits of KV cache compression", 4.1 and 4.3)
//
// One CTA streams a contiguous range of 128-entry tiles of one query (or, in
// pool mode, tiles of 16 pool blocks x 8 entries).  Warp roles:
//   warp 0      producer: a 2-D TMA load of the tile's FP4 codes (64 B/entry,
//               64-byte swizzle so that the row-per-thread reads below are free
//               of bank conflicts) and a 1-D bulk copy of its E8M0 scales
//               (4 B/entry) into an 8-stage shared-memory ring;
//   warp 1      allocates tensor memory and issues the MMAs (one thread):
//               D[128 entries x 32 heads] = A[128 x 128] * q^T, kind::f16,
//               A read from tensor memory, q from shared memory;
//   warps 2-5   dequantize: thread r owns entry r of the tile (TMEM lane r),
//               converts its 128 E2M1 codes with cvt.e2m1x2 -> f16x2, scales
//               each 32-element block by 2^(e_c - e_max) (exact, HMUL2), and
//               stores the row into the A tile in tensor memory;
//   warps 6-9   epilogue: read the row's 32 head dots from tensor memory,
//               score = 2^(e_max-127) * sum_h w'_h max(dot_h, 0); write the
//               score and/or the max of each 8-entry block.
// q^I is prescaled per head by a power of two 2^-s_h into f16 (exact for
// bf16 inputs) and w'_h = w_h 2^s_h, so the score is unchanged.
// Tensor memory: A tiles at columns [0,64) and [64,128), accumulators at
// [128,160) and [160,192) (two tiles in flight); 256 columns per CTA.
// Every mbarrier wait is bounded; a wait that gives up records
// CSA2_ERR_DEVICE_TIMEOUT and makes every role leave its loop.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "index_scan.cuh"
#include "codec.cuh"
#include "ptx.cuh"

namespace csa2 {

namespace {

constexpr int kTile = 128;
#ifndef CSA2_SCAN_STAGES
#define CSA2_SCAN_STAGES 8
#endif
constexpr int kStages = CSA2_SCAN_STAGES;  // shared-memory ring depth (tiles in flight)
constexpr int kAcc = 2;
// Dequant warps per TMEM lane quarter; each converts 1/kSplit of every row.
// Epilogue form of sum_h w_h ReLU(x_h): 1 = max then FMA, 0 = two FMAs with |x|.
#ifndef CSA2_SCAN_RELU_MAX
#define CSA2_SCAN_RELU_MAX 0
#endif
#ifndef CSA2_SCAN_SPLIT
#define CSA2_SCAN_SPLIT 1
#endif
constexpr int kSplit = CSA2_SCAN_SPLIT;
static_assert(kSplit == 1 || kSplit == 2, "row split must be 1 or 2");
constexpr int kDequantWarps = 4 * kSplit;
constexpr int kWordsPerThread = 16 / kSplit;  // 32-bit code words (8 elements each)
constexpr int kWarps = 2 + kDequantWarps + 4;
constexpr int kThreads = kWarps * 32;
constexpr int kEpiWarp0 = 2 + kDequantWarps;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kDCol0 = 128;
constexpr long long kWaitBudget = 1LL << 32;  // clock cycles (about 2 s)

struct __align__(1024) ScanSmem {
  uint8_t codes[kStages][kTile * 64];  // 1024-byte aligned stages (swizzle atoms)
  uint8_t scales[kStages][kTile * 4];
  uint16_t qB[16 * 32 * 8];  // f16 B operand: [k/8][head][k%8]
  float wq[32];
  float entry_scale[kAcc][kTile];
  uint64_t full[kStages], empty[kStages];
  uint64_t a_full[kAcc], mma_done[kAcc], d_free[kAcc];
  uint32_t tmem_base;
  int abort_flag;
};

struct ScanParams {
  const uint8_t* ix_codes;
  const uint8_t* ix_scales;
  int64_t seq_stride;
  const int32_t* n_entries;
  int64_t n_max;
  const uint16_t* q;
  const float* w;
  const int32_t* pool;  // pool mode when non-null (blocks of 8)
  int keep;
  int64_t ncand_max;
  int ctas_per_query;
  float* scores;
  int64_t score_stride;
  float* bmax;
  int64_t bmax_stride;
  void* ws;
};

__device__ __forceinline__ void scan_abort(ScanSmem& S, void* ws, int where) {
  *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
  report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, where);
}

// f16x2 holding 2^g in both halves, g <= 0 (0 below the f16 subnormal range)
__device__ __forceinline__ uint32_t pow2_f16x2(int g) {
  const uint32_t normal = (uint32_t)(15 + max(g, -14)) << 10;
  const uint32_t sub = g >= -24 ? (1u << ((g + 24) & 31)) : 0u;
  const uint32_t h = g >= -14 ? normal : sub;
  return h | (h << 16);
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// one 32-bit word of codes (elements 8i..8i+7) -> four f16x2 words; the word is
// unpacked into byte registers with a vector mov, which measured 1.8x faster
// than extracting each byte with shifts and masks before the conversion
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\tmov.b32 {t0, t1, t2, t3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t0;\n\tcvt.rn.f16x2.e2m1x2 %1, t1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, t2;\n\tcvt.rn.f16x2.e2m1x2 %3, t3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Where tile row r of tile t lives: entry index in the slot, validity, and
// whether its scale word came through the bulk copy.
struct RowInfo {
  int64_t j;
  bool valid;
  bool scale_in_smem;
};

__device__ __forceinline__ RowInfo row_info(const ScanParams& p, int b, int64_t n, int64_t t, int r,
                                            bool scale_bulk) {
  RowInfo ri;
  if (!p.pool) {
    const int64_t j0 = t * kTile;
    const int64_t cnt = min((int64_t)kTile, n - j0);
    ri.j = j0 + r;
    ri.valid = r < cnt;
    ri.scale_in_smem = scale_bulk && r < (cnt & ~3LL);
  } else {
    const int64_t slot = t * (kTile / 8) + r / 8;
    const int pb = slot < p.keep ? p.pool[(int64_t)b * p.keep + slot] : -1;
    const int64_t base = (int64_t)pb * 8;
    const int64_t cnt = (pb >= 0 && base < n) ? min((int64_t)8, n - base) : 0;
    ri.j = base + (r % 8);
    ri.valid = (r % 8) < cnt;
    ri.scale_in_smem = scale_bulk && (r % 8) < (cnt & ~3LL);
  }
  return ri;
}

__global__ void __launch_bounds__(kThreads, 2) k_scan_tc(const __grid_constant__ ScanParams p, const __grid_constant__ CUtensorMap map_tile,
              const __grid_constant__ CUtensorMap map_block) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  ScanSmem& S = *reinterpret_cast<ScanSmem*>(smem_raw);
  volatile int* abort_flag = &S.abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int b = blockIdx.y;

  int64_t n = p.n_entries[b];
  if (n > p.n_max) {
    if (threadIdx.x == 0 && blockIdx.x == 0) report_error(p.ws, CSA2_ERR_INDEX_RANGE, n);
    n = p.n_max;
  }
  if (n < 0) n = 0;
  const bool pooled = p.pool != nullptr;
  const int64_t ncand = pooled ? p.ncand_max : n;
  const int64_t ntiles = cdiv(ncand, kTile);
  const int64_t t_begin = ntiles * blockIdx.x / p.ctas_per_query;
  const int64_t t_end = ntiles * (blockIdx.x + 1) / p.ctas_per_query;
  const int my_tiles = (int)(t_end - t_begin);
  const bool scale_bulk = ((b * p.seq_stride) & 3) == 0;  // 16-byte aligned scale rows
  const uint8_t* scales_b = p.ix_scales + (int64_t)b * p.seq_stride * 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&S.full[s], 1);
      ptx::mbar_init(&S.empty[s], kDequantWarps);
    }
    for (int a = 0; a < kAcc; ++a) {
      ptx::mbar_init(&S.a_full[a], kDequantWarps);
      ptx::mbar_init(&S.mma_done[a], 1);
      ptx::mbar_init(&S.d_free[a], 4);
    }
    S.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (my_tiles > 0 && warp == 1) ptx::tmem_alloc(&S.tmem_base, kTmemCols);

  // q^I -> f16 B operand with a power-of-two prescale per head; w' = w 2^s
  for (int h = warp; h < kHIdx; h += kWarps) {
    const uint16_t* qh = p.q + ((int64_t)b * kHIdx + h) * kDIdx;
    const uint2 raw = *reinterpret_cast<const uint2*>(qh + 4 * lane);
    float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                  __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int sig = m > 0.0f ? floor_log2_f32(m) - 14 : 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = 4 * lane + e;
      const __half hv = __float2half_rn(ldexpf(v[e], -sig));
      S.qB[(k / 8) * 256 + h * 8 + (k % 8)] = *reinterpret_cast<const uint16_t*>(&hv);
    }
    if (lane == 0) S.wq[h] = ldexpf(p.w[(int64_t)b * kHIdx + h], sig);
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (my_tiles > 0) {
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        for (int i = 0; i < my_tiles; ++i) {
          const int s = i % kStages;
          const uint32_t ph = (uint32_t)(i / kStages) & 1u;
          if (!ptx::mbar_wait(&S.empty[s], ph ^ 1u, abort_flag, kWaitBudget)) {
            scan_abort(S, p.ws, 1);
            break;
          }
          const int64_t t = t_begin + i;
          if (!pooled) {
            const int64_t j0 = t * kTile;
            const uint32_t cnt = (uint32_t)min((int64_t)kTile, n - j0);
            const uint32_t cnt4 = scale_bulk ? (cnt & ~3u) : 0u;
            ptx::mbar_arrive_expect_tx(&S.full[s], kTile * 64u + cnt4 * 4u);
            ptx::tma_load_2d(S.codes[s], &map_tile, 0, (int)(b * p.seq_stride + j0), &S.full[s]);
            if (cnt4) ptx::bulk_g2s(S.scales[s], scales_b + j0 * 4, cnt4 * 4u, &S.full[s]);
          } else {
            int pbv[16];
            uint32_t cnt[16];
            uint32_t bytes = 0;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              const int64_t slot = t * 16 + u;
              pbv[u] = slot < p.keep ? p.pool[(int64_t)b * p.keep + slot] : -1;
              const int64_t base = (int64_t)pbv[u] * 8;
              cnt[u] = (pbv[u] >= 0 && base < n) ? (uint32_t)min((int64_t)8, n - base) : 0u;
              bytes += (cnt[u] ? 512u : 0u) + (scale_bulk ? (cnt[u] & ~3u) * 4u : 0u);
            }
            ptx::mbar_arrive_expect_tx(&S.full[s], bytes);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              if (!cnt[u]) continue;
              const int64_t base = (int64_t)pbv[u] * 8;
              ptx::tma_load_2d(S.codes[s] + u * 512, &map_block, 0, (int)(b * p.seq_stride + base),
                               &S.full[s]);
              const uint32_t c4 = scale_bulk ? (cnt[u] & ~3u) : 0u;
              if (c4) ptx::bulk_g2s(S.scales[s] + u * 32, scales_b + base * 4, c4 * 4u, &S.full[s]);
            }
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issue
      if (lane == 0) {
        constexpr uint32_t idesc = ptx::idesc_f16(128, 32, 0);
        for (int i = 0; i < my_tiles; ++i) {
          const int a = i % kAcc;
          const uint32_t u = (uint32_t)(i / kAcc) & 1u;
          if (!ptx::mbar_wait(&S.a_full[a], u, abort_flag, kWaitBudget) ||
              !ptx::mbar_wait(&S.d_free[a], u ^ 1u, abort_flag, kWaitBudget)) {
            scan_abort(S, p.ws, 2);
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_t = tmem + (uint32_t)a * 64u;
          const uint32_t d_t = tmem + kDCol0 + (uint32_t)a * 32u;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t bd = ptx::smem_desc_noswizzle(S.qB + ks * 512, 512, 128);
            ptx::mma_f16_ts(d_t, a_t + (uint32_t)ks * 8u, bd, idesc, ks > 0 ? 1u : 0u);
          }
          ptx::mma_commit(&S.mma_done[a]);
        }
      }
    } else if (warp < kEpiWarp0) {
      // ------------------------------------------------------------ dequant
      // warps w, w+4, ... share a TMEM lane quarter; part hf converts code
      // words hf*kWordsPerThread .. +kWordsPerThread-1 of each row
      const int sub = warp % 4;
      const int hf = (warp - 2) / 4;
      const int r = sub * 32 + lane;
      const uint32_t lane_addr =
          tmem + ((uint32_t)(sub * 32) << 16) + (uint32_t)(hf * kWordsPerThread * 4);
      for (int i = 0; i < my_tiles; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        const int a = i % kAcc;
        const uint32_t u = (uint32_t)(i / kAcc) & 1u;
        if (!ptx::mbar_wait_warp(&S.full[s], ph, abort_flag, kWaitBudget)) {
          scan_abort(S, p.ws, 3);
          break;
        }
        const RowInfo ri = row_info(p, b, n, t_begin + i, r, scale_bulk);
        uint32_t words[kWordsPerThread];
        uint32_t sc = 0;
        if (ri.valid) {
          // 64-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3)
          const unsigned char* row = S.codes[s] + r * 64;
          const int sw = (r >> 1) & 3;
#pragma unroll
          for (int c2 = 0; c2 < kWordsPerThread / 4; ++c2) {
            const int c = hf * (kWordsPerThread / 4) + c2;
            const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * (c ^ sw));
            words[4 * c2 + 0] = v.x;
            words[4 * c2 + 1] = v.y;
            words[4 * c2 + 2] = v.z;
            words[4 * c2 + 3] = v.w;
          }
          sc = ri.scale_in_smem ? *reinterpret_cast<const uint32_t*>(S.scales[s] + r * 4)
                                : *reinterpret_cast<const uint32_t*>(scales_b + ri.j * 4);
        } else {
#pragma unroll
          for (int k = 0; k < kWordsPerThread; ++k) words[k] = 0u;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.empty[s]);

        const int e0 = (int)(sc & 0xFFu), e1 = (int)((sc >> 8) & 0xFFu);
        const int e2 = (int)((sc >> 16) & 0xFFu), e3 = (int)(sc >> 24);
        const int emax = max(max(e0, e1), max(e2, e3));
        uint32_t mult[kWordsPerThread / 4];  // one per 32-element block this thread converts
#pragma unroll
        for (int c2 = 0; c2 < kWordsPerThread / 4; ++c2) {
          const int blk = hf * (kWordsPerThread / 4) + c2;
          mult[c2] = pow2_f16x2((blk == 0 ? e0 : blk == 1 ? e1 : blk == 2 ? e2 : e3) - emax);
        }

        // A[a] and entry_scale[a] are free once the epilogue released tile i-2
        if (!ptx::mbar_wait_warp(&S.d_free[a], u ^ 1u, abort_flag, kWaitBudget)) {
          scan_abort(S, p.ws, 4);
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int st32 = 0; st32 < kWordsPerThread / 8; ++st32) {
          uint32_t v[32];
#pragma unroll
          for (int wi = 0; wi < 8; ++wi) {  // code word -> elements 8*word .. 8*word+7
            const int word = st32 * 8 + wi;
            uint32_t h[4];
            e2m1x8_to_f16x2x4(words[word], h);
#pragma unroll
            for (int k = 0; k < 4; ++k) v[4 * wi + k] = hmul2_bits(h[k], mult[word / 4]);
          }
          ptx::tmem_st_32x32b_x32(lane_addr + (uint32_t)a * 64u + (uint32_t)st32 * 32u, v);
        }
        if (hf == 0) S.entry_scale[a][r] = ri.valid ? exp2i_f32(emax - 127) : 0.0f;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.a_full[a]);
      }
    } else {
      // ------------------------------------------------------------ epilogue
      const int sub = warp % 4;
      const int r = sub * 32 + lane;
      const uint32_t lane_addr = tmem + ((uint32_t)(sub * 32) << 16);
      for (int i = 0; i < my_tiles; ++i) {
        const int a = i % kAcc;
        const uint32_t u = (uint32_t)(i / kAcc) & 1u;
        if (!ptx::mbar_wait_warp(&S.mma_done[a], u, abort_flag, kWaitBudget) ||
            !ptx::mbar_wait_warp(&S.a_full[a], u, abort_flag, kWaitBudget)) {
          scan_abort(S, p.ws, 5);
          break;
        }
        ptx::tc_fence_after();
        uint32_t acc[32];
        ptx::tmem_ld_32x32b_x32(lane_addr + kDCol0 + (uint32_t)a * 32u, acc);
        ptx::tmem_wait_ld();
        const float es = S.entry_scale[a][r];
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.d_free[a]);

        const int64_t t = t_begin + i;
        const RowInfo ri = row_info(p, b, n, t, r, scale_bulk);
#if CSA2_SCAN_RELU_MAX
        float sum = 0.0f;
#pragma unroll
        for (int h = 0; h < 32; ++h) sum = fmaf(S.wq[h], fmaxf(__uint_as_float(acc[h]), 0.0f), sum);
        const float sp = sum, sa = sum;
#else
        // sum_h w_h max(x_h, 0) = (sum_h w_h x_h + sum_h w_h |x_h|) / 2 (|.| is a free
        // operand modifier, so this stays on the FMA pipe)
        float sp = 0.0f, sa = 0.0f;
        const float4* wq4 = reinterpret_cast<const float4*>(S.wq);
#pragma unroll
        for (int h4 = 0; h4 < 8; ++h4) {
          const float4 wv = wq4[h4];
          const float x0 = __uint_as_float(acc[4 * h4]), x1 = __uint_as_float(acc[4 * h4 + 1]);
          const float x2 = __uint_as_float(acc[4 * h4 + 2]), x3 = __uint_as_float(acc[4 * h4 + 3]);
          sp = fmaf(wv.x, x0, sp);
          sa = fmaf(wv.x, fabsf(x0), sa);
          sp = fmaf(wv.y, x1, sp);
          sa = fmaf(wv.y, fabsf(x1), sa);
          sp = fmaf(wv.z, x2, sp);
          sa = fmaf(wv.z, fabsf(x2), sa);
          sp = fmaf(wv.w, x3, sp);
          sa = fmaf(wv.w, fabsf(x3), sa);
        }
#endif
        const float score = ri.valid ? 0.5f * (sp + sa) * es : -INFINITY;
        const int64_t c = t * kTile + r;  // candidate index
        if (p.scores && c < ncand) p.scores[(int64_t)b * p.score_stride + c] = score;
        if (p.bmax) {
          float m = score;
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          if ((lane & 7) == 0 && c < ncand) p.bmax[(int64_t)b * p.bmax_stride + c / 8] = m;
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (my_tiles > 0 && warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

int choose_ctas_per_query(int64_t tiles, int B, int slots) {
  if (tiles <= 0) return 1;
  int best = 1;
  double best_cost = 1e300;
  const int64_t smax = std::min<int64_t>(tiles, 4096);
  for (int64_t S = 1; S <= smax; ++S) {
    const int64_t ctas = S * B;
    const int64_t waves = cdiv(ctas, slots);
    const double cost = (double)waves * ((double)cdiv(tiles, S) + 6.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = (int)S;
    }
  }
  return best;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// [rows][64] bytes of codes, box of `box_rows` rows, 64-byte swizzle
bool make_code_map(CUtensorMap* map, const uint8_t* codes, int64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {64, (cuuint64_t)rows};
  cuuint64_t strides[1] = {64};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

csa2_status launch_scan(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries, int64_t n_max,
                        int64_t ncand_max, const uint16_t* q, const float* w, const int32_t* pool,
                        int keep, float* scores, int64_t score_stride, float* bmax, int64_t bmax_stride,
                        void* ws, cudaStream_t st) {
  if (ncand_max <= 0) return CSA2_OK;
  const int64_t rows = (int64_t)B * kv->seq_stride;
  if (rows >= ((int64_t)1 << 31)) return CSA2_ERR_UNSUPPORTED;
  CUtensorMap map_tile, map_block;
  if (!make_code_map(&map_tile, kv->ix_codes, rows, kTile) ||
      !make_code_map(&map_block, kv->ix_codes, rows, 8))
    return CSA2_ERR_CUDA;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int smem = (int)sizeof(ScanSmem);
  if (cudaFuncSetAttribute(k_scan_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return CSA2_ERR_CUDA;
  const int64_t tiles = cdiv(ncand_max, kTile);
  const int S = choose_ctas_per_query(tiles, B, 2 * sms);
  ScanParams p{kv->ix_codes, kv->ix_scales, kv->seq_stride, n_entries, n_max, q, w, pool, keep,
               ncand_max, S, scores, score_stride, bmax, bmax_stride, ws};
  k_scan_tc<<<dim3((unsigned)S, (unsigned)B), kThreads, smem, st>>>(p, map_tile, map_block);
  return cudaGetLastError() == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

}  // namespace csa2
