// Lightning-indexer scan on the 5th-generation tensor cores.
//
//   I_j = sum_h w_h ReLU(q_h . K^I_j)   ("DeepSeek-V4: Towards Highly Efficient
//   Million-Token Context Intelligence", CSA step 2; "DeepSeek-V4.1-Flash:
//   pushing the limits of KV cache compression", 4.1 and 4.3)
//
// The indexer keys are MXFP4 (E2M1 codes, one E8M0 scale per 32 elements), a
// format the tensor cores read natively: the block-scaled MMA kind::mxf8f6f4
// multiplies E2M1 codes by E4M3 values and applies one UE8M0 scale per row and
// per 32-element K step of each operand.  The keys are never touched by a
// thread: the tensor-memory-access unit loads each tile of codes with its
// packed 4-bit element type (16 codes per 16-byte slot, 128-byte swizzle),
// which is the shared-memory operand layout of that MMA, and the entries'
// scale bytes go to tensor memory as they are stored.
//
// The bf16 query is split, per head and per 32-element block, into
//   q = 2^s (hi + lo),  hi = E4M3(q 2^-s),  lo = E4M3(q 2^-s - hi),
// with s = floor(log2 max|q_block|) - 7.  For every element of magnitude at
// least 2^-9 of its block maximum this is exact (hi holds the top four
// significant bits, lo the remaining four of bf16's eight); smaller elements
// are off by at most 2^-17 of the block maximum.  The halves are stacked along
// N (rows 0-31 hi, 32-63 lo of each head) in shared memory; per 32-element K
// step one MMA takes the hi rows and a second the lo rows into the same 32
// accumulator columns (both halves have the same scales), so the accumulator
// holds hi + lo and the epilogue reads one column per head.
//
// One CTA streams a contiguous range of 128-entry tiles of one query (or, in
// pool mode, tiles of 16 pool blocks x 8 entries).  Warp roles:
//   warp 0      producer: the tile's codes (one 2-D tensor load, 8 KB) and
//               scale words (one bulk copy, 512 B) into a shared-memory ring;
//   warps 1, 7  MMA issue, even and odd tiles (warp 1 also allocates tensor
//               memory): one thread copies the tile's scales into tensor
//               memory (tcgen05.cp) and issues per K step two MMAs
//               D[128 entries x 32] += A[128 x 32] * B[32 x 32]^T (the hi
//               rows, then the lo rows; one for an MXFP4 query), both
//               operands read from shared memory, into one of three
//               accumulators (tile i -> i mod 3); two issuers and three
//               accumulators keep the tensor core fed while the epilogue
//               drains earlier tiles;
//   warp 2      reorders the tile's 128 scale words into the layout the copy
//               replicates into the four lane quarters of tensor memory;
//   warps 3-6   epilogue: read the row's 32 dots from tensor memory,
//               score = sum_h w_h max(dot_h, 0) (packed
//               f32x2 arithmetic); write the score and/or the max of each
//               8-entry block.
// Every mbarrier wait is bounded; a wait that gives up records
// CSA2_ERR_DEVICE_TIMEOUT and makes every role leave its loop.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "index_scan.cuh"
#include "codec.cuh"
#include "ptx.cuh"
#include "timing.cuh"

namespace csa2 {

namespace {

constexpr int kTile = 128;
#ifndef CSA2_SCAN_STAGES
#define CSA2_SCAN_STAGES 6
#endif
constexpr int kStages = CSA2_SCAN_STAGES;  // shared-memory ring depth (tiles in flight)
constexpr int kAcc = 3;                    // accumulators in tensor memory
constexpr int kWarps = 8;
constexpr int kMmaWarp1 = 7;               // issues the odd tiles
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kCodeBytes = kTile * 64;  // bytes a tile of codes moves from global memory
// Tensor memory columns: accumulators (64 fp32 columns each), then a 4-column
// scale slot per ring stage and a query-scale slot per MMA warp.
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kDCol0 = 0;
constexpr uint32_t kSfaCol0 = 64u * kAcc;
constexpr uint32_t kSfbCol0 = kSfaCol0 + 4u * kStages;
static_assert(kSfbCol0 + 8u <= kTmemCols, "tensor memory layout");
constexpr long long kWaitBudget = 1LL << 32;  // clock cycles (about 2 s)

struct __align__(1024) ScanSmem {
  // codes of a tile: row r at 128 r, its 16-code group g in the 16-byte slot
  // g ^ (r % 8) (first 8 bytes; the other 8 are not written)
  uint8_t codes[kStages][kTile * 128];
  // E4M3 B operand [K step][16-byte K chunk][row][16 B]: rows 0-31 the hi
  // halves of the 32 heads, rows 32-63 the lo halves (K-major core matrices of
  // 8 rows x 16 bytes)
  uint8_t qB[4][2 * 64 * 16];
  uint8_t scales[kStages][kTile * 4];  // scale words of the tile's entries
  uint32_t sfT[kStages][32][4];        // sfT[l][j] = scale word of row 32 j + l
  uint32_t qsfT[32][4];                // query scales: [head][hi, lo, -, -]
  float w[32];
  uint64_t full[kStages], sfull[kStages], sf_ready[kStages], tile_done[kStages];
  uint64_t d_free[kAcc];
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
  int shared_slot;  // >= 0: every query reads this sequence slot (prefill); else query b reads slot b
};

__device__ __forceinline__ void scan_abort(ScanSmem& S, void* ws, int where) {
  *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
  report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, where);
}

// Slot and pass parity in a ring of N slots, stepped without divisions.
template <int N>
struct Ring {
  int slot;
  uint32_t phase;
  __device__ __forceinline__ explicit Ring(int start) : slot(start % N), phase((uint32_t)(start / N) & 1u) {}
  __device__ __forceinline__ void step(int k) {  // k <= N
    slot += k;
    if (slot >= N) {
      slot -= N;
      phase ^= 1u;
    }
  }
};

// packed fp32 pairs (one instruction for two lanes of arithmetic)
__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, z, d;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
      "mov.b64 z, {%6, %7};\n\tfma.rn.f32x2 d, x, y, z;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
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

// Head h of a bf16 query row (128 elements) as its E4M3 halves: lane l holds
// elements 4l..4l+3 (32-element block l / 8, `raw` = the row's bf16 at 4l) and
// gets them packed (element e in byte e), hi and lo, with the block's UE8M0 scale
// byte (the same in the block's eight lanes).  Callers load every row they split
// before splitting the first, so that the loads overlap.
struct QSplit {
  uint32_t hi4, lo4, scale_byte;
};
__device__ __forceinline__ uint2 load_query_lane(const uint16_t* qh, int lane) {
  return *reinterpret_cast<const uint2*>(qh + 4 * lane);
}
__device__ __forceinline__ QSplit split_query(uint2 raw) {
  const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
  const int sb = m > 0.0f ? max(floor_log2_f32(m) - 7, -127) : 0;
  const float inv = exp2i_f32(-sb);
  QSplit r{0u, 0u, (uint32_t)(sb + 127)};
  // pairs of elements through the two-wide conversions (round to nearest even)
#pragma unroll
  for (int e = 0; e < 4; e += 2) {
    const float x0 = v[e] * inv, x1 = v[e + 1] * inv;  // exact: a power-of-two scale, |x| < 256
    uint16_t hi2, lo2;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi2) : "f"(x1), "f"(x0));
    const float2 h = e4m3x2_to_float2(hi2);
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo2) : "f"(x1 - h.y), "f"(x0 - h.x));
    r.hi4 |= (uint32_t)hi2 << (8 * e);
    r.lo4 |= (uint32_t)lo2 << (8 * e);
  }
  return r;
}
// the four blocks' scale bytes of a head as one word (byte = block), in every lane
__device__ __forceinline__ uint32_t scale_word(uint32_t byte) {
  uint32_t word = 0;
#pragma unroll
  for (int blk = 0; blk < 4; ++blk) word |= __shfl_sync(0xffffffffu, byte, 8 * blk) << (8 * blk);
  return word;
}

__global__ void __launch_bounds__(kThreads, 2)
    k_scan_tc(const __grid_constant__ ScanParams p, const __grid_constant__ CUtensorMap map_tile,
              const __grid_constant__ CUtensorMap map_block) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  ScanSmem& S = *reinterpret_cast<ScanSmem*>(smem_raw);
  volatile int* abort_flag = &S.abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int b = blockIdx.y;
  ptx::griddep_wait();  // inputs may come from the previous kernel of the stream

  int64_t n = p.n_entries ? p.n_entries[b] : p.n_max;  // no counts: every slot holds n_max
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
  const int64_t srow = (int64_t)(p.shared_slot >= 0 ? p.shared_slot : b) * p.seq_stride;  // slot's first row
  const bool scale_bulk = (srow & 3) == 0;  // 16-byte aligned scale rows
  const uint8_t* scales_b = p.ix_scales + srow * 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&S.full[s], 1);
      ptx::mbar_init(&S.sfull[s], 1);
      ptx::mbar_init(&S.sf_ready[s], 1);
      ptx::mbar_init(&S.tile_done[s], 1);
    }
    for (int a = 0; a < kAcc; ++a) ptx::mbar_init(&S.d_free[a], 4);
    S.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (my_tiles > 0 && warp == 1) ptx::tmem_alloc(&S.tmem_base, kTmemCols);

  // q^I -> E4M3 halves hi, lo with one E8M0 scale per head and 32-element
  // block; lane l holds elements 4l..4l+3 (block l/8)
  bool lo_nonzero = false;
  uint2 qraw[kHIdx / kWarps];
#pragma unroll
  for (int u = 0; u < kHIdx / kWarps; ++u)
    qraw[u] = load_query_lane(p.q + ((int64_t)b * kHIdx + warp + kWarps * u) * kDIdx, lane);
#pragma unroll
  for (int u = 0; u < kHIdx / kWarps; ++u) {
    const int h = warp + kWarps * u;
    const QSplit qs = split_query(qraw[u]);
    // elements 4l..4l+3: K step l/8, chunk (l/4)%2, bytes 4(l%4)..+3 of row h / 32+h
    const int off = ((lane >> 2) & 1) * 1024 + (h >> 3) * 128 + (h & 7) * 16 + 4 * (lane & 3);
    *reinterpret_cast<uint32_t*>(&S.qB[lane >> 3][off]) = qs.hi4;
    *reinterpret_cast<uint32_t*>(&S.qB[lane >> 3][off + 512]) = qs.lo4;
    lo_nonzero |= qs.lo4 != 0u;
    const uint32_t word = scale_word(qs.scale_byte);
    if (lane == 0) {
      S.qsfT[h][0] = word;
      S.qsfT[h][1] = word;
      S.qsfT[h][2] = 0u;
      S.qsfT[h][3] = 0u;
    }
  }
  if (threadIdx.x < kHIdx) S.w[threadIdx.x] = p.w[(int64_t)b * kHIdx + threadIdx.x];
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  // A query whose every lo half is zero (an MXFP4 query: E2M1 codes under a
  // power-of-two scale fit E4M3 exactly) needs only the hi rows: the MMAs run
  // with N = 32 and the epilogue reads half the columns.
  const bool hi_only = __syncthreads_or(lo_nonzero ? 1 : 0) == 0;
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (my_tiles > 0) {
    if (warp == 0 && pooled) {
      // ------------------------------------------------------------ producer (pool)
      if (lane == 0) {
        Ring<kStages> st(0);
        for (int i = 0; i < my_tiles; ++i, st.step(1)) {
          const int s = st.slot;
          const uint32_t ph = st.phase;
          // stage s is free once the MMAs of tile i - kStages completed
          if (!ptx::mbar_wait(&S.tile_done[s], ph ^ 1u, abort_flag, kWaitBudget)) {
            scan_abort(S, p.ws, 1);
            break;
          }
          const int64_t t = t_begin + i;
          int pbv[16];
          uint32_t cnt[16];
          uint32_t cbytes = 0, sbytes = 0;
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int64_t slot = t * 16 + u;
            pbv[u] = slot < p.keep ? p.pool[(int64_t)b * p.keep + slot] : -1;
            const int64_t base = (int64_t)pbv[u] * 8;
            cnt[u] = (pbv[u] >= 0 && base < n) ? (uint32_t)min((int64_t)8, n - base) : 0u;
            cbytes += cnt[u] ? 8u * 64u : 0u;
            sbytes += scale_bulk ? (cnt[u] & ~3u) * 4u : 0u;
          }
          ptx::mbar_arrive_expect_tx(&S.sfull[s], sbytes);
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const uint32_t c4 = scale_bulk ? (cnt[u] & ~3u) : 0u;
            if (c4) ptx::bulk_g2s(S.scales[s] + u * 32, scales_b + (int64_t)pbv[u] * 8 * 4, c4 * 4u, &S.sfull[s]);
          }
          ptx::mbar_arrive_expect_tx(&S.full[s], cbytes);
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            if (!cnt[u]) continue;
            const int64_t base = (int64_t)pbv[u] * 8;
            ptx::tma_load_2d(S.codes[s] + u * 1024, &map_block, 0, (int)(srow + base), &S.full[s]);
          }
        }
      }
    } else if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        // the keys are read once: keep them from evicting the block maxima and
        // pool the selection kernels read back
        const uint64_t pol = ptx::policy_evict_first();
        Ring<kStages> st(0);
        for (int i = 0; i < my_tiles; ++i, st.step(1)) {
          const int s = st.slot;
          const uint32_t ph = st.phase;
          // stage s is free once the MMAs of tile i - kStages completed
          if (!ptx::mbar_wait(&S.tile_done[s], ph ^ 1u, abort_flag, kWaitBudget)) {
            scan_abort(S, p.ws, 1);
            break;
          }
          const int64_t j0 = (t_begin + i) * kTile;
          const uint32_t cnt = (uint32_t)min((int64_t)kTile, n - j0);
          const uint32_t cnt4 = scale_bulk ? (cnt & ~3u) : 0u;
          // scales first, on their own barrier, so that their reorder overlaps the codes' arrival
          ptx::mbar_arrive_expect_tx(&S.sfull[s], cnt4 * 4u);
          if (cnt4) ptx::bulk_g2s_hint(S.scales[s], scales_b + j0 * 4, cnt4 * 4u, &S.sfull[s], pol);
          ptx::mbar_arrive_expect_tx(&S.full[s], kCodeBytes);
          ptx::tma_load_2d_hint(S.codes[s], &map_tile, 0, (int)(srow + j0), &S.full[s], pol);
        }
      }
    } else if (warp == 1 || warp == kMmaWarp1) {
      // ------------------------------------------------------------ MMA issue
      const int par = warp == 1 ? 0 : 1;  // tile parity this warp issues
      if (lane == 0) {
        uint64_t bd[4];
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) bd[ks] = ptx::smem_desc_noswizzle(S.qB[ks], 1024, 128);
        // query scales, replicated into the four lane quarters; each issuer
        // copies them into its own slot, ordered before its MMAs
        const uint32_t sfb_t = tmem + kSfbCol0 + 4u * (uint32_t)par;
        ptx::tmem_cp_32x128b_warpx4(sfb_t, ptx::smem_desc_noswizzle(S.qsfT, 128, 128));
        // A operand descriptors of stage 0, K step 0; stage s and K step ks add
        // (s * stage bytes + 32 ks) / 16 to the start-address field
        const uint64_t ad0 = ptx::smem_desc_sw128(S.codes[0], 1024);
        Ring<kStages> st(par);
        Ring<kAcc> acc(par);
        for (int i = par; i < my_tiles; i += 2, st.step(2), acc.step(2)) {
          const int s = st.slot;
          const uint32_t ph = st.phase;
          const int a = acc.slot;
          const uint32_t u = acc.phase;
          if (!ptx::mbar_wait(&S.sf_ready[s], ph, abort_flag, kWaitBudget) ||
              !ptx::mbar_wait(&S.full[s], ph, abort_flag, kWaitBudget) ||
              !ptx::mbar_wait(&S.d_free[a], u ^ 1u, abort_flag, kWaitBudget)) {
            scan_abort(S, p.ws, 2);
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sfa_t = tmem + kSfaCol0 + (uint32_t)s * 4u;
          const uint32_t d_t = tmem + kDCol0 + (uint32_t)a * 64u;
          ptx::tmem_cp_32x128b_warpx4(sfa_t, ptx::smem_desc_noswizzle(S.sfT[s], 128, 128));
          const uint64_t ads = ad0 + (uint64_t)(s * (kTile * 128 / 16));
          // per K step: the hi rows (0-31 of the B tile), then the lo rows (32-63, 512 bytes on)
          // into the same 32 columns: hi + lo adds in the accumulator (both halves share
          // their scales)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t idesc = ptx::idesc_block_scaled(128, 32, ptx::kFmtE2M1, ptx::kFmtE4M3, ks, ks);
            ptx::mma_mxf8f6f4_ss(d_t, ads + (uint64_t)(2 * ks), bd[ks], idesc, sfa_t, sfb_t, ks > 0 ? 1u : 0u);
            if (!hi_only)
              ptx::mma_mxf8f6f4_ss(d_t, ads + (uint64_t)(2 * ks), bd[ks] + (uint64_t)(512 / 16), idesc, sfa_t, sfb_t, 1u);
          }
          ptx::mma_commit(&S.tile_done[s]);
        }
      }
    } else if (warp == 2) {
      // ------------------------------------------------------------ scale reorder
      Ring<kStages> st(0);
      for (int i = 0; i < my_tiles; ++i, st.step(1)) {
        const int s = st.slot;
        const uint32_t ph = st.phase;
        if (!ptx::mbar_wait_warp(&S.sfull[s], ph, abort_flag, kWaitBudget)) {
          scan_abort(S, p.ws, 3);
          break;
        }
        const int64_t t = t_begin + i;
        uint32_t w4[4];
        const uint32_t* sc = reinterpret_cast<const uint32_t*>(S.scales[s]);
        if (!pooled && scale_bulk && (t + 1) * kTile <= n) {  // a full tile: every word came in
#pragma unroll
          for (int j = 0; j < 4; ++j) w4[j] = sc[32 * j + lane];
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = 32 * j + lane;
            const RowInfo ri = row_info(p, b, n, t, r, scale_bulk);
            w4[j] = !ri.valid ? 0u
                    : ri.scale_in_smem ? sc[r]
                                       : *reinterpret_cast<const uint32_t*>(scales_b + ri.j * 4);
          }
        }
        *reinterpret_cast<uint4*>(S.sfT[s][lane]) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.sf_ready[s]);
      }
    } else if (warp < kMmaWarp1) {
      // ------------------------------------------------------------ epilogue
      const int sub = warp % 4;  // lane quarter this warp may access
      float wr[32];
#pragma unroll
      for (int h = 0; h < 32; ++h) wr[h] = S.w[h];
      const int r = sub * 32 + lane;
      const uint32_t lane_addr = tmem + ((uint32_t)(sub * 32) << 16);
      float* const score_row = p.scores ? p.scores + (int64_t)b * p.score_stride : nullptr;
      float* const bmax_row = p.bmax ? p.bmax + (int64_t)b * p.bmax_stride : nullptr;
      Ring<kStages> st(0);
      Ring<kAcc> acc(0);
      for (int i = 0; i < my_tiles; ++i, st.step(1), acc.step(1)) {
        const int s = st.slot;
        const uint32_t ph = st.phase;
        const int a = acc.slot;
        if (!ptx::mbar_wait_warp(&S.tile_done[s], ph, abort_flag, kWaitBudget)) {
          scan_abort(S, p.ws, 5);
          break;
        }
        ptx::tc_fence_after();
        // dot_h (hi + lo summed by the MMAs); the accumulator is released as soon as it is read
        uint32_t hi[32];
        const uint32_t d_addr = lane_addr + kDCol0 + (uint32_t)a * 64u;
        ptx::tmem_ld_32x32b_x16(d_addr, hi);
        ptx::tmem_ld_32x32b_x16(d_addr + 16u, hi + 16);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.d_free[a]);
        // sum_h w_h max(dot_h, 0) on head pairs, two accumulators
        float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int h4 = 0; h4 < 8; ++h4) {
          const float4 wv = make_float4(wr[4 * h4], wr[4 * h4 + 1], wr[4 * h4 + 2], wr[4 * h4 + 3]);
          const float2 x01 = make_float2(fmaxf(__uint_as_float(hi[4 * h4]), 0.0f),
                                         fmaxf(__uint_as_float(hi[4 * h4 + 1]), 0.0f));
          const float2 x23 = make_float2(fmaxf(__uint_as_float(hi[4 * h4 + 2]), 0.0f),
                                         fmaxf(__uint_as_float(hi[4 * h4 + 3]), 0.0f));
          acc0 = fma_f32x2(make_float2(wv.x, wv.y), x01, acc0);
          acc1 = fma_f32x2(make_float2(wv.z, wv.w), x23, acc1);
        }
        const float sum = (acc0.x + acc0.y) + (acc1.x + acc1.y);

        const int64_t t = t_begin + i;
        const int64_t c = t * kTile + r;  // candidate index
        const bool full_tile = !pooled && (t + 1) * kTile <= n;
        const bool valid = full_tile || row_info(p, b, n, t, r, scale_bulk).valid;
        const float score = valid ? sum : -INFINITY;
        // evict-first: 4 B per entry that only the pool entries are read back from,
        // which must not push the block maxima (read next) out of L2
        if (score_row && c < ncand) __stcs(score_row + c, score);
        if (bmax_row) {
          float m = score;
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          if ((lane & 7) == 0 && c < ncand) bmax_row[c >> 3] = m;
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

// ---------------------------------------------------------------------------
// Prefill scan.  Every query reads the same sequence slot, so a key tile (L2
// resident) serves kPG queries at once: their E4M3 halves are stacked along N
// (B rows 32 qi + h: hi; 32 kPG + 32 qi + h: lo), and per K step one MMA of the
// hi rows and one of the lo rows (N = 128) cover the four queries, so a tile's
// scale copy and MMAs are issued once for them.  One CTA per SM (the three
// 128-column accumulators take the tensor memory), 16 warps:
//   warp 0      producer (as in k_scan_tc, flat tiles only);
//   warps 1, 3  MMA issue, even and odd tiles, into accumulator i mod 3;
//   warp 2      scale reorder;
//   warps 4-15  three epilogue groups of four warps (one per lane quarter);
//               group g drains accumulator g, i.e. tiles i = g mod 3: per
//               query the row's 32 dots, score = sum_h w_h max(dot_h, 0),
//               written for candidates below that query's visible count.
constexpr int kPG = 4;
constexpr int kPStages = 6;
constexpr int kPTilesPerCta = 128;
constexpr int kPWarps = 16;
constexpr int kPThreads = kPWarps * 32;
constexpr int kPEpi0 = 4;                          // first epilogue warp
constexpr uint32_t kPAccCols = 32u * kPG;          // accumulator columns (32 heads x 4 queries)
constexpr uint32_t kPSfaCol0 = kPAccCols * kAcc;   // then a 4-column scale slot per stage
constexpr uint32_t kPSfbCol0 = kPSfaCol0 + 4u * kPStages;  // then a query-scale slot per MMA warp
constexpr uint32_t kPTmemCols = 512;
static_assert(kPSfbCol0 + 8u <= kPTmemCols, "tensor memory layout");
constexpr int kPMmaWarp1 = 3;  // issues the odd tiles
constexpr uint32_t kPRows = 64u * kPG;  // B rows per K step: 32 kPG hi, then 32 kPG lo

#define PSCAN_ABORT(where)                                           \
  do {                                                               \
    *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;             \
    report_error(p.ws, CSA2_ERR_DEVICE_TIMEOUT, (where));            \
  } while (0)

struct __align__(1024) PScanSmem {
  uint8_t codes[kPStages][kTile * 128];
  // E4M3 B operand [K step][16-byte K chunk][row][16 B]
  uint8_t qB[4][2 * kPRows * 16];
  uint8_t scales[kPStages][kTile * 4];
  uint32_t sfT[kPStages][32][4];
  uint32_t qsfT[32][4];  // query scales: [head][query]
  float w[kPG][32];
  uint64_t full[kPStages], sfull[kPStages], sf_ready[kPStages], tile_done[kPStages];
  uint64_t d_free[kAcc];
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(kPThreads, 1)
    k_scan_prefill(const __grid_constant__ ScanParams p, const __grid_constant__ CUtensorMap map_tile, int nq) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  PScanSmem& S = *reinterpret_cast<PScanSmem*>(smem_raw);
  volatile int* abort_flag = &S.abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // groups in reverse order: the causal bound gives the last queries the most
  // candidates, and the longest CTAs should start first
  const int b0 = (gridDim.y - 1 - blockIdx.y) * kPG;  // this CTA's first query
  ptx::griddep_wait();  // inputs may come from the previous kernel of the stream

  // visible candidates of each query (-1: no query), and of the group (the max)
  int64_t nqv[kPG], n = 0;
#pragma unroll
  for (int qi = 0; qi < kPG; ++qi) {
    int64_t v = -1;
    if (b0 + qi < nq) {
      v = p.n_entries[b0 + qi];
      if (v > p.n_max) {
        if (threadIdx.x == 0 && blockIdx.x == 0) report_error(p.ws, CSA2_ERR_INDEX_RANGE, v);
        v = p.n_max;
      }
      if (v < 0) v = 0;
    }
    nqv[qi] = v;
    n = max(n, v);
  }
  const int64_t ntiles = cdiv(n, kTile);
  const int64_t t_begin = ntiles * blockIdx.x / p.ctas_per_query;
  const int64_t t_end = ntiles * (blockIdx.x + 1) / p.ctas_per_query;
  const int my_tiles = (int)(t_end - t_begin);
  if (my_tiles <= 0) return;  // a short group: fewer tiles than CTAs
  const int64_t srow = (int64_t)p.shared_slot * p.seq_stride;  // the slot's first row
  const bool scale_bulk = (srow & 3) == 0;
  const uint8_t* scales_b = p.ix_scales + srow * 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      ptx::mbar_init(&S.full[s], 1);
      ptx::mbar_init(&S.sfull[s], 1);
      ptx::mbar_init(&S.sf_ready[s], 1);
      ptx::mbar_init(&S.tile_done[s], 1);
    }
    for (int a = 0; a < kAcc; ++a) ptx::mbar_init(&S.d_free[a], 4);
    S.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) ptx::tmem_alloc(&S.tmem_base, kPTmemCols);

  // the queries' E4M3 halves: warp w takes (query, head) pairs w, w + 16, ...
  bool lo_nonzero = false;
  constexpr int kPerWarp = kPG * kHIdx / kPWarps;
  uint2 qraw[kPerWarp];
#pragma unroll
  for (int v = 0; v < kPerWarp; ++v) {
    const int u = warp + kPWarps * v, qi = u / kHIdx, h = u % kHIdx;
    qraw[v] = b0 + qi < nq ? load_query_lane(p.q + ((int64_t)(b0 + qi) * kHIdx + h) * kDIdx, lane)
                           : make_uint2(0u, 0u);
  }
#pragma unroll
  for (int v = 0; v < kPerWarp; ++v) {
    const int u = warp + kPWarps * v, qi = u / kHIdx, h = u % kHIdx;
    const QSplit qs = split_query(qraw[v]);  // a missing query: zeros
    const int row = 32 * qi + h;
    const int off = ((lane >> 2) & 1) * (int)(kPRows * 16) + (row >> 3) * 128 + (row & 7) * 16 + 4 * (lane & 3);
    *reinterpret_cast<uint32_t*>(&S.qB[lane >> 3][off]) = qs.hi4;
    *reinterpret_cast<uint32_t*>(&S.qB[lane >> 3][off + 32 * kPG * 16]) = qs.lo4;
    lo_nonzero |= qs.lo4 != 0u;
    const uint32_t word = scale_word(qs.scale_byte);
    if (lane == 0) S.qsfT[h][qi] = word;
  }
  if (threadIdx.x < kPG * kHIdx) {
    const int qi = threadIdx.x / kHIdx;
    S.w[qi][threadIdx.x % kHIdx] = b0 + qi < nq ? p.w[(int64_t)(b0 + qi) * kHIdx + threadIdx.x % kHIdx] : 0.0f;
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  // queries whose every lo half is zero (MXFP4 queries) need only the hi rows
  const bool hi_only = __syncthreads_or(lo_nonzero ? 1 : 0) == 0;
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (my_tiles > 0) {
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        Ring<kPStages> st(0);
        for (int i = 0; i < my_tiles; ++i, st.step(1)) {
          const int s = st.slot;
          const uint32_t ph = st.phase;
          if (!ptx::mbar_wait(&S.tile_done[s], ph ^ 1u, abort_flag, kWaitBudget)) {
            PSCAN_ABORT(1);
            break;
          }
          const int64_t j0 = (t_begin + i) * kTile;
          const uint32_t cnt = (uint32_t)min((int64_t)kTile, n - j0);
          const uint32_t cnt4 = scale_bulk ? (cnt & ~3u) : 0u;
          ptx::mbar_arrive_expect_tx(&S.sfull[s], cnt4 * 4u);
          if (cnt4) ptx::bulk_g2s(S.scales[s], scales_b + j0 * 4, cnt4 * 4u, &S.sfull[s]);
          ptx::mbar_arrive_expect_tx(&S.full[s], kCodeBytes);
          ptx::tma_load_2d(S.codes[s], &map_tile, 0, (int)(srow + j0), &S.full[s]);
        }
      }
    } else if (warp == 1 || warp == kPMmaWarp1) {
      // ------------------------------------------------------------ MMA issue
      // warp 1 the even tiles, warp 3 the odd ones; each warp runs its loop together
      // (uniform waits and descriptors) and one elected lane issues each copy, MMA and commit
      const int par = warp == 1 ? 0 : 1;
      uint64_t bd[4];
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) bd[ks] = ptx::smem_desc_noswizzle(S.qB[ks], kPRows * 16, 128);
      // the query scales in this warp's own slot, ordered before its MMAs
      const uint32_t sfb_t = tmem + kPSfbCol0 + 4u * (uint32_t)par;
      ptx::tmem_cp_32x128b_warpx4_elect(sfb_t, ptx::smem_desc_noswizzle(S.qsfT, 128, 128));
      const uint64_t ad0 = ptx::smem_desc_sw128(S.codes[0], 1024);
      Ring<kPStages> st(par);
      Ring<kAcc> acc(par);
      for (int i = par; i < my_tiles; i += 2, st.step(2), acc.step(2)) {
        const int s = st.slot;
        const uint32_t ph = st.phase;
        const int a = acc.slot;
        const uint32_t u = acc.phase;
        if (!ptx::mbar_wait_warp(&S.sf_ready[s], ph, abort_flag, kWaitBudget) ||
            !ptx::mbar_wait_warp(&S.full[s], ph, abort_flag, kWaitBudget) ||
            !ptx::mbar_wait_warp(&S.d_free[a], u ^ 1u, abort_flag, kWaitBudget)) {
          if (lane == 0) PSCAN_ABORT(2);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sfa_t = tmem + kPSfaCol0 + (uint32_t)s * 4u;
        const uint32_t d_t = tmem + (uint32_t)a * kPAccCols;
        ptx::tmem_cp_32x128b_warpx4_elect(sfa_t, ptx::smem_desc_noswizzle(S.sfT[s], 128, 128));
        const uint64_t ads = ad0 + (uint64_t)(s * (kTile * 128 / 16));
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint32_t idesc = ptx::idesc_block_scaled(128, 32 * kPG, ptx::kFmtE2M1, ptx::kFmtE4M3, ks, ks);
          ptx::mma_mxf8f6f4_ss_elect(d_t, ads + (uint64_t)(2 * ks), bd[ks], idesc, sfa_t, sfb_t, ks > 0 ? 1u : 0u);
          if (!hi_only)
            ptx::mma_mxf8f6f4_ss_elect(d_t, ads + (uint64_t)(2 * ks), bd[ks] + (uint64_t)(32 * kPG * 16 / 16), idesc,
                                       sfa_t, sfb_t, 1u);
        }
        ptx::mma_commit_elect(&S.tile_done[s]);
      }
    } else if (warp == 2) {
      // ------------------------------------------------------------ scale reorder
      Ring<kPStages> st(0);
      for (int i = 0; i < my_tiles; ++i, st.step(1)) {
        const int s = st.slot;
        const uint32_t ph = st.phase;
        if (!ptx::mbar_wait_warp(&S.sfull[s], ph, abort_flag, kWaitBudget)) {
          PSCAN_ABORT(3);
          break;
        }
        const int64_t t = t_begin + i;
        uint32_t w4[4];
        const uint32_t* sc = reinterpret_cast<const uint32_t*>(S.scales[s]);
        if (scale_bulk && (t + 1) * kTile <= n) {
#pragma unroll
          for (int j = 0; j < 4; ++j) w4[j] = sc[32 * j + lane];
        } else {
          const int64_t j0 = t * kTile;
          const int64_t cnt = min((int64_t)kTile, n - j0);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = 32 * j + lane;
            w4[j] = r >= cnt ? 0u
                    : (scale_bulk && r < (cnt & ~3LL)) ? sc[r]
                                                        : *reinterpret_cast<const uint32_t*>(scales_b + (j0 + r) * 4);
          }
        }
        *reinterpret_cast<uint4*>(S.sfT[s][lane]) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.sf_ready[s]);
      }
    } else if (warp >= kPEpi0) {
      // ------------------------------------------------------------ epilogue
      const int g = (warp - kPEpi0) / 4;  // group: accumulator g, tiles i = g mod 3
      const int sub = warp % 4;           // lane quarter this warp may access
      const int r = sub * 32 + lane;
      const uint32_t lane_addr = tmem + ((uint32_t)(sub * 32) << 16) + (uint32_t)g * kPAccCols;
      Ring<kPStages> st(g);
      for (int i = g; i < my_tiles; i += kAcc, st.step(kAcc)) {
        const int s = st.slot;
        const uint32_t ph = st.phase;
        if (!ptx::mbar_wait_warp(&S.tile_done[s], ph, abort_flag, kWaitBudget)) {
          PSCAN_ABORT(5);
          break;
        }
        ptx::tc_fence_after();
        const int64_t c = (t_begin + i) * kTile + r;  // candidate index
        // query qi's 32 dots at columns 32 qi ..: queries 0 and 1 read together, then 2 into
        // the first buffer while query 1 is summed and 3 into the second; the accumulator is
        // released once the last read lands, before the last two sums
        uint32_t da[32], db[32];
        float bm[kPG];  // this entry's visible score per query (-inf if not visible), for the block maxima
        auto score = [&](int qi, const uint32_t (&d)[32]) {
          float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
          const float4* wq = reinterpret_cast<const float4*>(S.w[qi]);
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 wv = wq[h4];
            const float2 x01 = make_float2(fmaxf(__uint_as_float(d[4 * h4]), 0.0f),
                                           fmaxf(__uint_as_float(d[4 * h4 + 1]), 0.0f));
            const float2 x23 = make_float2(fmaxf(__uint_as_float(d[4 * h4 + 2]), 0.0f),
                                           fmaxf(__uint_as_float(d[4 * h4 + 3]), 0.0f));
            acc0 = fma_f32x2(make_float2(wv.x, wv.y), x01, acc0);
            acc1 = fma_f32x2(make_float2(wv.z, wv.w), x23, acc1);
          }
          const float sum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
          const bool vis = c < nqv[qi];
          if (vis) __stcs(p.scores + (int64_t)(b0 + qi) * p.score_stride + c, sum);
          bm[qi] = vis ? sum : -INFINITY;
        };
        static_assert(kPG == 4, "the epilogue reads the queries in pairs");
        ptx::tmem_ld_32x32b_x32(lane_addr, da);
        ptx::tmem_ld_32x32b_x32(lane_addr + 32u, db);
        ptx::tmem_wait_ld();
        score(0, da);
        ptx::tmem_ld_32x32b_x32(lane_addr + 64u, da);
        score(1, db);
        ptx::tmem_ld_32x32b_x32(lane_addr + 96u, db);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.d_free[g]);  // every column read: the accumulator is free
        score(2, da);
        score(3, db);
        if (p.bmax) {  // maxima of the 8-entry blocks (lanes 8 j .. 8 j + 7 hold one), the four queries interleaved
#pragma unroll
          for (int o = 1; o < 8; o <<= 1)
#pragma unroll
            for (int qi = 0; qi < kPG; ++qi) bm[qi] = fmaxf(bm[qi], __shfl_xor_sync(0xffffffffu, bm[qi], o));
          if ((lane & 7) == 0) {
#pragma unroll
            for (int qi = 0; qi < kPG; ++qi)
              if (c < nqv[qi]) p.bmax[(int64_t)(b0 + qi) * p.bmax_stride + c / 8] = bm[qi];
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kPTmemCols);
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

// [rows][64] bytes of codes as [rows][128] packed 4-bit elements, box of
// `box_rows` rows; shared memory gets 16 codes per 16-byte slot, 128-byte swizzle
bool make_code_map(CUtensorMap* map, const uint8_t* codes, int64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {64};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<uint8_t*>(codes), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

csa2_status launch_scan(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries, int64_t n_max,
                        int64_t ncand_max, const uint16_t* q, const float* w, const int32_t* pool,
                        int keep, float* scores, int64_t score_stride, float* bmax, int64_t bmax_stride,
                        void* ws, cudaStream_t st, int shared_slot) {
  if (ncand_max <= 0) return CSA2_OK;
  const int64_t rows = (int64_t)(shared_slot >= 0 ? shared_slot + 1 : B) * kv->seq_stride;
  if (rows >= ((int64_t)1 << 31)) return CSA2_ERR_UNSUPPORTED;
  if (!aligned(kv->ix_codes, 32)) return CSA2_ERR_INVALID_ARG;  // packed 4-bit tensor loads
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
               ncand_max, S, scores, score_stride, bmax, bmax_stride, ws, shared_slot};
  KernelTimer timer("k_scan_tc", st);
  launch_pdl(k_scan_tc, dim3((unsigned)S, (unsigned)B), dim3(kThreads), (size_t)smem, st, p, map_tile, map_block);
  return cudaGetLastError() == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

csa2_status launch_scan_prefill(const csa2_kv_planes* kv, int32_t Q, const int32_t* n_visible, int64_t n_max,
                                const uint16_t* q, const float* w, float* scores, int64_t score_stride, float* bmax,
                                int64_t bmax_stride, void* ws, cudaStream_t st, int slot) {
  if (n_max <= 0) return CSA2_OK;
  const int64_t rows = (int64_t)(slot + 1) * kv->seq_stride;
  if (rows >= ((int64_t)1 << 31)) return CSA2_ERR_UNSUPPORTED;
  if (!aligned(kv->ix_codes, 32)) return CSA2_ERR_INVALID_ARG;  // packed 4-bit tensor loads
  CUtensorMap map_tile;
  if (!make_code_map(&map_tile, kv->ix_codes, rows, kTile)) return CSA2_ERR_CUDA;
  const int smem = (int)sizeof(PScanSmem);
  if (cudaFuncSetAttribute(k_scan_prefill, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return CSA2_ERR_CUDA;
  // up to kPTilesPerCta tiles per CTA: the groups' candidate counts differ (causal), and
  // short CTAs let the GPU even out the work
  const int groups = (int)cdiv(Q, kPG);
  const int S = (int)std::max<int64_t>(1, cdiv(cdiv(n_max, kTile), kPTilesPerCta));
  ScanParams p{kv->ix_codes, kv->ix_scales, kv->seq_stride, n_visible, n_max, q, w, nullptr, 0,
               n_max, S, scores, score_stride, bmax, bmax_stride, ws, slot};
  KernelTimer timer("k_scan_prefill", st);
  launch_pdl(k_scan_prefill, dim3((unsigned)S, (unsigned)groups), dim3(kPThreads), (size_t)smem, st, p, map_tile,
             (int)Q);
  return cudaGetLastError() == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}

}  // namespace csa2
