// Prefill cache write: C = H W_KV, Z = H W_Z ("DeepSeek-V4.1-Flash course, 02
// Architecture", 2.2 Eq. (1)), per-channel softmax pooling of each group of m
// tokens and the indexer key K^I = Cbar W_IK ("DeepSeek-V4.1-Flash: pushing the
// limits of KV cache compression", 4.1), then the cache codec (section 5).
//
// The projection runs on the 5th-generation tensor cores (k_cw_tc): a
// persistent bf16 GEMM whose 128-token x 256-column tiles hold C and Z of the
// same 128 channels, so that the epilogue can pool them without another pass.
// H is the K-major A operand; the weights are read as given ([d][512], N
// contiguous) as an N-major B operand: four 64-column tensor loads per stage
// (two of W_KV, two of W_Z), 128-byte swizzle.  Warp roles: warp 0 loads the A
// (16 KB) and B (32 KB) tiles of each 64-wide K step with TMA into a 4-stage
// ring; warp 1 allocates tensor memory and issues 4 MMAs (M128 N256 K16,
// kind::f16, bf16 operands, fp32 accumulate) per stage into one of two
// 256-column accumulators; warps 2-5 read the finished accumulator (thread =
// token), pool each group of m adjacent tokens with a max-subtracted
// per-channel softmax through lane shuffles, and write Cbar (fp32).  K^I =
// Cbar W_IK follows on the tensor cores with every product exact (k_cw_ki_tc:
// Cbar split into three bf16 terms), then the codec.  A group of 64 tokens
// spans two lane quarters; m = 64 keeps the CUDA-core kernel k_cw_gemm_pool,
// which computes the same quantities.  Few tokens (a decode-time append) split
// the K range over the SMs instead (k_cw_finish_small sums the slices, pools,
// forms K^I and writes the entries).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "codec.cuh"
#include "index_scan.cuh"
#include "ptx.cuh"
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

// ------------------------------------------------------------ tensor-core path
constexpr int kTcM = 128;         // tokens per tile
constexpr int kTcN = 256;         // C and Z columns of 128 channels
constexpr int kTcBK = 64;         // K elements per stage (one 128-byte swizzle row)
constexpr int kTcStages = 4;
constexpr int kFillSms = 148;     // SMs the split plan fills (a shape-only constant)
constexpr int kTcThreads = 192;   // producer, MMA, 4 epilogue warps
constexpr uint32_t kTcTmemCols = 512;
constexpr long long kTcWaitBudget = 1LL << 32;

struct __align__(1024) TcSmem {
  uint8_t A[kTcStages][kTcM * 128];  // H tile, K-major, 128-byte swizzle
  // W tile, N-major: four 64-column blocks (W_KV 128 j .. + 127, then W_Z's), each
  // 64 K rows of 128 bytes with 128-byte swizzle, as the tensor loads write them
  uint8_t B[kTcStages][kTcN * 128];
  uint64_t full[kTcStages], empty[kTcStages];
  uint64_t acc_full[2], acc_free[2];
  uint32_t tmem_base;
  int abort_flag;
};

// Long inputs read the weights K-major from a per-call transposed copy
// Wt[channel block j][C rows | Z rows][d] (measured faster than the N-major
// reads once the transpose is spread over many token tiles): 64 x 64 tiles
// through shared memory, 16-byte global accesses on both sides.
constexpr int kWtTile = 64;
constexpr int64_t kDirectMaxT = 65536;  // tokens up to which W is read N-major as given
__global__ void __launch_bounds__(256) k_cw_wt(const uint16_t* __restrict__ Wkv,
                                               const uint16_t* __restrict__ Wz, int d,
                                               uint16_t* __restrict__ Wt) {
  __shared__ __align__(16) uint16_t tile[kWtTile][kWtTile + 8];  // [k][column], rows padded by 16 bytes
  const int k0 = blockIdx.x * kWtTile;    // K rows of W
  const int row0 = blockIdx.y * kWtTile;  // Wt rows (0 .. 1023)
  const int j = row0 / 256, rr = row0 % 256;
  const uint16_t* src = rr < 128 ? Wkv : Wz;
  const int c0 = 128 * j + (rr % 128);
  for (int i = threadIdx.x; i < kWtTile * 8; i += 256) {  // row i / 8, 8 columns from 8 (i % 8)
    const int r = i / 8, ch = i % 8;
    *reinterpret_cast<uint4*>(&tile[r][ch * 8]) =
        *reinterpret_cast<const uint4*>(src + (int64_t)(k0 + r) * kDMain + c0 + ch * 8);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kWtTile * 8; i += 256) {  // Wt row row0 + i % 64, K chunk i / 64
    const int nn = i % kWtTile, kc = i / kWtTile;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w[q] = (uint32_t)tile[kc * 8 + 2 * q][nn] | ((uint32_t)tile[kc * 8 + 2 * q + 1][nn] << 16);
    *reinterpret_cast<uint4*>(Wt + (int64_t)(row0 + nn) * d + k0 + kc * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__device__ __forceinline__ void tc_abort(TcSmem& S, void* ws, int where) {
  *reinterpret_cast<volatile int*>(&S.abort_flag) = 1;
  report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, where);
}

// kNMajorW: B tiles come N-major from W_KV and W_Z as given (map_wkv, map_wz);
// otherwise K-major from the transposed copy (map_wkv holds Wt, map_wz unused).
template <bool kNMajorW>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_cw_tc(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_wkv,
            const __grid_constant__ CUtensorMap map_wz, int64_t T,
            int d, int m, int width, float* __restrict__ cbar, float* __restrict__ zout, int ksplit,
            float* __restrict__ part, void* ws) {
  extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
  TcSmem& S = *reinterpret_cast<TcSmem*>(tc_smem_raw);
  volatile int* abort_flag = &S.abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t token_tiles = cdiv(T, kTcM);
  const int nblk = width / 128;  // 128-channel blocks of the output (C and Z of the same channels per tile)
  const int64_t ntiles = token_tiles * nblk;
  const int nk = d / kTcBK;
  // work item = (tile, K slice): with ksplit > 1 each item sums K steps
  // [ks nk / ksplit, (ks + 1) nk / ksplit) and writes raw partial C and Z to part
  const int64_t nitems = ntiles * ksplit;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      ptx::mbar_init(&S.full[s], 1);
      ptx::mbar_init(&S.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&S.acc_full[a], 1);
      ptx::mbar_init(&S.acc_free[a], 4);
    }
    S.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) ptx::tmem_alloc(&S.tmem_base, kTcTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      for (int64_t item = blockIdx.x; item < nitems; item += gridDim.x) {
        const int64_t tile = item / ksplit;
        const int ks = (int)(item % ksplit);
        const int t0 = (int)((tile / nblk) * kTcM), j = (int)(tile % nblk);
        for (int kb = ks * nk / ksplit; kb < (ks + 1) * nk / ksplit; ++kb) {
          if (!ptx::mbar_wait(&S.empty[s], ph ^ 1u, abort_flag, kTcWaitBudget)) {
            tc_abort(S, ws, 31);
            goto producer_done;
          }
          ptx::mbar_arrive_expect_tx(&S.full[s], (kTcM + kTcN) * 128);
          ptx::tma_load_2d(S.A[s], &map_h, kb * kTcBK, t0, &S.full[s]);
          if (kNMajorW) {
            ptx::tma_load_2d(S.B[s], &map_wkv, 128 * j, kb * kTcBK, &S.full[s]);
            ptx::tma_load_2d(S.B[s] + 8192, &map_wkv, 128 * j + 64, kb * kTcBK, &S.full[s]);
            ptx::tma_load_2d(S.B[s] + 16384, &map_wz, 128 * j, kb * kTcBK, &S.full[s]);
            ptx::tma_load_2d(S.B[s] + 24576, &map_wz, 128 * j + 64, kb * kTcBK, &S.full[s]);
          } else {
            ptx::tma_load_2d(S.B[s], &map_wkv, kb * kTcBK, j * kTcN, &S.full[s]);
          }
          if (++s == kTcStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
  producer_done:;
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_f16(kTcM, kTcN, 1) | (kNMajorW ? ptx::kIdescBMajorMN : 0u);
      int s = 0, local = 0;
      uint32_t ph = 0;
      for (int64_t item = blockIdx.x; item < nitems; item += gridDim.x, ++local) {
        const int ks = (int)(item % ksplit);
        const int kb0 = ks * nk / ksplit, kb1 = (ks + 1) * nk / ksplit;
        const int a = local & 1;
        const uint32_t u = (uint32_t)(local >> 1) & 1u;
        if (!ptx::mbar_wait(&S.acc_free[a], u ^ 1u, abort_flag, kTcWaitBudget)) {
          tc_abort(S, ws, 32);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_t = tmem + (uint32_t)a * kTcN;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait(&S.full[s], ph, abort_flag, kTcWaitBudget)) {
            tc_abort(S, ws, 33);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t ad = ptx::smem_desc_sw128(S.A[s], 1024);
          const uint64_t bd =
              kNMajorW ? ptx::smem_desc_sw128_mn(S.B[s], 8192, 1024) : ptx::smem_desc_sw128(S.B[s], 1024);
          // K step: 32 bytes of an A row; of B 16 rows (2 KB) N-major, 32 bytes of a row K-major
          constexpr uint64_t kBStep = kNMajorW ? 128 : 2;
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk)
            ptx::mma_f16_ss(d_t, ad + (uint64_t)(2 * kk), bd + kBStep * kk, idesc, (kb != kb0 || kk) ? 1u : 0u);
          ptx::mma_commit(&S.empty[s]);  // the stage is free once these MMAs have read it
          if (++s == kTcStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&S.acc_full[a]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int sub = warp % 4;  // lane quarter: tokens 32 sub .. 32 sub + 31 of the tile
    const uint32_t lane_addr = tmem + ((uint32_t)(sub * 32) << 16);
    const int64_t n = T / m;
    int local = 0;
    for (int64_t item = blockIdx.x; item < nitems; item += gridDim.x, ++local) {
      const int64_t tile = item / ksplit;
      const int ks = (int)(item % ksplit);
      const int a = local & 1;
      const uint32_t u = (uint32_t)(local >> 1) & 1u;
      if (!ptx::mbar_wait_warp(&S.acc_full[a], u, abort_flag, kTcWaitBudget)) {
        tc_abort(S, ws, 34);
        break;
      }
      ptx::tc_fence_after();
      const int64_t t = (tile / nblk) * kTcM + sub * 32 + lane;  // this thread's token
      const int ch0 = (int)(tile % nblk) * 128;
      const int64_t e = t / m;                               // its entry
      const bool writer = (lane % m) == 0 && e < n;           // first token of its group
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t cr[32], zr[32];
        const uint32_t base = lane_addr + (uint32_t)a * kTcN + (uint32_t)cb * 32u;
        ptx::tmem_ld_32x32b_x32(base, cr);
        ptx::tmem_ld_32x32b_x32(base + 128u, zr);
        ptx::tmem_wait_ld();
        if (part) {  // K slice ks of token t: raw C then Z, [ks][t][C 512 | Z 512]
          if (t < T) {
            float4* pc = reinterpret_cast<float4*>(part + ((int64_t)ks * T + t) * (2 * kDMain) + ch0 + cb * 32);
            float4* pz = pc + kDMain / 4;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              pc[q] = make_float4(__uint_as_float(cr[4 * q]), __uint_as_float(cr[4 * q + 1]),
                                  __uint_as_float(cr[4 * q + 2]), __uint_as_float(cr[4 * q + 3]));
              pz[q] = make_float4(__uint_as_float(zr[4 * q]), __uint_as_float(zr[4 * q + 1]),
                                  __uint_as_float(zr[4 * q + 2]), __uint_as_float(zr[4 * q + 3]));
            }
          }
          continue;
        }
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float cv = __uint_as_float(cr[c]), zv = __uint_as_float(zr[c]);
          if (m == 1) {
            v[c] = cv;  // the softmax over one token is exactly 1
          } else {
            float zmax = zv;
            for (int o = 1; o < m; o <<= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
            const float ez = expf(zv - zmax);
            float num = ez * cv, den = ez;
            for (int o = 1; o < m; o <<= 1) {
              num += __shfl_xor_sync(0xffffffffu, num, o);
              den += __shfl_xor_sync(0xffffffffu, den, o);
            }
            v[c] = __fdiv_rn(num, den);
          }
        }
        if (writer) {
          float4* dst = reinterpret_cast<float4*>(cbar + e * width + ch0 + cb * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          if (zout) {  // unpooled projections (m = 1): Z next to C
            float4* zd = reinterpret_cast<float4*>(zout + e * width + ch0 + cb * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              zd[q] = make_float4(__uint_as_float(zr[4 * q]), __uint_as_float(zr[4 * q + 1]),
                                  __uint_as_float(zr[4 * q + 2]), __uint_as_float(zr[4 * q + 3]));
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&S.acc_free[a]);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTcTmemCols);
  }
}

// K^I = Cbar W_IK on the tensor cores, exactly in every product: each fp32
// Cbar value splits into three bf16 terms, hi = its top 8 significant bits
// (truncated), mid = the next 8 of the remainder, lo = the rest (at most 8
// bits), so Cbar = hi + mid + lo exactly, and W_IK is bf16 already.  The three
// terms are three MMA sets into one fp32 accumulator; only the order of the
// fp32 additions differs from a sequential sum.  Persistent: one CTA per SM
// keeps all of W_IK in shared memory as the MMA's N-major B operand (tensor-loaded
// as given, [512 channels][128 outputs], 64-output blocks with 128-byte swizzle)
// and runs tiles of 128 entries, 64 channels (a chunk) at a time:
//   warp 17    tensor-loads each chunk of Cbar (fp32, two 32-channel boxes,
//              128-byte swizzle) into a three-stage ring;
//   warps 0-15 thread = (entry row, 16-channel quarter): read the row's quarter
//              from the ring, split it, and store the three bf16 terms as the
//              MMA's A operand in tensor memory (row m at lane m, two bf16 per
//              column; two buffers), so the operand never passes through shared
//              memory; warps 0-3 also read each finished tile's K^I out;
//   warp 16    issues 3 x 4 MMAs (M128 N128 K16, A from tensor memory, W from
//              shared memory) per chunk into one of two accumulators, so a
//              tile's K^I is read out while the next tile's chunks run.
// The codec runs here too: the read-out quantizes each K^I row (four MXFP4
// groups of 32) straight into the indexer-key planes, and, when the main KV
// takes neither RMSNorm nor RoPE, the split warps quantize each 16-channel group
// of Cbar they read (E2M1 x E4M3) into the main-KV planes, so Cbar is read once.
// Sixteen split warps (four per scheduler) hide the latency of that arithmetic.
struct KtOut {
  float* ki;                    // fp32 K^I [n][128], or null
  uint8_t *ix_codes, *ix_scales;  // indexer-key planes, or null
  uint8_t *kv_codes, *kv_scales;  // main-KV planes (plain codec), or null
  QDest d;
};
constexpr int kKtStreamWarps = 16;
constexpr int kKtMmaWarp = 16;
constexpr int kKtLoadWarp = 17;
constexpr int kKtThreads = 18 * 32;
// five warps share two of the schedulers, whose 16 K registers then allow 102 per thread: the
// bound below makes the compiler keep to that
constexpr int kKtBoundThreads = 20 * 32;
constexpr int kKtStages = 3;
constexpr uint32_t kKtAcol = 256;  // A operand buffer u: columns 256 + 128 u (term t: + 32 t)
constexpr long long kKtWaitBudget = 1LL << 32;

struct __align__(1024) KtSmem {
  uint8_t B[8][128 * 128];                 // W_IK chunk j: channels 64 j .. + 63, outputs 0-63 | 64-127
  float X[kKtStages][2][128 * 32];         // Cbar chunk: [half][row][32 channels], 128-byte swizzle
  uint64_t b_full, x_full[kKtStages], x_free[kKtStages], a_full[2], a_free[2], done[2], acc_free[2], drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Splits 16 fp32 values into the hi / mid / lo bf16 terms, packed in pairs
// (element 2c in the low half of word c).
__device__ __forceinline__ void kt_split(const float (&x)[16], uint32_t (&t3)[3][8]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint32_t h[2], md[2], lw[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float v = x[2 * q + u];
      const uint32_t hb = __float_as_uint(v) & 0xFFFF0000u;  // top 8 significant bits
      const float r1 = v - __uint_as_float(hb);               // exact
      const uint32_t mb = __float_as_uint(r1) & 0xFFFF0000u;
      const float r2 = r1 - __uint_as_float(mb);              // exact, <= 8 bits left
      h[u] = hb >> 16;
      md[u] = mb >> 16;
      lw[u] = __float_as_uint(r2) >> 16;                      // exact: low half is zero
    }
    t3[0][q] = h[0] | (h[1] << 16);
    t3[1][q] = md[0] | (md[1] << 16);
    t3[2][q] = lw[0] | (lw[1] << 16);
  }
}

// K^I rows of a finished tile (accumulator `acc`): warps 0-3, thread = entry row
__device__ __forceinline__ bool kt_epilogue(KtSmem& S, uint32_t tmem, int acc, uint32_t par, int64_t e0, int64_t n,
                                            const KtOut& o, int warp, int lane, volatile int* abort_flag, void* ws) {
  const bool landed = ptx::mbar_wait_warp(&S.done[acc], par, abort_flag, kKtWaitBudget);
  if (!landed) {
    if (lane == 0) report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 42);
    return false;
  }
  ptx::tc_fence_after();
  const int64_t e = e0 + warp * 32 + lane;
  const int64_t row = e < n && o.ix_codes ? dest_row(o.d, e) : -1;  // plane row of the entry
  float4* dst = reinterpret_cast<float4*>(o.ki + e * kDIdx);
#pragma unroll 1
  for (int cb = 0; cb < 4; ++cb) {
    uint32_t v[32];
    ptx::tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)acc * 128u + (uint32_t)cb * 32u, v);
    ptx::tmem_wait_ld();
    if (e < n && o.ki) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dst[8 * cb + q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                      __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
    }
    if (row >= 0) {  // MXFP4 group cb of the indexer key
      float g[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) g[i] = __uint_as_float(v[i]);
      quantize_index_group_vals(g, o.ix_codes + row * 64 + cb * 16, o.ix_scales + row * 4 + cb);
    }
  }
  ptx::tc_fence_before();
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(&S.acc_free[acc]);  // the accumulator may take the tile after next
  return true;
}

__global__ void __launch_bounds__(kKtBoundThreads, 1)
    k_cw_ki_tc(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_cbar, int64_t n,
               const __grid_constant__ KtOut o, void* ws) {
  extern __shared__ __align__(1024) unsigned char kt_smem_raw[];
  KtSmem& S = *reinterpret_cast<KtSmem*>(kt_smem_raw);
  volatile int* abort_flag = &S.abort_flag;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int64_t ntiles = cdiv(n, (int64_t)128);
  const int my = (int)((ntiles - (int64_t)blockIdx.x + gridDim.x - 1) / gridDim.x);  // this CTA's tiles
  const int nch = 8 * my;                                                            // its chunks
  auto tile_e0 = [&](int k) { return ((int64_t)blockIdx.x + (int64_t)k * gridDim.x) * 128; };
  if (tid == 0) {
    ptx::mbar_init(&S.b_full, 1);
    for (int i = 0; i < kKtStages; ++i) {
      ptx::mbar_init(&S.x_full[i], 1);
      ptx::mbar_init(&S.x_free[i], kKtStreamWarps);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&S.a_full[i], kKtStreamWarps);
      ptx::mbar_init(&S.a_free[i], 1);
      ptx::mbar_init(&S.done[i], 1);
      ptx::mbar_init(&S.acc_free[i], 4);  // the four read-out warps
    }
    ptx::mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) ptx::tmem_alloc(&S.tmem_base, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  bool good = true;

  if (warp == kKtLoadWarp) {
    // ------------------------------------------------------------ Cbar loads
    if (lane == 0 && my > 0) {
      ptx::mbar_arrive_expect_tx(&S.b_full, 8 * 128 * 128);
      for (int j = 0; j < 8; ++j) {  // two 64-output blocks of 64 channel rows each
        ptx::tma_load_2d(S.B[j], &map_w, 0, 64 * j, &S.b_full);
        ptx::tma_load_2d(S.B[j] + 8192, &map_w, 64, 64 * j, &S.b_full);
      }
      const uint64_t pol = ptx::policy_evict_first();  // Cbar is read once
      int s = 0;
      uint32_t ph = 0;
      for (int g = 0; g < nch; ++g) {
        if (g >= kKtStages && !ptx::mbar_wait(&S.x_free[s], ph ^ 1u, abort_flag, kKtWaitBudget)) {
          good = false;
          break;
        }
        const int j = g & 7;
        const int e0 = (int)tile_e0(g >> 3);
        ptx::mbar_arrive_expect_tx(&S.x_full[s], 2 * 128 * 32 * 4);
        ptx::tma_load_2d_hint(S.X[s][0], &map_cbar, 64 * j, e0, &S.x_full[s], pol);
        ptx::tma_load_2d_hint(S.X[s][1], &map_cbar, 64 * j + 32, e0, &S.x_full[s], pol);
        if (++s == kKtStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == kKtMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    good = my <= 0 || ptx::mbar_wait_warp(&S.b_full, 0, abort_flag, kKtWaitBudget);
    constexpr uint32_t idesc = ptx::idesc_f16(128, 128, 1) | ptx::kIdescBMajorMN;
    for (int k = 0; k < my && good; ++k) {
      const int acc = k & 1;
      // the accumulator's previous tile (k - 2) has been read out
      if (k >= 2) good = ptx::mbar_wait_warp(&S.acc_free[acc], (uint32_t)((k - 2) >> 1) & 1u, abort_flag, kKtWaitBudget);
      for (int j = 0; j < 8 && good; ++j) {
        const int buf = j & 1;
        const int g = 8 * k + j;
        good = ptx::mbar_wait_warp(&S.a_full[buf], (uint32_t)(g >> 1) & 1u, abort_flag, kKtWaitBudget);
        if (!good) break;
        ptx::tc_fence_after();
        // B N-major: the two 64-output blocks 8 KB apart, 8-row K groups 1 KB apart
        const uint64_t bd = ptx::smem_desc_sw128_mn(S.B[j], 8192, 1024);
#pragma unroll
        for (int t = 0; t < 3; ++t)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // A: 8 columns (16 bf16) per K step; B: 16 rows (2 KB) per K step
            ptx::mma_f16_ts_elect(tmem + (uint32_t)acc * 128u, tmem + kKtAcol + 128u * buf + 32u * t + 8u * kk,
                                  bd + (uint64_t)(128 * kk), idesc, (j | t | kk) ? 1u : 0u);
        ptx::mma_commit_elect(&S.a_free[buf]);
        if (j == 7) ptx::mma_commit_elect(&S.done[acc]);
      }
    }
    // every MMA issued has completed before tensor memory is freed
    ptx::mma_commit_elect(&S.drain);
    volatile int keep_waiting = 0;
    ptx::mbar_wait_warp(&S.drain, 0, &keep_waiting, kKtWaitBudget);
  } else {
    // ------------------------------------------------------------ split, read out
    const int q4 = warp & 3, cq = warp >> 2;  // lane quarter, 16-channel quarter of the chunk
    const int h = cq >> 1, sub = cq & 1;      // the quarter's half of the ring row, and which 16 of its 32
    const int r = 32 * q4 + lane;             // entry row of the tile
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    int s = 0;
    uint32_t ph = 0;
    for (int k = 0; k < my && good; ++k) {
      const int acc = k & 1;
      const int64_t e = tile_e0(k) + r;
      const int64_t mrow = e < n && o.kv_codes ? dest_row(o.d, e) : -1;  // main-KV plane row of the entry
      for (int j = 0; j < 8; ++j) {
        const int buf = j & 1;
        const int g = 8 * k + j;
        good = ptx::mbar_wait_warp(&S.x_full[s], ph, abort_flag, kKtWaitBudget);
        if (!good) break;
        float x[16];
        const float* row = S.X[s][h] + r * 32;
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // 16-byte chunk c of the row sits at slot c ^ (r % 8)
          const int c = 4 * sub + i;
          const float4 v = *reinterpret_cast<const float4*>(row + 4 * (c ^ (r & 7)));
          x[4 * i] = v.x;
          x[4 * i + 1] = v.y;
          x[4 * i + 2] = v.z;
          x[4 * i + 3] = v.w;
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.x_free[s]);
        if (++s == kKtStages) {
          s = 0;
          ph ^= 1u;
        }
        if (mrow >= 0) {  // main-KV group 4 j + cq of the entry
          const int grp = 4 * j + cq;
          quantize_main_group_vals(x, o.kv_codes + mrow * 256 + grp * 8, o.kv_scales + mrow * 32 + grp);
        }
        uint32_t t3[3][8];
        kt_split(x, t3);
        // operand buffer `buf` is free once the MMAs of chunk g - 2 completed
        if (g >= 2) good = ptx::mbar_wait_warp(&S.a_free[buf], (uint32_t)((g - 2) >> 1) & 1u, abort_flag, kKtWaitBudget);
        if (!good) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int t = 0; t < 3; ++t)
          ptx::tmem_st_32x32b_x8(tmem + lane_base + kKtAcol + 128u * buf + 32u * t + 8u * cq, t3[t]);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&S.a_full[buf]);
        // the previous tile's K^I, read out while this tile's chunks run
        if (j == 1 && k >= 1 && warp < 4)
          good = kt_epilogue(S, tmem, acc ^ 1, (uint32_t)((k - 1) >> 1) & 1u, tile_e0(k - 1), n, o, warp, lane,
                             abort_flag, ws);
        if (!good) break;
      }
    }
    if (good && my > 0 && warp < 4)  // the last tile
      good = kt_epilogue(S, tmem, (my - 1) & 1, (uint32_t)((my - 1) >> 1) & 1u, tile_e0(my - 1), n, o, warp, lane,
                         abort_flag, ws);
  }
  if (!good && lane == 0 && !*abort_flag) {
    *abort_flag = 1;
    report_error(ws, CSA2_ERR_DEVICE_TIMEOUT, 41);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// fp32 [rows][cols] in boxes of 32 columns x box_rows rows (128 bytes per box row), 128-byte swizzle;
// rows beyond the tensor read as zeros
bool make_f32_map(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_bf16_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTcBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Few tokens (split-K): one CTA per entry finishes it.  Thread c sums the K
// slices of channel c of C and Z for each of the entry's m rows, pools them as
// k_cw_tc's epilogue does (Cbar), then the CTA forms K^I = Cbar W_IK: thread t
// sums channels 128 (t / 128) .. + 127 for output t % 128 (every product exact
// inside its fp32 FMA), and the four quarter sums add in a fixed order.  Warp 0
// then writes the entry's main KV (RMSNorm / RoPE as the codec kernels do) and
// warp 1 its indexer key into the planes.
constexpr int kFinThreads = kDMain;
struct FinishOut {
  uint8_t *kv_codes, *kv_scales, *ix_codes, *ix_scales;
  QDest d;
  const float* norm_w;
  float eps;
  int rope;
};
__global__ void __launch_bounds__(kFinThreads) k_cw_finish_small(const float* __restrict__ part, int ksplit,
                                                                 int64_t T, int m,
                                                                 const uint16_t* __restrict__ Wik,
                                                                 const __grid_constant__ FinishOut fo,
                                                                 const __grid_constant__ RopeTheta th) {
  __shared__ __align__(16) float cb[kDMain];
  __shared__ __align__(16) float kis[kDIdx];
  __shared__ float quarter[4][kDIdx];
  const int64_t e = blockIdx.x;
  const int c = threadIdx.x;
  float zmax = -INFINITY, num = 0.0f, den = 0.0f, c0 = 0.0f;
  // two passes over the rows (max, then weighted sums): the partials are L2-resident
  for (int pass = 0; pass < (m == 1 ? 1 : 2); ++pass) {
    for (int r = 0; r < m; ++r) {
      const float* rowp = part + (e * m + r) * (2 * kDMain) + c;
      float cs = 0.0f, zs = 0.0f;
      int k = 0;
      for (; k + 4 <= ksplit; k += 4) {  // four slices' loads in flight
        float cv[4], zv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          cv[u] = rowp[(int64_t)(k + u) * T * (2 * kDMain)];
          zv[u] = rowp[(int64_t)(k + u) * T * (2 * kDMain) + kDMain];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          cs += cv[u];
          zs += zv[u];
        }
      }
      for (; k < ksplit; ++k) {
        cs += rowp[(int64_t)k * T * (2 * kDMain)];
        zs += rowp[(int64_t)k * T * (2 * kDMain) + kDMain];
      }
      if (m == 1) {
        c0 = cs;  // the softmax over one token is exactly 1
      } else if (pass == 0) {
        zmax = fmaxf(zmax, zs);
      } else {
        const float ez = expf(zs - zmax);
        num = fmaf(ez, cs, num);
        den += ez;
      }
    }
  }
  const float v = m == 1 ? c0 : __fdiv_rn(num, den);
  cb[c] = v;
  __syncthreads();
  const int o = c % kDIdx, qt = c / kDIdx;
  float acc = 0.0f;
#pragma unroll 16
  for (int i = 0; i < kDMain / 4; ++i) {
    const int ch = qt * (kDMain / 4) + i;
    acc = fmaf(cb[ch], __uint_as_float((uint32_t)__ldg(Wik + ch * kDIdx + o) << 16), acc);
  }
  quarter[qt][o] = acc;
  __syncthreads();
  if (c < kDIdx) kis[c] = ((quarter[0][c] + quarter[1][c]) + quarter[2][c]) + quarter[3][c];
  __syncthreads();
  const int warp = c / 32, lane = c % 32;
  if (warp == 0) {
    const int64_t row = dest_row(fo.d, e);
    if (row >= 0)
      quantize_main_entry_warp(cb, fo.norm_w, fo.eps, fo.rope, th, fo.rope ? (double)dest_pos(fo.d, e) : 0.0,
                               fo.kv_codes + row * 256, fo.kv_scales + row * 32, lane);
  } else if (warp == 1 && lane < 4) {
    const int64_t row = dest_row(fo.d, e);
    if (row >= 0) quantize_index_group(kis + lane * 32, fo.ix_codes + row * 64 + lane * 16, fo.ix_scales + row * 4 + lane);
  }
}

struct CwWs {
  float* cbar;
  float* ki;
  uint16_t* wt;  // transposed weights (long inputs only)
  float* part;  // split-K partial C and Z [ksplit][T][1024] (few tokens only)
  int ksplit;
  size_t bytes;
};

// K slices of the projection GEMM: few tokens leave most SMs idle with one CTA
// per 128 x 256 tile, so the K range is split until about one item per SM
// (the partials are summed by k_cw_reduce_pool).  Depends only on the shapes.
constexpr int kMaxKSplit = 32;
int cw_ksplit(int64_t T, int64_t d_model, int sms) {
  const int64_t ntiles = cdiv(T, kTcM) * (kDMain / 128);
  if (T <= 0 || ntiles * 2 > sms) return 1;
  int64_t ks = sms / ntiles;
  ks = std::min<int64_t>(ks, d_model / kTcBK);
  ks = std::min<int64_t>(ks, kMaxKSplit);
  return (int)std::max<int64_t>(ks, 1);
}

CwWs cw_ws_layout(void* ws, int64_t n, int64_t d_model, int m = 1) {
  CwWs L;
  char* base = (char*)ws;
  size_t off = kWsHeader;
  const int64_t T = n * m;
  L.ksplit = cw_ksplit(T, d_model, kFillSms);
  L.cbar = (float*)(base ? base + off : nullptr);
  off += align_up((size_t)n * kDMain * 4, 256);
  L.ki = (float*)(base ? base + off : nullptr);
  off += align_up((size_t)n * kDIdx * 4, 256);
  L.wt = nullptr;
  if (T > kDirectMaxT) {
    L.wt = (uint16_t*)(base ? base + off : nullptr);
    off += align_up((size_t)2 * kDMain * d_model * 2, 256);
  }
  L.part = nullptr;
  if (L.ksplit > 1) {
    L.part = (float*)(base ? base + off : nullptr);
    off += align_up((size_t)L.ksplit * T * 2 * kDMain * 4, 256);
  }
  L.bytes = off;
  return L;
}

}  // namespace

}  // namespace csa2

extern "C" size_t csa2_cache_write_workspace_size(int64_t T, int32_t d_model, int32_t m) {
  if (T < 0 || m < 1 || d_model < 0) return 0;
  return csa2::cw_ws_layout(nullptr, T / m, d_model, m).bytes;
}

namespace csa2 {
namespace {

// C = H W_KV, Z = H W_Z (bf16 operands, fp32 accumulation), softmax pooling over
// groups of m consecutive rows of H into L.cbar, then K^I = Cbar W_IK into L.ki:
// T / m entries.  Shared by the prefill write (one slot, contiguous entries) and
// the decode-time append (one group per slot).
// With few tokens (split-K) the finishing kernel also writes the entries into
// dst at d (*written = true); otherwise L.cbar and L.ki hold them for the codec.
csa2_status cw_compute(const void* H_bf16, int64_t T, int32_t d_model, const void* Wkv_bf16,
                       const void* Wz_bf16, const void* Wik_bf16, int32_t m, const CwWs& L, void* ws,
                       cudaStream_t st, const csa2_kv_planes* dst, const QDest& d, const csa2_norm_rope* nr,
                       bool* written) {
  *written = false;
  const int64_t n = T / m;
  if (m <= 32 && T < ((int64_t)1 << 31)) {
    // tensor cores: the persistent GEMM + pooling; W read N-major as given, or
    // (long inputs) K-major from a transposed copy
    const bool nmajor = T <= kDirectMaxT;
    CUtensorMap map_h, map_wkv, map_wz;
    if (nmajor) {
      if (!make_bf16_map(&map_wkv, Wkv_bf16, d_model, kDMain, kTcBK) ||
          !make_bf16_map(&map_wz, Wz_bf16, d_model, kDMain, kTcBK))
        return CSA2_ERR_CUDA;
    } else {
      {
        KernelTimer timer("k_cw_wt", st);
        k_cw_wt<<<dim3((unsigned)(d_model / kWtTile), 2 * kDMain / kWtTile), 256, 0, st>>>(
            (const uint16_t*)Wkv_bf16, (const uint16_t*)Wz_bf16, d_model, L.wt);
      }
      if (!make_bf16_map(&map_wkv, L.wt, 2 * kDMain, d_model, kTcN)) return CSA2_ERR_CUDA;
      map_wz = map_wkv;
    }
    if (!make_bf16_map(&map_h, H_bf16, T, d_model, kTcM)) return CSA2_ERR_CUDA;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int smem = (int)sizeof(TcSmem);
    auto kern = nmajor ? k_cw_tc<true> : k_cw_tc<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return CSA2_ERR_CUDA;
    const int64_t nitems = cdiv(T, kTcM) * (kDMain / 128) * L.ksplit;
    const int grid = (int)std::min<int64_t>(nitems, sms);
    {
      KernelTimer timer("k_cw_tc", st);
      kern<<<grid, kTcThreads, smem, st>>>(map_h, map_wkv, map_wz, T, d_model, m, kDMain, L.cbar, nullptr, L.ksplit,
                                           L.part, ws);
    }
    if (L.ksplit > 1) {  // the partials' sums, pooling, K^I and the codec in one kernel
      FinishOut fo{dst->kv_codes, dst->kv_scales, dst->ix_codes, dst->ix_scales, d,
                   nr ? nr->norm_weight : nullptr, nr ? nr->norm_eps : 0.0f, nr ? nr->rope : 0};
      const RopeTheta th = fo.rope ? make_rope_theta(nr->rope_base) : RopeTheta{};
      KernelTimer timer("k_cw_finish_small", st);
      k_cw_finish_small<<<(unsigned)n, kFinThreads, 0, st>>>(L.part, L.ksplit, T, m, (const uint16_t*)Wik_bf16, fo,
                                                             th);
      *written = true;
      return CSA2_OK;
    }
  } else {
    const int smem = (int)sizeof(GemmSmem);
    if (cudaFuncSetAttribute(k_cw_gemm_pool, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return CSA2_ERR_CUDA;
    KernelTimer timer("k_cw_gemm_pool", st);
    k_cw_gemm_pool<<<dim3((unsigned)cdiv(T, kTM), kDMain / kTN), kCT, smem, st>>>(
        (const uint16_t*)H_bf16, T, d_model, (const uint16_t*)Wkv_bf16, (const uint16_t*)Wz_bf16, m, L.cbar);
  }
  {
    // K^I on the tensor cores (exact three-way bf16 split of Cbar)
    CUtensorMap map_wik, map_cbar;  // W_IK as given: [512][128], 64 x 64 boxes
    if (!make_bf16_map(&map_wik, Wik_bf16, kDMain, kDIdx, 64) || !make_f32_map(&map_cbar, L.cbar, n, kDMain, 128))
      return CSA2_ERR_CUDA;
    const int smem = (int)sizeof(KtSmem);
    if (cudaFuncSetAttribute(k_cw_ki_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return CSA2_ERR_CUDA;
    KernelTimer timer("k_cw_ki_tc", st);
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t kt_tiles = cdiv(n, (int64_t)128);
    // the codec in the same pass: the indexer key always, the main KV when it takes no RMSNorm / RoPE
    const bool main_here = !(nr && (nr->norm_weight || nr->rope));
    const KtOut o{nullptr, dst->ix_codes, dst->ix_scales, main_here ? dst->kv_codes : nullptr,
                  main_here ? dst->kv_scales : nullptr, d};
    k_cw_ki_tc<<<(unsigned)std::min<int64_t>(kt_tiles, sms), kKtThreads, smem, st>>>(map_wik, map_cbar, n, o, ws);
    if (!main_here) launch_quantize(L.cbar, nullptr, n, dst, d, st, nr);
    *written = true;
  }
  return CSA2_OK;
}

}  // namespace
}  // namespace csa2

extern "C" csa2_status csa2_cache_write(const void* H_bf16, int64_t T, int32_t d_model,
                                        const void* Wkv_bf16, const void* Wz_bf16, const void* Wik_bf16,
                                        int32_t m, const csa2_kv_planes* dst, int32_t seq,
                                        int64_t entry_offset, const csa2_norm_rope* kv_nr,
                                        int64_t pos_first, void* ws, size_t ws_bytes, csa2_stream stream) {
  using namespace csa2;
  cudaStream_t st = (cudaStream_t)stream;
  if (!planes_ok(dst) || !H_bf16 || !Wkv_bf16 || !Wz_bf16 || !Wik_bf16 || T < 0 || seq < 0 ||
      entry_offset < 0)
    return CSA2_ERR_INVALID_ARG;
  if (m < 1 || m > 64 || 64 % m != 0 || T % m != 0) return CSA2_ERR_UNSUPPORTED;
  if (d_model < kTK || d_model % 64 != 0) return CSA2_ERR_UNSUPPORTED;
  if (!aligned(H_bf16, 16) || !aligned(Wkv_bf16, 16) || !aligned(Wz_bf16, 16) || !aligned(Wik_bf16, 16))
    return CSA2_ERR_INVALID_ARG;
  if (kv_nr && !norm_rope_ok(kv_nr)) return CSA2_ERR_INVALID_ARG;
  const int64_t n = T / m;
  if (entry_offset + n > dst->seq_stride) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  CwWs L = cw_ws_layout(ws, n, d_model, m);
  if (ws_bytes < L.bytes) return CSA2_ERR_WORKSPACE;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;
  if (T == 0) return CSA2_OK;
  QDest d{};
  d.e0 = (int64_t)seq * dst->seq_stride + entry_offset;
  d.pos_first = pos_first;
  d.pos_step = m;
  bool written = false;
  const csa2_status rc =
      cw_compute(H_bf16, T, d_model, Wkv_bf16, Wz_bf16, Wik_bf16, m, L, ws, st, dst, d, kv_nr, &written);
  if (rc != CSA2_OK) return rc;
  if (!written) launch_quantize(L.cbar, L.ki, n, dst, d, st, kv_nr);
  return launch_status();
}

extern "C" size_t csa2_cache_append_workspace_size(int32_t G, int32_t d_model, int32_t m) {
  if (G < 0 || d_model <= 0 || m < 1) return 0;
  return csa2::cw_ws_layout(nullptr, G, d_model, m).bytes;
}

extern "C" csa2_status csa2_cache_append(const void* H_bf16, int32_t G, int32_t d_model, const void* Wkv_bf16,
                                         const void* Wz_bf16, const void* Wik_bf16, int32_t m,
                                         const csa2_kv_planes* dst, int32_t n_slots, const int32_t* slot,
                                         const int64_t* entry, const csa2_norm_rope* kv_nr, const int64_t* pos,
                                         void* ws, size_t ws_bytes, csa2_stream stream) {
  using namespace csa2;
  cudaStream_t st = (cudaStream_t)stream;
  if (!planes_ok(dst) || !H_bf16 || !Wkv_bf16 || !Wz_bf16 || !Wik_bf16 || G < 0 || n_slots <= 0)
    return CSA2_ERR_INVALID_ARG;
  if (G > 0 && (!slot || !entry || !aligned(entry, 8) || !aligned(slot, 4))) return CSA2_ERR_INVALID_ARG;
  if (m < 1 || m > 64 || 64 % m != 0) return CSA2_ERR_UNSUPPORTED;
  if (d_model < kTK || d_model % 64 != 0) return CSA2_ERR_UNSUPPORTED;
  if (!aligned(H_bf16, 16) || !aligned(Wkv_bf16, 16) || !aligned(Wz_bf16, 16) || !aligned(Wik_bf16, 16))
    return CSA2_ERR_INVALID_ARG;
  if (kv_nr && (!norm_rope_ok(kv_nr) || (kv_nr->rope && (!pos || !aligned(pos, 8))))) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  CwWs L = cw_ws_layout(ws, G, d_model, m);
  if (ws_bytes < L.bytes) return CSA2_ERR_WORKSPACE;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;
  if (G == 0) return CSA2_OK;
  QDest d{};
  d.slot = slot;
  d.entry = entry;
  d.stride = dst->seq_stride;
  d.n_slots = n_slots;
  d.pos = pos;
  d.ws = ws;
  bool written = false;
  const csa2_status rc = cw_compute(H_bf16, (int64_t)G * m, d_model, Wkv_bf16, Wz_bf16, Wik_bf16, m, L, ws, st,
                                    dst, d, kv_nr, &written);
  if (rc != CSA2_OK) return rc;
  if (!written) launch_quantize(L.cbar, L.ki, G, dst, d, st, kv_nr);
  return launch_status();
}

// ---------------------------------------------------------------------------
// The V4 compressors ("DeepSeek-V4: Towards Highly Efficient Million-Token
// Context Intelligence", CSA step 1 and HCA): the projections run unpooled on
// the tensor cores (k_cw_tc with m = 1 writes C and Z), then a pooling kernel
// forms each entry with per-channel softmax weights that include the learned
// position biases.
namespace csa2 {
namespace {

// Pools rows 0 .. rows - 1 of a row source for one channel with softmax weights:
// one pass, eight rows' loads in flight at a time, the running sums rescaled when
// the maximum grows.  src(r, z, v) gives row r's biased score z and value v.
template <class Src>
__device__ __forceinline__ float pool_rows(int rows, const Src& src) {
  constexpr int kRows = 8;
  float zmax = -INFINITY, num = 0.0f, den = 0.0f;
  for (int r = 0; r < rows; r += kRows) {
    float z[kRows], v[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      z[u] = -INFINITY;
      v[u] = 0.0f;
      if (r + u < rows) src(r + u, z[u], v[u]);
    }
    float mx = z[0];
#pragma unroll
    for (int u = 1; u < kRows; ++u) mx = fmaxf(mx, z[u]);
    const float nm = fmaxf(zmax, mx);
    const float sc = expf(zmax - nm);  // 0 on the first chunk (zmax = -inf)
    num *= sc;
    den *= sc;
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const float e = expf(z[u] - nm);  // 0 for the rows past the end
      num = fmaf(e, v[u], num);
      den += e;
    }
    zmax = nm;
  }
  return __fdiv_rn(num, den);
}

// overlapping: entry i pools rows m i .. m i + m - 1 of (Ca, Za + Ba) and rows
// m (i - 1) .. m i - 1 of (Cb, Zb + Bb); entry 0 has only the first part.  One
// CTA per entry, one thread per channel.
__global__ void k_pool_overlap(const float* __restrict__ Ca, const float* __restrict__ Za,
                               const float* __restrict__ Cb, const float* __restrict__ Zb,
                               const float* __restrict__ Ba, const float* __restrict__ Bb, int m, int width,
                               float* __restrict__ out) {
  const int64_t i = blockIdx.x;  // the entry
  const int c = threadIdx.x;     // its channel (blockDim.x = width)
  const int64_t a0 = i * m * width + c, b0 = (i - 1) * m * width + c;
  out[i * width + c] = pool_rows(i > 0 ? 2 * m : m, [&](int r, float& z, float& v) {
    if (r < m) {
      const int64_t row = a0 + (int64_t)r * width;
      z = Za[row] + Ba[(int64_t)r * width + c];
      v = Ca[row];
    } else {
      const int64_t row = b0 + (int64_t)(r - m) * width;
      z = Zb[row] + Bb[(int64_t)(r - m) * width + c];
      v = Cb[row];
    }
  });
}

// The same for a compression rate M fixed at compile time (V4's CSA runs at m = 4):
// all 2 M rows' loads are issued before the first use, and no rescaling is needed.
template <int M>
__global__ void k_pool_overlap_m(const float* __restrict__ Ca, const float* __restrict__ Za,
                                 const float* __restrict__ Cb, const float* __restrict__ Zb,
                                 const float* __restrict__ Ba, const float* __restrict__ Bb, int width,
                                 float* __restrict__ out) {
  const int64_t i = blockIdx.x;  // the entry
  const int c = threadIdx.x;     // its channel (blockDim.x = width)
  const bool has_b = i > 0;
  float z[2 * M], v[2 * M];
#pragma unroll
  for (int r = 0; r < M; ++r) {
    const int64_t ra = (i * M + r) * width + c, rb = ((i - 1) * M + r) * width + c;
    z[r] = Za[ra] + Ba[r * width + c];
    v[r] = Ca[ra];
    z[M + r] = has_b ? Zb[rb] + Bb[r * width + c] : -INFINITY;
    v[M + r] = has_b ? Cb[rb] : 0.0f;
  }
  float zmax = z[0];
#pragma unroll
  for (int r = 1; r < 2 * M; ++r) zmax = fmaxf(zmax, z[r]);
  float num = 0.0f, den = 0.0f;
#pragma unroll
  for (int r = 0; r < 2 * M; ++r) {
    const float e = expf(z[r] - zmax);
    num = fmaf(e, v[r], num);
    den += e;
  }
  out[i * width + c] = __fdiv_rn(num, den);
}

// HCA: entry i pools rows m i .. m i + m - 1 of (C, Z + Bp).
__global__ void k_pool_bias(const float* __restrict__ C, const float* __restrict__ Z, const float* __restrict__ Bp,
                            int m, int width, float* __restrict__ out) {
  const int64_t i = blockIdx.x;  // the entry
  const int c = threadIdx.x;     // its channel (blockDim.x = width)
  const int64_t r0 = i * m * width + c;
  out[i * width + c] = pool_rows(m, [&](int r, float& z, float& v) {
    const int64_t row = r0 + (int64_t)r * width;
    z = Z[row] + Bp[(int64_t)r * width + c];
    v = C[row];
  });
}

struct CmpWs {
  float *c0, *z0, *c1, *z1;  // [T][width <= 512] each: the unpooled projections of up to two paths
  size_t bytes;
};
CmpWs cmp_ws_layout(void* ws, int64_t T, int64_t d_model) {
  CmpWs L{};
  char* base = (char*)ws;
  size_t off = kWsHeader;
  float** f[4] = {&L.c0, &L.z0, &L.c1, &L.z1};
  for (int i = 0; i < 4; ++i) {
    *f[i] = (float*)(base ? base + off : nullptr);
    off += align_up((size_t)T * kDMain * 4, 256);
  }
  (void)d_model;
  L.bytes = off;
  return L;
}

// C = H Wc, Z = H Wz (unpooled, fp32, [T][width]) on the tensor cores
csa2_status project_raw(const void* H, int64_t T, int32_t d_model, int32_t width, const void* Wc, const void* Wz,
                        float* C, float* Z, void* ws, cudaStream_t st) {
  CUtensorMap map_h, map_wc, map_wz;
  if (!make_bf16_map(&map_h, H, T, d_model, kTcM) || !make_bf16_map(&map_wc, Wc, d_model, width, kTcBK) ||
      !make_bf16_map(&map_wz, Wz, d_model, width, kTcBK))
    return CSA2_ERR_CUDA;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess) return CSA2_ERR_CUDA;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int smem = (int)sizeof(TcSmem);
  if (cudaFuncSetAttribute(k_cw_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return CSA2_ERR_CUDA;
  const int64_t ntiles = cdiv(T, kTcM) * (width / 128);
  KernelTimer timer("k_cw_tc", st);
  k_cw_tc<true><<<(int)std::min<int64_t>(ntiles, sms), kTcThreads, smem, st>>>(map_h, map_wc, map_wz, T, d_model, 1,
                                                                                width, C, Z, 1, nullptr, ws);
  return CSA2_OK;
}

csa2_status compress_checks(const void* H, int64_t T, int32_t d_model, int32_t m, int32_t width, float* out,
                            void* ws, size_t ws_bytes, size_t need) {
  if ((!H && T > 0) || !out || T < 0 || m < 1 || m > 1024) return CSA2_ERR_INVALID_ARG;
  if (width < 128 || width > kDMain || width % 128 != 0) return CSA2_ERR_UNSUPPORTED;
  if (T % m != 0) return CSA2_ERR_UNSUPPORTED;
  if (d_model < kTK || d_model % 64 != 0 || T >= ((int64_t)1 << 30)) return CSA2_ERR_UNSUPPORTED;
  if (!aligned(H, 16) || !aligned(out, 16)) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  if (ws_bytes < need) return CSA2_ERR_WORKSPACE;
  return CSA2_OK;
}

}  // namespace
}  // namespace csa2

extern "C" size_t csa2_compress_workspace_size(int64_t T, int32_t d_model) {
  if (T < 0 || d_model <= 0) return 0;
  return csa2::cmp_ws_layout(nullptr, T, d_model).bytes;
}

extern "C" csa2_status csa2_compress_overlap(const void* H_bf16, int64_t T, int32_t d_model, const void* Wa_kv,
                                             const void* Wb_kv, const void* Wa_z, const void* Wb_z, const float* Ba,
                                             const float* Bb, int32_t m, int32_t width, float* out, void* ws,
                                             size_t ws_bytes, csa2_stream stream) {
  using namespace csa2;
  const CmpWs L = cmp_ws_layout(ws, T, d_model);
  csa2_status rc = compress_checks(H_bf16, T, d_model, m, width, out, ws, ws_bytes, L.bytes);
  if (rc != CSA2_OK) return rc;
  if (!Wa_kv || !Wb_kv || !Wa_z || !Wb_z || !Ba || !Bb) return CSA2_ERR_INVALID_ARG;
  if (!aligned(Wa_kv, 16) || !aligned(Wb_kv, 16) || !aligned(Wa_z, 16) || !aligned(Wb_z, 16))
    return CSA2_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;
  if (T == 0) return CSA2_OK;
  if ((rc = project_raw(H_bf16, T, d_model, width, Wa_kv, Wa_z, L.c0, L.z0, ws, st)) != CSA2_OK) return rc;
  if ((rc = project_raw(H_bf16, T, d_model, width, Wb_kv, Wb_z, L.c1, L.z1, ws, st)) != CSA2_OK) return rc;
  const int64_t n = T / m;
  KernelTimer timer("k_pool_overlap", st);
  if (m == 4)
    k_pool_overlap_m<4><<<(unsigned)n, width, 0, st>>>(L.c0, L.z0, L.c1, L.z1, Ba, Bb, width, out);
  else
    k_pool_overlap<<<(unsigned)n, width, 0, st>>>(L.c0, L.z0, L.c1, L.z1, Ba, Bb, m, width, out);
  return launch_status();
}

extern "C" csa2_status csa2_compress_hca(const void* H_bf16, int64_t T, int32_t d_model, const void* W_kv,
                                         const void* W_z, const float* Bp, int32_t m, int32_t width, float* out,
                                         void* ws, size_t ws_bytes, csa2_stream stream) {
  using namespace csa2;
  const CmpWs L = cmp_ws_layout(ws, T, d_model);
  csa2_status rc = compress_checks(H_bf16, T, d_model, m, width, out, ws, ws_bytes, L.bytes);
  if (rc != CSA2_OK) return rc;
  if (!W_kv || !W_z || !Bp || !aligned(W_kv, 16) || !aligned(W_z, 16)) return CSA2_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;
  if (T == 0) return CSA2_OK;
  if ((rc = project_raw(H_bf16, T, d_model, width, W_kv, W_z, L.c0, L.z0, ws, st)) != CSA2_OK) return rc;
  const int64_t n = T / m;
  KernelTimer timer("k_pool_bias", st);
  k_pool_bias<<<(unsigned)n, width, 0, st>>>(L.c0, L.z0, Bp, m, width, out);
  return launch_status();
}
