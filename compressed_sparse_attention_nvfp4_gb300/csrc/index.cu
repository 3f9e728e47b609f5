// Lightning indexer + top-k selection.
//   I_j = sum_h w_h ReLU(q_h . K^I_j)   ("DeepSeek-V4: Towards Highly Efficient
//   Million-Token Context Intelligence", CSA step 2; "DeepSeek-V4.1-Flash: pushing
//   the limits of KV cache compression", 4.1), the hierarchical pool of the first
//   decoder Full layer and the Reindex layers' pool-restricted top-k (4.3).
#include <atomic>
#include <mutex>

#include <cooperative_groups.h>
#include <cub/block/block_scan.cuh>

#include "common.cuh"
#include "index_scan.cuh"
#include "timing.cuh"

namespace csa2 {

namespace cg = cooperative_groups;

// ------------------------------------------------------------------ selection
// Radix select of the k largest keys of one query (one CTA per query), then an
// ordered collection pass: everything above the k-th key, plus the first
// (lowest-index) candidates equal to it, written in ascending candidate order.
// Candidates are entries [0, n), blocks [0, ceil(n/8)), or the entries of the
// 8-entry blocks listed in `pool` (ascending) -- in every case candidate order
// is entry (or block) order, so ties go to the lower index.  The key of
// candidate c is keys[b*key_stride + c], or, with keys_by_entry (pool mode),
// the key of the candidate's entry: keys[b*key_stride + entry].
struct SelectArgs {
  const float* keys;    // [B][key_stride]
  int64_t key_stride;
  const int32_t* n_entries;
  const int32_t* pool;  // [B][keep] or nullptr
  int keep;
  int count_blocks;     // candidates are the 8-entry blocks of [0, n)
  int64_t ncand_fixed;  // candidate count when pool != nullptr
  int k;
  int32_t* out;         // [B][out_stride]
  int64_t out_stride;
  int64_t n_max;        // visible entries are clamped to this bound
  int keys_by_entry;    // pool mode: keys are indexed by entry id, not by candidate
  // queries whose candidate count lies outside [band_lo, band_hi] leave at once (all
  // CTAs of their cluster alike), so a launch can serve the queries of one size band
  int64_t band_lo = 0;
  int64_t band_hi = INT64_MAX;
};

constexpr int kSelItems = 4;   // consecutive candidates per thread per chunk
constexpr int kSelUnroll = 4;  // chunks whose loads are in flight together

// Keys (order-preserving u32, 0 = not a candidate) and entry ids of the four
// candidates c0..c0+3 (c0 a multiple of 4, so they share one pool block).
__device__ __forceinline__ void load_candidates(const SelectArgs& a, int b, int64_t n, int64_t ncand,
                                                int64_t c0, bool vec_ok, uint32_t (&key)[kSelItems],
                                                int64_t (&id)[kSelItems]) {
  const float* kb = a.keys + (int64_t)b * a.key_stride;
  float v[kSelItems];
  if (a.pool && a.keys_by_entry) {
    // four consecutive entries of one pool block (c0 % 8 is 0 or 4)
    const int p = c0 < ncand ? a.pool[(int64_t)b * a.keep + c0 / 8] : -1;
    const int64_t e0 = (int64_t)p * 8 + c0 % 8;
    if (p >= 0 && vec_ok && e0 + kSelItems <= n) {
      const float4 f = *reinterpret_cast<const float4*>(kb + e0);
      v[0] = f.x;
      v[1] = f.y;
      v[2] = f.z;
      v[3] = f.w;
    } else {
#pragma unroll
      for (int i = 0; i < kSelItems; ++i) v[i] = (p >= 0 && e0 + i < n) ? kb[e0 + i] : -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < kSelItems; ++i) {
      id[i] = e0 + i;
      key[i] = (c0 + i < ncand && p >= 0 && id[i] < n) ? score_key(v[i]) : 0u;
    }
    return;
  }
  if (vec_ok && c0 + kSelItems <= ncand) {
    const float4 f = *reinterpret_cast<const float4*>(kb + c0);
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  } else {
#pragma unroll
    for (int i = 0; i < kSelItems; ++i) v[i] = (c0 + i < ncand) ? kb[c0 + i] : -INFINITY;
  }
  if (a.pool) {
    const int p = c0 < ncand ? a.pool[(int64_t)b * a.keep + c0 / 8] : -1;
#pragma unroll
    for (int i = 0; i < kSelItems; ++i) {
      id[i] = (int64_t)p * 8 + (c0 + i) % 8;
      key[i] = (c0 + i < ncand && p >= 0 && id[i] < n) ? score_key(v[i]) : 0u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kSelItems; ++i) {
      id[i] = c0 + i;
      key[i] = c0 + i < ncand ? score_key(v[i]) : 0u;
    }
  }
}

// Digit passes over the four bytes of the key, most significant first, by a
// cluster of kSelCluster CTAs per query: CTA r owns the r-th contiguous slice of
// the candidates.  Each pass, every warp counts its keys into its own 256-bin
// histogram (a warp whose 32 digits agree adds 32 with one atomic), the CTA sums
// its warps, and every CTA of the cluster reads the other CTAs' sums through
// distributed shared memory, so all of them choose the same digit without a
// round trip through global memory.  The ordered collect uses the per-CTA
// counts of keys above / equal to the threshold the same way to place each
// CTA's output.  Loads are vectorised, 16 keys in flight per thread.
constexpr int kSelCluster = 8;
constexpr int kSelThreads = 256;

__global__ void __cluster_dims__(kSelCluster, 1, 1) __launch_bounds__(kSelThreads)
    k_select(SelectArgs a) {
  constexpr int NT = kSelThreads;
  constexpr int kBins = 256;
  constexpr int kWarpsSel = NT / 32;
  constexpr int64_t kChunk = (int64_t)NT * kSelItems;
  using ScanU = cub::BlockScan<unsigned, NT>;
  using ScanI = cub::BlockScan<int, NT>;
  __shared__ union {
    typename ScanU::TempStorage u;
    typename ScanI::TempStorage i;
  } scan_tmp;
  __shared__ unsigned whist[kWarpsSel][kBins];
  __shared__ unsigned chist[kBins];   // this CTA's histogram, read by the whole cluster
  __shared__ unsigned cvalid;         // this CTA's valid-candidate count
  __shared__ int ccount[2];           // this CTA's keys > T and == T
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_need;
  __shared__ int s_base_eq, s_base_out;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / kSelCluster;
  const int tid = threadIdx.x, lane = threadIdx.x % 32, wid = threadIdx.x / 32;
  const int64_t n = max((int64_t)0, min((int64_t)a.n_entries[b], a.n_max));
  const int64_t ncand = a.pool ? a.ncand_fixed : (a.count_blocks ? cdiv(n, 8) : n);
  if (ncand < a.band_lo || ncand > a.band_hi) return;  // another launch's query (uniform per cluster)
  const int64_t per = (int64_t)align_up((size_t)cdiv(ncand, kSelCluster), kSelItems);
  const int64_t lo = min(ncand, rank * per), hi = min(ncand, lo + per);
  const int64_t nchunks = cdiv(hi - lo, kChunk);
  const bool vec_ok = (a.key_stride % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.keys) & 15) == 0);
  int32_t* out = a.out + (int64_t)b * a.out_stride;
  unsigned* myhist = whist[wid];

  if (tid == 0) {
    cvalid = 0;
    s_prefix = 0;
    s_mask = 0;
  }
  __syncthreads();

  int need_total = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int d = lane; d < kBins; d += 32) myhist[d] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix, mask = s_mask;
    unsigned myvalid = 0;
    for (int64_t g = 0; g < nchunks; g += kSelUnroll) {
      uint32_t key[kSelUnroll][kSelItems];
      int64_t id[kSelUnroll][kSelItems];
#pragma unroll
      for (int u = 0; u < kSelUnroll; ++u) {
        const int64_t c0 = lo + (g + u) * kChunk + (int64_t)tid * kSelItems;
        if (c0 < hi) {
          load_candidates(a, b, n, hi, c0, vec_ok, key[u], id[u]);
        } else {
#pragma unroll
          for (int i = 0; i < kSelItems; ++i) key[u][i] = 0u;
        }
      }
#pragma unroll
      for (int u = 0; u < kSelUnroll; ++u)
#pragma unroll
        for (int i = 0; i < kSelItems; ++i) {
          const uint32_t kk = key[u][i];
          myvalid += kk != 0u;
          const bool in = kk != 0u && (kk & mask) == prefix;
          const uint32_t d = in ? ((kk >> shift) & 255u) : 0xFFFFFFFFu;
          const uint32_t d0 = __shfl_sync(0xffffffffu, d, 0);
          if (__all_sync(0xffffffffu, d == d0)) {
            if (lane == 0 && d0 != 0xFFFFFFFFu) atomicAdd(&myhist[d0], 32u);
          } else if (in) {
            atomicAdd(&myhist[d], 1u);
          }
        }
    }
    if (shift == 24) {
      myvalid = __reduce_add_sync(0xffffffffu, myvalid);
      if (lane == 0) atomicAdd(&cvalid, myvalid);
    }
    __syncthreads();
    {  // this CTA's bin totals (thread t <-> bin 255 - t)
      unsigned h = 0;
      const int bin = kBins - 1 - tid;
      for (int w = 0; w < kWarpsSel; ++w) h += whist[w][bin];
      chist[bin] = h;
    }
    cluster.sync();
    if (shift == 24) {
      if (tid == 0) {
        unsigned tv = 0;
        for (int r = 0; r < kSelCluster; ++r) tv += *cluster.map_shared_rank(&cvalid, r);
        s_need = (int)min((int64_t)a.k, (int64_t)tv);
      }
      __syncthreads();
      need_total = s_need;
      if (need_total == 0) break;  // uniform across the cluster
    }
    const int need = s_need;
    const int bin = kBins - 1 - tid;
    unsigned h = 0;
    for (int r = 0; r < kSelCluster; ++r) h += *cluster.map_shared_rank(&chist[bin], r);
    unsigned cum = h;
    ScanU(scan_tmp.u).InclusiveSum(cum, cum);
    if (cum >= (unsigned)need && cum - h < (unsigned)need) {
      s_prefix = prefix | ((uint32_t)bin << shift);
      s_mask = mask | (255u << shift);
      s_need = need - (int)(cum - h);
    }
    cluster.sync();  // every CTA has read the histograms before they are reused
  }
  const uint32_t T = s_prefix;
  const int take_eq = s_need;  // candidates equal to T to take (lowest indices first)

  if (need_total > 0) {
    // counts of this CTA's keys above and equal to T, shared with the cluster
    int gt = 0, eq = 0;
    for (int64_t c0 = lo + (int64_t)tid * kSelItems; c0 < hi; c0 += kChunk) {
      uint32_t key[kSelItems];
      int64_t id[kSelItems];
      load_candidates(a, b, n, hi, c0, vec_ok, key, id);
#pragma unroll
      for (int i = 0; i < kSelItems; ++i) {
        gt += key[i] != 0u && key[i] > T;
        eq += key[i] != 0u && key[i] == T;
      }
    }
    gt = __reduce_add_sync(0xffffffffu, (unsigned)gt);
    eq = __reduce_add_sync(0xffffffffu, (unsigned)eq);
    if (tid == 0) ccount[0] = ccount[1] = 0;
    __syncthreads();
    if (lane == 0) {
      atomicAdd(&ccount[0], gt);
      atomicAdd(&ccount[1], eq);
    }
    cluster.sync();
    if (tid == 0) {
      int eq_before = 0, out_before = 0;
      for (int r = 0; r < rank; ++r) {
        const int* cc = cluster.map_shared_rank(ccount, r);
        const int g_r = cc[0], e_r = cc[1];
        out_before += g_r + max(0, min(e_r, take_eq - eq_before));
        eq_before += e_r;
      }
      s_base_eq = eq_before;
      s_base_out = out_before;
    }
    __syncthreads();
    for (int64_t ch = 0; ch < nchunks; ++ch) {
      uint32_t key[kSelItems];
      int64_t id[kSelItems];
      const int64_t c0 = lo + ch * kChunk + (int64_t)tid * kSelItems;
      if (c0 < hi) {
        load_candidates(a, b, n, hi, c0, vec_ok, key, id);
      } else {
#pragma unroll
        for (int i = 0; i < kSelItems; ++i) {
          key[i] = 0u;
          id[i] = -1;
        }
      }
      int is_eq[kSelItems], eq_rank[kSelItems], take[kSelItems], pos[kSelItems];
#pragma unroll
      for (int i = 0; i < kSelItems; ++i) is_eq[i] = (key[i] != 0u && key[i] == T) ? 1 : 0;
      int eq_total, take_total;
      ScanI(scan_tmp.i).ExclusiveSum(is_eq, eq_rank, eq_total);
      __syncthreads();
      const int base_eq = s_base_eq;
#pragma unroll
      for (int i = 0; i < kSelItems; ++i)
        take[i] = (key[i] != 0u && key[i] > T) || (is_eq[i] && base_eq + eq_rank[i] < take_eq);
      ScanI(scan_tmp.i).ExclusiveSum(take, pos, take_total);
      const int base_out = s_base_out;
#pragma unroll
      for (int i = 0; i < kSelItems; ++i)
        if (take[i]) out[base_out + pos[i]] = (int32_t)id[i];
      __syncthreads();
      if (tid == 0) {
        s_base_eq += eq_total;
        s_base_out += take_total;
      }
      __syncthreads();
    }
  }
  if (rank == kSelCluster - 1) {  // padding after the last selected id
    const int taken = need_total > 0 ? need_total : 0;
    for (int i = taken + tid; i < a.k; i += NT) out[i] = -1;
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

// Resident form of the same selection, for slices of at most kResCap
// candidates per CTA: each CTA loads its slice once into shared memory (coalesced
// loads; thread t owns a contiguous run of kper candidates) and collects with one
// scan: a thread's run is contiguous, so per-thread counts of keys above / equal to
// the threshold, scanned in thread order and offset by the cluster's earlier CTAs,
// place every chosen id in candidate order.  The first digit is the key's offset from
// the cluster's smallest key in units of 2^shift0 (at most 255 units span the keys),
// which spreads keys that share their top bits over the histogram; each thread keeps
// its keys' first digits as bytes, so the keys above the threshold's first-digit bin
// and those in it come from byte-wise compares, and only the latter are looked at
// again.  When the bin's keys of the whole cluster fit kCompCap they are gathered in
// rank 0, which finds the remaining digits alone.  The per-CTA histograms alternate
// between two buffers so that one cluster barrier per pass suffices.  (A single
// 1024-thread CTA per query for the pool's 16,384 entries measured slower than eight
// CTAs: the load latency of one query's gather is then hidden by nothing.)
constexpr int kResMaxPer = 64;  // candidates per thread (a thread's keys fit one 64-bit mask)
constexpr int64_t kResCap = 256 * kResMaxPer;  // candidates per CTA: 64 KB of keys
constexpr int kCompCap = 4096;  // keys of the first digit's threshold bin kept for the later passes

// keys of candidates c0..c0+3 (c0 a multiple of 4; 0 = not a candidate)
__device__ __forceinline__ uint4 load_keys4(const SelectArgs& a, int b, int64_t n, int64_t ncand, int64_t c0,
                                            bool vec_ok) {
  const float* kb = a.keys + (int64_t)b * a.key_stride;
  float v[4];
  int64_t e0 = c0;  // index into the key row of candidate c0
  int64_t lim = ncand;
  bool ok = c0 < ncand;
  if (a.pool) {
    const int p = ok ? a.pool[(int64_t)b * a.keep + c0 / 8] : -1;
    ok = ok && p >= 0;
    if (a.keys_by_entry) {
      e0 = (int64_t)p * 8 + c0 % 8;
      lim = n;
    } else {
      lim = min(ncand, c0 + max((int64_t)0, n - ((int64_t)p * 8 + c0 % 8)));  // entries beyond n are out
    }
  }
  if (ok && vec_ok && e0 + 4 <= lim) {
    const float4 f = *reinterpret_cast<const float4*>(kb + e0);
    v[0] = f.x;
    v[1] = f.y;
    v[2] = f.z;
    v[3] = f.w;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (ok && e0 + i < lim) ? kb[e0 + i] : -INFINITY;
  }
  uint32_t k[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) k[i] = v[i] == -INFINITY ? 0u : score_key(v[i]);
  return make_uint4(k[0], k[1], k[2], k[3]);
}

// First digit of every key of a thread's run (NS slots of 4): counted in the warp's
// histogram and kept, + 1, as a byte in dg (0: no key).
template <int NS>
__device__ __forceinline__ void first_digits(const uint4* myslots, int swz, int shift, uint32_t base0,
                                             unsigned* myhist, uint32_t (&dg)[kResMaxPer / 4]) {
#pragma unroll
  for (int v = 0; v < NS; ++v) {
    const uint4 k4 = myslots[v ^ swz];
    const uint32_t kk4[4] = {k4.x, k4.y, k4.z, k4.w};
    uint32_t w = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (kk4[i] != 0u) {
        const uint32_t d = (kk4[i] >> shift) - base0;
        atomicAdd(&myhist[d], 1u);
        w |= (d + 1u) << (8 * i);
      }
    }
    dg[v] = w;
  }
}

// Bit 4 v + i of gtm / binm: key i of slot v has a first digit above / equal to the
// threshold's (j4: its digit + 1 in every byte), four keys per byte-wise compare.
template <int NS>
__device__ __forceinline__ void digit_masks(const uint32_t (&dg)[kResMaxPer / 4], uint32_t j4, uint64_t& gtm,
                                            uint64_t& binm) {
#pragma unroll
  for (int v = 0; v < NS; ++v) {
    // 0xFF per byte that compares true; the low bit of each byte moved to bits 24..27
    const uint32_t gt = ((__vcmpgtu4(dg[v], j4) & 0x01010101u) * 0x01020408u) >> 24;
    const uint32_t eq = ((__vcmpeq4(dg[v], j4) & 0x01010101u) * 0x01020408u) >> 24;
    gtm |= (uint64_t)gt << (4 * v);
    binm |= (uint64_t)eq << (4 * v);
  }
}

// The same two steps as rolled loops, the digits kept in shared memory (word v of a
// thread at dg[v * stride]).  A select that runs once per SM executes its code once per
// warp, so the unrolled form's length, not its trip count, sets how long the warps wait
// for instructions; a large grid keeps the code in the instruction caches instead, and
// the unrolled form is faster there.
__device__ __forceinline__ void first_digits_rolled(const uint4* myslots, int nslot, int swz, int shift,
                                                    uint32_t base0, unsigned* myhist, uint32_t* dg, int stride) {
#pragma unroll 1
  for (int v = 0; v < nslot; ++v) {
    const uint4 k4 = myslots[v ^ swz];
    const uint32_t kk4[4] = {k4.x, k4.y, k4.z, k4.w};
    uint32_t w = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (kk4[i] != 0u) {
        const uint32_t d = (kk4[i] >> shift) - base0;
        atomicAdd(&myhist[d], 1u);
        w |= (d + 1u) << (8 * i);
      }
    }
    dg[v * stride] = w;
  }
}
__device__ __forceinline__ void digit_masks_rolled(const uint32_t* dg, int stride, int nslot, uint32_t j4,
                                                   uint64_t& gtm, uint64_t& binm) {
#pragma unroll 1
  for (int v = 0; v < nslot; ++v) {
    const uint32_t d = dg[v * stride];
    const uint32_t gt = ((__vcmpgtu4(d, j4) & 0x01010101u) * 0x01020408u) >> 24;
    const uint32_t eq = ((__vcmpeq4(d, j4) & 0x01010101u) * 0x01020408u) >> 24;
    gtm |= (uint64_t)gt << (4 * v);
    binm |= (uint64_t)eq << (4 * v);
  }
}

// kRolled: the first-digit steps as rolled loops (grids of at most two CTAs per SM)
template <int NT, bool kRolled>
__global__ void __launch_bounds__(NT) k_select_res(SelectArgs a) {
  constexpr int kBins = 256;
  constexpr int kWarpsSel = NT / 32;
  using ScanI = cub::BlockScan<int, NT>;
  __shared__ typename ScanI::TempStorage scan_tmp;
  extern __shared__ uint4 keys_s[];  // thread t: 4-key slots t*S .. t*S+S-1, swizzled
  __shared__ unsigned whist[kWarpsSel][kBins];
  __shared__ unsigned chist[2][kBins];  // this CTA's histogram of pass p in chist[p & 1]
  __shared__ unsigned cvalid, ckmin, ckmax;  // this CTA's valid count and key range, read by the cluster
  __shared__ int ccount[2];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int s_need, s_shift0;
  __shared__ uint32_t s_base0;            // first digit of a key: (key >> shift0) - s_base0
  __shared__ int s_base_eq, s_base_out;
  __shared__ int s_ncomp;                 // keys in the compacted list (may exceed kCompCap: then unused)
  __shared__ int s_gtotal, s_goff;        // first digit's threshold bin: cluster total, this CTA's offset
  __shared__ uint32_t comp_s[kCompCap];   // keys in the first pass's threshold bin

  cg::cluster_group cluster = cg::this_cluster();
  const int ncl = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / ncl;
  const int tid = threadIdx.x, lane = threadIdx.x % 32, wid = threadIdx.x / 32;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the keys come from the previous kernel
  const int64_t n = max((int64_t)0, min((int64_t)a.n_entries[b], a.n_max));
  const int64_t ncand = a.pool ? a.ncand_fixed : (a.count_blocks ? cdiv(n, 8) : n);
  if (ncand < a.band_lo || ncand > a.band_hi) return;  // another launch's query (uniform per cluster)
  const int64_t per = (int64_t)align_up((size_t)cdiv(ncand, ncl), kSelItems);
  const int64_t lo = min(ncand, rank * per), hi = min(ncand, lo + per);
  // candidates per thread: a power of two >= 4 covering the slice (the launch
  // sized the shared buffer for the largest slice, n = n_max)
  int kper = 4;
  while ((int64_t)kper * NT < per) kper *= 2;
  const int nslot = kper / 4;
  const int64_t t0 = lo + (int64_t)tid * kper;
  const bool vec_ok = (a.key_stride % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.keys) & 15) == 0);
  int32_t* out = a.out + (int64_t)b * a.out_stride;
  unsigned* myhist = whist[wid];
  uint4* myslots = keys_s + (int64_t)tid * nslot;
  const int swz = tid & (nslot - 1);

  if (tid == 0) {
    cvalid = 0;
    ckmin = 0xFFFFFFFFu;
    ckmax = 0;
    s_ncomp = 0;
  }
  // load the slice once, up to kLoadBatch 4-key groups in flight per thread.  The loads
  // are coalesced (group g = tid + NT u: consecutive threads read consecutive 16 bytes)
  // and each group is stored to its owner's run: owner g / nslot, slot g % nslot
  constexpr int kLoadBatch = NT >= 1024 ? 4 : 16;  // within the register budget of NT threads
  unsigned myvalid = 0;
  uint32_t mykmin = 0xFFFFFFFFu, mykmax = 0;
  const bool contiguous = !a.pool && vec_ok;  // candidate c's key is keys[b][c]
  const float* krow = a.keys + (int64_t)b * a.key_stride;
  for (int v0 = 0; v0 < nslot; v0 += kLoadBatch) {
    uint4 k4[kLoadBatch];
    if (contiguous) {  // every load of the batch in flight before any is used
      float4 f[kLoadBatch];
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int64_t c0 = lo + 4 * ((int64_t)tid + (int64_t)NT * (v0 + u));
        f[u] = (v0 + u < nslot && c0 + 4 <= hi) ? __ldg(reinterpret_cast<const float4*>(krow + c0))
                                                 : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int64_t c0 = lo + 4 * ((int64_t)tid + (int64_t)NT * (v0 + u));
        float v[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
        if (v0 + u < nslot && c0 < hi && c0 + 4 > hi) {  // the slice's ragged end
#pragma unroll
          for (int i = 0; i < 4; ++i) v[i] = c0 + i < hi ? krow[c0 + i] : -INFINITY;
        }
        uint32_t kk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) kk[i] = v[i] == -INFINITY ? 0u : score_key(v[i]);
        k4[u] = make_uint4(kk[0], kk[1], kk[2], kk[3]);
      }
    } else {
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int64_t c0 = lo + 4 * ((int64_t)tid + (int64_t)NT * (v0 + u));
        k4[u] = (v0 + u < nslot && c0 < hi) ? load_keys4(a, b, n, hi, c0, vec_ok) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      if (v0 + u < nslot) {
        const int g = tid + NT * (v0 + u);
        const int o = g / nslot, vs = g % nslot;  // nslot is a power of two
        keys_s[(int64_t)o * nslot + (vs ^ (o & (nslot - 1)))] = k4[u];
        const uint32_t kv[4] = {k4[u].x, k4[u].y, k4[u].z, k4[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (kv[i] != 0u) {
            ++myvalid;
            mykmin = min(mykmin, kv[i]);
            mykmax = max(mykmax, kv[i]);
          }
      }
    }
  }
  myvalid = __reduce_add_sync(0xffffffffu, myvalid);
  mykmin = __reduce_min_sync(0xffffffffu, mykmin);
  mykmax = __reduce_max_sync(0xffffffffu, mykmax);
  __syncthreads();
  if (lane == 0) {
    atomicAdd(&cvalid, myvalid);
    atomicMin(&ckmin, mykmin);
    atomicMax(&ckmax, mykmax);
  }
  // the cluster's valid count and key range.  The first digit is the key's offset from
  // the smallest key in units of 2^shift0, shift0 the least shift that brings the range
  // within 256 units: it spreads the keys over the range's bins, where the key's own top
  // bits would put most of them in a few (scores within a few binades share them)
  cluster.sync();
  if (wid == 0) {  // lane r reads CTA r's values: one round trip
    unsigned tv = 0, kmn = 0xFFFFFFFFu, kmx = 0;
    if (lane < ncl) {
      tv = *cluster.map_shared_rank(&cvalid, lane);
      kmn = *cluster.map_shared_rank(&ckmin, lane);
      kmx = *cluster.map_shared_rank(&ckmax, lane);
    }
    tv = __reduce_add_sync(0xffffffffu, tv);
    kmn = __reduce_min_sync(0xffffffffu, kmn);
    kmx = __reduce_max_sync(0xffffffffu, kmx);
    if (lane == 0) {
      s_need = (int)min((int64_t)a.k, (int64_t)tv);
      int sh = 0;
      if (tv)
        while ((kmx >> sh) - (kmn >> sh) > 254u) ++sh;  // at most 24; digits 0..254
      s_shift0 = sh;
      s_base0 = tv ? kmn >> sh : 0u;
      s_mask = 0u;  // pass 0 takes every valid key
      s_prefix = 0u;
    }
  }
  __syncthreads();
  const int need_total = s_need;
  const int shift0 = s_shift0;
  const uint32_t base0 = s_base0;

  int pass = 0;
  // after the first digit, bit 4 v + i of each: this thread's candidate t0 + 4 v + i lies
  // above the threshold's first-digit bin / in it (only the latter need the final key)
  uint64_t gtm0 = 0, binm = 0;
  uint32_t dg[kResMaxPer / 4];  // first digit + 1 of the keys of slot v, a byte each (0: no key)
  uint32_t* dgr = nullptr;      // the same in shared memory (rolled form)
  if constexpr (kRolled) {
    __shared__ uint32_t dg_s[kResMaxPer / 4][NT];
    dgr = &dg_s[0][tid];
  }
  // digit of pass p: bits [shift + 7, shift] (the last pass may reach below bit 0)
  for (int shift = shift0; need_total > 0 && shift > -8; shift -= 8, ++pass) {
    for (int d = lane; d < kBins; d += 32) myhist[d] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix, mask = s_mask;
    const int ncomp = s_ncomp;
    if (pass > 0 && ncomp <= kCompCap) {  // the later digits only split the first digit's bin
      for (int j = tid; j < ncomp; j += NT) {
        const uint32_t kk = comp_s[j];
        if ((kk & mask) == prefix) atomicAdd(&myhist[(shift >= 0 ? kk >> shift : kk << -shift) & 255u], 1u);
      }
    }
    if (pass == 0) {  // every key: count its first digit and keep it in dg (unrolled per run length)
      if constexpr (kRolled) {
        first_digits_rolled(myslots, nslot, swz, shift, base0, myhist, dgr, NT);
      } else {
        switch (nslot) {
          case 1: first_digits<1>(myslots, swz, shift, base0, myhist, dg); break;
          case 2: first_digits<2>(myslots, swz, shift, base0, myhist, dg); break;
          case 4: first_digits<4>(myslots, swz, shift, base0, myhist, dg); break;
          case 8: first_digits<8>(myslots, swz, shift, base0, myhist, dg); break;
          default: first_digits<kResMaxPer / 4>(myslots, swz, shift, base0, myhist, dg); break;
        }
      }
    }
    const int vend = (pass > 0 && ncomp <= kCompCap) || pass == 0 ? 0 : nslot;
    for (int v = 0; v < vend; ++v) {
      const uint4 k4 = myslots[v ^ swz];
      const uint32_t kk4[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t kk = kk4[i];
        if (kk != 0u && (kk & mask) == prefix) {
          const uint32_t d = pass == 0 ? (kk >> shift) - base0 : (shift >= 0 ? kk >> shift : kk << -shift) & 255u;
          atomicAdd(&myhist[d], 1u);
        }
      }
    }
    __syncthreads();
    unsigned* ch = chist[pass & 1];
    if (tid < kBins) {  // this CTA's bin totals (thread t <-> bin 255 - t)
      unsigned h = 0;
      const int bin = kBins - 1 - tid;
#pragma unroll 8
      for (int w = 0; w < kWarpsSel; ++w) h += whist[w][bin];
      ch[bin] = h;
    }
    // one barrier per pass: the other buffer is rewritten two passes later,
    // after every CTA passed the next pass's barrier (and so finished reading)
    cluster.sync();
    const int need = s_need;
    const int bin = kBins - 1 - tid;  // negative for threads beyond the 256 bins
    unsigned h = 0, below = 0;  // the bin's cluster total and its count in the ranks before this CTA
    if (bin >= 0) {
      unsigned hr[kSelCluster];
#pragma unroll
      for (int r = 0; r < kSelCluster; ++r) hr[r] = r < ncl ? *cluster.map_shared_rank(&ch[bin], r) : 0u;
#pragma unroll
      for (int r = 0; r < kSelCluster; ++r) {
        h += hr[r];
        below += r < rank ? hr[r] : 0u;
      }
    }
    int cum = (int)h;
    ScanI(scan_tmp).InclusiveSum(cum, cum);
    __syncthreads();  // s_need read above before it is rewritten
    if (bin >= 0 && cum >= need && cum - (int)h < need) {
      if (pass == 0) {  // the keys whose bits from shift0 up equal base0 + bin
        s_prefix = (base0 + (uint32_t)bin) << shift;
        s_mask = 0xFFFFFFFFu << shift;
      } else {
        s_prefix = prefix | (shift >= 0 ? (uint32_t)bin << shift : (uint32_t)bin >> -shift);
        s_mask = mask | (shift >= 0 ? 255u << shift : 255u >> -shift);
      }
      s_need = need - (cum - (int)h);
      s_gtotal = (int)h;
      s_goff = (int)below;
    }
    __syncthreads();
    if (pass == 0) {  // from the kept digits: four keys per byte-wise compare
      const uint32_t j4 = (((s_prefix >> shift) - base0) + 1u) * 0x01010101u;  // the bin's digit + 1
      if constexpr (kRolled) {
        digit_masks_rolled(dgr, NT, nslot, j4, gtm0, binm);
      } else {
        switch (nslot) {
          case 1: digit_masks<1>(dg, j4, gtm0, binm); break;
          case 2: digit_masks<2>(dg, j4, gtm0, binm); break;
          case 4: digit_masks<4>(dg, j4, gtm0, binm); break;
          case 8: digit_masks<8>(dg, j4, gtm0, binm); break;
          default: digit_masks<kResMaxPer / 4>(dg, j4, gtm0, binm); break;
        }
      }
    }
    if (pass == 0 && shift > 0) {  // more digits follow: keep the threshold bin's keys
      // the bin's keys of the whole cluster fit one CTA: gather them into rank 0,
      // which finishes the digits alone (no cluster barrier per digit)
      const bool gather = s_gtotal <= kCompCap;
      uint32_t* dst = gather ? cluster.map_shared_rank(comp_s, 0) + s_goff : comp_s;
      // one slot reservation per thread and the few stores of its keys in the bin
      uint64_t mm = binm;
      if (mm) {
        int j = atomicAdd(&s_ncomp, __popcll(mm));
        while (mm) {
          const int bit = __ffsll((long long)mm) - 1;
          mm &= mm - 1;
          const uint32_t kk = reinterpret_cast<const uint32_t*>(&myslots[(bit >> 2) ^ swz])[bit & 3];
          if (j < kCompCap) dst[j] = kk;
          ++j;
        }
      }
      __syncthreads();
      if (gather) {
        cluster.sync();  // every CTA's keys are in rank 0
        if (rank == 0) {
          const int total = s_gtotal;
          for (int sh = shift - 8; sh > -8; sh -= 8) {
            for (int d = lane; d < kBins; d += 32) myhist[d] = 0;
            __syncthreads();
            const uint32_t pf = s_prefix, mk = s_mask;
            for (int j = tid; j < total; j += NT) {  // per-warp histograms, as in the cluster passes
              const uint32_t kk = comp_s[j];
              if ((kk & mk) == pf) atomicAdd(&myhist[(sh >= 0 ? kk >> sh : kk << -sh) & 255u], 1u);
            }
            __syncthreads();
            const int nd = s_need;
            unsigned hb = 0;
            if (bin >= 0) {
#pragma unroll 8
              for (int w = 0; w < kWarpsSel; ++w) hb += whist[w][bin];
            }
            int cb = (int)hb;
            ScanI(scan_tmp).InclusiveSum(cb, cb);
            __syncthreads();
            if (bin >= 0 && cb >= nd && cb - (int)hb < nd) {
              s_prefix = pf | (sh >= 0 ? (uint32_t)bin << sh : (uint32_t)bin >> -sh);
              s_mask = mk | (sh >= 0 ? 255u << sh : 255u >> -sh);
              s_need = nd - (cb - (int)hb);
            }
            __syncthreads();
          }
          if (wid == 0 && lane < ncl) {  // the threshold and the ties to take, to every CTA
            *cluster.map_shared_rank(&s_prefix, lane) = s_prefix;
            *cluster.map_shared_rank(&s_need, lane) = s_need;
          }
        }
        cluster.sync();
        break;
      }
    }
  }
  const uint32_t T = s_prefix;
  const int take_eq = s_need;  // candidates equal to T to take (lowest indices first)

  if (need_total > 0) {
    // bit 4 v + i of gtm / eqm: this thread's candidate t0 + 4 v + i is above / equal to T.
    // Keys above the first digit's bin are above T; only the bin's keys are compared
    uint64_t gtm = gtm0, eqm = 0;
    for (uint64_t bm = binm; bm; bm &= bm - 1) {
      const int bit = __ffsll((long long)bm) - 1;
      const uint32_t kk = reinterpret_cast<const uint32_t*>(&myslots[(bit >> 2) ^ swz])[bit & 3];
      gtm |= (uint64_t)(kk > T) << bit;
      eqm |= (uint64_t)(kk == T) << bit;
    }
    const int gt = __popcll(gtm), eq = __popcll(eqm);
    const int wgt = (int)__reduce_add_sync(0xffffffffu, (unsigned)gt);
    const int weq = (int)__reduce_add_sync(0xffffffffu, (unsigned)eq);
    if (tid == 0) ccount[0] = ccount[1] = 0;
    __syncthreads();
    if (lane == 0) {
      atomicAdd(&ccount[0], wgt);
      atomicAdd(&ccount[1], weq);
    }
    cluster.sync();
    if (wid == 0) {  // lane r reads CTA r's counts at once, then lane 0 combines them in rank order
      int g_r = 0, e_r = 0;
      if (lane < rank) {
        const int* cc = cluster.map_shared_rank(ccount, lane);
        g_r = cc[0];
        e_r = cc[1];
      }
      int eq_before = 0, out_before = 0;
      for (int r = 0; r < rank; ++r) {
        const int gr = __shfl_sync(0xffffffffu, g_r, r), er = __shfl_sync(0xffffffffu, e_r, r);
        out_before += gr + max(0, min(er, take_eq - eq_before));
        eq_before += er;
      }
      if (lane == 0) {
        s_base_eq = eq_before;
        s_base_out = out_before;
      }
    }
    __syncthreads();
    int eq_rank;
    ScanI(scan_tmp).ExclusiveSum(eq, eq_rank);
    __syncthreads();
    const int eq_start = s_base_eq + eq_rank;  // cluster-wide rank of my first key equal to T
    const int eq_take = max(0, min(eq, take_eq - eq_start));
    int pos;
    ScanI(scan_tmp).ExclusiveSum(gt + eq_take, pos);
    pos += s_base_out;
    uint64_t take = gtm;
    for (int q = 0; q < eq_take; ++q) {  // the lowest eq_take candidates equal to T
      take |= eqm & (~eqm + 1);
      eqm &= eqm - 1;
    }
    while (take) {  // ascending candidate order
      const int j = __ffsll((long long)take) - 1;
      take &= take - 1;
      const int64_t c = t0 + j;
      out[pos++] = a.pool ? (int32_t)((int64_t)a.pool[(int64_t)b * a.keep + c / 8] * 8 + c % 8) : (int32_t)c;
    }
  }
  if (rank == ncl - 1) {  // padding after the last selected id
    const int taken = need_total > 0 ? need_total : 0;
    for (int i = taken + tid; i < a.k; i += NT) out[i] = -1;
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

template <int NT>
void launch_select_res(const SelectArgs& a, int B, int ncl, int64_t per, cudaStream_t st) {
  int kper = 4;
  while ((int64_t)kper * NT < per) kper *= 2;
  const int smem = NT * kper * 4;
  // a failure here surfaces as the launch error that launch_status() reports
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // one CTA per select slot or fewer: the rolled form (its code runs once per warp)
  const bool rolled = (int64_t)B * ncl <= 2 * (int64_t)(sms > 0 ? sms : 148);
  auto kern = rolled ? k_select_res<NT, true> : k_select_res<NT, false>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kResCap * 4));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * ncl));
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ncl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // starts with griddepcontrol.wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  KernelTimer timer("k_select_res", st);
  cudaLaunchKernelEx(&cfg, kern, a);
}

void launch_select(const SelectArgs& a, int B, cudaStream_t st) {
  // slice per CTA: the pool candidates, the blocks, or up to n_max entries
  const int64_t ncand_max = a.pool ? a.ncand_fixed : (a.count_blocks ? cdiv(a.n_max, 8) : a.n_max);
  // 8 CTAs per query, or fewer when the batch alone overfills the resident slots
  // (two select CTAs per SM) and each CTA's slice still fits its shared memory:
  // one wave of clusters instead of several
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t slots = 2 * (int64_t)(sms > 0 ? sms : 148);
  int ncl = kSelCluster;
  while (ncl > 1 && (int64_t)B * ncl > slots && cdiv(ncand_max, ncl / 2) <= kResCap) ncl /= 2;
  const int64_t per = (int64_t)align_up((size_t)cdiv(ncand_max, ncl), kSelItems);
  if (per <= kResCap) {
    launch_select_res<256>(a, B, ncl, per, st);
  } else {
    KernelTimer timer("k_select", st);
    k_select<<<B * kSelCluster, kSelThreads, 0, st>>>(a);
  }
}

// FLAT selects of queries whose candidate counts differ widely (the prefill
// indexer's causal bounds): one launch per size band, each with the smallest
// cluster whose CTAs hold a query's slice (1, 2, 4 CTAs for up to 1, 2, 4 x kResCap
// candidates, then launch_select's choice), so a query of few candidates does not
// hold eight CTAs through the cluster's barriers; a query outside a launch's band
// leaves that launch at once.
void launch_select_banded(SelectArgs a, int B, int64_t n_max, cudaStream_t st) {
  int64_t lo = 0;
  for (int ncl = 1; ncl < kSelCluster; ncl *= 2) {
    const int64_t hi = std::min<int64_t>(n_max, (int64_t)ncl * kResCap);
    a.band_lo = lo;
    a.band_hi = hi;
    launch_select_res<256>(a, B, ncl, (int64_t)align_up((size_t)cdiv(std::max<int64_t>(hi, 1), ncl), kSelItems),
                           st);
    if (hi >= n_max) return;
    lo = hi + 1;
  }
  a.band_lo = lo;
  a.band_hi = INT64_MAX;
  launch_select(a, B, st);
}

// ------------------------------------------------------------------ workspace
struct IndexWs {
  float* scores;
  float* bmax;
  int32_t* pool;
  uint8_t* stage_codes;   // POOL mode: the pool blocks' keys gathered contiguously
  uint8_t* stage_scales;  // [B][keep * block] entries of 64 + 4 bytes
  int64_t score_cols, bmax_cols;
  size_t bytes;
};

// FLAT over this many entries or more selects through the 8-entry block maxima: the k
// best blocks hold the k best entries (a block holding one of them has its own best
// entry among them, and blocks rank as their best entries do: by maximum, then block
// id, i.e. entry id), so a pool of k blocks and a select over its 8k entries give the
// flat top-k exactly, from two selections of n/8 and 8k keys instead of one of n.
constexpr int64_t kFlatViaPoolMin = 65536;
inline int32_t flat_pool_blocks(int64_t n_max, int32_t k) { return n_max >= kFlatViaPoolMin ? k : 0; }

// with_stage = false: the layout without the POOL-mode staging part (which sits last),
// for a POOL call over planes the caller staged once (csa2_index_topk_staged).
// The pool part also holds a FLAT call's k blocks (flat_pool_blocks).
static IndexWs index_ws_layout(void* ws, int32_t B, int64_t n_max, int32_t block, int32_t keep, int32_t k,
                               bool with_stage = true) {
  IndexWs L;
  L.score_cols = (int64_t)align_up((size_t)std::max<int64_t>(n_max, (int64_t)keep * block), 64);
  L.bmax_cols = (int64_t)align_up((size_t)cdiv(n_max, block), 64);
  size_t off = kWsHeader;
  size_t s_bytes = (size_t)B * L.score_cols * 4;
  size_t b_bytes = (size_t)B * L.bmax_cols * 4;
  size_t p_bytes = align_up((size_t)B * std::max(keep, flat_pool_blocks(n_max, k)) * 4, 256);
  char* base = (char*)ws;
  L.scores = (float*)(base ? base + off : nullptr);
  off += align_up(s_bytes, 256);
  L.bmax = (float*)(base ? base + off : nullptr);
  off += align_up(b_bytes, 256);
  L.pool = (int32_t*)(base ? base + off : nullptr);
  off += p_bytes;
  const size_t stage_rows = with_stage ? (size_t)B * keep * block : 0;
  L.stage_codes = (uint8_t*)(base ? base + off : nullptr);
  off += align_up(stage_rows * 64, 256);
  L.stage_scales = (uint8_t*)(base ? base + off : nullptr);
  off += align_up(stage_rows * 4, 256);
  L.bytes = off;
  return L;
}

// POOL mode gather: block u of query b's pool -> staged entries (b*keep + u)*8 ..+7
// (codes 512 B, scales 32 B); a warp copies kGatherBlocks blocks with all their
// 16-byte loads in flight.  Blocks that are padding (-1) or start at or beyond n
// are left as they are: the selector masks their candidates by the pool ids.
constexpr int kGatherBlocks = 4;

__global__ void __launch_bounds__(256) k_pool_gather(const uint8_t* __restrict__ ix_codes,
                                                     const uint8_t* __restrict__ ix_scales, int64_t seq_stride,
                                                     const int32_t* __restrict__ n_entries, int64_t n_max,
                                                     const int32_t* __restrict__ pool, int keep, int B,
                                                     uint8_t* __restrict__ st_codes, uint8_t* __restrict__ st_scales) {
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32 * kGatherBlocks;
  const int lane = threadIdx.x % 32;
  const int64_t total = (int64_t)B * keep;
  uint4 code[kGatherBlocks];
  uint32_t scale[kGatherBlocks];
  bool cp_code[kGatherBlocks], cp_scale[kGatherBlocks];
#pragma unroll
  for (int g = 0; g < kGatherBlocks; ++g) {
    const int64_t wg = w0 + g;
    cp_code[g] = cp_scale[g] = false;
    if (wg >= total) continue;
    const int b = (int)(wg / keep);
    const int64_t n = max((int64_t)0, min((int64_t)n_entries[b], n_max));
    const int pb = pool[wg];
    if (pb < 0 || (int64_t)pb * 8 >= n) continue;
    const int rows = (int)min((int64_t)8, seq_stride - (int64_t)pb * 8);  // rows inside the slot
    const int64_t src = (int64_t)b * seq_stride + (int64_t)pb * 8;       // first entry of the block
    cp_code[g] = lane / 4 < rows;  // a quarter of a 64-byte row per lane
    cp_scale[g] = lane < rows;
    if (cp_code[g]) code[g] = reinterpret_cast<const uint4*>(ix_codes + src * 64)[lane];
    if (cp_scale[g]) scale[g] = reinterpret_cast<const uint32_t*>(ix_scales + src * 4)[lane];
  }
#pragma unroll
  for (int g = 0; g < kGatherBlocks; ++g) {
    const int64_t wg = w0 + g;
    if (cp_code[g]) reinterpret_cast<uint4*>(st_codes + wg * 8 * 64)[lane] = code[g];
    if (cp_scale[g]) reinterpret_cast<uint32_t*>(st_scales + wg * 8 * 4)[lane] = scale[g];
  }
}

void launch_pool_gather(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries, int64_t n_max, int32_t keep,
                        const int32_t* pool, uint8_t* st_codes, uint8_t* st_scales, cudaStream_t st) {
  KernelTimer timer("k_pool_gather", st);
  const int64_t warps = cdiv((int64_t)B * keep, kGatherBlocks);
  k_pool_gather<<<(unsigned)cdiv(warps * 32, 256), 256, 0, st>>>(kv->ix_codes, kv->ix_scales, kv->seq_stride,
                                                                 n_entries, n_max, pool, keep, B, st_codes,
                                                                 st_scales);
}

// POOL mode over staged planes ([B][keep * block] entries): the scan scores every
// staged entry as a flat slot, the select keeps the k best of the pool's visible
// blocks (padding and blocks at or beyond n_entries[b] are masked by their ids)
csa2_status pool_scan_select(const uint8_t* st_codes, const uint8_t* st_scales, int32_t B,
                             const int32_t* n_entries, int64_t n_max, const uint16_t* q, const float* w, int32_t k,
                             int32_t block, int32_t keep, const int32_t* pool, int32_t* topk_out,
                             float* scores_out, const IndexWs& L, void* ws, cudaStream_t st) {
  const int64_t keep_c = (int64_t)keep * block;
  float* sc = scores_out ? scores_out : L.scores;
  const int64_t sc_stride = scores_out ? keep_c : L.score_cols;
  csa2_kv_planes staged{};
  staged.ix_codes = const_cast<uint8_t*>(st_codes);
  staged.ix_scales = const_cast<uint8_t*>(st_scales);
  staged.seq_stride = keep_c;
  csa2_status rs = launch_scan(&staged, B, nullptr, keep_c, keep_c, q, w, nullptr, 0, sc, sc_stride, nullptr,
                               0, ws, st);
  if (rs != CSA2_OK) return rs;
  SelectArgs a{sc, sc_stride, n_entries, pool, keep, 0, keep_c, k, topk_out, k, n_max};
  launch_select(a, B, st);
  return CSA2_OK;
}

}  // namespace csa2

namespace csa2 {
namespace {
// Prefill indexer: queries per scan launch, so that their fp32 scores (and, over long
// slots, their block maxima and pools) fit in about 1.25 GiB of workspace (at least one
// query, at most all of them; 2,048 queries over 131,072 entries take one launch).
// Slots of kFlatViaPoolMin entries or more select each query's top-k through a pool of
// k blocks, as csa2_index_topk's FLAT mode does.
constexpr int64_t kPrefillScoreBytes = (int64_t)5 << 28;
struct PrefillWs {
  int64_t cols, bcols, qb;
  bool pooled;
  size_t score_bytes, bmax_bytes, pool_bytes, bytes;
};
PrefillWs prefill_ws(int32_t Q, int64_t n_max, int32_t k) {
  PrefillWs L;
  L.cols = (int64_t)align_up((size_t)std::max<int64_t>(n_max, 1), 64);
  L.pooled = flat_pool_blocks(n_max, k) > 0;
  L.bcols = L.pooled ? (int64_t)align_up((size_t)cdiv(n_max, 8), 64) : 0;
  const int64_t per_query = (L.cols + L.bcols + (L.pooled ? k : 0)) * 4;
  L.qb = std::max<int64_t>(1, std::min<int64_t>(Q, kPrefillScoreBytes / per_query));
  L.score_bytes = align_up((size_t)L.qb * L.cols * 4, 256);
  L.bmax_bytes = align_up((size_t)L.qb * L.bcols * 4, 256);
  L.pool_bytes = L.pooled ? align_up((size_t)L.qb * k * 4, 256) : 0;
  L.bytes = kWsHeader + L.score_bytes + L.bmax_bytes + L.pool_bytes;
  return L;
}
}  // namespace
}  // namespace csa2

extern "C" size_t csa2_index_topk_prefill_workspace_size(int32_t Q, int64_t n_max, int32_t k) {
  if (Q <= 0 || n_max < 0 || k < 0) return 0;
  return csa2::prefill_ws(Q, n_max, k).bytes;
}

extern "C" csa2_status csa2_index_topk_prefill(const csa2_kv_planes* kv, int32_t seq, int32_t Q,
                                               const int32_t* n_visible, int64_t n_max, const void* qidx_bf16,
                                               const float* w, int32_t k, int32_t* topk_out, void* ws,
                                               size_t ws_bytes, csa2_stream stream) {
  using namespace csa2;
  cudaStream_t st = (cudaStream_t)stream;
  if (!planes_ok(kv) || seq < 0 || Q <= 0 || !n_visible || !qidx_bf16 || !w || !topk_out)
    return CSA2_ERR_INVALID_ARG;
  if (k < 1 || k > CSA2_MAX_TOPK || n_max < 0 || n_max > kv->seq_stride || n_max >= ((int64_t)1 << 31))
    return CSA2_ERR_INVALID_ARG;
  if (!aligned(qidx_bf16, 16) || !aligned(w, 16)) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  const PrefillWs L = prefill_ws(Q, n_max, k);
  if (ws_bytes < L.bytes) return CSA2_ERR_WORKSPACE;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;
  char* base = (char*)ws + kWsHeader;
  float* scores = (float*)base;
  float* bmax = L.pooled ? (float*)(base + L.score_bytes) : nullptr;
  int32_t* pool = L.pooled ? (int32_t*)(base + L.score_bytes + L.bmax_bytes) : nullptr;
  const uint16_t* q = (const uint16_t*)qidx_bf16;
  for (int64_t q0 = 0; q0 < Q; q0 += L.qb) {
    const int32_t nb = (int32_t)std::min<int64_t>(L.qb, Q - q0);
    csa2_status rs = launch_scan_prefill(kv, nb, n_visible + q0, n_max, q + q0 * kHIdx * kDIdx, w + q0 * kHIdx,
                                         scores, L.cols, bmax, L.bcols, ws, st, seq);
    if (rs != CSA2_OK) return rs;
    if (L.pooled) {  // the k best blocks by maximum, then the k best entries of those blocks
      SelectArgs pa{bmax, L.bcols, n_visible + q0, nullptr, 0, 1, 0, k, pool, k, n_max};
      launch_select(pa, nb, st);
      SelectArgs ta{scores, L.cols, n_visible + q0, pool, k, 0, (int64_t)k * 8, k, topk_out + q0 * k, k, n_max, 1};
      launch_select(ta, nb, st);
    } else {
      launch_select_banded(
          SelectArgs{scores, L.cols, n_visible + q0, nullptr, 0, 0, 0, k, topk_out + q0 * k, k, n_max}, nb, n_max,
          st);
    }
  }
  return launch_status();
}

extern "C" size_t csa2_index_topk_workspace_size(int32_t B, int64_t n_max, int32_t k, int32_t block,
                                                 int32_t n_blocks_keep) {
  if (B <= 0 || n_max < 0 || block <= 0 || n_blocks_keep < 0 || k < 0) return 0;
  return csa2::index_ws_layout(nullptr, B, n_max, block, n_blocks_keep, k).bytes;
}

extern "C" csa2_status csa2_index_topk(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries,
                                       int64_t n_max, const void* qidx_bf16, const float* w, int32_t k,
                                       csa2_topk_mode mode, int32_t block, int32_t n_blocks_keep,
                                       const int32_t* pool_in, int32_t* topk_out, int32_t* pool_out,
                                       float* scores_out, void* ws, size_t ws_bytes,
                                       csa2_stream stream) {
  using namespace csa2;
  cudaStream_t st = (cudaStream_t)stream;
  if (!planes_ok(kv) || B <= 0 || !n_entries || !qidx_bf16 || !w || !topk_out) return CSA2_ERR_INVALID_ARG;
  if (k < 1 || k > CSA2_MAX_TOPK || n_max < 0 || n_max > kv->seq_stride || n_max >= ((int64_t)1 << 31))
    return CSA2_ERR_INVALID_ARG;
  if (mode != CSA2_TOPK_FLAT && mode != CSA2_TOPK_HIER_BUILD && mode != CSA2_TOPK_POOL)
    return CSA2_ERR_INVALID_ARG;
  if (mode != CSA2_TOPK_FLAT) {
    if (block != 8) return CSA2_ERR_UNSUPPORTED;
    if (n_blocks_keep < 1 || (int64_t)n_blocks_keep * block > 16384) return CSA2_ERR_INVALID_ARG;
    if (mode == CSA2_TOPK_POOL && !pool_in) return CSA2_ERR_INVALID_ARG;
  } else {
    block = 8;
    n_blocks_keep = 0;
  }
  if (!aligned(qidx_bf16, 16) || !aligned(w, 16)) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  IndexWs L = index_ws_layout(ws, B, n_max, block, n_blocks_keep, k);
  if (ws_bytes < L.bytes) return CSA2_ERR_WORKSPACE;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;

  const uint16_t* q = (const uint16_t*)qidx_bf16;
  const int64_t keep_c = (int64_t)n_blocks_keep * block;

  if (mode == CSA2_TOPK_POOL) {
    // gather the pool's blocks into contiguous staged entries, then scan those
    // as flat slots of keep_c entries (one tensor load per 128 entries instead
    // of one per 8-entry block)
    launch_pool_gather(kv, B, n_entries, n_max, n_blocks_keep, pool_in, L.stage_codes, L.stage_scales, st);
    csa2_status rs = pool_scan_select(L.stage_codes, L.stage_scales, B, n_entries, n_max, q, w, k, block,
                                      n_blocks_keep, pool_in, topk_out, scores_out, L, ws, st);
    if (rs != CSA2_OK) return rs;
    return launch_status();
  }

  if (mode == CSA2_TOPK_FLAT && flat_pool_blocks(n_max, k) > 0) {
    // long contexts: the same top-k through a pool of k blocks (flat_pool_blocks)
    n_blocks_keep = flat_pool_blocks(n_max, k);
  } else if (mode == CSA2_TOPK_FLAT) {
    float* sc = scores_out ? scores_out : L.scores;
    int64_t sc_stride = scores_out ? n_max : L.score_cols;
    csa2_status rs = launch_scan(kv, B, n_entries, n_max, n_max, q, w, nullptr, 0, sc, sc_stride,
                                 nullptr, 0, ws, st);
    if (rs != CSA2_OK) return rs;
    SelectArgs a{sc, sc_stride, n_entries, nullptr, 0, 0, 0, k, topk_out, k, n_max};
    launch_select(a, B, st);
    return launch_status();
  }

  // HIER_BUILD (and FLAT over long contexts): one full scan writes every entry's
  // score and the block maxima; the pool is selected from the maxima, and the token
  // top-k reads the scores of the pool's entries where the scan left them (4 bytes
  // written per entry instead of a second pass over the pool's keys).
  const int64_t keep_p = (int64_t)n_blocks_keep * 8;
  float* sc = scores_out ? scores_out : L.scores;
  const int64_t sc_stride = scores_out ? n_max : L.score_cols;
  csa2_status rs = launch_scan(kv, B, n_entries, n_max, n_max, q, w, nullptr, 0, sc, sc_stride, L.bmax,
                               L.bmax_cols, ws, st);
  if (rs != CSA2_OK) return rs;
  int32_t* pool = pool_out && mode == CSA2_TOPK_HIER_BUILD ? pool_out : L.pool;
  SelectArgs pa{L.bmax, L.bmax_cols, n_entries, nullptr, 0, 1, 0, n_blocks_keep, pool, n_blocks_keep,
                n_max};
  launch_select(pa, B, st);
  SelectArgs ta{sc, sc_stride, n_entries, pool, n_blocks_keep, 0, keep_p, k, topk_out, k, n_max, 1};
  launch_select(ta, B, st);
  return launch_status();
}

extern "C" csa2_status csa2_pool_stage(const csa2_kv_planes* kv, int32_t B, const int32_t* n_entries,
                                       int64_t n_max, int32_t block, int32_t n_blocks_keep, const int32_t* pool,
                                       uint8_t* stage_codes, uint8_t* stage_scales, csa2_stream stream) {
  using namespace csa2;
  if (!planes_ok(kv) || B <= 0 || !n_entries || !pool || !stage_codes || !stage_scales) return CSA2_ERR_INVALID_ARG;
  if (n_max < 0 || n_max > kv->seq_stride || n_max >= ((int64_t)1 << 31)) return CSA2_ERR_INVALID_ARG;
  if (block != 8) return CSA2_ERR_UNSUPPORTED;
  if (n_blocks_keep < 1 || (int64_t)n_blocks_keep * block > 16384) return CSA2_ERR_INVALID_ARG;
  if (!aligned(stage_codes, 32) || !aligned(stage_scales, 16)) return CSA2_ERR_INVALID_ARG;
  launch_pool_gather(kv, B, n_entries, n_max, n_blocks_keep, pool, stage_codes, stage_scales,
                     (cudaStream_t)stream);
  return launch_status();
}

extern "C" csa2_status csa2_index_topk_staged(const uint8_t* stage_codes, const uint8_t* stage_scales, int32_t B,
                                              const int32_t* n_entries, int64_t n_max, const void* qidx_bf16,
                                              const float* w, int32_t k, int32_t block, int32_t n_blocks_keep,
                                              const int32_t* pool_in, int32_t* topk_out, float* scores_out,
                                              void* ws, size_t ws_bytes, csa2_stream stream) {
  using namespace csa2;
  cudaStream_t st = (cudaStream_t)stream;
  if (!stage_codes || !stage_scales || B <= 0 || !n_entries || !qidx_bf16 || !w || !pool_in || !topk_out)
    return CSA2_ERR_INVALID_ARG;
  if (k < 1 || k > CSA2_MAX_TOPK || n_max < 0 || n_max >= ((int64_t)1 << 31)) return CSA2_ERR_INVALID_ARG;
  if (block != 8) return CSA2_ERR_UNSUPPORTED;
  if (n_blocks_keep < 1 || (int64_t)n_blocks_keep * block > 16384) return CSA2_ERR_INVALID_ARG;
  if (!aligned(stage_codes, 32) || !aligned(stage_scales, 16)) return CSA2_ERR_INVALID_ARG;
  if (!aligned(qidx_bf16, 16) || !aligned(w, 16)) return CSA2_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return CSA2_ERR_WORKSPACE;
  IndexWs L = index_ws_layout(ws, B, n_max, block, n_blocks_keep, k, false);
  if (ws_bytes < L.bytes) return CSA2_ERR_WORKSPACE;
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;
  csa2_status rs = pool_scan_select(stage_codes, stage_scales, B, n_entries, n_max, (const uint16_t*)qidx_bf16, w,
                                    k, block, n_blocks_keep, pool_in, topk_out, scores_out, L, ws, st);
  if (rs != CSA2_OK) return rs;
  return launch_status();
}

// ---------------------------------------------------------------------------
// Allocation-free variant of csa2_index_topk.
//
// Some callers cannot allocate device memory at the point where they run the
// indexer: an inference-engine plugin that is handed only its input and output
// buffers, a serving loop whose memory is carved up once at start-up with no
// allocator reachable from the hot path, or a runtime that forbids allocation
// while it records a replayable command sequence.  For them this entry point
// keeps its scratch (block maxima, candidate scores, the pool, the error word)
// in one file-scope device array of CSA2_NOALLOC_SCRATCH_BYTES, which every GPU
// that loads the library holds until the process exits.  The host code below
// looks up that array's device address once per device and passes it to the
// same kernels csa2_index_topk launches.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CSA2_NOALLOC_SCRATCH_BYTES];

namespace csa2 {
namespace {

constexpr int kMaxDevices = 64;

// The array's device address belongs to the CUDA context that loaded this
// module: after a device reset the next context loads it afresh, possibly at
// another address.  So the cached address is keyed on the context's unique id
// (cuCtxGetId), and a call from a new context looks it up again.
struct NoallocSlot {
  unsigned long long ctx_id;  // 0: not looked up yet
  void* addr;
};
NoallocSlot g_noalloc_slot[kMaxDevices];
std::mutex g_noalloc_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// id of the current thread's CUDA context (0 if it cannot be read)
unsigned long long current_ctx_id() {
  static CtxGetCurrentFn get_cur = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (CtxGetCurrentFn) nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  static CtxGetIdFn get_id = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (CtxGetIdFn) nullptr;
    return reinterpret_cast<CtxGetIdFn>(f);
  }();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current device's context, looked
// up with that device current on the first call in each context.
csa2_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CSA2_ERR_CUDA;
  unsigned long long id = current_ctx_id();  // 0 before the runtime made a context current here
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocSlot& s = g_noalloc_slot[dev];
  if (id == 0 || s.ctx_id != id || !s.addr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return CSA2_ERR_CUDA;
    s.addr = p;
    s.ctx_id = current_ctx_id();  // the lookup made the device's primary context current
  }
  *out = s.addr;
  return CSA2_OK;
}

}  // namespace
}  // namespace csa2

extern "C" csa2_status csa2_index_topk_noalloc(const csa2_kv_planes* kv, int32_t B,
                                               const int32_t* n_entries, int64_t n_max,
                                               const void* qidx_bf16, const float* w, int32_t k,
                                               csa2_topk_mode mode, int32_t block,
                                               int32_t n_blocks_keep, const int32_t* pool_in,
                                               int32_t* topk_out, int32_t* pool_out,
                                               csa2_stream stream) {
  using namespace csa2;
  cudaStream_t st = (cudaStream_t)stream;
  if (!planes_ok(kv) || B <= 0 || !n_entries || !qidx_bf16 || !w || !topk_out) return CSA2_ERR_INVALID_ARG;
  if (k < 1 || k > CSA2_MAX_TOPK || n_max < 0 || n_max > kv->seq_stride || n_max >= ((int64_t)1 << 31))
    return CSA2_ERR_INVALID_ARG;
  if (mode != CSA2_TOPK_FLAT && mode != CSA2_TOPK_HIER_BUILD && mode != CSA2_TOPK_POOL)
    return CSA2_ERR_INVALID_ARG;
  if (mode != CSA2_TOPK_FLAT) {
    if (block != 8) return CSA2_ERR_UNSUPPORTED;
    if (n_blocks_keep < 1 || (int64_t)n_blocks_keep * block > 16384) return CSA2_ERR_INVALID_ARG;
    if (mode == CSA2_TOPK_POOL && !pool_in) return CSA2_ERR_INVALID_ARG;
  } else {
    block = 8;
    n_blocks_keep = 0;
  }
  if (!aligned(qidx_bf16, 16) || !aligned(w, 16)) return CSA2_ERR_INVALID_ARG;

  // scratch layout of this mode: [error word | scores | block maxima | pool]
  const int64_t keep_c = (int64_t)n_blocks_keep * block;
  const int64_t score_cols = (int64_t)align_up((size_t)(mode == CSA2_TOPK_FLAT ? n_max : keep_c), 64);
  const int64_t bmax_cols = mode == CSA2_TOPK_HIER_BUILD ? (int64_t)align_up((size_t)cdiv(n_max, 8), 64) : 0;
  const size_t s_bytes = align_up((size_t)B * score_cols * 4, 256);
  const size_t b_bytes = align_up((size_t)B * bmax_cols * 4, 256);
  const size_t p_bytes =
      mode == CSA2_TOPK_HIER_BUILD && !pool_out ? align_up((size_t)B * n_blocks_keep * 4, 256) : 0;
  if (kWsHeader + s_bytes + b_bytes + p_bytes > (size_t)CSA2_NOALLOC_SCRATCH_BYTES) return CSA2_ERR_WORKSPACE;

  void* ws = nullptr;
  csa2_status rs = noalloc_scratch(&ws);
  if (rs != CSA2_OK) return rs;
  char* base = (char*)ws;
  float* scores = (float*)(base + kWsHeader);
  float* bmax = (float*)(base + kWsHeader + s_bytes);
  int32_t* pool_tmp = (int32_t*)(base + kWsHeader + s_bytes + b_bytes);
  if (reset_error(ws, st) != CSA2_OK) return CSA2_ERR_CUDA;  // the error word starts at zero
  const uint16_t* q = (const uint16_t*)qidx_bf16;

  if (mode == CSA2_TOPK_POOL) {
    rs = launch_scan(kv, B, n_entries, n_max, keep_c, q, w, pool_in, n_blocks_keep, scores, score_cols,
                     nullptr, 0, ws, st);
    if (rs != CSA2_OK) return rs;
    SelectArgs a{scores, score_cols, n_entries, pool_in, n_blocks_keep, 0, keep_c, k, topk_out, k, n_max};
    launch_select(a, B, st);
    return launch_status();
  }
  if (mode == CSA2_TOPK_FLAT) {
    rs = launch_scan(kv, B, n_entries, n_max, n_max, q, w, nullptr, 0, scores, score_cols, nullptr, 0, ws,
                     st);
    if (rs != CSA2_OK) return rs;
    SelectArgs a{scores, score_cols, n_entries, nullptr, 0, 0, 0, k, topk_out, k, n_max};
    launch_select(a, B, st);
    return launch_status();
  }
  rs = launch_scan(kv, B, n_entries, n_max, n_max, q, w, nullptr, 0, nullptr, 0, bmax, bmax_cols, ws, st);
  if (rs != CSA2_OK) return rs;
  int32_t* pool = pool_out ? pool_out : pool_tmp;
  SelectArgs pa{bmax, bmax_cols, n_entries, nullptr, 0, 1, 0, n_blocks_keep, pool, n_blocks_keep, n_max};
  launch_select(pa, B, st);
  rs = launch_scan(kv, B, n_entries, n_max, keep_c, q, w, pool, n_blocks_keep, scores, score_cols, nullptr,
                   0, ws, st);
  if (rs != CSA2_OK) return rs;
  SelectArgs ta{scores, score_cols, n_entries, pool, n_blocks_keep, 0, keep_c, k, topk_out, k, n_max};
  launch_select(ta, B, st);
  return launch_status();
}

extern "C" csa2_status csa2_index_topk_noalloc_check(csa2_stream stream, int64_t* detail) {
  void* ws = nullptr;
  csa2_status rs = csa2::noalloc_scratch(&ws);
  if (rs != CSA2_OK) return rs;
  return csa2_check(ws, stream, detail);
}
