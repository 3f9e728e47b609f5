// Group quantizers of the cache format, usable from any kernel (the codec entry
// point and the cache-write epilogue share them so the bytes always agree).
#pragma once

#include "common.cuh"

namespace csa2 {

// Main KV: 16 channels -> 8 bytes of E2M1 codes + 1 E4M3 scale byte.
// x16 must be 16-byte aligned; codes8 8-byte aligned.
// x / s correctly rounded, for a positive E4M3 scale s and r = RN(1 / s), by Markstein's
// FMA correction of the reciprocal product (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990):
// q0 = x r, then q = q0 + (x - q0 s) r in two fused steps.  For every positive E4M3 s and
// every fp32 significand of x with x / s in [2^-5, 2^7) -- the range a group's values take,
// below which the E2M1 code is 0 either way -- it equals the correctly rounded division bit
// for bit: csa2_selftest_codec_division checks exactly that set.
__device__ __forceinline__ float div_by_e4m3(float x, float s, float r) {
  const float q0 = x * r;
  return fmaf(fmaf(-q0, s, x), r, q0);
}

__device__ __forceinline__ void quantize_main_group_vals(const float (&v)[16], uint8_t* codes8,
                                                         uint8_t* scale1) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  float t = __fdiv_rn(amax, 6.0f);
  uint32_t sb = float_to_e4m3(t);
  float s = e4m3_to_float(sb);
  uint32_t c0 = 0, c1 = 0;
  if (s != 0.0f) {
    const float r = __frcp_rn(s);
    auto quo = [&](float x) { return div_by_e4m3(x, s, r); };
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c0 |= float2_to_e2m1x2(quo(v[2 * i]), quo(v[2 * i + 1])) << (8 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c1 |= float2_to_e2m1x2(quo(v[8 + 2 * i]), quo(v[9 + 2 * i])) << (8 * i);
  }
  *reinterpret_cast<uint2*>(codes8) = make_uint2(c0, c1);
  *scale1 = (uint8_t)sb;
}

__device__ __forceinline__ void quantize_main_group(const float* __restrict__ x16, uint8_t* codes8,
                                                    uint8_t* scale1) {
  float v[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 f = reinterpret_cast<const float4*>(x16)[i];
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
  quantize_main_group_vals(v, codes8, scale1);
}

// ---------------------------------------------------------------- RMSNorm / RoPE
// Partial RoPE of a 512-channel vector: pair i (channels 448 + 2i, 449 + 2i,
// i < 32) turns by pos * theta_i, theta_i = base^(-i/32).  The angles are
// formed and reduced modulo 2 pi in fp64 (positions reach millions), then
// sin / cos in fp32.
constexpr int kRopeFirst = kDMain - 64;
struct RopeTheta {
  double t[32];
};
inline RopeTheta make_rope_theta(double base) {
  RopeTheta r;
  for (int i = 0; i < 32; ++i) r.t[i] = pow(base, -2.0 * i / 64.0);
  return r;
}
__device__ __forceinline__ void rope_cos_sin(double theta, double pos, float& c, float& s) {
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  constexpr double kInvTwoPi = 0.15915494309189533576888376337251;
  const double a = pos * theta;
  // a - 2 pi n with n the nearest integer to a / 2 pi (a product, not an fp64
  // division): |red| <= pi up to a last-bit slip near a half turn, which sincosf
  // takes as it is
  const double red = fma(-kTwoPi, rint(a * kInvTwoPi), a);
  sincosf((float)red, &s, &c);
}
// (x, y) turned counter-clockwise by the angle with cosine c, sine s
__device__ __forceinline__ void rope_pair(float& x, float& y, float c, float s) {
  const float nx = x * c - y * s, ny = x * s + y * c;
  x = nx;
  y = ny;
}

// floor(log2 a) of a finite fp32 a > 0 (normal or subnormal), exactly
__device__ __forceinline__ int floor_log2_f32(float a) {
  uint32_t u = __float_as_uint(a);
  int ef = (int)((u >> 23) & 0xFFu);
  if (ef) return ef - 127;
  return (31 - __clz((int)(u & 0x7FFFFFu))) - 149;
}

// 2^k as fp32 for k in [-127, 127] (2^-127 is the subnormal 0x00400000)
__device__ __forceinline__ float exp2i_f32(int k) {
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}

// Indexer key (MXFP4): 32 elements -> 16 bytes of codes + 1 E8M0 byte.
__device__ __forceinline__ void quantize_index_group_vals(const float (&v)[32], uint8_t* codes16,
                                                          uint8_t* scale1) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  int e = -127;
  if (amax > 0.0f) {
    e = floor_log2_f32(amax) - 2;
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
  }
  uint32_t c[4] = {0u, 0u, 0u, 0u};
  if (amax > 0.0f) {
    float inv = exp2i_f32(-e);  // x / 2^e = x * 2^-e, exact where a code can be nonzero
#pragma unroll
    for (int i = 0; i < 16; ++i)
      c[i / 4] |= float2_to_e2m1x2(__fmul_rn(v[2 * i], inv), __fmul_rn(v[2 * i + 1], inv))
                  << (8 * (i % 4));
  }
  *reinterpret_cast<uint4*>(codes16) = make_uint4(c[0], c[1], c[2], c[3]);
  *scale1 = (uint8_t)(e + 127);
}

__device__ __forceinline__ void quantize_index_group(const float* __restrict__ x32, uint8_t* codes16,
                                                     uint8_t* scale1) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4 f = reinterpret_cast<const float4*>(x32)[i];
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
  quantize_index_group_vals(v, codes16, scale1);
}

// Where the entries of a quantize launch go (and, for RoPE, their positions).
struct QDest {
  int64_t e0;             // contiguous: entry e -> plane row e0 + e
  const int32_t* slot;    // or scattered: entry e -> row slot[e] * stride + entry[e]
  const int64_t* entry;
  int64_t stride;
  int32_t n_slots;
  const int64_t* pos;     // positions of the entries, or pos_first + e * pos_step
  int64_t pos_first, pos_step;
  void* ws;               // error word for destinations outside the planes
};

// Entry e of a quantize launch goes to plane row dest_row(d, e): contiguous rows
// e0 + e, or (scattered) slot[e] * stride + entry[e], skipped and reported when
// outside the planes.
__device__ __forceinline__ int64_t dest_row(const QDest& d, int64_t e) {
  if (!d.slot) return d.e0 + e;
  const int32_t sl = d.slot[e];
  const int64_t en = d.entry[e];
  if (sl < 0 || sl >= d.n_slots || en < 0 || en >= d.stride) {
    if (d.ws) report_error(d.ws, CSA2_ERR_INDEX_RANGE, sl < 0 || sl >= d.n_slots ? (long long)sl : en);
    return -1;
  }
  return (int64_t)sl * d.stride + en;
}
__device__ __forceinline__ int64_t dest_pos(const QDest& d, int64_t e) {
  return d.pos ? d.pos[e] : d.pos_first + e * d.pos_step;
}

// One entry's main-KV copy by one warp: optional RMSNorm (weight w, eps) and
// RoPE at position pos, then the E2M1 / E4M3 quantizer; lane l holds channels
// 16 l .. 16 l + 15 (its quantization group), the rotated pairs sit in lanes
// 28-31.  x: the entry's 512 fp32 values (16-byte aligned, global or shared).
__device__ __forceinline__ void quantize_main_entry_warp(const float* x, const float* w, float eps, int rope,
                                                         const RopeTheta& th, double pos, uint8_t* codes_row,
                                                         uint8_t* scales_row, int lane) {
  float v[16];
  const float4* src = reinterpret_cast<const float4*>(x + lane * 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = src[i];
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
  if (w) {
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ss = fmaf(v[i], v[i], ss);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.0f / sqrtf(ss / (float)kDMain + eps);
    const float4* wv = reinterpret_cast<const float4*>(w + lane * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 g = wv[i];
      v[4 * i] = g.x * (v[4 * i] * inv);
      v[4 * i + 1] = g.y * (v[4 * i + 1] * inv);
      v[4 * i + 2] = g.z * (v[4 * i + 2] * inv);
      v[4 * i + 3] = g.w * (v[4 * i + 3] * inv);
    }
  }
  if (rope && lane * 16 >= kRopeFirst) {
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      float c, s;
      rope_cos_sin(th.t[(lane * 16 - kRopeFirst) / 2 + p], pos, c, s);
      rope_pair(v[2 * p], v[2 * p + 1], c, s);
    }
  }
  quantize_main_group_vals(v, codes_row + lane * 8, scales_row + lane);
}
void launch_quantize(const float* Cbar, const float* KI, int64_t n, const csa2_kv_planes* dst, const QDest& d,
                     cudaStream_t st, const csa2_norm_rope* nr);

}  // namespace csa2
