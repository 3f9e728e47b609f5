/*
 * Seeded, counter-based synthetic input generator.
 *
 * This header holds ONLY input synthesis: 64-bit counter-based random draws and
 * the conversions that turn them into the value distributions of the decode and
 * prefill workloads (N(0,1), U(0,1), their bf16 roundings, and an FP8 E4M3
 * rounding used to synthesise the sliding-window rows).  It holds none of the
 * arithmetic of the attention method: no quantizer of the cache format, no
 * pooling, no scoring, no selection, no attention.
 *
 * The same header is compiled by the host C build (synth_host.c) and by the
 * CUDA build (synth_dev.cu), so a value drawn on the host and on the device for
 * the same (seed, tensor id, element index) is bit-identical.  Every step is
 * integer arithmetic or an exactly rounded IEEE operation; no libm call whose
 * result could differ between machines is used.
 *
 * Definition (stated so that anyone can re-implement it):
 *   fmix64(z)  : z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27;
 *                z *= 0x94D049BB133111EB; z ^= z>>31            (SplitMix64 output mix)
 *   key(s, t)  : fmix64( fmix64(s + G) + (t + 1) * 0xD1B54A32D192ED03 ),  G = 0x9E3779B97F4A7C15
 *   u64(k, i)  : fmix64( k + (i + 1) * G )     (the (i+1)-th SplitMix64 output from state k)
 *   normal(k,i): the twelve 16-bit fields of u64(k,3i), u64(k,3i+1), u64(k,3i+2) summed to S;
 *                value = (S - 393210) / 65536, i.e. sum of twelve (u + 1/2)/65536 minus 6
 *                (Irwin-Hall, mean 0, variance 1, bounded by +-6); exact in fp32.
 *   uniform(k,i): (u64(k,i) >> 11) * 2^-53 in fp64, rounded to fp32 (nearest-even).
 */
#ifndef CSA2_SYNTH_CORE_H
#define CSA2_SYNTH_CORE_H

#include <stdint.h>
#include <string.h>
#include <math.h>

#ifdef __CUDACC__
#define SYN_FN __host__ __device__ static inline
#else
#define SYN_FN static inline
#endif

#define SYN_GAMMA 0x9E3779B97F4A7C15ULL
#define SYN_TGAMMA 0xD1B54A32D192ED03ULL

SYN_FN uint64_t syn_fmix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

SYN_FN uint64_t syn_key(uint64_t seed, uint64_t tid) {
  return syn_fmix64(syn_fmix64(seed + SYN_GAMMA) + (tid + 1ULL) * SYN_TGAMMA);
}

SYN_FN uint64_t syn_u64(uint64_t key, uint64_t i) {
  return syn_fmix64(key + (i + 1ULL) * SYN_GAMMA);
}

SYN_FN int32_t syn_fields16(uint64_t x) {
  return (int32_t)(x & 0xFFFFu) + (int32_t)((x >> 16) & 0xFFFFu) +
         (int32_t)((x >> 32) & 0xFFFFu) + (int32_t)(x >> 48);
}

/* N(0,1) by the Irwin-Hall sum of twelve 16-bit uniforms; exact in fp32. */
SYN_FN float syn_normal(uint64_t key, uint64_t i) {
  int32_t s = syn_fields16(syn_u64(key, 3 * i)) + syn_fields16(syn_u64(key, 3 * i + 1)) +
              syn_fields16(syn_u64(key, 3 * i + 2));
  return (float)(s - 393210) * (1.0f / 65536.0f);
}

/* U(0,1): 53 random bits as an fp64 in [0,1), rounded to fp32. */
SYN_FN float syn_uniform(uint64_t key, uint64_t i) {
  double d = (double)(syn_u64(key, i) >> 11) * (1.0 / 9007199254740992.0);
  return (float)d;
}

SYN_FN uint32_t syn_f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

/* fp32 -> bf16, round to nearest even (finite inputs). */
SYN_FN uint16_t syn_bf16_rne(float f) {
  uint32_t u = syn_f32_bits(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* fp32 -> FP8 E4M3 byte, round to nearest even, saturating at +-448.
 * Only used to synthesise sliding-window rows that are stored as FP8. */
SYN_FN uint8_t syn_e4m3_rne(float f) {
  uint32_t u = syn_f32_bits(f);
  uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
  float a = fabsf(f);
  if (a >= 464.0f) return (uint8_t)(sign | 0x7Eu);
  if (a < 0.015625f) { /* below 2^-6: subnormal grid of step 2^-9 */
    float q = rintf(a * 512.0f);
    return (uint8_t)(sign | (uint8_t)q);
  }
  int e = (int)((syn_f32_bits(a) >> 23) & 0xFFu) - 127; /* floor(log2 a), a normal */
  uint32_t pbits = (uint32_t)(127 + 3 - e) << 23;        /* 2^(3-e), e in [-6, 8] */
  float p;
  memcpy(&p, &pbits, 4);
  float scaled = a * p;                                  /* in [8,16), exact */
  int q = (int)rintf(scaled);
  if (q == 16) { q = 8; e += 1; }
  return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | (q - 8)));
}

#endif /* CSA2_SYNTH_CORE_H */
