/*
 * CSA2 ORACLE -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU restatement of what the CSA2 decode path
 * and its cache writer compute, written from the design description:
 *   [V41]  "DeepSeek-V4.1-Flash: pushing the limits of KV cache compression"
 *          section 2 (890 bytes/token), 4.1 (single-layer computation),
 *          4.2 (Full/Reindex/Reuse table), 4.3 (Hierarchical Sparse Indexer),
 *          5 (FP4 Main KV Cache).
 *   [CRS]  "DeepSeek-V4.1-Flash course, 02 Architecture", section 2.2 Eq. (1),
 *          2.3 CSA2, 2.3.1, 2.3.2 (Fig. 5), 2.4.4 FP4 main KV cache.
 *   [V4]   "DeepSeek-V4: Towards Highly Efficient Million-Token Context
 *          Intelligence", CSA step 1 (two-path overlapping compressor), step 2
 *          (lightning indexer, top-k) and step 3 (shared-KV MQA), the
 *          sliding-window branch, and HCA (m' tokens per entry, dense).
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this library.  It shares no code with the CUDA library: nothing here is
 * included from, or included by, the kernels.  Floating point is fp64 unless a
 * step of the cache format fixes fp32 (the quantizers' divisions, see below).
 * Build with -O2 -ffp-contract=off so no multiply-add is fused behind our back.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - E2M1 / E4M3 rounding is round-to-nearest with ties to the even code, and
 *    saturates at the largest finite magnitude (6 and 448).  A negative value
 *    that rounds to zero keeps its sign bit.
 *  - Main-KV scale: s = E4M3(fp32(amax / 6)); codes E2M1(fp32(x / s)); a zero
 *    scale gives all-zero codes.
 *  - Indexer-K scale (OCP MX rule): X = 2^(floor(log2 amax) - 2), clamped to
 *    [2^-127, 2^127]; codes E2M1(x / X); amax = 0 gives byte 0 and zero codes.
 *  - Nibble order: element 2i in the low nibble of byte i.
 *  - Top-k order: score descending, then entry index ascending; the output
 *    lists the chosen indices in ascending order, padded with -1.
 *  - Blocks of the hierarchical indexer are aligned at entry 0; a partial last
 *    block scores the entries it has.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D_MAIN 512
#define D_IDX 128
#define H_IDX 32
#define H_ATT 64
#define MAIN_GROUP 16
#define IDX_GROUP 32

/* ========================================================================== */
/* Element formats                                                            */
/* ========================================================================== */

/* FP4 E2M1 magnitudes by 3-bit code (OCP MX element format, as used by NVFP4):
 * [CRS] 2.4.4 and [V41] 5 give the largest magnitude 6 (= 448 x 6 / 448). */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double o_e2m1_value(int code) {
  double v = E2M1_MAG[code & 7];
  return (code & 8) ? -v : v;
}

/* Nearest E2M1 code; ties go to the even code; beyond 6 saturates to 6. */
int o_e2m1_encode(float x) {
  int sign = signbit(x) ? 8 : 0;
  if (isnan(x)) return sign | 7;
  double a = fabs((double)x);
  if (a >= 6.0) return sign | 7; /* saturate: nothing lies beyond the largest magnitude */
  int best = 0;
  double bd = a;
  for (int c = 1; c < 8; ++c) {
    double d = fabs(a - E2M1_MAG[c]);
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return sign | best;
}

/* FP8 E4M3 ("fn": no infinities, S.1111.111 is NaN), bias 7. */
double o_e4m3_value(int b) {
  int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^-6 */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Nearest finite E4M3 code (magnitudes of codes 0..126 increase with the code);
 * ties go to the even code; beyond 448 saturates to 448. */
int o_e4m3_encode(float x) {
  int sign = signbit(x) ? 0x80 : 0;
  if (isnan(x)) return 0x7F;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  int lo = 0, hi = 126; /* largest code with value <= a */
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (o_e4m3_value(mid) <= a)
      lo = mid;
    else
      hi = mid - 1;
  }
  int c = lo;
  if (c == 126) return sign | c;
  double dl = a - o_e4m3_value(c), du = o_e4m3_value(c + 1) - a;
  if (du < dl || (du == dl && ((c + 1) & 1) == 0)) c = c + 1;
  return sign | c;
}

/* E8M0 scale: 2^(b - 127); 255 is NaN. */
double o_e8m0_value(int b) {
  if (b == 255) return NAN;
  return ldexp(1.0, b - 127);
}

/* ========================================================================== */
/* Quantizers of the cache format ([V41] 2 and 5, [CRS] 2.4.4)                */
/* ========================================================================== */

/* Main KV: 512 channels, one E4M3 scale per 16 channels, E2M1 codes.
 * s_g = E4M3(amax/6);  xhat_i = s_g * E2M1(x_i / s_g).   288 bytes per entry. */
void o_quantize_main(const float* x, int64_t n, uint8_t* codes, uint8_t* scales) {
  for (int64_t r = 0; r < n; ++r) {
    const float* xr = x + r * D_MAIN;
    for (int g = 0; g < D_MAIN / MAIN_GROUP; ++g) {
      float amax = 0.0f;
      for (int i = 0; i < MAIN_GROUP; ++i) {
        float a = fabsf(xr[g * MAIN_GROUP + i]);
        if (a > amax) amax = a;
      }
      volatile float t = amax / 6.0f; /* fp32, correctly rounded */
      int sb = o_e4m3_encode(t);
      float s = (float)o_e4m3_value(sb);
      scales[r * 32 + g] = (uint8_t)sb;
      for (int i = 0; i < MAIN_GROUP; i += 2) {
        int c0 = 0, c1 = 0;
        if (s != 0.0f) {
          volatile float y0 = xr[g * MAIN_GROUP + i] / s;
          volatile float y1 = xr[g * MAIN_GROUP + i + 1] / s;
          c0 = o_e2m1_encode(y0);
          c1 = o_e2m1_encode(y1);
        }
        codes[r * 256 + (g * MAIN_GROUP + i) / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
  }
}

/* floor(log2 a) for a finite a > 0, exactly (frexp is exact). */
static int floor_log2(double a) {
  int e;
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
  return e - 1;
}

/* Indexer K: 128 elements, MXFP4 (OCP MX): one E8M0 scale per 32 elements,
 * shared exponent floor(log2 amax) - emax(E2M1) with emax = 2.  68 bytes. */
void o_quantize_index(const float* x, int64_t n, uint8_t* codes, uint8_t* scales) {
  for (int64_t r = 0; r < n; ++r) {
    const float* xr = x + r * D_IDX;
    for (int g = 0; g < D_IDX / IDX_GROUP; ++g) {
      float amax = 0.0f;
      for (int i = 0; i < IDX_GROUP; ++i) {
        float a = fabsf(xr[g * IDX_GROUP + i]);
        if (a > amax) amax = a;
      }
      int e = -127;
      if (amax > 0.0f) {
        e = floor_log2((double)amax) - 2;
        if (e < -127) e = -127;
        if (e > 127) e = 127;
      }
      scales[r * 4 + g] = (uint8_t)(e + 127);
      double X = ldexp(1.0, e);
      for (int i = 0; i < IDX_GROUP; i += 2) {
        int c0 = 0, c1 = 0;
        if (amax > 0.0f) {
          /* x / 2^e is exact in fp64 and, where a code can be nonzero, in fp32 */
          c0 = o_e2m1_encode((float)((double)xr[g * IDX_GROUP + i] / X));
          c1 = o_e2m1_encode((float)((double)xr[g * IDX_GROUP + i + 1] / X));
        }
        codes[r * 64 + (g * IDX_GROUP + i) / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
  }
}

void o_dequant_main(const uint8_t* codes, const uint8_t* scales, int64_t n, double* out) {
  for (int64_t r = 0; r < n; ++r)
    for (int c = 0; c < D_MAIN; ++c) {
      int byte = codes[r * 256 + c / 2];
      int code = (c & 1) ? (byte >> 4) : (byte & 15);
      out[r * D_MAIN + c] = o_e2m1_value(code) * o_e4m3_value(scales[r * 32 + c / MAIN_GROUP]);
    }
}

void o_dequant_index(const uint8_t* codes, const uint8_t* scales, int64_t n, double* out) {
  for (int64_t r = 0; r < n; ++r)
    for (int c = 0; c < D_IDX; ++c) {
      int byte = codes[r * 64 + c / 2];
      int code = (c & 1) ? (byte >> 4) : (byte & 15);
      out[r * D_IDX + c] = o_e2m1_value(code) * o_e8m0_value(scales[r * 4 + c / IDX_GROUP]);
    }
}

/* Distance, relative to the value, of one input to the nearest rounding decision
 * point of the main-KV quantizer of its group (scale rounding and element
 * rounding).  Used by tests to separate groups whose bytes are fixed by the
 * mathematics from groups that sit on a rounding boundary.  x: 16 values. */
double o_main_group_margin(const double* x) {
  static const double MID[7] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0};
  double amax = 0.0;
  for (int i = 0; i < MAIN_GROUP; ++i)
    if (fabs(x[i]) > amax) amax = fabs(x[i]);
  if (amax == 0.0) return INFINITY;
  double t = amax / 6.0, margin = INFINITY;
  /* scale rounding: midpoints between adjacent finite E4M3 magnitudes */
  for (int c = 0; c < 126; ++c) {
    double mid = 0.5 * (o_e4m3_value(c) + o_e4m3_value(c + 1));
    double d = fabs(t - mid) / t;
    if (d < margin) margin = d;
  }
  int sb = o_e4m3_encode((float)t);
  double s = o_e4m3_value(sb);
  if (s == 0.0) return margin;
  for (int i = 0; i < MAIN_GROUP; ++i) {
    double y = fabs(x[i]) / s;
    if (y == 0.0) continue;
    for (int k = 0; k < 7; ++k) {
      double d = fabs(y - MID[k]) / y;
      if (d < margin) margin = d;
    }
  }
  return margin;
}

/* Same for the indexer-K quantizer: the power-of-two boundary of amax and the
 * element midpoints.  x: 32 values. */
double o_index_group_margin(const double* x) {
  static const double MID[7] = {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0};
  double amax = 0.0;
  for (int i = 0; i < IDX_GROUP; ++i)
    if (fabs(x[i]) > amax) amax = fabs(x[i]);
  if (amax == 0.0) return INFINITY;
  int e = floor_log2(amax);
  double lo = ldexp(1.0, e), hi = ldexp(1.0, e + 1);
  double margin = fmin((amax - lo) / amax, (hi - amax) / amax);
  int es = e - 2;
  if (es < -127) es = -127;
  double X = ldexp(1.0, es);
  for (int i = 0; i < IDX_GROUP; ++i) {
    double y = fabs(x[i]) / X;
    if (y == 0.0) continue;
    for (int k = 0; k < 7; ++k) {
      double d = fabs(y - MID[k]) / y;
      if (d < margin) margin = d;
    }
  }
  return margin;
}

/* ========================================================================== */
/* Q/KV RMSNorm and partial RoPE ([V4] CSA, "other details": RMSNorm of every  */
/* query head and of each compressed entry before the core attention; RoPE on */
/* the last 64 channels of query, KV and output)                              */
/* ========================================================================== */

#define ROPE_DIMS 64
#define ROPE_FIRST (D_MAIN - ROPE_DIMS)

/* y = w * x / sqrt(mean(x^2) + eps) over n channels (w = NULL: all ones) */
void o_rmsnorm(const double* x, int n, const float* w, double eps, double* y) {
  double ss = 0.0;
  for (int c = 0; c < n; ++c) ss += x[c] * x[c];
  const double inv = 1.0 / sqrt(ss / n + eps);
  for (int c = 0; c < n; ++c) y[c] = (w ? (double)w[c] : 1.0) * x[c] * inv;
}

/* Rotates the last 64 channels of a 512-vector in place by position pos: pair
 * i, channels (448 + 2i, 449 + 2i), turns by the angle pos * base^(-2i/64). */
void o_rope(double* x, double pos, double base) {
  for (int i = 0; i < ROPE_DIMS / 2; ++i) {
    const double theta = pos * pow(base, -2.0 * i / ROPE_DIMS);
    const double c = cos(theta), s = sin(theta);
    double* v = x + ROPE_FIRST + 2 * i;
    const double a = v[0], b = v[1];
    v[0] = a * c - b * s;
    v[1] = a * s + b * c;
  }
}

/* One sliding-window row ([V4] sliding-window branch; [CRS] 2.4.4: the window
 * stays FP8): RMSNorm (w, or none when NULL), RoPE at pos (rope), then E4M3 of
 * the value rounded to fp32 (nearest even, saturating at 448, no scale).
 * pre (or NULL) gets the values before the encoding. */
void o_swa_row(const double* x, const float* w, double eps, int rope, double base, double pos,
               uint8_t* out, double* pre) {
  double y[D_MAIN];
  if (w)
    o_rmsnorm(x, D_MAIN, w, eps, y);
  else
    memcpy(y, x, sizeof(y));
  if (rope) o_rope(y, pos, base);
  for (int c = 0; c < D_MAIN; ++c) out[c] = (uint8_t)o_e4m3_encode((float)y[c]);
  if (pre) memcpy(pre, y, sizeof(y));
}

/* ========================================================================== */
/* Compressor / cache write ([CRS] Eq. (1) and 2.3; [V41] 4.1)                */
/* ========================================================================== */

static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* C = H W_KV, Z = H W_Z (fp64 sums); each non-overlapping group B_j of m tokens
 * pools per channel as  Cbar_j[c] = sum_i softmax_i(Z_i[c]) C_i[c];  the
 * indexer key is K^I_j = Cbar_j W_IK; both are quantized into the entry. */
typedef struct {
  const uint16_t *H, *Wkv, *Wz, *Wik;
  int64_t T;
  int d, m;
  uint8_t *kvc, *kvs, *ixc, *ixs;
  double *cbar_out, *ki_out, *att_out;
  const float* norm_w; /* RMSNorm weight of the attention copy, or NULL: no RMSNorm */
  double eps;
  int rope;
  double rope_base, pos_first, pos_step;
  int64_t j_lo, j_hi;
} cw_job;

static void cache_write_range(const cw_job* jb) {
  int d = jb->d, m = jb->m;
  double* C = (double*)malloc(sizeof(double) * (size_t)m * D_MAIN);
  double* Z = (double*)malloc(sizeof(double) * (size_t)m * D_MAIN);
  double* Wkv = (double*)malloc(sizeof(double) * (size_t)d * D_MAIN);
  double* Wz = (double*)malloc(sizeof(double) * (size_t)d * D_MAIN);
  double cbar[D_MAIN], ki[D_IDX], att[D_MAIN];
  float cbar32[D_MAIN], ki32[D_IDX];
  for (int64_t i = 0; i < (int64_t)d * D_MAIN; ++i) {
    Wkv[i] = bf16_value(jb->Wkv[i]);
    Wz[i] = bf16_value(jb->Wz[i]);
  }
  for (int64_t j = jb->j_lo; j < jb->j_hi; ++j) {
    for (int r = 0; r < m; ++r) {
      const uint16_t* h = jb->H + ((size_t)j * m + r) * d;
      double* cr = C + (size_t)r * D_MAIN;
      double* zr = Z + (size_t)r * D_MAIN;
      for (int c = 0; c < D_MAIN; ++c) cr[c] = zr[c] = 0.0;
      for (int k = 0; k < d; ++k) {
        double hv = bf16_value(h[k]);
        if (hv == 0.0) continue;
        const double* wk = Wkv + (size_t)k * D_MAIN;
        const double* wz = Wz + (size_t)k * D_MAIN;
        for (int c = 0; c < D_MAIN; ++c) {
          cr[c] += hv * wk[c];
          zr[c] += hv * wz[c];
        }
      }
    }
    for (int c = 0; c < D_MAIN; ++c) {
      double zmax = -INFINITY;
      for (int r = 0; r < m; ++r)
        if (Z[(size_t)r * D_MAIN + c] > zmax) zmax = Z[(size_t)r * D_MAIN + c];
      double num = 0.0, den = 0.0;
      for (int r = 0; r < m; ++r) {
        double e = exp(Z[(size_t)r * D_MAIN + c] - zmax);
        num += e * C[(size_t)r * D_MAIN + c];
        den += e;
      }
      cbar[c] = num / den;
    }
    for (int o = 0; o < D_IDX; ++o) {
      double s = 0.0;
      for (int c = 0; c < D_MAIN; ++c) s += cbar[c] * bf16_value(jb->Wik[(size_t)c * D_IDX + o]);
      ki[o] = s;
    }
    /* the attention copy: RMSNorm, then RoPE at the entry's position, then the
     * FP4 quantization ([V41] 2.4.4: the cache is quantized after RoPE); the
     * indexer key keeps the pooled latent */
    if (jb->norm_w)
      o_rmsnorm(cbar, D_MAIN, jb->norm_w, jb->eps, att);
    else
      memcpy(att, cbar, sizeof(att));
    if (jb->rope) o_rope(att, jb->pos_first + (double)j * jb->pos_step, jb->rope_base);
    for (int c = 0; c < D_MAIN; ++c) cbar32[c] = (float)att[c];
    for (int o = 0; o < D_IDX; ++o) ki32[o] = (float)ki[o];
    o_quantize_main(cbar32, 1, jb->kvc + j * 256, jb->kvs + j * 32);
    o_quantize_index(ki32, 1, jb->ixc + j * 64, jb->ixs + j * 4);
    if (jb->cbar_out) memcpy(jb->cbar_out + j * D_MAIN, cbar, sizeof(cbar));
    if (jb->ki_out) memcpy(jb->ki_out + j * D_IDX, ki, sizeof(ki));
    if (jb->att_out) memcpy(jb->att_out + j * D_MAIN, att, sizeof(att));
  }
  free(C);
  free(Z);
  free(Wkv);
  free(Wz);
}

static void* cache_write_worker(void* p) {
  cache_write_range((const cw_job*)p);
  return NULL;
}

/* Writes entries 0 .. T/m - 1 into the four planes (T must be a multiple of m).
 * norm_w (or NULL), eps, rope, rope_base: RMSNorm and RoPE of the main-KV copy;
 * entry j sits at position pos_first + j * pos_step.  att_out (or NULL) gets
 * the values the main quantizer saw. */
int o_cache_write(const uint16_t* H, int64_t T, int d, const uint16_t* Wkv, const uint16_t* Wz,
                  const uint16_t* Wik, int m, uint8_t* kv_codes, uint8_t* kv_scales,
                  uint8_t* ix_codes, uint8_t* ix_scales, double* cbar_out, double* ki_out,
                  int nthreads, const float* norm_w, double eps, int rope, double rope_base,
                  double pos_first, double pos_step, double* att_out) {
  if (m < 1 || T % m != 0 || d < 1) return 1;
  int64_t n = T / m;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 128) nthreads = 128;
  if (nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  pthread_t th[128];
  cw_job jobs[128];
  int64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    cw_job jb = {H,        Wkv,   Wz,       Wik,        T,         d,         m,
                 kv_codes, kv_scales, ix_codes, ix_scales, cbar_out, ki_out, att_out,
                 norm_w,   eps,   rope,     rope_base,  pos_first, pos_step,
                 (int64_t)t * per, (int64_t)(t + 1) * per};
    if (jb.j_hi > n) jb.j_hi = n;
    jobs[t] = jb;
  }
  for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, cache_write_worker, &jobs[t]);
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  return 0;
}

/* Softmax pooling alone, for tests: C, Z fp64 [T, width]; out [T/m, width]. */
void o_pool(const double* C, const double* Z, int64_t T, int width, int m, double* out) {
  for (int64_t j = 0; j < T / m; ++j)
    for (int c = 0; c < width; ++c) {
      double zmax = -INFINITY;
      for (int r = 0; r < m; ++r)
        if (Z[(j * m + r) * width + c] > zmax) zmax = Z[(j * m + r) * width + c];
      double num = 0.0, den = 0.0;
      for (int r = 0; r < m; ++r) {
        double e = exp(Z[(j * m + r) * width + c] - zmax);
        num += e * C[(j * m + r) * width + c];
        den += e;
      }
      out[j * width + c] = num / den;
    }
}

/* ========================================================================== */
/* V4 compressors ([V4] CSA step 1: two paths with overlapping blocks; HCA:   */
/* one path, m' tokens per entry).  Position biases B join the scores before  */
/* the per-channel softmax over the rows an entry draws from.                */
/* ========================================================================== */

typedef struct {
  const uint16_t *H, *W;
  int64_t r_lo, r_hi;
  int d, width;
  double* out;
} proj_job;

static void* project_worker(void* p) {
  const proj_job* jb = (const proj_job*)p;
  int d = jb->d, w = jb->width;
  double* W = (double*)malloc(sizeof(double) * (size_t)d * w);
  for (int64_t i = 0; i < (int64_t)d * w; ++i) W[i] = bf16_value(jb->W[i]);
  for (int64_t r = jb->r_lo; r < jb->r_hi; ++r) {
    double* o = jb->out + r * w;
    for (int c = 0; c < w; ++c) o[c] = 0.0;
    for (int k = 0; k < d; ++k) {
      double hv = bf16_value(jb->H[r * d + k]);
      if (hv == 0.0) continue;
      const double* wk = W + (size_t)k * w;
      for (int c = 0; c < w; ++c) o[c] += hv * wk[c];
    }
  }
  free(W);
  return NULL;
}

/* out [T][width] = H [T][d] W [d][width], bf16 operands, fp64 sums */
void o_project(const uint16_t* H, int64_t T, int d, int width, const uint16_t* W, double* out, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 128) nthreads = 128;
  if (nthreads > T) nthreads = (int)(T > 0 ? T : 1);
  pthread_t th[128];
  proj_job jobs[128];
  int64_t per = (T + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    proj_job jb = {H, W, (int64_t)t * per, (int64_t)(t + 1) * per, d, width, out};
    if (jb.r_hi > T) jb.r_hi = T;
    if (jb.r_lo > T) jb.r_lo = T;
    jobs[t] = jb;
  }
  for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, project_worker, &jobs[t]);
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* Overlapping pool.  Entry i draws from rows m i .. m i + m - 1 of path a
 * (scores Za + Ba[r]) and rows m (i - 1) .. m i - 1 of path b (scores
 * Zb + Bb[r]); per channel the 2m scores go through one softmax and weight
 * their rows of Ca / Cb.  Entry 0 has no previous block: its path-b rows count
 * as score -inf and value 0, i.e. they drop out.  C*, Z* fp64 [T][width];
 * B* fp32 [m][width]; out [T/m][width]. */
void o_pool_overlap(const double* Ca, const double* Za, const double* Cb, const double* Zb,
                    const float* Ba, const float* Bb, int64_t T, int width, int m, double* out) {
  for (int64_t i = 0; i < T / m; ++i)
    for (int c = 0; c < width; ++c) {
      double zmax = -INFINITY;
      for (int r = 0; r < m; ++r) {
        double z = Za[(i * m + r) * width + c] + (double)Ba[r * width + c];
        if (z > zmax) zmax = z;
      }
      if (i > 0)
        for (int r = 0; r < m; ++r) {
          double z = Zb[((i - 1) * m + r) * width + c] + (double)Bb[r * width + c];
          if (z > zmax) zmax = z;
        }
      double num = 0.0, den = 0.0;
      for (int r = 0; r < m; ++r) {
        int64_t row = (i * m + r) * width + c;
        double e = exp(Za[row] + (double)Ba[r * width + c] - zmax);
        num += e * Ca[row];
        den += e;
      }
      if (i > 0)
        for (int r = 0; r < m; ++r) {
          int64_t row = ((i - 1) * m + r) * width + c;
          double e = exp(Zb[row] + (double)Bb[r * width + c] - zmax);
          num += e * Cb[row];
          den += e;
        }
      out[i * width + c] = num / den;
    }
}

/* HCA pool: entry i = per-channel softmax over rows m i .. m i + m - 1 of
 * Z + B[r], weighting the same rows of C. */
void o_pool_bias(const double* C, const double* Z, const float* Bp, int64_t T, int width, int m,
                 double* out) {
  for (int64_t i = 0; i < T / m; ++i)
    for (int c = 0; c < width; ++c) {
      double zmax = -INFINITY;
      for (int r = 0; r < m; ++r) {
        double z = Z[(i * m + r) * width + c] + (double)Bp[r * width + c];
        if (z > zmax) zmax = z;
      }
      double num = 0.0, den = 0.0;
      for (int r = 0; r < m; ++r) {
        int64_t row = (i * m + r) * width + c;
        double e = exp(Z[row] + (double)Bp[r * width + c] - zmax);
        num += e * C[row];
        den += e;
      }
      out[i * width + c] = num / den;
    }
}

/* The two compressors end to end: projections of H, then the pool.  Returns 1
 * when T is not a multiple of m (or an allocation fails). */
int o_compress_overlap(const uint16_t* H, int64_t T, int d, int width, const uint16_t* Wa_kv,
                       const uint16_t* Wb_kv, const uint16_t* Wa_z, const uint16_t* Wb_z, const float* Ba,
                       const float* Bb, int m, double* out, int nthreads) {
  if (m < 1 || d < 1 || width < 1 || T < 0 || T % m != 0) return 1;
  size_t sz = sizeof(double) * (size_t)(T > 0 ? T : 1) * width;
  double *Ca = (double*)malloc(sz), *Za = (double*)malloc(sz), *Cb = (double*)malloc(sz),
         *Zb = (double*)malloc(sz);
  int rc = 1;
  if (Ca && Za && Cb && Zb) {
    o_project(H, T, d, width, Wa_kv, Ca, nthreads);
    o_project(H, T, d, width, Wa_z, Za, nthreads);
    o_project(H, T, d, width, Wb_kv, Cb, nthreads);
    o_project(H, T, d, width, Wb_z, Zb, nthreads);
    o_pool_overlap(Ca, Za, Cb, Zb, Ba, Bb, T, width, m, out);
    rc = 0;
  }
  free(Ca);
  free(Za);
  free(Cb);
  free(Zb);
  return rc;
}

int o_compress_hca(const uint16_t* H, int64_t T, int d, int width, const uint16_t* Wkv, const uint16_t* Wz,
                   const float* Bp, int m, double* out, int nthreads) {
  if (m < 1 || d < 1 || width < 1 || T < 0 || T % m != 0) return 1;
  size_t sz = sizeof(double) * (size_t)(T > 0 ? T : 1) * width;
  double *C = (double*)malloc(sz), *Z = (double*)malloc(sz);
  int rc = 1;
  if (C && Z) {
    o_project(H, T, d, width, Wkv, C, nthreads);
    o_project(H, T, d, width, Wz, Z, nthreads);
    o_pool_bias(C, Z, Bp, T, width, m, out);
    rc = 0;
  }
  free(C);
  free(Z);
  return rc;
}

/* ========================================================================== */
/* Lightning indexer score ([V4] CSA step 2; [V41] 4.1)                      */
/*   I_j = sum_h w_h * ReLU(q_h . K^I_j)   over 32 heads of dimension 128      */
/* ========================================================================== */

static void score_one(const uint8_t* codes, const uint8_t* scales, const double* q,
                      const double* w, double* out) {
  double k[D_IDX];
  for (int c = 0; c < D_IDX; ++c) {
    int byte = codes[c / 2];
    int code = (c & 1) ? (byte >> 4) : (byte & 15);
    k[c] = o_e2m1_value(code) * o_e8m0_value(scales[c / IDX_GROUP]);
  }
  double s = 0.0;
  for (int h = 0; h < H_IDX; ++h) {
    double dot = 0.0;
    for (int c = 0; c < D_IDX; ++c) dot += q[h * D_IDX + c] * k[c];
    s += w[h] * (dot > 0.0 ? dot : 0.0);
  }
  *out = s;
}

typedef struct {
  const uint8_t *codes, *scales;
  const double *q, *w;
  double* scores;
  int64_t lo, hi;
} sc_job;

static void* score_worker(void* p) {
  const sc_job* j = (const sc_job*)p;
  for (int64_t e = j->lo; e < j->hi; ++e)
    score_one(j->codes + e * 64, j->scales + e * 4, j->q, j->w, j->scores + e);
  return NULL;
}

/* Scores of entries 0..n-1 of one sequence's indexer planes.
 * q_bf16: [32,128] bf16 bit patterns; w: [32] fp32. */
void o_index_scores(const uint8_t* ix_codes, const uint8_t* ix_scales, int64_t n,
                    const uint16_t* q_bf16, const float* w, double* scores, int nthreads) {
  double q[H_IDX * D_IDX], wd[H_IDX];
  for (int i = 0; i < H_IDX * D_IDX; ++i) q[i] = bf16_value(q_bf16[i]);
  for (int h = 0; h < H_IDX; ++h) wd[h] = (double)w[h];
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 128) nthreads = 128;
  if (n < 4096) nthreads = 1;
  pthread_t th[128];
  sc_job jobs[128];
  int64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    sc_job jb = {ix_codes, ix_scales, q, wd, scores, (int64_t)t * per, (int64_t)(t + 1) * per};
    if (jb.hi > n) jb.hi = n;
    if (jb.lo > n) jb.lo = n;
    jobs[t] = jb;
  }
  if (nthreads == 1) {
    score_worker(&jobs[0]);
    return;
  }
  for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, score_worker, &jobs[t]);
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* Scores of selected entries (idx[i] < 0 gives -inf). */
void o_index_scores_at(const uint8_t* ix_codes, const uint8_t* ix_scales, const int64_t* idx,
                       int64_t count, const uint16_t* q_bf16, const float* w, double* scores) {
  double q[H_IDX * D_IDX], wd[H_IDX];
  for (int i = 0; i < H_IDX * D_IDX; ++i) q[i] = bf16_value(q_bf16[i]);
  for (int h = 0; h < H_IDX; ++h) wd[h] = (double)w[h];
  for (int64_t i = 0; i < count; ++i) {
    if (idx[i] < 0) {
      scores[i] = -INFINITY;
      continue;
    }
    score_one(ix_codes + idx[i] * 64, ix_scales + idx[i] * 4, q, wd, scores + i);
  }
}

/* ========================================================================== */
/* Selection ([V4] CSA step 2 top-k; [V41] 4.3 and [CRS] 2.3.2 hierarchy)     */
/* ========================================================================== */

typedef struct {
  double s;
  int64_t i;
} keyed;

/* score descending, then index ascending */
static int cmp_keyed(const void* a, const void* b) {
  const keyed *x = (const keyed*)a, *y = (const keyed*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->i > y->i) - (x->i < y->i);
}

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* Top-k of the candidates idx[0..count) by (score desc, index asc); writes the
 * chosen indices ascending into out[0..k), -1 padded.  Returns the number chosen. */
static int topk_of(const double* scores_by_cand, const int64_t* idx, int64_t count, int k,
                   int32_t* out) {
  keyed* v = (keyed*)malloc(sizeof(keyed) * (size_t)(count > 0 ? count : 1));
  for (int64_t c = 0; c < count; ++c) {
    v[c].s = scores_by_cand[c];
    v[c].i = idx[c];
  }
  qsort(v, (size_t)count, sizeof(keyed), cmp_keyed);
  int took = (int)(count < k ? count : k);
  for (int t = 0; t < took; ++t) out[t] = (int32_t)v[t].i;
  qsort(out, (size_t)took, sizeof(int32_t), cmp_i32);
  for (int t = took; t < k; ++t) out[t] = -1;
  free(v);
  return took;
}

/* FLAT: top-k over entries 0..n-1. */
int o_topk(const double* scores, int64_t n, int k, int32_t* out) {
  int64_t* idx = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
  for (int64_t j = 0; j < n; ++j) idx[j] = j;
  int r = topk_of(scores, idx, n, k, out);
  free(idx);
  return r;
}

/* s_b = max of the scores of block b = [blk*b, blk*b + blk) within [0, n). */
void o_block_max(const double* scores, int64_t n, int blk, double* bmax) {
  int64_t nb = (n + blk - 1) / blk;
  for (int64_t b = 0; b < nb; ++b) {
    double m = -INFINITY;
    for (int64_t j = b * blk; j < (b + 1) * blk && j < n; ++j)
      if (scores[j] > m) m = scores[j];
    bmax[b] = m;
  }
}

/* Candidate pool: the top `keep` blocks by (block max desc, block index asc),
 * listed ascending, -1 padded to `keep`.  Returns the number of blocks kept. */
int o_hier_pool(const double* bmax, int64_t nb, int keep, int32_t* pool) {
  return o_topk(bmax, nb, keep, pool);
}

/* Top-k over the entries of the pool's blocks (entries < n).  scores: all n. */
int o_pool_topk(const double* scores, int64_t n, const int32_t* pool, int keep, int blk, int k,
                int32_t* out) {
  int64_t* idx = (int64_t*)malloc(sizeof(int64_t) * (size_t)keep * blk + 1);
  double* s = (double*)malloc(sizeof(double) * (size_t)keep * blk + 1);
  int64_t cnt = 0;
  for (int p = 0; p < keep; ++p) {
    if (pool[p] < 0) continue;
    for (int t = 0; t < blk; ++t) {
      int64_t j = (int64_t)pool[p] * blk + t;
      if (j >= n) break;
      idx[cnt] = j;
      s[cnt] = scores[j];
      ++cnt;
    }
  }
  int r = topk_of(s, idx, cnt, k, out);
  free(idx);
  free(s);
  return r;
}

/* ========================================================================== */
/* Sparse MQA over the selected entries plus the sliding window               */
/* ([V4] CSA step 3 and the sliding-window branch; [V41] 4.1)                 */
/*   X = [dequant(main KV rows of topk) ; E4M3 SWA rows],  K = V = X,          */
/*   o_h = sum_s softmax_s(scale * q_h . X_s) X_s                               */
/* ========================================================================== */

/* kv planes of one sequence; topk [k] (entries < 0 are skipped);
 * swa [n_swa,512] E4M3 bytes; q [64,512] bf16; out [64,512]; lse [64] (natural
 * log of the softmax denominator of the scaled logits, incl. the max).
 * Extras ([V4] CSA, "other details"), each off when NULL / 0:
 *   q_norm_w [512]: RMSNorm of every query head (eps) before the logits;
 *   rope: RoPE of the query's last 64 channels at position qpos (base), and of
 *     the output at position -qpos (the cached entries carry their own);
 *   sink [64]: per-head logit z'_h whose exp joins the softmax denominator
 *     (and lse).
 * o_attention_rows takes the rows X [rows,512] (fp64) directly. */
void o_attention_rows(const double* X, int rows, const uint16_t* q_bf16, double scale,
                      const float* q_norm_w, double eps, int rope, double rope_base, double qpos,
                      const float* sink, double* out, double* lse) {
  double* logit = (double*)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1));
  for (int h = 0; h < H_ATT; ++h) {
    double q[D_MAIN];
    for (int c = 0; c < D_MAIN; ++c) q[c] = bf16_value(q_bf16[h * D_MAIN + c]);
    if (q_norm_w) o_rmsnorm(q, D_MAIN, q_norm_w, eps, q);
    if (rope) o_rope(q, qpos, rope_base);
    double mx = -INFINITY;
    for (int s = 0; s < rows; ++s) {
      double dot = 0.0;
      for (int c = 0; c < D_MAIN; ++c) dot += q[c] * X[(size_t)s * D_MAIN + c];
      logit[s] = scale * dot;
      if (logit[s] > mx) mx = logit[s];
    }
    /* the sink joins the denominator: sum_s exp(l_s) + exp(z'_h), kept relative
     * to the larger of the logits' maximum and z'_h */
    const double z = sink ? (double)sink[h] : -INFINITY;
    const double ref = (rows > 0 && mx > z) ? mx : z;
    double den = 0.0;
    for (int s = 0; s < rows; ++s) den += exp(logit[s] - ref);
    if (sink) den += exp(z - ref);
    for (int c = 0; c < D_MAIN; ++c) out[h * D_MAIN + c] = 0.0;
    for (int s = 0; s < rows; ++s) {
      double p = exp(logit[s] - ref) / den;
      for (int c = 0; c < D_MAIN; ++c) out[h * D_MAIN + c] += p * X[(size_t)s * D_MAIN + c];
    }
    if (rope) o_rope(out + h * D_MAIN, -qpos, rope_base);
    if (lse) lse[h] = (rows > 0 || sink) ? ref + log(den) : -INFINITY;
  }
  free(logit);
}

/* The same over dequantized cache rows: the selected main entries, then the
 * window rows. */
void o_attention_ex(const uint8_t* kv_codes, const uint8_t* kv_scales, const int32_t* topk, int k,
                    const uint8_t* swa, int n_swa, const uint16_t* q_bf16, double scale,
                    const float* q_norm_w, double eps, int rope, double rope_base, double qpos,
                    const float* sink, double* out, double* lse) {
  int rows = 0;
  for (int i = 0; i < k; ++i)
    if (topk[i] >= 0) ++rows;
  rows += n_swa;
  double* X = (double*)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1) * D_MAIN);
  int r = 0;
  for (int i = 0; i < k; ++i) {
    if (topk[i] < 0) continue;
    o_dequant_main(kv_codes + (int64_t)topk[i] * 256, kv_scales + (int64_t)topk[i] * 32, 1,
                   X + (size_t)r * D_MAIN);
    ++r;
  }
  for (int i = 0; i < n_swa; ++i, ++r)
    for (int c = 0; c < D_MAIN; ++c) X[(size_t)r * D_MAIN + c] = o_e4m3_value(swa[i * D_MAIN + c]);
  o_attention_rows(X, rows, q_bf16, scale, q_norm_w, eps, rope, rope_base, qpos, sink, out, lse);
  free(X);
}

void o_attention(const uint8_t* kv_codes, const uint8_t* kv_scales, const int32_t* topk, int k,
                 const uint8_t* swa, int n_swa, const uint16_t* q_bf16, double scale,
                 double* out, double* lse) {
  o_attention_ex(kv_codes, kv_scales, topk, k, swa, n_swa, q_bf16, scale, NULL, 0.0, 0, 0.0, 0.0,
                 NULL, out, lse);
}

/* ========================================================================== */
/* Array forms of the element encoders (for exhaustive checks in tests)       */
/* ========================================================================== */

void o_e2m1_encode_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)o_e2m1_encode(x[i]);
}

void o_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)o_e4m3_encode(x[i]);
}
