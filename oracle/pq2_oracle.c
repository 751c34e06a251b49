/*
 * pq2_oracle.c — plain, slow CPU oracle for the ternary (PQ2) x INT8 matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header or table with the CUDA library.
 *
 * Build: gcc -O2 -std=c11 -fno-fast-math -ffp-contract=off -fPIC -shared
 * (no FMA contraction, IEEE single/double, round-to-nearest-even mode).
 *
 * Sources (page "Kernel experiments: recorded evidence", abbreviated KE, and
 * page "Baseline and the integer breakthrough", abbreviated BIB):
 *   - block format: KE, Test 1 ("Packed loading, unpacking and scheduling"),
 *     Diagram 1 and the prepare_pq2 listing: 34-byte blocks, fp16 scale in
 *     bytes 0-1, then 32 code bytes; weight k of a group sits in bits
 *     2(k%4)..2(k%4)+1 of code byte k/4.
 *   - decode: KE Test 1 slow path of _expand_byte: code c means c-1.
 *   - quantiser: KE Test 6 (_quantize listing) and BIB "Calculate with small
 *     integers", step 1: per 128-group scale = max|x|/127 in fp32, IEEE
 *     division by (scale>0 ? scale : 1), round half to even, clamp to +-127.
 *   - group dot and scale: BIB steps 3-4: 32 DP4A per 128-group in int32,
 *     then multiply by (activation scale x weight scale) once per group and
 *     accumulate across groups in fp32.
 *   - plane order of q and per-group sum of q: KE Test 21 ("Masked-plane
 *     Triton small-batch MMA", Diagram 7 and the plane-order quantisation
 *     listing): element i of a group is stored at (i%4)*32 + i/4, and
 *     T = sum of q removes the -1 offset of the codes once per group.
 *   - gated output of a gate/up projection: KE Test 12 ("Single-token
 *     geometry, PRMT, chaining and fusion screens"), the "activated" and
 *     gated-fusion calls: the projection's output is split in halves along
 *     the output dimension, gate first, and the result is silu(gate) * up,
 *     with silu(v) = v * sigmoid(v) = v / (1 + e^-v).
 *   - smaller activation groups: KE Test 9 ("Smaller Q8 activation groups"):
 *     the activations get one scale per A = 64 or 32 elements, the weights
 *     keep their 128-groups and scales; each 128-group's dot splits into
 *     128/A partial dots, each scaled by its own activation scale.
 *   - fused preparation of the activations: KE Test 18 ("RMSNorm + Hadamard
 *     + Q8 fusion"): h = x (+ residual) in fp32; the sum of h^2 over the row
 *     kept in 2048 strided partial sums, then summed; inv = 1/sqrt(mean +
 *     eps); normalised = bf16((h * inv) * (w + 1)); v = normalised * sign;
 *     a 1024-point Walsh-Hadamard transform; bf16; then the group-128 INT8
 *     quantiser above.
 *   - PTQ1_0 weights: page "KERNEL_REPORT: PTQ1_0 small-batch decoding on the
 *     PrismML fork, RTX 3060 12GB" (abbreviated KR), "What the source said":
 *     a 28-byte block per 128 weights; 24 qs bytes of five trits each,
 *     unpacked by repeatedly multiplying by 3 (a 16-bit lane) and taking the
 *     part above the low byte; qh, two bytes holding the other 8 trits; the
 *     fp16 scale d in the last two bytes; trit t means weight t - 1.  The
 *     page does not say which trit is which weight; the reading taken here:
 *     trit n of qs byte j is weight 24n + j, trit n (n < 4) of qh byte j is
 *     weight 120 + 2n + j.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <fenv.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORC_GROUP 128
#define ORC_BLOCK_BYTES 34

/* ---------------------------------------------------------------- scalars */

/* One 2-bit field of a code byte decoded to its signed weight: c - 1.
 * KE Test 1, slow path of _expand_byte: ((p >> 2i) & 3) - 1. */
int orc_decode_field(uint8_t byte, int field) {
  return (int)((byte >> (2 * field)) & 3u) - 1;
}

/* IEEE-754 binary16 -> binary32, written from the format definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits).
 * Every binary16 value is exactly representable in binary32. */
float orc_half_to_float(uint16_t h) {
  uint32_t sign = (uint32_t)(h >> 15) & 1u;
  uint32_t expo = (uint32_t)(h >> 10) & 0x1fu;
  uint32_t frac = (uint32_t)h & 0x3ffu;
  double mag;
  if (expo == 0x1f) {
    mag = frac ? NAN : INFINITY;
  } else if (expo == 0) {
    mag = ldexp((double)frac, -24);             /* subnormal: frac * 2^-24 */
  } else {
    mag = ldexp((double)(frac | 0x400u), (int)expo - 25); /* 1.frac * 2^(e-15) */
  }
  float f = (float)mag;
  return sign ? -f : f;
}

/* bfloat16 -> binary32: the bf16 bits are the top half of a binary32. */
float orc_bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* binary32 -> bfloat16 with round to nearest, ties to even (finite inputs). */
uint16_t orc_float_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint32_t lower = u & 0xffffu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

/* ------------------------------------------------------------- preparation */

/* Split raw blocks into a code plane and a scale plane (pure byte move).
 * KE Test 1 prepare_pq2 (separate=True) and Test 4: the prepared matrix keeps
 * exactly 34 bytes per 128 weights, codes first, then fp16 scales.
 *   raw    : N rows, row stride raw_stride bytes, K/128 blocks of 34 bytes
 *   codes  : [N][K/4] bytes
 *   scales : [N][K/128] fp16 bit patterns */
void orc_prepare(const uint8_t *raw, int64_t raw_stride, int64_t N, int64_t K,
                 uint8_t *codes, uint16_t *scales) {
  int64_t G = K / ORC_GROUP;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t g = 0; g < G; ++g) {
      const uint8_t *blk = raw + n * raw_stride + g * ORC_BLOCK_BYTES;
      scales[n * G + g] = (uint16_t)(blk[0] | (blk[1] << 8)); /* little-endian */
      for (int j = 0; j < 32; ++j) codes[n * (K / 4) + g * 32 + j] = blk[2 + j];
    }
  }
}

/* Dense signed weights from the code plane: w[n][k] = c - 1. */
void orc_decode_matrix(const uint8_t *codes, int64_t N, int64_t K, int8_t *w) {
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      w[n * K + k] =
          (int8_t)orc_decode_field(codes[n * (K / 4) + k / 4], (int)(k % 4));
}

/* ------------------------------------------------------------------ PTQ1_0 */

#define ORC_PTQ_BLOCK_BYTES 28

/* Trit `level` (0 first) of a five-trit byte, KR: v <- 3v in a 16-bit lane,
 * the trit is the part above the low byte, the low byte carries on. */
int orc_ptq_trit(uint8_t byte, int level) {
  unsigned v = byte, t = 0;
  for (int n = 0; n <= level; ++n) {
    unsigned w = 3u * v;
    t = w >> 8;
    v = w & 0xFFu;
  }
  return (int)t;
}

/* PTQ1_0 rows -> the code plane used everywhere in this file (code = trit, so
 * the weight is code - 1) and the fp16 scale bits.
 *   raw    : N rows, row stride raw_stride bytes, K/128 blocks of 28 bytes:
 *            qs bytes 0-23, qh bytes 24-25, d bytes 26-27 (little-endian)
 *   codes  : [N][K/4], weight k of a group in bits 2(k%4).. of byte k/4
 *   scales : [N][K/128] */
void orc_ptq_unpack(const uint8_t *raw, int64_t raw_stride, int64_t N, int64_t K,
                    uint8_t *codes, uint16_t *scales) {
  int64_t G = K / ORC_GROUP;
  for (int64_t n = 0; n < N; ++n) {
    uint8_t *crow = codes + n * (K / 4);
    memset(crow, 0, (size_t)(K / 4));
    for (int64_t g = 0; g < G; ++g) {
      const uint8_t *blk = raw + n * raw_stride + g * ORC_PTQ_BLOCK_BYTES;
      uint8_t *cg = crow + g * 32;
      for (int j = 0; j < 24; ++j)
        for (int lv = 0; lv < 5; ++lv) {
          int k = 24 * lv + j;
          cg[k / 4] |= (uint8_t)(orc_ptq_trit(blk[j], lv) << (2 * (k % 4)));
        }
      for (int j = 0; j < 2; ++j)
        for (int lv = 0; lv < 4; ++lv) {
          int k = 120 + 2 * lv + j;
          cg[k / 4] |= (uint8_t)(orc_ptq_trit(blk[24 + j], lv) << (2 * (k % 4)));
        }
      scales[n * G + g] = (uint16_t)(blk[26] | (blk[27] << 8));
    }
  }
}

/* ------------------------------------------------------------ quantisation */

/* Per-group INT8 quantisation of an fp32 activation matrix a[M][K].
 * KE Test 6 _quantize and BIB step 1:
 *   s = max|a| / 127            (fp32 IEEE division)
 *   d = s > 0 ? s : 1
 *   q = clamp(nearbyint(a / d), -127, 127)   (fp32 IEEE division, ties even)
 * Outputs q[M][K] (row-major, natural order) and sx[M][K/128]. */
void orc_quantize(const float *a, int64_t M, int64_t K, int8_t *q, float *sx) {
  int saved = fegetround();
  fesetround(FE_TONEAREST);
  int64_t G = K / ORC_GROUP;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t g = 0; g < G; ++g) {
      const float *x = a + m * K + g * ORC_GROUP;
      float amax = 0.0f;
      for (int i = 0; i < ORC_GROUP; ++i) {
        float v = fabsf(x[i]);
        if (v > amax) amax = v;
      }
      float s = amax / 127.0f;
      float d = (s > 0.0f) ? s : 1.0f;
      for (int i = 0; i < ORC_GROUP; ++i) {
        float r = nearbyintf(x[i] / d);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[m * K + g * ORC_GROUP + i] = (int8_t)r;
      }
      sx[m * G + g] = s;
    }
  }
  fesetround(saved);
}

/* Widen bf16 (kind 0), fp16 (kind 1) or fp32 (kind 2) activations to fp32.
 * x has row stride ldx elements. */
void orc_widen(const void *x, int kind, int64_t ldx, int64_t M, int64_t K,
               float *a) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t k = 0; k < K; ++k) {
      int64_t i = m * ldx + k;
      if (kind == 0)
        a[m * K + k] = orc_bf16_to_float(((const uint16_t *)x)[i]);
      else if (kind == 1)
        a[m * K + k] = orc_half_to_float(((const uint16_t *)x)[i]);
      else
        a[m * K + k] = ((const float *)x)[i];
    }
}

/* Plane order of q inside each 128-group (KE Test 21):
 * qp[g*128 + s*32 + j] = q[g*128 + 4*j + s], s = 0..3, j = 0..31, so plane s
 * holds the activations that meet bit field s of the 32 code bytes. */
void orc_q_planes(const int8_t *q, int64_t M, int64_t K, int8_t *qp) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t g = 0; g < K / ORC_GROUP; ++g)
      for (int s = 0; s < 4; ++s)
        for (int j = 0; j < 32; ++j)
          qp[m * K + g * ORC_GROUP + s * 32 + j] =
              q[m * K + g * ORC_GROUP + 4 * j + s];
}

/* T[m][g] = sum of q over the group (KE Test 21). */
void orc_qsum(const int8_t *q, int64_t M, int64_t K, int32_t *T) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t g = 0; g < K / ORC_GROUP; ++g) {
      int32_t t = 0;
      for (int i = 0; i < ORC_GROUP; ++i) t += q[m * K + g * ORC_GROUP + i];
      T[m * (K / ORC_GROUP) + g] = t;
    }
}

/* ---------------------------------------------------------- matmul pieces */

/* Exact per-group integer dots, BIB step 3:
 * dots[m][n][g] = sum_{k in g} (c_{n,k} - 1) * q_{m,k}   (int32, exact). */
void orc_group_dots(const int8_t *q, const uint8_t *codes, int64_t M,
                    int64_t N, int64_t K, int32_t *dots) {
  int64_t G = K / ORC_GROUP;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t g = 0; g < G; ++g) {
        int32_t acc = 0;
        for (int i = 0; i < ORC_GROUP; ++i) {
          int64_t k = g * ORC_GROUP + i;
          int w = orc_decode_field(codes[n * (K / 4) + k / 4], (int)(k % 4));
          acc += w * (int32_t)q[m * K + k];
        }
        dots[(m * N + n) * G + g] = acc;
      }
}

/* Scale and accumulate, BIB step 4, in sequential fp32 with no FMA:
 * y32[m][n] = sum over g = 0..G-1 of ((float)dot * s_x[m][g]) * s_w[n][g].
 * Optionally also the fp64 value and the error-bound weight
 * B[m][n] = sum_g |s_x * s_w * dot| (both in double).  scales are fp16 bits. */
void orc_scale_accumulate(const int32_t *dots, const float *sx,
                          const uint16_t *scales, int64_t M, int64_t N,
                          int64_t K, float *y32, double *y64, double *bound) {
  int64_t G = K / ORC_GROUP;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      float acc = 0.0f;
      double acc64 = 0.0, b = 0.0;
      for (int64_t g = 0; g < G; ++g) {
        int32_t dot = dots[(m * N + n) * G + g];
        float xs = sx[m * G + g];
        float ws = orc_half_to_float(scales[n * G + g]);
        float t = (float)dot * xs;
        t = t * ws;
        acc = acc + t;
        double term = (double)dot * (double)xs * (double)ws;
        acc64 += term;
        b += fabs(term);
      }
      if (y32) y32[m * N + n] = acc;
      if (y64) y64[m * N + n] = acc64;
      if (bound) bound[m * N + n] = b;
    }
}

/* Quantiser with activation groups of A elements (A = 128, 64 or 32; KE
 * Test 9): per A-group s = max|x| / 127, q = clamp(rne(x / d)) as
 * orc_quantize; sx is [M][K/A]. */
void orc_quantize_grouped(const float *a, int64_t M, int64_t K, int A, int8_t *q, float *sx) {
  int saved = fegetround();
  fesetround(FE_TONEAREST);
  int64_t GA = K / A;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t g = 0; g < GA; ++g) {
      const float *x = a + m * K + g * A;
      float amax = 0.0f;
      for (int i = 0; i < A; ++i) {
        float v = fabsf(x[i]);
        if (v > amax) amax = v;
      }
      float s = amax / 127.0f;
      float d = (s > 0.0f) ? s : 1.0f;
      for (int i = 0; i < A; ++i) {
        float r = nearbyintf(x[i] / d);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[m * K + g * A + i] = (int8_t)r;
      }
      sx[m * GA + g] = s;
    }
  }
  fesetround(saved);
}

/* Sum of q over each A-group: T[m][j], j = 0..K/A-1 (the masked-plane
 * decoder's offset term, KE Test 21, per activation group). */
void orc_qsum_grouped(const int8_t *q, int64_t M, int64_t K, int A, int32_t *T) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t j = 0; j < K / A; ++j) {
      int32_t t = 0;
      for (int i = 0; i < A; ++i) t += q[m * K + j * A + i];
      T[m * (K / A) + j] = t;
    }
}

/* Partial dots over each A-group: dots[m][n][j] = sum over k in
 * [jA, jA + A) of (c_{n,k} - 1) q_{m,k}, j = 0..K/A-1. */
void orc_group_dots_grouped(const int8_t *q, const uint8_t *codes, int64_t M, int64_t N,
                            int64_t K, int A, int32_t *dots) {
  int64_t GA = K / A;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t j = 0; j < GA; ++j) {
        int32_t acc = 0;
        for (int i = 0; i < A; ++i) {
          int64_t k = j * A + i;
          int w = orc_decode_field(codes[n * (K / 4) + k / 4], (int)(k % 4));
          acc += w * (int32_t)q[m * K + k];
        }
        dots[(m * N + n) * GA + j] = acc;
      }
}

/* Scale and accumulate with activation groups of A elements (KE Test 9):
 * y32[m][n] = sum over the weight groups g, then over their activation
 * groups h = 0..128/A-1, of ((float)dot_{gh} * s_x[m][g*128/A + h]) *
 * s_w[n][g], in sequential fp32; y64 the same in double; bound B = the sum
 * of |s_x * s_w * dot| (double). */
void orc_scale_accumulate_grouped(const int32_t *dots, const float *sx, const uint16_t *scales,
                                  int64_t M, int64_t N, int64_t K, int A, float *y32,
                                  double *y64, double *bound) {
  int64_t G = K / ORC_GROUP, GA = K / A, H = ORC_GROUP / A;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      float acc = 0.0f;
      double acc64 = 0.0, b = 0.0;
      for (int64_t g = 0; g < G; ++g) {
        float ws = orc_half_to_float(scales[n * G + g]);
        for (int64_t h = 0; h < H; ++h) {
          int32_t dot = dots[(m * N + n) * GA + g * H + h];
          float xs = sx[m * GA + g * H + h];
          float t = (float)dot * xs;
          t = t * ws;
          acc = acc + t;
          double term = (double)dot * (double)xs * (double)ws;
          acc64 += term;
          b += fabs(term);
        }
      }
      if (y32) y32[m * N + n] = acc;
      if (y64) y64[m * N + n] = acc64;
      if (bound) bound[m * N + n] = b;
    }
}

/* Gated output, KE Test 12: y64 [M][N] (N even) holds the projection's
 * output, gate = columns 0..N/2-1, up = columns N/2..N-1;
 * out64[m][n] = silu(gate) * up = gate / (1 + exp(-gate)) * up, in double. */
void orc_gated(const double *y64, int64_t M, int64_t N, double *out64) {
  int64_t I = N / 2;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < I; ++n) {
      double g = y64[m * N + n];
      double u = y64[m * N + I + n];
      out64[m * I + n] = g / (1.0 + exp(-g)) * u;
    }
}

/* Orthonormal Walsh-Hadamard transform of 1024 values in place, fp32:
 * butterfly passes with half-width 1, 2, 4, .., 512 (pairs j, j + h inside
 * blocks of 2h become a + b, a - b), then the factor 1/32 = 1/sqrt(1024),
 * exact.  (KE Test 18 applies it to each 1024-element block of a row.) */
void orc_fwht1024(float *v) {
  for (int h = 1; h < 1024; h *= 2)
    for (int b = 0; b < 1024; b += 2 * h)
      for (int j = b; j < b + h; ++j) {
        float a = v[j], c = v[j + h];
        v[j] = a + c;
        v[j + h] = a - c;
      }
  for (int j = 0; j < 1024; ++j) v[j] = v[j] * 0.03125f;
}

/* Sum of squares of one row in the reduction structure of KE Test 18:
 * partial p[i] = sum of h[j]^2 over j = i, i + 2048, i + 4096, .. (in that
 * order, fp32), then the 2048 partials summed pairwise: p[i] += p[i + len]
 * for len = 1024, 512, .., 1; the result is p[0]. */
float orc_sumsq2048(const float *h, int64_t K) {
  static float p[2048];
  for (int i = 0; i < 2048; ++i) p[i] = 0.0f;
  for (int64_t j = 0; j < K; ++j) {
    float t = h[j] * h[j];
    p[j % 2048] = p[j % 2048] + t;
  }
  for (int len = 1024; len >= 1; len /= 2)
    for (int i = 0; i < len; ++i) p[i] = p[i] + p[i + len];
  return p[0];
}

/* Fused preparation, KE Test 18, for M rows of K (K % 1024 == 0) bf16
 * activations x (bits), optional bf16 residual (bits, NULL if none):
 *   h      = x + residual (fp32; x alone without residual)
 *   inv    = 1 / sqrt(sumsq2048(h) / K + eps)     (IEEE sqrt and division)
 *   n      = bf16_rne((h * inv) * (w + 1))        (w: bf16 bits, per column)
 *   v      = float(n) * sign                       (sign: +1 / -1 per column)
 *   v      = bf16_rne(fwht1024(v)) per 1024-column block
 *   q, sx  = orc_quantize(v)                       (group 128)
 * Optional outputs (NULL to skip): norm_out (bits of n), res_out (bits of
 * bf16_rne(h)). */
void orc_norm_hadamard_quantize(const uint16_t *x, const uint16_t *residual,
                                const uint16_t *w, const int8_t *sign, float eps,
                                int64_t M, int64_t K, uint16_t *norm_out,
                                uint16_t *res_out, int8_t *q, float *sx) {
  int saved = fegetround();
  fesetround(FE_TONEAREST);
  static float h[1 << 20], v[1 << 20];
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t j = 0; j < K; ++j) {
      float a = orc_bf16_to_float(x[m * K + j]);
      if (residual) a = a + orc_bf16_to_float(residual[m * K + j]);
      h[j] = a;
      if (res_out) res_out[m * K + j] = orc_float_to_bf16_rne(a);
    }
    float mean = orc_sumsq2048(h, K) / (float)K;
    float inv = 1.0f / sqrtf(mean + eps);
    for (int64_t j = 0; j < K; ++j) {
      float t = (h[j] * inv) * (orc_bf16_to_float(w[j]) + 1.0f);
      uint16_t nb = orc_float_to_bf16_rne(t);
      if (norm_out) norm_out[m * K + j] = nb;
      v[j] = orc_bf16_to_float(nb) * (float)sign[j];
    }
    for (int64_t b = 0; b < K; b += 1024) {
      orc_fwht1024(v + b);
      for (int j = 0; j < 1024; ++j) v[b + j] = orc_bf16_to_float(orc_float_to_bf16_rne(v[b + j]));
    }
    orc_quantize(v, 1, K, q + m * K, sx + m * (K / ORC_GROUP));
  }
  fesetround(saved);
}

/* Whole path on already-prepared planes: y32 for an activation matrix x.
 * Used for the timed CPU baseline (quantise + group dots + scale). */
void orc_linear(const void *x, int kind, int64_t ldx, int64_t M, int64_t N,
                int64_t K, const uint8_t *codes, const uint16_t *scales,
                float *a_tmp, int8_t *q_tmp, float *sx_tmp, int32_t *dots_tmp,
                float *y32) {
  orc_widen(x, kind, ldx, M, K, a_tmp);
  orc_quantize(a_tmp, M, K, q_tmp, sx_tmp);
  orc_group_dots(q_tmp, codes, M, N, K, dots_tmp);
  orc_scale_accumulate(dots_tmp, sx_tmp, scales, M, N, K, y32, NULL, NULL);
}
