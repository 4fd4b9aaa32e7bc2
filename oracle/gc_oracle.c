/*
 * gc_oracle.c -- CPU oracle for the error-feedback gradient compressor.
 *
 * TEST INFRASTRUCTURE.  This is the slow, plain, single-threaded statement of
 * what the compressor computes.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load it.  It shares no code,
 * header, table or helper with the CUDA library; the only thing both sides
 * see is the seeded synthetic input.
 *
 * Sources (cited by page title and section):
 *   [P1] hotdry blog, "gradient-compression-quantization-sparsification":
 *        1.1 QSGD and TernGrad, 1.2 trade-offs (deterministic vs stochastic
 *        rounding, groups of 64), 2.1 Top-K with error feedback,
 *        3.1 PowerSGD.
 *   [P2] "分布式训练中的梯度压缩算法：性能瓶颈、收敛性影响与实现细节":
 *        二.1 线性量化 (q = round((g-min)/scale), g_hat = q*scale+min,
 *        scale = (max-min)/(2^b-1)); 二.2 Top-K 稀疏化; 三 误差补偿代码示例
 *        (c = g + e, e' = c - g_hat).
 *   [P3] "4、梯度累积与梯度压缩": 4.2.1 TopK稀疏化 (k = max(1, n*ratio),
 *        torch.topk on |g|, return (indices, values)); 4.2.2 QSGD量化压缩;
 *        4.3 TopK(1%) + 8-bit QSGD combination.
 *   [P4] "梯度聚合通信优化实战方案": 梯度压缩原理 (error compensation);
 *        Python 演示 (error_feedback_compress, quantize, topk_sparsify).
 *   Philox-4x32-10: J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel Random
 *        Numbers: As Easy as 1, 2, 3", SC'11, section 3 (Philox S-box and
 *        key schedule).
 *   QSGD: D. Alistarh et al., "QSGD: Communication-Efficient SGD via Gradient
 *        Quantization and Encoding", NeurIPS 2017, section 3.1 (s levels on
 *        the L2 norm, stochastic rounding between adjacent levels).
 *   TernGrad: W. Wen et al., "TernGrad: Ternary Gradients to Reduce
 *        Communication in Distributed Deep Learning", NeurIPS 2017, eq. 2
 *        (s = max|g|, Bernoulli(|g|/s) times sign times s).
 *   Cody-Waite: W. J. Cody, W. Waite, "Software Manual for the Elementary
 *        Functions", Prentice-Hall 1980, the ALOG and EXP chapters (argument
 *        reduction by ln 2 split in two parts, a series in s = (m-1)/(m+1)
 *        for the logarithm, a polynomial for exp on [-ln2/2, ln2/2]).
 *   PowerSGD: T. Vogels, S. P. Karimireddy, M. Jaggi, "PowerSGD: Practical
 *        Low-Rank Gradient Compression for Distributed Optimization",
 *        NeurIPS 2019, Algorithm 1 (P = MQ, orthogonalise, Q = M^T P,
 *        reconstruct P Q^T, error feedback).
 *
 * Precision: the pages' gradients are float32 arrays (P4 Python 演示 casts
 * with astype(np.float32)); every floating-point step below is one IEEE-754
 * binary32 operation rounded to nearest-even.  The file must be compiled with
 * -ffp-contract=off (no fused multiply-add) and without -ffast-math.
 * PowerSGD is the exception: it is computed in binary64 and cast at the end,
 * because its parity bar is a relative Frobenius tolerance.
 *
 * Readings of points the pages leave open are listed where they are used.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_EUNSUP (-2)
#define ORC_ENOMEM (-7)

#define ORC_MINMAX 0
#define ORC_QSGD 1
#define ORC_TERN 2
#define ORC_LOG 3

#define ORC_NEAREST_EVEN 0
#define ORC_STOCHASTIC 1

/* ------------------------------------------------------------------------ */
/* Philox-4x32-10 (Salmon et al., SC'11, section 3).                         */
/* ------------------------------------------------------------------------ */

/* Multipliers and Weyl key increments published with Philox-4x32. */
#define PHILOX_MUL_A 0xD2511F53u
#define PHILOX_MUL_B 0xCD9E8D57u
#define PHILOX_WEYL_A 0x9E3779B9u
#define PHILOX_WEYL_B 0xBB67AE85u

void orc_philox4x32_10(const uint32_t counter[4], const uint32_t key[2],
                       uint32_t out[4]) {
  uint32_t x0 = counter[0], x1 = counter[1], x2 = counter[2], x3 = counter[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { /* key schedule: bump by the Weyl constants */
      k0 += PHILOX_WEYL_A;
      k1 += PHILOX_WEYL_B;
    }
    uint64_t pa = (uint64_t)PHILOX_MUL_A * (uint64_t)x0;
    uint64_t pb = (uint64_t)PHILOX_MUL_B * (uint64_t)x2;
    uint32_t hi_a = (uint32_t)(pa >> 32), lo_a = (uint32_t)pa;
    uint32_t hi_b = (uint32_t)(pb >> 32), lo_b = (uint32_t)pb;
    /* S-box: the two products, the other two words and the round key. */
    uint32_t y0 = hi_b ^ x1 ^ k0;
    uint32_t y1 = lo_b;
    uint32_t y2 = hi_a ^ x3 ^ k1;
    uint32_t y3 = lo_a;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/*
 * Uniform draw for element i of a call (reading: the pages ask for
 * stochastic rounding [P1 1.1, 1.2] but fix no generator).  Element i uses
 * word (i mod 4) of Philox-4x32-10 at counter
 *   {low32(i/4), high32(i/4), low32(step), high32(step)}
 * with key {low32(seed), high32(seed)}; the word's top 24 bits scaled by
 * 2^-24 give u in [0, 1), exactly representable in binary32.
 */
float orc_uniform(uint64_t seed, uint64_t step, uint64_t i) {
  uint64_t block = i >> 2;
  uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), (uint32_t)step,
                     (uint32_t)(step >> 32)};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t r[4];
  orc_philox4x32_10(ctr, key, r);
  uint32_t word = r[i & 3u];
  return (float)(word >> 8) * 0x1p-24f;
}

/*
 * Key of bucket b of a bucketed call (reading: the pages compress bucket by
 * bucket [P3 4.3, P4 通信计算重叠] and fix no stream per bucket).  Bucket b
 * draws with the key seed XOR (b * 0x9E3779B97F4A7C15), the 64-bit
 * golden-ratio constant floor(2^64 / phi): bucket 0 keeps the call's seed,
 * and buckets of calls whose seeds differ by small amounts never share a
 * key.
 */
uint64_t orc_bucket_seed(uint64_t seed, int64_t b) {
  return seed ^ ((uint64_t)b * UINT64_C(0x9E3779B97F4A7C15));
}

/* ------------------------------------------------------------------------ */
/* Sizes of the compressed formats.                                          */
/* ------------------------------------------------------------------------ */

static int64_t round_up16(int64_t bytes) { return (bytes + 15) / 16 * 16; }

static int valid_bits(int bits) {
  return bits == 1 || bits == 2 || bits == 4 || bits == 8;
}

/*
 * Packed code buffer: the b-bit codes of all n elements, least-significant
 * bit first, padded with zero bytes to a multiple of 16 bytes; for QSGD a
 * one-bit-per-element sign plane follows in the same way.  (Reading: P2
 * 二.1 and P4 Python 演示 send integer codes plus the scale and minimum;
 * P3 4.2.2 states 8-bit codes are 1/4 and 4-bit codes 1/8 of fp32, so codes
 * are packed b bits each.)
 */
int64_t orc_codes_bytes(int64_t n, int bits, int mode) {
  if (n < 0 || !valid_bits(bits)) return -1;
  int64_t mag = round_up16((n * bits + 7) / 8);
  if (mode == ORC_QSGD) return mag + round_up16((n + 7) / 8);
  return mag;
}

static int64_t group_len(int64_t n, int64_t group) {
  return group == 0 ? n : group;
}

static int64_t num_groups(int64_t n, int64_t group) {
  if (n == 0) return 0;
  int64_t G = group_len(n, group);
  return (n + G - 1) / G;
}

/* Scale buffer: min-max stores {scale, min} per group, QSGD and TernGrad
 * store {scale} per group.  group == 0 means one group over all n. */
int64_t orc_scales_floats(int64_t n, int64_t group, int mode) {
  if (n < 0 || group < 0) return -1;
  return num_groups(n, group) * (mode == ORC_MINMAX ? 2 : 1);
}

/* ------------------------------------------------------------------------ */
/* Top-K selection with error feedback.                                      */
/* ------------------------------------------------------------------------ */

/* |x| as an unsigned integer: the IEEE bits with the sign cleared.  For
 * finite values this orders exactly like |x| and makes -0 equal to +0. */
static uint32_t magnitude_key(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  return u & 0x7fffffffu;
}

typedef struct {
  uint32_t key;
  int64_t index;
} rank_rec;

/* Larger |c| first; among equal |c| the smaller index first. */
static int rank_cmp(const void* pa, const void* pb) {
  const rank_rec* a = (const rank_rec*)pa;
  const rank_rec* b = (const rank_rec*)pb;
  if (a->key != b->key) return a->key > b->key ? -1 : 1;
  if (a->index != b->index) return a->index < b->index ? -1 : 1;
  return 0;
}

/*
 * Marks in keep[0..n) the k entries of c with the largest |c| ([P2 二.2
 * Top-K 稀疏化]: keep the K entries of largest absolute value; [P3 4.2.1]:
 * exactly k via torch.topk).  Reading for ties: the order is (|c|
 * descending, index ascending), so exactly k entries are kept.
 */
static int topk_mark(const float* c, int64_t n, int64_t k, unsigned char* keep) {
  memset(keep, 0, (size_t)n);
  if (k == 0) return ORC_OK;
  rank_rec* recs = (rank_rec*)malloc((size_t)n * sizeof(rank_rec));
  if (!recs) return ORC_ENOMEM;
  for (int64_t i = 0; i < n; ++i) {
    recs[i].key = magnitude_key(c[i]);
    recs[i].index = i;
  }
  qsort(recs, (size_t)n, sizeof(rank_rec), rank_cmp);
  for (int64_t j = 0; j < k; ++j) keep[recs[j].index] = 1;
  free(recs);
  return ORC_OK;
}

/*
 * EF + Top-K ([P2 三 误差补偿], [P4 Python 演示 error_feedback_compress],
 * [P1 2.1]):
 *   c = g + e;  kept = Top-K(|c|);  idx = kept positions in ascending order
 *   (the order np.where gives in P4);  val = c[idx];
 *   e' = c with the kept positions set to zero (what was not sent is carried
 *   to the next step).
 * err == NULL selects from grad alone and writes no residual.
 */
int orc_ef_topk(const float* grad, float* err, int64_t n, int64_t k,
                int32_t* idx_out, float* val_out) {
  if (n < 0 || k < 0 || k > n || n > INT32_MAX) return ORC_EINVAL;
  if (n == 0) return ORC_OK;
  float* c = (float*)malloc((size_t)n * sizeof(float));
  unsigned char* keep = (unsigned char*)malloc((size_t)n);
  if (!c || !keep) { free(c); free(keep); return ORC_ENOMEM; }
  for (int64_t i = 0; i < n; ++i) c[i] = err ? grad[i] + err[i] : grad[i];
  int st = topk_mark(c, n, k, keep);
  if (st == ORC_OK) {
    int64_t j = 0;
    for (int64_t i = 0; i < n; ++i) {
      if (keep[i]) {
        idx_out[j] = (int32_t)i;
        val_out[j] = c[i];
        ++j;
      }
    }
    if (err)
      for (int64_t i = 0; i < n; ++i) err[i] = keep[i] ? 0.0f : c[i];
  }
  free(c);
  free(keep);
  return st;
}

/* ------------------------------------------------------------------------ */
/* Group statistics.                                                         */
/* ------------------------------------------------------------------------ */

/*
 * Sum of x[i]^2 over a group, added in a fixed order (reading: the pages
 * fix no order).  The order is the perfect binary tree over the group's
 * squares padded with zeros to a power of two, adjacent pairs first.  Adding
 * a zero is exact, so the padded tree equals this level-by-level pairing in
 * which an unpaired last entry is carried up unchanged.
 */
static float tree_sum_squares(const float* x, int64_t len, float* scratch) {
  if (len == 0) return 0.0f;
  for (int64_t i = 0; i < len; ++i) scratch[i] = x[i] * x[i];
  int64_t m = len;
  while (m > 1) {
    int64_t half = m / 2;
    for (int64_t j = 0; j < half; ++j)
      scratch[j] = scratch[2 * j] + scratch[2 * j + 1];
    if (m & 1) scratch[half] = scratch[m - 1];
    m = half + (m & 1);
  }
  return scratch[0];
}

/* ------------------------------------------------------------------------ */
/* Natural logarithm and exponential in binary32 (logarithmic quantisation). */
/* ------------------------------------------------------------------------ */

/*
 * [P2 二.1 对数量化] needs log and exp, and its level q = round(log(|g|+1) /
 * scale) is an integer that a one-ulp difference in log can change.
 * Reading: the pages do not fix the functions to the bit, so log and exp are
 * defined here by the Cody-Waite method, every step one binary32 operation
 * (the CUDA library implements the same definition independently); their
 * accuracy against the true functions is checked by the tests.
 *
 * ln 2 = LN2_HI + LN2_LO: LN2_HI = 45426 / 2^16 (16 significant bits, so
 * k * LN2_HI is exact for |k| < 2^8) and LN2_LO = ln 2 - LN2_HI rounded to
 * binary32.  The series coefficients are 1/(2j+1) and 1/j! rounded to
 * binary32.
 */
#define LN2_HI 0x1.62e4p-1f
#define LN2_LO 0x1.7f7d1cp-20f
#define INV_LN2 0x1.715476p+0f
#define SQRT2_F 0x1.6a09e6p+0f

/*
 * log(x) for finite x >= 1: x = 2^k m with m in [sqrt(2)/2, sqrt(2)],
 * s = (m - 1) / (m + 1), log m = 2 atanh(s) = 2s (1 + z/3 + z^2/5 + ...
 * + z^5/11), z = s^2 (|s| <= 0.1716, the first omitted term is below
 * 2^-36 of 2s); log x = k LN2_HI + (k LN2_LO + log m).
 */
float orc_logf(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  int k = (int)(u >> 23) - 127;
  u = (u & 0x007fffffu) | 0x3f800000u;
  float m;
  memcpy(&m, &u, 4);
  if (m > SQRT2_F) {
    m = m * 0.5f;
    k += 1;
  }
  float f = m - 1.0f;
  float s = f / (f + 2.0f);
  float z = s * s;
  float r = 0x1.745d18p-4f;             /* 1/11 */
  r = 0x1.c71c72p-4f + z * r;           /* 1/9 */
  r = 0x1.24924ap-3f + z * r;           /* 1/7 */
  r = 0x1.99999ap-3f + z * r;           /* 1/5 */
  r = 0x1.555556p-2f + z * r;           /* 1/3 */
  r = z * r;
  float w = s + s;
  float logm = w + w * r;
  float kf = (float)k;
  return kf * LN2_HI + (kf * LN2_LO + logm);
}

/*
 * exp(y) for 0 <= y < 89: k = rint(y / ln 2), r = (y - k LN2_HI) - k LN2_LO
 * (|r| <= ln2 / 2), exp r = 1 + r + r^2/2! + ... + r^8/8! (Horner; the first
 * omitted term is below 2^-31), exp y = 2^k exp r (an exact scaling; k = 128
 * overflows to +inf).
 */
float orc_expf(float y) {
  float kf = rintf(y * INV_LN2);
  float r = (y - kf * LN2_HI) - kf * LN2_LO;
  float p = 0x1.a01a02p-16f;            /* 1/8! */
  p = 0x1.a01a02p-13f + r * p;          /* 1/7! */
  p = 0x1.6c16c2p-10f + r * p;          /* 1/6! */
  p = 0x1.111112p-7f + r * p;           /* 1/5! */
  p = 0x1.555556p-5f + r * p;           /* 1/4! */
  p = 0x1.555556p-3f + r * p;           /* 1/3! */
  p = 0.5f + r * p;                     /* 1/2! */
  p = 1.0f + r * p;
  p = 1.0f + r * p;
  int k = (int)kf;
  if (k >= 128) return INFINITY;
  uint32_t bits = (uint32_t)(k + 127) << 23;
  float two_k;
  memcpy(&two_k, &bits, 4);
  return p * two_k;
}

typedef struct {
  float scale;  /* step between levels (0 means every code is 0) */
  float offset; /* min-max: the group minimum; otherwise unused */
} group_param;

/*
 * Per-group parameters.
 *  min-max  [P2 二.1 线性量化]: scale = (max - min) / (2^b - 1), offset = min.
 *           Reading: min and max are canonicalised by adding +0 so that -0
 *           and +0 give the same bits.
 *  QSGD     [P1 1.1; Alistarh et al. 3.1]: s = 2^b - 1 levels of the group's
 *           L2 norm; scale = ||c||_2 / s.  The norm is the correctly rounded
 *           square root of tree_sum_squares.
 *  TernGrad [P1 1.1 "逐层归一化"; Wen et al. eq. 2]: scale = max |c| over the
 *           group (the group is the whole tensor for layer-wise scaling).
 *  log      [P2 二.1 对数量化]: scale = log(max |c| + 1) / (2^(b-1) - 1), one
 *           bit being the sign; max over the group (the page's example takes
 *           the whole tensor: group 0).
 */
static group_param group_stats(const float* x, int64_t len, int bits, int mode,
                               float* scratch) {
  group_param p = {0.0f, 0.0f};
  if (mode == ORC_MINMAX) {
    float mn = x[0], mx = x[0];
    for (int64_t i = 1; i < len; ++i) {
      if (x[i] < mn) mn = x[i];
      if (x[i] > mx) mx = x[i];
    }
    mn = mn + 0.0f;
    mx = mx + 0.0f;
    float levels = (float)((1 << bits) - 1);
    p.scale = (mx - mn) / levels;
    p.offset = mn;
  } else if (mode == ORC_QSGD) {
    float ss = tree_sum_squares(x, len, scratch);
    float norm = sqrtf(ss);
    float levels = (float)((1 << bits) - 1);
    p.scale = norm / levels;
  } else { /* ORC_TERN, ORC_LOG */
    float mx = 0.0f;
    for (int64_t i = 0; i < len; ++i) {
      float a = fabsf(x[i]);
      if (a > mx) mx = a;
    }
    if (mode == ORC_TERN) {
      p.scale = mx;
    } else {
      float levels = (float)((1 << (bits - 1)) - 1);
      p.scale = orc_logf(mx + 1.0f) / levels;
    }
  }
  return p;
}

/* ------------------------------------------------------------------------ */
/* Rounding, packing, quantize / dequantize.                                 */
/* ------------------------------------------------------------------------ */

/*
 * Integer level for the real level position t >= 0 ([P1 1.2]: deterministic
 * or stochastic rounding).
 *  nearest-even: rint(t), round half to even, as np.round / torch.round do
 *                in [P2 二.1], [P3 4.2.2] and [P4 Python 演示].
 *  stochastic:   floor(t) + 1 with probability t - floor(t), else floor(t)
 *                ([P1 1.1]: unbiased in expectation); the draw is
 *                orc_uniform for this element, and "u < t - floor(t)" rounds
 *                up.
 * The result is clamped to [0, top] (reading: the pages never clamp; the
 * clamp only acts when a rounded t lands one step past the top level).
 */
static uint32_t round_level(float t, int rounding, uint64_t seed, uint64_t step,
                            uint64_t i, uint32_t top) {
  float q;
  if (rounding == ORC_NEAREST_EVEN) {
    q = rintf(t);
  } else {
    float fl = floorf(t);
    float frac = t - fl;
    float u = orc_uniform(seed, step, i);
    q = fl + (u < frac ? 1.0f : 0.0f);
  }
  if (!(q > 0.0f)) return 0;
  if (q >= (float)top) return top;
  return (uint32_t)q;
}

/* Bit i*bits.. of a little-endian bit stream. */
static void put_bits(uint8_t* buf, int64_t i, int bits, uint32_t code) {
  int64_t bit = i * bits;
  buf[bit >> 3] |= (uint8_t)(code << (bit & 7));
}

static uint32_t get_bits(const uint8_t* buf, int64_t i, int bits) {
  int64_t bit = i * bits;
  return (buf[bit >> 3] >> (bit & 7)) & ((1u << bits) - 1u);
}

static int check_quant_args(int64_t n, int bits, int64_t group, int mode,
                            int rounding) {
  if (n < 0 || n > INT32_MAX || group < 0) return ORC_EINVAL;
  if (!valid_bits(bits)) return ORC_EUNSUP;
  if (mode != ORC_MINMAX && mode != ORC_QSGD && mode != ORC_TERN && mode != ORC_LOG)
    return ORC_EINVAL;
  if (mode == ORC_TERN && bits != 2) return ORC_EUNSUP;
  if (mode == ORC_LOG && bits == 1) return ORC_EUNSUP; /* no magnitude bit */
  if (rounding != ORC_NEAREST_EVEN && rounding != ORC_STOCHASTIC)
    return ORC_EINVAL;
  return ORC_OK;
}

/* Dequantised value of one element ([P2 二.1]: g_hat = q*scale + min, two
 * separate roundings; QSGD / TernGrad: sign times q*scale; log: sign times
 * exp(q*scale) - 1). */
static float dequant_one(uint32_t q, int negative, group_param p, int mode) {
  float mag = (float)q * p.scale;
  if (mode == ORC_MINMAX) return mag + p.offset;
  if (mode == ORC_LOG) mag = orc_expf(mag) - 1.0f;
  return negative ? -mag : mag;
}

/*
 * Quantises x[0..n) group by group.  Writes the packed codes and scales and,
 * when x_hat != NULL, the dequantised values.
 *  min-max:  t = (x - min) / scale, q in [0, 2^b - 1].
 *  QSGD:     t = |x| / scale, q in [0, 2^b - 1], sign in the sign plane.
 *  TernGrad: t = |x| / scale, q in {0, 1}, 2-bit code (sign << 1) | q.
 *  log:      t = log(|x| + 1) / scale, q in [0, 2^(b-1) - 1], b-bit
 *            sign-magnitude code (sign << (b-1)) | q.
 * scale == 0 (a constant group for min-max, an all-zero group otherwise)
 * gives q = 0 without dividing.  A sign is recorded only when q != 0, so a
 * zero code always dequantises to +0.
 */
static int quant_core(const float* x, int64_t n, int64_t base, int bits,
                      int64_t group, int mode, int rounding, uint64_t seed,
                      uint64_t step, uint8_t* codes_out, float* scales_out,
                      float* x_hat) {
  int st = check_quant_args(n, bits, group, mode, rounding);
  if (st != ORC_OK) return st;
  int64_t total = orc_codes_bytes(n, bits, mode);
  memset(codes_out, 0, (size_t)total);
  if (n == 0) return ORC_OK;
  int64_t mag_bytes = round_up16((n * bits + 7) / 8);
  uint8_t* sign_plane = codes_out + mag_bytes;
  int64_t G = group_len(n, group);
  int64_t ng = num_groups(n, group);
  float* scratch = (float*)malloc((size_t)G * sizeof(float));
  if (!scratch) return ORC_ENOMEM;
  uint32_t top = (mode == ORC_TERN)  ? 1u
                 : (mode == ORC_LOG) ? ((1u << (bits - 1)) - 1u)
                                     : ((1u << bits) - 1u);
  for (int64_t g = 0; g < ng; ++g) {
    int64_t start = g * G;
    int64_t len = (n - start < G) ? (n - start) : G;
    group_param p = group_stats(x + start, len, bits, mode, scratch);
    if (mode == ORC_MINMAX) {
      scales_out[2 * g] = p.scale;
      scales_out[2 * g + 1] = p.offset;
    } else {
      scales_out[g] = p.scale;
    }
    for (int64_t i = start; i < start + len; ++i) {
      float t;
      if (mode == ORC_MINMAX)
        t = p.scale == 0.0f ? 0.0f : (x[i] - p.offset) / p.scale;
      else if (mode == ORC_LOG)
        t = p.scale == 0.0f ? 0.0f : orc_logf(fabsf(x[i]) + 1.0f) / p.scale;
      else
        t = p.scale == 0.0f ? 0.0f : fabsf(x[i]) / p.scale;
      uint32_t q = p.scale == 0.0f
                       ? 0u
                       : round_level(t, rounding, seed, step,
                                     (uint64_t)(base + i), top);
      int negative = (mode != ORC_MINMAX) && q != 0 && x[i] < 0.0f;
      if (mode == ORC_TERN) {
        put_bits(codes_out, i, 2, ((uint32_t)negative << 1) | q);
      } else if (mode == ORC_LOG) {
        put_bits(codes_out, i, bits, ((uint32_t)negative << (bits - 1)) | q);
      } else {
        put_bits(codes_out, i, bits, q);
        if (mode == ORC_QSGD && negative) put_bits(sign_plane, i, 1, 1u);
      }
      if (x_hat) x_hat[i] = dequant_one(q, negative, p, mode);
    }
  }
  free(scratch);
  return ORC_OK;
}

int orc_quant(const float* x, int64_t n, int bits, int64_t group, int mode,
              int rounding, uint64_t seed, uint64_t step, uint8_t* codes_out,
              float* scales_out) {
  return quant_core(x, n, 0, bits, group, mode, rounding, seed, step,
                    codes_out, scales_out, NULL);
}

/*
 * Same as orc_quant on the slice x[0..n) of a larger call whose element 0
 * is element `base` of that call: the groups are taken relative to the
 * slice (so the slice must start on a group boundary of the call) and the
 * stochastic draw of slice element i is that of call element base + i.
 * Lets a test check a sampled range of a call too large for the oracle.
 */
int orc_quant_at(const float* x, int64_t n, int64_t base, int bits,
                 int64_t group, int mode, int rounding, uint64_t seed,
                 uint64_t step, uint8_t* codes_out, float* scales_out) {
  if (base < 0) return ORC_EINVAL;
  return quant_core(x, n, base, bits, group, mode, rounding, seed, step,
                    codes_out, scales_out, NULL);
}

/* Inverse of the packing above: g_hat from codes and scales. */
int orc_dequant(const uint8_t* codes, const float* scales, int64_t n, int bits,
                int64_t group, int mode, float* x_out) {
  int st = check_quant_args(n, bits, group, mode, ORC_NEAREST_EVEN);
  if (st != ORC_OK) return st;
  if (n == 0) return ORC_OK;
  int64_t mag_bytes = round_up16((n * bits + 7) / 8);
  const uint8_t* sign_plane = codes + mag_bytes;
  int64_t G = group_len(n, group);
  for (int64_t i = 0; i < n; ++i) {
    int64_t g = i / G;
    group_param p;
    if (mode == ORC_MINMAX) {
      p.scale = scales[2 * g];
      p.offset = scales[2 * g + 1];
    } else {
      p.scale = scales[g];
      p.offset = 0.0f;
    }
    uint32_t code = get_bits(codes, i, bits);
    uint32_t q;
    int negative;
    if (mode == ORC_TERN) {
      q = code & 1u;
      negative = (int)(code >> 1);
    } else if (mode == ORC_LOG) {
      q = code & ((1u << (bits - 1)) - 1u);
      negative = (int)(code >> (bits - 1));
    } else {
      q = code;
      negative = mode == ORC_QSGD ? (int)get_bits(sign_plane, i, 1) : 0;
    }
    x_out[i] = dequant_one(q, negative, p, mode);
  }
  return ORC_OK;
}

/*
 * EF + quantisation ([P2 三 quantize_with_error_compensation]):
 *   c = g + e;  (codes, scales) = quant(c);  g_hat = dequant(codes, scales);
 *   e' = c - g_hat, written over err.
 */
int orc_ef_quant(const float* grad, float* err, int64_t n, int bits,
                 int64_t group, int mode, int rounding, uint64_t seed,
                 uint64_t step, uint8_t* codes_out, float* scales_out) {
  int st = check_quant_args(n, bits, group, mode, rounding);
  if (st != ORC_OK) return st;
  if (n == 0) return quant_core(grad, 0, 0, bits, group, mode, rounding, seed,
                                step, codes_out, scales_out, NULL);
  float* c = (float*)malloc((size_t)n * sizeof(float));
  float* g_hat = (float*)malloc((size_t)n * sizeof(float));
  if (!c || !g_hat) { free(c); free(g_hat); return ORC_ENOMEM; }
  for (int64_t i = 0; i < n; ++i) c[i] = grad[i] + err[i];
  st = quant_core(c, n, 0, bits, group, mode, rounding, seed, step, codes_out,
                  scales_out, g_hat);
  if (st == ORC_OK)
    for (int64_t i = 0; i < n; ++i) err[i] = c[i] - g_hat[i];
  free(c);
  free(g_hat);
  return st;
}

/*
 * Differential quantisation ([P2 二.4 差分量化]): only the difference between
 * the gradient and the previous one is sent, quantised with few bits; the
 * page notes that both sides keep a gradient history and that errors pile up
 * over the steps unless corrected from time to time.  Reading: the history
 * ref is the gradient the receiver reconstructed last (closed loop, the
 * same on both sides, so quantisation errors do not pile up in it), and a
 * refresh step (the periodic correction) sends the full gradient, as if ref
 * were 0.  With error feedback ([P4 梯度压缩原理]):
 *   c = g + e (or g);  r = refresh ? 0 : ref;  d = c - r;
 *   (codes, scales) = quant(d);  d_hat = dequant(codes, scales);
 *   g_hat = r + d_hat;  e' = c - g_hat (when e is given);  ref' = g_hat.
 * Every step is one binary32 operation.
 */
int orc_ef_diff_quant(const float* grad, float* err, float* ref, int64_t n, int bits,
                      int64_t group, int mode, int rounding, uint64_t seed, uint64_t step,
                      int refresh, uint8_t* codes_out, float* scales_out) {
  int st = check_quant_args(n, bits, group, mode, rounding);
  if (st != ORC_OK) return st;
  if (!ref && n > 0) return ORC_EINVAL;
  float* c = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
  float* d = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
  float* d_hat = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
  if (!c || !d || !d_hat) { free(c); free(d); free(d_hat); return ORC_ENOMEM; }
  for (int64_t i = 0; i < n; ++i) {
    c[i] = err ? grad[i] + err[i] : grad[i];
    float r = refresh ? 0.0f : ref[i];
    d[i] = c[i] - r;
  }
  st = quant_core(d, n, 0, bits, group, mode, rounding, seed, step, codes_out, scales_out,
                  d_hat);
  if (st == ORC_OK) {
    for (int64_t i = 0; i < n; ++i) {
      float r = refresh ? 0.0f : ref[i];
      float g_hat = r + d_hat[i];
      if (err) err[i] = c[i] - g_hat;
      ref[i] = g_hat;
    }
  }
  free(c);
  free(d);
  free(d_hat);
  return st;
}

/* The receiving side: ref' = (refresh ? 0 : ref) + dequant(codes, scales). */
int orc_diff_dequant(const uint8_t* codes, const float* scales, int64_t n, int bits,
                     int64_t group, int mode, int refresh, float* ref) {
  float* d_hat = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
  if (!d_hat) return ORC_ENOMEM;
  int st = orc_dequant(codes, scales, n, bits, group, mode, d_hat);
  if (st == ORC_OK)
    for (int64_t i = 0; i < n; ++i) ref[i] = (refresh ? 0.0f : ref[i]) + d_hat[i];
  free(d_hat);
  return st;
}

/*
 * Hybrid: EF + Top-K, then QSGD on the kept values ([P3 4.3]: TopK 1% plus
 * 8-bit QSGD; [P1 三 混合压缩]).
 *   c = g + e;  (idx, val) = Top-K(c) in ascending index order;
 *   (codes, scales) = QSGD(val[0..k), bits, group) where element j of the
 *   quantised array is val[j] (its stochastic draw uses index j);
 *   e'[idx[j]] = val[j] - g_hat[j];  e'[i] = c[i] at every other i.
 */
int orc_ef_topk_quant(const float* grad, float* err, int64_t n, int64_t k,
                      int bits, int64_t group, int rounding, uint64_t seed,
                      uint64_t step, int32_t* idx_out, uint8_t* codes_out,
                      float* scales_out) {
  if (n < 0 || k < 0 || k > n || n > INT32_MAX || !err) return ORC_EINVAL;
  int st = check_quant_args(k, bits, group, ORC_QSGD, rounding);
  if (st != ORC_OK) return st;
  float* val = (float*)malloc((size_t)(k > 0 ? k : 1) * sizeof(float));
  float* g_hat = (float*)malloc((size_t)(k > 0 ? k : 1) * sizeof(float));
  if (!val || !g_hat) { free(val); free(g_hat); return ORC_ENOMEM; }
  st = orc_ef_topk(grad, err, n, k, idx_out, val); /* err := c, kept -> 0 */
  if (st == ORC_OK)
    st = quant_core(val, k, 0, bits, group, ORC_QSGD, rounding, seed, step,
                    codes_out, scales_out, g_hat);
  if (st == ORC_OK)
    for (int64_t j = 0; j < k; ++j) err[idx_out[j]] = val[j] - g_hat[j];
  free(val);
  free(g_hat);
  return st;
}

/* ------------------------------------------------------------------------ */
/* Random sparsification with error feedback.                                */
/* ------------------------------------------------------------------------ */

/*
 * [P2 二.2 随机稀疏化]: every element is kept with probability p (the page's
 * mask = rand(n) < p); [P1 2.2]: random sparsification keeps the traffic
 * steady.  With error feedback ([P4 梯度压缩原理]) the unsent entries stay in
 * the residual, as for Top-K:
 *   c = g + e;  keep i when u_i < p, u_i = orc_uniform(seed, step, i)
 *   (reading: the same Philox-4x32-10 draw as stochastic rounding);
 *   emit (i, c_i) of the kept entries in ascending index order;
 *   e'_i = +0 when kept, c_i otherwise.
 * At most `capacity` entries are written; *count receives how many were kept
 * (ORC_EINVAL when that exceeds the capacity, the first `capacity` written).
 * err == NULL selects from grad alone and writes no residual.
 */
int orc_ef_randk(const float* grad, float* err, int64_t n, float p, uint64_t seed,
                 uint64_t step, int32_t* idx_out, float* val_out, int64_t capacity,
                 int64_t* count) {
  if (n < 0 || n > INT32_MAX || capacity < 0 || !count) return ORC_EINVAL;
  int64_t kept = 0;
  for (int64_t i = 0; i < n; ++i) {
    float c = err ? grad[i] + err[i] : grad[i];
    int keep = orc_uniform(seed, step, (uint64_t)i) < p;
    if (keep) {
      if (kept < capacity) {
        idx_out[kept] = (int32_t)i;
        val_out[kept] = c;
      }
      ++kept;
    }
    if (err) err[i] = keep ? 0.0f : c;
  }
  *count = kept;
  return kept <= capacity ? ORC_OK : ORC_EINVAL;
}

/* ------------------------------------------------------------------------ */
/* Diagnostics of one compressed bucket.                                      */
/* ------------------------------------------------------------------------ */

/*
 * [P1 3.2]: production systems watch the ratio of the gradient norm after
 * compression to the norm before it; [P4 Python 演示] prints the error
 * energy, the sum of the squared residual, after each compression.  For one
 * compressed bucket, from the call's inputs and its transmitted values:
 *   c_i = g_i + e_i (binary32; g_i when e is NULL);
 *   g_hat_j, j < k: the value the receiver reconstructs for kept index
 *   idx[j] (strictly increasing);
 *   e'_i = c_i - g_hat_j (binary32) where i = idx[j], c_i elsewhere
 *   (for Top-K g_hat_j = c_i, so e'_i = +0: the residual the call stores);
 *   out[0] = sum_i c_i^2,  out[1] = sum_j g_hat_j^2,  out[2] = sum_i e'_i^2.
 * Reading: "before compression" is the gradient the compressor sees, c
 * (with error feedback the corrected gradient), so the norm ratio is
 * sqrt(out[1] / out[0]).  Every square of a binary32 value is exact in
 * binary64; the sums run in binary64 in index order.
 */
int orc_diagnostics(const float* grad, const float* err, int64_t n, const int32_t* idx,
                    const float* g_hat, int64_t k, double* out) {
  if (n < 0 || k < 0 || k > n || !out) return ORC_EINVAL;
  double s_c = 0.0, s_g = 0.0, s_e = 0.0;
  int64_t j = 0;
  for (int64_t i = 0; i < n; ++i) {
    float c = err ? grad[i] + err[i] : grad[i];
    float r = c;
    if (j < k && idx[j] == i) {
      r = c - g_hat[j];
      s_g += (double)g_hat[j] * (double)g_hat[j];
      ++j;
    }
    s_c += (double)c * (double)c;
    s_e += (double)r * (double)r;
  }
  if (j != k) return ORC_EINVAL; /* indices not increasing or out of range */
  out[0] = s_c;
  out[1] = s_g;
  out[2] = s_e;
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Aggregation of several ranks' compressed gradients.                       */
/* ------------------------------------------------------------------------ */

/*
 * [P2 四, the All-Reduce flow with compression]: every worker compresses its
 * local gradient, the compressed gradients are aggregated and decompressed,
 * and every worker applies the result.  With Top-K each rank keeps its own
 * positions and, quantised, its own scales, so the aggregate is the sum of
 * the ranks' decompressed sparse vectors.  Reading: the ranks are added in
 * rank order, one binary32 addition per present entry:
 *   out[i] = 0;  for w = 0 .. W-1:  out[idx_w[j]] += v_w[j]  (j ascending)
 * Inputs follow the compressor's output: rank w's k indices at
 * idx[w*K ..], K = k rounded up to a multiple of 4 (every rank's entries
 * start on a 16-byte boundary), strictly increasing in [0, n) (ORC_EINVAL
 * otherwise); values at the same positions.
 */
static int64_t rank_stride(int64_t k) { return (k + 3) / 4 * 4; }

static int check_aggregate_idx(int W, int64_t k, const int32_t* idx, int64_t n) {
  if (W < 1 || k < 0 || n < 0 || k > n) return ORC_EINVAL;
  for (int w = 0; w < W; ++w) {
    const int32_t* iw = idx + (int64_t)w * rank_stride(k);
    for (int64_t j = 0; j < k; ++j) {
      if (iw[j] < 0 || (int64_t)iw[j] >= n) return ORC_EINVAL;
      if (j > 0 && iw[j] <= iw[j - 1]) return ORC_EINVAL;
    }
  }
  return ORC_OK;
}

/* Rank w's values are val[w*K .. w*K + k). */
int orc_topk_aggregate(int W, int64_t k, const int32_t* idx, const float* val, int64_t n,
                       float* out) {
  int st = check_aggregate_idx(W, k, idx, n);
  if (st != ORC_OK) return st;
  for (int64_t i = 0; i < n; ++i) out[i] = 0.0f;
  for (int w = 0; w < W; ++w)
    for (int64_t j = 0; j < k; ++j) {
      int64_t at = (int64_t)w * rank_stride(k) + j;
      out[idx[at]] = out[idx[at]] + val[at];
    }
  return ORC_OK;
}

/*
 * QSGD-compressed ranks (the hybrid's output): rank w's values are
 * dequant(codes_w, scales_w, k, bits, group, QSGD) with codes_w at
 * codes + w * orc_codes_bytes(k, bits, QSGD) and scales_w at
 * scales + w * S, S = orc_scales_floats(k, group, QSGD) rounded up to a
 * multiple of 4 (each rank's scales start on a 16-byte boundary, as the
 * compressor writes them).
 */
int orc_topk_quant_aggregate(int W, int64_t k, const int32_t* idx, const uint8_t* codes,
                             const float* scales, int bits, int64_t group, int64_t n,
                             float* out) {
  int st = check_aggregate_idx(W, k, idx, n);
  if (st != ORC_OK) return st;
  st = check_quant_args(k, bits, group, ORC_QSGD, ORC_NEAREST_EVEN);
  if (st != ORC_OK) return st;
  int64_t cb = orc_codes_bytes(k, bits, ORC_QSGD);
  int64_t sf = (orc_scales_floats(k, group, ORC_QSGD) + 3) / 4 * 4;
  float* val = (float*)malloc((size_t)(k > 0 ? k : 1) * sizeof(float));
  if (!val) return ORC_ENOMEM;
  for (int64_t i = 0; i < n; ++i) out[i] = 0.0f;
  for (int w = 0; w < W && st == ORC_OK; ++w) {
    st = orc_dequant(codes + (int64_t)w * cb, scales + (int64_t)w * sf, k, bits, group,
                     ORC_QSGD, val);
    const int32_t* iw = idx + (int64_t)w * rank_stride(k);
    for (int64_t j = 0; st == ORC_OK && j < k; ++j) out[iw[j]] = out[iw[j]] + val[j];
  }
  free(val);
  return st;
}

/* ------------------------------------------------------------------------ */
/* PowerSGD step (binary64).                                                 */
/* ------------------------------------------------------------------------ */

/*
 * One rank-r PowerSGD step with error feedback ([P1 3.1]: a low-rank
 * approximation, send the two thin matrices, rebuild on the receiver;
 * [P4 梯度压缩原理]: error compensation makes PowerSGD work; Vogels et al.
 * Algorithm 1):
 *   M = G + E                      (m x n, row-major)
 *   P = M Q                        (m x r)
 *   P_hat = Gram-Schmidt(P)        (modified Gram-Schmidt, column by column;
 *                                   a column of norm 0 is left as zeros)
 *   Q' = M^T P_hat                 (n x r)
 *   E' = M - P_hat Q'^T
 * Inputs grad (m x n), err (m x n, overwritten with E'), Q_inout (n x r,
 * overwritten with Q'); P_out receives P_hat.
 */
int orc_powersgd_step(const float* grad, float* err, int64_t m, int64_t n,
                      int r, float* P_out, float* Q_inout) {
  if (m < 0 || n < 0 || r < 1) return ORC_EINVAL;
  if (m == 0 || n == 0) return ORC_OK;
  double* M = (double*)malloc((size_t)(m * n) * sizeof(double));
  double* P = (double*)calloc((size_t)(m * r), sizeof(double));
  double* Q = (double*)calloc((size_t)(n * r), sizeof(double));
  if (!M || !P || !Q) { free(M); free(P); free(Q); return ORC_ENOMEM; }
  for (int64_t i = 0; i < m * n; ++i) M[i] = (double)grad[i] + (double)err[i];
  for (int64_t i = 0; i < m; ++i)
    for (int c = 0; c < r; ++c) {
      double s = 0.0;
      for (int64_t j = 0; j < n; ++j)
        s += M[i * n + j] * (double)Q_inout[j * r + c];
      P[i * r + c] = s;
    }
  for (int c = 0; c < r; ++c) {
    for (int l = 0; l < c; ++l) {
      double d = 0.0;
      for (int64_t i = 0; i < m; ++i) d += P[i * r + l] * P[i * r + c];
      for (int64_t i = 0; i < m; ++i) P[i * r + c] -= d * P[i * r + l];
    }
    double nrm = 0.0;
    for (int64_t i = 0; i < m; ++i) nrm += P[i * r + c] * P[i * r + c];
    nrm = sqrt(nrm);
    if (nrm > 0.0)
      for (int64_t i = 0; i < m; ++i) P[i * r + c] /= nrm;
  }
  for (int64_t j = 0; j < n; ++j)
    for (int c = 0; c < r; ++c) {
      double s = 0.0;
      for (int64_t i = 0; i < m; ++i) s += M[i * n + j] * P[i * r + c];
      Q[j * r + c] = s;
    }
  for (int64_t i = 0; i < m; ++i)
    for (int64_t j = 0; j < n; ++j) {
      double a = 0.0;
      for (int c = 0; c < r; ++c) a += P[i * r + c] * Q[j * r + c];
      err[i * n + j] = (float)(M[i * n + j] - a);
    }
  for (int64_t i = 0; i < m * r; ++i) P_out[i] = (float)P[i];
  for (int64_t i = 0; i < n * r; ++i) Q_inout[i] = (float)Q[i];
  free(M);
  free(P);
  free(Q);
  return ORC_OK;
}
