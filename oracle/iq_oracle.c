/*
 * Plain CPU oracle for the importance-weighted GGML IQ codebook encoder, its decoder and the
 * per-expert imatrix statistic.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, includes or calls this file; only the
 * tests, the package's smoke() check and the benchmark's CPU-baseline leg load it.  It shares no
 * code, header, table or constant with the CUDA path: every format constant below is written out
 * again from the format description.
 *
 * It is deliberately slow and literal: every search evaluates the weighted squared error
 * sum_i w_i (x_i - q_i)^2 directly in fp64 for every candidate, with q the decoded fp32 value.
 * Blocks are independent, so the OpenMP loop over blocks does not change any result.
 *
 * Sources (pages are cited by title and section):
 *  - "Add imatrix calibration for the GGML formats and use it for fused MoE experts" (PR #2735),
 *    "What imatrix does": importance = sqrt(E[x_j^2]) per column, per routed expert; idle experts
 *    get the plain search; input rows squared 1,024 at a time; widths not a multiple of 256 refused.
 *  - "MoE expert coverage in imatrix calibration", Facts: top-k routed sum of squares and per-expert
 *    counts; non-finite sums checked only for touched experts; count 0 -> weight 1 on every channel;
 *    the per-expert slice of a merged tensor is global row / rows per expert.
 *  - PR #2513 (IQ2_XXS, IQ2_S, IQ1_M commit texts): 256-value blocks, fp16 super-block scale fixed
 *    (anchored) before a single-pass grid search; IQ2_XXS 4-bit sub-block scale packed with four
 *    7-bit sign indices in one 32-bit word; even-parity sign rule (flip the weakest element) for
 *    IQ2_XXS/IQ2_XS; IQ2_S full 8-bit sign mask taken as is; IQ1 +-1/8 delta shift; IQ1_M scale
 *    split over the top nibbles of four scale words, local scale per two groups, delta per group,
 *    tie order (lower shift, then lower entry); IQ1_S flat anchor 0.61, IQ1_M anchor
 *    clamp(0.58 + 0.035 * peak_to_rms, 0.65, 0.95); bits per weight of each format.
 *  - PR #3157 "[1/5] Let the GGML IQ encoders take fixed per-group choices": one choice per group
 *    (local scale, plus the delta sign for IQ1_S) picked by least weighted squared error; fixed
 *    choices keep the entry/sign search; choices must lie in [0, num_choices); all-zero blocks give
 *    all-zero payloads.  PR #3159 (one-pass every-choice encode): every choice's result from one
 *    sweep.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_IQ2_XXS = 0, OR_IQ2_XS = 1, OR_IQ2_S = 2, OR_IQ1_S = 3, OR_IQ1_M = 4 };

/* status bits (same meaning as the library's, written independently) */
#define OR_ST_BAD_CHOICE 1
#define OR_ST_BAD_EXPERT_ID 2
#define OR_ST_NONFINITE_SUM2 4
#define OR_ST_DUP_EXPERT_ID 8
#define OR_ST_BAD_INPUT 16
#define OR_ST_BAD_IMPORTANCE 32
#define OR_ST_BAD_SCALE 64
#define OR_ST_BAD_GRID 128

typedef struct {
  int block_bytes;   /* payload bytes per 256 values */
  int groups;        /* choice groups per block */
  int num_choices;   /* choices per group */
  int entries;       /* grid entries */
  int vpg;           /* 8-value vectors per choice group */
  int iq1;           /* 1: ternary grid with delta shift; 0: magnitude grid with signs */
} or_fmt;

static int or_get_fmt(int f, or_fmt *o) {
  switch (f) {
    case OR_IQ2_XXS: *o = (or_fmt){66, 8, 16, 256, 4, 0}; return 0;
    case OR_IQ2_XS:  *o = (or_fmt){74, 16, 16, 512, 2, 0}; return 0;
    case OR_IQ2_S:   *o = (or_fmt){82, 16, 16, 1024, 2, 0}; return 0;
    case OR_IQ1_S:   *o = (or_fmt){50, 8, 16, 2048, 4, 1}; return 0;
    case OR_IQ1_M:   *o = (or_fmt){56, 16, 8, 2048, 2, 1}; return 0;
  }
  return -1;
}

int or_format_info(int f, int *block_bytes, int *groups, int *num_choices, int *entries, int *vpg) {
  or_fmt o;
  if (or_get_fmt(f, &o)) return -1;
  *block_bytes = o.block_bytes; *groups = o.groups; *num_choices = o.num_choices;
  *entries = o.entries; *vpg = o.vpg;
  return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32, written from the format definition (round to nearest, ties to even). */

uint16_t or_half_from_float(float f) {
  uint32_t x; memcpy(&x, &f, 4);
  uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  uint32_t ex = (x >> 23) & 0xffu, man = x & 0x7fffffu;
  if (ex == 0xffu) return (uint16_t)(sign | 0x7c00u | (man ? 0x200u : 0u)); /* inf / nan */
  int e = (int)ex - 127;             /* unbiased exponent of a normal float */
  if (ex == 0) return sign;          /* float subnormals are far below half's range: +-0 */
  uint32_t sig = man | 0x800000u;    /* 24-bit significand, value = sig * 2^(e-23) */
  if (e > 15) return (uint16_t)(sign | 0x7c00u);
  int shift;                         /* bits of sig to drop */
  uint32_t hexp;
  if (e >= -14) { shift = 13; hexp = (uint32_t)(e + 15); }          /* normal half */
  else { shift = 13 + (-14 - e); hexp = 0; if (shift > 24) return sign; } /* subnormal half */
  uint32_t keep = sig >> shift;
  uint32_t rem = sig & ((1u << shift) - 1u);
  uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (keep & 1u))) keep += 1;
  uint32_t out;
  if (hexp == 0) {
    out = keep;                       /* may carry into the smallest normal: still correct */
  } else {
    if (keep >= 0x800u) { keep >>= 1; hexp += 1; }  /* significand overflow after rounding */
    if (hexp >= 31) return (uint16_t)(sign | 0x7c00u);
    out = (hexp << 10) | (keep & 0x3ffu);
  }
  return (uint16_t)(sign | out);
}

float or_float_from_half(uint16_t h) {
  uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  uint32_t ex = (h >> 10) & 0x1fu, man = h & 0x3ffu;
  float v;
  if (ex == 0) v = ldexpf((float)man, -24);
  else if (ex == 31) v = man ? NAN : INFINITY;
  else v = ldexpf((float)(man | 0x400u), (int)ex - 25);
  uint32_t b; memcpy(&b, &v, 4); b |= sign; memcpy(&v, &b, 4);
  return v;
}

void or_half_from_float_n(const float *in, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = or_half_from_float(in[i]);
}
void or_float_from_half_n(const uint16_t *in, float *out, int64_t n) {
  for (int64_t i = 0; i < n; i++) out[i] = or_float_from_half(in[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* imatrix: per routed expert, sum of squared activations and token counts.
 * Order (our reading of "squares 1,024 rows at a time"): for each chunk of rows_per_chunk rows, a
 * partial sum per (expert, column) starts at +0 and adds the square of each token of the chunk
 * routed to the expert, in ascending token order: the square is one rounded fp32 multiply, sq =
 * fl(x*x), and it is added with one rounded fp32 add, partial = fl(partial + sq) (the page squares
 * the rows, then sums them; this file is built without FMA contraction, so the two steps stay
 * apart); then in_sum2 += partial (one rounded fp32 add), chunk by chunk, for experts the chunk
 * routed at least one token to.  The same two steps serve bf16 activations (widened exactly):
 * their squares are exact in fp32 except below its normal range, where they round as well.
 * A token's top-k slots are read as a set: a repeated id counts once (and is reported). */
int or_imatrix_accumulate(const float *x, int64_t tokens, int64_t cols, const int32_t *ids, int top_k,
                          int E, int64_t rows_per_chunk, float *in_sum2, int64_t *counts,
                          int32_t *status) {
  if (tokens < 0 || cols <= 0 || top_k <= 0 || E <= 0 || rows_per_chunk <= 0) return -1;
  int32_t st = 0;
  float *partial = (float *)malloc(sizeof(float) * (size_t)E * (size_t)cols);
  unsigned char *touched = (unsigned char *)malloc((size_t)E);
  unsigned char *touched_call = (unsigned char *)calloc((size_t)E, 1);
  unsigned char *member = (unsigned char *)malloc((size_t)E);
  if (!partial || !touched || !touched_call || !member) return -2;
  for (int64_t t0 = 0; t0 < tokens; t0 += rows_per_chunk) {
    int64_t t1 = t0 + rows_per_chunk < tokens ? t0 + rows_per_chunk : tokens;
    memset(touched, 0, (size_t)E);
    for (int64_t t = t0; t < t1; t++) {
      memset(member, 0, (size_t)E);
      for (int k = 0; k < top_k; k++) {
        int32_t e = ids[t * top_k + k];
        if (e < 0 || e >= E) { st |= OR_ST_BAD_EXPERT_ID; continue; }
        if (member[e]) { st |= OR_ST_DUP_EXPERT_ID; continue; }
        member[e] = 1;
        if (!touched[e]) {
          touched[e] = 1;
          for (int64_t j = 0; j < cols; j++) partial[(int64_t)e * cols + j] = 0.0f;
        }
        counts[e] += 1;
        touched_call[e] = 1;
        const float *xr = x + t * cols;
        float *pr = partial + (int64_t)e * cols;
        for (int64_t j = 0; j < cols; j++) {
          const float sq = xr[j] * xr[j];
          pr[j] = pr[j] + sq;
        }
      }
    }
    for (int e = 0; e < E; e++) {
      if (!touched[e]) continue;
      for (int64_t j = 0; j < cols; j++)
        in_sum2[(int64_t)e * cols + j] = in_sum2[(int64_t)e * cols + j] + partial[(int64_t)e * cols + j];
    }
  }
  for (int e = 0; e < E; e++) {
    if (!touched_call[e]) continue;
    for (int64_t j = 0; j < cols; j++)
      if (!isfinite(in_sum2[(int64_t)e * cols + j])) { st |= OR_ST_NONFINITE_SUM2; break; }
  }
  free(partial); free(touched); free(touched_call); free(member);
  if (status) *status |= st;
  return 0;
}

/* importance weights: w = sqrt(in_sum2 / count), 1 for count 0; optional floor on the mean. */
int or_imatrix_weights(const float *in_sum2, const int64_t *counts, int E, int64_t cols, float floor_,
                       float *w) {
  if (E <= 0 || cols <= 0) return -1;
  for (int e = 0; e < E; e++) {
    for (int64_t j = 0; j < cols; j++) {
      int64_t i = (int64_t)e * cols + j;
      if (counts[e] == 0) { w[i] = 1.0f; continue; }
      float m = in_sum2[i] / (float)counts[e];
      if (floor_ > 0.0f && m < floor_) m = floor_;
      w[i] = sqrtf(m);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Super-block scale anchor.  d = (ratio * amax) / K, K = largest grid magnitude times the largest
 * local-scale multiplier: IQ2 43 * 31/8 = 166.625, IQ1 1 * 15 = 15.  IQ2 ratio = 1 (the pages give
 * none), IQ1_S 0.61, IQ1_M clamp(0.58 + 0.035 * amax/rms, 0.65, 0.95) with the sum of squares in a
 * fixed tree: 32 partial sums of 8 consecutive squares, then pairs (l, l+16), (l, l+8), ... */
static int block_finite(const float *x) {
  for (int i = 0; i < 256; i++) if (!isfinite(x[i])) return 0;
  return 1;
}

static float anchor_d(int f, const float *x) {
  float amax = 0.0f;
  for (int i = 0; i < 256; i++) { float a = fabsf(x[i]); if (a > amax) amax = a; }
  float ratio, K;
  if (f == OR_IQ1_S) { ratio = 0.61f; K = 15.0f; }
  else if (f == OR_IQ1_M) {
    float v[32];
    for (int l = 0; l < 32; l++) {
      float s = 0.0f;
      for (int i = 0; i < 8; i++) { float sq = x[8 * l + i] * x[8 * l + i]; s = s + sq; }
      v[l] = s;
    }
    for (int h = 16; h >= 1; h >>= 1)
      for (int l = 0; l < h; l++) v[l] = v[l] + v[l + h];
    float mean = v[0] / 256.0f;
    float rms = sqrtf(mean);
    float p2r = amax / rms;
    float r = 0.035f * p2r;
    r = 0.58f + r;
    if (r < 0.65f) r = 0.65f;
    if (r > 0.95f) r = 0.95f;
    ratio = r; K = 15.0f;
    if (amax == 0.0f) return 0.0f;
  } else { ratio = 1.0f; K = 166.625f; }
  float num = ratio * amax;
  return num / K;
}

static uint16_t anchor_d16(int f, const float *x) {
  float d = anchor_d(f, x);
  if (d > 65504.0f) d = 65504.0f;
  return or_half_from_float(d);
}

int or_anchor_scales(int f, const float *W, int64_t rows, int64_t cols, uint16_t *d16, int32_t *status) {
  or_fmt o;
  if (or_get_fmt(f, &o) || rows < 0 || cols <= 0 || cols % 256) return -1;
  int64_t nb = rows * (cols / 256);
  int32_t st = 0;
  for (int64_t b = 0; b < nb; b++) {
    const float *x = W + b * 256;
    if (!block_finite(x)) { d16[b] = 0; st |= OR_ST_BAD_INPUT; continue; }
    d16[b] = anchor_d16(f, x);
  }
  if (status) *status |= st;
  return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Decoded values.  IQ2: q = (d * (2s+1) * 1/8) * g, negated where the sign bit is set.
 * IQ1: q = (d * (2s+1)) * (g + delta), delta = +1/8 (delta bit 0) or -1/8 (delta bit 1). */
static inline float iq2_dl(float d, int s) { float a = d * (float)(2 * s + 1); return a * 0.125f; }
static inline float iq1_dl(float d, int s) { return d * (float)(2 * s + 1); }
static inline float iq1_delta(int dbit) { return dbit ? -0.125f : 0.125f; }

static inline void q_iq2(float dl, const float *g, int sgn8, float *q) {
  for (int i = 0; i < 8; i++) { float v = dl * g[i]; q[i] = ((sgn8 >> i) & 1) ? -v : v; }
}
static inline void q_iq1(float dl, const float *g, int dbit, float *q) {
  float dlt = iq1_delta(dbit);
  for (int i = 0; i < 8; i++) { float gd = g[i] + dlt; q[i] = dl * gd; }
}

static inline double vec_err(const float *x, const float *w, const float *q) {
  double acc = 0.0;
  for (int i = 0; i < 8; i++) {
    double d = (double)x[i] - (double)q[i];
    double t = (double)w[i] * (d * d);
    acc = acc + t;
  }
  return acc;
}

static inline int parity7(int s) { int p = 0; for (int i = 0; i < 7; i++) p ^= (s >> i) & 1; return p; }

/* Sign rule.  IQ2_XXS / IQ2_XS: signs of x; if an odd number are negative, flip the sign bit of
 * the weakest element, argmin_i w_i * x_i^2 in fp32 (lowest index on ties), so the stored 7 bits
 * imply the 8th by even parity.  IQ2_S: the 8-bit sign mask as is. */
static int sign_mask(int f, const float *x, const float *w) {
  int m = 0;
  for (int i = 0; i < 8; i++) if (x[i] < 0.0f) m |= 1 << i;
  if (f == OR_IQ2_S) return m;
  int pop = 0;
  for (int i = 0; i < 8; i++) pop += (m >> i) & 1;
  if (pop & 1) {
    int best = 0; float bk = 0.0f;
    for (int i = 0; i < 8; i++) {
      float sq = x[i] * x[i];
      float k = w[i] * sq;
      if (i == 0 || k < bk) { bk = k; best = i; }
    }
    m ^= 1 << best;
  }
  return m;
}

/* ------------------------------------------------------------------------------------------ */
/* Packing and unpacking (bit layout: the library header documents the same layout). */
typedef struct {
  uint16_t d16;
  int idx[32];
  int sgn[32];      /* IQ2: 8-bit mask (bit 7 implied by parity for XXS/XS) */
  int dbit[32];     /* IQ1_M: per-group delta bit */
  int choice[16];   /* per choice group */
} blockfields;

static void pack_block(int f, const blockfields *bf, uint8_t *p) {
  or_fmt o; or_get_fmt(f, &o);
  memset(p, 0, (size_t)o.block_bytes);
  if (f != OR_IQ1_M) { p[0] = (uint8_t)(bf->d16 & 0xff); p[1] = (uint8_t)(bf->d16 >> 8); }
  if (f == OR_IQ2_XXS) {
    for (int s = 0; s < 8; s++) {
      uint8_t *q = p + 2 + 8 * s;
      uint32_t word = 0;
      for (int k = 0; k < 4; k++) {
        q[k] = (uint8_t)bf->idx[4 * s + k];
        word |= (uint32_t)(bf->sgn[4 * s + k] & 0x7f) << (7 * k);
      }
      word |= (uint32_t)(bf->choice[s] & 0xf) << 28;
      for (int k = 0; k < 4; k++) q[4 + k] = (uint8_t)(word >> (8 * k));
    }
  } else if (f == OR_IQ2_XS) {
    for (int g = 0; g < 32; g++) {
      uint32_t v = (uint32_t)(bf->idx[g] & 0x1ff) | ((uint32_t)(bf->sgn[g] & 0x7f) << 9);
      p[2 + 2 * g] = (uint8_t)(v & 0xff); p[3 + 2 * g] = (uint8_t)(v >> 8);
    }
    for (int s = 0; s < 8; s++)
      p[66 + s] = (uint8_t)((bf->choice[2 * s] & 0xf) | ((bf->choice[2 * s + 1] & 0xf) << 4));
  } else if (f == OR_IQ2_S) {
    for (int g = 0; g < 32; g++) { p[2 + g] = (uint8_t)(bf->idx[g] & 0xff); p[34 + g] = (uint8_t)bf->sgn[g]; }
    for (int s = 0; s < 8; s++) {
      int h = 0;
      for (int k = 0; k < 4; k++) h |= ((bf->idx[4 * s + k] >> 8) & 3) << (2 * k);
      p[66 + s] = (uint8_t)h;
      p[74 + s] = (uint8_t)((bf->choice[2 * s] & 0xf) | ((bf->choice[2 * s + 1] & 0xf) << 4));
    }
  } else if (f == OR_IQ1_S) {
    for (int g = 0; g < 32; g++) p[2 + g] = (uint8_t)(bf->idx[g] & 0xff);
    for (int s = 0; s < 8; s++) {
      uint32_t v = 0;
      for (int k = 0; k < 4; k++) v |= (uint32_t)((bf->idx[4 * s + k] >> 8) & 7) << (3 * k);
      v |= (uint32_t)(bf->choice[s] & 7) << 12;
      v |= (uint32_t)((bf->choice[s] >> 3) & 1) << 15;
      p[34 + 2 * s] = (uint8_t)(v & 0xff); p[35 + 2 * s] = (uint8_t)(v >> 8);
    }
  } else { /* IQ1_M */
    for (int g = 0; g < 32; g++) p[g] = (uint8_t)(bf->idx[g] & 0xff);
    for (int g = 0; g < 32; g++) {
      int nib = ((bf->idx[g] >> 8) & 7) | ((bf->dbit[g] & 1) << 3);
      p[32 + g / 2] |= (uint8_t)(nib << (4 * (g & 1)));
    }
    for (int k = 0; k < 4; k++) {
      uint32_t v = 0;
      for (int j = 0; j < 4; j++) v |= (uint32_t)(bf->choice[4 * k + j] & 7) << (3 * j);
      v |= (uint32_t)((bf->d16 >> (4 * k)) & 0xf) << 12;
      p[48 + 2 * k] = (uint8_t)(v & 0xff); p[49 + 2 * k] = (uint8_t)(v >> 8);
    }
  }
}

/* Unpack into per-group (per 8 values) decode parameters: d, local scale s, grid index, 8-bit sign
 * mask (IQ2) or delta bit (IQ1). */
static void unpack_block(int f, const uint8_t *p, uint16_t *d16, int *s, int *idx, int *sgn, int *dbit) {
  if (f != OR_IQ1_M) *d16 = (uint16_t)(p[0] | (p[1] << 8));
  if (f == OR_IQ2_XXS) {
    for (int sb = 0; sb < 8; sb++) {
      const uint8_t *q = p + 2 + 8 * sb;
      uint32_t word = (uint32_t)q[4] | ((uint32_t)q[5] << 8) | ((uint32_t)q[6] << 16) | ((uint32_t)q[7] << 24);
      for (int k = 0; k < 4; k++) {
        int g = 4 * sb + k;
        idx[g] = q[k];
        int s7 = (int)((word >> (7 * k)) & 0x7f);
        sgn[g] = s7 | (parity7(s7) << 7);
        s[g] = (int)(word >> 28);
        dbit[g] = 0;
      }
    }
  } else if (f == OR_IQ2_XS) {
    for (int g = 0; g < 32; g++) {
      int v = p[2 + 2 * g] | (p[3 + 2 * g] << 8);
      idx[g] = v & 0x1ff;
      int s7 = (v >> 9) & 0x7f;
      sgn[g] = s7 | (parity7(s7) << 7);
      int sc = p[66 + g / 4];
      s[g] = ((g % 4) < 2) ? (sc & 0xf) : (sc >> 4);
      dbit[g] = 0;
    }
  } else if (f == OR_IQ2_S) {
    for (int g = 0; g < 32; g++) {
      int hi = (p[66 + g / 4] >> (2 * (g % 4))) & 3;
      idx[g] = p[2 + g] | (hi << 8);
      sgn[g] = p[34 + g];
      int sc = p[74 + g / 4];
      s[g] = ((g % 4) < 2) ? (sc & 0xf) : (sc >> 4);
      dbit[g] = 0;
    }
  } else if (f == OR_IQ1_S) {
    for (int g = 0; g < 32; g++) {
      int sb = g / 4, k = g % 4;
      int v = p[34 + 2 * sb] | (p[35 + 2 * sb] << 8);
      idx[g] = p[2 + g] | (((v >> (3 * k)) & 7) << 8);
      s[g] = (v >> 12) & 7;
      dbit[g] = (v >> 15) & 1;
      sgn[g] = 0;
    }
  } else {
    uint16_t d = 0;
    for (int k = 0; k < 4; k++) {
      int v = p[48 + 2 * k] | (p[49 + 2 * k] << 8);
      d |= (uint16_t)(((v >> 12) & 0xf) << (4 * k));
    }
    *d16 = d;
    for (int g = 0; g < 32; g++) {
      int nib = (p[32 + g / 2] >> (4 * (g & 1))) & 0xf;
      idx[g] = p[g] | ((nib & 7) << 8);
      dbit[g] = nib >> 3;
      int cg = g / 2, k = cg / 4, j = cg % 4;
      int v = p[48 + 2 * k] | (p[49 + 2 * k] << 8);
      s[g] = (v >> (3 * j)) & 7;
      sgn[g] = 0;
    }
  }
}

static void decode_block(int f, const uint8_t *p, const float *grid, float *out) {
  uint16_t d16 = 0; int s[32], idx[32], sgn[32], dbit[32];
  unpack_block(f, p, &d16, s, idx, sgn, dbit);
  float d = or_float_from_half(d16);
  for (int g = 0; g < 32; g++) {
    if (f >= OR_IQ1_S) q_iq1(iq1_dl(d, s[g]), grid + 8 * idx[g], dbit[g], out + 8 * g);
    else q_iq2(iq2_dl(d, s[g]), grid + 8 * idx[g], sgn[g], out + 8 * g);
  }
}

int or_decode(int f, const uint8_t *payload, int64_t rows, int64_t cols, const float *grid, float *out) {
  or_fmt o;
  if (or_get_fmt(f, &o) || rows < 0 || cols <= 0 || cols % 256) return -1;
  int64_t nb = rows * (cols / 256);
  for (int64_t b = 0; b < nb; b++) decode_block(f, payload + b * o.block_bytes, grid, out + b * 256);
  return 0;
}

/* ------------------------------------------------------------------------------------------ */
static int grid_ok(int f, const float *grid, int n) {
  for (int i = 0; i < 8 * n; i++) {
    float v = grid[i];
    if (f >= OR_IQ1_S) { if (!(v == -1.0f || v == 0.0f || v == 1.0f)) return 0; }
    else { if (!(v >= 1.0f && v <= 127.0f && v == floorf(v))) return 0; }
  }
  return 1;
}

static const float *row_importance(const float *imp, int64_t rows_per_expert, int64_t cols, int64_t row) {
  if (!imp) return NULL;
  if (rows_per_expert <= 0) return imp;
  return imp + (row / rows_per_expert) * cols;
}

/* Per-vector error at one choice, minimised over the vector's candidates.  For IQ2 the candidate
 * is the grid entry; for IQ1_S the delta comes with the choice; for IQ1_M the candidate is
 * (delta bit, entry) in that key order.  Candidates are visited in ascending key order and only a
 * strictly smaller error replaces the best, so ties go to the lowest key. */
static double vec_best(int f, const or_fmt *o, const float *x, const float *w, const float *grid,
                       float d, int c, int sgn8, int *best_idx, int *best_dbit, double *second) {
  double best = INFINITY, sec = INFINITY;
  int bi = 0, bd = 0;
  float q[8];
  if (f < OR_IQ1_S) {
    float dl = iq2_dl(d, c);
    for (int e = 0; e < o->entries; e++) {
      q_iq2(dl, grid + 8 * e, sgn8, q);
      double err = vec_err(x, w, q);
      if (err < best) { sec = best; best = err; bi = e; }
      else if (err < sec) sec = err;
    }
  } else if (f == OR_IQ1_S) {
    float dl = iq1_dl(d, c & 7);
    int db = c >> 3;
    for (int e = 0; e < o->entries; e++) {
      q_iq1(dl, grid + 8 * e, db, q);
      double err = vec_err(x, w, q);
      if (err < best) { sec = best; best = err; bi = e; }
      else if (err < sec) sec = err;
    }
    bd = db;
  } else {
    float dl = iq1_dl(d, c);
    for (int db = 0; db < 2; db++)
      for (int e = 0; e < o->entries; e++) {
        q_iq1(dl, grid + 8 * e, db, q);
        double err = vec_err(x, w, q);
        if (err < best) { sec = best; best = err; bi = e; bd = db; }
        else if (err < sec) sec = err;
      }
  }
  *best_idx = bi; *best_dbit = bd;
  if (second) *second = sec;
  return best;
}

/* Encode.  Optional outputs for the tests:
 *   table   [B, G, C]  weighted squared error of every (choice group, choice); NaN for choices a
 *                      fixed-choice call did not evaluate
 *   gbest   [B, G]     error of the chosen choice;  gsecond [B, G] best error of any other choice
 *   vbest   [B, 32]    error of each vector's chosen candidate; vsecond [B, 32] its runner-up
 *   chosen  [B, G]     the chosen choice */
int or_encode(int f, const float *W, int64_t rows, int64_t cols, const float *importance,
              int64_t rows_per_expert, const float *grid, const uint16_t *d16_in, const uint8_t *choices,
              uint8_t *payload, double *table, double *gbest, double *gsecond, double *vbest,
              double *vsecond, uint8_t *chosen, int32_t *status, int threads, int entries) {
  or_fmt o;
  if (or_get_fmt(f, &o) || rows < 0 || cols <= 0 || cols % 256) return -1;
  /* entries > 0 searches only the first `entries` codebook rows (a smaller codebook in the same
   * layout); the brute-force tests use it to enumerate whole groups. */
  if (entries > 0) { if (entries > o.entries) return -1; o.entries = entries; }
  if (rows_per_expert > 0 && rows % rows_per_expert) return -1;
  const int64_t bpr = cols / 256, nb = rows * bpr;
  int32_t st = 0;
  if (!grid_ok(f, grid, o.entries)) {
    memset(payload, 0, (size_t)(nb * o.block_bytes));
    if (status) *status |= OR_ST_BAD_GRID;
    return 0;
  }
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : st)
#endif
  for (int64_t b = 0; b < nb; b++) {
    const int64_t row = b / bpr, kb = b % bpr;
    const float *x = W + b * 256;
    const float *wr = row_importance(importance, rows_per_expert, cols, row);
    float w[256];
    for (int i = 0; i < 256; i++) w[i] = wr ? wr[kb * 256 + i] : 1.0f;
    uint8_t *p = payload + b * o.block_bytes;
    if (table) for (int i = 0; i < o.groups * o.num_choices; i++) table[b * o.groups * o.num_choices + i] = NAN;
    if (gbest) for (int i = 0; i < o.groups; i++) { gbest[b * o.groups + i] = 0.0; gsecond[b * o.groups + i] = NAN; }
    if (vbest) for (int i = 0; i < 32; i++) { vbest[b * 32 + i] = 0.0; vsecond[b * 32 + i] = NAN; }
    if (chosen) memset(chosen + b * o.groups, 0, (size_t)o.groups);
    int bad = 0;
    if (!block_finite(x)) { st |= OR_ST_BAD_INPUT; bad = 1; }
    for (int i = 0; i < 256 && !bad; i++) if (!(w[i] >= 0.0f) || !isfinite(w[i])) { st |= OR_ST_BAD_IMPORTANCE; bad = 1; }
    uint16_t d16 = 0;
    if (!bad) {
      d16 = d16_in ? d16_in[b] : anchor_d16(f, x);
      if ((d16 & 0x8000u) || (d16 & 0x7c00u) == 0x7c00u) {
        if ((d16 & 0x7fffu) != 0 || (d16 & 0x7c00u) == 0x7c00u) { st |= OR_ST_BAD_SCALE; bad = 1; }
        else d16 = 0; /* -0 is a zero scale */
      }
    }
    if (!bad && choices)
      for (int g = 0; g < o.groups; g++) if (choices[b * o.groups + g] >= o.num_choices) { st |= OR_ST_BAD_CHOICE; bad = 1; }
    if (bad || d16 == 0) {
      memset(p, 0, (size_t)o.block_bytes);
      if (!bad) {
        /* a zero scale decodes every choice to zeros: report that payload's error */
        float zq[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int g = 0; g < o.groups; g++) {
          double Eg = 0.0;
          for (int k = 0; k < o.vpg; k++) {
            int v = g * o.vpg + k;
            double e = vec_err(x + 8 * v, w + 8 * v, zq);
            if (vbest) vbest[b * 32 + v] = e;
            Eg = Eg + e;
          }
          if (table) for (int c = 0; c < o.num_choices; c++) table[(b * o.groups + g) * o.num_choices + c] = Eg;
          if (gbest) gbest[b * o.groups + g] = Eg;
        }
      }
      continue;
    }
    const float d = or_float_from_half(d16);
    blockfields bf; memset(&bf, 0, sizeof bf);
    bf.d16 = d16;
    int sg[32];
    for (int v = 0; v < 32; v++) sg[v] = (f < OR_IQ1_S) ? sign_mask(f, x + 8 * v, w + 8 * v) : 0;
    for (int g = 0; g < o.groups; g++) {
      double bestE = INFINITY, secE = INFINITY;
      int bestc = 0;
      int c0 = 0, c1 = o.num_choices;
      if (choices) { c0 = choices[b * o.groups + g]; c1 = c0 + 1; }
      for (int c = c0; c < c1; c++) {
        double Eg = 0.0;
        for (int k = 0; k < o.vpg; k++) {
          int v = g * o.vpg + k, bi, bd;
          Eg = Eg + vec_best(f, &o, x + 8 * v, w + 8 * v, grid, d, c, sg[v], &bi, &bd, NULL);
        }
        if (table) table[(b * o.groups + g) * o.num_choices + c] = Eg;
        if (Eg < bestE) { secE = bestE; bestE = Eg; bestc = c; }
        else if (Eg < secE) secE = Eg;
      }
      bf.choice[g] = bestc;
      if (chosen) chosen[b * o.groups + g] = (uint8_t)bestc;
      if (gbest) { gbest[b * o.groups + g] = bestE; gsecond[b * o.groups + g] = choices ? NAN : secE; }
      for (int k = 0; k < o.vpg; k++) {
        int v = g * o.vpg + k, bi, bd;
        double sec;
        double be = vec_best(f, &o, x + 8 * v, w + 8 * v, grid, d, bestc, sg[v], &bi, &bd, &sec);
        bf.idx[v] = bi; bf.dbit[v] = bd; bf.sgn[v] = sg[v];
        if (vbest) { vbest[b * 32 + v] = be; vsecond[b * 32 + v] = sec; }
      }
    }
    pack_block(f, &bf, p);
  }
  if (status) *status |= st;
  return 0;
}

/* Weighted squared error of a given payload, per choice group and per vector (decode, then the
 * direct fp64 form).  The parity tests use it to judge a differing group under the near-tie rule. */
int or_payload_errors(int f, const float *W, int64_t rows, int64_t cols, const float *importance,
                      int64_t rows_per_expert, const float *grid, const uint8_t *payload, double *gerr,
                      double *verr) {
  or_fmt o;
  if (or_get_fmt(f, &o) || rows < 0 || cols <= 0 || cols % 256) return -1;
  const int64_t bpr = cols / 256, nb = rows * bpr;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
  for (int64_t b = 0; b < nb; b++) {
    const int64_t row = b / bpr, kb = b % bpr;
    const float *x = W + b * 256;
    const float *wr = row_importance(importance, rows_per_expert, cols, row);
    float w[256], q[256];
    for (int i = 0; i < 256; i++) w[i] = wr ? wr[kb * 256 + i] : 1.0f;
    decode_block(f, payload + b * o.block_bytes, grid, q);
    for (int g = 0; g < o.groups; g++) {
      double Eg = 0.0;
      for (int k = 0; k < o.vpg; k++) {
        int v = g * o.vpg + k;
        double e = vec_err(x + 8 * v, w + 8 * v, q + 8 * v);
        if (verr) verr[b * 32 + v] = e;
        Eg = Eg + e;
      }
      if (gerr) gerr[b * o.groups + g] = Eg;
    }
  }
  return 0;
}
