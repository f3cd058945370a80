/*
 * kvq_oracle.c -- plain scalar CPU oracle for the KV-cache codec.
 *
 * TEST INFRASTRUCTURE ONLY (see kvq_oracle.h).  Slow on purpose: one element at a
 * time, in the order the method states, so that a reader can check it by eye.
 *
 * Sources (page title, then the section of the page):
 *  - "vllm-rlt PR #166: INT4 KV packing/unpacking and cross-loop residual
 *    reconstruction", Purpose: the INT4 affine codec works in FP32 and keeps its
 *    minimum and scale as FP16; the NVFP4 codec rounds elements to the nearest
 *    E2M1 value (ties even) under E4M3 scales of 16-value blocks and one FP32
 *    scale; a scale so small that its reciprocal is infinite is divided by
 *    directly; K groups run along token rows at a fixed (head, channel) and V
 *    groups along channels at a fixed (token, head); a residual is the current
 *    tensor minus the reconstruction of its predecessor, taken in bf16; sparse
 *    residuals keep their rows packed together with an int32 map of positions,
 *    and a row missing from the map keeps its predecessor.  Review by 0z5a: the
 *    G64 format spends 4 + 32/64 bits on each element; the codes come from the
 *    FP32 minimum and scale, which are rounded to FP16 only afterwards.
 *  - "feat(kvcache): add nvfp4 kv quantization (FreeToken PR #408)", Summary and the
 *    codec-delta port note: each (token, KV head) row has its own FP32 scale; two
 *    E2M1 codes share a byte, the even element in the low nibble; every 16 values
 *    share an E4M3 scale, and elements are quantised against that scale after
 *    its rounding; a head_dim-128 row takes 76 B; the paged store reads its
 *    destination slots from a device tensor.
 *
 * Readings where the pages leave a step open, one per step of the method:
 *  R1  row scale rs = amax / 2688 (2688 = 6 * 448), stored as the decode multiplier.
 *  R2  block scale target t = (vb / 6) / rs, clamped to 448, then E4M3 RNE.
 *  R3  s = bs * rs; s == 0 -> every code is a signed zero; inv = 1/s; if inv is
 *      infinite the element is divided by s instead of multiplied by inv.
 *  R4  decode y = bf16((e2m1 * bs) * rs): the inner product is exact.
 *  R5  INT4: sc = (mx - mn) / 15; sc == 0 -> codes 0; code = clamp(rint((x-mn)/sc),0,15)
 *      with ties to even; decode y = bf16(code * sc16 + mn16) as a mul then an add.
 *  R6  INT4 nibble order: low nibble = even channel.
 *  R7  residual r = bf16(cur - prev) in fp32; decode out = bf16(prev + unpack(r)).
 */
#include "kvq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* bit views                                                                  */
/* ------------------------------------------------------------------------- */
static uint32_t f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}
static float bits_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ------------------------------------------------------------------------- */
/* bf16: the upper 16 bits of a binary32                                      */
/* ------------------------------------------------------------------------- */
float orc_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/* Round a binary32 to the nearest bf16, ties to the even bf16.  In sign-magnitude
 * form the bf16 just below |f| is the top 16 bits; the 16 dropped bits decide
 * whether the magnitude steps up by one unit (a carry into the exponent, or to
 * infinity, is the correct result of that step). */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u = f32_bits(f);
  if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t kept = u >> 16;
  uint32_t dropped = u & 0xFFFFu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

/* ------------------------------------------------------------------------- */
/* IEEE binary16 (used for the INT4 min/scale metadata)                       */
/* ------------------------------------------------------------------------- */
float orc_f16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  float v;
  if (e == 0)
    v = ldexpf((float)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = (m == 0) ? INFINITY : NAN;
  else
    v = ldexpf((float)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/* Nearest binary16, ties to even.  The value is split as n * ulp with ulp the
 * spacing of binary16 at |f|; n is rounded to the nearest integer (ties even),
 * which is exact in double because |f| has 24 significant bits. */
uint16_t orc_f32_to_f16(float f) {
  uint16_t sign = signbit(f) ? 0x8000u : 0;
  double a = fabs((double)f);
  if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
  if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u); /* beyond the 65504/65536 midpoint */
  if (a == 0.0) return sign;
  int ex;
  frexp(a, &ex);        /* a = mant * 2^ex with mant in [0.5, 1) */
  int e = ex - 1;       /* floor(log2 a) */
  if (e < -14) e = -14; /* subnormal range shares the spacing of the smallest binade */
  double ulp = ldexp(1.0, e - 10);
  double n = nearbyint(a / ulp); /* default rounding mode: nearest, ties to even */
  uint32_t bits;
  if (a < ldexp(1.0, -14)) {
    bits = (uint32_t)n; /* subnormal (n == 1024 is exactly the smallest normal) */
  } else {
    /* normal: n in [1024, 2048]; n == 2048 carries into the next exponent */
    bits = ((uint32_t)(e + 15) << 10) + (uint32_t)(n - 1024.0);
  }
  return (uint16_t)(sign | bits);
}

/* ------------------------------------------------------------------------- */
/* E2M1 (FP4): sign, 2 exponent bits (bias 1), 1 mantissa bit                 */
/* ------------------------------------------------------------------------- */
static double e2m1_magnitude(int mag_code) { /* mag_code in 0..7 */
  int e = (mag_code >> 1) & 3;
  int m = mag_code & 1;
  if (e == 0) return 0.5 * m;                    /* subnormal: 2^(1-1) * m/2 */
  return ldexp(1.0 + 0.5 * m, e - 1);            /* 2^(e-1) * (1 + m/2) */
}

float orc_e2m1_value(uint8_t code) {
  double v = e2m1_magnitude(code & 7);
  return (float)((code & 8) ? -v : v);
}

/* Index of the value nearest to a among n ascending non-negative values (vals[0]
 * == 0); ties go to the even index, which is the even significand; a at or above
 * the largest value saturates to it.  Midpoints of neighbouring values of these
 * tiny formats are exact in double, so every comparison is exact. */
static int nearest_even_index(double a, const double* vals, int n) {
  if (a >= vals[n - 1]) return n - 1;
  int i = 0;
  while (vals[i + 1] <= a) i++; /* vals[i] <= a < vals[i+1] */
  double mid = 0.5 * (vals[i] + vals[i + 1]);
  if (a < mid) return i;
  if (a > mid) return i + 1;
  return (i % 2 == 0) ? i : i + 1;
}

uint8_t orc_e2m1_encode(float q) {
  double mags[8];
  for (int c = 0; c < 8; c++) mags[c] = e2m1_magnitude(c);
  double a = fabs((double)q);
  int c = nearest_even_index(a, mags, 8); /* saturates at 6 */
  return (uint8_t)((signbit(q) ? 8 : 0) | c);
}

/* ------------------------------------------------------------------------- */
/* E4M3 ("fn"): sign, 4 exponent bits (bias 7), 3 mantissa bits; no infinity, */
/* 0x7F / 0xFF are NaN; largest finite 448, smallest subnormal 2^-9.          */
/* ------------------------------------------------------------------------- */
static double e4m3_magnitude(int code7) { /* code7 in 0..126 */
  int e = (code7 >> 3) & 15;
  int m = code7 & 7;
  if (e == 0) return ldexp((double)m, -9);       /* 2^(1-7) * m/8 */
  return ldexp(1.0 + m / 8.0, e - 7);             /* 2^(e-7) * (1 + m/8) */
}

float orc_e4m3_value(uint8_t code) {
  if ((code & 0x7F) == 0x7F) return NAN;
  double v = e4m3_magnitude(code & 0x7F);
  return (float)((code & 0x80) ? -v : v);
}

uint8_t orc_e4m3_encode(float t) {
  double mags[127];
  for (int c = 0; c < 127; c++) mags[c] = e4m3_magnitude(c);
  double a = fabs((double)t);
  int c = nearest_even_index(a, mags, 127); /* saturates at 448 */
  return (uint8_t)((signbit(t) ? 0x80 : 0) | c);
}

int orc_subnormals_kept(void) {
  /* volatile operands: the products are computed at run time, under the FPU modes
   * this process runs with */
  volatile float smallest_normal = 0x1p-126f, half = 0.5f, sub = 0x1p-140f, two = 2.0f;
  const float r1 = smallest_normal * half; /* a subnormal result: 2^-127 */
  const float r2 = sub * two;              /* a subnormal operand and result: 2^-139 */
  return r1 == 0x1p-127f && r2 == 0x1p-139f && r2 != 0.0f;
}

void orc_f32_to_bf16_n(const float* x, int64_t n, uint16_t* y) {
  for (int64_t i = 0; i < n; i++) y[i] = orc_f32_to_bf16(x[i]);
}
void orc_f32_to_f16_n(const float* x, int64_t n, uint16_t* y) {
  for (int64_t i = 0; i < n; i++) y[i] = orc_f32_to_f16(x[i]);
}
void orc_e2m1_encode_n(const float* x, int64_t n, uint8_t* y) {
  for (int64_t i = 0; i < n; i++) y[i] = orc_e2m1_encode(x[i]);
}
void orc_e4m3_encode_n(const float* x, int64_t n, uint8_t* y) {
  for (int64_t i = 0; i < n; i++) y[i] = orc_e4m3_encode(x[i]);
}

/* ------------------------------------------------------------------------- */
/* NVFP4 row codec                                                            */
/* ------------------------------------------------------------------------- */
void orc_nvfp4_encode_row(const uint16_t* x, int D, uint8_t* codes, uint8_t* bscale,
                          float* rscale) {
  /* row amax and the FP32 row scale (R1) */
  float amax = 0.0f;
  for (int i = 0; i < D; i++) amax = fmaxf(amax, fabsf(orc_bf16_to_f32(x[i])));
  const float E2M1_MAX = 6.0f, E4M3_MAX = 448.0f;
  float rs = amax / (E2M1_MAX * E4M3_MAX);
  *rscale = rs;

  for (int i = 0; i < D / 2; i++) codes[i] = 0;
  for (int b = 0; b < D / 16; b++) {
    /* block amax and the E4M3 block scale (R2) */
    float vb = 0.0f;
    for (int j = 0; j < 16; j++) vb = fmaxf(vb, fabsf(orc_bf16_to_f32(x[16 * b + j])));
    float t = 0.0f;
    if (rs != 0.0f) t = (vb / E2M1_MAX) / rs;
    if (t > E4M3_MAX) t = E4M3_MAX;
    uint8_t bsb = orc_e4m3_encode(t);
    bscale[b] = bsb;
    float bs = orc_e4m3_value(bsb); /* quantise against the STORED block scale */

    /* element codes against s = bs * rs (R3) */
    float s = bs * rs;
    float inv = 0.0f;
    if (s != 0.0f) inv = 1.0f / s;
    for (int j = 0; j < 16; j++) {
      int i = 16 * b + j;
      float xi = orc_bf16_to_f32(x[i]);
      float q;
      if (s == 0.0f)
        q = copysignf(0.0f, xi);
      else if (isinf(inv))
        q = xi / s; /* tiny scale: direct division */
      else
        q = xi * inv;
      uint8_t c = orc_e2m1_encode(q);
      c = (uint8_t)((c & 7) | (signbit(xi) ? 8 : 0)); /* the sign is always x's */
      codes[i / 2] |= (uint8_t)((i % 2 == 0) ? c : (c << 4)); /* low nibble first */
    }
  }
}

void orc_nvfp4_decode_row(const uint8_t* codes, const uint8_t* bscale, float rscale, int D,
                          uint16_t* y) {
  for (int i = 0; i < D; i++) {
    uint8_t byte = codes[i / 2];
    uint8_t c = (i % 2 == 0) ? (byte & 15) : (byte >> 4);
    float bs = orc_e4m3_value(bscale[i / 16]);
    float v = orc_e2m1_value(c) * bs; /* exact: 2 x 4 significant bits */
    v = v * rscale;                   /* the one fp32 rounding (R4) */
    y[i] = orc_f32_to_bf16(v);
  }
}

void orc_nvfp4_encode_rows(const uint16_t* x, int64_t n, int D, uint8_t* codes,
                           uint8_t* bscale, float* rscale) {
  for (int64_t r = 0; r < n; r++)
    orc_nvfp4_encode_row(x + r * D, D, codes + r * (D / 2), bscale + r * (D / 16), rscale + r);
}

void orc_nvfp4_decode_rows(const uint8_t* codes, const uint8_t* bscale, const float* rscale,
                           int64_t n, int D, uint16_t* y) {
  for (int64_t r = 0; r < n; r++)
    orc_nvfp4_decode_row(codes + r * (D / 2), bscale + r * (D / 16), rscale[r], D, y + r * D);
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 row codec ("feat(kvcache): add nvfp4 kv quantization (FreeToken PR */
/* #408)", fp8 store notes: every element of a row is stored as one E4M3     */
/* byte, and the row has one FP32 scale).  Readings, as for NVFP4:             */
/* rs = amax / 448 stored as the decode multiplier; q = x * (1 / rs), or       */
/* x / rs when the reciprocal                                                  */
/* overflows; code = e4m3_rne(q) (saturating at 448, sign of x);               */
/* decode y = bf16(e4m3 * rs).                                                 */
/* ------------------------------------------------------------------------- */
void orc_fp8_encode_row(const uint16_t* x, int D, uint8_t* codes, float* rscale) {
  float amax = 0.0f;
  for (int i = 0; i < D; i++) amax = fmaxf(amax, fabsf(orc_bf16_to_f32(x[i])));
  const float E4M3_MAX = 448.0f;
  float rs = amax / E4M3_MAX;
  *rscale = rs;
  float inv = 0.0f;
  if (rs != 0.0f) inv = 1.0f / rs;
  for (int i = 0; i < D; i++) {
    float xi = orc_bf16_to_f32(x[i]);
    float q;
    if (rs == 0.0f)
      q = copysignf(0.0f, xi);
    else if (isinf(inv))
      q = xi / rs;
    else
      q = xi * inv;
    uint8_t c = orc_e4m3_encode(q);
    codes[i] = (uint8_t)((c & 0x7F) | (signbit(xi) ? 0x80 : 0));
  }
}

void orc_fp8_decode_row(const uint8_t* codes, float rscale, int D, uint16_t* y) {
  for (int i = 0; i < D; i++) y[i] = orc_f32_to_bf16(orc_e4m3_value(codes[i]) * rscale);
}

void orc_fp8_encode_rows(const uint16_t* x, int64_t n, int D, uint8_t* codes, float* rscale) {
  for (int64_t r = 0; r < n; r++) orc_fp8_encode_row(x + r * D, D, codes + r * D, rscale + r);
}

void orc_fp8_decode_rows(const uint8_t* codes, const float* rscale, int64_t n, int D, uint16_t* y) {
  for (int64_t r = 0; r < n; r++) orc_fp8_decode_row(codes + r * D, rscale[r], D, y + r * D);
}

/* ------------------------------------------------------------------------- */
/* paged store and restore                                                    */
/* ------------------------------------------------------------------------- */
uint32_t orc_nvfp4_scatter(const uint16_t* x, int64_t row_pitch, int64_t head_pitch, int T,
                           int H, int D, const int64_t* slot_ids, int64_t num_slots,
                           uint8_t* codes, uint8_t* bscale, float* rscale) {
  uint32_t status = 0;
  uint16_t row[4096];
  for (int t = 0; t < T; t++) {
    int64_t slot = slot_ids[t];
    if (slot < 0) continue; /* padding token */
    if (slot >= num_slots) {
      status |= ORC_BAD_SLOT;
      continue;
    }
    for (int h = 0; h < H; h++) {
      for (int d = 0; d < D; d++) row[d] = x[(int64_t)t * row_pitch + (int64_t)h * head_pitch + d];
      int64_t r = slot * H + h;
      orc_nvfp4_encode_row(row, D, codes + r * (D / 2), bscale + r * (D / 16), rscale + r);
    }
  }
  return status;
}

uint32_t orc_nvfp4_restore(const uint8_t* codes, const uint8_t* bscale, const float* rscale,
                           int64_t num_slots, int H, int D, int block_size,
                           const int32_t* block_table, int S, int max_blocks,
                           const int32_t* seq_lens, int Tmax, uint16_t* out) {
  uint32_t status = 0;
  int64_t num_blocks = num_slots / block_size;
  int64_t cap = (int64_t)max_blocks * block_size;
  if (cap > Tmax) cap = Tmax;
  for (int s = 0; s < S; s++) {
    int len = seq_lens[s];
    if (len < 0 || len > cap) {
      status |= ORC_BAD_SEQLEN;
      continue;
    }
    for (int t = 0; t < len; t++) {
      int32_t block = block_table[(int64_t)s * max_blocks + t / block_size];
      if (block < 0 || block >= num_blocks) {
        status |= ORC_BAD_BLOCK;
        continue;
      }
      int64_t slot = (int64_t)block * block_size + t % block_size;
      for (int h = 0; h < H; h++) {
        int64_t r = slot * H + h;
        uint16_t* y = out + (((int64_t)s * Tmax + t) * H + h) * D;
        orc_nvfp4_decode_row(codes + r * (D / 2), bscale + r * (D / 16), rscale[r], D, y);
      }
    }
  }
  return status;
}

uint32_t orc_fp8_scatter(const uint16_t* x, int64_t row_pitch, int64_t head_pitch, int T, int H,
                         int D, const int64_t* slot_ids, int64_t num_slots, uint8_t* codes,
                         float* rscale) {
  uint32_t status = 0;
  uint16_t row[4096];
  for (int t = 0; t < T; t++) {
    int64_t slot = slot_ids[t];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      status |= ORC_BAD_SLOT;
      continue;
    }
    for (int h = 0; h < H; h++) {
      for (int d = 0; d < D; d++) row[d] = x[(int64_t)t * row_pitch + (int64_t)h * head_pitch + d];
      int64_t r = slot * H + h;
      orc_fp8_encode_row(row, D, codes + r * D, rscale + r);
    }
  }
  return status;
}

uint32_t orc_fp8_restore(const uint8_t* codes, const float* rscale, int64_t num_slots, int H,
                         int D, int block_size, const int32_t* block_table, int S,
                         int max_blocks, const int32_t* seq_lens, int Tmax, uint16_t* out) {
  uint32_t status = 0;
  int64_t num_blocks = num_slots / block_size;
  int64_t cap = (int64_t)max_blocks * block_size;
  if (cap > Tmax) cap = Tmax;
  for (int s = 0; s < S; s++) {
    int len = seq_lens[s];
    if (len < 0 || len > cap) {
      status |= ORC_BAD_SEQLEN;
      continue;
    }
    for (int t = 0; t < len; t++) {
      int32_t block = block_table[(int64_t)s * max_blocks + t / block_size];
      if (block < 0 || block >= num_blocks) {
        status |= ORC_BAD_BLOCK;
        continue;
      }
      int64_t slot = (int64_t)block * block_size + t % block_size;
      for (int h = 0; h < H; h++) {
        int64_t r = slot * H + h;
        orc_fp8_decode_row(codes + r * D, rscale[r], D, out + (((int64_t)s * Tmax + t) * H + h) * D);
      }
    }
  }
  return status;
}

/* ------------------------------------------------------------------------- */
/* NVFP4 with one FP32 scale per tensor ("vllm-rlt PR #166", Purpose: blocks   */
/* of 16 with E4M3 scales, plus one FP32 number for the whole tensor, as in     */
/* vLLM's reference; K blocks run along token rows, V blocks along channels;   */
/* the last block may be short).  The scale is the tensor's amax / 2688,       */
/* stored as the decode multiplier (R1 read per tensor); each block follows    */
/* R2-R3 against it.                                                           */
/* ------------------------------------------------------------------------- */
static int64_t nvfp4t_elem(int kind, int H, int D, int g, int h, int j, int k) {
  /* element k (0..15) of block j: VALUE block j = (t, h, 16-channel block), KEY block = (group, h, d) */
  if (kind == ORC_KIND_VALUE) return ((int64_t)g * H + h) * D + 16 * j + k;
  return ((int64_t)(16 * g + k) * H + h) * D + j;
}

void orc_nvfp4t_pack(const uint16_t* x, int T, int H, int D, int kind, uint8_t* codes,
                     uint8_t* bscale, float* rscale) {
  const float E2M1_MAX = 6.0f, E4M3_MAX = 448.0f;
  int64_t n = (int64_t)T * H * D;
  float amax = 0.0f;
  for (int64_t i = 0; i < n; i++) amax = fmaxf(amax, fabsf(orc_bf16_to_f32(x[i])));
  float rs = amax / (E2M1_MAX * E4M3_MAX);
  rscale[0] = rs;
  for (int64_t i = 0; i < n / 2; i++) codes[i] = 0;
  int groups = (kind == ORC_KIND_VALUE) ? T : (T + 15) / 16; /* outer index of a block */
  int per = (kind == ORC_KIND_VALUE) ? D / 16 : D;            /* blocks per (outer, h) */
  for (int g = 0; g < groups; g++)
    for (int h = 0; h < H; h++)
      for (int j = 0; j < per; j++) {
        int len = (kind == ORC_KIND_VALUE) ? 16 : (T - 16 * g < 16 ? T - 16 * g : 16);
        /* block amax and the E4M3 block scale (R2) */
        float vb = 0.0f;
        for (int k = 0; k < len; k++) vb = fmaxf(vb, fabsf(orc_bf16_to_f32(x[nvfp4t_elem(kind, H, D, g, h, j, k)])));
        float t = 0.0f;
        if (rs != 0.0f) t = (vb / E2M1_MAX) / rs;
        if (t > E4M3_MAX) t = E4M3_MAX;
        uint8_t bsb = orc_e4m3_encode(t);
        bscale[((int64_t)g * H + h) * per + j] = bsb;
        float bs = orc_e4m3_value(bsb);
        /* element codes against s = bs * rs (R3) */
        float s = bs * rs;
        float inv = 0.0f;
        if (s != 0.0f) inv = 1.0f / s;
        for (int k = 0; k < len; k++) {
          int64_t e = nvfp4t_elem(kind, H, D, g, h, j, k);
          float xi = orc_bf16_to_f32(x[e]);
          float q;
          if (s == 0.0f)
            q = copysignf(0.0f, xi);
          else if (isinf(inv))
            q = xi / s;
          else
            q = xi * inv;
          uint8_t c = orc_e2m1_encode(q);
          c = (uint8_t)((c & 7) | (signbit(xi) ? 8 : 0));
          codes[e / 2] |= (uint8_t)((e % 2 == 0) ? c : (c << 4)); /* low nibble = even channel */
        }
      }
}

void orc_nvfp4t_unpack(const uint8_t* codes, const uint8_t* bscale, const float* rscale, int T, int H,
                       int D, int kind, uint16_t* y) {
  for (int t = 0; t < T; t++)
    for (int h = 0; h < H; h++)
      for (int d = 0; d < D; d++) {
        int64_t e = ((int64_t)t * H + h) * D + d;
        uint8_t c = (e % 2 == 0) ? (uint8_t)(codes[e / 2] & 15) : (uint8_t)(codes[e / 2] >> 4);
        int64_t b = (kind == ORC_KIND_VALUE) ? ((int64_t)t * H + h) * (D / 16) + d / 16
                                             : ((int64_t)(t / 16) * H + h) * D + d;
        float v = orc_e2m1_value(c) * orc_e4m3_value(bscale[b]); /* exact */
        y[e] = orc_f32_to_bf16(v * rscale[0]);                    /* R4 */
      }
}

/* ------------------------------------------------------------------------- */
/* paged decode attention (NEXT row f1: "feat(kvcache): add nvfp4 kv quantization */
/* (FreeToken PR #408)", Summary and fp8 store notes -- dequantise in registers,  */
/* the row scale applied to the score / output -- and the vllm-rlt review's note  */
/* to dequantise in registers and keep the 16-bit MMA).  The definition is plain  */
/* softmax attention of one query over the decoded rows, in double precision.     */
/* ------------------------------------------------------------------------- */
/* Exact value of element d of a pool row (double holds every product exactly). */
static double pool_value(const uint8_t* codes, const uint8_t* bscale, const float* rscale, int fmt,
                         int64_t r, int D, int d) {
  if (fmt == ORC_FMT_FP8) return (double)orc_e4m3_value(codes[r * D + d]) * (double)rscale[r];
  uint8_t byte = codes[r * (D / 2) + d / 2];
  uint8_t nib = (d % 2 == 0) ? (uint8_t)(byte & 15) : (uint8_t)(byte >> 4);
  return (double)orc_e2m1_value(nib) * (double)orc_e4m3_value(bscale[r * (D / 16) + d / 16]) *
         (double)rscale[r];
}

uint32_t orc_decode_attention(const uint8_t* k_codes, const uint8_t* k_bscale, const float* k_rscale,
                              int fmt_k, const uint8_t* v_codes, const uint8_t* v_bscale,
                              const float* v_rscale, int fmt_v, int64_t num_slots, int H, int D,
                              int block_size, const int32_t* block_table, int S, int max_blocks,
                              const int32_t* seq_lens, const uint16_t* q, int Hq, double scale,
                              double* out) {
  uint32_t status = 0;
  int64_t num_blocks = num_slots / block_size;
  int64_t cap = (int64_t)max_blocks * block_size;
  int group = Hq / H;
  for (int s = 0; s < S; s++) {
    int len = seq_lens[s];
    if (len < 0 || len > cap) {
      status |= ORC_BAD_SEQLEN;
      continue;
    }
    int bad = 0;
    for (int t = 0; t < len && !bad; t++) {
      int32_t block = block_table[(int64_t)s * max_blocks + t / block_size];
      if (block < 0 || block >= num_blocks) bad = 1;
    }
    if (bad) {
      status |= ORC_BAD_BLOCK;
      continue;
    }
    double* sc = (double*)malloc(sizeof(double) * (len > 0 ? len : 1));
    for (int qh = 0; qh < Hq; qh++) {
      int h = qh / group;
      const uint16_t* qv = q + ((int64_t)s * Hq + qh) * D;
      double* o = out + ((int64_t)s * Hq + qh) * D;
      for (int d = 0; d < D; d++) o[d] = 0.0;
      if (len == 0) continue;
      double mx = -INFINITY;
      for (int t = 0; t < len; t++) {
        int64_t slot = (int64_t)block_table[(int64_t)s * max_blocks + t / block_size] * block_size + t % block_size;
        int64_t r = slot * H + h;
        double dot = 0.0;
        for (int d = 0; d < D; d++)
          dot += (double)orc_bf16_to_f32(qv[d]) * pool_value(k_codes, k_bscale, k_rscale, fmt_k, r, D, d);
        sc[t] = scale * dot;
        if (sc[t] > mx) mx = sc[t];
      }
      double l = 0.0;
      for (int t = 0; t < len; t++) {
        sc[t] = exp(sc[t] - mx);
        l += sc[t];
      }
      for (int t = 0; t < len; t++) {
        int64_t slot = (int64_t)block_table[(int64_t)s * max_blocks + t / block_size] * block_size + t % block_size;
        int64_t r = slot * H + h;
        double p = sc[t] / l;
        for (int d = 0; d < D; d++) o[d] += p * pool_value(v_codes, v_bscale, v_rscale, fmt_v, r, D, d);
      }
    }
    free(sc);
  }
  return status;
}

/* ------------------------------------------------------------------------- */
/* INT4 affine codec                                                          */
/* ------------------------------------------------------------------------- */
static void put_nibble(uint8_t* codes, int64_t elem, int code) {
  uint8_t* b = codes + elem / 2;
  if (elem % 2 == 0)
    *b = (uint8_t)((*b & 0xF0) | code);
  else
    *b = (uint8_t)((*b & 0x0F) | (code << 4));
}
static int get_nibble(const uint8_t* codes, int64_t elem) {
  uint8_t b = codes[elem / 2];
  return (elem % 2 == 0) ? (b & 15) : (b >> 4);
}

/* Minimum and maximum in the total order of IEEE 754-2019 minimum/maximum for finite
 * values: -0 is below +0.  (C's fminf may return either zero for a (-0, +0) pair, and
 * which one changes the sign bit of the stored FP16 minimum.) */
static float min_signed0(float a, float b) {
  if (a == 0.0f && b == 0.0f) return signbit(a) ? a : b;
  return b < a ? b : a;
}
static float max_signed0(float a, float b) {
  if (a == 0.0f && b == 0.0f) return signbit(a) ? b : a;
  return b > a ? b : a;
}

/* One group of n elements at x[idx[k]] (R5). */
static void int4_quantize_group(const uint16_t* x, const int64_t* idx, int n, uint8_t* codes,
                                uint16_t* mn16, uint16_t* sc16) {
  float mn = orc_bf16_to_f32(x[idx[0]]), mx = mn;
  for (int k = 1; k < n; k++) {
    float v = orc_bf16_to_f32(x[idx[k]]);
    mn = min_signed0(mn, v);
    mx = max_signed0(mx, v);
  }
  float sc = (mx - mn) / 15.0f;
  for (int k = 0; k < n; k++) {
    int code = 0;
    if (sc != 0.0f) {
      float v = orc_bf16_to_f32(x[idx[k]]);
      float r = rintf((v - mn) / sc); /* codes from the FP32 min and scale */
      if (r < 0.0f) r = 0.0f;
      if (r > 15.0f) r = 15.0f;
      code = (int)r;
    }
    put_nibble(codes, idx[k], code);
  }
  *mn16 = orc_f32_to_f16(mn); /* metadata rounded to FP16 only afterwards */
  *sc16 = orc_f32_to_f16(sc);
}

void orc_int4_pack(const uint16_t* x, int T, int H, int D, int kind, int G, uint8_t* codes,
                   uint16_t* mn16, uint16_t* sc16) {
  int64_t idx[4096];
  if (kind == ORC_KIND_KEY) {
    int ng = (T + G - 1) / G;
    for (int g = 0; g < ng; g++)
      for (int h = 0; h < H; h++)
        for (int d = 0; d < D; d++) {
          int n = 0;
          for (int t = g * G; t < T && t < (g + 1) * G; t++)
            idx[n++] = ((int64_t)t * H + h) * D + d;
          int64_t m = ((int64_t)g * H + h) * D + d;
          int4_quantize_group(x, idx, n, codes, mn16 + m, sc16 + m);
        }
  } else {
    int ng = (D + G - 1) / G;
    for (int t = 0; t < T; t++)
      for (int h = 0; h < H; h++)
        for (int g = 0; g < ng; g++) {
          int n = 0;
          for (int d = g * G; d < D && d < (g + 1) * G; d++)
            idx[n++] = ((int64_t)t * H + h) * D + d;
          int64_t m = ((int64_t)t * H + h) * ng + g;
          int4_quantize_group(x, idx, n, codes, mn16 + m, sc16 + m);
        }
  }
}

void orc_int4_unpack(const uint8_t* codes, const uint16_t* mn16, const uint16_t* sc16, int T,
                     int H, int D, int kind, int G, uint16_t* y) {
  int ngv = (D + G - 1) / G;
  for (int t = 0; t < T; t++)
    for (int h = 0; h < H; h++)
      for (int d = 0; d < D; d++) {
        int64_t e = ((int64_t)t * H + h) * D + d;
        int64_t m = (kind == ORC_KIND_KEY) ? ((int64_t)(t / G) * H + h) * D + d
                                           : ((int64_t)t * H + h) * ngv + d / G;
        float v = (float)get_nibble(codes, e) * orc_f16_to_f32(sc16[m]);
        v = v + orc_f16_to_f32(mn16[m]);
        y[e] = orc_f32_to_bf16(v);
      }
}

/* ------------------------------------------------------------------------- */
/* residual encode / decode (R7)                                              */
/* ------------------------------------------------------------------------- */
static uint32_t check_positions(const int32_t* pos, int P, int T) {
  uint32_t st = 0;
  for (int p = 0; p < P; p++) {
    if (pos[p] < 0 || pos[p] >= T) st |= ORC_BAD_POS;
    if (p > 0 && pos[p] <= pos[p - 1]) st |= ORC_BAD_POS;
  }
  return st;
}

uint32_t orc_residual_encode(const uint16_t* cur, const uint16_t* prev, int T, int H, int D,
                             const int32_t* pos, int P, int fmt, int kind, int G,
                             uint8_t* codes, void* meta_a, void* meta_b, float* rscale,
                             int32_t* pos_out) {
  uint32_t status = 0;
  if (pos == NULL) P = T;
  else status |= check_positions(pos, P, T);
  int64_t row = (int64_t)H * D;
  uint16_t* r = (uint16_t*)calloc((size_t)(P > 0 ? P : 1) * (size_t)row, sizeof(uint16_t));
  for (int p = 0; p < P; p++) {
    int t = pos ? pos[p] : p;
    if (pos_out) pos_out[p] = t;
    if (t < 0 || t >= T) continue; /* left as +0 */
    for (int64_t k = 0; k < row; k++) {
      float c = orc_bf16_to_f32(cur[(int64_t)t * row + k]);
      float q = orc_bf16_to_f32(prev[(int64_t)t * row + k]);
      r[(int64_t)p * row + k] = orc_f32_to_bf16(c - q);
    }
  }
  if (P > 0) {
    if (fmt == ORC_FMT_NVFP4)
      orc_nvfp4_encode_rows(r, (int64_t)P * H, D, codes, (uint8_t*)meta_a, rscale);
    else if (fmt == ORC_FMT_FP8)
      orc_fp8_encode_rows(r, (int64_t)P * H, D, codes, rscale);
    else
      orc_int4_pack(r, P, H, D, kind, G, codes, (uint16_t*)meta_a, (uint16_t*)meta_b);
  }
  free(r);
  return status;
}

uint32_t orc_residual_decode(const uint8_t* codes, const void* meta_a, const void* meta_b,
                             const float* rscale, int fmt, int kind, int G, const int32_t* pos,
                             int P, const uint16_t* prev, int T, int H, int D, uint16_t* out) {
  uint32_t status = 0;
  if (pos == NULL) P = T;
  else status |= check_positions(pos, P, T);
  int64_t row = (int64_t)H * D;
  if (out != prev) memcpy(out, prev, (size_t)T * (size_t)row * sizeof(uint16_t));
  if (P == 0) return status;
  uint16_t* y = (uint16_t*)malloc((size_t)P * (size_t)row * sizeof(uint16_t));
  if (fmt == ORC_FMT_NVFP4)
    orc_nvfp4_decode_rows(codes, (const uint8_t*)meta_a, rscale, (int64_t)P * H, D, y);
  else if (fmt == ORC_FMT_FP8)
    orc_fp8_decode_rows(codes, rscale, (int64_t)P * H, D, y);
  else
    orc_int4_unpack(codes, (const uint16_t*)meta_a, (const uint16_t*)meta_b, P, H, D, kind, G, y);
  for (int p = 0; p < P; p++) {
    int t = pos ? pos[p] : p;
    if (t < 0 || t >= T) continue;
    for (int64_t k = 0; k < row; k++) {
      float a = orc_bf16_to_f32(out[(int64_t)t * row + k]); /* == prev: each row written once */
      float b = orc_bf16_to_f32(y[(int64_t)p * row + k]);
      out[(int64_t)t * row + k] = orc_f32_to_bf16(a + b);
    }
  }
  free(y);
  return status;
}

/* ------------------------------------------------------------------------- */
/* storage accounting                                                         */
/* ------------------------------------------------------------------------- */
int64_t orc_storage_bytes(int fmt, int kind, int G, int64_t T, int H, int D) {
  if (fmt == ORC_FMT_NVFP4) /* codes D/2 + one E4M3 per 16 + one FP32 per row */
    return T * H * (D / 2 + D / 16 + 4);
  if (fmt == ORC_FMT_FP8) /* one E4M3 per value + one FP32 per row */
    return T * H * (D + 4);
  if (fmt == ORC_FMT_NVFP4_TENSOR) { /* codes D/2 + one E4M3 per 16-block + one FP32 per tensor */
    int64_t blocks = (kind == ORC_KIND_KEY) ? ((T + 15) / 16) * H * D : T * H * (D / 16);
    return T * H * (D / 2) + blocks + 4;
  }
  int64_t code_bytes = T * H * (D / 2);
  int64_t groups = (kind == ORC_KIND_KEY) ? ((T + G - 1) / G) * H * D
                                          : T * H * ((D + G - 1) / G);
  return code_bytes + groups * 4; /* FP16 min + FP16 scale per group */
}
