/*
 * trace_oracle.c - CPU oracle for the guided-NVFP4 hot path of TRACE.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the CUDA library.  Plain C,
 * single-threaded, binary32 arithmetic with round-to-nearest-even, no fused
 * multiply-add (built with -ffp-contract=off) and subnormals kept.
 *
 * What it follows:
 *   [EN] "Alibaba Qwen Proposes TRACE for 5.4x Faster FP4 RL Rollouts":
 *     - "Why Does FP4 Rollout 'Break' RL Training?", the worked example after
 *       Fig. 1: both sides share a global and a block scale, normalise to
 *       2.51 / 2.49 and round-to-nearest takes them to E2M1 values 3 and 2.
 *     - "TRACE Core Concept", first design: rollout records the FP4 results
 *       of routed-expert activations and KV states; the training side still
 *       picks one of the two adjacent E2M1 points, preferring the one closer
 *       to the rollout's actual point instead of plain RTN.
 *     - "TRACE Core Concept", second design (after Fig. 3): the training
 *       value already narrows the candidates, so a little mantissa
 *       information plus the scale tells the training side which way to
 *       round; full records are costly to move GPU->CPU->disk->GPU.
 *   The pages leave the arithmetic open.  The readings taken here (each also
 *   listed in the design notes of the repository) are marked READING below.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include "trace_oracle.h"

#include <math.h>
#include <stddef.h>
#include <string.h>

/* ======================================================================== */
/* Number formats                                                           */
/* ======================================================================== */

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bfloat16 is the upper 16 bits of a binary32, so widening is exact. */
float orc_bf16_to_f32(uint16_t h) { return u2f((uint32_t)h << 16); }

/* binary32 -> bfloat16, round to nearest, ties to an even last kept bit.
 * The 16 dropped bits decide: above half an ulp rounds up, below rounds
 * down, exactly half rounds to make the kept field even.  A carry out of
 * the significand moves into the exponent, which is how the largest finite
 * values round up to infinity.  NaN stays NaN (quiet bit forced). */
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u = f2u(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t kept = u >> 16;
  uint32_t dropped = u & 0xFFFFu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

/* OCP FP8 E4M3 ("E4M3FN"): 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, only S.1111.111 is NaN, so the largest finite
 * magnitude is 2^8 * 1.75 = 448.  Exponent field 0 holds subnormals
 * m * 2^-9.  Encoding: round to nearest with ties to an even significand,
 * saturating (any magnitude >= 448, infinities included, becomes 448). */
uint8_t orc_e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  /* binade [2^e, 2^(e+1)); everything below 2^-6 uses the subnormal step */
  int e = -6;
  while (e < 8 && a >= ldexp(1.0, e + 1)) e++;
  double ulp = ldexp(1.0, e - 3);
  double q = a / ulp; /* exact: a power-of-two scaling */
  double n = floor(q);
  double rem = q - n;
  if (rem > 0.5 || (rem == 0.5 && fmod(n, 2.0) == 1.0)) n += 1.0;
  int code;
  if (a < ldexp(1.0, -6)) {
    code = (int)n; /* 0..8; 8 is the smallest normal, 1.000 x 2^-6 */
  } else {
    code = ((e + 7) << 3) + ((int)n - 8); /* n == 16 carries into the exponent */
  }
  if (code > 0x7E) code = 0x7E;
  return (uint8_t)(sign | code);
}

float orc_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9);
  else
    mag = ldexp(8.0 + m, e - 10);
  return (float)(s ? -mag : mag);
}

/* OCP FP4 E2M1: index m = (exponent field << 1) | mantissa bit, bias 1.
 * Exponent field 0 is subnormal: 0.5 * mantissa.  Otherwise
 * 2^(e-1) * (1 + mantissa/2).  This gives 0, .5, 1, 1.5, 2, 3, 4, 6. */
float orc_e2m1_value(int m) {
  int e = (m >> 1) & 3, mb = m & 1;
  if (e == 0) return 0.5f * (float)mb;
  return (float)ldexp(1.0 + 0.5 * mb, e - 1);
}

/* Step "bracket": lo = the largest index whose magnitude does not exceed t,
 * hi = the smallest index whose magnitude is not below t.  On a code point
 * lo == hi.  Above the largest point (t > 6, infinity included) both are 7,
 * the saturation reading. */
void orc_e2m1_bracket(float t, int* lo, int* hi) {
  int l = 0, h = 7;
  if (!(t > 6.0f)) {
    for (int m = 0; m < 8; ++m)
      if (orc_e2m1_value(m) <= t) l = m;
    for (int m = 7; m >= 0; --m)
      if (orc_e2m1_value(m) >= t) h = m;
  } else {
    l = 7;
  }
  if (isnan(t)) { l = 0; h = 0; }
  *lo = l;
  *hi = h;
}

/* Round-to-nearest onto the E2M1 grid ([EN] names RTN as the default the
 * guided rule replaces).  READING: ties go to the even index (the OCP /
 * IEEE convention), values above 6 saturate to index 7. */
int orc_e2m1_rtn(float t) {
  int lo, hi;
  orc_e2m1_bracket(t, &lo, &hi);
  if (lo == hi) return lo;
  double dl = (double)t - orc_e2m1_value(lo); /* exact in binary64 */
  double dh = (double)orc_e2m1_value(hi) - (double)t;
  if (dl < dh) return lo;
  if (dh < dl) return hi;
  return (lo & 1) ? hi : lo;
}

/* ======================================================================== */
/* Scalar pieces of the method                                              */
/* ======================================================================== */

/* Per-segment FP32 global scale: the NVFP4 convention maps the segment amax
 * to E2M1's largest magnitude (6) times E4M3's largest (448), so
 * gs = amax / 2688 in binary32.  READING: a zero amax (or a quotient that
 * underflows to zero) gives gs = 0, and every block of the segment then
 * gets a zero scale. */
float orc_global_scale(float amax) {
  if (!(amax > 0.0f)) return 0.0f;
  float gs = amax / 2688.0f;
  return gs > 0.0f ? gs : 0.0f;
}

/* Per-block E4M3 scale: the block's largest magnitude over 6 * gs (the
 * product is formed first, then one division), then E4M3 encoding. */
uint8_t orc_block_scale(float bamax, float gs) {
  if (!(gs > 0.0f)) return 0;
  float denom = gs * 6.0f;
  float q = bamax / denom;
  return orc_e4m3_encode(q);
}

/* The block's real scale S = decode(bs) * gs and its reciprocal.
 * READING: elements are scaled by the reciprocal of S (one IEEE division
 * per block) rather than divided by S one by one.  A block whose S is zero,
 * or so small that 1/S overflows binary32, is flushed: inv = 0, so every
 * element normalises to 0. */
void orc_scale_pair(uint8_t bs, float gs, float* S, float* inv) {
  float s = orc_e4m3_decode(bs) * gs;
  float r = 0.0f;
  if (s > 0.0f) {
    r = 1.0f / s;
    if (isinf(r)) r = 0.0f;
  }
  *S = s;
  *inv = r;
}

/* Compact record decoding ([EN] "TRACE Core Concept", after Fig. 3: the
 * training value narrows the candidates, the stored mantissa bit picks the
 * direction).  READING: the reference value is bracketed in the rollout's
 * own scale frame; of the two adjacent candidates exactly one has the stored
 * low bit, and that one is the decoded index.  A single-point bracket needs
 * no bit. */
int orc_unpack_index(float t_ref, int lsb) {
  int lo, hi;
  orc_e2m1_bracket(t_ref, &lo, &hi);
  if (lo == hi) return lo;
  return ((lo & 1) == (lsb & 1)) ? lo : hi;
}

/* Rollout-guided rounding of one training element ([EN] "TRACE Core
 * Concept", first design).  t = |x| * inv_t; the two adjacent E2M1
 * candidates lo/hi of t are dequantised with the training side's own scale
 * S_t, the rollout code with the rollout's scale S_r, and the candidate whose
 * dequantised value is closer to the rollout's reconstructed value wins.
 * READING: distances are |v_c - v_r| in binary32; equal distances, a
 * single-point bracket or a missing guide fall back to RTN. */
int orc_guided_index(float x, float S_t, float inv_t, int have_guide,
                     int nib_r, float S_r) {
  float t = fabsf(x) * inv_t;
  int lo, hi;
  orc_e2m1_bracket(t, &lo, &hi);
  int m_rtn = orc_e2m1_rtn(t);
  if (!have_guide || lo == hi) return m_rtn;
  int s_t = signbit(x) ? 1 : 0;
  int s_r = (nib_r >> 3) & 1;
  int m_r = nib_r & 7;
  float v_r = orc_e2m1_value(m_r) * S_r;
  if (s_r) v_r = -v_r;
  float v_lo = orc_e2m1_value(lo) * S_t;
  float v_hi = orc_e2m1_value(hi) * S_t;
  if (s_t) { v_lo = -v_lo; v_hi = -v_hi; }
  float d_lo = fabsf(v_lo - v_r);
  float d_hi = fabsf(v_hi - v_r);
  if (d_lo < d_hi) return lo;
  if (d_hi < d_lo) return hi;
  return m_rtn;
}

void orc_e2m1_rtn_array(const float* t, int64_t n, uint8_t* m_out) {
  for (int64_t i = 0; i < n; ++i) m_out[i] = (uint8_t)orc_e2m1_rtn(t[i]);
}

void orc_e2m1_bracket_array(const float* t, int64_t n, uint8_t* lo,
                            uint8_t* hi) {
  for (int64_t i = 0; i < n; ++i) {
    int l, h;
    orc_e2m1_bracket(t[i], &l, &h);
    lo[i] = (uint8_t)l;
    hi[i] = (uint8_t)h;
  }
}

void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

void orc_f32_to_bf16_array(const float* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(v[i]);
}

/* ======================================================================== */
/* Whole-tensor steps                                                       */
/* ======================================================================== */

/* Validates a segment table; NULL stands for one segment over all rows. */
static int check_segments(const int64_t* seg, int32_t n_seg, int64_t rows) {
  if (seg == NULL) return n_seg == 1 || n_seg == 0 ? 0 : -1;
  if (n_seg < 1) return -1;
  if (seg[0] != 0 || seg[n_seg] != rows) return -1;
  for (int32_t s = 0; s < n_seg; ++s)
    if (seg[s + 1] < seg[s]) return -1;
  return 0;
}

static int check_shape(int64_t rows, int64_t cols) {
  if (rows < 0 || cols <= 0 || cols % 32 != 0) return -1;
  return 0;
}

static int64_t seg_begin(const int64_t* seg, int32_t s) { return seg ? seg[s] : 0; }
static int64_t seg_end(const int64_t* seg, int32_t s, int64_t rows) {
  return seg ? seg[s + 1] : rows;
}
static int32_t seg_count(const int64_t* seg, int32_t n_seg) { return seg ? n_seg : 1; }

/* Which segment holds a row (linear search: the oracle favours plainness). */
static int32_t seg_of_row(const int64_t* seg, int32_t n_seg, int64_t row) {
  if (!seg) return 0;
  int32_t s = 0;
  while (s + 1 < n_seg && seg[s + 1] <= row) ++s;
  return s;
}

/* Largest magnitude over each segment's rows; an empty segment gives 0. */
int orc_segment_amax(const uint16_t* x, int64_t rows, int64_t cols,
                     const int64_t* seg, int32_t n_seg, float* amax) {
  if (check_shape(rows, cols) || check_segments(seg, n_seg, rows)) return -1;
  int32_t ns = seg_count(seg, n_seg);
  for (int32_t s = 0; s < ns; ++s) {
    float m = 0.0f;
    for (int64_t r = seg_begin(seg, s); r < seg_end(seg, s, rows); ++r)
      for (int64_t c = 0; c < cols; ++c) {
        float a = fabsf(orc_bf16_to_f32(x[r * cols + c]));
        if (a > m) m = a;
      }
    amax[s] = m;
  }
  return 0;
}

static float block_amax(const uint16_t* xb) {
  float m = 0.0f;
  for (int j = 0; j < 16; ++j) {
    float a = fabsf(orc_bf16_to_f32(xb[j]));
    if (a > m) m = a;
  }
  return m;
}

/* Rollout side: NVFP4 quantisation with the compact record.  Per segment the
 * global scale, per block the E4M3 scale, per element the RTN code; the
 * compact word stores each element's sign and the low bit of its index
 * ([EN] "TRACE Core Concept", after Fig. 3: "a small amount of mantissa
 * information, along with the scale" -- in E2M1 the index's low bit is the
 * single mantissa bit). */
int orc_rollout_quant(const uint16_t* x, int64_t rows, int64_t cols,
                      const int64_t* seg, int32_t n_seg, uint8_t* codes,
                      uint8_t* bs, float* gs, uint32_t* guide) {
  return orc_rollout_quant_given(x, rows, cols, seg, n_seg, NULL, codes, bs, gs, guide);
}

int orc_rollout_quant_given(const uint16_t* x, int64_t rows, int64_t cols,
                            const int64_t* seg, int32_t n_seg, const float* amax_in,
                            uint8_t* codes, uint8_t* bs, float* gs, uint32_t* guide) {
  if (check_shape(rows, cols) || check_segments(seg, n_seg, rows)) return -1;
  int32_t ns = seg_count(seg, n_seg);
  int64_t nb = cols / 16;
  for (int32_t s = 0; s < ns; ++s) {
    int64_t r0 = seg_begin(seg, s), r1 = seg_end(seg, s, rows);
    float amax;
    int64_t one[2] = {0, r1 - r0};
    if (amax_in)
      amax = amax_in[s];
    else
      orc_segment_amax(x + r0 * cols, r1 - r0, cols, one, 1, &amax);
    float g = orc_global_scale(amax);
    gs[s] = g;
    for (int64_t r = r0; r < r1; ++r) {
      for (int64_t b = 0; b < nb; ++b) {
        const uint16_t* xb = x + r * cols + b * 16;
        uint8_t code_s = orc_block_scale(block_amax(xb), g);
        float S, inv;
        orc_scale_pair(code_s, g, &S, &inv);
        bs[r * nb + b] = code_s;
        uint32_t word = 0;
        for (int j = 0; j < 16; ++j) {
          float v = orc_bf16_to_f32(xb[j]);
          float t = fabsf(v) * inv;
          int m = orc_e2m1_rtn(t);
          int sgn = signbit(v) ? 1 : 0;
          uint8_t nib = (uint8_t)((sgn << 3) | m);
          int64_t e = r * cols + b * 16 + j;
          uint8_t* byte = codes + e / 2;
          if ((e & 1) == 0)
            *byte = (uint8_t)((*byte & 0xF0) | nib);
          else
            *byte = (uint8_t)((*byte & 0x0F) | (nib << 4));
          word |= (uint32_t)sgn << j;
          word |= (uint32_t)(m & 1) << (16 + j);
        }
        if (guide) guide[r * nb + b] = word;
      }
    }
  }
  return 0;
}

static int nibble_at(const uint8_t* codes, int64_t e) {
  uint8_t byte = codes[e / 2];
  return (e & 1) ? (byte >> 4) : (byte & 0x0F);
}

/* Full codes -> compact words: keep bit 3 (sign) and bit 0 (mantissa bit). */
int orc_guide_pack(const uint8_t* codes, int64_t rows, int64_t cols,
                   uint32_t* guide) {
  if (check_shape(rows, cols)) return -1;
  int64_t nb = cols / 16;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      uint32_t word = 0;
      for (int j = 0; j < 16; ++j) {
        int nib = nibble_at(codes, r * cols + b * 16 + j);
        word |= (uint32_t)((nib >> 3) & 1) << j;
        word |= (uint32_t)(nib & 1) << (16 + j);
      }
      guide[r * nb + b] = word;
    }
  return 0;
}

/* Compact words + reference values -> full rollout codes (see
 * orc_unpack_index).  The rollout scales come from the rollout's own block
 * scale codes and per-segment global scales. */
int orc_guide_unpack(const uint16_t* x_ref, const uint32_t* guide,
                     const uint8_t* bs_r, const float* gs_r,
                     const int64_t* seg_r, int32_t n_seg_r, int64_t rows,
                     int64_t cols, uint8_t* codes) {
  if (check_shape(rows, cols) || check_segments(seg_r, n_seg_r, rows)) return -1;
  int64_t nb = cols / 16;
  for (int64_t r = 0; r < rows; ++r) {
    float g = gs_r[seg_of_row(seg_r, n_seg_r, r)];
    for (int64_t b = 0; b < nb; ++b) {
      float S, inv;
      orc_scale_pair(bs_r[r * nb + b], g, &S, &inv);
      uint32_t word = guide[r * nb + b];
      for (int j = 0; j < 16; ++j) {
        int64_t e = r * cols + b * 16 + j;
        float t = fabsf(orc_bf16_to_f32(x_ref[e])) * inv;
        int m = orc_unpack_index(t, (int)((word >> (16 + j)) & 1));
        int sgn = (int)((word >> j) & 1);
        uint8_t nib = (uint8_t)((sgn << 3) | m);
        uint8_t* byte = codes + e / 2;
        if ((e & 1) == 0)
          *byte = (uint8_t)((*byte & 0xF0) | nib);
        else
          *byte = (uint8_t)((*byte & 0x0F) | (nib << 4));
      }
    }
  }
  return 0;
}

static int signed_index(int sgn, int m) { return sgn ? -m : m; }

static int dist_bucket(int a, int b) {
  int d = a > b ? a - b : b - a;
  return d >= 3 ? 3 : d;
}

/* Training side: guided fake quantisation with the training tensor's own
 * scales.  Writes the bf16 dequantised values, the straight-through mask and
 * optionally the chosen codes and mismatch statistics.
 *
 * READING (mask): the pages are silent on the backward pass; "QAT" implies a
 * straight-through estimator.  An element is cut from the gradient (bit 0)
 * exactly when its block scale is positive and |x| > 6 * S, i.e. it was
 * clipped by the saturating top code; every other element passes (bit 1).
 *
 * READING (statistics): signed index k = sign ? -m : m (so +0 and -0 agree);
 * an element mismatches when its k differs from the rollout's; histogram
 * buckets count |dk| = 0, 1, 2, >= 3, before (RTN) and after guidance. */
int orc_train_fakequant(const uint16_t* x, int64_t rows, int64_t cols,
                        const int64_t* seg_t, int32_t n_seg_t, int kind,
                        const void* guide, const uint8_t* bs_r,
                        const float* gs_r, const int64_t* seg_r,
                        int32_t n_seg_r, uint16_t* y, uint32_t* mask,
                        uint8_t* codes_t, uint64_t* stats) {
  return orc_train_fakequant_given(x, rows, cols, seg_t, n_seg_t, NULL, kind, guide, bs_r,
                                   gs_r, seg_r, n_seg_r, y, mask, codes_t, stats);
}

int orc_train_fakequant_given(const uint16_t* x, int64_t rows, int64_t cols,
                              const int64_t* seg_t, int32_t n_seg_t,
                              const float* amax_t_in, int kind, const void* guide,
                              const uint8_t* bs_r, const float* gs_r,
                              const int64_t* seg_r, int32_t n_seg_r, uint16_t* y,
                              uint32_t* mask, uint8_t* codes_t, uint64_t* stats) {
  if (check_shape(rows, cols) || check_segments(seg_t, n_seg_t, rows)) return -1;
  if (kind != ORC_GUIDE_NONE) {
    if (!guide || !bs_r || !gs_r) return -1;
    if (check_segments(seg_r, n_seg_r, rows)) return -1;
  }
  int64_t nb = cols / 16;
  int32_t ns = seg_count(seg_t, n_seg_t);
  for (int32_t s = 0; s < ns; ++s) {
    int64_t r0 = seg_begin(seg_t, s), r1 = seg_end(seg_t, s, rows);
    float amax;
    int64_t one[2] = {0, r1 - r0};
    if (amax_t_in)
      amax = amax_t_in[s];
    else
      orc_segment_amax(x + r0 * cols, r1 - r0, cols, one, 1, &amax);
    float g_t = orc_global_scale(amax);
    for (int64_t r = r0; r < r1; ++r) {
      float g_r = 0.0f;
      if (kind != ORC_GUIDE_NONE) g_r = gs_r[seg_of_row(seg_r, n_seg_r, r)];
      for (int64_t b = 0; b < nb; ++b) {
        const uint16_t* xb = x + r * cols + b * 16;
        uint8_t code_s = orc_block_scale(block_amax(xb), g_t);
        float S_t, inv_t;
        orc_scale_pair(code_s, g_t, &S_t, &inv_t);
        float S_r = 0.0f, inv_r = 0.0f;
        uint32_t word = 0;
        if (kind != ORC_GUIDE_NONE) orc_scale_pair(bs_r[r * nb + b], g_r, &S_r, &inv_r);
        if (kind == ORC_GUIDE_COMPACT) word = ((const uint32_t*)guide)[r * nb + b];
        for (int j = 0; j < 16; ++j) {
          int64_t e = r * cols + b * 16 + j;
          float v = orc_bf16_to_f32(xb[j]);
          int s_t = signbit(v) ? 1 : 0;
          int nib_r = 0;
          if (kind == ORC_GUIDE_FULL) {
            nib_r = nibble_at((const uint8_t*)guide, e);
          } else if (kind == ORC_GUIDE_COMPACT) {
            float t_ref = fabsf(v) * inv_r;
            int m_r = orc_unpack_index(t_ref, (int)((word >> (16 + j)) & 1));
            nib_r = (int)(((word >> j) & 1) << 3) | m_r;
          }
          int m = orc_guided_index(v, S_t, inv_t, kind != ORC_GUIDE_NONE, nib_r, S_r);
          float out = orc_e2m1_value(m) * S_t;
          if (s_t) out = -out;
          y[e] = orc_f32_to_bf16(out);
          if (mask) {
            int clipped = (S_t > 0.0f) && (fabsf(v) > 6.0f * S_t);
            uint32_t* w = mask + e / 32;
            if (e % 32 == 0) *w = 0;
            if (!clipped) *w |= 1u << (e % 32);
          }
          if (codes_t) {
            uint8_t nib = (uint8_t)((s_t << 3) | m);
            uint8_t* byte = codes_t + e / 2;
            if ((e & 1) == 0)
              *byte = (uint8_t)((*byte & 0xF0) | nib);
            else
              *byte = (uint8_t)((*byte & 0x0F) | (nib << 4));
          }
          if (stats) {
            stats[ORC_STAT_N] += 1;
            if (kind != ORC_GUIDE_NONE) {
              int k_r = signed_index((nib_r >> 3) & 1, nib_r & 7);
              int m_rtn = orc_e2m1_rtn(fabsf(v) * inv_t);
              int k_rtn = signed_index(s_t, m_rtn);
              int k_g = signed_index(s_t, m);
              if (k_rtn != k_r) stats[ORC_STAT_MISMATCH_RTN] += 1;
              if (k_g != k_r) stats[ORC_STAT_MISMATCH_GUIDED] += 1;
              stats[ORC_STAT_HIST_RTN + dist_bucket(k_rtn, k_r)] += 1;
              stats[ORC_STAT_HIST_GUIDED + dist_bucket(k_g, k_r)] += 1;
            }
          }
        }
      }
    }
  }
  return 0;
}

/* Straight-through estimator ("QAT" in the article's title implies a
 * fake quantiser trained through; READING: the gradient passes unchanged for
 * kept elements and is cut to +0 for elements clipped by the top code). */
int orc_ste_backward(const uint16_t* g, const uint32_t* mask, int64_t rows, int64_t cols,
                     uint16_t* out) {
  if (check_shape(rows, cols)) return -1;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      int64_t e = r * cols + c;
      int kept = (int)((mask[e / 32] >> (e % 32)) & 1u);
      out[e] = kept ? g[e] : (uint16_t)0;
    }
  return 0;
}

/* ---- block scales for tensor cores, and the NVFP4 GEMM that uses them ---- */

static int64_t ceil_to(int64_t v, int64_t q) { return (v + q - 1) / q * q; }

int64_t orc_mma_scales_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols <= 0 || cols % 16) return -1;
  return ceil_to(rows, 128) * ceil_to(cols / 16, 4);
}

/* Layout per NVIDIA's cuBLAS documentation, "1D block scaling factors
 * layout": 512-byte tiles of 128 rows x 4 scale columns, tiles running along
 * the scale columns, (r, c) inside a tile at 16 (r mod 32) + 4 (r div 32) + c. */
int orc_mma_scales(const uint8_t* bs, int64_t rows, int64_t cols, uint8_t* out) {
  int64_t bytes = orc_mma_scales_bytes(rows, cols);
  if (bytes < 0) return -1;
  int64_t sc = cols / 16;                  /* scale columns               */
  int64_t tiles_per_row = ceil_to(sc, 4) / 4;
  for (int64_t i = 0; i < bytes; ++i) out[i] = 0;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < sc; ++c) {
      int64_t tile = (r / 128) * tiles_per_row + c / 4;
      int64_t rr = r % 128, cc = c % 4;
      out[tile * 512 + 16 * (rr % 32) + 4 * (rr / 32) + cc] = bs[r * sc + c];
    }
  return 0;
}

static double nvfp4_value(const uint8_t* codes, const uint8_t* bs, int64_t cols, int64_t r,
                          int64_t c) {
  int64_t e = r * cols + c;
  uint8_t byte = codes[e / 2];
  int nib = (e % 2) ? (byte >> 4) : (byte & 15);
  double v = (double)orc_e2m1_value(nib & 7) * (double)orc_e4m3_decode(bs[r * (cols / 16) + c / 16]);
  return (nib & 8) ? -v : v;
}

int orc_nvfp4_gemm(const uint8_t* a_codes, const uint8_t* a_bs, float a_gs,
                   const uint8_t* b_codes, const uint8_t* b_bs, float b_gs,
                   int64_t m, int64_t n, int64_t k, double* d) {
  if (m < 0 || n < 0 || k <= 0 || k % 32) return -1;
  float alpha = a_gs * b_gs;               /* binary32, as the GEMM's scale */
  for (int64_t i = 0; i < m; ++i)
    for (int64_t j = 0; j < n; ++j) {
      double acc = 0.0;
      for (int64_t q = 0; q < k; ++q)
        acc += nvfp4_value(a_codes, a_bs, k, i, q) * nvfp4_value(b_codes, b_bs, k, j, q);
      d[i * n + j] = (double)alpha * acc;
    }
  return 0;
}
