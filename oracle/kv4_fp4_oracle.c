/*
 * kv4_fp4_oracle.c -- plain, slow CPU reference for the FP4 probe formats that
 * KV4-RL compares with affine INT4 (App. D.4, Fig. A4(c)): NVFP4 (E2M1 values,
 * 16-element E4M3 block scales and one FP32 global scale per token-head
 * vector) and MXFP4 (E2M1 values, 32-element E8M0 block scales).  The probe
 * reconstructs the stored cache and attends with BF16 operands.
 *
 * TEST INFRASTRUCTURE ONLY, like kv4_oracle.c: it shares no code with the CUDA
 * library and restates the element formats from their published definitions
 * (OCP Microscaling Formats v1.0 for E2M1 and E8M0; OCP 8-bit floating point
 * for E4M3) and the scale rules below from the pages' description.
 *
 * Reading R13 (the pages name the formats, not the scale arithmetic):
 *   E2M1   sign, 2 exponent bits (bias 1), 1 mantissa bit: magnitudes 0, 0.5,
 *          1, 1.5, 2, 3, 4, 6.  Rounding to nearest, ties to the even code,
 *          magnitudes above 6 saturate to 6; the sign is kept (-0 included).
 *   E4M3   sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities:
 *          largest finite 448, subnormals m/8 * 2^-6.  Ties to even, values
 *          above 448 saturate to 448.
 *   E8M0   the power of two 2^(e - 127), e = 0..254.
 *   NVFP4  vector x[0..n):  a = max|x|;  S = fl(a / 2688) (2688 = 6 * 448,
 *          so that the largest block scale lands on E4M3's largest value);
 *          block b of 16:  s_b = E4M3(fl(amax_b / fl(6 S)));
 *          e_b = fl(E4M3value(s_b) * S);  q_i = E2M1(fl(x_i / e_b)), q = 0
 *          when e_b = 0.  Reconstruction x^_i = E2M1value(q_i) * e_b.
 *   MXFP4  block of 32:  E = floor(log2 amax_b) - 2 (2 = E2M1's largest
 *          exponent), clamped to [-127, 127], E = -127 when amax_b = 0;
 *          q_i = E2M1(x_i * 2^-E);  x^_i = E2M1value(q_i) * 2^E.
 *   A vector with a non-finite element stores all zeros (codes, scales,
 *   global) and sets the non-finite status bit, as the INT4 writer does.
 *   The probe's attention operands are x^ rounded to bf16 (nearest even).
 *
 * fl() is one fp32 operation rounded to nearest even.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#pragma STDC FENV_ACCESS ON

#define FP4O_NVFP4 1
#define FP4O_MXFP4 2
#define FP4O_ST_BAD_PAGE 1
#define FP4O_ST_BAD_POS 2
#define FP4O_ST_BAD_SEQ 4
#define FP4O_ST_NONFINITE 8

/* ------------------------------------------------------------ E2M1 */

static const float kE2M1[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float fp4o_e2m1_value(int code) {
  float v = kE2M1[code & 7];
  return (code & 8) ? -v : v;
}

/* nearest E2M1 code of y (ties to the even code, saturating at 6) */
int fp4o_e2m1_round(float y) {
  int sign = signbit(y) ? 8 : 0;
  float a = fabsf(y);
  if (a >= 6.0f) return sign | 7;
  int k = 0;
  while (k < 7 && kE2M1[k + 1] <= a) ++k;   /* v[k] <= a < v[k+1] */
  float lo = kE2M1[k], hi = kE2M1[k + 1];
  float mid = 0.5f * (lo + hi);             /* exact: two-bit significands */
  int c;
  if (a < mid) c = k;
  else if (a > mid) c = k + 1;
  else c = (k % 2 == 0) ? k : k + 1;
  return sign | c;
}

/* ------------------------------------------------------------ E4M3 */

float fp4o_e4m3_value(int code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return (float)(s ? -v : v);
}

/* nearest finite E4M3 code of t (ties to the even code, saturating at 448),
 * by scanning every finite non-negative code */
int fp4o_e4m3_round(float t) {
  int sign = signbit(t) ? 0x80 : 0;
  double a = fabs((double)t);
  if (a >= 448.0) return sign | 0x7E;
  int best = 0;
  double bd = a;
  for (int c = 1; c <= 0x7E; ++c) {
    double d = fabs((double)fp4o_e4m3_value(c) - a);
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return sign | best;
}

/* ------------------------------------------------------------ encoders */

/* NVFP4-encode one vector of n values (n a multiple of 16).  codes: n bytes
 * (one E2M1 code each); bscale: n/16 E4M3 codes; *global: S. */
int fp4o_nvfp4_encode(const float* x, int n, uint8_t* codes, uint8_t* bscale, float* global) {
  if (n <= 0) return 0;
  int old = fegetround();
  fesetround(FE_TONEAREST);
  float a = 0.0f;
  int nf = 0;
  for (int i = 0; i < n; ++i) {
    if (!isfinite(x[i])) nf = 1;
    else if (fabsf(x[i]) > a) a = fabsf(x[i]);
  }
  memset(codes, 0, (size_t)n);
  memset(bscale, 0, (size_t)n / 16);
  *global = 0.0f;
  if (nf) {
    fesetround(old);
    return FP4O_ST_NONFINITE;
  }
  float S = a / 2688.0f;
  float six_s = 6.0f * S;
  *global = S;
  for (int b = 0; b < n / 16; ++b) {
    float am = 0.0f;
    for (int i = 0; i < 16; ++i)
      if (fabsf(x[16 * b + i]) > am) am = fabsf(x[16 * b + i]);
    int sc = six_s > 0.0f ? fp4o_e4m3_round(am / six_s) : 0;
    bscale[b] = (uint8_t)sc;
    float eb = fp4o_e4m3_value(sc) * S;
    for (int i = 0; i < 16; ++i)
      codes[16 * b + i] = (uint8_t)(eb != 0.0f ? fp4o_e2m1_round(x[16 * b + i] / eb) : 0);
  }
  fesetround(old);
  return 0;
}

/* MXFP4-encode one vector of n values (n a multiple of 32).  codes: n bytes;
 * bscale: n/32 E8M0 codes. */
int fp4o_mxfp4_encode(const float* x, int n, uint8_t* codes, uint8_t* bscale) {
  if (n <= 0) return 0;
  int old = fegetround();
  fesetround(FE_TONEAREST);
  int nf = 0;
  for (int i = 0; i < n; ++i)
    if (!isfinite(x[i])) nf = 1;
  memset(codes, 0, (size_t)n);
  memset(bscale, 0, (size_t)n / 32);
  if (nf) {
    fesetround(old);
    return FP4O_ST_NONFINITE;
  }
  for (int b = 0; b < n / 32; ++b) {
    float am = 0.0f;
    for (int i = 0; i < 32; ++i)
      if (fabsf(x[32 * b + i]) > am) am = fabsf(x[32 * b + i]);
    int E = -127;
    if (am > 0.0f) {
      int e2;
      frexpf(am, &e2); /* am = f 2^e2, f in [0.5, 1): floor(log2 am) = e2 - 1 */
      E = e2 - 1 - 2;
      if (E < -127) E = -127;
      if (E > 127) E = 127;
    }
    bscale[b] = (uint8_t)(E + 127);
    for (int i = 0; i < 32; ++i)
      codes[32 * b + i] = (uint8_t)fp4o_e2m1_round(ldexpf(x[32 * b + i], -E));
  }
  fesetround(old);
  return 0;
}

/* reconstruction of one encoded vector, fp32 */
void fp4o_decode(int fmt, int n, const uint8_t* codes, const uint8_t* bscale, float global,
                 float* out) {
  for (int i = 0; i < n; ++i) {
    float s;
    if (fmt == FP4O_NVFP4) s = fp4o_e4m3_value(bscale[i / 16]) * global;
    else s = ldexpf(1.0f, (int)bscale[i / 32] - 127);
    out[i] = fp4o_e2m1_value(codes[i]) * s;
  }
}

/* ---------------------------------------------- packed probe cache (bytes) */
/*
 * Probe cache layout, restated from the library's description in words:
 *   [num_pages][h_kv][K, V][16 slots][row],  row = d_h/2 + 16 bytes:
 *   bytes [0, d_h/2): E2M1 codes, byte i = channel 2i (low nibble) and
 *   channel 2i+1 (high nibble); then the block scales, one byte each
 *   (NVFP4: d_h/16 E4M3 codes, MXFP4: d_h/32 E8M0 codes); NVFP4 keeps its
 *   global scale S as a little-endian fp32 at byte d_h/2 + 12.  Other bytes
 *   are never written.  Position p of request slot s: page block_table[s][p/16],
 *   slot p % 16.
 */
static long fp4_row_bytes(int d_h) { return d_h / 2 + 16; }

extern void kv4o_hadamard_f32(float* x, int n);
extern float kv4o_bf16_to_f32(uint16_t b);

static void fp4_encode_row(int fmt, const float* x, int d_h, uint8_t* row, int* status) {
  uint8_t codes[256], bs[16];
  float g = 0.0f;
  int st = fmt == FP4O_NVFP4 ? fp4o_nvfp4_encode(x, d_h, codes, bs, &g)
                             : fp4o_mxfp4_encode(x, d_h, codes, bs);
  *status |= st;
  for (int i = 0; i < d_h / 2; ++i) row[i] = (uint8_t)((codes[2 * i] & 15) | ((codes[2 * i + 1] & 15) << 4));
  const int nb = fmt == FP4O_NVFP4 ? d_h / 16 : d_h / 32;
  for (int b = 0; b < nb; ++b) row[d_h / 2 + b] = bs[b];
  if (fmt == FP4O_NVFP4) {
    uint32_t u;
    memcpy(&u, &g, 4);
    for (int k = 0; k < 4; ++k) row[d_h / 2 + 12 + k] = (uint8_t)(u >> (8 * k));
  }
}

/* Append T tokens into the probe cache; rotate_k: K rotated by
 * kv4o_hadamard_f32 first (V never is).  Returns the OR of status bits. */
int fp4o_append(int h_kv, int d_h, int fmt, int rotate_k, int max_seqs, int num_pages,
                int max_pages_per_seq, uint8_t* cache, const uint16_t* k_new,
                const uint16_t* v_new, const int32_t* tok_seq, const int32_t* tok_pos, int T,
                const int32_t* seq_lens, const int32_t* block_table) {
  int status = 0;
  const long rb = fp4_row_bytes(d_h);
  for (int t = 0; t < T; ++t) {
    int s = tok_seq[t], p = tok_pos[t];
    if (s < 0 || s >= max_seqs) {
      status |= FP4O_ST_BAD_SEQ;
      continue;
    }
    if (p < 0 || p >= seq_lens[s] || p >= max_pages_per_seq * 16) {
      status |= FP4O_ST_BAD_POS;
      continue;
    }
    int page = block_table[(long)s * max_pages_per_seq + p / 16];
    if (page < 0 || page >= num_pages) {
      status |= FP4O_ST_BAD_PAGE;
      continue;
    }
    for (int h = 0; h < h_kv; ++h)
      for (int kv = 0; kv < 2; ++kv) {
        const uint16_t* src = (kv == 0 ? k_new : v_new) + ((long)t * h_kv + h) * d_h;
        float x[256];
        for (int i = 0; i < d_h; ++i) x[i] = kv4o_bf16_to_f32(src[i]);
        if (rotate_k && kv == 0) kv4o_hadamard_f32(x, d_h);
        uint8_t* row = cache + ((((long)page * h_kv + h) * 2 + kv) * 16 + p % 16) * rb;
        fp4_encode_row(fmt, x, d_h, row, &status);
      }
  }
  return status;
}

static double bf16_round_d(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* The probe's attention operands for one sequence: every position's K and V
 * encoded, reconstructed and rounded to bf16, as fp64 [h_kv][L][d_h]. */
int fp4o_dequant_seq(int h_kv, int d_h, int fmt, int rotate_k, int L, const uint16_t* k_src,
                     const uint16_t* v_src, double* k_hat, double* v_hat) {
  int status = 0;
  int old = fegetround();
  fesetround(FE_TONEAREST);
  for (int h = 0; h < h_kv; ++h)
    for (int p = 0; p < L; ++p)
      for (int kv = 0; kv < 2; ++kv) {
        const uint16_t* src = (kv == 0 ? k_src : v_src) + ((long)h * L + p) * d_h;
        float x[256], y[256];
        for (int i = 0; i < d_h; ++i) x[i] = kv4o_bf16_to_f32(src[i]);
        if (rotate_k && kv == 0) kv4o_hadamard_f32(x, d_h);
        uint8_t codes[256], bs[16];
        float g = 0.0f;
        status |= fmt == FP4O_NVFP4 ? fp4o_nvfp4_encode(x, d_h, codes, bs, &g)
                                    : fp4o_mxfp4_encode(x, d_h, codes, bs);
        fp4o_decode(fmt, d_h, codes, bs, g, y);
        double* dst = (kv == 0 ? k_hat : v_hat) + ((long)h * L + p) * d_h;
        for (int i = 0; i < d_h; ++i) dst[i] = bf16_round_d(y[i]);
      }
  fesetround(old);
  return status;
}

/* array helpers for the tests */
void fp4o_e2m1_round_n(const float* y, long n, uint8_t* out) {
  for (long i = 0; i < n; ++i) out[i] = (uint8_t)fp4o_e2m1_round(y[i]);
}
void fp4o_e4m3_round_n(const float* t, long n, uint8_t* out) {
  int old = fegetround();
  fesetround(FE_TONEAREST);
  for (long i = 0; i < n; ++i) out[i] = (uint8_t)fp4o_e4m3_round(t[i]);
  fesetround(old);
}
int fp4o_encode_n(int fmt, const float* x, long nvec, int n, uint8_t* codes, uint8_t* bscale,
                  float* global) {
  int st = 0;
  const int nb = fmt == FP4O_NVFP4 ? n / 16 : n / 32;
  for (long v = 0; v < nvec; ++v)
    st |= fmt == FP4O_NVFP4
              ? fp4o_nvfp4_encode(x + v * n, n, codes + v * n, bscale + v * nb, global + v)
              : fp4o_mxfp4_encode(x + v * n, n, codes + v * n, bscale + v * nb);
  return st;
}
void fp4o_decode_n(int fmt, const uint8_t* codes, const uint8_t* bscale, const float* global,
                   long nvec, int n, float* out) {
  int old = fegetround();
  fesetround(FE_TONEAREST);
  const int nb = fmt == FP4O_NVFP4 ? n / 16 : n / 32;
  for (long v = 0; v < nvec; ++v)
    fp4o_decode(fmt, n, codes + v * n, bscale + v * nb, fmt == FP4O_NVFP4 ? global[v] : 0.0f,
                out + v * n);
  fesetround(old);
}
