/*
 * kv4_oracle.c -- plain, slow, CPU reference for the KV4-RL mixed INT4/INT8
 * KV cache: quantize-on-append and decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library; the packed byte layout it
 * writes is restated here from the layout description in words.
 *
 * Sources (paper: "KV4-RL: Unlocking Faster Asynchronous Rollouts for RLVR with
 * INT4 KV Cache Quantization"):
 *   - affine b-bit quantizer x^ = Delta*c + m, c in {0..2^b-1}   (Sec. 3, eq. 3.3)
 *   - affine INT4 codes with FP16 scale and offset per group      (Sec. 5.1; App. A.3)
 *   - INT8 side entries: symmetric per token/head scale, computed
 *     from the source vector, not from the INT4 reconstruction    (App. A.3)
 *   - protected set = first s positions + most recent w positions (Sec. 5.2)
 *   - protected and INT4 regions are disjoint                     (Sec. 5.3)
 *   - regional softmax merge z = log(e^z4 + e^z8), o = sum e^(zr-z) o_r
 *                                                                 (App. A.3, eq. A1)
 *   - INT8 scale = max|x| / 127 per token-head (course page "KV cache
 *     quantization", INT8 per-token-head write path)
 *
 * Readings where the pages leave a step open:
 *   R1 group size g is a parameter (the paper deploys 128; its ablation uses 32).
 *   R2 Delta and m come from the group min/max (asymmetric).  m is the FP16 value
 *      rounded DOWN from the min; Delta is the FP16 value rounded UP from
 *      (max -up m) /up 15, both fp32 operations rounded upward.  This makes
 *      m <= x <= m + 15*Delta hold exactly, so codes never clamp.
 *   R3 codes c = round-half-to-even((x -rn m) /rn Delta), clamped to [0,15];
 *      Delta == 0 (constant group) gives c = 0.
 *   R4 INT8: a = max|x|, s = fp16_up(a /up 127), c = rne(x /rn s) clamped to
 *      [-127,127]; s == 0 gives c = 0.
 *   R5 protected set of a sequence of length L: [0, min(S,L)) U [max(S,L-R), L).
 *      Sink slot of position p < S is p; ring slot of p >= S is S + (p mod R).
 *   R6 in a multi-token append a position is written to the ring only if it lies
 *      in the window of its sequence's length after the append (seq_lens).
 *   R7 attention is fp64 softmax over the dequantized cache, bf16 query used as
 *      is, softmax scale passed in (1/sqrt(d_h) by convention), query head j
 *      reads kv head j / (h_q / h_kv).
 *   R8 a non-finite input element, or metadata that overflows FP16, marks the
 *      status word and stores an all-zero group (codes 0, Delta 0, m 0).
 *   R9 Hadamard K-rotation (Sec. 3 eq. 3.4; App. A.3 "Encoding and
 *      allocation"; App. D.4 keeps K-only): the fixed normalized Sylvester
 *      matrix of order d_h (no random signs), applied to the bf16 K vector of
 *      every token-head before both encoders (INT4 and INT8), V unrotated; the
 *      query is rotated by the same matrix and rounded to bf16.  The pages fix
 *      no precision: fp32, in the order kv4o_hadamard_f32 states, so that the
 *      quantization decisions are reproducible bit for bit.
 *
 * Every function pins against closed forms / invariants / brute force in
 * tests/test_oracle_*.py.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#pragma STDC FENV_ACCESS ON

#define KV4O_RNE 0
#define KV4O_DOWN 1
#define KV4O_UP 2

#define KV4O_ST_BAD_PAGE 1
#define KV4O_ST_BAD_POS 2
#define KV4O_ST_BAD_SEQ 4
#define KV4O_ST_NONFINITE 8

/* ---------------------------------------------------------------- scalars */

float kv4o_bf16_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* IEEE binary16 -> binary32, from the format definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float kv4o_f16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 0x1F;
  int fr = h & 0x3FF;
  double v;
  if (ex == 0x1F) {
    v = fr ? NAN : INFINITY;
  } else if (ex == 0) {
    v = ldexp((double)fr, -24); /* subnormal: fr * 2^-24 */
  } else {
    v = ldexp((double)(1024 + fr), ex - 25); /* (1 + fr/1024) * 2^(ex-15) */
  }
  return (float)(sign ? -v : v);
}

/* binary32 -> binary16 with a chosen rounding direction.  The magnitude is
 * written as an integer multiple of the binary16 quantum of its binade and that
 * integer is rounded; overflow follows IEEE 754 (round-to-nearest and
 * round-away-from-zero give infinity, round-toward-zero gives 65504). */
uint16_t kv4o_f32_to_f16(float xf, int mode) {
  uint32_t bits;
  memcpy(&bits, &xf, 4);
  uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
  if (isnan(xf)) return 0x7E00;
  if (isinf(xf)) return (uint16_t)(sign | 0x7C00);
  double x = fabs((double)xf);
  if (x == 0.0) return sign;
  /* magnitude rounding: 0 nearest-even, 1 toward zero, 2 away from zero */
  int mag;
  if (mode == KV4O_RNE)
    mag = 0;
  else if (mode == KV4O_DOWN)
    mag = sign ? 2 : 1;
  else
    mag = sign ? 1 : 2;
  int e2;
  frexp(x, &e2);   /* x in [2^(e2-1), 2^e2) */
  int E = e2 - 1;  /* unbiased exponent of x */
  if (E < -14) E = -14; /* subnormal binade shares the quantum 2^-24 */
  double quantum = ldexp(1.0, E - 10);
  double n = x / quantum; /* exact: power-of-two division of a binary32 */
  double r;
  if (mag == 0) {
    r = floor(n);
    double frac = n - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  } else if (mag == 1) {
    r = floor(n);
  } else {
    r = ceil(n);
  }
  double y = r * quantum;
  if (y > 65504.0) {
    if (mag == 1) return (uint16_t)(sign | 0x7BFF);
    return (uint16_t)(sign | 0x7C00);
  }
  if (y == 0.0) return sign;
  uint16_t out;
  if (y < ldexp(1.0, -14)) {
    out = (uint16_t)(y / ldexp(1.0, -24)); /* subnormal fraction field */
  } else {
    int ey;
    frexp(y, &ey);
    int Ey = ey - 1;
    int frac = (int)(y / ldexp(1.0, Ey - 10)) - 1024;
    out = (uint16_t)(((Ey + 15) << 10) | frac);
  }
  return (uint16_t)(sign | out);
}

/* fp32 subtraction / division under an explicit IEEE rounding direction. */
float kv4o_sub_dir(float a, float b, int mode) {
  int old = fegetround();
  fesetround(mode == KV4O_UP ? FE_UPWARD : (mode == KV4O_DOWN ? FE_DOWNWARD : FE_TONEAREST));
  volatile float va = a, vb = b;
  volatile float r = va - vb;
  fesetround(old);
  return r;
}

float kv4o_div_dir(float a, float b, int mode) {
  int old = fegetround();
  fesetround(mode == KV4O_UP ? FE_UPWARD : (mode == KV4O_DOWN ? FE_DOWNWARD : FE_TONEAREST));
  volatile float va = a, vb = b;
  volatile float r = va / vb;
  fesetround(old);
  return r;
}

/* round half to even, binary32 -> integer (value as double for range) */
static double rne_int(float v) {
  double d = (double)v;
  double r = floor(d);
  double frac = d - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  return r;
}

/* ------------------------------------------------------------ encoders */

/* INT4 affine encode of one group of g values (readings R2, R3, R8).
 * Returns 0, or KV4O_ST_NONFINITE (and an all-zero group). */
int kv4o_int4_encode_group(const float* x, int g, uint8_t* codes, uint16_t* delta16,
                           uint16_t* off16) {
  float mn = x[0], mx = x[0];
  int bad = 0;
  for (int i = 0; i < g; ++i) {
    if (!isfinite(x[i])) bad = 1;
    if (x[i] < mn) mn = x[i];
    if (x[i] > mx) mx = x[i];
  }
  uint16_t m16 = 0, d16 = 0;
  float mf = 0.f, df = 0.f;
  if (!bad) {
    m16 = kv4o_f32_to_f16(mn, KV4O_DOWN);
    mf = kv4o_f16_to_f32(m16);
    float span = kv4o_sub_dir(mx, mf, KV4O_UP);
    float step = kv4o_div_dir(span, 15.0f, KV4O_UP);
    d16 = kv4o_f32_to_f16(step, KV4O_UP);
    df = kv4o_f16_to_f32(d16);
    if (!isfinite(mf) || !isfinite(df)) bad = 1;
  }
  if (bad) {
    for (int i = 0; i < g; ++i) codes[i] = 0;
    *delta16 = 0;
    *off16 = 0;
    return KV4O_ST_NONFINITE;
  }
  for (int i = 0; i < g; ++i) {
    int c = 0;
    if (df != 0.0f) {
      float t = kv4o_div_dir(kv4o_sub_dir(x[i], mf, KV4O_RNE), df, KV4O_RNE);
      double r = rne_int(t);
      if (r < 0) r = 0;
      if (r > 15) r = 15;
      c = (int)r;
    }
    codes[i] = (uint8_t)c;
  }
  *delta16 = d16;
  *off16 = m16;
  return 0;
}

/* INT8 symmetric encode of one token-head vector of n values (reading R4, R8). */
int kv4o_int8_encode_vec(const float* x, int n, int8_t* codes, uint16_t* scale16) {
  float a = 0.f;
  int bad = 0;
  for (int i = 0; i < n; ++i) {
    if (!isfinite(x[i])) bad = 1;
    float ax = fabsf(x[i]);
    if (ax > a) a = ax;
  }
  uint16_t s16 = 0;
  float sf = 0.f;
  if (!bad) {
    s16 = kv4o_f32_to_f16(kv4o_div_dir(a, 127.0f, KV4O_UP), KV4O_UP);
    sf = kv4o_f16_to_f32(s16);
    if (!isfinite(sf)) bad = 1;
  }
  if (bad) {
    for (int i = 0; i < n; ++i) codes[i] = 0;
    *scale16 = 0;
    return KV4O_ST_NONFINITE;
  }
  for (int i = 0; i < n; ++i) {
    int c = 0;
    if (sf != 0.0f) {
      double r = rne_int(kv4o_div_dir(x[i], sf, KV4O_RNE));
      if (r < -127) r = -127;
      if (r > 127) r = 127;
      c = (int)r;
    }
    codes[i] = (int8_t)c;
  }
  *scale16 = s16;
  return 0;
}

/* ------------------------------------------------------ protection rule */

/* Reading R5: is position p of a length-L sequence protected (kept in INT8)? */
int kv4o_is_protected(int p, int L, int S, int R) {
  if (p < S) return 1;
  if (p >= L - R) return 1;
  return 0;
}

/* side-cache slot of a protected position */
int kv4o_side_slot(int p, int S, int R) { return p < S ? p : S + (p % R); }

/* Normalized Hadamard rotation of n values (n a power of two), in place:
 * y = H_n x / sqrt(n), with the Sylvester matrix H_1 = [1],
 * H_2m = [[H_m, H_m], [H_m, -H_m]] (Sec. 3 eq. 3.4: an orthogonal rotation
 * leaves q.k unchanged; App. D.4 rotates K only).  Evaluated in fp32 with
 * round-to-nearest in this order: butterfly stages h = 1, 2, 4, ..., n/2, in
 * which each pair (i, i + h) with bit h of i clear becomes (a + b, a - b);
 * then every value is multiplied by the fp32 value nearest to 1/sqrt(n). */
void kv4o_hadamard_f32(float* x, int n) {
  int old = fegetround();
  fesetround(FE_TONEAREST);
  for (int h = 1; h < n; h <<= 1)
    for (int i = 0; i < n; ++i)
      if (!(i & h)) {
        float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
  float c = (float)(1.0 / sqrt((double)n));
  for (int i = 0; i < n; ++i) x[i] = x[i] * c;
  fesetround(old);
}

void kv4o_hadamard_f32_n(float* x, long rows, int n) {
  for (long r = 0; r < rows; ++r) kv4o_hadamard_f32(x + r * n, n);
}

/* ------------------------------------------------- packed append (bytes) */
/*
 * Packed layout, restated from the library's layout description:
 *
 *   paged cache = [num_pages][h_kv][chunk], chunk bytes = 16*d_h + 128*(d_h/g)
 *   (page size 16), and inside one chunk:
 *     K codes  [16 slots][d_h/2 bytes]   a byte holds two consecutive channels,
 *                                        the even one in its low nibble; a slot
 *                                        row is 4 quarters q = 0..3 of d_h/32
 *                                        four-byte words, and word b of quarter
 *                                        q holds channels 32b + 8q .. 32b + 8q + 7
 *                                        in increasing byte order
 *     V codes  [16 slots][d_h/2 bytes]   logical byte i of a slot row holds
 *                                        channel 2i in its low nibble and channel
 *                                        2i+1 in its high nibble; the row is cut
 *                                        into 16-byte pieces of 32 channels and
 *                                        piece P of slot t is stored at piece
 *                                        position P xor ((t / 2) mod (d_h / 32))
 *     K meta   [16 slots][d_h/g][2 x u16] (Delta16, m16) per group
 *     V Delta  [4 quads][d_h/g][4 x u16]  Delta16 of (slot, group); quad u lists
 *                                        slots 2u, 2u+1, 2u+8, 2u+9 in that order
 *     V m      [4 quads][d_h/g][4 x u16]  m16, same order
 *
 *   side cache = [max_seqs][h_kv][block], NS = S + R, NSP = NS rounded up to
 *   a multiple of 8, block bytes = 2*NS*d_h + 4*NSP, and inside one block:
 *     K8 codes [NS][d_h] int8, V8 codes [NS][d_h] int8,
 *     K8 scale [NSP] u16 (fp16), V8 scale [NSP] u16 (fp16); scale entries
 *     NS..NSP-1 are padding that is never written.  A code row (one slot) is
 *     cut into 16-byte pieces of 16 channels; piece P of slot t is stored at
 *     piece position P xor (t mod (d_h / 16)).
 *
 * All multi-byte fields are little-endian.
 */
static long chunk_bytes(int d_h, int g) { return 16L * d_h + 128L * (d_h / g); }
static long side_scale_entries(int S, int R) { return ((long)S + R + 7) / 8 * 8; }
static long side_block_bytes(int d_h, int S, int R) {
  return 2L * (S + R) * d_h + 4L * side_scale_entries(S, R);
}

static void put_u16(uint8_t* p, uint16_t v) {
  p[0] = (uint8_t)(v & 0xFF);
  p[1] = (uint8_t)(v >> 8);
}

/* Append T tokens: INT4 for every position, INT8 side entry for protected
 * positions of the final length seq_lens[seq] (ring entries only for positions
 * inside the final recent window, reading R6).  rotate_k: K is first rotated
 * by kv4o_hadamard_f32 (reading R9; V never is).  Returns the OR of status bits. */
int kv4o_quant_append(int h_kv, int d_h, int g, int S, int R, int max_seqs, int num_pages,
                      int max_pages_per_seq, uint8_t* paged, uint8_t* side,
                      const uint16_t* k_new, const uint16_t* v_new, const int32_t* tok_seq,
                      const int32_t* tok_pos, int T, const int32_t* seq_lens,
                      const int32_t* block_table, int rotate_k) {
  int status = 0;
  int ng = d_h / g;
  long cb = chunk_bytes(d_h, g);
  long sb = side_block_bytes(d_h, S, R);
  int NS = S + R;
  float x[1024];
  uint8_t c4[1024];
  int8_t c8[1024];
  for (int t = 0; t < T; ++t) {
    int s = tok_seq[t], p = tok_pos[t];
    if (s < 0 || s >= max_seqs) {
      status |= KV4O_ST_BAD_SEQ;
      continue;
    }
    int L = seq_lens[s];
    if (p < 0 || p >= L || p >= max_pages_per_seq * 16) {
      status |= KV4O_ST_BAD_POS;
      continue;
    }
    int page = block_table[(long)s * max_pages_per_seq + p / 16];
    if (page < 0 || page >= num_pages) {
      status |= KV4O_ST_BAD_PAGE;
      continue;
    }
    int slot = p % 16;
    int prot = kv4o_is_protected(p, L, S, R) && (p < S || R > 0);
    for (int h = 0; h < h_kv; ++h) {
      uint8_t* chunk = paged + ((long)page * h_kv + h) * cb;
      for (int kv = 0; kv < 2; ++kv) {
        const uint16_t* src = (kv == 0 ? k_new : v_new) + ((long)t * h_kv + h) * d_h;
        for (int d = 0; d < d_h; ++d) x[d] = kv4o_bf16_to_f32(src[d]);
        if (rotate_k && kv == 0) kv4o_hadamard_f32(x, d_h);
        uint8_t* rows = chunk + (long)kv * 16 * (d_h / 2) + (long)slot * (d_h / 2);
        for (int j = 0; j < ng; ++j) {
          uint16_t d16, m16;
          status |= kv4o_int4_encode_group(x + j * g, g, c4 + j * g, &d16, &m16);
          if (kv == 0) {
            uint8_t* meta = chunk + 16L * d_h + (long)slot * ng * 4 + 4 * j;
            put_u16(meta, d16);
            put_u16(meta + 2, m16);
          } else {
            /* quad of the slot, its place among the quad's 4 entries */
            int quad = (slot % 8) / 2, at = 2 * (slot / 8) + slot % 2;
            long entry = ((long)quad * ng + j) * 4 + at;
            uint8_t* vmeta = chunk + 16L * d_h + 64L * ng;
            put_u16(vmeta + 2 * entry, d16);
            put_u16(vmeta + 32L * ng + 2 * entry, m16);
          }
        }
        int npieces = d_h / 32;
        for (int i = 0; i < d_h / 2; ++i) {
          int dst;
          if (kv == 0) {
            int ch = 2 * i, blk = ch / 32, quarter = (ch % 32) / 8;
            dst = 4 * (quarter * npieces + blk) + (ch % 8) / 2;
          } else {
            int piece = i / 16, within = i % 16;
            dst = 16 * (piece ^ ((slot / 2) % npieces)) + within;
          }
          rows[dst] = (uint8_t)(c4[2 * i] | (c4[2 * i + 1] << 4));
        }
        if (prot) {
          int ss = kv4o_side_slot(p, S, R);
          uint8_t* blk = side + ((long)s * h_kv + h) * sb;
          uint8_t* codes = blk + (long)kv * NS * d_h + (long)ss * d_h;
          uint8_t* scl = blk + 2L * NS * d_h + (long)kv * side_scale_entries(S, R) * 2 + (long)ss * 2;
          uint16_t s16;
          status |= kv4o_int8_encode_vec(x, d_h, c8, &s16);
          for (int i = 0; i < d_h; ++i) {
            int dst = 16 * ((i / 16) ^ (ss % (d_h / 16))) + i % 16;
            codes[dst] = c8[i];
          }
          put_u16(scl, s16);
        }
      }
    }
  }
  return status;
}

/* ------------------------------------------------------------ decoding */

/* Dequantized cache of one sequence, fp64, for all L positions (reading R5):
 * protected positions decode the INT8 entry s*c, the rest the INT4 entry
 * Delta*c + m (Sec. 3 eq. 3.3).  k_src/v_src: [h_kv][L][d_h] bf16 bits.
 * k_hat/v_hat: [h_kv][L][d_h].  rotate_k: K is rotated (kv4o_hadamard_f32)
 * before it is quantized.  Returns status bits. */
int kv4o_dequant_seq(int h_kv, int d_h, int g, int S, int R, int L, const uint16_t* k_src,
                     const uint16_t* v_src, double* k_hat, double* v_hat, int rotate_k) {
  int status = 0;
  int ng = d_h / g;
  float x[1024];
  uint8_t c4[1024];
  int8_t c8[1024];
  for (int h = 0; h < h_kv; ++h) {
    for (int p = 0; p < L; ++p) {
      for (int kv = 0; kv < 2; ++kv) {
        const uint16_t* src = (kv == 0 ? k_src : v_src) + ((long)h * L + p) * d_h;
        double* dst = (kv == 0 ? k_hat : v_hat) + ((long)h * L + p) * d_h;
        for (int d = 0; d < d_h; ++d) x[d] = kv4o_bf16_to_f32(src[d]);
        if (rotate_k && kv == 0) kv4o_hadamard_f32(x, d_h);
        if (kv4o_is_protected(p, L, S, R)) {
          uint16_t s16;
          status |= kv4o_int8_encode_vec(x, d_h, c8, &s16);
          double sf = (double)kv4o_f16_to_f32(s16);
          for (int d = 0; d < d_h; ++d) dst[d] = sf * (double)c8[d];
        } else {
          for (int j = 0; j < ng; ++j) {
            uint16_t d16, m16;
            status |= kv4o_int4_encode_group(x + j * g, g, c4 + j * g, &d16, &m16);
            double df = (double)kv4o_f16_to_f32(d16), mf = (double)kv4o_f16_to_f32(m16);
            for (int i = 0; i < g; ++i) dst[j * g + i] = df * (double)c4[j * g + i] + mf;
          }
        }
      }
    }
  }
  return status;
}

/* Plain softmax attention in fp64 over a dequantized sequence (reading R7).
 * q: [h_q][d_h] bf16 bits; k_hat/v_hat: [h_kv][L][d_h]; out: [h_q][d_h];
 * lse: [h_q] (natural log of the softmax normaliser of the scaled scores).
 * scratch: L doubles.  L == 0 gives out = 0 and lse = -inf. */
void kv4o_attend(int h_q, int h_kv, int d_h, int L, const uint16_t* q, const double* k_hat,
                 const double* v_hat, double sm_scale, double* out, double* lse,
                 double* scratch) {
  int G = h_q / h_kv;
  for (int j = 0; j < h_q; ++j) {
    int h = j / G;
    double* o = out + (long)j * d_h;
    for (int d = 0; d < d_h; ++d) o[d] = 0.0;
    if (L == 0) {
      lse[j] = -INFINITY;
      continue;
    }
    double M = -INFINITY;
    for (int p = 0; p < L; ++p) {
      const double* k = k_hat + ((long)h * L + p) * d_h;
      double s = 0.0;
      for (int d = 0; d < d_h; ++d) s += (double)kv4o_bf16_to_f32(q[(long)j * d_h + d]) * k[d];
      s *= sm_scale;
      scratch[p] = s;
      if (s > M) M = s;
    }
    double Z = 0.0;
    for (int p = 0; p < L; ++p) {
      double w = exp(scratch[p] - M);
      scratch[p] = w;
      Z += w;
    }
    for (int p = 0; p < L; ++p) {
      const double* v = v_hat + ((long)h * L + p) * d_h;
      double w = scratch[p] / Z;
      for (int d = 0; d < d_h; ++d) o[d] += w * v[d];
    }
    lse[j] = M + log(Z);
  }
}

/* Regional / split merge (App. A.3 eq. A1), generalised to n parts:
 * z = log sum_r e^{z_r}, o = sum_r e^{z_r - z} o_r; parts with z_r = -inf have
 * weight 0; all parts empty gives o = 0, z = -inf.
 * o_parts: [n][d]; z_parts: [n]. */
void kv4o_combine(int n, int d, const double* o_parts, const double* z_parts, double* out,
                  double* out_z) {
  double M = -INFINITY;
  for (int r = 0; r < n; ++r)
    if (z_parts[r] > M) M = z_parts[r];
  for (int i = 0; i < d; ++i) out[i] = 0.0;
  if (M == -INFINITY) {
    *out_z = -INFINITY;
    return;
  }
  double Z = 0.0;
  for (int r = 0; r < n; ++r) Z += exp(z_parts[r] - M);
  double z = M + log(Z);
  for (int r = 0; r < n; ++r) {
    if (z_parts[r] == -INFINITY) continue;
    double w = exp(z_parts[r] - z);
    for (int i = 0; i < d; ++i) out[i] += w * o_parts[(long)r * d + i];
  }
  *out_z = z;
}

/* ------------------------------------------- array helpers for the tests */

void kv4o_f32_to_f16_n(const float* x, long n, int mode, uint16_t* out) {
  for (long i = 0; i < n; ++i) out[i] = kv4o_f32_to_f16(x[i], mode);
}

void kv4o_sub_dir_n(const float* a, const float* b, long n, int mode, float* out) {
  for (long i = 0; i < n; ++i) out[i] = kv4o_sub_dir(a[i], b[i], mode);
}

void kv4o_div_dir_n(const float* a, const float* b, long n, int mode, float* out) {
  for (long i = 0; i < n; ++i) out[i] = kv4o_div_dir(a[i], b[i], mode);
}

int kv4o_int4_encode_n(const float* x, long ngroups, int g, uint8_t* codes, uint16_t* delta16,
                       uint16_t* off16) {
  int st = 0;
  for (long k = 0; k < ngroups; ++k)
    st |= kv4o_int4_encode_group(x + k * g, g, codes + k * g, delta16 + k, off16 + k);
  return st;
}

int kv4o_int8_encode_n(const float* x, long nvec, int n, int8_t* codes, uint16_t* scale16) {
  int st = 0;
  for (long k = 0; k < nvec; ++k) st |= kv4o_int8_encode_vec(x + k * n, n, codes + k * n, scale16 + k);
  return st;
}
