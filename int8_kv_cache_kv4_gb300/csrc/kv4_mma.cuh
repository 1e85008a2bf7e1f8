// kv4_mma.cuh -- warp-level tensor-core helpers shared by the decode kernels:
// the m16n8k16 fp16 MMA, transposing shared-memory matrix loads, and the
// conversions that widen packed 4-bit / 8-bit codes to exact fp16 values.
#pragma once
#include "kv4_common.cuh"

namespace kv4 {

// (no side effects besides its register results: not volatile, so the
// compiler may schedule shared-memory reads across it)
__device__ inline void mma_f16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                               uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ inline void ldsm_x4_trans(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ inline uint32_t hfma2(uint32_t x, uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(x), "r"(a), "r"(b));
  return d;
}

__device__ inline float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ inline uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// (low half of a, low half of b)
__device__ inline uint32_t lo_lo(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x5410); }

__device__ inline float2 h2f2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

__device__ inline uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ inline uint32_t u4word(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Shared-memory loads at 32-bit shared addresses (base register + immediate
// offsets).  Volatile: kept after the mbarrier wait and before the refill
// that reuses the stage, which are volatile too.
__device__ inline uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ inline uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ inline uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

__device__ inline void sts16(uint32_t a, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"((unsigned short)v));
}

// (a & m) | c as one three-input logic op.  Written as C++ the same
// expression compiled to two logic ops per value on sm_103a (measured with
// the executed-instruction counters); the widening routines below are the
// decode kernels' busiest code.
__device__ inline uint32_t and_or(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(m), "r"(c));
  return d;
}

// fp16 pairs: 1.0, -1032 (= -(1024 + 8)), 1/16, -72 (= -(64 + 8))
constexpr uint32_t kOne2 = 0x3C003C00u, kM1032 = 0xE408E408u;
constexpr uint32_t kSixteenth2 = 0x2C002C00u, kM72 = 0xD480D480u;

// Widen 8 V codes (two tokens x four channels, nibbles 0-3 and 4-7 of w) to
// fp16 pairs (token a, token b) of the centred value c - 8, channel +0..+3.
__device__ inline void widen_v(uint32_t w, uint32_t x[4]) {
  x[0] = hfma2(and_or(w, 0x000F000Fu, 0x64006400u), kOne2, kM1032);
  x[1] = hfma2(and_or(w, 0x00F000F0u, 0x64006400u), kSixteenth2, kM72);
  const uint32_t w8 = w >> 8;
  x[2] = hfma2(and_or(w8, 0x000F000Fu, 0x64006400u), kOne2, kM1032);
  x[3] = hfma2(and_or(w8, 0x00F000F0u, 0x64006400u), kSixteenth2, kM72);
}

// Widen 8 V codes (two tokens x four channels) to fp16 pairs whose bit
// patterns are the codes themselves: subnormal values c * 2^-24 (low nibbles,
// pairs 0 and 2) and 16 c * 2^-24 (high nibbles, pairs 1 and 3).  One logic
// op per pair; the consumer scales its accumulators by 2^24 and 2^20.
__device__ inline void widen_v_sub(uint32_t w, uint32_t x[4]) {
  x[0] = w & 0x000F000Fu;
  x[1] = w & 0x00F000F0u;
  const uint32_t w8 = w >> 8;
  x[2] = w8 & 0x000F000Fu;
  x[3] = w8 & 0x00F000F0u;
}

// Widen one K code word (8 channels of one token) to 4 fp16 pairs without
// removing the exponent offset: pairs 0 and 2 hold 1024 + c (channels i and
// i + 4 of the low nibbles), pairs 1 and 3 hold 1024 + 16 c (high nibbles).
// The consumer folds the 1024 and the 16 into its other operand.
__device__ inline void widen_k_biased(uint32_t w, uint32_t x[4]) {
  x[0] = and_or(w, 0x000F000Fu, 0x64006400u);
  x[1] = and_or(w, 0x00F000F0u, 0x64006400u);
  const uint32_t w8 = w >> 8;
  x[2] = and_or(w8, 0x000F000Fu, 0x64006400u);
  x[3] = and_or(w8, 0x00F000F0u, 0x64006400u);
}

// fp16 pairs -1024 and -64
constexpr uint32_t kM1024 = 0xE400E400u, kM64 = 0xD400D400u;

// Widen one K code word (8 channels of one token) to 4 fp16 pairs of exact
// codes: pair i = (channel i, channel i + 4).
__device__ inline void widen_k(uint32_t w, uint32_t x[4]) {
  x[0] = hfma2(and_or(w, 0x000F000Fu, 0x64006400u), kOne2, kM1024);
  x[1] = hfma2(and_or(w, 0x00F000F0u, 0x64006400u), kSixteenth2, kM64);
  const uint32_t w8 = w >> 8;
  x[2] = hfma2(and_or(w8, 0x000F000Fu, 0x64006400u), kOne2, kM1024);
  x[3] = hfma2(and_or(w8, 0x00F000F0u, 0x64006400u), kSixteenth2, kM64);
}

// (Delta, m) of V for slot t and group grp of a chunk, as one word (Delta in
// the low half), gathered from the V metadata's two arrays.
__device__ inline uint32_t vmeta_word(const uint8_t* chunk, int t, int grp, int d_h, int g) {
  return (uint32_t)*reinterpret_cast<const uint16_t*>(chunk + v_delta_byte(t, grp, d_h, g)) |
         ((uint32_t)*reinterpret_cast<const uint16_t*>(chunk + v_offset_byte(t, grp, d_h, g))
          << 16);
}
// The four words of a K code row that hold block blk (channels 32 blk ..
// 32 blk + 31), in channel order.
__device__ inline uint4 k_block_words(const uint8_t* row, int blk, int d_h) {
  uint4 w;
  w.x = *reinterpret_cast<const uint32_t*>(row + k_row_byte(32 * blk, d_h));
  w.y = *reinterpret_cast<const uint32_t*>(row + k_row_byte(32 * blk + 8, d_h));
  w.z = *reinterpret_cast<const uint32_t*>(row + k_row_byte(32 * blk + 16, d_h));
  w.w = *reinterpret_cast<const uint32_t*>(row + k_row_byte(32 * blk + 24, d_h));
  return w;
}

template <int NG>
struct MetaRow;  // one slot's NG (Delta, m) words
template <>
struct MetaRow<4> {
  uint4 v;
  __device__ void load(const uint8_t* p) { v = *reinterpret_cast<const uint4*>(p); }
  __device__ void load_v(const uint8_t* c, int t, int d_h) {
    v = make_uint4(vmeta_word(c, t, 0, d_h, d_h / 4), vmeta_word(c, t, 1, d_h, d_h / 4),
                   vmeta_word(c, t, 2, d_h, d_h / 4), vmeta_word(c, t, 3, d_h, d_h / 4));
  }
  __device__ void load_s(uint32_t a) { v = lds128(a); }
  __device__ uint32_t get(int g) const { return u4word(v, g); }
  __device__ void zero() { v = make_uint4(0u, 0u, 0u, 0u); }
};
template <>
struct MetaRow<2> {
  uint2 v;
  __device__ void load(const uint8_t* p) { v = *reinterpret_cast<const uint2*>(p); }
  __device__ void load_v(const uint8_t* c, int t, int d_h) {
    v = make_uint2(vmeta_word(c, t, 0, d_h, d_h / 2), vmeta_word(c, t, 1, d_h, d_h / 2));
  }
  __device__ void load_s(uint32_t a) { v = lds64(a); }
  __device__ uint32_t get(int g) const { return g == 0 ? v.x : v.y; }
  __device__ void zero() { v = make_uint2(0u, 0u); }
};
template <>
struct MetaRow<1> {
  uint32_t v;
  __device__ void load(const uint8_t* p) { v = *reinterpret_cast<const uint32_t*>(p); }
  __device__ void load_v(const uint8_t* c, int t, int d_h) { v = vmeta_word(c, t, 0, d_h, d_h); }
  __device__ void load_s(uint32_t a) { v = lds32(a); }
  __device__ uint32_t get(int) const { return v; }
  __device__ void zero() { v = 0u; }
};

__device__ inline float lo_f(uint32_t w) { return f16_bits_to_f32(w & 0xFFFFu); }
__device__ inline float hi_f(uint32_t w) { return f16_bits_to_f32(w >> 16); }

// 8-bit codes: x ^ 0x80 turns a signed code c into the byte c + 128; with the
// byte placed under an fp16 exponent of 2^10 the half is 1024 + 128 + c, and
// subtracting 1152 leaves c exactly.
constexpr uint32_t kMagic64 = 0x64646464u, kF1152x2 = 0x64806480u;
__device__ inline uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// fp16 pair (code of byte i, code of byte j) of the biased word xb = w ^ 0x80808080;
// sel = 0x4j4i selects the two bytes under the 0x64 exponent byte
__device__ inline uint32_t i8pair(uint32_t xb, uint32_t sel) {
  return hsub2(__byte_perm(xb, kMagic64, sel), kF1152x2);
}

}  // namespace kv4
