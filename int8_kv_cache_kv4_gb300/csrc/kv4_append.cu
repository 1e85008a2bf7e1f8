// kv4_append.cu -- quantize-on-append: each new K/V token-head vector is
// written as head-wise affine INT4 (per group of g channels: FP16 scale Delta
// and offset m, 4-bit codes c with x^ = Delta*c + m; KV4-RL Sec. 3 eq. 3.3,
// Sec. 5.1, App. A.3) into its 16-token page, and -- when the position is a
// sink or inside the final recent window (Sec. 5.2) -- also as a symmetric
// INT8 side entry computed from the same source vector (App. A.3).
//
// One warp per (token, kv head); lane l owns channels [4l, 4l+4) of K and V
// (head_dim 128; head_dim 64 uses lanes 0..15).  Group min/max and the INT8
// absolute maximum are warp-shuffle reductions; codes are packed two per byte
// (low nibble = even channel) and stored as one 16-bit word per lane, so a
// slot row of 64 bytes is one coalesced store.  Rounding follows the layout
// header's rules exactly (directed fp32 ops and fp16 conversions), which makes
// the written bytes bit-identical to the CPU oracle.
//
// The rotating variant first turns each K vector into H k with H the
// normalized Sylvester-Hadamard matrix of order head_dim (KV4-RL Sec. 3
// eq. 3.4: an orthogonal H applied to both q and k leaves q.k unchanged;
// App. A.3 "Encoding and allocation": K rotated after RoPE, V in its own
// basis; App. D.4 keeps the rotation K-only).  The query side of the same
// rotation is hadamard_bf16_kernel below.
#include <cmath>

#include "kv4_common.cuh"

namespace kv4 {

// Reduce over the `span` lanes of a group (span a power of two <= 32).
__device__ inline float group_min(float v, int span) {
  for (int o = 1; o < span; o <<= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ inline float group_max(float v, int span) {
  for (int o = 1; o < span; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ inline int group_or(int v, int span) {
  for (int o = 1; o < span; o <<= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// INT4-encode this lane's 4 channels of a group whose lanes span `span`
// lanes.  Returns the packed 16-bit code word and, via meta, (Delta, m) bits.
__device__ inline uint32_t encode_int4(const float x[4], int span, uint32_t* meta, int* bad) {
  float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
  float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  int nf = !(isfinite(x[0]) && isfinite(x[1]) && isfinite(x[2]) && isfinite(x[3]));
  mn = group_min(mn, span);
  mx = group_max(mx, span);
  nf = group_or(nf, span);
  uint32_t codes = 0;
  uint16_t d16 = 0, m16 = 0;
  if (!nf) {
    __half mh = __float2half_rd(mn);
    float mf = __half2float(mh);
    float span_f = __fsub_ru(mx, mf);
    float step = __fdiv_ru(span_f, 15.0f);
    __half dh = __float2half_ru(step);
    float df = __half2float(dh);
    if (!isfinite(mf) || !isfinite(df)) {
      nf = 1;
    } else {
      m16 = __half_as_ushort(mh);
      d16 = __half_as_ushort(dh);
      if (df != 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          int c = __float2int_rn(__fdiv_rn(__fsub_rn(x[i], mf), df));
          c = min(max(c, 0), 15);
          codes |= (uint32_t)c << (4 * i);
        }
      }
    }
  }
  if (nf) {
    codes = 0;
    d16 = 0;
    m16 = 0;
  }
  *bad |= nf;
  *meta = (uint32_t)d16 | ((uint32_t)m16 << 16);
  return codes;
}

// INT8-encode this lane's 4 channels of a token-head vector spread over
// `lanes` lanes.  Returns 4 packed int8 codes and, via scale, the fp16 bits.
__device__ inline uint32_t encode_int8(const float x[4], int lanes, uint16_t* scale, int* bad) {
  float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  int nf = !(isfinite(x[0]) && isfinite(x[1]) && isfinite(x[2]) && isfinite(x[3]));
  a = group_max(a, lanes);
  nf = group_or(nf, lanes);
  uint32_t out = 0;
  uint16_t s16 = 0;
  if (!nf) {
    __half sh = __float2half_ru(__fdiv_ru(a, 127.0f));
    float sf = __half2float(sh);
    if (!isfinite(sf)) {
      nf = 1;
    } else {
      s16 = __half_as_ushort(sh);
      if (sf != 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          int c = __float2int_rn(__fdiv_rn(x[i], sf));
          c = min(max(c, -127), 127);
          out |= ((uint32_t)c & 0xFFu) << (8 * i);
        }
      }
    }
  }
  if (nf) {
    out = 0;
    s16 = 0;
  }
  *bad |= nf;
  *scale = s16;
  return out;
}

// Validate a token; returns the physical page or -1 (status already set).
__device__ inline int token_page(const Layout& L, int s, int p, const int32_t* seq_lens,
                                 const int32_t* block_table, int32_t* status, bool report,
                                 int* seq_len_out) {
  if (s < 0 || s >= L.max_seqs) {
    if (report) set_status(status, KV4_STATUS_BAD_SEQ);
    return -1;
  }
  int len = seq_lens[s];
  if (p < 0 || p >= len || p >= L.max_pages * kPage) {
    if (report) set_status(status, KV4_STATUS_BAD_POS);
    return -1;
  }
  int page = block_table[(long long)s * L.max_pages + p / kPage];
  if (page < 0 || page >= L.num_pages) {
    if (report) set_status(status, KV4_STATUS_BAD_PAGE);
    return -1;
  }
  *seq_len_out = len;
  return page;
}

template <bool kRotateK>
__global__ void __launch_bounds__(256) quant_append_kernel(
    Layout L, uint8_t* __restrict__ paged, uint8_t* __restrict__ side,
    const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
    const int32_t* __restrict__ tok_seq, const int32_t* __restrict__ tok_pos, int T,
    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
    int32_t* status, float hc) {
  // A decode launched next as a programmatic dependent may start its set-up
  // now: it waits for this grid before it reads any page.  (Before its own
  // wait below this kernel only reads its inputs, which no kernel of this
  // library writes.)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= (long long)T * L.h_kv) return;
  const int t = (int)(w / L.h_kv);
  const int h = (int)(w % L.h_kv);
  const int d_h = L.d_h, g = L.g, ng = d_h / g;
  const int lanes = d_h / 4;  // active lanes (32 at d_h = 128, 16 at 64)
  const int span = g / 4;     // lanes per INT4 group
  const bool active = lane < lanes;
  const int c0 = (active ? lane : 0) * 4;
  // The new K and V rows are read and encoded first: they do not depend on
  // the page lookup (token -> length -> block table), so the two latencies
  // overlap.  Both encodings are formed; the INT8 one is stored only for a
  // protected position (non-finite input is flagged by either).
  int bad = 0;
  uint32_t codes[2], meta[2], c8[2];
  uint16_t s16[2];
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {  // 4 bf16, 8-byte aligned
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>((kv == 0 ? k_new : v_new) +
                                                         ((long long)t * L.h_kv + h) * d_h + c0));
    float x[4] = {bf16_bits_to_f32(raw.x & 0xFFFFu), bf16_bits_to_f32(raw.x >> 16),
                  bf16_bits_to_f32(raw.y & 0xFFFFu), bf16_bits_to_f32(raw.y >> 16)};
    if (!active) x[0] = x[1] = x[2] = x[3] = 0.f;
    if (kRotateK && kv == 0) hadamard_warp(x, d_h, hc);  // before both encoders
    codes[kv] = encode_int4(x, span, &meta[kv], &bad);
    c8[kv] = encode_int8(x, lanes < 32 ? lanes : 32, &s16[kv], &bad);
  }
  const int s = tok_seq[t], p = tok_pos[t];
  int len = 0;
  const int page = token_page(L, s, p, seq_lens, block_table, status, lane == 0 && h == 0, &len);
  if (page < 0) return;
  // Launched as a programmatic dependent of the kernel before it (often the
  // previous step's decode, which reads the side-cache ring slot this token
  // may overwrite): nothing of the cache is written before that kernel has
  // completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int slot = p % kPage;
  const bool prot = (p < L.S) || (L.R > 0 && p >= len - L.R);
  uint8_t* chunk = paged + ((long long)page * L.h_kv + h) * chunk_bytes(d_h, g);
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    if (active) {
      uint8_t* row = chunk + (kv == 0 ? 0 : codes_off_v(d_h)) + slot * (d_h / 2);
      // 4 codes of channels c0..c0+3 -> two bytes (low nibble = even channel)
      const int b = kv == 0 ? k_row_byte(c0, d_h) : row_byte(2 * lane, slot, d_h);
      *reinterpret_cast<uint16_t*>(row + b) = (uint16_t)codes[kv];
      if ((lane % span) == 0) {
        const int grp = lane / span;
        if (kv == 0) {
          *reinterpret_cast<uint32_t*>(chunk + meta_off_k(d_h) + slot * ng * 4 + 4 * grp) = meta[kv];
        } else {
          *reinterpret_cast<uint16_t*>(chunk + v_delta_byte(slot, grp, d_h, g)) = (uint16_t)meta[kv];
          *reinterpret_cast<uint16_t*>(chunk + v_offset_byte(slot, grp, d_h, g)) =
              (uint16_t)(meta[kv] >> 16);
        }
      }
    }
    if (prot) {
      const int NS = L.S + L.R;
      const int ss = side_slot(p, L.S, L.R);
      uint8_t* blk = side + ((long long)s * L.h_kv + h) * side_block_bytes(d_h, L.S, L.R);
      if (active)
        *reinterpret_cast<uint32_t*>(blk + (long long)kv * NS * d_h + (long long)ss * d_h +
                                     side_byte(c0, ss, d_h)) = c8[kv];
      if (lane == 0)
        *reinterpret_cast<uint16_t*>(blk + 2LL * NS * d_h +
                                     (long long)kv * side_scale_entries(L.S, L.R) * 2 + ss * 2) =
            s16[kv];
    }
  }
  if (bad && lane == 0) set_status(status, KV4_STATUS_NONFINITE);
  // V metadata outside the range of the tensor-core decode's fp16 PV operand
  // (P' = p Delta, p <= 2^8): Delta >= 256 (fp16 bits 0x5C00 and up; Delta is
  // never negative) or a nonzero subnormal Delta (bits below 0x0400), and the
  // same for a stored INT8 scale
  auto out_of_range = [](uint32_t h) { return h >= 0x5C00u || (h != 0u && h < 0x0400u); };
  const bool v_out = (active && out_of_range(meta[1] & 0xFFFFu)) || (prot && out_of_range(s16[1]));
  if (__any_sync(0xffffffffu, v_out) && lane == 0) set_status(status, KV4_STATUS_V_RANGE);
}

// Comparator cache: [page][h_kv][K|V][16][d_h] bf16, plain copy.
__global__ void __launch_bounds__(256) bf16_append_kernel(
    Layout L, uint16_t* __restrict__ cache, const uint16_t* __restrict__ k_new,
    const uint16_t* __restrict__ v_new, const int32_t* __restrict__ tok_seq,
    const int32_t* __restrict__ tok_pos, int T, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ block_table, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= (long long)T * L.h_kv) return;
  const int t = (int)(w / L.h_kv);
  const int h = (int)(w % L.h_kv);
  int len = 0;
  const int page =
      token_page(L, tok_seq[t], tok_pos[t], seq_lens, block_table, status, lane == 0 && h == 0,
                 &len);
  if (page < 0) return;
  const int d_h = L.d_h;
  const int slot = tok_pos[t] % kPage;
  uint16_t* base = cache + ((long long)page * L.h_kv + h) * 2 * kPage * d_h;
  for (int c = lane * 4; c < d_h; c += 128) {
    const long long src = ((long long)t * L.h_kv + h) * d_h + c;
    *reinterpret_cast<uint2*>(base + slot * d_h + c) = *reinterpret_cast<const uint2*>(k_new + src);
    *reinterpret_cast<uint2*>(base + (kPage + slot) * d_h + c) =
        *reinterpret_cast<const uint2*>(v_new + src);
  }
}

cudaError_t launch_quant_append(const Layout& L, void* paged, void* side, const uint16_t* k_new,
                                const uint16_t* v_new, const int32_t* tok_seq,
                                const int32_t* tok_pos, int T, const int32_t* seq_lens,
                                const int32_t* block_table, int32_t* status, bool rotate_k,
                                cudaStream_t st) {
  const long long warps = (long long)T * L.h_kv;
  const int wpb = 8;
  const long long blocks = (warps + wpb - 1) / wpb;
  // A programmatic dependent of the kernel before it: the grid may start (and
  // read and encode its tokens) while that kernel still runs, and waits for it
  // before writing the cache.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(wpb * 32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (rotate_k)
    return cudaLaunchKernelEx(&cfg, quant_append_kernel<true>, L, (uint8_t*)paged, (uint8_t*)side,
                              k_new, v_new, tok_seq, tok_pos, T, seq_lens, block_table, status,
                              hadamard_scale(L.d_h));
  return cudaLaunchKernelEx(&cfg, quant_append_kernel<false>, L, (uint8_t*)paged, (uint8_t*)side,
                            k_new, v_new, tok_seq, tok_pos, T, seq_lens, block_table, status, 1.0f);
}

// Query side of the K rotation: each row of d bf16 values becomes H x rounded
// to bf16 (nearest even).  One warp per row; lane l reads and writes channels
// 4l..4l+3 as one 8-byte word.  x and y may be the same array: a warp reads its
// whole row into registers before any lane writes.
__global__ void __launch_bounds__(256) hadamard_bf16_kernel(const uint16_t* x, uint16_t* y,
                                                            long long rows, int d, float hc) {
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const bool active = 4 * lane < d;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (active) {
    const uint2 raw = *reinterpret_cast<const uint2*>(x + r * d + 4 * lane);
    v[0] = bf16_bits_to_f32(raw.x & 0xFFFFu);
    v[1] = bf16_bits_to_f32(raw.x >> 16);
    v[2] = bf16_bits_to_f32(raw.y & 0xFFFFu);
    v[3] = bf16_bits_to_f32(raw.y >> 16);
  }
  hadamard_warp(v, d, hc);
  if (active) {
    uint2 o;
    o.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[0])) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[1])) << 16);
    o.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[2])) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[3])) << 16);
    *reinterpret_cast<uint2*>(y + r * d + 4 * lane) = o;
  }
}

cudaError_t launch_hadamard_bf16(const uint16_t* x, uint16_t* y, long long rows, int d,
                                 cudaStream_t st) {
  const int wpb = 8;
  const long long blocks = (rows + wpb - 1) / wpb;
  hadamard_bf16_kernel<<<(unsigned)blocks, wpb * 32, 0, st>>>(x, y, rows, d, hadamard_scale(d));
  return cudaGetLastError();
}

cudaError_t launch_bf16_append(const Layout& L, void* cache, const uint16_t* k_new,
                               const uint16_t* v_new, const int32_t* tok_seq,
                               const int32_t* tok_pos, int T, const int32_t* seq_lens,
                               const int32_t* block_table, int32_t* status, cudaStream_t st) {
  const long long warps = (long long)T * L.h_kv;
  const int wpb = 8;
  const long long blocks = (warps + wpb - 1) / wpb;
  bf16_append_kernel<<<(unsigned)blocks, wpb * 32, 0, st>>>(
      L, (uint16_t*)cache, k_new, v_new, tok_seq, tok_pos, T, seq_lens, block_table, status);
  return cudaGetLastError();
}

// ------------------------------------------------- FP4 probe formats
// KV4-RL App. D.4 (Fig. A4(c)) compares affine INT4 with two FP4 formats as
// fidelity probes that reconstruct the stored cache and attend with bf16
// operands: NVFP4 (E2M1 values, one E4M3 scale per 16 elements, one fp32
// global scale per token-head vector) and MXFP4 (E2M1 values, one E8M0 scale
// per 32 elements).  Scale rules (the pages name the formats only):
//   NVFP4  S = a / 2688 (a = max|x| of the vector, 2688 = 6 * 448);
//          s_b = E4M3(amax_b / (6 S)) per block of 16; e_b = E4M3value(s_b) * S;
//          q = E2M1(x / e_b)                      (q = 0 when e_b = 0)
//   MXFP4  E = floor(log2 amax_b) - 2 per block of 32, clamped to [-127, 127]
//          (-127 for an all-zero block); q = E2M1(x * 2^-E)
// each step one fp32 operation rounded to nearest even; E2M1 rounds to the
// nearest of 0, .5, 1, 1.5, 2, 3, 4, 6 with ties to the even code, saturating
// at 6 and keeping the sign; E4M3 rounds to nearest even, saturating at 448.
// Probe cache: [page][h_kv][K, V][16 slots][row], row = d/2 + 16 bytes: the
// codes (byte i = channel 2i low nibble, 2i+1 high), then the block scales,
// and for NVFP4 the fp32 S at byte d/2 + 12.

constexpr int kFp4Nv = 1, kFp4Mx = 2;
__host__ __device__ inline int fp4_row_bytes(int d_h) { return d_h / 2 + 16; }

// E2M1 code of y: nearest magnitude, ties to the even code (strict '>' at the
// midpoints that round down, '>=' where they round up), saturating at 6.
__device__ inline uint32_t e2m1_code(float y) {
  const float a = fabsf(y);
  uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
               (a >= 3.5f) + (a > 5.0f);
  return c | (signbit(y) ? 8u : 0u);
}
__device__ inline float e2m1_value(uint32_t c) {
  const uint32_t e = (c >> 1) & 3u, m = c & 1u;
  const float v = e == 0 ? 0.5f * (float)m : __uint_as_float(((e + 126u) << 23) | (m << 22));
  return (c & 8u) ? -v : v;
}
// E4M3 code of t >= 0 (nearest even, saturating at 448), and its value
__device__ inline uint32_t e4m3_code(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
  return r & 0xFFu;
}
__device__ inline float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  const float v = e == 0 ? (float)m * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (c & 0x80u) ? -v : v;
}
// 2^k as an fp32 for k in [-127, 127] (2^-127 is subnormal)
__device__ inline float pow2f(int k) {
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}
// floor(log2 a) of a finite a > 0
__device__ inline int ilog2f(float a) {
  const uint32_t u = __float_as_uint(a);
  const int ex = (int)(u >> 23);
  return ex ? ex - 127 : (31 - __clz((int)(u & 0x7FFFFFu))) - 149;
}

template <int kFmt, bool kRotateK>
__global__ void __launch_bounds__(256) fp4_append_kernel(
    Layout L, uint8_t* __restrict__ cache, const uint16_t* __restrict__ k_new,
    const uint16_t* __restrict__ v_new, const int32_t* __restrict__ tok_seq,
    const int32_t* __restrict__ tok_pos, int T, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ block_table, int32_t* status, float hc) {
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= (long long)T * L.h_kv) return;
  const int t = (int)(w / L.h_kv);
  const int h = (int)(w % L.h_kv);
  const int s = tok_seq[t], p = tok_pos[t];
  int len = 0;
  const int page = token_page(L, s, p, seq_lens, block_table, status, lane == 0 && h == 0, &len);
  if (page < 0) return;
  const int d_h = L.d_h, lanes = d_h / 4, rb = fp4_row_bytes(d_h);
  const bool active = lane < lanes;
  const int c0 = (active ? lane : 0) * 4;
  int bad = 0;
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    const uint16_t* src = (kv == 0 ? k_new : v_new) + ((long long)t * L.h_kv + h) * d_h + c0;
    const uint2 raw = *reinterpret_cast<const uint2*>(src);
    float x[4] = {bf16_bits_to_f32(raw.x & 0xFFFFu), bf16_bits_to_f32(raw.x >> 16),
                  bf16_bits_to_f32(raw.y & 0xFFFFu), bf16_bits_to_f32(raw.y >> 16)};
    if (!active) x[0] = x[1] = x[2] = x[3] = 0.f;
    if (kRotateK && kv == 0) hadamard_warp(x, d_h, hc);
    const int nf = group_or(!(isfinite(x[0]) && isfinite(x[1]) && isfinite(x[2]) && isfinite(x[3])), 32);
    float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    uint32_t codes = 0, bsc = 0;
    float S = 0.f;
    if (!nf) {
      float scale;  // the divisor (NVFP4) or multiplier (MXFP4) of x
      bool zero;
      if (kFmt == kFp4Nv) {
        S = __fdiv_rn(group_max(am, 32), 2688.0f);
        const float six_s = __fmul_rn(6.0f, S);
        const float ab = group_max(am, 4);  // block of 16 channels = 4 lanes
        bsc = six_s > 0.f ? e4m3_code(__fdiv_rn(ab, six_s)) : 0u;
        scale = __fmul_rn(e4m3_value(bsc), S);
        zero = scale == 0.f;
      } else {
        const float ab = group_max(am, 8);  // block of 32 channels = 8 lanes
        const int E = ab > 0.f ? max(-127, min(127, ilog2f(ab) - 2)) : -127;
        bsc = (uint32_t)(E + 127);
        scale = pow2f(-E);
        zero = false;
      }
      if (!zero) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float y = kFmt == kFp4Nv ? __fdiv_rn(x[i], scale) : __fmul_rn(x[i], scale);
          codes |= e2m1_code(y) << (4 * i);
        }
      }
    }
    bad |= nf;
    if (active) {
      uint8_t* row = cache + ((((long long)page * L.h_kv + h) * 2 + kv) * 16 + p % 16) * rb;
      *reinterpret_cast<uint16_t*>(row + 2 * lane) = (uint16_t)codes;
      if (kFmt == kFp4Nv) {
        if ((lane & 3) == 0) row[d_h / 2 + lane / 4] = (uint8_t)bsc;
        if (lane == 0) *reinterpret_cast<float*>(row + d_h / 2 + 12) = S;
      } else if ((lane & 7) == 0) {
        row[d_h / 2 + lane / 8] = (uint8_t)bsc;
      }
    }
  }
  if (bad && lane == 0) set_status(status, KV4_STATUS_NONFINITE);
}

// Reconstruction into the bf16 comparator cache ([page][h_kv][K, V][16][d]):
// one warp per row, lane l producing channels 4l .. 4l + 3.
template <int kFmt>
__global__ void __launch_bounds__(256) fp4_to_bf16_kernel(Layout L, const uint8_t* __restrict__ cache,
                                                          uint16_t* __restrict__ out, long long rows) {
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int d_h = L.d_h;
  if (r >= rows || 4 * lane >= d_h) return;
  const uint8_t* row = cache + r * fp4_row_bytes(d_h);
  const uint32_t codes = *reinterpret_cast<const uint16_t*>(row + 2 * lane);
  float scale;
  if (kFmt == kFp4Nv) {
    const float S = *reinterpret_cast<const float*>(row + d_h / 2 + 12);
    scale = __fmul_rn(e4m3_value(row[d_h / 2 + lane / 4]), S);
  } else {
    scale = pow2f((int)row[d_h / 2 + lane / 8] - 127);
  }
  uint32_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) b[i] = f32_to_bf16_bits(__fmul_rn(e2m1_value((codes >> (4 * i)) & 15u), scale));
  *reinterpret_cast<uint2*>(out + r * d_h + 4 * lane) = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
}

cudaError_t launch_fp4_append(const Layout& L, int fmt, bool rotate_k, void* cache,
                              const uint16_t* k_new, const uint16_t* v_new,
                              const int32_t* tok_seq, const int32_t* tok_pos, int T,
                              const int32_t* seq_lens, const int32_t* block_table, int32_t* status,
                              cudaStream_t st) {
  const long long warps = (long long)T * L.h_kv;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  const float hc = hadamard_scale(L.d_h);
  uint8_t* c = (uint8_t*)cache;
#define KV4_FP4_LAUNCH(F, R)                                                                   \
  fp4_append_kernel<F, R><<<blocks, 256, 0, st>>>(L, c, k_new, v_new, tok_seq, tok_pos, T, seq_lens, \
                                                  block_table, status, hc)
  if (fmt == kFp4Nv) {
    if (rotate_k) KV4_FP4_LAUNCH(kFp4Nv, true);
    else KV4_FP4_LAUNCH(kFp4Nv, false);
  } else {
    if (rotate_k) KV4_FP4_LAUNCH(kFp4Mx, true);
    else KV4_FP4_LAUNCH(kFp4Mx, false);
  }
#undef KV4_FP4_LAUNCH
  return cudaGetLastError();
}

cudaError_t launch_fp4_to_bf16(const Layout& L, int fmt, const void* cache, void* out,
                               cudaStream_t st) {
  const long long rows = (long long)L.num_pages * L.h_kv * 2 * 16;
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  if (fmt == kFp4Nv)
    fp4_to_bf16_kernel<kFp4Nv><<<blocks, 256, 0, st>>>(L, (const uint8_t*)cache, (uint16_t*)out, rows);
  else
    fp4_to_bf16_kernel<kFp4Mx><<<blocks, 256, 0, st>>>(L, (const uint8_t*)cache, (uint16_t*)out, rows);
  return cudaGetLastError();
}

}  // namespace kv4
