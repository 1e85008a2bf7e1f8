// kv4_stream_common.cuh -- the unit stream of the work-balanced decode kernel
// (KV4-RL Sec. 5.3, App. A.3): per (sequence, kv head) pair, its protected
// INT8 units, then its INT4 units; the cost model that cuts the stream over
// CTAs, segment walking, the protected slot test and the query conversion.
#pragma once
#include "kv4_common.cuh"

namespace kv4 {
namespace {

constexpr int SD = 128, SG = 4;     // head_dim, query heads per kv head
constexpr int kSPages = 2;          // 16-token INT4 pages per unit (and per stage)
constexpr int kProtUnit = 16;       // side-cache slots per protected unit
// Online softmax with a lazily moved reference: the running reference m
// (log2 domain) is raised only when a score exceeds it by more than this, so
// probabilities 2^(s - m) stay below 2^kLazyLog2 = 256 (fp16-safe in P')
// and the accumulators are rescaled on a few pages only.  The split's
// log-normaliser m + log2(l) is exact for any reference.
constexpr float kLazyLog2 = 8.f;
// One segment of the stream: the units of pair (b, h), its protected units
// first (np of them), then its INT4 units (n - np).
struct Seg {
  long long start;  // stream index of its first unit
  long long cs;     // cost of the stream before it (see seg_cost)
  int b, h, len, np, n;
};

// Cost model of the stream for splitting it over CTAs: an INT4 unit counts 4,
// a protected unit 7, and the start of a segment 24 more (its share of the
// barriers, merge and query setup at a segment boundary).  Ratios measured on
// GB300 (per-CTA timelines of the work-balanced kernel).
constexpr int kCost4 = 4, kCost8 = 7, kCostSeg = 24;
// cost of a pair with np protected and n4 INT4 units
__host__ __device__ inline long long seg_cost(int np, int n4) {
  return np + n4 ? kCostSeg + (long long)np * kCost8 + (long long)n4 * kCost4 : 0;
}
// stream cost of unit j of a segment from the segment's start: unit 0 is at
// 0 (the segment start is counted with its first unit), unit j > 0 at
// kCostSeg + the cost of units 0 .. j - 1
__device__ inline long long unit_cost_at(int j, int np) {
  if (j <= 0) return 0;
  return kCostSeg + (j <= np ? (long long)j * kCost8
                             : (long long)np * kCost8 + (long long)(j - np) * kCost4);
}
// the first unit j of a segment (np protected, n units) with
// unit_cost_at(j) >= x; n when there is none
__device__ inline int unit_at_within(long long x, int np, int n) {
  if (x <= 0) return 0;
  const long long y = x - kCostSeg;
  long long j;
  if (y <= (long long)np * kCost8) j = (y + kCost8 - 1) / kCost8;
  else j = np + (y - (long long)np * kCost8 + kCost4 - 1) / kCost4;
  return (int)min((long long)n, max(1LL, j));
}

__device__ inline int clamp_len(int len, const Layout& L) {
  return (len < 0 || len > L.max_pages * kPage) ? 0 : len;
}
// protected units of a sequence of length len: the sink slots alone while
// len <= S, else every side slot (the ring is masked to the window)
__device__ inline int prot_units(int len, const Layout& L) {
  if (len <= 0) return 0;
  const int ns = len <= L.S ? len : L.S + L.R;
  return (ns + kProtUnit - 1) / kProtUnit;
}
// INT4 pages of a sequence of length len (between the sinks and the window)
__device__ inline int int4_pages(int len, const Layout& L) {
  const Regions rg = regions(len, L.S, L.R);
  return rg.rec_start > rg.sink_end ? (rg.rec_start + kPage - 1) / kPage - rg.sink_end / kPage
                                    : 0;
}
__device__ inline int int4_units(int len, const Layout& L) {
  return (int4_pages(len, L) + kSPages - 1) / kSPages;
}
// the segment fields of sequence b's kv head h (start and cs are the caller's)
__device__ inline void seg_set(Seg& s, int b, int h, int len, const Layout& L) {
  s.b = b;
  s.h = h;
  s.len = len;
  s.np = prot_units(len, L);
  s.n = s.np + int4_units(len, L);
}

// Next non-empty segment (b == B when the stream is exhausted).  Sequences of
// length 0 are skipped whole, one length load each.  A caller that needs no
// segment starting at or after stream position `stop` passes it: the walk then
// ends (b = B) as soon as the position reaches it, instead of crossing the
// empty sequences that may follow (idle slots of a batch).
__device__ inline void seg_next(Seg& s, const Layout& L, const int32_t* seq_lens, int B,
                                long long stop = 0x7fffffffffffffffLL) {
  s.start += s.n;
  s.cs += seg_cost(s.np, s.n - s.np);
  if (s.start >= stop) {
    s.b = B;
    return;
  }
  // the next kv head of the same sequence has the same units; past the last
  // one, the next sequence that is not empty
  if (++s.h == L.h_kv) {
    int b = s.b, len = 0;
    do {
      ++b;
      len = b < B ? clamp_len(__ldg(seq_lens + b), L) : 0;
    } while (len == 0 && b < B);
    seg_set(s, b, 0, len, L);
  }
}

// Atomic add with release semantics at GPU scope; returns the old value.
__device__ inline int atom_add_release_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.add.release.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Is side slot sl part of the protected set of a sequence of length len?
// Sinks: sl < min(S, len).  Ring slot S + r: holds a position p of the final
// window [ws, len) with p = r (mod R).
__device__ inline bool slot_valid(int sl, int len, const Layout& L, int ws_mod, int n_rec) {
  if (sl < L.S) return sl < len;
  if (sl >= L.S + L.R) return false;
  int d = sl - L.S - ws_mod;
  if (d < 0) d += L.R;
  return d < n_rec;
}

// A query element (bf16 bits) as fp16 bits (the INT8 units' query operand).
__device__ inline uint32_t q16(uint32_t bf) {
  return __half_as_ushort(__float2half_rn(bf16_bits_to_f32(bf)));
}
// bf16 bits times 2^e (exact in fp32) as fp16 bits, rounded to nearest even.
__device__ inline uint32_t q16_scaled(uint32_t bf, float two_e) {
  return __half_as_ushort(__float2half_rn(bf16_bits_to_f32(bf) * two_e));
}

// One pair's query in the forms the tensor-core units use (16-byte
// multiple, so that it can be bulk-copied).
//
// INT4 units compute S = K_codes x Q^T with the tokens as MMA rows (A = the K
// codes of 16 tokens, entered as fp16 subnormals whose bit pattern is the
// code) and the query as B, one 32-channel block per pair of k-steps.  B's
// eight columns are (head j, parity p) = (n >> 1, n & 1): block b contributes
// to the columns of parity b & 1 only, so that one accumulator holds two
// blocks and every lane ends with the four blocks of one head.  Lane
// (r', q') (lane = 4 r' + q') of block b holds, for head j = r' >> 1 when
// b & 1 == r' & 1 (else zeros), the channels c0 = 32 b + 8 q':
//   lo k-step: (16 q~[c0], 16 q~[c0 + 4]), (16 q~[c0 + 2], 16 q~[c0 + 6])
//   hi k-step: (q~[c0 + 1], q~[c0 + 5]),   (q~[c0 + 3], q~[c0 + 7])
// matching the widened code words (low nibbles c 2^-24, high nibbles
// 16 c 2^-24), so every product is q~ c 2^-20.  q~ = q 2^e_j is the head's
// query scaled by a power of two that puts max |q~| in [2^10, 2^11): exact,
// inside fp16's normal range for all but negligible elements, and 16 q~ below
// fp16's largest value.  The score of token t for head j (log2 domain) is then
//   s = ks[j] * sum_b Delta_(t, group(b)) S_(t, j, b) + sum_g m_(t, g) qs[j][g]
// with ks[j] = scale_log2 2^20 2^-e_j and qs[j][g] = scale_log2 sum_(d in g) q_d
// (eq. 5.1 per group).  The offset part sum_g m qs is one more MMA per page:
// A = each token's offsets m_(t, g) at k = 2 g and 2 g + 1, B = qs[j][g]
// split into an fp16 head and tail (k = 2 g, 2 g + 1) in the parity-0
// columns, so that its products are exact and the tensor core sums them in
// fp32 (qm: lane (r', q') holds the (head, tail) of group q' of head r' >> 1
// when r' is even and q' < NG, else zeros).
struct __align__(16) QPrep {
  uint4 qb[4][32];            // INT4 path: B fragments [block][lane]: lo b0, lo b1, hi b0, hi b1
  uint2 qfrag8[8][16];        // INT8 path: query fragments (a0, a2) of lanes 0..15
  uint32_t qm[32];            // INT4 path: B fragment (b0) of the offset-term MMA, per lane
  float ks[SG];               // [head]: scale_log2 x 2^20 x 2^-e_head
};
static_assert(sizeof(QPrep) % 16 == 0, "QPrep is copied in 16-byte units");

// Everything the units of one pair need from its query (qr: G rows of D
// bf16), built by 128 threads (t = thread index; warp j builds head j's
// entries: its exponent, group sums and B fragments, then a share of the
// INT8 fragments).
template <int NG>
__device__ inline void build_qprep(const uint16_t* qr, QPrep& qp, int t, float scale_log2) {
  constexpr int GS = SD / NG;
  const int j = t >> 5, ln = t & 31;
  // lane ln of warp j: channels 4 ln .. 4 ln + 3 of head j
  const uint2 raw = reinterpret_cast<const uint2*>(qr + j * SD)[ln];
  const uint32_t b4[4] = {raw.x & 0xFFFFu, raw.x >> 16, raw.y & 0xFFFFu, raw.y >> 16};
  float mx = 0.f, sq = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float v = bf16_bits_to_f32(b4[i]);
    sq += v;
    mx = fmaxf(mx, fabsf(v));
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
  for (int o = 1; o < GS / 4; o <<= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  // e_j: max |q| 2^e in [2^10, 2^11); a zero or non-finite head keeps e = 0
  int e = 0;
  if (mx > 0.f && mx <= 3.0e38f) {
    const int ex = (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127;  // floor(log2 mx), normal mx
    e = min(40, max(-20, 10 - max(ex, -126)));
  }
  const float two_e = __int_as_float((127 + e) << 23);
  // lanes 8 j .. 8 j + 7 of the offset-term fragment: group q' of head j
  // (lane ln < 4 reads group ln's sum from lane ln * GS / 4)
  {
    const float qsg = scale_log2 * __shfl_sync(0xffffffffu, sq, (ln & 3) * (GS / 4));
    if (ln < 8) {
      uint32_t w = 0u;
      if (ln < 4 && ln < NG) {
        const __half hi = __float2half_rn(qsg);
        const __half lo = __float2half_rn(qsg - __half2float(hi));
        w = (uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16);
      }
      qp.qm[8 * j + ln] = w;
    }
  }
  if (ln == 0) qp.ks[j] = scale_log2 * __int_as_float((127 + 20 - e) << 23);
  {
    // thread ln of warp j: lane (r', q') = (2 j + (ln >> 4), (ln >> 2) & 3), block ln & 3
    const int rp = 2 * j + (ln >> 4), qp_ = (ln >> 2) & 3, blk = ln & 3;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if ((blk & 1) == (rp & 1)) {
      const uint16_t* c0 = qr + j * SD + 32 * blk + 8 * qp_;
      const float two_e4 = two_e * 16.f;
      w.x = q16_scaled(c0[0], two_e4) | (q16_scaled(c0[4], two_e4) << 16);
      w.y = q16_scaled(c0[2], two_e4) | (q16_scaled(c0[6], two_e4) << 16);
      w.z = q16_scaled(c0[1], two_e) | (q16_scaled(c0[5], two_e) << 16);
      w.w = q16_scaled(c0[3], two_e) | (q16_scaled(c0[7], two_e) << 16);
    }
    qp.qb[blk][4 * rp + qp_] = w;
  }
  // INT8 fragments: A rows = heads 0..3; k-step s, lane quad qd covers
  // channels 32*qd + 4*s + {0,1} (a0) and + {2,3} (a2)
  // (lanes 16..31, rows 4..7, read lane - 16's words: they duplicate heads
  // 0..3, whose results those lanes never publish)
  for (int idx = t; idx < 8 * 16; idx += 128) {
    const int s_ = idx >> 4, l2 = idx & 15;
    const int rr = l2 >> 2, qq = l2 & 3;
    const uint16_t* src = qr + rr * SD + 32 * qq + 4 * s_;
    uint2 w;
    w.x = q16(src[0]) | (q16(src[1]) << 16);
    w.y = q16(src[2]) | (q16(src[3]) << 16);
    qp.qfrag8[s_][l2] = w;
  }
}

}  // namespace
}  // namespace kv4
