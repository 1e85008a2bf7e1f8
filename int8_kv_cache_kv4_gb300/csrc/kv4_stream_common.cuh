// kv4_stream_common.cuh -- the unit stream shared by the work-balanced decode
// kernels (KV4-RL Sec. 5.3, App. A.3): per (sequence, kv head) pair, its
// protected INT8 units, then its INT4 units; segment walking, the protected
// slot test and the query conversion both kernels use.
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
// INT4 QK^T with the codes' exponent offset folded into the query side
// (1024 + c against q, 1024 + 16 c against q / 16, accumulators started at
// minus the constant part): exact-enough only while a group's constant part
// (1024 x the sum of its query values) stays small, i.e. for 32-channel
// groups; larger groups widen the codes to their exact values instead.
template <int NG>
__host__ __device__ constexpr bool fold_k_offset() { return NG >= 4; }
// One segment of the stream: region `type` (0 protected, 1 INT4) of pair (b, h).
struct Seg {
  long long start;  // stream index of its first unit
  long long cs;     // cost of the stream before it (see seg_cost)
  int b, h, type, len, n;
};

// Cost model of the stream for splitting it over CTAs: an INT4 unit counts 4,
// a protected unit 7, and the start of a segment 24 more (its share of the
// barriers, merge and query setup at a segment boundary).  Ratios measured on
// GB300 (per-CTA timelines of the work-balanced kernel).
constexpr int kCost4 = 4, kCost8 = 7, kCostSeg = 24;
__host__ __device__ inline long long seg_cost(int n, int type) {
  return n ? kCostSeg + (long long)n * (type == 0 ? kCost8 : kCost4) : 0;
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

// Next non-empty segment (b == B when the stream is exhausted).  Sequences of
// length 0 are skipped whole, one length load each.  A caller that needs no
// segment starting at or after stream position `stop` passes it: the walk then
// ends (b = B) as soon as the position reaches it, instead of crossing the
// empty sequences that may follow (idle slots of a batch).
__device__ inline void seg_next(Seg& s, const Layout& L, const int32_t* seq_lens, int B,
                                long long stop = 0x7fffffffffffffffLL) {
  s.start += s.n;
  s.cs += seg_cost(s.n, s.type);
  if (s.start >= stop) {
    s.b = B;
    return;
  }
  do {  // empty segments add nothing to start or cs
    if (s.type == 0) {
      s.type = 1;
      s.n = int4_units(s.len, L);
    } else {
      s.type = 0;
      if (++s.h == L.h_kv) {
        s.h = 0;
        do {
          ++s.b;
          s.len = s.b < B ? clamp_len(__ldg(seq_lens + s.b), L) : 0;
        } while (s.len == 0 && s.b < B);
      }
      s.n = prot_units(s.len, L);
    }
  } while (s.n == 0 && s.b < B);
}

// Atomic add with release semantics at GPU scope; returns the old value.
__device__ inline int atom_add_release_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.add.release.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// CTA holding stream unit u when U >= C units are split over C CTAs as
// [c*U/C, (c+1)*U/C) (every CTA then holds at least one unit); the
// stream kernel (decode_stream_kernel) cuts by cost instead.
__device__ inline int cta_of(long long u, long long U, int C) {
  return (int)(((u + 1) * C - 1) / U);
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

// A query element (bf16 bits) as fp16 bits, optionally divided by 16 (the
// same two roundings wherever the value is used).
__device__ inline uint32_t q16(uint32_t bf, bool sixteenth) {
  __half h = __float2half_rn(bf16_bits_to_f32(bf));
  if (sixteenth) h = __float2half_rn(__half2float(h) * 0.0625f);
  return __half_as_ushort(h);
}

// One pair's query in the forms the tensor-core units use (16-byte
// multiple, so that it can be bulk-copied).
struct __align__(16) QPrep {
  uint32_t qfrag4[8][32][4];  // INT4 path: block-diagonal query fragments per k-step and lane
  uint2 qfrag8[8][16];        // INT8 path: query fragments (a0, a2) of lanes 0..15
  float qsum[SD / 32][SG];    // per 32-channel block sums of the query
  float kc[4][SG];            // per (group, head): the constant part of the INT4 QK sums
};
static_assert(sizeof(QPrep) % 16 == 0, "QPrep is copied in 16-byte units");

// Everything the units of one pair need from its query (qr: G rows of D
// bf16), built by 128 threads (t = thread index): per-32-channel-block sums,
// both fragment sets, and per (group, head) the constant 1024-part of the
// INT4 QK sums.
template <int NG>
__device__ inline void build_qprep(const uint16_t* qr, QPrep& qp, int t) {
  constexpr int GS = SD / NG;
  {
    // warp j: head j, lane: channels 4 * lane .. + 3
    const int jj = t >> 5, ln = t & 31;
    const uint2 raw = reinterpret_cast<const uint2*>(qr)[t];
    const uint32_t b[4] = {raw.x & 0xFFFFu, raw.x >> 16, raw.y & 0xFFFFu, raw.y >> 16};
    float sq = 0.f, sa = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      sq += bf16_bits_to_f32(b[i]);
      sa += __half2float(__ushort_as_half((unsigned short)q16(b[i], i & 1)));
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
#pragma unroll
    for (int o = 1; o < GS / 4; o <<= 1) sa += __shfl_xor_sync(0xffffffffu, sa, o);
    if ((ln & 7) == 0) qp.qsum[ln >> 3][jj] = sq;
    if ((ln % (GS / 4)) == 0) qp.kc[ln / (GS / 4)][jj] = fold_k_offset<NG>() ? 1024.f * sa : 0.f;
  }
  // INT4 fragments: A rows (group, head), block diagonal; k-index order as the
  // widened K words produce it.  The B values are 1024 + c for even channels
  // (low nibbles) and 1024 + 16 c for odd ones (high nibbles, k-indices 8..15
  // of each step, A registers 2 and 3), so the odd channels' query values are
  // stored divided by 16 (exact in fp16 for |q| >= 2^-10).
  {
    // thread t (< 128) fills word k of lane ln at every k-step: row (group,
    // head) and the channel block are the same at every step
    const int ln = (t >> 2) & 31, k = t & 3;
    const int rr = ln >> 2, qq = ln & 3;
    const int row = rr + 8 * (k & 1);
    const int grp = row >> 2, jj = row & 3;
    // the step's channels 32 qq + [0, 32) lie in group (32 qq) / GS
    const bool in_group = grp < NG && (32 * qq) / GS == grp;
    const bool sixteenth = fold_k_offset<NG>() && (k & 2);
    const uint16_t* qrow = qr + jj * SD + 32 * qq + ((k & 2) ? 1 : 0);
#pragma unroll
    for (int s_ = 0; s_ < 8; ++s_) {
      const int off = 8 * (s_ >> 1) + 2 * (s_ & 1);  // channels off and off + 4 of the block
      uint32_t w = 0u;
      if (in_group)
        w = q16(qrow[off], sixteenth) | (q16(qrow[off + 4], sixteenth) << 16);
      qp.qfrag4[s_][ln][k] = w;
    }
  }
  // INT8 fragments: A rows = heads 0..3; k-step s, lane quad qd covers
  // channels 32*qd + 4*s + {0,1} (a0) and + {2,3} (a2)
  // (lanes 16..31, rows 4..7, read lane - 16's words: they duplicate heads
  // 0..3, whose results those lanes never publish)
  for (int idx = t; idx < 8 * 16; idx += 128) {
    const int s_ = idx >> 4, ln = idx & 15;
    const int rr = ln >> 2, qq = ln & 3;
    const uint16_t* src = qr + rr * SD + 32 * qq + 4 * s_;
    uint2 w;
    w.x = q16(src[0], false) | (q16(src[1], false) << 16);
    w.y = q16(src[2], false) | (q16(src[3], false) << 16);
    qp.qfrag8[s_][ln] = w;
  }
}

}  // namespace
}  // namespace kv4
