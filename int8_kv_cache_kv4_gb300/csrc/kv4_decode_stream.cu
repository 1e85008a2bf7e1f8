// kv4_decode_stream.cu -- work-balanced persistent decode over the mixed
// INT4 / INT8 cache (KV4-RL Sec. 5.3 and eq. 5.1; App. A.3 "Protected path"
// and eq. A1), head_dim 128 with 4 query heads per kv head.
//
// Work is one stream of units over all (sequence, kv head) pairs.  For each
// pair, in order: its protected units (16 consecutive INT8 side-cache slots
// each, the sink slots and the recent-window ring), then one unit per two
// 16-token INT4 pages of the region between the sinks and the recent window.
// A pair's units form one segment of the stream.  The grid is sized to fill
// the GPU once, and the stream is cut into contiguous CTA shares of equal
// cost: an INT4 unit counts 4, a protected unit 7 and a segment start 24
// (seg_cost), the measured ratios of their times, so that CTAs whose share
// crosses many short segments take fewer units and all CTAs finish together.
//
// Inside a CTA the four warps take the units of the current segment
// round-robin; each warp streams its units through its own two-stage ring of
// bulk copies (the copy engine, one mbarrier per stage), issued ahead across
// segment boundaries.  A warp runs its protected units of the segment, then
// its INT4 units, carrying one online-softmax state across.  When a segment
// ends the warps' states are merged into one partial result (a locally
// normalised output and its log-normaliser) for the pair's four query heads.
// A pair held by one CTA is written out directly; otherwise each CTA adds its
// unit count to the pair's ticket after storing its partial, and the one that
// completes the count merges the partials (eq. A1) into the output.
// The CTA c holding units of pair p writes partial p + c: CTA ranges are
// contiguous, ordered and non-empty, so these indices are distinct and below
// pairs + C.
//
// Per-unit math on the tensor cores (m16n8k16, fp16 operands, fp32
// accumulation):
//  INT4 unit: the tokens as MMA rows -- the 4-bit K codes entered as fp16
//    subnormals (bit pattern = code) against the pair's query scaled by a
//    power of two per head, one 32-channel block per two k-steps; scores by
//    eq. 5.1 per group with the offset term as one more MMA; then the
//    transposed V codes (subnormals as well) against P' = p * Delta_v, plus
//    the offset term sum p m as one MMA whose rows are the V offsets.
//  INT8 unit: the query (rows = heads) against the 16 slots' K codes widened
//    exactly to fp16, scores scaled by each slot's K scale; then the
//    transposed V codes against P' = p * s_v.  Slots outside the protected
//    set (not yet written, or outside the final recent window) are masked.
#include <algorithm>
#include <type_traits>

#include "kv4_decode_common.cuh"
#include "kv4_mma.cuh"
#include "kv4_stream_common.cuh"

namespace kv4 {
namespace {

// warps per CTA of this kernel, and its threads
constexpr int kSW = 4;
constexpr int kST = kSW * 32;
// Copy stages per warp and CTAs per SM (build-time constants; the defaults
// are the measured best on GB300).
#ifndef KV4_STREAM_STAGES
#define KV4_STREAM_STAGES 2
#endif
#ifndef KV4_STREAM_CTAS_PER_SM
#define KV4_STREAM_CTAS_PER_SM 4
#endif
constexpr int kSStages = KV4_STREAM_STAGES;
constexpr int kStreamMinBlocks = KV4_STREAM_CTAS_PER_SM;
// The thread that keeps the segment bookkeeping and takes the completion
// tickets: lane 0 of the last warp, which the round-robin unit assignment
// never gives more units than the others.
constexpr int kTicketThread = (kSW - 1) * 32;

// Share weights by launch rank.  The grid holds kStreamMinBlocks CTAs per
// SM, placed in block order (CTA c is the (c / SMs)-th on its SM), and the
// warp schedulers favour the older CTAs of an SM: measured on GB300, the
// first CTA of an SM streams its share about 18% faster than the fourth.  The
// stream is therefore cut into shares proportional to these weights, so that
// an SM's CTAs finish together.
#ifndef KV4_STREAM_RANK_STEP
#define KV4_STREAM_RANK_STEP 6
#endif
constexpr int kRankW0 = 118, kRankStep = KV4_STREAM_RANK_STEP;  // weight of rank k: 118 - 6 k
__host__ __device__ constexpr int rank_w(int k) { return kRankW0 - kRankStep * k; }
static_assert(rank_w(kStreamMinBlocks - 1) > 0, "positive weights");
// CTAs per launch rank of a grid of C CTAs (C / kStreamMinBlocks, at least 1)
__device__ inline int rank_width(int C) { return max(1, C / kStreamMinBlocks); }
// summed weight of CTAs 0 .. c - 1 (S CTAs per rank; the last rank takes the rest)
__device__ inline long long share_weight(int c, int S) {
  long long f = 0;
#pragma unroll
  for (int k = 0; k < kStreamMinBlocks; ++k) {
    const int lo = k * S, hi = k == kStreamMinBlocks - 1 ? c : min(c, lo + S);
    if (hi > lo) f += (long long)rank_w(k) * (hi - lo);
  }
  return f;
}
// The stream of cost Wc cut over Cw CTAs: CTA c holds the units whose cost
// lies in [T(c), T(c + 1)), T(c) = ceil(Wc F(c) / F(Cw)) with F = share_weight.
struct Cut {
  long long Wc, Ft;  // stream cost, summed weight of all Cw CTAs
  int Cw, S;
  __device__ long long start(int c) const { return (Wc * share_weight(c, S) + Ft - 1) / Ft; }
  // the CTA holding stream cost x (0 <= x < Wc): the last c with
  // F(c) <= floor(x F(Cw) / Wc)
  __device__ int cta_of(long long x) const {
    const long long Y = (x * Ft) / Wc;
    long long f = 0;
#pragma unroll
    for (int k = 0; k < kStreamMinBlocks; ++k) {
      const int lo = k * S;
      if (lo >= Cw) break;
      const int hi = k == kStreamMinBlocks - 1 ? Cw : min(Cw, lo + S);
      const long long fk = (long long)rank_w(k) * (hi - lo);
      if (Y < f + fk) return min(Cw - 1, lo + (int)((Y - f) / rank_w(k)));
      f += fk;
    }
    return Cw - 1;
  }
};
// The cut of a stream of cost Wc over a grid of C CTAs: at most C shares, and
// few enough that every share is at least one unit's cost wide (no CTA is left
// without units): a share is at least Wc w_min / (w_max Cw) wide, and
// consecutive units start at most kCostSeg + kCost8 apart.
__device__ inline Cut stream_cut(long long Wc, int C) {
  Cut k;
  k.Wc = Wc;
  constexpr long long w_min = rank_w(kStreamMinBlocks - 1), w_max = rank_w(0);
  k.Cw = Wc > 0 ? (int)max(1LL, min((long long)C, Wc * w_min / ((kCostSeg + kCost8) * w_max))) : 0;
  k.S = rank_width(C);
  k.Ft = share_weight(k.Cw, k.S);
  return k;
}

// First unit whose stream cost (the cost of all units before it, a segment's
// start counted with its first unit) is at least T, for T inside the cost of
// sequences [b_lo, b_hi); pre_u / pre_c: units and cost before b_lo.
__device__ inline long long unit_at_cost(long long T, int b_lo, int b_hi, long long pre_u,
                                         long long pre_c, const Layout& L,
                                         const int32_t* __restrict__ seq_lens) {
  for (int b = b_lo; b < b_hi; ++b) {
    const int len = clamp_len(__ldg(seq_lens + b), L);
    const int np = prot_units(len, L), n = np + int4_units(len, L);
    const long long pc = seg_cost(np, n - np);  // one pair
    if (T < pre_c + (long long)L.h_kv * pc) {
      const long long h = (T - pre_c) / pc;
      // j = n: the next segment's first unit
      return pre_u + h * n + unit_at_within(T - pre_c - h * pc, np, n);
    }
    pre_c += (long long)L.h_kv * pc;
    pre_u += (long long)L.h_kv * n;
  }
  return pre_u;  // (not reached: T lies in these sequences)
}

// CTAs c0 .. c0 + n0 - 1 holding the units of a pair (np protected, n in
// all) whose first unit lies at stream cost pcs.
__device__ inline void pair_ctas(long long pcs, int np, int n, const Cut& k, int& c0, int& n0) {
  c0 = k.cta_of(pcs);
  n0 = k.cta_of(pcs + unit_cost_at(n - 1, np)) - c0 + 1;
}

// A pair whose partial results are to be merged, with where they are.
struct Pend {
  long long row0;  // first output row (sequence * h_q + kv head * G)
  long long pcs;   // stream cost before the pair's first unit
  int pair;        // sequence * h_kv + kv head
  int np, n;       // the pair's protected and total unit counts
  int mine;        // units of the pair this CTA holds
  int direct;      // this CTA holds all of them
  int valid;
  int c0, n0;      // (merging CTA) the CTAs holding the pair's partials
};

// Where one CTA of the decode grid starts: the first unit of its share and
// the segment holding it.
struct __align__(16) StreamStart {
  long long u_begin;
  Seg cs;
};
// The stream's cut over the decode grid, written by stream_prep_kernel and
// read once by every CTA of decode_stream_kernel at its start: CTA c's share
// ends where CTA c + 1's begins (start[C].u_begin = the stream's length).
struct __align__(16) StreamPlan {
  Cut cut;
  long long total;  // units in the stream
  StreamStart start[kMaxStreamCtas + 1];
};

struct __align__(16) StreamSmem {
  QPrep qp;                         // the current pair's query fragments and sums
  float mrg_o[kSW][SG][SD];         // per-warp unnormalised outputs at a segment end
  uint16_t qraw[SG * SD];           // next pair's query (bf16), bulk-copied ahead
  float mrg_m[kSW][SG];
  float mrg_l[kSW][SG];
  float mrg_mt[kSW][SG][SD / 32];
  Cut cut;                          // the stream's cut over the CTAs
  long long u_begin, u_end;         // this CTA's share of the stream
  Seg cs;                           // current segment of this CTA
  Seg prod[kSW];                    // producer cursors (segment of each warp's next unit)
  Seg nx;                           // segment after cs (ticket thread, at segment start)
  Pend pcur;                        // partial bookkeeping of segment cs (ticket thread)
  Pend pend;                        // partial whose ticket is in flight (ticket thread)
  Pend comb[2];                     // pair to merge at boundary k (slot k & 1)
  int go[2];                        // comb[k & 1] is valid
  int new_q;                        // a next segment follows (its query is being copied)
  uint64_t bar[kSW][kSStages];      // stage completion (one per warp and stage)
  uint64_t qbar;                    // completion of the qraw copy
};

// One thread: start the bulk copy of pair `row0`'s query (G rows of D bf16,
// 1 KB, 16-byte aligned) into sm.qraw; it completes on sm.qbar.
__device__ inline void stream_query_fetch(StreamSmem& sm, const uint16_t* __restrict__ q,
                                          long long row0) {
  mbar_arrive_expect_tx(&sm.qbar, SG * SD * 2);
  bulk_g2s(sm.qraw, q + row0 * SD, SG * SD * 2, &sm.qbar);
}

// Everything the units need from the query of the next pair, built from
// sm.qraw once its copy has completed.  No warp may still read the old values.
// q_rot != 0: the query is first rotated by the normalized Hadamard matrix of
// the keys (KV4-RL eq. 3.4; q_rot is the fp32 value nearest 1/sqrt(128)) and
// rounded to bf16, the same steps in the same order as kv4_hadamard_bf16, so
// that the result equals a decode of the separately rotated query.  Called
// by every thread of the CTA.
template <int NG>
__device__ __noinline__ void stream_query_setup(StreamSmem& sm, float scale_log2, float q_rot) {
  static_assert(kST == 32 * SG, "one warp per query head");
  if (q_rot != 0.f) {
    uint2* row = reinterpret_cast<uint2*>(sm.qraw + (threadIdx.x >> 5) * SD) + (threadIdx.x & 31);
    const uint2 raw = *row;
    float v[4] = {bf16_bits_to_f32(raw.x & 0xFFFFu), bf16_bits_to_f32(raw.x >> 16),
                  bf16_bits_to_f32(raw.y & 0xFFFFu), bf16_bits_to_f32(raw.y >> 16)};
    hadamard_warp(v, SD, q_rot);
    *row = make_uint2((uint32_t)f32_to_bf16_bits(v[0]) | ((uint32_t)f32_to_bf16_bits(v[1]) << 16),
                      (uint32_t)f32_to_bf16_bits(v[2]) | ((uint32_t)f32_to_bf16_bits(v[3]) << 16));
    __syncthreads();
  }
  build_qprep<NG>(sm.qraw, sm.qp, threadIdx.x, scale_log2);
}

// Merge the warps' states of one segment (after a barrier that follows every
// warp's publish).  Warp j < G merges query head j: the warps' weights
// 2^(m_w - M) / L are formed once, then each lane combines four channels.
// The result is stored as partial P, or, for a pair no other CTA holds
// (direct), as the pair's output rows row0 .. row0 + G - 1 and their
// log-normalisers.
__device__ inline void stream_merge_store(StreamSmem& sm, float* __restrict__ part_o,
                                          float* __restrict__ part_lse, long long P, bool direct,
                                          long long row0, uint16_t* __restrict__ out,
                                          float* __restrict__ out_lse) {
  const int j = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (j >= SG) return;
  const float mw = lane < kSW ? sm.mrg_m[lane][j] : -INFINITY;
  const float lw = lane < kSW ? sm.mrg_l[lane][j] : 0.f;
  float M = mw;
#pragma unroll
  for (int o = 1; o < kSW; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  M = __shfl_sync(0xffffffffu, M, 0);
  const float e = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
  float Lt = e * lw;
#pragma unroll
  for (int o = 1; o < kSW; o <<= 1) Lt += __shfl_xor_sync(0xffffffffu, Lt, o);
  Lt = __shfl_sync(0xffffffffu, Lt, 0);
  const bool empty = !(Lt > 0.f);
  const float f = empty ? 0.f : e * __frcp_rn(Lt);  // lanes 0 .. kSW-1: weight of warp `lane`
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 0; w < kSW; ++w) {
    const float fw = __shfl_sync(0xffffffffu, f, w);
    const float4 a = reinterpret_cast<const float4*>(&sm.mrg_o[w][j][0])[lane];
    const float mt = sm.mrg_mt[w][j][lane >> 3];  // channels 4*lane.. lie in block lane/8
    o.x = fmaf(fw, a.x + mt, o.x);
    o.y = fmaf(fw, a.y + mt, o.y);
    o.z = fmaf(fw, a.z + mt, o.z);
    o.w = fmaf(fw, a.w + mt, o.w);
  }
  const float lse2 = empty ? -INFINITY : M + log2f(Lt);  // log2 domain
  if (direct) {
    const long long row = row0 + j;
    uint16_t* po = out + row * SD + 4 * lane;  // the output need only be 2-byte aligned
    po[0] = f32_to_bf16_bits(o.x);
    po[1] = f32_to_bf16_bits(o.y);
    po[2] = f32_to_bf16_bits(o.z);
    po[3] = f32_to_bf16_bits(o.w);
    if (out_lse && lane == 0) out_lse[row] = lse2 * kLn2;
  } else {
    reinterpret_cast<float4*>(part_o + (P * SG + j) * SD)[lane] = o;
    if (lane == 0) part_lse[P * SG + j] = lse2 * kLn2;
  }
}

// Eq. A1, folded online: the partials P0 + k, k = k0, k0 + step, ... < n of
// query head j, this lane's four channels.  Each batch of kB partials' outputs
// and log-normalisers is requested at once (one round of L2 latency), then
// folded into the running maximum log-normaliser m, the sum l of e^(z - m) and
// the weighted output sum acc.  Empty partials (z = -inf) weigh nothing.
template <int kB>
__device__ inline void fold_partials(const float* __restrict__ part_o,
                                     const float* __restrict__ part_lse, long long P0, int n,
                                     int k0, int step, int j, int lane, float& m, float& l,
                                     float4& acc) {
  for (int kb = k0; kb < n; kb += kB * step) {
    float z[kB];
    float4 o[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int k = kb + u * step;
      const bool in = k < n;
      z[u] = in ? __ldcg(part_lse + (P0 + k) * SG + j) : -INFINITY;
      o[u] = in ? __ldcg(reinterpret_cast<const float4*>(part_o + ((P0 + k) * SG + j) * SD) + lane)
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mb = m;
#pragma unroll
    for (int u = 0; u < kB; ++u) mb = fmaxf(mb, z[u]);
    if (mb == -INFINITY) continue;
    const float sc = m == -INFINITY ? 0.f : exp2f((m - mb) * kLog2e);
    l *= sc;
    acc.x *= sc;
    acc.y *= sc;
    acc.z *= sc;
    acc.w *= sc;
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      if (z[u] != -INFINITY) {
        const float w = exp2f((z[u] - mb) * kLog2e);
        l += w;
        acc.x = fmaf(w, o[u].x, acc.x);
        acc.y = fmaf(w, o[u].y, acc.y);
        acc.z = fmaf(w, o[u].z, acc.z);
        acc.w = fmaf(w, o[u].w, acc.w);
      }
    }
    m = mb;
  }
}

// Eq. A1 over the n partials P0 .. P0 + n - 1 of one pair; warp j merges
// query head j.
__device__ inline void stream_combine(const float* __restrict__ part_o,
                                      const float* __restrict__ part_lse, long long P0, int n,
                                      long long row0, uint16_t* __restrict__ out,
                                      float* __restrict__ out_lse) {
  const int j = threadIdx.x >> 5, lane = threadIdx.x & 31;  // warp j < G: query head j
  if (j >= SG) return;
  float m = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  fold_partials<4>(part_o, part_lse, P0, n, 0, 1, j, lane, m, l, acc);
  const bool empty = !(l > 0.f);
  const float inv = empty ? 0.f : 1.f / l;
  const long long row = row0 + j;
  uint16_t* o = out + row * SD + 4 * lane;  // the output need only be 2-byte aligned
  o[0] = f32_to_bf16_bits(acc.x * inv);
  o[1] = f32_to_bf16_bits(acc.y * inv);
  o[2] = f32_to_bf16_bits(acc.z * inv);
  o[3] = f32_to_bf16_bits(acc.w * inv);
  if (out_lse && lane == 0) out_lse[row] = empty ? -INFINITY : m + logf(l);
}

// Ticket thread, at boundary k: did the ticket taken for partial sm.pend
// (old value t) bring the pair's count of finished units to its total?  Then
// this CTA merges the pair after the boundary: the CTAs holding its partials
// are worked out here, once per pair.  Slot k & 1 is read after the boundary's
// second barrier; it is written again two boundaries later, when every thread
// has passed the barriers in between.
__device__ inline void pend_take(StreamSmem& sm, int t, int k) {
  int go = 0;
  if (sm.pend.valid && t + sm.pend.mine == sm.pend.n) {
    __threadfence();  // acquire: the other CTAs' partials are visible
    Pend cm = sm.pend;
    pair_ctas(cm.pcs, cm.np, cm.n, sm.cut, cm.c0, cm.n0);
    sm.comb[k & 1] = cm;
    go = 1;
  }
  sm.go[k & 1] = go;
}

template <int NG>
__global__ void __launch_bounds__(kST, kStreamMinBlocks) decode_stream_kernel(
    Layout L, const uint8_t* __restrict__ paged, const uint8_t* __restrict__ side,
    const uint16_t* __restrict__ q, const int32_t* __restrict__ seq_lens, int B,
    const int32_t* __restrict__ block_table, float scale_log2, float* __restrict__ part_o,
    float* __restrict__ part_lse, int32_t* __restrict__ tickets, uint16_t* __restrict__ out,
    float* __restrict__ out_lse, int32_t* status, int defer, float q_rot,
    const StreamPlan* __restrict__ plan) {
  constexpr int D = SD;
  constexpr int GS = D / NG;  // channels per INT4 group
  constexpr int cb = 16 * D + 128 * NG;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  StreamSmem& sm = *reinterpret_cast<StreamSmem*>(smem_raw);
  uint8_t* stage_base = smem_raw + ((sizeof(StreamSmem) + 127) / 128) * 128;
  const int C = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ------------------------------------------------ this CTA's share (plan)
  if (lane == 0) {  // (made visible by the barrier below)
    for (int st = 0; st < kSStages; ++st) mbar_init(&sm.bar[warp][st], 1);
    if (warp == 0) mbar_init(&sm.qbar, 1);
    fence_mbar_init();
  }
  // The plan is written by stream_prep_kernel, launched just before this grid
  // (a programmatic dependent of it, this grid may start as it exits); the
  // wait also covers every kernel before it on the stream (the prep kernel
  // waited for them), so that the cache pages and tickets are ready.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) {
    const StreamStart s = plan->start[c];
    const long long u_end = plan->start[c + 1].u_begin;
    sm.cut = plan->cut;
    sm.u_begin = s.u_begin;
    sm.u_end = u_end;
    sm.cs = s.cs;
    sm.pend.valid = 0;
    // the first pair's query, fetched ahead of the page copies issued below
    // (the copy engine serves one SM's copies in order: behind them it would
    // arrive last)
    if (s.u_begin < u_end)
      stream_query_fetch(sm, q, (long long)s.cs.b * L.h_q + (long long)s.cs.h * SG);
  }
  __syncthreads();
  // Every CTA has read its plan entry: the next kernels on the stream may
  // launch (the next call's prep kernel rewrites the plan; an append waits for
  // this grid before it writes the cache).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long u_begin = sm.u_begin;
  // sequences with nothing to attend: zero output, log-normaliser -inf
  // (written at the end, off the path to the first page copies)
  auto zero_empty = [&]() {
    for (int b = c; b < B; b += C) {
      if (clamp_len(__ldg(seq_lens + b), L) != 0) continue;
      for (int idx = threadIdx.x; idx < L.h_q * D; idx += kST)
        out[(long long)b * L.h_q * D + idx] = 0;
      if (out_lse)
        for (int idx = threadIdx.x; idx < L.h_q; idx += kST)
          out_lse[(long long)b * L.h_q + idx] = -INFINITY;
    }
  };
  if (u_begin >= sm.u_end) {  // no units for this CTA
    zero_empty();
    return;
  }

  // ------------------------------------------------------ producer (lane 0)
  const int NS = L.S + L.R;
  const int NSP = side_scale_entries(L.S, L.R);
  const long long side_blk = side_block_bytes(D, L.S, L.R);
  constexpr int SB = kSPages * cb;  // stage bytes: two INT4 chunks or one 16-slot INT8 unit
  static_assert(2 * kProtUnit * SD + 4 * kProtUnit <= SB, "an INT8 unit fits a stage");
  uint8_t* my_stages = stage_base + (size_t)warp * kSStages * SB;
  // Producer: lane 0 of each warp.  A unit is one 1-D bulk copy
  // (cp.async.bulk, executed by the copy engine) per INT4 page, or four for a
  // protected unit, completing on the stage's mbarrier.  Its segment cursor
  // lives in shared memory and moves only when a segment is used up; what
  // each unit needs is kept in registers: the unit index in the segment and
  // its end, the segment's protected unit count, INT4 page count and
  // block-table row, the pair's column of the page pool and its side block,
  // and the next INT4 unit's pages, read one unit ahead so that the load's
  // latency is not waited for at the issue.  vbits (lane 0) records which
  // pages of each stage were copied; the consumers read it with a shuffle.
  int p_more = 0, p_j = 0, p_hi = 0, p_np = 0, p_np4 = 0, p_ns = 0, p_hcb = 0;
  const int32_t* p_bt = block_table;
  const uint8_t* p_src8 = side;
  int pphys = -1, pphys1 = -1;  // the INT4 unit's two pages (-2: no second page)
  uint32_t vbits = 0;           // bit 2 st + p: page p of stage st was copied
  const uint32_t stages_s = smem_u32(my_stages), bars_s = smem_u32(&sm.bar[warp][0]);
  // pages of INT4 unit p_j - p_np
  auto prod_pages = [&]() {
    const int j2 = kSPages * (p_j - p_np);
    pphys = __ldg(p_bt + j2);
    pphys1 = j2 + 1 < p_np4 ? __ldg(p_bt + j2 + 1) : -2;
  };
  // slow path: (cursor, p_j) may lie past its segment's end; move over
  // segments until it names a unit of this warp
  auto prod_next = [&]() {
    Seg& s_ = sm.prod[warp];
    const long long ub = sm.u_begin, ue = sm.u_end;
    while (true) {
      if (s_.b >= B || s_.start >= ue) {
        p_more = 0;
        return;
      }
      p_hi = (int)(min(ue, s_.start + s_.n) - s_.start);
      if (p_j < p_hi) break;
      seg_next(s_, L, seq_lens, B, ue);
      p_j = (int)(max(ub, s_.start) - s_.start) + warp;
    }
    p_more = 1;
    p_np = s_.np;
    p_bt = block_table + (long long)s_.b * L.max_pages + min(s_.len, L.S) / kPage;
    p_np4 = int4_pages(s_.len, L);
    p_ns = s_.len <= L.S ? s_.len : NS;
    p_hcb = s_.h * cb;
    p_src8 = side + ((long long)s_.b * L.h_kv + s_.h) * side_blk;
    if (p_j >= p_np) prod_pages();
  };
  auto issue = [&](int st) {
    const uint32_t bar = bars_s + 8u * st;
    const uint32_t dst = stages_s + (uint32_t)(st * SB);
    if (p_j >= p_np) {
      // INT4 pages 2 j and 2 j + 1 of the region (the second may not exist:
      // -2); a page id outside the pool is not copied and its slots are masked
      const bool good0 = (unsigned)pphys < (unsigned)L.num_pages;
      const bool good1 = (unsigned)pphys1 < (unsigned)L.num_pages;
      if (!good0 || (pphys1 != -2 && !good1)) set_status(status, KV4_STATUS_BAD_PAGE);
      vbits = (vbits & ~(3u << (2 * st))) | ((good0 ? 1u : 0u) << (2 * st)) |
              ((good1 ? 1u : 0u) << (2 * st + 1));
      const long long page_stride = (long long)L.h_kv * cb;  // bytes between pages of one head
      const uint8_t* src = paged + p_hcb;
      mbar_arrive_expect_tx_s(bar, (good0 ? (uint32_t)cb : 0u) + (good1 ? (uint32_t)cb : 0u));
      if (good0) bulk_g2s_s(dst, src + pphys * page_stride, (uint32_t)cb, bar);
      if (good1) bulk_g2s_s(dst + cb, src + pphys1 * page_stride, (uint32_t)cb, bar);
    } else {
      const int slot0 = p_j * kProtUnit;
      const uint32_t rows = (uint32_t)min(kProtUnit, p_ns - slot0);
      vbits |= 3u << (2 * st);  // (a protected unit is always copied)
      // scales of the 8-slot runs that hold copied rows (within the NSP padding)
      const uint32_t sbytes = 16u * ((rows + 7) / 8);
      mbar_arrive_expect_tx_s(bar, 2u * rows * D + 2u * sbytes);
      bulk_g2s_s(dst, p_src8 + (long long)slot0 * D, rows * D, bar);
      bulk_g2s_s(dst + kProtUnit * D, p_src8 + (long long)(NS + slot0) * D, rows * D, bar);
      bulk_g2s_s(dst + 2 * kProtUnit * D, p_src8 + 2LL * NS * D + 2 * slot0, sbytes, bar);
      bulk_g2s_s(dst + 2 * kProtUnit * D + 2 * kProtUnit,
                 p_src8 + 2LL * NS * D + 2LL * NSP + 2 * slot0, sbytes, bar);
    }
  };
  if (lane == 0) {  // the warp's first units into its stages
    sm.prod[warp] = sm.cs;
    p_j = (int)(max(u_begin, sm.cs.start) - sm.cs.start) + warp;
    prod_next();
    for (int st = 0; st < kSStages && p_more; ++st) {
      issue(st);
      p_j += kSW;
      if (p_j < p_hi) {
        if (p_j >= p_np) prod_pages();
      } else {
        prod_next();
      }
    }
  }
  // After the warp consumed the unit in stage st: the next unit into it.
  auto refill = [&](int st) {
    __syncwarp();  // every lane is past its reads of stage st
    if (lane == 0 && p_more) {
      issue(st);
      p_j += kSW;
      if (p_j < p_hi) {  // fast path: next unit of the same segment
        if (p_j >= p_np) prod_pages();
      } else {
        prod_next();
      }
    }
  };
  uint32_t phase = 0;  // bit st: parity of stage st's next completion
  // Wait for the unit in stage st (bounded: a wait that expires sets
  // KV4_STATUS_TIMEOUT and the unit is treated as not copied).  Returns which
  // of its pages were copied (bits 0, 1; a protected unit reads 3).
  auto stage_wait = [&](int st) -> uint32_t {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.bar[warp][st], (phase >> st) & 1u));
    phase ^= 1u << st;
    if (!ok && lane == 0) set_status(status, KV4_STATUS_TIMEOUT);
    const uint32_t pv = __shfl_sync(0xffffffffu, vbits >> (2 * st), 0) & 3u;
    return ok ? pv : 0u;
  };

  // ------------------------------------------------------ per-lane constants
  const int r = lane >> 2, qd = lane & 3;
  const uint32_t p_keep = (r < 4) ? 0xFFFFFFFFu : 0u;  // INT8 path: lanes of heads 0..3
  // INT4 V ldmatrix rows: matrix lane/8 = tokens (mi&1)*8.., piece mi>>1 (+2)
  const int lm_tok = ((lane >> 3) & 1) * 8 + (lane & 7);
  const int lm_p = lane >> 4;
  const uint32_t lm_off0 = lm_tok * 64 + 16 * ((lm_p) ^ ((lm_tok >> 1) & 3));
  const uint32_t lm_off1 = lm_tok * 64 + 16 * ((lm_p + 2) ^ ((lm_tok >> 1) & 3));
  // INT8 V ldmatrix rows: matrix lane/8 = (slots 0-7 | 8-15) x (piece, piece + 1),
  // row lane & 7; pieces are swizzled by slot
  const int l8_t = lane & 7, l8_row = ((lane >> 3) & 1) * 8 + l8_t, l8_pp = lane >> 4;
  constexpr int TK8[4] = {0, 1, 8, 9};  // INT8 unit: this lane's slots 2 * qd + TK8[e]

  int it = 0;  // stage of this warp's next unit (0 .. kSStages - 1)
  int pend_t = 0;  // ticket thread: ticket value returned for the pending partial
  int nb = 0;               // segment boundaries passed
  uint32_t qphase = 0;  // completed copies into sm.qraw
  if (!mbar_wait(&sm.qbar, qphase & 1) && threadIdx.x == 0) set_status(status, KV4_STATUS_TIMEOUT);
  ++qphase;
  stream_query_setup<NG>(sm, scale_log2, q_rot);
  __syncthreads();
  // The current segment lives in sm.cs (advanced by the ticket thread between
  // the boundary barriers); the loop below keeps only what the units need.
  while (true) {
    const Seg cs = sm.cs;
    if (cs.b >= B || cs.start >= sm.u_end) break;
    if (threadIdx.x == kTicketThread) {
      // the next segment (its pair's query is read ahead: the previous copy
      // was consumed before the last barrier), and this segment's partial
      // bookkeeping -- none of it is waited for by a barrier
      Seg nx = cs;
      seg_next(nx, L, seq_lens, B, sm.u_end);
      const bool new_q = nx.b < B && nx.start < sm.u_end;
      sm.new_q = new_q;
      if (new_q) stream_query_fetch(sm, q, (long long)nx.b * L.h_q + (long long)nx.h * SG);
      sm.nx = nx;
      Pend pd;
      pd.row0 = (long long)cs.b * L.h_q + (long long)cs.h * SG;
      pd.pcs = cs.cs;
      pd.pair = cs.b * L.h_kv + cs.h;
      pd.np = cs.np;
      pd.n = cs.n;
      pd.mine = (int)(min(sm.u_end, cs.start + cs.n) - max(sm.u_begin, cs.start));
      pd.direct = pd.mine == cs.n;
      pd.valid = 1;
      sm.pcur = pd;
    }
    const int lo = (int)(max(sm.u_begin, cs.start) - cs.start);
    const int hi = (int)(min(sm.u_end, cs.start + cs.n) - cs.start);
    const Regions rg = regions(cs.len, L.S, L.R);
    const int np = cs.np;
    // this warp's units of the segment: jj = lo + warp, lo + warp + kSW, ...;
    // the protected ones (jj < np) first
    int jj = lo + warp;
    const int e8 = min(hi, np);
    const bool have8 = jj < e8;
    if (have8) {
      // ================================= INT8 protected units (App. A.3)
      // Per unit of 16 side slots: QK^T with the query rows (heads) against
      // the slots' codes widened exactly to fp16 (two 8-slot tiles), scores
      // scaled by each slot's K scale; then PV with the transposed codes
      // against P' = p * s_v.  Slots outside the protected set are masked.
      const int n_rec = cs.len > L.S ? cs.len - rg.rec_start : 0;
      const int ws_mod = L.R > 0 ? rg.rec_start % L.R : 0;
      float m8 = -INFINITY, l8 = 0.f;
      float acc8[8][4];
#pragma unroll
      for (int P = 0; P < 8; ++P)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc8[P][i] = 0.f;
      const uint2* q8 = &sm.qp.qfrag8[0][lane & 15];  // + 16 * s
      for (; jj < e8; jj += kSW, it = it + 1 == kSStages ? 0 : it + 1) {
        const int st = it;
        const bool ok = stage_wait(st) != 0u;
        const uint32_t stg = smem_u32(my_stages) + st * SB;
        if (ok) {
          const int sl0 = jj * kProtUnit + 2 * qd;  // this lane's slots sl0 + {0, 1, 8, 9}
          // a sequence of at least S + R tokens fills every sink and ring slot:
          // only a unit reaching into the padding past NS needs the test
          const bool all_in = cs.len >= NS && (jj + 1) * kProtUnit <= NS;
          bool okv[4] = {true, true, true, true};
          if (!all_in) {
#pragma unroll
            for (int e = 0; e < 4; ++e) okv[e] = slot_valid(sl0 + TK8[e], cs.len, L, ws_mod, n_rec);
          }
          // ---- QK: B = K codes of slot r (tile 0) and slot r + 8 (tile 1),
          // channels 32*qd + [0, 32); pieces are swizzled by slot (r + 8 & 7 = r)
          const uint4 kA0 = lds128(stg + r * D + 16 * ((2 * qd) ^ r));
          const uint4 kB0 = lds128(stg + r * D + 16 * ((2 * qd + 1) ^ r));
          const uint4 kA1 = lds128(stg + (r + 8) * D + 16 * ((2 * qd) ^ r));
          const uint4 kB1 = lds128(stg + (r + 8) * D + 16 * ((2 * qd + 1) ^ r));
          float dq0[4] = {0.f, 0.f, 0.f, 0.f}, dq1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int s_ = 0; s_ < 8; ++s_) {
            const uint32_t x0 = (s_ < 4 ? u4word(kA0, s_) : u4word(kB0, s_ - 4)) ^ 0x80808080u;
            const uint32_t x1 = (s_ < 4 ? u4word(kA1, s_) : u4word(kB1, s_ - 4)) ^ 0x80808080u;
            const uint2 qa = q8[16 * s_];
            mma_f16(dq0, qa.x, 0u, qa.y, 0u, i8pair(x0, 0x4140u), i8pair(x0, 0x4342u));
            mma_f16(dq1, qa.x, 0u, qa.y, 0u, i8pair(x1, 0x4140u), i8pair(x1, 0x4342u));
          }
          // scores of head r & 3 for the four slots
          const float2 ksA = h2f2(lds32(stg + 2 * kProtUnit * D + 4 * qd));
          const float2 ksB = h2f2(lds32(stg + 2 * kProtUnit * D + 16 + 4 * qd));
          float sv[4] = {dq0[0] * ksA.x, dq0[1] * ksA.y, dq1[0] * ksB.x, dq1[1] * ksB.y};
#pragma unroll
          for (int e = 0; e < 4; ++e) sv[e] = okv[e] ? sv[e] * scale_log2 : -INFINITY;
          float tmax = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
          tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
          if (__any_sync(0xffffffffu, tmax > m8 + kLazyLog2)) {  // lazy rescaling, as above
            const float mnew = fmaxf(m8, tmax);
            const float alpha = mnew == -INFINITY ? 1.f : ex2(m8 - mnew);
            const float aA = __shfl_sync(0xffffffffu, alpha, 4 * ((2 * qd) & 3));
            const float aB = __shfl_sync(0xffffffffu, alpha, 4 * ((2 * qd + 1) & 3));
#pragma unroll
            for (int P = 0; P < 8; ++P) {
              acc8[P][0] *= aA;
              acc8[P][1] *= aB;
              acc8[P][2] *= aA;
              acc8[P][3] *= aB;
            }
            l8 *= alpha;
            m8 = mnew;
          }
          const float mref = m8 == -INFINITY ? 0.f : m8;
          float pv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) pv[e] = ex2(sv[e] - mref);
          l8 += (pv[0] + pv[1]) + (pv[2] + pv[3]);
          // ---- PV: A = V codes transposed (rows = channels, k = 16 slots), B = p * s_v
          uint32_t vsA = lds32(stg + 2 * kProtUnit * D + 2 * kProtUnit + 4 * qd);
          uint32_t vsB = lds32(stg + 2 * kProtUnit * D + 2 * kProtUnit + 16 + 4 * qd);
          vsA &= (okv[0] ? 0x0000FFFFu : 0u) | (okv[1] ? 0xFFFF0000u : 0u);
          vsB &= (okv[2] ? 0x0000FFFFu : 0u) | (okv[3] ? 0xFFFF0000u : 0u);
          const uint32_t pb0 = hmul2(pack_f16(pv[0], pv[1]) & p_keep, vsA);
          const uint32_t pb1 = hmul2(pack_f16(pv[2], pv[3]) & p_keep, vsB);
          const uint32_t vbase = stg + kProtUnit * D;
#pragma unroll
          for (int c2 = 0; c2 < 4; ++c2) {  // pieces 2 c2 and 2 c2 + 1
            uint32_t vr[4];  // (slots 0-7, piece), (slots 8-15, piece), same for piece + 1
            ldsm_x4_trans(vr, vbase + l8_row * D + 16 * ((2 * c2 + l8_pp) ^ l8_t));
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const uint32_t xlo = vr[2 * h2] ^ 0x80808080u, xhi = vr[2 * h2 + 1] ^ 0x80808080u;
              // rows r / r+8 = channels 16P + 2r / 16P + 2r + 1; k = slots 2qd,
              // 2qd+1 (a0, a1) and 2qd+8, 2qd+9 (a2, a3)
              mma_f16(acc8[2 * c2 + h2], i8pair(xlo, 0x4240u), i8pair(xlo, 0x4341u),
                      i8pair(xhi, 0x4240u), i8pair(xhi, 0x4341u), pb0, pb1);
            }
          }
        }
        refill(st);
      }
      // publish this warp's state (it is read back below if INT4 units follow)
      float lsum = (r < 4) ? l8 : 0.f;
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
      if (qd == 0 && r < 4) {
        sm.mrg_m[warp][r] = m8;
        sm.mrg_l[warp][r] = lsum;
      }
      if (lane < SG * (D / 32)) sm.mrg_mt[warp][lane / (D / 32)][lane % (D / 32)] = 0.f;
      if (qd < 2) {
        const int hA = 2 * qd, hB = 2 * qd + 1;
#pragma unroll
        for (int P = 0; P < 8; ++P) {
          const int dd = 16 * P + 2 * r;
          sm.mrg_o[warp][hA][dd] = acc8[P][0];
          sm.mrg_o[warp][hB][dd] = acc8[P][1];
          sm.mrg_o[warp][hA][dd + 1] = acc8[P][2];
          sm.mrg_o[warp][hB][dd + 1] = acc8[P][3];
        }
      }
    }
    if (jj < hi || !have8) {
      // ============================================= INT4 pages (eq. 5.1)
      // Per unit of two pages.  QK^T with the tokens as MMA rows: A = the K
      // codes of the page's 16 tokens entered as fp16 subnormals (bit
      // pattern = code: one logic op per pair of values), B = the scaled
      // query fragments of the pair (in registers for the whole segment),
      // one 32-channel block per two k-steps; accumulator set A holds blocks
      // 0 and 1, set B blocks 2 and 3, so each lane ends with the four
      // per-block sums of tokens r and r + 8 for head q.  Scores by eq. 5.1
      // per group, one online-softmax step for both pages.  The probabilities
      // are moved into the PV operand layout by two shuffles per page; per
      // page PV against the transposed V codes (subnormals as well) with
      // P' = p * Delta_v, and the offset term sum_t p_t m_t of every group as
      // one more MMA whose A rows are the page's V offsets.  Units inside the
      // region with both pages copied (all but its first and last) skip every
      // mask.  A warp without units here publishes an empty state.
      uint4 qbf[4];  // this lane's B fragments of the four blocks (lo b0, lo b1, hi b0, hi b1)
#pragma unroll
      for (int bl = 0; bl < 4; ++bl) qbf[bl] = sm.qp.qb[bl][lane];
      const uint32_t qmf = sm.qp.qm[lane];  // offset-term B fragment
      const float ksc = sm.qp.ks[qd];
      const int first_page = rg.sink_end / kPage;
      const int len = cs.len;
      const int n4 = cs.n - np;
      float m_run = -INFINITY, l_run = 0.f, m_thr = -INFINITY;  // m_thr = m_run + kLazyLog2
      float mtacc[4] = {0.f, 0.f, 0.f, 0.f};  // rows = groups (V offsets), columns = heads
      float acc[4][2][4];
#pragma unroll
      for (int G_ = 0; G_ < 4; ++G_)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[G_][hh][i] = 0.f;
      if (have8) {
        // carry the state of this warp's protected units over, from the
        // publish above: the reference and sum of head q (the sum in the
        // row-0 lanes, which the publish below adds up), and the outputs in
        // this layout (even channels carry 2^-24, odd ones 2^-20)
        __syncwarp();
        m_run = sm.mrg_m[warp][qd];
        m_thr = m_run + kLazyLog2;
        if (r == 0) l_run = sm.mrg_l[warp][qd];
        if (qd < 2) {
#pragma unroll
          for (int P = 0; P < 4; ++P)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int dd = 32 * P + 4 * r + 2 * hh;
              acc[P][hh][0] = sm.mrg_o[warp][2 * qd][dd] * 0x1p-24f;
              acc[P][hh][1] = sm.mrg_o[warp][2 * qd + 1][dd] * 0x1p-24f;
              acc[P][hh][2] = sm.mrg_o[warp][2 * qd][dd + 1] * 0x1p-20f;
              acc[P][hh][3] = sm.mrg_o[warp][2 * qd + 1][dd + 1] * 0x1p-20f;
            }
        }
        __syncwarp();  // every lane has read before the publish below rewrites
      }
      const int mrow = r < NG ? r : 0;  // offset-term MMA: this lane's A row group
      // lane offsets inside a page chunk: K codes (row r, quarter q: one word
      // per block), K meta of row r, this lane's quad of V Deltas (all
      // groups) and of V offsets (group mrow)
      const uint32_t kq_off = r * 64 + 16 * qd;
      const uint32_t km_off = meta_off_k(D) + r * NG * 4;
      const uint32_t vd_off = meta_off_v(D, GS) + qd * NG * 8;
      const uint32_t vm_off = meta_off_v(D, GS) + 32 * NG + (qd * NG + mrow) * 8;
      const uint32_t vc_off = codes_off_v(D);
      // probabilities of tokens (r, r + 8) for head q, moved to the PV B
      // layout (tokens 2 q' + {0, 1} and 2 q' + {8, 9} of head r'): the lanes
      // holding tokens 2 q' and 2 q' + 1 for head r' (any value for r' > 3)
      const int src_a = (8 * qd + r) & 31, src_b = (8 * qd + 4 + r) & 31;

      for (; jj < hi; jj += kSW) {
        const int j4 = jj - np;  // INT4 unit of the region
        const int ST = it;
        const uint32_t sb = stages_s + (uint32_t)(ST * SB);
        const uint32_t pv = stage_wait(ST);  // pages copied
        const bool clean = (unsigned)(j4 - 1) < (unsigned)(n4 - 2) && pv == 3u;
        const int pg0 = first_page + kSPages * j4;
        // ---------------- S = K codes x Q^T and scores (eq. 5.1 per group),
        // log2 domain, relative to the running reference
        const float mref = m_run == -INFINITY ? 0.f : m_run;
        float sc[2][2];  // [page][token r | r + 8]
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const uint32_t pb = sb + pp * cb;
          const uint4 w0 = lds128(pb + kq_off), w1 = lds128(pb + kq_off + 512);
          float sA[4] = {0.f, 0.f, 0.f, 0.f}, sB[4] = {0.f, 0.f, 0.f, 0.f};
          // offset part sum_g m_(t, g) qs_g of tokens r and r + 8 (columns of parity 0)
          float sM[4] = {0.f, 0.f, 0.f, 0.f};
          {
            const uint32_t m0 = qd < NG ? lds32(pb + km_off + 4 * qd) : 0u;
            const uint32_t m1 = qd < NG ? lds32(pb + km_off + 8 * NG * 4 + 4 * qd) : 0u;
            mma_f16(sM, __byte_perm(m0, 0u, 0x3232), __byte_perm(m1, 0u, 0x3232), 0u, 0u, qmf, 0u);
          }
#pragma unroll
          for (int bl = 0; bl < 4; ++bl) {
            uint32_t x0[4], x1[4];
            widen_v_sub(u4word(w0, bl), x0);
            widen_v_sub(u4word(w1, bl), x1);
            float* d = bl < 2 ? sA : sB;
            mma_f16(d, x0[0], x1[0], x0[2], x1[2], qbf[bl].x, qbf[bl].y);
            mma_f16(d, x0[1], x1[1], x0[3], x1[3], qbf[bl].z, qbf[bl].w);
          }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            MetaRow<NG> km;
            km.load_s(pb + km_off + e * 8 * NG * 4);
            // block sums of this token: blocks 0, 1 in set A, 2, 3 in set B
            const float s0 = sA[2 * e], s1 = sA[2 * e + 1];
            const float s2 = sB[2 * e], s3 = sB[2 * e + 1];
            float dsum;
            if (NG == 4) {
              dsum = fmaf(lo_f(km.get(3)), s3, fmaf(lo_f(km.get(2)), s2,
                          fmaf(lo_f(km.get(1)), s1, lo_f(km.get(0)) * s0)));
            } else if (NG == 2) {
              dsum = fmaf(lo_f(km.get(1)), s2 + s3, lo_f(km.get(0)) * (s0 + s1));
            } else {
              dsum = lo_f(km.get(0)) * ((s0 + s1) + (s2 + s3));
            }
            sc[pp][e] = fmaf(ksc, dsum, sM[2 * e] - mref);
          }
        }
        if (!clean) {
          // first / last unit of the segment, or a page not copied: mask the
          // scores outside the INT4 region, and zero the V metadata of slots
          // that hold no data of this sequence (a page not copied, or slots
          // at or past the length: their bytes may be anything), so that
          // their P' = p Delta and offset p m are exactly zero in the PV
          // products below, which then need no mask
#pragma unroll
          for (int pp = 0; pp < 2; ++pp)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int pos = (pg0 + pp) * kPage + r + 8 * e;
              const bool in = ((pv >> pp) & 1u) && pos >= rg.sink_end && pos < rg.rec_start;
              if (!in) sc[pp][e] = -INFINITY;
            }
          if (lane < 2 * kPage) {
            const int pp = lane >> 4, t = lane & 15;
            if (!((pv >> pp) & 1u) || (pg0 + pp) * kPage + t >= len) {
              const uint32_t ch = sb + pp * cb;  // (volatile stores: kept before the loads below)
#pragma unroll
              for (int gg = 0; gg < NG; ++gg) {
                sts16(ch + v_delta_byte(t, gg, D, GS), 0u);
                sts16(ch + v_offset_byte(t, gg, D, GS), 0u);
              }
            }
          }
          __syncwarp();
        }
        // ---------------- online softmax for head q over both pages.  Lazy
        // rescaling: the reference m_run moves only when a score exceeds it
        // by more than kLazyLog2 (p then stays below 2^kLazyLog2).
        const float tmax = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1])) + mref;
        if (__any_sync(0xffffffffu, tmax > m_thr)) {
          float hm = tmax;  // the head's maximum over the warp's 32 tokens
          hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 4));
          hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 8));
          hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 16));
          const float mnew = fmaxf(m_run, hm);
          const float alpha = mnew == -INFINITY ? 1.f : ex2(m_run - mnew);
          // PV accumulators of this lane: heads 2 q and 2 q + 1 (columns)
          const float aA = __shfl_sync(0xffffffffu, alpha, (2 * qd) & 3);
          const float aB = __shfl_sync(0xffffffffu, alpha, (2 * qd + 1) & 3);
#pragma unroll
          for (int G_ = 0; G_ < 4; ++G_)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              acc[G_][hh][0] *= aA;
              acc[G_][hh][1] *= aB;
              acc[G_][hh][2] *= aA;
              acc[G_][hh][3] *= aB;
            }
          mtacc[0] *= aA;
          mtacc[1] *= aB;
          l_run *= alpha;
          const float shift = mnew == -INFINITY ? 0.f : mnew - mref;  // new reference vs old
#pragma unroll
          for (int pp = 0; pp < 2; ++pp)
#pragma unroll
            for (int e = 0; e < 2; ++e) sc[pp][e] -= shift;
          m_run = mnew;
          m_thr = mnew + kLazyLog2;
        }
        float pr_[2][2];
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
#pragma unroll
          for (int e = 0; e < 2; ++e) pr_[pp][e] = ex2(sc[pp][e]);  // masked: 0
        l_run += (pr_[0][0] + pr_[0][1]) + (pr_[1][0] + pr_[1][1]);
        // ---------------- PV, one page at a time
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const uint32_t pb = sb + pp * cb;
          // p of tokens 2 q + {0, 1} (b0) and 2 q + {8, 9} (b1), head r
          const uint32_t ph = pack_f16(pr_[pp][0], pr_[pp][1]);
          const uint32_t hA = __shfl_sync(0xffffffffu, ph, src_a);
          const uint32_t hB = __shfl_sync(0xffffffffu, ph, src_b);
          const uint32_t p01 = __byte_perm(hA, hB, 0x5410);
          const uint32_t p23 = __byte_perm(hA, hB, 0x7632);
          uint32_t va[4], vb[4];
          ldsm_x4_trans(va, pb + vc_off + lm_off0);
          ldsm_x4_trans(vb, pb + vc_off + lm_off1);
          // V Deltas of the lane's four tokens, words (t0, t1), (t2, t3) per group
          uint32_t dl[4][2];
          if (NG == 4) {
            const uint4 a = lds128(pb + vd_off), b = lds128(pb + vd_off + 16);
            dl[0][0] = a.x; dl[0][1] = a.y; dl[1][0] = a.z; dl[1][1] = a.w;
            dl[2][0] = b.x; dl[2][1] = b.y; dl[3][0] = b.z; dl[3][1] = b.w;
          } else if (NG == 2) {
            const uint4 a = lds128(pb + vd_off);
            dl[0][0] = a.x; dl[0][1] = a.y; dl[1][0] = a.z; dl[1][1] = a.w;
          } else {
            const uint2 a = lds64(pb + vd_off);
            dl[0][0] = a.x; dl[0][1] = a.y;
          }
          const uint2 mw = lds64(pb + vm_off);  // V offsets of group mrow, same tokens
          // offset term: rows = groups (their m), columns = heads, against p
          mma_f16(mtacc, mw.x, 0u, mw.y, 0u, p01, p23);
#pragma unroll
          for (int P = 0; P < 4; ++P) {
            const int grp = (P * 32) / GS;
            const uint32_t b0 = hmul2(p01, dl[grp][0]);
            const uint32_t b1 = hmul2(p23, dl[grp][1]);
            const uint32_t wlo = (P < 2) ? va[2 * P] : vb[2 * (P - 2)];
            const uint32_t whi = (P < 2) ? va[2 * P + 1] : vb[2 * (P - 2) + 1];
            uint32_t xl[4], xh[4];
            widen_v_sub(wlo, xl);
            widen_v_sub(whi, xh);
            mma_f16(acc[P][0], xl[0], xl[1], xh[0], xh[1], b0, b1);
            mma_f16(acc[P][1], xl[2], xl[3], xh[2], xh[3], b0, b1);
          }
        }
        refill(ST);
        it = it + 1 == kSStages ? 0 : it + 1;
      }

      // publish this warp's state: head q's running max and sum over the
      // lanes of rows r = 0..7 (lane q holds the totals)
      float lsum = l_run;
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 4);
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 8);
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
      if (r == 0) {
        sm.mrg_m[warp][qd] = m_run;
        sm.mrg_l[warp][qd] = lsum;
      }
      // offset term of group g (row g, in lanes 4 g + q): sum_t p m for heads
      // 2 q and 2 q + 1
      if (r < NG && qd < 2) {
        for (int blk = r * (GS / 32); blk < (r + 1) * (GS / 32); ++blk) {
          sm.mrg_mt[warp][2 * qd][blk] = mtacc[0];
          sm.mrg_mt[warp][2 * qd + 1][blk] = mtacc[1];
        }
      }
      if (qd < 2) {
        const int hA = 2 * qd, hB = 2 * qd + 1;
#pragma unroll
        for (int P = 0; P < 4; ++P)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            // codes entered as c 2^-24 (even channels) and 16 c 2^-24 (odd)
            const int dd = 32 * P + 4 * r + 2 * hh;
            sm.mrg_o[warp][hA][dd] = acc[P][hh][0] * 0x1p24f;
            sm.mrg_o[warp][hB][dd] = acc[P][hh][1] * 0x1p24f;
            sm.mrg_o[warp][hA][dd + 1] = acc[P][hh][2] * 0x1p20f;
            sm.mrg_o[warp][hB][dd + 1] = acc[P][hh][3] * 0x1p20f;
          }
      }
    }

    // ----------------------------------------- segment end: partial + merge
    // the previous partial's ticket (taken one boundary ago) decides whether
    // this CTA merges that pair after this boundary
    if (threadIdx.x == kTicketThread) pend_take(sm, pend_t, nb);
    // B1: every warp has published; merge into partial pair + c, or into the
    // output when no other CTA holds the pair (sm.pcur, sm.new_q: written at
    // this segment's start; the ticket thread rewrites sm.cs before the next
    // barrier)
    __syncthreads();
    const bool direct = sm.pcur.direct;
    stream_merge_store(sm, part_o, part_lse, (long long)sm.pcur.pair + c, direct, sm.pcur.row0,
                       out, out_lse);
    if (threadIdx.x == kTicketThread) sm.cs = sm.nx;  // read by all after the next barrier
    if (sm.new_q) {  // fragments are not read again before the next barrier
      if (!mbar_wait(&sm.qbar, qphase & 1) && threadIdx.x == 0)
        set_status(status, KV4_STATUS_TIMEOUT);
      ++qphase;
      stream_query_setup<NG>(sm, scale_log2, q_rot);
    }
    __syncthreads();  // B2: partial stored; next pair's query set up; comb, cs written
    if (threadIdx.x == kTicketThread) {
      // take this partial's ticket with release semantics (the barrier above
      // makes the CTA's partial stores part of what is released); the
      // result is read at the next boundary.  A pair written directly, or
      // merged by the separate kernel (defer), takes none.
      if (!defer && !direct) {
        pend_t = atom_add_release_gpu(&tickets[sm.pcur.pair], sm.pcur.mine);
        sm.pend = sm.pcur;
      } else {
        sm.pend.valid = 0;
      }
    }
    if (sm.go[nb & 1]) {
      const Pend& cm = sm.comb[nb & 1];
      stream_combine(part_o, part_lse, (long long)cm.pair + cm.c0, cm.n0, cm.row0, out, out_lse);
    }
    ++nb;
  }
  // the last partial's ticket
  if (threadIdx.x == kTicketThread) pend_take(sm, pend_t, nb);
  __syncthreads();
  if (sm.go[nb & 1]) {
    const Pend& cm = sm.comb[nb & 1];
    stream_combine(part_o, part_lse, (long long)cm.pair + cm.c0, cm.n0, cm.row0, out, out_lse);
  }
  zero_empty();
}

// The stream's cut over the decode grid of C CTAs: per CTA the first unit of
// its share and the segment holding it, then, once the kernels before it on
// the stream have completed, the completion tickets of the fused merge set to
// zero.  Launched as a programmatic dependent of the kernel before it (the
// previous decode call lets its dependents launch once its CTAs have read
// their plan entries), the cut is worked out while that kernel finishes; the
// decode grid, launched as this kernel's dependent, starts as it exits.
// Each CTA counts the whole stream (the lengths) and its thread k works out
// share boundary k of the CTAs it serves (boundaries 0 .. C).
constexpr int kPrepThreads = 128;
// the last thread t whose prefix ex[t] is at most x (ex nondecreasing, ex[0] = 0)
__device__ inline int prep_owner(const long long* ex, long long x) {
  int lo = 0, hi = kPrepThreads - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ex[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}
__global__ void __launch_bounds__(kPrepThreads) stream_prep_kernel(
    Layout L, const int32_t* __restrict__ seq_lens, int B, int C, StreamPlan* __restrict__ plan,
    const int32_t* __restrict__ block_table, const uint16_t* __restrict__ q,
    int32_t* __restrict__ tickets, int n_tickets, int32_t* status) {
  __shared__ long long ex_u[kPrepThreads], ex_c[kPrepThreads];
  __shared__ long long wsum[2][kPrepThreads / 32];
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  // units and cost of this thread's sequences
  const int per = (B + kPrepThreads - 1) / kPrepThreads;
  auto b_lo = [&](int tt) { return min(B, tt * per); };
  auto b_hi = [&](int tt) { return min(B, tt * per + per); };
  long long mine = 0, mine_c = 0;
  bool bad_len = false;
  for (int b = b_lo(t); b < b_hi(t); ++b) {
    const int raw = __ldg(seq_lens + b);
    const int len = clamp_len(raw, L);
    bad_len |= len != raw;
    const int np = prot_units(len, L), n4 = int4_units(len, L);
    mine += (long long)L.h_kv * (np + n4);
    mine_c += (long long)L.h_kv * seg_cost(np, n4);
  }
  if (bad_len && blockIdx.x == 0) set_status(status, KV4_STATUS_BAD_LEN);
  // exclusive prefixes over the threads: within each warp, then over warps
  long long iu = mine, ic = mine_c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long yu = __shfl_up_sync(0xffffffffu, iu, o);
    const long long yc = __shfl_up_sync(0xffffffffu, ic, o);
    if (lane >= o) {
      iu += yu;
      ic += yc;
    }
  }
  if (lane == 31) {
    wsum[0][warp] = iu;
    wsum[1][warp] = ic;
  }
  __syncthreads();
  long long bu = 0, bc = 0, U = 0, Wc = 0;
#pragma unroll
  for (int w = 0; w < kPrepThreads / 32; ++w) {
    if (w < warp) {
      bu += wsum[0][w];
      bc += wsum[1][w];
    }
    U += wsum[0][w];
    Wc += wsum[1][w];
  }
  ex_u[t] = bu + iu - mine;
  ex_c[t] = bc + ic - mine_c;
  __syncthreads();
  // The stream is cut by cost over Cw CTAs: CTA c takes the units from the
  // first whose stream cost reaches T(c) up to the first whose cost reaches
  // T(c + 1) (Cut: shares weighted by launch rank).  Cw keeps every share at
  // least one unit's cost wide, so every working CTA holds a unit (the
  // partial counts rely on it).  Boundaries from Cw on are the stream's end.
  const Cut cut = stream_cut(Wc, C);
  if (blockIdx.x == 0 && t == 0) {
    plan->cut = cut;
    plan->total = U;
  }
  const int k = blockIdx.x * kPrepThreads + t;
  if (k <= C) {
    StreamStart s;
    s.u_begin = U;
    s.cs.start = U;
    s.cs.cs = Wc;
    s.cs.b = B;
    s.cs.h = 0;
    s.cs.len = 0;
    s.cs.np = 0;
    s.cs.n = 0;
    if (k < cut.Cw) {
      const long long Tb = cut.start(k);
      const int tb = prep_owner(ex_c, Tb);
      s.u_begin = unit_at_cost(Tb, b_lo(tb), b_hi(tb), ex_u[tb], ex_c[tb], L, seq_lens);
    }
    if (k < C && s.u_begin < U) {
      // the segment holding unit u_begin: in the sequences of the thread
      // whose unit range holds it
      const int tu = prep_owner(ex_u, s.u_begin);
      long long pre = ex_u[tu], pre_c = ex_c[tu];
      for (int b = b_lo(tu); b < b_hi(tu); ++b) {
        const int len = clamp_len(__ldg(seq_lens + b), L);
        const int np = prot_units(len, L), n4 = int4_units(len, L);
        const long long ub = (long long)L.h_kv * (np + n4);
        if (s.u_begin < pre + ub) {
          Seg cs;
          seg_set(cs, b, 0, len, L);
          cs.start = pre;
          cs.cs = pre_c;
          while (cs.start + cs.n <= s.u_begin) seg_next(cs, L, seq_lens, B);
          s.cs = cs;
          // into L2 ahead of the decode grid: the pair's query rows and the
          // block-table entries of its first INT4 units
          const char* qr = reinterpret_cast<const char*>(
              q + ((long long)cs.b * L.h_q + (long long)cs.h * SG) * SD);
#pragma unroll
          for (int o = 0; o < SG * SD * 2; o += 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(qr + o));
          const int j0 = (int)(s.u_begin - cs.start);
          const int p0 = kSPages * max(0, j0 - cs.np);
          if (cs.n > cs.np)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(block_table + (long long)cs.b * L.max_pages +
                                                           min(len, L.S) / kPage + p0));
          break;
        }
        pre += ub;
        pre_c += (long long)L.h_kv * seg_cost(np, n4);
      }
    }
    plan->start[k] = s;
  }
  // The tickets may still be in use by the kernels before this one (a decode
  // call on the same workspace): zero them once those have completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = k; i < n_tickets; i += gridDim.x * kPrepThreads) tickets[i] = 0;
}

// Eq. A1 for pairs whose partials are spread over many CTAs (few, long
// sequences): run after decode_stream_kernel, one CTA per (pair, query head),
// eight warps splitting the pair's partials.  The partial positions follow
// from the stream's share arithmetic, recounted from the lengths.
constexpr int kMergeThreads = 256;
__global__ void __launch_bounds__(kMergeThreads) stream_merge_kernel(
    Layout L, const int32_t* __restrict__ seq_lens, int B, const float* __restrict__ part_o,
    const float* __restrict__ part_lse, int C, uint16_t* __restrict__ out,
    float* __restrict__ out_lse) {
  __shared__ long long red64[2][kMergeThreads / 32];
  __shared__ float red_m[kMergeThreads / 32], red_l[kMergeThreads / 32];
  __shared__ float4 acc_s[kMergeThreads / 32][32];
  // the next call's prep kernel may start (it writes the plan, and the
  // tickets only after waiting for this grid; nothing here reads either)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int pair = blockIdx.x / SG, j = blockIdx.x % SG;
  const int b = pair / L.h_kv, h = pair % L.h_kv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int len = clamp_len(__ldg(seq_lens + b), L);
  if (len == 0) return;  // the decode kernel wrote its zero output
  // stream cost of the pair's first unit (the cost of all earlier sequences,
  // then of the sequence's earlier kv heads), and the stream's cost Wc, by the
  // decode kernel's own count
  long long v[2] = {0, 0};  // cost before sequence b; cost of all
  for (int bb = threadIdx.x; bb < B; bb += kMergeThreads) {
    const int lb = clamp_len(__ldg(seq_lens + bb), L);
    const long long c_ = (long long)L.h_kv * seg_cost(prot_units(lb, L), int4_units(lb, L));
    if (bb < b) v[0] += c_;
    v[1] += c_;
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[i] += __shfl_xor_sync(0xffffffffu, v[i], o);
    if (lane == 0) red64[i][warp] = v[i];
  }
  __syncthreads();
  long long pre_c = 0, Wc = 0;
  for (int w = 0; w < kMergeThreads / 32; ++w) {
    pre_c += red64[0][w];
    Wc += red64[1][w];
  }
  const int np = prot_units(len, L), nu = np + int4_units(len, L);
  const long long pcs = pre_c + (long long)h * seg_cost(np, nu - np);
  int c0 = 0, n = 0;
  pair_ctas(pcs, np, nu, stream_cut(Wc, C), c0, n);
  if (n == 1) return;  // a pair held by one CTA: the decode kernel wrote it
  const long long P0 = (long long)pair + c0;
  // Everything above reads only the inputs; what follows reads what the decode
  // kernel wrote (launched as its programmatic dependent, this is where the
  // merge waits for it to complete; otherwise the wait returns at once).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // warp w folds partials k = w, w + 8, ... (ten at a time: one round of L2
  // latency for up to 80 partials); warp 0 then folds the warps' states
  constexpr int NW = kMergeThreads / 32;
  float m = -INFINITY, l = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  fold_partials<10>(part_o, part_lse, P0, n, warp, NW, j, lane, m, l, a);
  if (lane == 0) {
    red_m[warp] = m;
    red_l[warp] = l;
  }
  acc_s[warp][lane] = a;
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w]);
    float Z = 0.f;
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = red_m[w];
      if (mw == -INFINITY) continue;
      const float e = exp2f((mw - M) * kLog2e);
      const float4 aw = acc_s[w][lane];
      Z = fmaf(e, red_l[w], Z);
      t.x = fmaf(e, aw.x, t.x);
      t.y = fmaf(e, aw.y, t.y);
      t.z = fmaf(e, aw.z, t.z);
      t.w = fmaf(e, aw.w, t.w);
    }
    const bool empty = !(Z > 0.f);
    const float inv = empty ? 0.f : 1.f / Z;
    const long long row = (long long)b * L.h_q + (long long)h * SG + j;
    uint16_t* o = out + row * SD + 4 * lane;
    o[0] = f32_to_bf16_bits(t.x * inv);
    o[1] = f32_to_bf16_bits(t.y * inv);
    o[2] = f32_to_bf16_bits(t.z * inv);
    o[3] = f32_to_bf16_bits(t.w * inv);
    if (out_lse && lane == 0) out_lse[row] = empty ? -INFINITY : M + logf(Z);
  }
}

}  // namespace

bool stream_supported(const Layout& L) { return L.d_h == SD && L.h_q == SG * L.h_kv; }

// Partial results the stream kernel may write for num_seqs sequences.
long long stream_partials(const Layout& L, int num_seqs) {
  return (long long)num_seqs * L.h_kv + kMaxStreamCtas;
}

// Bytes of the stream's plan (the per-CTA start table) in the workspace.
size_t stream_plan_bytes() { return sizeof(StreamPlan); }

// Eq. A1 for every pair held by more than one CTA, from the partials the
// work-balanced decode kernel left on a grid of C CTAs; the merge recounts
// the stream from the lengths.
cudaError_t launch_stream_merge(const Layout& L, const int32_t* seq_lens, int num_seqs,
                                const float* part_o, const float* part_lse, int C, bool overlap,
                                uint16_t* out, float* out_lse, cudaStream_t st) {
  // overlap: the previous kernel on the stream lets its dependents start early
  // (griddepcontrol.launch_dependents); this kernel then starts on the SMs its
  // CTAs free and waits for its completion only before reading its results
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_seqs * L.h_kv * SG));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, stream_merge_kernel, L, seq_lens, num_seqs, part_o, part_lse, C,
                            out, out_lse);
}

template <int NG>
cudaError_t launch_stream_t(const Layout& L, const void* paged, const void* side,
                            const uint16_t* q, const int32_t* seq_lens, int num_seqs,
                            const int32_t* block_table, float sm_scale, float* part_o,
                            float* part_lse, int32_t* tickets, void* plan, uint16_t* out,
                            float* out_lse, int32_t* status, float q_rot, cudaStream_t st) {
  constexpr int cb = 16 * SD + 128 * NG;
  constexpr size_t smem =
      ((sizeof(StreamSmem) + 127) / 128) * 128 + (size_t)kSW * kSStages * kSPages * cb;
  // four CTAs per SM: 228 KB per SM, 1 KB of it reserved per CTA
  static_assert(smem <= 228 * 1024 / kStreamMinBlocks - 1024, "shared memory per CTA");
  // once per device: the shared-memory attribute and the resident-CTA capacity
  static OnceSetup setup;
  int grid = 0;
  cudaError_t e = once_per_device(
      setup,
      [&](int dev, int* g) {
        cudaError_t r = cudaFuncSetAttribute(decode_stream_kernel<NG>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        int sms = 0, per_sm = 0;
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (r == cudaSuccess)
          r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_stream_kernel<NG>,
                                                            kST, smem);
        *g = std::max(1, std::min(kMaxStreamCtas, sms * std::max(1, per_sm)));
        return r;
      },
      &grid);
  if (e != cudaSuccess) return e;
  // With few pairs each one spreads over many CTAs; its merge then runs as a
  // separate, wider kernel instead of in the last CTA.
  const int defer = 8LL * num_seqs * L.h_kv < grid ? 1 : 0;
  // The prep kernel cuts the stream over the grid into the plan and zeroes
  // the completion tickets of the in-kernel merge; it is a programmatic
  // dependent of the kernel before it, and the decode grid of it.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  StreamPlan* sp = static_cast<StreamPlan*>(plan);
  {
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3((unsigned)(grid / kPrepThreads + 1));  // boundaries 0 .. grid
    pc.blockDim = dim3(kPrepThreads);
    pc.stream = st;
    pc.attrs = attr;
    pc.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&pc, stream_prep_kernel, L, seq_lens, num_seqs, grid, sp,
                                block_table, q, tickets, defer ? 0 : num_seqs * L.h_kv,
                                status)) != cudaSuccess)
      return e;
  }
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kST);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_stream_kernel<NG>, L, (const uint8_t*)paged,
                           (const uint8_t*)side, q, seq_lens, num_seqs, block_table,
                           sm_scale * kLog2e, part_o, part_lse, tickets, out, out_lse, status, defer,
                           q_rot, (const StreamPlan*)sp);
    if (e != cudaSuccess) return e;
  }
  if (defer)
    e = launch_stream_merge(L, seq_lens, num_seqs, part_o, part_lse, grid, true, out, out_lse, st);
  return e;
}

cudaError_t launch_decode_stream(const Layout& L, const void* paged, const void* side,
                                 const uint16_t* q, const int32_t* seq_lens, int num_seqs,
                                 const int32_t* block_table, float sm_scale, float* part_o,
                                 float* part_lse, int32_t* tickets, void* plan, uint16_t* out,
                                 float* out_lse, int32_t* status, bool rotate_q, cudaStream_t st) {
  // the query rotated in the kernel's query set-up (Hadamard K-rotation)
  const float q_rot = rotate_q ? hadamard_scale(SD) : 0.f;
  switch (L.d_h / L.g) {
    case 4:
      return launch_stream_t<4>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale,
                                part_o, part_lse, tickets, plan, out, out_lse, status, q_rot, st);
    case 2:
      return launch_stream_t<2>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale,
                                part_o, part_lse, tickets, plan, out, out_lse, status, q_rot, st);
    case 1:
      return launch_stream_t<1>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale,
                                part_o, part_lse, tickets, plan, out, out_lse, status, q_rot, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kv4
