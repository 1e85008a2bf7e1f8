// kv4_decode_sm.cu -- SM-persistent decode over the mixed INT4 / INT8 cache
// (KV4-RL Sec. 5.3 and eq. 5.1; App. A.3 "Protected path" and eq. A1),
// head_dim 128 with 4 query heads per kv head.
//
// The work is the unit stream of the work-balanced kernel: per (sequence,
// kv head) pair its protected units (16 INT8 side-cache slots each), then
// its INT4 units (two 16-token pages each).  One CTA of sixteen warps runs on
// each SM and takes the units [c*U/C, (c+1)*U/C).  After start-up the CTA has
// no barrier: each warp claims the CTA's units one at a time from a shared
// counter, streams them through its own two-stage ring of bulk copies, and
// keeps one online-softmax state for the segment (a pair's protected or INT4
// units) it is in.  A warp that moves on to another segment hands its state
// over without a lock: it takes the segment's published state (if any),
// merges it into its own registers and publishes the result; the warp whose
// state comes to cover all of the segment's units in this CTA writes the
// partial result (2 * pair + region + c, as in the work-balanced kernel).
// The separate merge kernel then applies eq. A1 to every pair's partials.  A
// warp that runs ahead never waits for the others except on its own deposit
// area or a query buffer whose earlier pair has not finished, so the SM stays
// busy until its units are done.
//
// The per-pair query fragments are built once per call by
// decode_sm_qprep_kernel and bulk-copied into one of four buffers when a
// pair's first unit in the CTA is claimed.  The per-unit arithmetic is that of
// the work-balanced kernel.
#include <algorithm>

#include "kv4_decode_common.cuh"
#include "kv4_mma.cuh"
#include "kv4_stream_common.cuh"

namespace kv4 {
namespace {

constexpr int kMW = 16;                 // warps per CTA, one CTA per SM
constexpr int kMThreads = kMW * 32;
constexpr int kMStages = 2;             // bulk-copy stages per warp
constexpr int kQBufs = 4;               // query-fragment buffers (pairs in flight)
constexpr int kRing = 32;               // segment completion counters (segments in flight)
constexpr uint32_t kSpinLimit = 1u << 23;  // bound on a (backed-off) spin over a shared-memory flag

// What the consumer lanes need about the unit in a stage; written by the
// warp's producer lane before the copy's arrive.
struct StageRec {
  long long start;         // first stream unit of the unit's segment
  int b, h, type, len, n;  // the segment (pair b, h; region type; its sequence length; units)
  int j;                   // unit index inside the segment
  int sig, pord;           // ordinals of the segment and its pair among this CTA's
  int phys0, phys1;        // INT4: the two physical pages (< 0: not loaded)
};

// Producer cursor of one warp (lane 0): the segment of its last claimed unit.
struct ProdM {
  Seg s;
  int sig, pord;
  long long u;  // claimed unit, not yet issued
  int more;     // u is valid
};

// One warp's state at the end of its part of a segment, deposited for the
// merge: for the 16 lanes that hold query heads 0-3 (lane 4r + qd, qd < 2,
// at index 2r + qd) the 32 accumulators of the warp layout and, for INT4
// units, two offset-term values, component-major so that the lanes' accesses
// do not conflict; per head the reference m and the sum l.
struct Dep {
  float acc[34][16];
  float m[SG], l[SG];
  int n;    // units the state covers
  int sig;  // segment held (-1: the area is free)
  int pad_[2];
};

// The published state of one segment in this CTA (entry sig mod kRing).
struct SegDone {
  int gen;   // segment ordinal the entry serves
  int held;  // warp whose deposit holds the segment's merged-so-far state, or -1
};

struct __align__(16) SmSmem {
  QPrep qb[kQBufs];
  union {
    Dep dep[kMW];
    long long scan[kMThreads];  // start-up: per-thread unit counts, then their prefix
  };
  SegDone ring[kRing];
  StageRec rec[kMW][kMStages];
  ProdM prod[kMW];
  float tmt[kMW][SG][SD / 32];  // finalize: offset term per (head, 32-channel block)
  // per query buffer, in one word so that both change together: the pair
  // ordinal loaded (or loading) into it (high half, biased by kQBufs) and the
  // units of that pair in this CTA not yet processed (low half)
  unsigned long long qb_state[kQBufs];
  long long total, u_begin, u_end;
  Seg cs0;                      // segment of the first unit
  int next;                     // units claimed so far (from u_begin)
  uint64_t qb_bar[kQBufs];
  uint64_t bar[kMW][kMStages];
};

__device__ inline unsigned long long qb_word(int pord, int left) {
  return ((unsigned long long)(unsigned)(pord + kQBufs) << 32) | (unsigned)left;
}
__device__ inline int qb_pair(unsigned long long w) { return (int)(w >> 32) - kQBufs; }

__device__ inline int vload(const int* p) { return *reinterpret_cast<const volatile int*>(p); }
__device__ inline float vloadf(const float* p) { return *reinterpret_cast<const volatile float*>(p); }

// Units of the pair whose segment is s that lie in [ub, ue).
__device__ inline int pair_units_in(const Seg& s, const Layout& L, long long ub, long long ue) {
  const int np = prot_units(s.len, L), n4 = int4_units(s.len, L);
  const long long gs = s.type == 0 ? s.start : s.start - np;
  return (int)(min(ue, gs + np + n4) - max(ub, gs));
}

// One CTA per pair: the pair's query fragments and sums (QPrep).
template <int NG>
__global__ void __launch_bounds__(128) decode_sm_qprep_kernel(Layout L,
                                                              const uint16_t* __restrict__ q,
                                                              QPrep* __restrict__ qprep) {
  __shared__ __align__(16) uint16_t qraw[SG * SD];
  __shared__ QPrep qp;
  const int pair = blockIdx.x;
  const long long row0 = (long long)(pair / L.h_kv) * L.h_q + (long long)(pair % L.h_kv) * SG;
  const uint4* src = reinterpret_cast<const uint4*>(q + row0 * SD);
  if (threadIdx.x < SG * SD / 8)  // G rows of D bf16: 64 x 16 B
    reinterpret_cast<uint4*>(qraw)[threadIdx.x] = __ldg(src + threadIdx.x);
  __syncthreads();
  build_qprep<NG>(qraw, qp, threadIdx.x);
  __syncthreads();
  const uint4* s4 = reinterpret_cast<const uint4*>(&qp);
  uint4* d4 = reinterpret_cast<uint4*>(qprep + pair);
  for (int i = threadIdx.x; i < (int)(sizeof(QPrep) / 16); i += 128) d4[i] = s4[i];
}

template <int NG>
__global__ void __launch_bounds__(kMThreads, 1) decode_sm_kernel(
    Layout L, const uint8_t* __restrict__ paged, const uint8_t* __restrict__ side,
    const QPrep* __restrict__ qprep, const int32_t* __restrict__ seq_lens, int B,
    const int32_t* __restrict__ block_table, float scale_log2, float* __restrict__ part_o,
    float* __restrict__ part_lse, uint16_t* __restrict__ out, float* __restrict__ out_lse,
    int32_t* status) {
  constexpr int D = SD;
  constexpr int GS = D / NG;  // channels per INT4 group
  constexpr int cb = 16 * D + 128 * NG;
  constexpr int SB = kSPages * cb;  // stage bytes: two INT4 chunks or one 16-slot INT8 unit
  static_assert(2 * kProtUnit * SD + 4 * kProtUnit <= SB, "an INT8 unit fits a stage");
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmSmem& sm = *reinterpret_cast<SmSmem*>(smem_raw);
  uint8_t* stage_base = smem_raw + ((sizeof(SmSmem) + 127) / 128) * 128;
  const int C = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ------------------------------------------ stream size and this CTA's share
  const int per = (B + kMThreads - 1) / kMThreads;
  const int b_lo = min(B, (int)threadIdx.x * per), b_hi = min(B, b_lo + per);
  long long mine = 0;
  bool bad_len = false;
  for (int b = b_lo; b < b_hi; ++b) {
    const int raw = __ldg(seq_lens + b);
    const int len = clamp_len(raw, L);
    bad_len |= len != raw;
    mine += (long long)L.h_kv * (prot_units(len, L) + int4_units(len, L));
  }
  if (c == 0 && bad_len) set_status(status, KV4_STATUS_BAD_LEN);
  sm.scan[threadIdx.x] = mine;
  __syncthreads();
  if (warp == 0) {  // exclusive prefix over the 512 per-thread counts
    constexpr int E = kMThreads / 32;
    long long v[E], run = 0;
#pragma unroll
    for (int k = 0; k < E; ++k) {
      v[k] = run;
      run += sm.scan[E * lane + k];
    }
    long long incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const long long excl = incl - run;
    __syncwarp();
#pragma unroll
    for (int k = 0; k < E; ++k) sm.scan[E * lane + k] = excl + v[k];
    if (lane == 31) sm.total = incl;
  }
  __syncthreads();
  const long long U = sm.total;
  const int Cw = (int)min((long long)C, U);
  const long long u_begin = c < Cw ? U * c / Cw : U, u_end = c < Cw ? U * (c + 1) / Cw : U;
  if (threadIdx.x == 0) {
    sm.u_begin = u_begin;
    sm.u_end = u_end;
  }
  if (u_begin < u_end) {  // the thread whose sequences hold u_begin: its segment
    const long long ex = sm.scan[threadIdx.x];
    if (u_begin >= ex && u_begin < ex + mine) {
      long long pre = ex;
      for (int b = b_lo; b < b_hi; ++b) {
        const int len = clamp_len(__ldg(seq_lens + b), L);
        const int np = prot_units(len, L), pu = np + int4_units(len, L);
        const long long ub = (long long)L.h_kv * pu;
        if (u_begin < pre + ub) {
          Seg sg;
          sg.cs = 0;
          sg.b = b;
          sg.len = len;
          const long long off = u_begin - pre;
          sg.h = (int)(off / pu);
          const int w = (int)(off - (long long)sg.h * pu);
          sg.type = w < np ? 0 : 1;
          sg.start = pre + (long long)sg.h * pu + (sg.type ? np : 0);
          sg.n = sg.type ? pu - np : np;
          sm.cs0 = sg;
          break;
        }
        pre += ub;
      }
    }
  }
  // sequences with nothing to attend: zero output, log-normaliser -inf
  for (int b = c; b < B; b += C) {
    if (clamp_len(__ldg(seq_lens + b), L) != 0) continue;
    for (int idx = threadIdx.x; idx < L.h_q * D; idx += kMThreads)
      out[(long long)b * L.h_q * D + idx] = 0;
    if (out_lse)
      for (int idx = threadIdx.x; idx < L.h_q; idx += kMThreads)
        out_lse[(long long)b * L.h_q + idx] = -INFINITY;
  }
  __syncthreads();  // the prefix is no longer read: the slots may reuse its memory
  if (u_begin >= u_end) return;
  if (threadIdx.x < kMW) sm.dep[threadIdx.x].sig = -1;
  if (threadIdx.x < kRing) {
    sm.ring[threadIdx.x].gen = threadIdx.x;
    sm.ring[threadIdx.x].held = -1;
  }
  if (threadIdx.x < kQBufs) {
    sm.qb_state[threadIdx.x] = qb_word(threadIdx.x - kQBufs, 0);  // "previous" user: pair i - 4
    mbar_init(&sm.qb_bar[threadIdx.x], 1);
  }
  if (threadIdx.x == 0) sm.next = 0;
  if (lane == 0) {
    for (int st = 0; st < kMStages; ++st) mbar_init(&sm.bar[warp][st], 1);
  }
  fence_mbar_init();
  __syncthreads();

  // ------------------------------------------------------ producer (lane 0)
  const int NS = L.S + L.R;
  const int NSP = side_scale_entries(L.S, L.R);
  const long long side_blk = side_block_bytes(D, L.S, L.R);
  uint8_t* my_stages = stage_base + (size_t)warp * kMStages * SB;
  int pphys = -1, pphys1 = -1;  // the claimed unit's INT4 pages (-2: no second page)

  // Lane 0: start loading pair `pord`'s query fragments into its buffer if
  // the buffer's previous pair is done; returns whether the load is started
  // (or was already).
  auto try_qload = [&](int pord, const Seg& s) -> bool {
    const int qb = (int)((unsigned)pord % kQBufs);
    const unsigned long long w = *reinterpret_cast<volatile unsigned long long*>(&sm.qb_state[qb]);
    if (qb_pair(w) == pord) return true;
    if (w != qb_word(pord - kQBufs, 0)) return false;  // the previous pair still in use
    const unsigned long long nw = qb_word(pord, pair_units_in(s, L, sm.u_begin, sm.u_end));
    if (atomicCAS(&sm.qb_state[qb], w, nw) != w)
      return qb_pair(*reinterpret_cast<volatile unsigned long long*>(&sm.qb_state[qb])) == pord;
    fence_proxy_async_smem();  // earlier reads of the buffer before the copy rewrites it
    mbar_arrive_expect_tx(&sm.qb_bar[qb], (uint32_t)sizeof(QPrep));
    bulk_g2s(&sm.qb[qb], qprep + (s.b * L.h_kv + s.h), (uint32_t)sizeof(QPrep), &sm.qb_bar[qb]);
    return true;
  };
  // Lane 0: claim the CTA's next unit for this warp, move the cursor to its
  // segment, start reading its block-table entries (consumed at the next
  // issue, so their latency is not waited for here).
  auto claim = [&]() {
    ProdM& pr = sm.prod[warp];
    const long long u = sm.u_begin + atomicAdd(&sm.next, 1);
    if (u >= sm.u_end) {
      pr.more = 0;
      return;
    }
    Seg s = pr.s;
    int sig = pr.sig, pord = pr.pord;
    bool new_pair = false;
    while (u >= s.start + s.n && s.b < B) {
      const int ob = s.b, oh = s.h;
      seg_next(s, L, seq_lens, B);
      ++sig;
      if (s.b != ob || s.h != oh) {
        ++pord;
        new_pair = true;
      }
    }
    if (s.b >= B) {  // (cannot happen: u < U) stop rather than read past the stream
      set_status(status, KV4_STATUS_BAD_LEN);
      pr.more = 0;
      return;
    }
    pr.s = s;
    pr.sig = sig;
    pr.pord = pord;
    pr.u = u;
    pr.more = 1;
    if (s.type == 1) {
      const int jj = (int)(u - s.start);
      const int pg = min(s.len, L.S) / kPage + kSPages * jj;  // < max_pages: len is clamped
      const int32_t* bt = block_table + (long long)s.b * L.max_pages + pg;
      if (jj < 0 || pg >= L.max_pages) {
        set_status(status, KV4_STATUS_INTERNAL);
        pphys = -1;
        pphys1 = -2;
      } else {
        pphys = __ldg(bt);
        pphys1 = kSPages * jj + 1 < int4_pages(s.len, L) ? __ldg(bt + 1) : -2;
      }
    }
    if (new_pair) try_qload(pord, s);  // prefetch; the first consumer retries if refused
  };
  // Lane 0: copy the claimed unit into stage st and describe it there.
  auto issue = [&](int st) {
    const ProdM& pr = sm.prod[warp];
    const Seg& ps = pr.s;
    const int pj = (int)(pr.u - ps.start);
    uint64_t* bar = &sm.bar[warp][st];
    uint8_t* dst = my_stages + (size_t)st * SB;
    StageRec& rc = sm.rec[warp][st];
    rc.start = ps.start;
    rc.b = ps.b;
    rc.h = ps.h;
    rc.type = ps.type;
    rc.len = ps.len;
    rc.n = ps.n;
    rc.j = pj;
    rc.sig = pr.sig;
    rc.pord = pr.pord;
    if (ps.type == 1) {
      // pages 2j and 2j + 1 of the segment (the second may not exist: -2)
      const bool good0 = pphys >= 0 && pphys < L.num_pages;
      const bool good1 = pphys1 >= 0 && pphys1 < L.num_pages;
      if (!good0 || (pphys1 != -2 && !good1)) set_status(status, KV4_STATUS_BAD_PAGE);
      rc.phys0 = good0 ? pphys : -1;  // published by the arrive below
      rc.phys1 = good1 ? pphys1 : -1;
      const uint32_t bytes = (good0 ? (uint32_t)cb : 0u) + (good1 ? (uint32_t)cb : 0u);
      if (bytes) {
        mbar_arrive_expect_tx(bar, bytes);
        if (good0) bulk_g2s(dst, paged + ((long long)pphys * L.h_kv + ps.h) * cb, (uint32_t)cb, bar);
        if (good1)
          bulk_g2s(dst + cb, paged + ((long long)pphys1 * L.h_kv + ps.h) * cb, (uint32_t)cb, bar);
      } else {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
      }
    } else {
      const uint8_t* blk = side + ((long long)ps.b * L.h_kv + ps.h) * side_blk;
      const int slot0 = pj * kProtUnit;
      const int ns = ps.len <= L.S ? ps.len : NS;
      uint32_t rows = (uint32_t)min(kProtUnit, ns - slot0);
      if (slot0 < 0 || (int)rows <= 0 || slot0 + (int)rows > NS) {  // (cannot happen)
        set_status(status, KV4_STATUS_INTERNAL);
        rows = 0;
      }
      // scales of the 8-slot runs that hold copied rows (within the NSP padding)
      const uint32_t sbytes = 16u * ((rows + 7) / 8);
      if (rows == 0) {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
      } else {
        mbar_arrive_expect_tx(bar, 2u * rows * D + 2u * sbytes);
        bulk_g2s(dst, blk + (long long)slot0 * D, rows * D, bar);
        bulk_g2s(dst + kProtUnit * D, blk + (long long)(NS + slot0) * D, rows * D, bar);
        bulk_g2s(dst + 2 * kProtUnit * D, blk + 2LL * NS * D + 2 * slot0, sbytes, bar);
        bulk_g2s(dst + 2 * kProtUnit * D + 2 * kProtUnit,
                 blk + 2LL * NS * D + 2LL * NSP + 2 * slot0, sbytes, bar);
      }
    }
  };
  int issued = 0;
  if (lane == 0) {
    ProdM& pr = sm.prod[warp];
    pr.s = sm.cs0;
    pr.sig = 0;
    pr.pord = 0;
    pr.u = -1;
    if (warp == 0) try_qload(0, sm.cs0);
    claim();
    for (int st = 0; st < kMStages && pr.more; ++st) {
      issue(st);
      ++issued;
      claim();
    }
  }
  int inflight = __shfl_sync(0xffffffffu, issued, 0);

  // ------------------------------------------------------ per-lane constants
  const int r = lane >> 2, qd = lane & 3;
  const int jh = r & 3;                 // this lane's softmax head
  const int g0 = r >> 2, g1 = g0 + 2;   // INT4 path: groups of QK rows r and r+8
  const bool v0 = NG == 4 || g0 < NG, v1 = NG == 4 || g1 < NG;
  const uint32_t p_keep = (r < 4) ? 0xFFFFFFFFu : 0u;
  const int lm_tok = ((lane >> 3) & 1) * 8 + (lane & 7);
  const int lm_p = lane >> 4;
  const uint32_t lm_off0 = lm_tok * 64 + 16 * ((lm_p) ^ ((lm_tok >> 1) & 3));
  const uint32_t lm_off1 = lm_tok * 64 + 16 * ((lm_p + 2) ^ ((lm_tok >> 1) & 3));
  const int l8_t = lane & 7, l8_row = ((lane >> 3) & 1) * 8 + l8_t, l8_pp = lane >> 4;
  constexpr int TK[4] = {0, 1, 8, 9};   // this lane's tokens / slots: 2 * qd + TK[e]
  const uint32_t stages_u32 = smem_u32(my_stages);
  const uint32_t k_lane = stages_u32 + r * 64 + row_byte(16 * qd, r, D);  // (+512: r + 8)
  const uint32_t km_lane = stages_u32 + meta_off_k(D) + (2 * qd * NG + g0) * 4;
  const uint32_t vm_lane = stages_u32 + meta_off_v(D, GS) + 2 * qd * NG * 4;
  const int mt_g = r >> 1;                  // offset-term MMA: this lane's A row group
  const bool mt_row = mt_g < NG;
  const uint32_t mt_sel = (r & 1) ? 0x7632u : 0x5410u;  // Delta (low) or m (high) halves
  const uint32_t v_lane = stages_u32 + codes_off_v(D);

  // ------------------------------------------------------ per-warp state
  float acc[32];          // INT4: [P][hh][i] = P*8 + hh*4 + i; INT8: [P][i] = P*4 + i
  float mtacc[4] = {0.f, 0.f, 0.f, 0.f};  // INT4 offset term (rows group x (Delta | m), heads)
  float m_run = -INFINITY, l_run = 0.f;
  int cur_sig = -1, cur_pord = -1, cur_type = 0, my_n = 0, qb = 0;
  int cur_b = 0, cur_h = 0, cur_len = 0, cur_n = 0;
  long long cur_start = 0;
  float qs0 = 0.f, qs1 = 0.f, kc0 = 0.f, kc1 = 0.f;

  // End of this warp's part of its segment.  The segment keeps at most one
  // published state (a warp's deposit).  The warp takes it if there is one,
  // merges it into its own registers, and publishes the result in its own
  // deposit area; if another state was published meanwhile it takes that one
  // too.  The warp whose state comes to cover all of the segment's units in
  // this CTA writes the partial result.  A warp
  // waits only for its own deposit area (its previous deposit not yet taken)
  // or a segment entry still serving an older segment.
  auto retire = [&]() {
    SegDone& E = sm.ring[(unsigned)cur_sig % kRing];
    Dep& Dw = sm.dep[warp];
    const int n_seg = (int)(min(sm.u_end, cur_start + cur_n) - max(sm.u_begin, cur_start));
    float lsum = (r < 4) ? l_run : 0.f;
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    float m4[SG], l4[SG];  // per head, the same in every lane
#pragma unroll
    for (int h = 0; h < SG; ++h) {
      m4[h] = __shfl_sync(0xffffffffu, m_run, 4 * h);
      l4[h] = __shfl_sync(0xffffffffu, lsum, 4 * h);
    }
    const int ci = 2 * r + qd;  // (lanes qd >= 2 hold padding heads: nothing to keep)
    int n = my_n;
    if (lane == 0) {
      uint32_t k = 0;
      while (vload(&E.gen) != cur_sig && ++k < kSpinLimit) __nanosleep(64);
      if (k >= kSpinLimit) set_status(status, KV4_STATUS_TIMEOUT);
    }
    __syncwarp();
    for (int round = 0; round <= 2 * kMW; ++round) {
      if (n < n_seg) {  // take the published state, if any, and merge it
        int h = -1;
        if (lane == 0) {
          h = atomicExch(&E.held, -1);
          if (h >= 0) __threadfence_block();
        }
        h = __shfl_sync(0xffffffffu, h, 0);
        __syncwarp();
        if (h >= kMW) {  // (cannot happen)
          if (lane == 0) set_status(status, KV4_STATUS_INTERNAL);
          h = -1;
        }
        if (h >= 0) {
          const Dep& Dd = sm.dep[h];
          float s0[SG], s1[SG];
#pragma unroll
          for (int hh = 0; hh < SG; ++hh) {
            const float md = vloadf(&Dd.m[hh]), ld = vloadf(&Dd.l[hh]);
            const float M = fmaxf(m4[hh], md);
            s0[hh] = m4[hh] == -INFINITY ? 0.f : ex2(m4[hh] - M);
            s1[hh] = md == -INFINITY ? 0.f : ex2(md - M);
            l4[hh] = s0[hh] * l4[hh] + s1[hh] * ld;
            m4[hh] = M;
          }
          const float a0 = qd == 0 ? s0[0] : s0[2], a1 = qd == 0 ? s0[1] : s0[3];
          const float b0 = qd == 0 ? s1[0] : s1[2], b1 = qd == 0 ? s1[1] : s1[3];
          if (qd < 2) {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              acc[k] = fmaf(Dd.acc[k][ci], (k & 1) ? b1 : b0, acc[k] * ((k & 1) ? a1 : a0));
            mtacc[0] = fmaf(Dd.acc[32][ci], b0, mtacc[0] * a0);
            mtacc[1] = fmaf(Dd.acc[33][ci], b1, mtacc[1] * a1);
          }
          n += vload(&Dd.n);
          __syncwarp();
          if (lane == 0) {  // the deposit is read: its area is free again
            __threadfence_block();
            *reinterpret_cast<volatile int*>(&sm.dep[h].sig) = -1;
          }
        }
      }
      if (n >= n_seg) break;
      // publish this state in the warp's own area
      if (lane == 0) {
        uint32_t k = 0;
        while (vload(&Dw.sig) != -1 && ++k < kSpinLimit) __nanosleep(64);
        if (k >= kSpinLimit) set_status(status, KV4_STATUS_TIMEOUT);
        __threadfence_block();
      }
      __syncwarp();
      if (qd < 2) {
#pragma unroll
        for (int k = 0; k < 32; ++k) Dw.acc[k][ci] = acc[k];
        Dw.acc[32][ci] = mtacc[0];
        Dw.acc[33][ci] = mtacc[1];
      }
      if (lane < SG) {
        Dw.m[lane] = lane == 0 ? m4[0] : lane == 1 ? m4[1] : lane == 2 ? m4[2] : m4[3];
        Dw.l[lane] = lane == 0 ? l4[0] : lane == 1 ? l4[1] : lane == 2 ? l4[2] : l4[3];
      }
      if (lane == 0) Dw.n = n;
      __syncwarp();
      int ok = 0;
      if (lane == 0) {
        *reinterpret_cast<volatile int*>(&Dw.sig) = cur_sig;
        __threadfence_block();  // the deposit before its publication
        ok = atomicCAS(&E.held, -1, warp) == -1;
        if (!ok) *reinterpret_cast<volatile int*>(&Dw.sig) = -1;  // not published: still ours
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (ok) return;  // a later warp takes it
    }
    if (n != n_seg) {  // (cannot happen: every unit is merged exactly once)
      if (lane == 0) set_status(status, KV4_STATUS_INTERNAL);
      return;
    }
    if (lane == 0) {  // the entry is free for segment cur_sig + kRing
      __threadfence_block();
      *reinterpret_cast<volatile int*>(&E.gen) = cur_sig + kRing;
    }
    float Lh = lane == 0 ? l4[0] : lane == 1 ? l4[1] : lane == 2 ? l4[2] : l4[3];
    float Mh = lane == 0 ? m4[0] : lane == 1 ? m4[1] : lane == 2 ? m4[2] : m4[3];
    // ---- the partial: o = (acc + offset term) / L per head and channel
    const int pair = cur_b * L.h_kv + cur_h;
    const long long P = 2LL * pair + cur_type + c;  // this CTA's partial of the segment
    if (cur_b < 0 || cur_b >= B || cur_h < 0 || cur_h >= L.h_kv) {  // (cannot happen)
      if (lane == 0) set_status(status, KV4_STATUS_INTERNAL);
      return;
    }
    if (cur_type == 1) {
      // offset term of group g, heads 2qd, 2qd+1: sum p m + 8 sum p Delta
      // (rows 2g and 2g + 1 live in lanes 8g + qd and 8g + 4 + qd)
      const float om0 = __shfl_xor_sync(0xffffffffu, mtacc[0], 4);
      const float om1 = __shfl_xor_sync(0xffffffffu, mtacc[1], 4);
      if ((r & 1) == 0 && mt_row && qd < 2) {
        const float tA = fmaf(8.f, mtacc[0], om0), tB = fmaf(8.f, mtacc[1], om1);
        for (int blk = mt_g * (GS / 32); blk < (mt_g + 1) * (GS / 32); ++blk) {
          sm.tmt[warp][2 * qd][blk] = tA;
          sm.tmt[warp][2 * qd + 1][blk] = tB;
        }
      }
      __syncwarp();
    }
    const float lA = qd == 0 ? l4[0] : l4[2], lB = qd == 0 ? l4[1] : l4[3];
    if (qd < 2) {
      const int hA = 2 * qd, hB = 2 * qd + 1;
      const float iA = lA > 0.f ? 1.f / lA : 0.f;
      const float iB = lB > 0.f ? 1.f / lB : 0.f;
      float* oA = part_o + (P * SG + hA) * SD;
      float* oB = part_o + (P * SG + hB) * SD;
      if (cur_type == 1) {
#pragma unroll
        for (int Pb = 0; Pb < 4; ++Pb) {
          const float tA = sm.tmt[warp][hA][Pb], tB = sm.tmt[warp][hB][Pb];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int dd = 32 * Pb + 4 * r + 2 * hh, k = Pb * 8 + hh * 4;
            *reinterpret_cast<float2*>(oA + dd) =
                make_float2((acc[k] + tA) * iA, (acc[k + 2] + tA) * iA);
            *reinterpret_cast<float2*>(oB + dd) =
                make_float2((acc[k + 1] + tB) * iB, (acc[k + 3] + tB) * iB);
          }
        }
      } else {
#pragma unroll
        for (int Pb = 0; Pb < 8; ++Pb) {
          const int dd = 16 * Pb + 2 * r, k = Pb * 4;
          *reinterpret_cast<float2*>(oA + dd) = make_float2(acc[k] * iA, acc[k + 2] * iA);
          *reinterpret_cast<float2*>(oB + dd) = make_float2(acc[k + 1] * iB, acc[k + 3] * iB);
        }
      }
    }
    if (lane < SG) part_lse[P * SG + lane] = Lh > 0.f ? (Mh + log2f(Lh)) * kLn2 : -INFINITY;
    __syncwarp();
  };

  int it = 0;  // this warp's consumed units (stage it % 2, phase (it / 2) & 1)
  while (inflight > 0) {
    const int ST = (int)((unsigned)it % kMStages);
    const uint32_t SO = (uint32_t)(ST * SB);  // stage offset
    const bool ok =
        __all_sync(0xffffffffu, mbar_wait(&sm.bar[warp][ST], ((unsigned)it / kMStages) & 1));
    if (!ok && lane == 0) set_status(status, KV4_STATUS_TIMEOUT);
    const StageRec& rc = sm.rec[warp][ST];
    const int sig = rc.sig;
    if (sig != cur_sig) {
      if (cur_sig >= 0) retire();
      const int pord = rc.pord;
      Seg sg;
      sg.cs = 0;
      sg.start = rc.start;
      sg.b = rc.b;
      sg.h = rc.h;
      sg.type = rc.type;
      sg.len = rc.len;
      sg.n = rc.n;
      if (pord != cur_pord) {
        // this pair's query fragments: load them if no one has, then wait
        qb = (int)((unsigned)pord % kQBufs);
        if (lane == 0) {
          uint32_t k = 0;
          while (!try_qload(pord, sg) && ++k < kSpinLimit) __nanosleep(128);
          if (k >= kSpinLimit) set_status(status, KV4_STATUS_TIMEOUT);
        }
        __syncwarp();
        const bool qok = __all_sync(
            0xffffffffu, mbar_wait(&sm.qb_bar[qb], ((unsigned)pord / kQBufs) & 1));
        if (!qok && lane == 0) set_status(status, KV4_STATUS_TIMEOUT);
        cur_pord = pord;
        const QPrep& qp = sm.qb[qb];
        qs0 = 0.f;
        qs1 = 0.f;
#pragma unroll
        for (int bq = 0; bq < D / 32; ++bq) {
          if (v0 && (bq * 32) / GS == g0) qs0 += qp.qsum[bq][jh];
          if (v1 && (bq * 32) / GS == g1) qs1 += qp.qsum[bq][jh];
        }
        kc0 = v0 ? qp.kc[g0][jh] : 0.f;
        kc1 = v1 ? qp.kc[g1][jh] : 0.f;
      }
      cur_sig = sig;
      cur_type = sg.type;
      cur_b = sg.b;
      cur_h = sg.h;
      cur_len = sg.len;
      cur_n = sg.n;
      cur_start = sg.start;
      my_n = 0;
      m_run = -INFINITY;
      l_run = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) acc[k] = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) mtacc[k] = 0.f;
    }
    const int jj = rc.j;
    const Regions rg = regions(cur_len, L.S, L.R);
    if (ok && cur_type == 1) {
      // ============================================= INT4 pages (eq. 5.1)
      const int ph0 = rc.phys0, ph1 = rc.phys1;
      const uint4* qa_s = reinterpret_cast<const uint4*>(&sm.qb[qb].qfrag4[0][0][0]) + lane;
      const int pg0 = rg.sink_end / kPage + kSPages * jj;
      uint4 kw[2][2];
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        kw[pp][0] = lds128(k_lane + SO + pp * cb);
        kw[pp][1] = lds128(k_lane + SO + pp * cb + 512);
      }
      float d[2][2][4];  // [page][tokens 0-7 | 8-15][accumulator]
#pragma unroll
      for (int pp = 0; pp < 2; ++pp)
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          d[pp][t2][0] = d[pp][t2][1] = -kc0;
          d[pp][t2][2] = d[pp][t2][3] = -kc1;
        }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 qa0 = qa_s[32 * (2 * u)], qa1 = qa_s[32 * (2 * u + 1)];
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          uint32_t x0[4], x1[4];
          if (fold_k_offset<NG>()) {
            widen_k_biased(u4word(kw[pp][0], u), x0);
            widen_k_biased(u4word(kw[pp][1], u), x1);
          } else {
            widen_k(u4word(kw[pp][0], u), x0);
            widen_k(u4word(kw[pp][1], u), x1);
          }
          mma_f16(d[pp][0], qa0.x, qa0.y, qa0.z, qa0.w, x0[0], x0[1]);
          mma_f16(d[pp][1], qa0.x, qa0.y, qa0.z, qa0.w, x1[0], x1[1]);
          mma_f16(d[pp][0], qa1.x, qa1.y, qa1.z, qa1.w, x0[2], x0[3]);
          mma_f16(d[pp][1], qa1.x, qa1.y, qa1.z, qa1.w, x1[2], x1[3]);
        }
      }
      float sc[2][4];
#pragma unroll
      for (int pp = 0; pp < 2; ++pp)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float raw0 = e < 2 ? d[pp][0][e] : d[pp][1][e - 2];  // row r   (group g0)
          const float raw1 = e < 2 ? d[pp][0][e + 2] : d[pp][1][e];  // row r+8 (group g1)
          float part = 0.f;
          if (v0) {
            const float2 dm = h2f2(lds32(km_lane + SO + pp * cb + TK[e] * NG * 4));
            part = fmaf(dm.x, raw0, dm.y * qs0);
          }
          if (v1) {
            const float2 dm = h2f2(lds32(km_lane + SO + pp * cb + TK[e] * NG * 4 + 8));
            part += fmaf(dm.x, raw1, dm.y * qs1);
          }
          part += __shfl_xor_sync(0xffffffffu, part, 16);
          sc[pp][e] = part * scale_log2;
        }
      // first / last unit of the segment, or a page not loaded: mask
      if (jj == 0 || jj == cur_n - 1 || ph0 < 0 || ph1 < 0) {
#pragma unroll
        for (int pp = 0; pp < 2; ++pp)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pos = (pg0 + pp) * kPage + 2 * qd + TK[e];
            const bool in = (pp == 0 ? ph0 : ph1) >= 0 && pos >= rg.sink_end && pos < rg.rec_start;
            if (!in) sc[pp][e] = -INFINITY;
          }
      }
      float tmax = fmaxf(fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[0][2], sc[0][3])),
                         fmaxf(fmaxf(sc[1][0], sc[1][1]), fmaxf(sc[1][2], sc[1][3])));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      if (__any_sync(0xffffffffu, tmax > m_run + kLazyLog2)) {
        const float mnew = fmaxf(m_run, tmax);
        const float alpha = mnew == -INFINITY ? 1.f : ex2(m_run - mnew);
        const float aA = __shfl_sync(0xffffffffu, alpha, 4 * ((2 * qd) & 3));
        const float aB = __shfl_sync(0xffffffffu, alpha, 4 * ((2 * qd + 1) & 3));
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[k] *= (k & 1) ? aB : aA;
        mtacc[0] *= aA;
        mtacc[1] *= aB;
        l_run *= alpha;
        m_run = mnew;
      }
      const float mref = m_run == -INFINITY ? 0.f : m_run;
      float pr_[2][4];
#pragma unroll
      for (int pp = 0; pp < 2; ++pp)
#pragma unroll
        for (int e = 0; e < 4; ++e) pr_[pp][e] = ex2(sc[pp][e] - mref);  // masked: 0
      l_run += ((pr_[0][0] + pr_[0][1]) + (pr_[0][2] + pr_[0][3])) +
               ((pr_[1][0] + pr_[1][1]) + (pr_[1][2] + pr_[1][3]));
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        if ((pp == 0 ? ph0 : ph1) < 0) continue;  // not loaded: all its p are 0
        MetaRow<NG> vm[4];
        uint32_t mw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          vm[e].load_s(vm_lane + SO + pp * cb + TK[e] * NG * 4);
          mw[e] = mt_row ? lds32(vm_lane + SO + pp * cb + TK[e] * NG * 4 + mt_g * 4) : 0u;
        }
        uint32_t va[4], vb[4];
        ldsm_x4_trans(va, v_lane + SO + pp * cb + lm_off0);
        ldsm_x4_trans(vb, v_lane + SO + pp * cb + lm_off1);
        if ((pg0 + pp + 1) * kPage > cur_len) {  // slots at or past the length were never written
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if ((pg0 + pp) * kPage + 2 * qd + TK[e] >= cur_len) {
              vm[e].zero();
              mw[e] = 0u;
            }
        }
        const uint32_t p01 = pack_f16(pr_[pp][0], pr_[pp][1]) & p_keep;
        const uint32_t p23 = pack_f16(pr_[pp][2], pr_[pp][3]) & p_keep;
        mma_f16(mtacc, __byte_perm(mw[0], mw[1], mt_sel), 0u, __byte_perm(mw[2], mw[3], mt_sel),
                0u, p01, p23);
#pragma unroll
        for (int Pb = 0; Pb < 4; ++Pb) {
          const int grp = (Pb * 32) / GS;
          const uint32_t b0 = hmul2(p01, lo_lo(vm[0].get(grp), vm[1].get(grp)));
          const uint32_t b1 = hmul2(p23, lo_lo(vm[2].get(grp), vm[3].get(grp)));
          const uint32_t wlo = (Pb < 2) ? va[2 * Pb] : vb[2 * (Pb - 2)];
          const uint32_t whi = (Pb < 2) ? va[2 * Pb + 1] : vb[2 * (Pb - 2) + 1];
          uint32_t xl[4], xh[4];
          widen_v(wlo, xl);
          widen_v(whi, xh);
          mma_f16(&acc[Pb * 8], xl[0], xl[1], xh[0], xh[1], b0, b1);
          mma_f16(&acc[Pb * 8 + 4], xl[2], xl[3], xh[2], xh[3], b0, b1);
        }
      }
    } else if (ok) {
      // ================================= INT8 protected units (App. A.3)
      const int n_rec = cur_len > L.S ? cur_len - rg.rec_start : 0;
      const int ws_mod = L.R > 0 ? rg.rec_start % L.R : 0;
      const uint2* q8 = &sm.qb[qb].qfrag8[0][lane & 15];
      const uint32_t stg = stages_u32 + SO;
      const int sl0 = jj * kProtUnit + 2 * qd;  // this lane's slots sl0 + {0, 1, 8, 9}
      bool okv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) okv[e] = slot_valid(sl0 + TK[e], cur_len, L, ws_mod, n_rec);
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
      const float2 ksA = h2f2(lds32(stg + 2 * kProtUnit * D + 4 * qd));
      const float2 ksB = h2f2(lds32(stg + 2 * kProtUnit * D + 16 + 4 * qd));
      float sv[4] = {dq0[0] * ksA.x, dq0[1] * ksA.y, dq1[0] * ksB.x, dq1[1] * ksB.y};
#pragma unroll
      for (int e = 0; e < 4; ++e) sv[e] = okv[e] ? sv[e] * scale_log2 : -INFINITY;
      float tmax = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      if (__any_sync(0xffffffffu, tmax > m_run + kLazyLog2)) {  // lazy rescaling, as above
        const float mnew = fmaxf(m_run, tmax);
        const float alpha = mnew == -INFINITY ? 1.f : ex2(m_run - mnew);
        const float aA = __shfl_sync(0xffffffffu, alpha, 4 * ((2 * qd) & 3));
        const float aB = __shfl_sync(0xffffffffu, alpha, 4 * ((2 * qd + 1) & 3));
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[k] *= (k & 1) ? aB : aA;
        l_run *= alpha;
        m_run = mnew;
      }
      const float mref = m_run == -INFINITY ? 0.f : m_run;
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pv[e] = ex2(sv[e] - mref);
      l_run += (pv[0] + pv[1]) + (pv[2] + pv[3]);
      uint32_t vsA = lds32(stg + 2 * kProtUnit * D + 2 * kProtUnit + 4 * qd);
      uint32_t vsB = lds32(stg + 2 * kProtUnit * D + 2 * kProtUnit + 16 + 4 * qd);
      vsA &= (okv[0] ? 0x0000FFFFu : 0u) | (okv[1] ? 0xFFFF0000u : 0u);
      vsB &= (okv[2] ? 0x0000FFFFu : 0u) | (okv[3] ? 0xFFFF0000u : 0u);
      const uint32_t pb0 = hmul2(pack_f16(pv[0], pv[1]) & p_keep, vsA);
      const uint32_t pb1 = hmul2(pack_f16(pv[2], pv[3]) & p_keep, vsB);
      const uint32_t vbase = stg + kProtUnit * D;
#pragma unroll
      for (int c2 = 0; c2 < 4; ++c2) {  // pieces 2 c2 and 2 c2 + 1
        uint32_t vr[4];
        ldsm_x4_trans(vr, vbase + l8_row * D + 16 * ((2 * c2 + l8_pp) ^ l8_t));
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const uint32_t xlo = vr[2 * h2] ^ 0x80808080u, xhi = vr[2 * h2 + 1] ^ 0x80808080u;
          mma_f16(&acc[(2 * c2 + h2) * 4], i8pair(xlo, 0x4240u), i8pair(xlo, 0x4341u),
                  i8pair(xhi, 0x4240u), i8pair(xhi, 0x4341u), pb0, pb1);
        }
      }
    }
    ++my_n;
    // the unit's query fragments are no longer read; then refill the stage
    __syncwarp();
    int n_is = 0;
    if (lane == 0) {
      atomicAdd(&sm.qb_state[qb], ~0ull);  // one unit of the buffer's pair done (low half - 1)
      ProdM& pr = sm.prod[warp];
      if (pr.more) {
        issue(ST);
        n_is = 1;
        claim();
      }
    }
    inflight += __shfl_sync(0xffffffffu, n_is, 0) - 1;
    ++it;
  }
  if (cur_sig >= 0) retire();
}

}  // namespace

cudaError_t launch_stream_merge(const Layout& L, const int32_t* seq_lens, int num_seqs,
                                const float* part_o, const float* part_lse, int C, int by_cost,
                                bool overlap, uint16_t* out, float* out_lse, cudaStream_t st);

bool sm_supported(const Layout& L) { return L.d_h == SD && L.h_q == SG * L.h_kv; }

size_t sm_qprep_bytes(const Layout& L, int num_seqs) {
  return (size_t)num_seqs * L.h_kv * sizeof(QPrep);
}

template <int NG>
cudaError_t launch_sm_t(const Layout& L, const void* paged, const void* side, const uint16_t* q,
                        const int32_t* seq_lens, int num_seqs, const int32_t* block_table,
                        float sm_scale, void* qprep, float* part_o, float* part_lse,
                        uint16_t* out, float* out_lse, int32_t* status, cudaStream_t st) {
  constexpr int cb = 16 * SD + 128 * NG;
  constexpr size_t smem =
      ((sizeof(SmSmem) + 127) / 128) * 128 + (size_t)kMW * kMStages * kSPages * cb;
  static_assert(smem <= 227 * 1024, "shared memory of one CTA per SM");
  // once per device: the shared-memory attribute and the SM count
  static OnceSetup setup;
  int grid = 0;
  cudaError_t e = once_per_device(
      setup,
      [&](int dev, int* g) {
        cudaError_t r = cudaFuncSetAttribute(decode_sm_kernel<NG>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        int sms = 0;
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        *g = std::max(1, std::min(kMaxStreamCtas, sms));
        return r;
      },
      &grid);
  if (e != cudaSuccess) return e;
  const int pairs = num_seqs * L.h_kv;
  decode_sm_qprep_kernel<NG><<<pairs, 128, 0, st>>>(L, q, (QPrep*)qprep);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  decode_sm_kernel<NG><<<grid, kMThreads, smem, st>>>(
      L, (const uint8_t*)paged, (const uint8_t*)side, (const QPrep*)qprep, seq_lens, num_seqs,
      block_table, sm_scale * kLog2e, part_o, part_lse, out, out_lse, status);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // every pair's partials are merged by the separate merge kernel: a warp of
  // this kernel that merged them itself would hold up its claimed units for
  // the whole of the pair's eq. A1 (measured: slower than one more launch)
  e = launch_stream_merge(L, seq_lens, num_seqs, part_o, part_lse, grid, 0, false, out, out_lse,
                          st);
  return e;
}

cudaError_t launch_decode_sm(const Layout& L, const void* paged, const void* side,
                             const uint16_t* q, const int32_t* seq_lens, int num_seqs,
                             const int32_t* block_table, float sm_scale, void* qprep,
                             float* part_o, float* part_lse, uint16_t* out,
                             float* out_lse, int32_t* status, cudaStream_t st) {
  switch (L.d_h / L.g) {
    case 4:
      return launch_sm_t<4>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, qprep,
                            part_o, part_lse, out, out_lse, status, st);
    case 2:
      return launch_sm_t<2>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, qprep,
                            part_o, part_lse, out, out_lse, status, st);
    case 1:
      return launch_sm_t<1>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, qprep,
                            part_o, part_lse, out, out_lse, status, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kv4
