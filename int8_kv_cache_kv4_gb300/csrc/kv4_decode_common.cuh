// kv4_decode_common.cuh -- pieces shared by the decode kernels: shared-memory
// plan, online-softmax state, query staging, the protected (INT8 side cache)
// split, and the cross-warp merge that emits one split's partial result
// (KV4-RL App. A.3 eq. A1 is applied to these partials by the combine).
#pragma once
#include <math.h>

#include "kv4_common.cuh"

namespace kv4 {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// exact small-integer -> float (c < 2^23) without the conversion pipe
__device__ inline float u2f(uint32_t c) { return __uint_as_float(0x4B000000u | c) - 8388608.0f; }

template <int D, int G>
struct Smem {
  float q[G][2][D / 2 + 4];      // query, split in two halves (padded: no bank conflicts)
  float qsum[D / 32][G];         // per 32-channel block sum of q (combined per group)
  float p[kWarps][16][G];        // probabilities of the current tile, per warp
  float mrg_m[kWarps][G];
  float mrg_l[kWarps][G];
  union __align__(128) {
    float mrg_o[kWarps][G][D];      // per-warp unnormalised outputs (end of a split)
    uint32_t qfrag[8][32][4];       // mma.sync query fragments (start of a split)
    struct {
      uint16_t bq[16 * D];          // tcgen05: block-diagonal query operand (K-major)
      uint16_t bp[16 * D];          // tcgen05: probability operand P' (MN-major)
    } tc;
  };
  float tc_wmax[kWarps][G];         // tcgen05: per-warp tile maxima
  float tc_red[kWarps][G][5];       // tcgen05: per-warp l and offset-term partials
  int32_t tc_phys[2][8];            // tcgen05: physical pages of a staged tile
  uint64_t tc_bar[4];               // tcgen05: tile full x2, QK done, PV done
  uint32_t tc_tmem;                 // tcgen05: tensor-memory base address
  int32_t tc_abort;
  float mrg_mt[kWarps][G][D / 32];  // additive term per 32-channel block (tensor-core path)
  uint16_t qh[G][D];                // query as fp16 bits
  int32_t phys[kWarps][kStages];    // physical page of each in-flight stage
  int32_t ticket;
  uint64_t bar[kWarps][kStages];
};

// Online softmax state of one warp: lanes own D/32 output channels.
template <int D, int G>
struct WarpState {
  static constexpr int PD = D / 32;
  float m[G];       // running max (log2 domain), uniform across the warp
  float l[G];       // partial sum of p over this lane's tokens
  float acc[G][PD];  // unnormalised output channels [lane*PD, lane*PD+PD)
  __device__ void init() {
#pragma unroll
    for (int j = 0; j < G; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.f;
#pragma unroll
      for (int i = 0; i < PD; ++i) acc[j][i] = 0.f;
    }
  }
};

// Given this lane's score s[j] for token t = lane>>1 (both lanes of a token
// hold the same value; -inf = masked), update the running max, rescale, and
// publish p[t][j] to shared memory.
template <int D, int G>
__device__ inline void softmax_tile(WarpState<D, G>& ws, const float s[G], float (*p)[G],
                                    int lane) {
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float tmax = warp_max(s[j]);
    float mnew = fmaxf(ws.m[j], tmax);
    float alpha, pj;
    if (mnew == -INFINITY) {
      alpha = 1.f;
      pj = 0.f;
    } else {
      alpha = exp2f(ws.m[j] - mnew);
      pj = exp2f(s[j] - mnew);
    }
    ws.m[j] = mnew;
    ws.l[j] = ws.l[j] * alpha + ((lane & 1) ? 0.f : pj);
#pragma unroll
    for (int i = 0; i < WarpState<D, G>::PD; ++i) ws.acc[j][i] *= alpha;
    if ((lane & 1) == 0) p[lane >> 1][j] = pj;
  }
}

// ---------------------------------------------------------------- INT4 tile
// QK for one 16-token page chunk in shared memory.  Lane (t, half) covers
// channels [half*D/2, half*D/2 + D/2) of token t.
template <int D, int G>
__device__ inline void qk_int4(const Smem<D, G>& sm, const uint8_t* chunk, int g, int t, int half,
                               float s[G]) {
  const int ng = D / g;
  const uint8_t* krow = chunk + t * (D / 2);
  const uint32_t* kmeta = reinterpret_cast<const uint32_t*>(chunk + meta_off_k(D) + t * ng * 4);
#pragma unroll
  for (int j = 0; j < G; ++j) s[j] = 0.f;
  float part[G];
#pragma unroll
  for (int j = 0; j < G; ++j) part[j] = 0.f;
  constexpr int WORDS = D / 16;  // 8 nibbles per word, D/2 channels per lane
#pragma unroll
  for (int w = 0; w < WORDS; ++w) {
    // channels half * D/2 + 8 w .. + 7: one word of the K row
    const uint32_t word =
        *reinterpret_cast<const uint32_t*>(krow + k_row_byte(half * (D / 2) + 8 * w, D));
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float c = u2f((word >> (4 * n)) & 0xFu);
      const int k = w * 8 + n;
#pragma unroll
      for (int j = 0; j < G; ++j) part[j] = fmaf(sm.q[j][half][k], c, part[j]);
    }
    const int ch_end = half * (D / 2) + w * 8 + 8;  // channel after this word
    if (ch_end % g == 0 || w == WORDS - 1) {
      const int grp = (ch_end - 1) / g;
      const uint32_t mt = kmeta[grp];
      const float delta = f16_bits_to_f32(mt & 0xFFFFu);
      const float off = f16_bits_to_f32(mt >> 16);
      // sum of q over this lane's part of the group
      const int lo = max(grp * g, half * (D / 2)) / 32, hi = min((grp + 1) * g, half * (D / 2) + D / 2) / 32;
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float qs = 0.f;
        for (int bq = lo; bq < hi; ++bq) qs += sm.qsum[bq][j];
        s[j] = fmaf(delta, part[j], fmaf(off, qs, s[j]));
        part[j] = 0.f;
      }
    }
  }
}

// PV for one 16-token page: lane owns channels [lane*PD, lane*PD + PD).
template <int D, int G>
__device__ inline void pv_int4(WarpState<D, G>& ws, const uint8_t* chunk, int g, const float (*p)[G],
                               int lane, uint32_t tok_mask) {
  constexpr int PD = D / 32;
  const int c0 = lane * PD;
  const int grp = c0 / g;
  const uint8_t* vcodes = chunk + codes_off_v(D);
  for (int t = 0; t < kPage; ++t) {
    if (!((tok_mask >> (2 * t)) & 1u)) continue;  // masked slot: may hold stale bytes
    uint32_t bits;
    if (PD == 4)
      bits = *reinterpret_cast<const uint16_t*>(vcodes + t * (D / 2) + row_byte(c0 / 2, t, D));
    else
      bits = vcodes[t * (D / 2) + row_byte(c0 / 2, t, D)];
    const float delta =
        f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(chunk + v_delta_byte(t, grp, D, g)));
    const float off =
        f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(chunk + v_offset_byte(t, grp, D, g)));
    float v[PD];
#pragma unroll
    for (int i = 0; i < PD; ++i) v[i] = fmaf(delta, u2f((bits >> (4 * i)) & 0xFu), off);
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const float pj = p[t][j];
#pragma unroll
      for (int i = 0; i < PD; ++i) ws.acc[j][i] = fmaf(pj, v[i], ws.acc[j][i]);
    }
  }
}

// ------------------------------------------------------------ merge + store
// Publish one warp's CUDA-core online-softmax state to shared memory.
template <int D, int G>
__device__ inline void write_state(Smem<D, G>& sm, WarpState<D, G>& ws, int warp, int lane) {
  constexpr int PD = D / 32;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const float lsum = warp_sum(ws.l[j]);
    if (lane == 0) {
      sm.mrg_m[warp][j] = ws.m[j];
      sm.mrg_l[warp][j] = lsum;
    }
#pragma unroll
    for (int i = 0; i < PD; ++i) sm.mrg_o[warp][j][lane * PD + i] = ws.acc[j][i];
    if (lane < D / 32) sm.mrg_mt[warp][j][lane] = 0.f;
  }
}

// Merge the warps' states (each: running max m, sum l, unnormalised output o
// plus a per-32-channel-block additive term mt) and store the split's locally
// normalised output and natural-log normaliser.
template <int D, int G>
__device__ inline void merge_store(Smem<D, G>& sm, float* part_o, float* part_lse, long long row0,
                                   int n_split, int split) {
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int j = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.mrg_m[w][j]);
    float Lt = 0.f, o = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = sm.mrg_m[w][j];
        if (mw == -INFINITY) continue;
        const float sc = exp2f(mw - M);
        Lt += sm.mrg_l[w][j] * sc;
        o += (sm.mrg_o[w][j][d] + sm.mrg_mt[w][j][d / 32]) * sc;
      }
    }
    const long long row = row0 + j;  // (seq * h_q + head)
    const bool empty = !(Lt > 0.f);
    part_o[(row * n_split + split) * D + d] = empty ? 0.f : o / Lt;
    if (d == 0) part_lse[row * n_split + split] = empty ? -INFINITY : (M + log2f(Lt)) * kLn2;
  }
}

// Eq. A1 over the n_split partials of `G` consecutive rows, done by the last
// CTA of a (sequence, kv head) to finish.  An atomic ticket per pair counts
// finished CTAs: the CTA barrier makes every thread's partial writes visible
// to thread 0, whose device-scope fence then orders them (cumulatively)
// before its ticket increment; the last CTA fences again before reading.
template <int D, int G>
__device__ inline void combine_if_last(Smem<D, G>& sm, int32_t* tickets, int pair,
                                       const float* part_o, const float* part_lse,
                                       long long row0, int n_split, uint16_t* out,
                                       float* out_lse) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    sm.ticket = atomicAdd(&tickets[pair], 1);
    if (sm.ticket == n_split - 1) __threadfence();
  }
  __syncthreads();
  if (sm.ticket != n_split - 1) return;
  constexpr int PD = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < G; j += kWarps) {
    const long long row = row0 + j;
    const float* lse = part_lse + row * n_split;
    float M = -INFINITY;
    for (int r = lane; r < n_split; r += 32) M = fmaxf(M, __ldcg(lse + r));
    M = warp_max(M);
    float acc[PD];
#pragma unroll
    for (int i = 0; i < PD; ++i) acc[i] = 0.f;
    float Zl = 0.f;
    if (M != -INFINITY) {
      for (int r0 = 0; r0 < n_split; r0 += 32) {
        const int r = r0 + lane;
        const float z = r < n_split ? __ldcg(lse + r) : -INFINITY;
        const float wl = z == -INFINITY ? 0.f : exp2f((z - M) * kLog2e);
        Zl += wl;
        const int nr = min(32, n_split - r0);
        // four parts' outputs in flight at a time
        for (int rr = 0; rr < nr; rr += 4) {
          float wv[4], o[4][PD];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            wv[u] = __shfl_sync(0xffffffffu, wl, (rr + u) & 31);
            const bool use = rr + u < nr && wv[u] != 0.f;
            const float* op = part_o + (row * n_split + r0 + rr + u) * D + lane * PD;
#pragma unroll
            for (int i = 0; i < PD; ++i) o[u][i] = use ? __ldcg(op + i) : 0.f;
            if (!use) wv[u] = 0.f;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < PD; ++i) acc[i] = fmaf(wv[u], o[u][i], acc[i]);
        }
      }
    }
    const float Z = warp_sum(Zl);
    const bool empty = !(Z > 0.f);
#pragma unroll
    for (int i = 0; i < PD; ++i)
      out[row * D + lane * PD + i] = f32_to_bf16_bits(empty ? 0.f : acc[i] / Z);
    if (out_lse && lane == 0) out_lse[row] = empty ? -INFINITY : M + logf(Z);
  }
}

template <int D, int G>
__device__ inline void load_query(Smem<D, G>& sm, const uint16_t* q, long long row0) {
  // A warp's 32 lanes hold 32 consecutive channels of one head, so the
  // per-32-channel query sums are warp reductions.
  const int lane = threadIdx.x & 31;
  constexpr int kIters = (G * D + kThreads - 1) / kThreads;
  uint16_t raw[kIters];
#pragma unroll
  for (int it = 0; it < kIters; ++it) {  // all loads in flight first
    const int idx = it * kThreads + threadIdx.x;
    raw[it] = idx < G * D ? q[(row0 + idx / D) * D + idx % D] : (uint16_t)0;
  }
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int idx = it * kThreads + threadIdx.x;
    const bool ok = idx < G * D;
    const int j = idx / D, d = idx % D;
    const float x = bf16_bits_to_f32(raw[it]);
    if (ok) {
      sm.qh[j][d] = __half_as_ushort(__float2half_rn(x));
      sm.q[j][d / (D / 2)][d % (D / 2)] = x;
    }
    const float s = warp_sum(x);
    if (ok && lane == 0) sm.qsum[d / 32][j] = s;
  }
  __syncthreads();
}

// ----------------------------------------- protected (INT8 side) split
// Positions of the sink and recent windows (KV4-RL Sec. 5.2), read from the
// INT8 side cache (App. A.3 "Protected path"): the k-th protected split covers
// protected positions [k*prot_per_split, (k+1)*prot_per_split).  CUDA-core
// fp32 math; lanes (t, half) as in the INT4 path for QK, lane-owned channels
// for PV.
template <int D, int G>
__device__ inline void prot_split(Smem<D, G>& sm, WarpState<D, G>& ws, const Layout& L,
                                  const uint8_t* __restrict__ side, int b, int h,
                                  const Regions& rg, int k, int prot_per_split, float scale_log2,
                                  int warp, int lane) {
  const int t = lane >> 1, half = lane & 1;
  const int i_lo = k * prot_per_split;
  const int i_hi = min(rg.n_prot, i_lo + prot_per_split);
  const int NS = L.S + L.R;
  const uint8_t* blk = side + ((long long)b * L.h_kv + h) * side_block_bytes(D, L.S, L.R);
  const int8_t* k8 = reinterpret_cast<const int8_t*>(blk);
  const int8_t* v8 = reinterpret_cast<const int8_t*>(blk + (long long)NS * D);
  const uint16_t* ks = reinterpret_cast<const uint16_t*>(blk + 2LL * NS * D);
  const uint16_t* vs = ks + side_scale_entries(L.S, L.R);
  constexpr int PD = D / 32;
  for (int base = i_lo + warp * 16; base < i_hi; base += kWarps * 16) {
    const int i = base + t;
    const bool tok_ok = i < i_hi;
    const int slot = tok_ok ? side_slot(prot_pos(rg, i), L.S, L.R) : 0;
    const int ntok = min(16, i_hi - base);
    // every global load of this 16-position block is issued before any use;
    // V scales stay packed as fp16 pairs to keep the register count down
    // this lane's half of the K row: pieces half*D/32 + i, stored swizzled
    const int8_t* krow = k8 + (long long)slot * D;
    auto kpiece = [&](int i) {
      return tok_ok ? *reinterpret_cast<const uint4*>(krow + side_byte(16 * (half * (D / 32) + i), slot, D))
                    : make_uint4(0u, 0u, 0u, 0u);
    };
    uint4 kraw0 = kpiece(0);
    uint4 kraw1 = kpiece(1);
    const float ksc = tok_ok ? f16_bits_to_f32(ks[slot]) : 0.f;
    uint32_t vword[16];
    uint32_t vsc2[8];
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
      const bool ok = tt < ntok;
      const int slot2 = ok ? side_slot(prot_pos(rg, base + tt), L.S, L.R) : 0;
      const uint32_t sbits = ok ? (uint32_t)vs[slot2] : 0u;
      if (tt & 1)
        vsc2[tt >> 1] |= sbits << 16;
      else
        vsc2[tt >> 1] = sbits;
      const int8_t* vp = v8 + (long long)slot2 * D + side_byte(lane * PD, slot2, D);
      if (PD == 4)
        vword[tt] = ok ? *reinterpret_cast<const uint32_t*>(vp) : 0u;
      else
        vword[tt] = ok ? *reinterpret_cast<const uint16_t*>(vp) : 0u;
    }
    float s[G];
#pragma unroll
    for (int j = 0; j < G; ++j) s[j] = 0.f;
#pragma unroll
    for (int w = 0; w < D / 32; ++w) {
      if (w == 2) {  // second half of this lane's 64 channels
        kraw0 = kpiece(2);
        kraw1 = kpiece(3);
      }
      const uint4 kr = (w & 1) ? kraw1 : kraw0;
      const uint32_t words[4] = {kr.x, kr.y, kr.z, kr.w};
#pragma unroll
      for (int wi = 0; wi < 4; ++wi)
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          const float c = (float)(int8_t)((words[wi] >> (8 * n)) & 0xFFu);
#pragma unroll
          for (int j = 0; j < G; ++j) s[j] = fmaf(sm.q[j][half][16 * w + 4 * wi + n], c, s[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
      s[j] *= ksc;
      s[j] += __shfl_xor_sync(0xffffffffu, s[j], 1);
      s[j] = tok_ok ? s[j] * scale_log2 : -INFINITY;
    }
    softmax_tile<D, G>(ws, s, sm.p[warp], lane);
    __syncwarp();
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
      if (tt < ntok) {
        float v[PD];
        const float vsc = f16_bits_to_f32((vsc2[tt >> 1] >> (16 * (tt & 1))) & 0xFFFFu);
#pragma unroll
        for (int ii = 0; ii < PD; ++ii) v[ii] = vsc * (float)(int8_t)((vword[tt] >> (8 * ii)) & 0xFFu);
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float pj = sm.p[warp][tt][j];
#pragma unroll
          for (int ii = 0; ii < PD; ++ii) ws.acc[j][ii] = fmaf(pj, v[ii], ws.acc[j][ii]);
        }
      }
    }
    __syncwarp();
  }
}

}  // namespace kv4
