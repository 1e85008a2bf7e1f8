// kv4_decode_mma.cu -- tensor-core variant of the INT4-region split of the
// mixed-cache decode (KV4-RL Sec. 5.3, eq. 5.1; App. A.3) for head_dim 128
// and 4 query heads per kv head (the Qwen3/Llama-3 layers the paper runs).
//
// The TMA staging, split plan, protected (INT8) split and merge are those of
// the CUDA-core kernel.  What changes is the per-page math, which moves from
// fp32 FMAs onto warp-level tensor-core MMAs (m16n8k16):
//
// QK^T, fp16 in, fp32 accumulate.  Rows of the 16-row A operand are the
//   (group, head) pairs -- 4 groups x 4 heads at g = 32 -- and A holds each
//   head's query restricted to that group's channels (block diagonal), so one
//   accumulator row is the group-partial dot product  D_g = sum_{d in g} q_d c_d.
//   B is the page's 4-bit codes widened in registers to exact fp16 integers
//   (magic-number OR, then one fp16 fma per pair).  The score then follows
//   eq. 5.1 per group:  s = sum_g Delta_g * D_g + m_g * sum_{d in g} q_d,
//   so the codes enter the product exactly.  16 MMAs per 16-token page.  The
//   bf16 query converts to fp16 without loss (|q| within fp16's normal range).
//
// PV, fp16 in, fp32 accumulate.  A is the page's V codes transposed
//   (channels x tokens), fetched with ldmatrix.trans and widened to the exact
//   centred values c - 8 in fp16; B is P' = p * Delta_v per group (rounded to
//   fp16 once).  The offset term sum_t p_t (m_t + 8 Delta_t) is accumulated on
//   the CUDA cores per group.  8 MMAs per page.
//
// The QK accumulator layout equals the PV operand layout for the tokens each
// lane holds, so probabilities never leave registers.
#include "kv4_decode_common.cuh"
#include "kv4_mma.cuh"

namespace kv4 {

constexpr int D128 = 128, G4 = 4;
// Two page stages per warp and the query fragments in shared memory keep the
// kernel at <= 102 registers and ~38 KB of shared memory, so five CTAs (20
// warps) share an SM.
constexpr int kStagesMma = 2;

template <int NG>
__global__ void __launch_bounds__(kThreads, 5) decode_mma_kernel(
    Layout L, const uint8_t* __restrict__ paged, const uint8_t* __restrict__ side,
    const uint16_t* __restrict__ q, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ block_table, float scale_log2, int n4, int pages_per_split,
    int prot_per_split, float* __restrict__ part_o, float* __restrict__ part_lse,
    int32_t* __restrict__ tickets, uint16_t* __restrict__ out, float* __restrict__ out_lse,
    int32_t* status) {
  constexpr int D = D128, G = G4;
  constexpr int GS = D / NG;  // channels per INT4 group
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<D, G>& sm = *reinterpret_cast<Smem<D, G>*>(smem_raw);
  constexpr int cb = 16 * D + 128 * NG;
  uint8_t* stage_base = smem_raw + ((sizeof(Smem<D, G>) + 127) / 128) * 128;
  uint32_t* qfrag = reinterpret_cast<uint32_t*>(stage_base + (size_t)kWarps * kStagesMma * cb);

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n_split = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row0 = (long long)b * L.h_q + (long long)h * G;

  int len = seq_lens[b];
  if (len < 0 || len > L.max_pages * kPage) {
    if (threadIdx.x == 0 && split == 0 && h == 0) set_status(status, KV4_STATUS_BAD_LEN);
    len = 0;
  }
  const Regions rg = regions(len, L.S, L.R);
  const int first_page = rg.sink_end / kPage;
  const int end_page = (rg.rec_start + kPage - 1) / kPage;
  const int p_lo = first_page + split * pages_per_split;
  const int p_hi = min(end_page, p_lo + pages_per_split);
  const bool empty_int4 =
      split < n4 && !(rg.rec_start > rg.sink_end && p_hi > p_lo);
  const bool empty_prot = split >= n4 && (split - n4) * prot_per_split >= rg.n_prot;
  if (empty_int4 || empty_prot) {
    // nothing to attend: an empty part (weight 0 in the merge)
    if (threadIdx.x < G) part_lse[(row0 + threadIdx.x) * n_split + split] = -INFINITY;
    combine_if_last<D, G>(sm, tickets, b * L.h_kv + h, part_o, part_lse, row0, n_split, out,
                          out_lse);
    return;
  }
  load_query(sm, q, row0);

  if (split >= n4) {
    WarpState<D, G> ws;
    ws.init();
    prot_split<D, G>(sm, ws, L, side, b, h, rg, split - n4, prot_per_split, scale_log2, warp,
                     lane);
    write_state<D, G>(sm, ws, warp, lane);
    merge_store<D, G>(sm, part_o, part_lse, row0, n_split, split);
    combine_if_last<D, G>(sm, tickets, b * L.h_kv + h, part_o, part_lse, row0, n_split, out,
                          out_lse);
    return;
  }

  // ------------------------------------------------ per-lane constant setup
  const int r = lane >> 2, qd = lane & 3;
  const int j = r & 3;                        // this lane's softmax head
  const int g0 = r >> 2, g1 = g0 + 2;         // groups of QK rows r and r+8
  const bool v0 = g0 < NG, v1 = g1 < NG;
  // Q operand fragments: block-diagonal (group, head) rows, fp16.  Identical
  // for the CTA's four warps: built once into shared memory ([s][lane][4]
  // words) and read back per k-step.
  for (int idx = threadIdx.x; idx < 8 * 32 * 4; idx += kThreads) {
    const int s = idx >> 7, ln = (idx >> 2) & 31, k = idx & 3;
    const int rr = ln >> 2, qq = ln & 3;
    const int row = rr + 8 * (k & 1);              // A rows r (k = 0, 2) and r + 8 (k = 1, 3)
    const int grp = row >> 2, jj = row & 3;
    const int base = 32 * qq + 8 * (s >> 1) + 2 * (s & 1) + ((k & 2) ? 1 : 0);
    uint32_t w = 0u;
    if (grp < NG) {
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int d = base + 4 * e2;               // k-index 2qd+e2 (k<2) or 2qd+8+e2 (k>=2)
        if (d / GS == grp) w |= (uint32_t)sm.qh[jj][d] << (16 * e2);
      }
    }
    qfrag[idx] = w;
  }
  __syncthreads();
  const uint4* qa_s = reinterpret_cast<const uint4*>(qfrag) + lane;  // + 32 * s
  float qs0 = 0.f, qs1 = 0.f;
  for (int bq = 0; bq < D / 32; ++bq) {
    if (v0 && (bq * 32) / GS == g0) qs0 += sm.qsum[bq][j];
    if (v1 && (bq * 32) / GS == g1) qs1 += sm.qsum[bq][j];
  }

  // ------------------------------------------------------ running state
  float m_run = -INFINITY, l_run = 0.f;
  constexpr int NGH = NG > 1 ? NG / 2 : 1;  // m-term groups per lane half
  const int mt_g0 = (r >= 4) ? NG / 2 : 0;
  const bool mt_on = (r < 4) || NG > 1;
  float mt_m[NGH], mt_d[NGH];  // sum_t p_t m_t and sum_t p_t Delta_t per handled group
#pragma unroll
  for (int i = 0; i < NGH; ++i) mt_m[i] = mt_d[i] = 0.f;
  float acc[4][2][4];
#pragma unroll
  for (int G_ = 0; G_ < 4; ++G_)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[G_][hh][i] = 0.f;

  // ------------------------------------------------------ page pipeline
  const int n_my = rg.rec_start > rg.sink_end && p_hi > p_lo + warp
                       ? (p_hi - p_lo - warp + kWarps - 1) / kWarps
                       : 0;
  uint8_t* my_stages = stage_base + (size_t)warp * kStagesMma * cb;
  const int32_t* bt_row = block_table + (long long)b * L.max_pages;
  if (lane == 0) {
    for (int st = 0; st < kStagesMma; ++st) mbar_init(&sm.bar[warp][st], 1);
    fence_mbar_init();
  }
  __syncwarp();
  // Lane 0 issues the bulk copies; the block-table entry of each page is
  // read one iteration before its copy is issued, so the issue never waits
  // on global-memory latency.
  auto issue = [&](int i, int phys) {
    uint64_t* bar = &sm.bar[warp][i % kStagesMma];
    const bool good = phys >= 0 && phys < L.num_pages;
    sm.phys[warp][i % kStagesMma] = good ? phys : -1;  // published by the arrive below
    if (good) {
      mbar_arrive_expect_tx(bar, (uint32_t)cb);
      bulk_g2s(my_stages + (size_t)(i % kStagesMma) * cb,
               paged + ((long long)phys * L.h_kv + h) * cb, (uint32_t)cb, bar);
    } else {
      set_status(status, KV4_STATUS_BAD_PAGE);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
    }
  };
  int next_phys = -1;  // lane 0: block-table entry of page i + kStagesMma
  if (lane == 0) {
    for (int i = 0; i < min(kStagesMma, n_my); ++i) issue(i, bt_row[p_lo + warp + i * kWarps]);
    if (kStagesMma < n_my) next_phys = bt_row[p_lo + warp + kStagesMma * kWarps];
  }

  // ldmatrix row addresses (relative to the V code block): matrix mi = lane/8
  // holds tokens (mi&1)*8 + 0..7 of channel piece P = mi>>1 (+2 on the second
  // load); pieces are XOR-swizzled by token pair.
  const int lm_tok = ((lane >> 3) & 1) * 8 + (lane & 7);
  const int lm_p = lane >> 4;
  const uint32_t lm_off0 = lm_tok * 64 + 16 * ((lm_p) ^ ((lm_tok >> 1) & 3));
  const uint32_t lm_off1 = lm_tok * 64 + 16 * ((lm_p + 2) ^ ((lm_tok >> 1) & 3));
  const int tk[4] = {2 * qd, 2 * qd + 1, 8 + 2 * qd, 9 + 2 * qd};  // this lane's tokens

  const uint32_t p_keep = (r < 4) ? 0xFFFFFFFFu : 0u;  // lanes r >= 4 feed zero PV columns
  for (int i = 0; i < n_my; ++i) {
    const int pg = p_lo + warp + i * kWarps;
    const bool ok =
        __all_sync(0xffffffffu, mbar_wait(&sm.bar[warp][i % kStagesMma], (i / kStagesMma) & 1));
    const bool valid = ok && sm.phys[warp][i % kStagesMma] >= 0;
    if (!ok && lane == 0) set_status(status, KV4_STATUS_BAD_PAGE);
    const uint8_t* chunk = my_stages + (size_t)(i % kStagesMma) * cb;
    if (valid) {
      // slots at or beyond the sequence length were never written: their
      // metadata may be any bit pattern, so it is zeroed before use
      const bool tail = (pg + 1) * kPage > len;
      // ---------------- QK^T on tensor cores
      const uint4 k0 = k_block_words(chunk + r * 64, qd, D);        // block qd of row r
      const uint4 k1 = k_block_words(chunk + (r + 8) * 64, qd, D);  // ... and of row r + 8
      // four independent accumulator chains (tokens 0-7 / 8-15 x even / odd
      // k-steps), summed afterwards
      float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
      float e0[4] = {0.f, 0.f, 0.f, 0.f}, e1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t x0[4], x1[4];
        widen_k(u4word(k0, u), x0);
        widen_k(u4word(k1, u), x1);
        const uint4 qa0 = qa_s[32 * (2 * u)], qa1 = qa_s[32 * (2 * u + 1)];
        // k-steps 2u and 2u+1 use pairs (0,1) and (2,3) of word u
        mma_f16(d0, qa0.x, qa0.y, qa0.z, qa0.w, x0[0], x0[1]);
        mma_f16(d1, qa0.x, qa0.y, qa0.z, qa0.w, x1[0], x1[1]);
        mma_f16(e0, qa1.x, qa1.y, qa1.z, qa1.w, x0[2], x0[3]);
        mma_f16(e1, qa1.x, qa1.y, qa1.z, qa1.w, x1[2], x1[3]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        d0[k] += e0[k];
        d1[k] += e1[k];
      }
      // ---------------- scores (eq. 5.1 per group) for this lane's 4 tokens
      const float draw0[4] = {d0[0], d0[1], d1[0], d1[1]};  // row r   (group g0)
      const float draw1[4] = {d0[2], d0[3], d1[2], d1[3]};  // row r+8 (group g1)
      const uint8_t* kmeta = chunk + meta_off_k(D);
      float sc[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float part = 0.f;
        if (v0) {
          const float2 dm = h2f2(*reinterpret_cast<const uint32_t*>(kmeta + (tk[e] * NG + g0) * 4));
          part = fmaf(dm.x, draw0[e], dm.y * qs0);
        }
        if (v1) {
          const float2 dm = h2f2(*reinterpret_cast<const uint32_t*>(kmeta + (tk[e] * NG + g1) * 4));
          part += fmaf(dm.x, draw1[e], dm.y * qs1);
        }
        sc[e] = part;
      }
      const bool interior = pg * kPage >= rg.sink_end && (pg + 1) * kPage <= rg.rec_start;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sc[e] += __shfl_xor_sync(0xffffffffu, sc[e], 16);
        sc[e] *= scale_log2;
      }
      if (!interior) {  // first / last page of the region: mask positions outside it
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pos = pg * kPage + tk[e];
          if (!(pos >= rg.sink_end && pos < rg.rec_start)) sc[e] = -INFINITY;
        }
      }
      // metadata for PV, loaded early so its latency overlaps the softmax
      MetaRow<NG> vm[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) vm[e].load_v(chunk, tk[e], D);
      uint32_t mtw[4][NGH];
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int gi = 0; gi < NGH; ++gi) mtw[e][gi] = vmeta_word(chunk, tk[e], mt_g0 + gi, D, GS);
      // ---------------- online softmax for head j over this page
      float tmax = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      const float mnew = fmaxf(m_run, tmax);
      const float mref = mnew == -INFINITY ? 0.f : mnew;
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) p[e] = ex2(sc[e] - mref);  // masked: ex2(-inf) = 0
      if (__any_sync(0xffffffffu, mnew > m_run)) {
        const float alpha = ex2(m_run - mref);
        const float aA = __shfl_sync(0xffffffffu, alpha, 4 * ((2 * qd) & 3));
        const float aB = __shfl_sync(0xffffffffu, alpha, 4 * ((2 * qd + 1) & 3));
#pragma unroll
        for (int G_ = 0; G_ < 4; ++G_)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            acc[G_][hh][0] *= aA;
            acc[G_][hh][1] *= aB;
            acc[G_][hh][2] *= aA;
            acc[G_][hh][3] *= aB;
          }
#pragma unroll
        for (int gi = 0; gi < NGH; ++gi) {
          mt_m[gi] *= alpha;
          mt_d[gi] *= alpha;
        }
        l_run *= alpha;
        m_run = mnew;
      }
      l_run += (p[0] + p[1]) + (p[2] + p[3]);

      // ---------------- PV on tensor cores
      uint32_t va[4], vb[4];
      const uint32_t vbase = smem_u32(chunk + codes_off_v(D));
      ldsm_x4_trans(va, vbase + lm_off0);  // pieces 0,1: (tok lo, P0) (tok hi, P0) (lo, P1) (hi, P1)
      ldsm_x4_trans(vb, vbase + lm_off1);  // pieces 2,3
      if (tail) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (pg * kPage + tk[e] >= len) vm[e].zero();
      }
      // offset term: sum_t p_t (m_t + 8 Delta_t) per group, fp32; this lane
      // handles groups [mt_g0, mt_g0 + NGH)
      if (mt_on) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int gi = 0; gi < NGH; ++gi) {
            const float2 dm = h2f2(tail && pg * kPage + tk[e] >= len ? 0u : mtw[e][gi]);
            mt_d[gi] = fmaf(p[e], dm.x, mt_d[gi]);
            mt_m[gi] = fmaf(p[e], dm.y, mt_m[gi]);
          }
      }
      // P' = p * Delta_v per group, formed in fp16x2 (token pairs)
      const uint32_t p01 = pack_f16(p[0], p[1]) & p_keep;
      const uint32_t p23 = pack_f16(p[2], p[3]) & p_keep;
#pragma unroll
      for (int P = 0; P < 4; ++P) {
        const int grp = (P * 32) / GS;
        const uint32_t b0 = hmul2(p01, lo_lo(vm[0].get(grp), vm[1].get(grp)));
        const uint32_t b1 = hmul2(p23, lo_lo(vm[2].get(grp), vm[3].get(grp)));
        const uint32_t wlo = (P < 2) ? va[2 * P] : vb[2 * (P - 2)];
        const uint32_t whi = (P < 2) ? va[2 * P + 1] : vb[2 * (P - 2) + 1];
        uint32_t xl[4], xh[4];
        widen_v(wlo, xl);
        widen_v(whi, xh);
        mma_f16(acc[P][0], xl[0], xl[1], xh[0], xh[1], b0, b1);
        mma_f16(acc[P][1], xl[2], xl[3], xh[2], xh[3], b0, b1);
      }
    }
    __syncwarp();
    if (lane == 0 && i + kStagesMma < n_my) {
      issue(i + kStagesMma, next_phys);
      if (i + kStagesMma + 1 < n_my) next_phys = bt_row[p_lo + warp + (i + kStagesMma + 1) * kWarps];
    }
  }

  // ------------------------------------------------ publish warp state
  float lsum = (r < 4) ? l_run : 0.f;
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
  float mt[NGH];
#pragma unroll
  for (int gi = 0; gi < NGH; ++gi) {
    mt[gi] = fmaf(8.f, mt_d[gi], mt_m[gi]);
    mt[gi] += __shfl_xor_sync(0xffffffffu, mt[gi], 1);
    mt[gi] += __shfl_xor_sync(0xffffffffu, mt[gi], 2);
  }
  if (qd == 0 && r < 4) {
    sm.mrg_m[warp][j] = m_run;
    sm.mrg_l[warp][j] = lsum;
  }
  if (qd == 0 && mt_on) {
#pragma unroll
    for (int gi = 0; gi < NGH; ++gi) {
      const int grp = mt_g0 + gi;
      for (int blk = grp * (GS / 32); blk < (grp + 1) * (GS / 32); ++blk)
        sm.mrg_mt[warp][j][blk] = mt[gi];
    }
  }
  if (qd < 2) {
    const int hA = 2 * qd, hB = 2 * qd + 1;
#pragma unroll
    for (int P = 0; P < 4; ++P)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int d = 32 * P + 4 * r + 2 * hh;
        sm.mrg_o[warp][hA][d] = acc[P][hh][0];
        sm.mrg_o[warp][hB][d] = acc[P][hh][1];
        sm.mrg_o[warp][hA][d + 1] = acc[P][hh][2];
        sm.mrg_o[warp][hB][d + 1] = acc[P][hh][3];
      }
  }
  merge_store<D, G>(sm, part_o, part_lse, row0, n_split, split);
  combine_if_last<D, G>(sm, tickets, b * L.h_kv + h, part_o, part_lse, row0, n_split, out,
                        out_lse);
}

template <int NG>
cudaError_t launch_mma_t(const Layout& L, const void* paged, const void* side, const uint16_t* q,
                         const int32_t* seq_lens, int num_seqs, const int32_t* block_table,
                         float sm_scale, int n4, int pages_per_split, int n8, int prot_per_split,
                         float* part_o, float* part_lse, int32_t* tickets, uint16_t* out,
                         float* out_lse, int32_t* status, cudaStream_t st) {
  constexpr int cb = 16 * D128 + 128 * NG;
  const size_t smem = ((sizeof(Smem<D128, G4>) + 127) / 128) * 128 +
                      (size_t)kWarps * kStagesMma * cb + 8 * 32 * 4 * sizeof(uint32_t);
  static OnceSetup setup;  // the shared-memory attribute, once per device
  int unused = 0;
  cudaError_t e = once_per_device(
      setup,
      [&](int, int*) {
        return cudaFuncSetAttribute(decode_mma_kernel<NG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem);
      },
      &unused);
  if (e != cudaSuccess) return e;
  dim3 grid(n4 + n8, L.h_kv, num_seqs);
  decode_mma_kernel<NG><<<grid, kThreads, smem, st>>>(
      L, (const uint8_t*)paged, (const uint8_t*)side, q, seq_lens, block_table,
      sm_scale * kLog2e, n4, pages_per_split, prot_per_split, part_o, part_lse, tickets, out,
      out_lse, status);
  return cudaGetLastError();
}

bool mma_supported(const Layout& L) { return L.d_h == 128 && L.h_q == 4 * L.h_kv; }

cudaError_t launch_decode_mma(const Layout& L, const void* paged, const void* side,
                              const uint16_t* q, const int32_t* seq_lens, int num_seqs,
                              const int32_t* block_table, float sm_scale, int n4,
                              int pages_per_split, int n8, int prot_per_split, float* part_o,
                              float* part_lse, int32_t* tickets, uint16_t* out, float* out_lse,
                              int32_t* status, cudaStream_t st) {
  switch (L.d_h / L.g) {
    case 4:
      return launch_mma_t<4>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, n4,
                             pages_per_split, n8, prot_per_split, part_o, part_lse, tickets, out,
                             out_lse, status, st);
    case 2:
      return launch_mma_t<2>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, n4,
                             pages_per_split, n8, prot_per_split, part_o, part_lse, tickets, out,
                             out_lse, status, st);
    case 1:
      return launch_mma_t<1>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, n4,
                             pages_per_split, n8, prot_per_split, part_o, part_lse, tickets, out,
                             out_lse, status, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kv4
