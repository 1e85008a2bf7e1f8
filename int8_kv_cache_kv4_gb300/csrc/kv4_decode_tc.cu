// kv4_decode_tc.cu -- fifth-generation tensor-core (tcgen05 / tensor memory)
// variant of the INT4-region split of the mixed-cache decode (KV4-RL
// Sec. 5.3, eq. 5.1; App. A.3) for head_dim 128 and 4 query heads per kv head.
//
// A CTA (4 warps) streams its split's pages in tiles of 8 pages = 128 tokens,
// staged by 1-D bulk copies (TMA engine) into a 2-deep shared-memory ring.
// Per tile:
//   1. every thread owns one token: it reads the token's K code row, widens
//      the codes to exact fp16 integers and stores them into tensor memory
//      (lane = token), the A operand of QK^T;
//   2. one thread issues QK^T = A_K x B_Q as asynchronous tcgen05.mma (M=128
//      tokens, N=16 = 4 groups x 4 heads, K=128 channels) with fp32
//      accumulation in tensor memory.  B_Q is the block-diagonal query: column
//      (g, j) holds head j's query on group g's channels, so accumulator
//      column (g, j) is the group-partial dot product D_gj = sum_{d in g} q_jd c_d;
//   3. meanwhile every warp fetches its 32-channel piece of the tile's V codes
//      transposed (ldmatrix.trans), widens them to exact centred fp16 values
//      c - 8, and, once QK has finished with the A columns, stores them into
//      tensor memory with lane = channel: the A operand of PV;
//   4. scores follow eq. 5.1 per group, s_j = sum_g Delta_g D_gj + m_g sum_{d in g} q_jd;
//      the softmax maximum is shared by the CTA per tile (one barrier);
//   5. each thread writes its token's row of P' = p_j * Delta_v,g (fp16) into
//      shared memory and one thread issues PV = A_V x B_P' (M=128 channels,
//      N=16, K=128 tokens).  The offset term sum_t p_t (m_t + 8 Delta_t) is
//      accumulated on the CUDA cores;
//   6. the next tile reads PV back (one tensor-memory load per thread) into
//      register accumulators rescaled by the running-max correction.
// Tensor memory: 128 columns per CTA (A 64 | S 16 | PV 16), so four CTAs fit
// an SM.  Every wait is bounded; on a timeout the CTA records
// KV4_STATUS_TIMEOUT, drains, frees its tensor memory and stops.
#include "kv4_decode_common.cuh"

namespace kv4 {
namespace tc {

constexpr int D = 128, G = 4;
constexpr int kTilePages = 8, kTileTok = 128, kStagesTc = 2;
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColA = 0, kColS = 64, kColPV = 80;

__device__ inline void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ inline void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ inline void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ inline void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ inline void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ inline void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ inline void st_x16(uint32_t taddr, const uint32_t v[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ inline void st_16x256b(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(a),
               "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ inline void ld_x16(uint32_t taddr, float v[16]) {
  uint32_t u[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
        "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]),
        "=r"(u[14]), "=r"(u[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(u[i]);
}
__device__ inline void ld_x4(uint32_t taddr, float v[4]) {
  uint32_t u[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3])
               : "r"(taddr)
               : "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(u[i]);
}
__device__ inline void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ inline void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// Shared-memory matrix descriptor, no swizzle: lbo = byte stride between
// 8x16-byte core matrices along K, sbo = along M/N.
__device__ inline uint64_t sdesc(const void* p, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((smem_u32(p) >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}
// Instruction descriptor, kind::f16: fp32 accumulate, fp16 A and B, A K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int b_mn_major) {
  return (1u << 4) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Canonical no-swizzle layouts: a core matrix is 8 rows x 16 bytes.
// K-major R x K (element (row, k)); MN-major K x N (element (k, n)).
__device__ inline int kmaj(int row, int k, int K) {
  return ((row >> 3) * (K >> 3) + (k >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2;
}
__device__ inline int mnmaj(int k, int n, int K) {
  return ((n >> 3) * (K >> 3) + (k >> 3)) * 128 + (k & 7) * 16 + (n & 7) * 2;
}

// Channel of the K operand's contraction index k: tensor-memory column c = k/2
// holds the widened pair (channel 8u + i, channel 8u + i + 4), u = c/4, i = c%4.
__device__ inline int k_channel(int k) {
  const int c = k >> 1;
  return 8 * (c >> 2) + (c & 3) + 4 * (k & 1);
}
// Contraction index of a tile token (page pp, slot) in the PV operand: the
// 16x256b store puts token pair (2q, 2q+1) of slot half h in column 2q + h.
__device__ inline int pv_k(int pp, int slot) {
  const int h = slot >> 3, q2 = (slot & 7) >> 1, e = slot & 1;
  return 2 * (8 * pp + 2 * q2 + h) + e;
}

}  // namespace tc

// Code widening: magic-number OR, then one fp16 fma per pair.
__device__ inline uint32_t tc_hfma2(uint32_t x, uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(x), "r"(a), "r"(b));
  return d;
}
__device__ inline void tc_widen(uint32_t w, uint32_t x[4], uint32_t b1, uint32_t b16) {
  // pair i = (nibble i, nibble i + 4) -> fp16 (value - bias): b1 for x1 slots,
  // b16 (with the 1/16 scale) for the x16 slots
  x[0] = tc_hfma2((w & 0x000F000Fu) | 0x64006400u, 0x3C003C00u, b1);
  x[1] = tc_hfma2((w & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, b16);
  const uint32_t w8 = w >> 8;
  x[2] = tc_hfma2((w8 & 0x000F000Fu) | 0x64006400u, 0x3C003C00u, b1);
  x[3] = tc_hfma2((w8 & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, b16);
}
// exact code c: biases -1024 / -64; centred c - 8: -1032 / -72
constexpr uint32_t kKb1 = 0xE400E400u, kKb16 = 0xD400D400u;
constexpr uint32_t kVb1 = 0xE408E408u, kVb16 = 0xD480D480u;

__device__ inline float tc_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ inline float2 tc_h2f2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

template <int NG>
__global__ void __launch_bounds__(kThreads, 4) decode_tc_kernel(
    Layout L, const uint8_t* __restrict__ paged, const uint8_t* __restrict__ side,
    const uint16_t* __restrict__ q, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ block_table, float scale_log2, int n4, int pages_per_split,
    int prot_per_split, float* __restrict__ part_o, float* __restrict__ part_lse,
    int32_t* __restrict__ tickets, uint16_t* __restrict__ out, float* __restrict__ out_lse,
    int32_t* status) {
  using namespace tc;
  constexpr int GS = D / NG;
  constexpr int cb = 16 * D + 128 * NG;
  constexpr int kTileBytes = kTilePages * cb;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem<D, G>& sm = *reinterpret_cast<Smem<D, G>*>(smem_raw);
  uint8_t* stage_base = smem_raw + ((sizeof(Smem<D, G>) + 1023) / 1024) * 1024;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n_split = gridDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long row0 = (long long)b * L.h_q + (long long)h * G;

  int len = seq_lens[b];
  if (len < 0 || len > L.max_pages * kPage) {
    if (tid == 0 && split == 0 && h == 0) set_status(status, KV4_STATUS_BAD_LEN);
    len = 0;
  }
  const Regions rg = regions(len, L.S, L.R);
  load_query(sm, q, row0);

  if (split >= n4) {  // protected positions: the INT8 side cache (CUDA cores)
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

  const int first_page = rg.sink_end / kPage;
  const int end_page = (rg.rec_start + kPage - 1) / kPage;
  const int p_lo = first_page + split * pages_per_split;
  const int p_hi = rg.rec_start > rg.sink_end ? min(end_page, p_lo + pages_per_split) : p_lo;
  const int n_pages = max(0, p_hi - p_lo);
  const int n_tiles = (n_pages + kTilePages - 1) / kTilePages;

  // running state (CTA-uniform maxima; per-thread partial sums)
  float m_run[G], l_run[G], alpha_prev[G];
  float mt[G][NG];  // sum_t p_tj (m_tg + 8 Delta_tg) over this thread's tokens
  float O[G];       // PV accumulator of this thread's channel
#pragma unroll
  for (int j = 0; j < G; ++j) {
    m_run[j] = -INFINITY;
    l_run[j] = 0.f;
    alpha_prev[j] = 1.f;
    O[j] = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) mt[j][g] = 0.f;
  }
  // per-group query sums (eq. 5.1 offset term), this CTA's heads
  float qsg[NG][G];
#pragma unroll
  for (int g = 0; g < NG; ++g)
#pragma unroll
    for (int j = 0; j < G; ++j) {
      float qs = 0.f;
#pragma unroll
      for (int bq = 0; bq < GS / 32; ++bq) qs += sm.qsum[g * (GS / 32) + bq][j];
      qsg[g][j] = qs;
    }
  // this thread's PV channel (tensor-memory lane of its warp quarter)
  const int my_ch = 32 * warp + 4 * (lane & 7) + (lane >> 3);
  const int my_grp = (32 * warp) / GS;

  if (n_tiles > 0) {
    // ---------------------------------------------------------- set-up
    for (int idx = tid; idx < 16 * D; idx += kThreads) {
      const int n = idx / D, k = idx % D;  // B_Q[n][k], n = 4g + j
      const int g = n >> 2, j = n & 3;
      const int ch = k_channel(k);
      const uint16_t v = (g < NG && ch / GS == g) ? sm.qh[j][ch] : (uint16_t)0;
      *reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(sm.tc.bq) + kmaj(n, k, D)) = v;
    }
    if (warp == 0) tmem_alloc(&sm.tc_tmem, kTmemCols);
    if (tid == 0) {
      for (int i = 0; i < 4; ++i) mbar_init(&sm.tc_bar[i], 1);
      fence_mbar_init();
      sm.tc_abort = 0;
    }
    fence_proxy_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
  }
  const uint32_t tm = sm.tc_tmem;
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  uint64_t* bar_full = &sm.tc_bar[0];
  uint64_t* bar_s = &sm.tc_bar[2];
  uint64_t* bar_pv = &sm.tc_bar[3];
  const int32_t* bt_row = block_table + (long long)b * L.max_pages;

  // Tile loads are issued by lanes 0..7 of warp 0, one page each: the lane
  // holds its page's block-table entry (read one tile ahead), lane 0 posts the
  // byte count of the valid pages, then every lane issues its bulk copy.
  // Pages past the split or with a bad block-table entry are recorded as -1
  // and masked.
  auto fetch_id = [&](int t) -> int {
    const int pg = p_lo + t * kTilePages + lane;
    return (lane < kTilePages && t < n_tiles && pg < p_hi) ? bt_row[pg] : -2;  // -2: past the split
  };
  auto issue_tile = [&](int t, int id) {  // called by all of warp 0
    const int st = t & 1;
    int ph = id;
    if (ph != -2 && (ph < 0 || ph >= L.num_pages)) {
      set_status(status, KV4_STATUS_BAD_PAGE);
      ph = -1;
    }
    ph = ph < 0 ? -1 : ph;
    if (lane < kTilePages) sm.tc_phys[st][lane] = ph;
    const uint32_t valid = __ballot_sync(0xffffffffu, lane < kTilePages && ph >= 0);
    if (lane == 0) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bar_full[st], (uint32_t)__popc(valid) * cb);
    }
    __syncwarp();
    if (lane < kTilePages && ph >= 0)
      bulk_g2s(stage_base + (size_t)st * kTileBytes + lane * cb,
               paged + ((long long)ph * L.h_kv + h) * cb, (uint32_t)cb, &bar_full[st]);
  };
  int next_id = -2;  // warp 0, lane < 8: entry of tile t + kStagesTc
  if (warp == 0) {
    for (int t = 0; t < min(kStagesTc, n_tiles); ++t) issue_tile(t, fetch_id(t));
    next_id = fetch_id(kStagesTc);
  }

  constexpr uint32_t kIdescQK = idesc_f16(128, 16, 0);
  constexpr uint32_t kIdescPV = idesc_f16(128, 16, 1);
  // operand descriptors of k-step 0; step s adds s*256 bytes (encoded >> 4)
  const uint64_t desc_q0 = sdesc(sm.tc.bq, 128, (D / 8) * 128);
  const uint64_t desc_p0 = sdesc(sm.tc.bp, 128, (kTileTok / 8) * 128);
  const int my_pp = tid >> 4, my_slot = tid & 15;
  bool dead = false;

  for (int t = 0; t < n_tiles; ++t) {
    const int st = t & 1;
    const uint8_t* tile = stage_base + (size_t)st * kTileBytes;
    // -------- 0. previous tile's PV result -> registers (frees A and PV)
    if (t > 0) {
      if (!mbar_wait(bar_pv, (t - 1) & 1)) dead = true;
      fence_after();
      float v4[4];
      ld_x4(tm + lane_base + kColPV + 4 * my_grp, v4);
      wait_ld();
#pragma unroll
      for (int j = 0; j < G; ++j) O[j] = fmaf(O[j], alpha_prev[j], v4[j]);
    }
    // -------- 1. tile data
    if (!mbar_wait(&bar_full[st], (t >> 1) & 1)) dead = true;
    if (__syncthreads_or(dead)) break;
    const int my_phys = sm.tc_phys[st][my_pp];
    const int my_pos = (p_lo + t * kTilePages + my_pp) * kPage + my_slot;
    const bool tok_ok = my_phys >= 0 && my_pos >= rg.sink_end && my_pos < rg.rec_start;
    const uint8_t* page = tile + my_pp * cb;
    // -------- 2. K codes of my token -> tensor memory (lane = token)
    {
      const uint8_t* krow = page + my_slot * (D / 2);
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) {
        const uint4 raw =
            *reinterpret_cast<const uint4*>(krow + 16 * (pc ^ ((my_slot >> 1) & 3)));
        uint32_t x[16];
        tc_widen(raw.x, x + 0, kKb1, kKb16);
        tc_widen(raw.y, x + 4, kKb1, kKb16);
        tc_widen(raw.z, x + 8, kKb1, kKb16);
        tc_widen(raw.w, x + 12, kKb1, kKb16);
        st_x16(tm + lane_base + kColA + 16 * pc, x);
      }
      wait_st();
    }
    fence_before();
    __syncthreads();
    fence_after();
    // -------- 3. QK^T (one thread)
    if (tid == 0) {
#pragma unroll
      for (int s = 0; s < D / 16; ++s)
        mma_ts(tm + kColS, tm + kColA + 8 * s, desc_q0 + (uint64_t)(16 * s), kIdescQK, s > 0);
      mma_commit(bar_s);
    }
    // -------- 4. while QK runs: V codes (transposed), metadata
    uint32_t vraw[4][4];
    {
      const int tok = ((lane >> 3) & 1) * 8 + (lane & 7);
      const uint32_t off = codes_off_v(D) + tok * (D / 2) + 16 * (warp ^ ((tok >> 1) & 3));
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int pp = 2 * m + (lane >> 4);
        const uint32_t addr = smem_u32(tile + pp * cb + off);
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                     : "=r"(vraw[m][0]), "=r"(vraw[m][1]), "=r"(vraw[m][2]), "=r"(vraw[m][3])
                     : "r"(addr));
      }
    }
    uint32_t kmeta[NG], vmeta[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      kmeta[g] = tok_ok ? *reinterpret_cast<const uint32_t*>(page + meta_off_k(D) +
                                                               (my_slot * NG + g) * 4)
                        : 0u;
      vmeta[g] = tok_ok ? *reinterpret_cast<const uint32_t*>(page + meta_off_v(D, GS) +
                                                               (my_slot * NG + g) * 4)
                        : 0u;
    }
    // -------- 5. scores
    if (!mbar_wait(bar_s, t & 1)) dead = true;
    fence_after();
    float S[16];
    ld_x16(tm + lane_base + kColS, S);
    wait_ld();
    // -------- 6. V -> tensor memory (lane = channel); A columns are free now
    {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {  // pages 2m and 2m+1
          uint32_t xa[4], xb[4];
          tc_widen(vraw[m][2 * hp], xa, kVb1, kVb16);      // tokens (2q, 2q+1)
          tc_widen(vraw[m][2 * hp + 1], xb, kVb1, kVb16);  // tokens (8+2q, 9+2q)
          const uint32_t col = kColA + 8 * (2 * m + hp);
          st_16x256b(tm + (((uint32_t)(32 * warp)) << 16) + col, xa[0], xb[0], xa[1], xb[1]);
          st_16x256b(tm + (((uint32_t)(32 * warp + 16)) << 16) + col, xa[2], xb[2], xa[3], xb[3]);
        }
      }
      wait_st();
    }
    float sc[G];
    {
      float2 dm[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) dm[g] = tc_h2f2(kmeta[g]);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float s = 0.f;
#pragma unroll
        for (int g = 0; g < NG; ++g) s = fmaf(dm[g].x, S[4 * g + j], fmaf(dm[g].y, qsg[g][j], s));
        sc[j] = tok_ok ? s * scale_log2 : -INFINITY;
      }
      float wm[G];
#pragma unroll
      for (int j = 0; j < G; ++j) wm[j] = sc[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int j = 0; j < G; ++j) wm[j] = fmaxf(wm[j], __shfl_xor_sync(0xffffffffu, wm[j], o));
      if (lane == 0)
#pragma unroll
        for (int j = 0; j < G; ++j) sm.tc_wmax[warp][j] = wm[j];
    }
    fence_before();
    __syncthreads();
    fence_after();
    // -------- 7. next loads into this stage (its shared memory has been read)
    if (warp == 0 && t + kStagesTc < n_tiles) {
      issue_tile(t + kStagesTc, next_id);
      next_id = fetch_id(t + kStagesTc + 1);
    }
    // -------- 8. softmax, P', offset term
    float p[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      float M = fmaxf(fmaxf(sm.tc_wmax[0][j], sm.tc_wmax[1][j]),
                      fmaxf(sm.tc_wmax[2][j], sm.tc_wmax[3][j]));
      const float mnew = fmaxf(m_run[j], M);
      const float mref = mnew == -INFINITY ? 0.f : mnew;
      const float alpha = tc_ex2(m_run[j] - mref);
      alpha_prev[j] = alpha;
      m_run[j] = mnew;
      p[j] = tc_ex2(sc[j] - mref);  // masked tokens: 0
      l_run[j] = fmaf(l_run[j], alpha, p[j]);
    }
    {
      float dv[NG], mv[NG];
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const float2 dm = tc_h2f2(vmeta[g]);
        dv[g] = dm.x;
        mv[g] = fmaf(8.f, dm.x, dm.y);
      }
#pragma unroll
      for (int j = 0; j < G; ++j)
#pragma unroll
        for (int g = 0; g < NG; ++g) mt[j][g] = fmaf(mt[j][g], alpha_prev[j], p[j] * mv[g]);
      // P' row of my token: columns n = 4g + j (zero for g >= NG)
      uint32_t w8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int n0 = 2 * i, n1 = 2 * i + 1;
        const float a = (n0 >> 2) < NG ? p[n0 & 3] * dv[(n0 >> 2) < NG ? (n0 >> 2) : 0] : 0.f;
        const float c = (n1 >> 2) < NG ? p[n1 & 3] * dv[(n1 >> 2) < NG ? (n1 >> 2) : 0] : 0.f;
        __half2 hv = __floats2half2_rn(a, c);
        w8[i] = *reinterpret_cast<uint32_t*>(&hv);
      }
      const int k = pv_k(my_pp, my_slot);
      uint8_t* bp = reinterpret_cast<uint8_t*>(sm.tc.bp);
      *reinterpret_cast<uint4*>(bp + mnmaj(k, 0, kTileTok)) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
      *reinterpret_cast<uint4*>(bp + mnmaj(k, 8, kTileTok)) = make_uint4(w8[4], w8[5], w8[6], w8[7]);
    }
    fence_proxy_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    // -------- 9. PV (one thread)
    if (tid == 0) {
#pragma unroll
      for (int s = 0; s < kTileTok / 16; ++s)
        mma_ts(tm + kColPV, tm + kColA + 8 * s, desc_p0 + (uint64_t)(16 * s), kIdescPV, s > 0);
      mma_commit(bar_pv);
    }
  }

  if (n_tiles > 0) {
    if (!dead) {
      if (!mbar_wait(bar_pv, (n_tiles - 1) & 1)) dead = true;
      fence_after();
      float v4[4];
      ld_x4(tm + lane_base + kColPV + 4 * my_grp, v4);
      wait_ld();
#pragma unroll
      for (int j = 0; j < G; ++j) O[j] = fmaf(O[j], alpha_prev[j], v4[j]);
    }
    if (__syncthreads_or(dead)) {
      if (tid == 0) set_status(status, KV4_STATUS_TIMEOUT);
      // drain: bounded waits for copies and MMAs still in flight
      if (tid == 0) {
        for (int i = 0; i < 4; ++i) {
          mbar_wait(&sm.tc_bar[i], 0, 100000u);
          mbar_wait(&sm.tc_bar[i], 1, 100000u);
        }
      }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tm, kTmemCols);
  }

  // -------------------------------------------- reduce and store the split
  // l and offset-term partials over the CTA's 128 tokens
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float ls = warp_sum(l_run[j]);
    if (lane == 0) sm.tc_red[warp][j][4] = ls;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const float v = warp_sum(mt[j][g]);
      if (lane == 0) sm.tc_red[warp][j][g] = v;
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float Lt = 0.f, MT = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      Lt += sm.tc_red[w][j][4];
      MT += sm.tc_red[w][j][my_grp];
    }
    const long long row = row0 + j;
    const bool empty = !(Lt > 0.f) || n_tiles == 0;
    part_o[(row * n_split + split) * D + my_ch] = empty ? 0.f : (O[j] + MT) / Lt;
    if (tid == 0)
      part_lse[row * n_split + split] = empty ? -INFINITY : (m_run[j] + log2f(Lt)) * kLn2;
  }
  combine_if_last<D, G>(sm, tickets, b * L.h_kv + h, part_o, part_lse, row0, n_split, out,
                        out_lse);
}

template <int NG>
cudaError_t launch_tc_t(const Layout& L, const void* paged, const void* side, const uint16_t* q,
                        const int32_t* seq_lens, int num_seqs, const int32_t* block_table,
                        float sm_scale, int n4, int pages_per_split, int n8, int prot_per_split,
                        float* part_o, float* part_lse, int32_t* tickets, uint16_t* out,
                        float* out_lse, int32_t* status, cudaStream_t st) {
  constexpr int cb = 16 * tc::D + 128 * NG;
  const size_t smem = ((sizeof(Smem<tc::D, tc::G>) + 1023) / 1024) * 1024 +
                      (size_t)tc::kStagesTc * tc::kTilePages * cb;
  static OnceSetup setup;  // the shared-memory attribute, once per device
  int unused = 0;
  cudaError_t e = once_per_device(
      setup,
      [&](int, int*) {
        return cudaFuncSetAttribute(decode_tc_kernel<NG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem);
      },
      &unused);
  if (e != cudaSuccess) return e;
  dim3 grid(n4 + n8, L.h_kv, num_seqs);
  decode_tc_kernel<NG><<<grid, kThreads, smem, st>>>(
      L, (const uint8_t*)paged, (const uint8_t*)side, q, seq_lens, block_table,
      sm_scale * kLog2e, n4, pages_per_split, prot_per_split, part_o, part_lse, tickets, out,
      out_lse, status);
  return cudaGetLastError();
}

cudaError_t launch_decode_tc(const Layout& L, const void* paged, const void* side,
                             const uint16_t* q, const int32_t* seq_lens, int num_seqs,
                             const int32_t* block_table, float sm_scale, int n4,
                             int pages_per_split, int n8, int prot_per_split, float* part_o,
                             float* part_lse, int32_t* tickets, uint16_t* out, float* out_lse,
                             int32_t* status, cudaStream_t st) {
  switch (L.d_h / L.g) {
    case 4:
      return launch_tc_t<4>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, n4,
                            pages_per_split, n8, prot_per_split, part_o, part_lse, tickets, out,
                            out_lse, status, st);
    case 2:
      return launch_tc_t<2>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, n4,
                            pages_per_split, n8, prot_per_split, part_o, part_lse, tickets, out,
                            out_lse, status, st);
    case 1:
      return launch_tc_t<1>(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, n4,
                            pages_per_split, n8, prot_per_split, part_o, part_lse, tickets, out,
                            out_lse, status, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kv4
