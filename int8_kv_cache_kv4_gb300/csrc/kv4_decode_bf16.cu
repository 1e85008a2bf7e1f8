// kv4_decode_bf16.cu -- the bf16-KV paged decode comparator on the tensor
// cores (head_dim 128, 4 query heads per kv head): the same paged GQA decode
// as the mixed INT4/INT8 path, over an unquantized cache, so that the two can
// be timed on the same pages and block table.
//
// Work items are chunks of kChunk consecutive pages of one (sequence, kv
// head) pair (64 pages: measured on GB300 on the batch-64 layer, 128-page
// items ran 23 %, 32-page items 4 %, 16-page items 17 % and 8-page items
// 63 % slower; claiming the next item ahead, or prefetching its block-table
// entries and query rows, gained nothing).  Every warp works alone: it claims items from a global counter,
// streams each item's pages through its own ring of shared-memory stages
// (cp.async, 16 bytes per lane and copy, placed with an XOR swizzle so that
// the tensor-core fragment loads hit distinct banks), and keeps one online
// softmax state per item.  Per page:
//   S = K Q^T with the 16 tokens as MMA rows (m16n8k16, bf16 operands, fp32
//   accumulation; the query B operand holds each head in two columns),
//   an online-softmax step in the log2 domain with a lazily moved reference,
//   O^T += V^T P^T with P = p split into a bf16 head and tail (two products,
//   so that p keeps 16 significant bits).
// An item ends with its partial result (a locally normalised output and its
// log-normaliser per query head) and a ticket on its pair; the warp whose
// ticket completes the pair merges the pair's partials (eq. A1, in chunk
// order).  Items are computed the same way whichever warp takes them, so the
// result does not depend on the claiming order.
#include <algorithm>

#include "kv4_decode_common.cuh"
#include "kv4_mma.cuh"

namespace kv4 {
namespace {

constexpr int BD = 128, BG = 4;
constexpr int kBW = 4, kBT = kBW * 32;     // warps and threads per CTA
constexpr int kBStages = 3;                // stages per warp
constexpr int kChunk = 64;                 // pages per work item
constexpr int kTile = kPage * BD * 2;      // bytes of one page's K (or V) for one head
constexpr int kPageBytes = 2 * kTile;      // K then V: 8 KB
constexpr int kBMaxSeqs = 2048;            // sequences the per-CTA item prefix holds

struct BfRec {     // what a stage holds
  int item;        // work item (-1: nothing)
  int page;        // page index in the sequence
  int last;        // the item's last page
  int ok;          // the page was copied
};

struct __align__(16) BfSmem {
  int pre[kBMaxSeqs + 1];   // work items before sequence b (prefix over sequences)
  int total;                // work items in all
  BfRec rec[kBW][kBStages];
};

__device__ inline void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ inline void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ inline void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ inline void ldsm_x4(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ inline void mma_bf16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// bf16 pair (lo, hi) rounded to nearest even
__device__ inline uint32_t pack_bf16(float lo, float hi) {
  return (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
}
// Byte offset of 16-byte piece c (0..15) of row t (0..15) inside a staged
// 4 KB tile: pieces are XOR-swizzled by the row, so that eight rows read at
// the same piece fall on eight different bank groups.
__device__ inline uint32_t tile_off(int t, int c) { return (uint32_t)(t * 256 + ((c ^ (t & 7)) << 4)); }

__device__ inline int chunks_of(int len) { return ((len + kPage - 1) / kPage + kChunk - 1) / kChunk; }

__global__ void __launch_bounds__(kBT, 2) bf16_decode_mma_kernel(
    Layout L, const uint8_t* __restrict__ cache, const uint16_t* __restrict__ q,
    const int32_t* __restrict__ seq_lens, int B, const int32_t* __restrict__ block_table,
    float scale_log2, float* __restrict__ part_o, float* __restrict__ part_lse,
    int32_t* __restrict__ tickets, int32_t* __restrict__ claim, uint16_t* __restrict__ out,
    float* __restrict__ out_lse, int32_t* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  BfSmem& sm = *reinterpret_cast<BfSmem*>(smem_raw);
  uint8_t* stage_base = smem_raw + ((sizeof(BfSmem) + 127) / 128) * 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, qd = lane & 3;

  // ---- items per sequence (h_kv x chunks), prefix over the sequences
  {
    const int per = (B + kBT - 1) / kBT;
    const int b_lo = min(B, (int)threadIdx.x * per), b_hi = min(B, b_lo + per);
    int mine = 0;
    bool bad = false;
    for (int b = b_lo; b < b_hi; ++b) {
      int len = __ldg(seq_lens + b);
      if (len < 0 || len > L.max_pages * kPage) {
        bad = true;
        len = 0;
      }
      mine += L.h_kv * chunks_of(len);
    }
    if (bad && blockIdx.x == 0) set_status(status, KV4_STATUS_BAD_LEN);
    // exclusive scan of the per-thread counts (through pre[] as scratch)
    sm.pre[threadIdx.x] = mine;
    __syncthreads();
    if (warp == 0) {
      constexpr int E = kBT / 32;
      int v[E], run = 0;
#pragma unroll
      for (int k = 0; k < E; ++k) {
        v[k] = run;
        run += sm.pre[E * lane + k];
      }
      int incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      __syncwarp();
#pragma unroll
      for (int k = 0; k < E; ++k) sm.pre[E * lane + k] = incl - run + v[k];
      if (lane == 31) sm.total = incl;
    }
    __syncthreads();
    int base = sm.pre[threadIdx.x];
    __syncthreads();
    for (int b = b_lo; b < b_hi; ++b) {
      sm.pre[b] = base;
      int len = __ldg(seq_lens + b);
      if (len < 0 || len > L.max_pages * kPage) len = 0;
      base += L.h_kv * chunks_of(len);
    }
    if (threadIdx.x == 0) sm.pre[B] = sm.total;
    __syncthreads();
  }
  const int total = sm.total;
  // item -> (sequence, kv head, chunk)
  auto locate = [&](int it, int& b, int& h, int& ch, int& len) {
    int lo = 0, hi = B;  // last b with pre[b] <= it
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sm.pre[mid] <= it) lo = mid;
      else hi = mid;
    }
    b = lo;
    len = __ldg(seq_lens + b);
    if (len < 0 || len > L.max_pages * kPage) len = 0;  // (such a sequence has no items)
    const int nc = chunks_of(len);
    const int rr = it - sm.pre[b];
    h = rr / nc;
    ch = rr - h * nc;
  };

  uint8_t* my_st = stage_base + (size_t)warp * kBStages * kPageBytes;
  const uint32_t st_s = smem_u32(my_st);
  BfRec* rec = sm.rec[warp];

  // ---- producer state (every lane keeps the same copy): the item being
  // issued and its next page
  int pi = -1, pb = 0, ph = 0, pp = 0, pend = 0, plen = 0;
  auto claim_item = [&]() {
    int it = 0;
    if (lane == 0) it = atomicAdd(claim, 1);
    it = __shfl_sync(0xffffffffu, it, 0);
    if (it >= total) {
      pi = -1;
      return;
    }
    int ch;
    locate(it, pb, ph, ch, plen);
    pi = it;
    pp = ch * kChunk;
    pend = min((plen + kPage - 1) / kPage, pp + kChunk);
  };
  // copy the producer's next page into stage st (one commit group per stage,
  // empty when nothing is left, so that the wait counts stay aligned)
  auto issue = [&](int st) {
    BfRec rc;
    rc.item = -1;
    if (pi >= 0) {
      const int phys = __ldg(block_table + (long long)pb * L.max_pages + pp);
      rc.item = pi;
      rc.page = pp;
      rc.last = pp + 1 == pend;
      rc.ok = (unsigned)phys < (unsigned)L.num_pages;
      if (rc.ok) {
        const uint8_t* src = cache + ((long long)phys * L.h_kv + ph) * kPageBytes;
        const uint32_t dst = st_s + (uint32_t)(st * kPageBytes);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int k = lane + 32 * i;  // piece k of the page: tile k / 256, row, piece
          const int tile = k >> 8, t = (k >> 4) & 15, c = k & 15;
          cp_async16(dst + tile * kTile + tile_off(t, c), src + 16 * k);
        }
      } else if (lane == 0) {
        set_status(status, KV4_STATUS_BAD_PAGE);
      }
      if (++pp == pend) claim_item();
    }
    cp_async_commit();
    if (lane == 0) rec[st] = rc;
  };

  claim_item();
  for (int st = 0; st < kBStages; ++st) issue(st);

  // ldmatrix row addresses: K as A (tokens = rows, 16 channels per k-step):
  // matrix m = lane / 8: rows (m & 1) * 8 + lane % 8, piece 2 kk + m / 2
  const int lk_t = ((lane >> 3) & 1) * 8 + (lane & 7), lk_c = lane >> 4;
  // V^T as A (channels = rows, tokens = k) with .trans: matrix m: tokens
  // (m / 2) * 8 + lane % 8, piece 2 cb + (m & 1)
  const int lv_t = ((lane >> 4) & 1) * 8 + (lane & 7), lv_c = (lane >> 3) & 1;

  int cur = -1;            // item of the state below
  int cur_b = 0, cur_h = 0, cur_ch = 0, cur_len = 0;  // the item's sequence, kv head, chunk
  uint32_t qb[8][2];       // query B fragments of the current item: head r / 2
  float m_run = -INFINITY, l_run = 0.f, m_thr = -INFINITY;
  float acc[8][4];         // O^T: rows = channels 16 cb + r (+8), columns = heads 2 qd, 2 qd + 1
  int st = 0;
  while (true) {
    cp_async_wait<kBStages - 1>();
    __syncwarp();
    const BfRec rc = rec[st];
    if (rc.item < 0) break;
    if (rc.item != cur) {  // a new item: its query and a fresh state
      cur = rc.item;
      locate(cur, cur_b, cur_h, cur_ch, cur_len);
      const uint16_t* qrow = q + ((long long)cur_b * L.h_q + (long long)cur_h * BG + (r >> 1)) * BD;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qb[kk][0] = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * qd));
        qb[kk][1] = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * qd));
      }
      m_run = -INFINITY;
      l_run = 0.f;
      m_thr = -INFINITY;
#pragma unroll
      for (int c = 0; c < 8; ++c)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;
    }
    const uint32_t kt = st_s + (uint32_t)(st * kPageBytes), vt = kt + kTile;
    const int ntok = min(kPage, cur_len - rc.page * kPage);  // tokens of this page (>= 1)
    if (rc.ok) {
      if (ntok < kPage) {  // (uniform: every lane passes the __syncwarp below)
        // slots past the length may hold anything: zero their V rows
        if (lane < kPage - ntok) {
          const int t = ntok + lane;
#pragma unroll
          for (int c = 0; c < 16; ++c)
            *reinterpret_cast<uint4*>(my_st + st * kPageBytes + kTile + tile_off(t, c)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
      }
      // ---- S = K Q^T: lane holds tokens r, r + 8 of head qd (twice)
      float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a[4];
        ldsm_x4(a, kt + tile_off(lk_t, 2 * kk + lk_c));
        mma_bf16(s, a, qb[kk][0], qb[kk][1]);
      }
      float s0 = r < ntok ? s[0] * scale_log2 : -INFINITY;
      float s1 = r + 8 < ntok ? s[2] * scale_log2 : -INFINITY;
      // ---- online softmax of head qd (lazy reference, p <= 2^kLazy)
      const float tmax = fmaxf(s0, s1);
      if (__any_sync(0xffffffffu, tmax > m_thr)) {
        float hm = tmax;
        hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 4));
        hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 8));
        hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 16));
        const float mnew = fmaxf(m_run, hm);
        const float alpha = (mnew == -INFINITY) ? 1.f : ex2(m_run - mnew);
        // accumulator columns: heads 2 qd and 2 qd + 1
        const float aA = __shfl_sync(0xffffffffu, alpha, (2 * qd) & 3);
        const float aB = __shfl_sync(0xffffffffu, alpha, (2 * qd + 1) & 3);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          acc[c][0] *= aA;
          acc[c][1] *= aB;
          acc[c][2] *= aA;
          acc[c][3] *= aB;
        }
        l_run *= alpha;
        m_run = mnew;
        m_thr = mnew + 8.f;
      }
      const float mref = m_run == -INFINITY ? 0.f : m_run;
      const float p0 = ex2(s0 - mref), p1 = ex2(s1 - mref);  // masked: 0
      l_run += p0 + p1;
      // ---- P^T as the B operand: lane (r, q) needs head r's tokens 2 q, 2 q + 1
      // (b0) and 2 q + 8, 2 q + 9 (b1), held by lanes (2 q, r) and (2 q + 1, r)
      // as (token, token + 8); p = hi + lo, both bf16
      const uint32_t hi01 = pack_bf16(p0, p1);
      const float r0 = p0 - bf16_bits_to_f32(hi01 & 0xFFFFu);
      const float r1 = p1 - bf16_bits_to_f32(hi01 >> 16);
      const uint32_t lo01 = pack_bf16(r0, r1);
      const int srcA = (8 * qd + (r & 3)) & 31, srcB = (8 * qd + 4 + (r & 3)) & 31;
      const uint32_t hA = __shfl_sync(0xffffffffu, hi01, srcA);
      const uint32_t hB = __shfl_sync(0xffffffffu, hi01, srcB);
      const uint32_t lA = __shfl_sync(0xffffffffu, lo01, srcA);
      const uint32_t lB = __shfl_sync(0xffffffffu, lo01, srcB);
      const uint32_t keep = r < BG ? 0xFFFFFFFFu : 0u;  // columns 4..7: no head
      const uint32_t bh0 = __byte_perm(hA, hB, 0x5410) & keep, bh1 = __byte_perm(hA, hB, 0x7632) & keep;
      const uint32_t bl0 = __byte_perm(lA, lB, 0x5410) & keep, bl1 = __byte_perm(lA, lB, 0x7632) & keep;
      // ---- O^T += V^T P^T over 8 blocks of 16 channels
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t a[4];
        ldsm_x4_trans(a, vt + tile_off(lv_t, 2 * c + lv_c));
        mma_bf16(acc[c], a, bh0, bh1);
        mma_bf16(acc[c], a, bl0, bl1);
      }
    }
    __syncwarp();  // every lane is past its reads of the stage
    if (rc.last) {
      // ---- the item's partial: head j's sum over the lanes of rows r = 0..7
      float lsum = l_run;
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 4);
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 8);
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 16);
      // lanes (., q) hold head q's m and l; columns of this lane: 2 q, 2 q + 1
      const float mA = __shfl_sync(0xffffffffu, m_run, (2 * qd) & 3);
      const float mB = __shfl_sync(0xffffffffu, m_run, (2 * qd + 1) & 3);
      const float lA = __shfl_sync(0xffffffffu, lsum, (2 * qd) & 3);
      const float lB = __shfl_sync(0xffffffffu, lsum, (2 * qd + 1) & 3);
      const float iA = lA > 0.f ? 1.f / lA : 0.f, iB = lB > 0.f ? 1.f / lB : 0.f;
      const long long P = cur;
      if (qd < 2) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float* oA = part_o + (P * BG + 2 * qd) * BD + 16 * c + r;
          float* oB = part_o + (P * BG + 2 * qd + 1) * BD + 16 * c + r;
          oA[0] = acc[c][0] * iA;
          oB[0] = acc[c][1] * iB;
          oA[8] = acc[c][2] * iA;
          oB[8] = acc[c][3] * iB;
        }
      }
      if (r == 0) part_lse[P * BG + qd] = lsum > 0.f ? (m_run + log2f(lsum)) * kLn2 : -INFINITY;
      // ticket of the pair (release over the warp's stores); the warp that
      // completes the count merges the pair's chunks in order
      const int nc = chunks_of(cur_len);
      const int pair = cur_b * L.h_kv + cur_h;
      __syncwarp();
      int t = 0;
      if (lane == 0) {
        __threadfence();
        t = atomicAdd(&tickets[pair], 1);
      }
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t == nc - 1) {
        __threadfence();
        const long long P0 = cur - cur_ch;  // the pair's chunks are consecutive items
        const long long row0 = (long long)cur_b * L.h_q + (long long)cur_h * BG;
#pragma unroll 1
        for (int j = 0; j < BG; ++j) {
          float M = -INFINITY;
          for (int k = lane; k < nc; k += 32) M = fmaxf(M, __ldcg(part_lse + (P0 + k) * BG + j));
          M = warp_max(M);
          float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
          float Zl = 0.f;
          if (M != -INFINITY) {
            for (int k0 = 0; k0 < nc; k0 += 32) {
              const int k = k0 + lane;
              const float z = k < nc ? __ldcg(part_lse + (P0 + k) * BG + j) : -INFINITY;
              const float wl = z == -INFINITY ? 0.f : exp2f((z - M) * kLog2e);
              Zl += wl;
              const int nr = min(32, nc - k0);
              for (int u0 = 0; u0 < nr; u0 += 4) {
                float wv[4];
                float4 ov[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  wv[u] = __shfl_sync(0xffffffffu, wl, (u0 + u) & 31);
                  const bool use = u0 + u < nr && wv[u] != 0.f;
                  ov[u] = use ? __ldcg(reinterpret_cast<const float4*>(
                                    part_o + ((P0 + k0 + u0 + u) * BG + j) * BD) + lane)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
                  if (!use) wv[u] = 0.f;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  o.x = fmaf(wv[u], ov[u].x, o.x);
                  o.y = fmaf(wv[u], ov[u].y, o.y);
                  o.z = fmaf(wv[u], ov[u].z, o.z);
                  o.w = fmaf(wv[u], ov[u].w, o.w);
                }
              }
            }
          }
          const float Z = warp_sum(Zl);
          const bool empty = !(Z > 0.f);
          const float inv = empty ? 0.f : 1.f / Z;
          uint16_t* po = out + (row0 + j) * BD + 4 * lane;
          po[0] = f32_to_bf16_bits(o.x * inv);
          po[1] = f32_to_bf16_bits(o.y * inv);
          po[2] = f32_to_bf16_bits(o.z * inv);
          po[3] = f32_to_bf16_bits(o.w * inv);
          if (out_lse && lane == 0) out_lse[row0 + j] = empty ? -INFINITY : M + logf(Z);
        }
      }
    }
    issue(st);  // the producer's next page into the consumed stage
    st = st + 1 == kBStages ? 0 : st + 1;
  }
  cp_async_wait<0>();
  // sequences with nothing to attend: zero output, log-normaliser -inf
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    const int len = __ldg(seq_lens + b);
    if (len > 0 && len <= L.max_pages * kPage) continue;
    for (int i = threadIdx.x; i < L.h_q * BD; i += kBT) out[(long long)b * L.h_q * BD + i] = 0;
    if (out_lse)
      for (int i = threadIdx.x; i < L.h_q; i += kBT) out_lse[(long long)b * L.h_q + i] = -INFINITY;
  }
}

}  // namespace

bool bf16_mma_supported(const Layout& L, int num_seqs) {
  return L.d_h == BD && L.h_q == BG * L.h_kv && num_seqs <= kBMaxSeqs;
}

// Work items (and partial results) of the tensor-core comparator: at most one
// per kChunk pages of every (sequence, kv head) pair.
long long bf16_mma_items(const Layout& L, int num_seqs) {
  return (long long)num_seqs * L.h_kv * ((L.max_pages + kChunk - 1) / kChunk);
}

cudaError_t launch_bf16_decode_mma(const Layout& L, const void* cache, const uint16_t* q,
                                   const int32_t* seq_lens, int num_seqs,
                                   const int32_t* block_table, float sm_scale, float* part_o,
                                   float* part_lse, int32_t* tickets, int32_t* claim,
                                   uint16_t* out, float* out_lse, int32_t* status,
                                   cudaStream_t st) {
  constexpr size_t smem =
      ((sizeof(BfSmem) + 127) / 128) * 128 + (size_t)kBW * kBStages * kPageBytes;
  static_assert(2 * smem <= 228 * 1024 - 2048, "two CTAs per SM");
  static OnceSetup setup;
  int grid = 0;
  cudaError_t e = once_per_device(
      setup,
      [&](int dev, int* g) {
        cudaError_t r = cudaFuncSetAttribute(bf16_decode_mma_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        int sms = 0, per_sm = 0;
        if (r == cudaSuccess) r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (r == cudaSuccess)
          r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bf16_decode_mma_kernel, kBT,
                                                            smem);
        *g = std::max(1, sms * std::max(1, per_sm));
        return r;
      },
      &grid);
  if (e != cudaSuccess) return e;
  bf16_decode_mma_kernel<<<grid, kBT, smem, st>>>(
      L, (const uint8_t*)cache, q, seq_lens, num_seqs, block_table, sm_scale * kLog2e, part_o,
      part_lse, tickets, claim, out, out_lse, status);
  return cudaGetLastError();
}

}  // namespace kv4
