// kv4_decode.cu -- split-KV GQA decode attention over the mixed INT4/INT8
// paged cache (KV4-RL Sec. 5.3; App. A.3), the eq. A1 split/region merge, and
// the bf16-cache comparator.
//
// Work decomposition.  One CTA per (split, kv head, sequence).  The INT4
// region of a sequence, [min(S,L), max(S,L-R)), is cut into splits of
// `pages_per_split` pages; the protected positions (sinks and the recent
// window, read from the INT8 side cache) form up to `n8` further splits.
// Every split emits a locally normalised output and log-normaliser per query
// head; kv4_split_combine merges them (eq. A1), with zero weight for empty
// splits.
//
// Inside a CTA, 4 warps each stream their own pages: lane 0 of a warp issues a
// 1-D bulk asynchronous copy (cp.async.bulk, TMA engine) of the whole
// (page, kv head) chunk -- codes and metadata, 2.5 KB at d=128, g=32 -- into a
// 4-stage shared-memory ring guarded by mbarriers, so each warp keeps up to
// four chunks in flight while it computes.  The warps merge their online-
// softmax states through shared memory at the end.
//
// Scores use the affine factorisation of eq. 5.1 per group:
//   q . k^ = Delta * (q . c) + m * sum(q)
// so the INT4 codes enter the dot product exactly and scale/offset are applied
// once per group; softmax runs in the log2 domain with sm_scale*log2(e) folded
// into the scores.  All accumulation is fp32.
#include "kv4_decode_common.cuh"

namespace kv4 {

// ------------------------------------------------------------ main kernel
template <int D, int G>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(
    Layout L, const uint8_t* __restrict__ paged, const uint8_t* __restrict__ side,
    const uint16_t* __restrict__ q, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ block_table, float scale_log2, int n4, int pages_per_split,
    int prot_per_split, float* __restrict__ part_o, float* __restrict__ part_lse,
    int32_t* __restrict__ tickets, uint16_t* __restrict__ out, float* __restrict__ out_lse,
    int32_t* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<D, G>& sm = *reinterpret_cast<Smem<D, G>*>(smem_raw);
  const int cb = chunk_bytes(D, L.g);
  uint8_t* stage_base = smem_raw + ((sizeof(Smem<D, G>) + 127) / 128) * 128;

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

  WarpState<D, G> ws;
  ws.init();
  load_query(sm, q, row0);

  const int t = lane >> 1, half = lane & 1;
  if (split < n4) {
    // ---------------------------------------------------- INT4 region split
    const int first_page = rg.sink_end / kPage;
    const int end_page = (rg.rec_start + kPage - 1) / kPage;
    const int p_lo = first_page + split * pages_per_split;
    const int p_hi = min(end_page, p_lo + pages_per_split);
    const int n_my = rg.rec_start > rg.sink_end && p_hi > p_lo + warp
                         ? (p_hi - p_lo - warp + kWarps - 1) / kWarps
                         : 0;
    uint8_t* my_stages = stage_base + (size_t)warp * kStages * cb;
    const int32_t* bt_row = block_table + (long long)b * L.max_pages;
    if (lane == 0) {
      for (int st = 0; st < kStages; ++st) mbar_init(&sm.bar[warp][st], 1);
      fence_mbar_init();
    }
    __syncwarp();
    auto issue = [&](int i) {
      const int pg = p_lo + warp + i * kWarps;
      const int phys = bt_row[pg];
      uint64_t* bar = &sm.bar[warp][i % kStages];
      if (phys >= 0 && phys < L.num_pages) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, (uint32_t)cb);
        bulk_g2s(my_stages + (size_t)(i % kStages) * cb,
                 paged + ((long long)phys * L.h_kv + h) * cb, (uint32_t)cb, bar);
      } else {
        set_status(status, KV4_STATUS_BAD_PAGE);
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
      }
    };
    if (lane == 0)
      for (int i = 0; i < min(kStages, n_my); ++i) issue(i);
    for (int i = 0; i < n_my; ++i) {
      const int pg = p_lo + warp + i * kWarps;
      const int phys = bt_row[pg];
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.bar[warp][i % kStages], (i / kStages) & 1));
      const bool valid = ok && phys >= 0 && phys < L.num_pages;
      if (!ok && lane == 0) set_status(status, KV4_STATUS_BAD_PAGE);
      const uint8_t* chunk = my_stages + (size_t)(i % kStages) * cb;
      const int pos = pg * kPage + t;
      const bool tok_ok = valid && pos >= rg.sink_end && pos < rg.rec_start;
      const uint32_t tok_mask = __ballot_sync(0xffffffffu, tok_ok);
      float s[G];
      if (valid) {
        qk_int4<D, G>(sm, chunk, L.g, t, half, s);
#pragma unroll
        for (int j = 0; j < G; ++j) s[j] += __shfl_xor_sync(0xffffffffu, s[j], 1);
      }
#pragma unroll
      for (int j = 0; j < G; ++j) s[j] = tok_ok ? s[j] * scale_log2 : -INFINITY;
      softmax_tile<D, G>(ws, s, sm.p[warp], lane);
      __syncwarp();
      if (valid) pv_int4<D, G>(ws, chunk, L.g, sm.p[warp], lane, tok_mask);
      __syncwarp();
      if (lane == 0 && i + kStages < n_my) issue(i + kStages);
    }
  } else {
    prot_split<D, G>(sm, ws, L, side, b, h, rg, split - n4, prot_per_split, scale_log2, warp, lane);
  }
  write_state<D, G>(sm, ws, warp, lane);
  merge_store<D, G>(sm, part_o, part_lse, row0, n_split, split);
  combine_if_last<D, G>(sm, tickets, b * L.h_kv + h, part_o, part_lse, row0, n_split, out,
                        out_lse);
}

// ------------------------------------------------- bf16 comparator kernel
template <int D, int G>
__global__ void __launch_bounds__(kThreads) bf16_decode_split_kernel(
    Layout L, const uint16_t* __restrict__ cache, const uint16_t* __restrict__ q,
    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ block_table,
    float scale_log2, int pages_per_split, float* __restrict__ part_o,
    float* __restrict__ part_lse, int32_t* __restrict__ tickets, uint16_t* __restrict__ out,
    float* __restrict__ out_lse, int32_t* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<D, G>& sm = *reinterpret_cast<Smem<D, G>*>(smem_raw);
  constexpr int cb = 2 * kPage * D * 2;
  uint8_t* stage_base = smem_raw + ((sizeof(Smem<D, G>) + 127) / 128) * 128;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int n_split = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row0 = (long long)b * L.h_q + (long long)h * G;
  int len = seq_lens[b];
  if (len < 0 || len > L.max_pages * kPage) {
    if (threadIdx.x == 0 && split == 0 && h == 0) set_status(status, KV4_STATUS_BAD_LEN);
    len = 0;
  }
  WarpState<D, G> ws;
  ws.init();
  load_query(sm, q, row0);
  const int t = lane >> 1, half = lane & 1;
  const int end_page = (len + kPage - 1) / kPage;
  const int p_lo = split * pages_per_split;
  const int p_hi = min(end_page, p_lo + pages_per_split);
  const int n_my = p_hi > p_lo + warp ? (p_hi - p_lo - warp + kWarps - 1) / kWarps : 0;
  uint8_t* my_stages = stage_base + (size_t)warp * kStages * cb;
  const int32_t* bt_row = block_table + (long long)b * L.max_pages;
  if (lane == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&sm.bar[warp][st], 1);
    fence_mbar_init();
  }
  __syncwarp();
  auto issue = [&](int i) {
    const int pg = p_lo + warp + i * kWarps;
    const int phys = bt_row[pg];
    uint64_t* bar = &sm.bar[warp][i % kStages];
    if (phys >= 0 && phys < L.num_pages) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, (uint32_t)cb);
      bulk_g2s(my_stages + (size_t)(i % kStages) * cb,
               reinterpret_cast<const uint8_t*>(cache) + ((long long)phys * L.h_kv + h) * cb,
               (uint32_t)cb, bar);
    } else {
      set_status(status, KV4_STATUS_BAD_PAGE);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
    }
  };
  if (lane == 0)
    for (int i = 0; i < min(kStages, n_my); ++i) issue(i);
  constexpr int PD = D / 32;
  for (int i = 0; i < n_my; ++i) {
    const int pg = p_lo + warp + i * kWarps;
    const int phys = bt_row[pg];
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.bar[warp][i % kStages], (i / kStages) & 1));
    const bool valid = ok && phys >= 0 && phys < L.num_pages;
    if (!ok && lane == 0) set_status(status, KV4_STATUS_BAD_PAGE);
    const uint16_t* kc = reinterpret_cast<const uint16_t*>(my_stages + (size_t)(i % kStages) * cb);
    const uint16_t* vc = kc + kPage * D;
    const int pos = pg * kPage + t;
    float s[G];
#pragma unroll
    for (int j = 0; j < G; ++j) s[j] = 0.f;
    if (valid) {
      const uint32_t* row = reinterpret_cast<const uint32_t*>(kc + t * D + half * (D / 2));
#pragma unroll 8
      for (int w = 0; w < D / 4; ++w) {
        const uint32_t word = row[w];
        const float x0 = bf16_bits_to_f32(word & 0xFFFFu), x1 = bf16_bits_to_f32(word >> 16);
#pragma unroll
        for (int j = 0; j < G; ++j)
          s[j] = fmaf(sm.q[j][half][2 * w], x0, fmaf(sm.q[j][half][2 * w + 1], x1, s[j]));
      }
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
      s[j] += __shfl_xor_sync(0xffffffffu, s[j], 1);
      s[j] = (valid && pos < len) ? s[j] * scale_log2 : -INFINITY;
    }
    const uint32_t tok_mask = __ballot_sync(0xffffffffu, valid && pos < len);
    softmax_tile<D, G>(ws, s, sm.p[warp], lane);
    __syncwarp();
    if (valid) {
      for (int tt = 0; tt < kPage; ++tt) {
        if (!((tok_mask >> (2 * tt)) & 1u)) continue;
        float v[PD];
        if (PD == 4) {
          const uint2 raw = *reinterpret_cast<const uint2*>(vc + tt * D + lane * PD);
          v[0] = bf16_bits_to_f32(raw.x & 0xFFFFu);
          v[1] = bf16_bits_to_f32(raw.x >> 16);
          v[2] = bf16_bits_to_f32(raw.y & 0xFFFFu);
          v[3] = bf16_bits_to_f32(raw.y >> 16);
        } else {
          const uint32_t raw = *reinterpret_cast<const uint32_t*>(vc + tt * D + lane * PD);
          v[0] = bf16_bits_to_f32(raw & 0xFFFFu);
          v[PD - 1] = bf16_bits_to_f32(raw >> 16);
        }
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float pj = sm.p[warp][tt][j];
#pragma unroll
          for (int ii = 0; ii < PD; ++ii) ws.acc[j][ii] = fmaf(pj, v[ii], ws.acc[j][ii]);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && i + kStages < n_my) issue(i + kStages);
  }
  write_state<D, G>(sm, ws, warp, lane);
  merge_store<D, G>(sm, part_o, part_lse, row0, n_split, split);
  combine_if_last<D, G>(sm, tickets, b * L.h_kv + h, part_o, part_lse, row0, n_split, out,
                        out_lse);
}

// ------------------------------------------------------------ combine kernel
// Eq. A1 over n parts per row; one warp per row, lane owns D/32 channels.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ part_o,
                                                      const float* __restrict__ part_lse, int rows,
                                                      int n, uint16_t* __restrict__ out,
                                                      float* __restrict__ out_lse) {
  constexpr int PD = D / 32;
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* lse = part_lse + row * n;
  float M = -INFINITY;
  for (int r = lane; r < n; r += 32) M = fmaxf(M, lse[r]);
  M = warp_max(M);
  float acc[PD];
#pragma unroll
  for (int i = 0; i < PD; ++i) acc[i] = 0.f;
  float Z = 0.f;
  if (M != -INFINITY) {
    for (int r = 0; r < n; ++r) {
      const float z = lse[r];
      if (z == -INFINITY) continue;
      const float w = __expf(z - M);
      Z += w;
      const float* o = part_o + (row * n + r) * D + lane * PD;
#pragma unroll
      for (int i = 0; i < PD; ++i) acc[i] = fmaf(w, o[i], acc[i]);
    }
  }
  const bool empty = !(Z > 0.f);
#pragma unroll
  for (int i = 0; i < PD; ++i)
    out[row * D + lane * PD + i] = f32_to_bf16_bits(empty ? 0.f : acc[i] / Z);
  if (out_lse && lane == 0) out_lse[row] = empty ? -INFINITY : M + logf(Z);
}

// ------------------------------------------------------------ launchers
template <int D, int G>
size_t decode_smem_bytes(int cb) {
  return ((sizeof(Smem<D, G>) + 127) / 128) * 128 + (size_t)kWarps * kStages * cb;
}

template <int D, int G>
cudaError_t launch_decode_t(const Layout& L, const void* paged, const void* side,
                            const uint16_t* q, const int32_t* seq_lens, int num_seqs,
                            const int32_t* block_table, float sm_scale, int n4,
                            int pages_per_split, int n8, int prot_per_split, float* part_o,
                            float* part_lse, int32_t* tickets, uint16_t* out, float* out_lse,
                            int32_t* status, cudaStream_t st) {
  const size_t smem = decode_smem_bytes<D, G>(chunk_bytes(D, L.g));
  // the attribute, once per device, for the largest chunk (group 32)
  const size_t smem_max = decode_smem_bytes<D, G>(chunk_bytes(D, 32));
  static OnceSetup setup;
  int unused = 0;
  cudaError_t e = once_per_device(
      setup,
      [&](int, int*) {
        return cudaFuncSetAttribute(decode_split_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem_max);
      },
      &unused);
  if (e != cudaSuccess) return e;
  dim3 grid(n4 + n8, L.h_kv, num_seqs);
  decode_split_kernel<D, G><<<grid, kThreads, smem, st>>>(
      L, (const uint8_t*)paged, (const uint8_t*)side, q, seq_lens, block_table,
      sm_scale * kLog2e, n4, pages_per_split, prot_per_split, part_o, part_lse, tickets, out,
      out_lse, status);
  return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_bf16_decode_t(const Layout& L, const void* cache, const uint16_t* q,
                                 const int32_t* seq_lens, int num_seqs,
                                 const int32_t* block_table, float sm_scale, int n_split,
                                 int pages_per_split, float* part_o, float* part_lse,
                                 int32_t* tickets, uint16_t* out, float* out_lse,
                                 int32_t* status, cudaStream_t st) {
  const size_t smem = decode_smem_bytes<D, G>(2 * kPage * D * 2);
  static OnceSetup setup;  // the shared-memory attribute, once per device
  int unused = 0;
  cudaError_t e = once_per_device(
      setup,
      [&](int, int*) {
        return cudaFuncSetAttribute(bf16_decode_split_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem);
      },
      &unused);
  if (e != cudaSuccess) return e;
  dim3 grid(n_split, L.h_kv, num_seqs);
  bf16_decode_split_kernel<D, G><<<grid, kThreads, smem, st>>>(
      L, (const uint16_t*)cache, q, seq_lens, block_table, sm_scale * kLog2e, pages_per_split,
      part_o, part_lse, tickets, out, out_lse, status);
  return cudaGetLastError();
}

#define KV4_DISPATCH_DG(D_, G_, CALL)                                                   \
  do {                                                                                  \
    if ((D_) == 128) {                                                                  \
      switch (G_) {                                                                     \
        case 1: { constexpr int D = 128, G = 1; return CALL; }                          \
        case 2: { constexpr int D = 128, G = 2; return CALL; }                          \
        case 4: { constexpr int D = 128, G = 4; return CALL; }                          \
        case 8: { constexpr int D = 128, G = 8; return CALL; }                          \
      }                                                                                 \
    } else if ((D_) == 64) {                                                            \
      switch (G_) {                                                                     \
        case 1: { constexpr int D = 64, G = 1; return CALL; }                           \
        case 2: { constexpr int D = 64, G = 2; return CALL; }                           \
        case 4: { constexpr int D = 64, G = 4; return CALL; }                           \
        case 8: { constexpr int D = 64, G = 8; return CALL; }                           \
      }                                                                                 \
    }                                                                                   \
    return cudaErrorInvalidValue;                                                       \
  } while (0)

cudaError_t launch_decode(const Layout& L, const void* paged, const void* side, const uint16_t* q,
                          const int32_t* seq_lens, int num_seqs, const int32_t* block_table,
                          float sm_scale, int n4, int pages_per_split, int n8, int prot_per_split,
                          float* part_o, float* part_lse, int32_t* tickets, uint16_t* out,
                          float* out_lse, int32_t* status, cudaStream_t st) {
  KV4_DISPATCH_DG(L.d_h, L.h_q / L.h_kv,
                  (launch_decode_t<D, G>(L, paged, side, q, seq_lens, num_seqs, block_table,
                                         sm_scale, n4, pages_per_split, n8, prot_per_split,
                                         part_o, part_lse, tickets, out, out_lse, status, st)));
}

cudaError_t launch_bf16_decode(const Layout& L, const void* cache, const uint16_t* q,
                               const int32_t* seq_lens, int num_seqs, const int32_t* block_table,
                               float sm_scale, int n_split, int pages_per_split, float* part_o,
                               float* part_lse, int32_t* tickets, uint16_t* out, float* out_lse,
                               int32_t* status, cudaStream_t st) {
  KV4_DISPATCH_DG(L.d_h, L.h_q / L.h_kv,
                  (launch_bf16_decode_t<D, G>(L, cache, q, seq_lens, num_seqs, block_table,
                                              sm_scale, n_split, pages_per_split, part_o,
                                              part_lse, tickets, out, out_lse, status, st)));
}

cudaError_t launch_combine(const float* part_o, const float* part_lse, int rows, int n, int d_h,
                           uint16_t* out, float* out_lse, cudaStream_t st) {
  const int blocks = (rows + 3) / 4;
  if (blocks == 0) return cudaSuccess;
  if (d_h == 128)
    combine_kernel<128><<<blocks, 128, 0, st>>>(part_o, part_lse, rows, n, out, out_lse);
  else if (d_h == 64)
    combine_kernel<64><<<blocks, 128, 0, st>>>(part_o, part_lse, rows, n, out, out_lse);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace kv4
