#include <algorithm>
// kv4_abi.cu -- the extern "C" boundary declared in include/kv4.h: argument
// validation, buffer sizing, the split plan, and kernel launches.  No entry
// point allocates, frees or synchronises.
#include <stdint.h>

#include "kv4_common.cuh"

namespace kv4 {
cudaError_t launch_quant_append(const Layout&, void*, void*, const uint16_t*, const uint16_t*,
                                const int32_t*, const int32_t*, int, const int32_t*,
                                const int32_t*, int32_t*, bool, cudaStream_t);
cudaError_t launch_hadamard_bf16(const uint16_t*, uint16_t*, long long, int, cudaStream_t);
cudaError_t launch_fp4_append(const Layout&, int, bool, void*, const uint16_t*, const uint16_t*,
                              const int32_t*, const int32_t*, int, const int32_t*, const int32_t*,
                              int32_t*, cudaStream_t);
cudaError_t launch_fp4_to_bf16(const Layout&, int, const void*, void*, cudaStream_t);
cudaError_t launch_bf16_append(const Layout&, void*, const uint16_t*, const uint16_t*,
                               const int32_t*, const int32_t*, int, const int32_t*, const int32_t*,
                               int32_t*, cudaStream_t);
cudaError_t launch_decode(const Layout&, const void*, const void*, const uint16_t*, const int32_t*,
                          int, const int32_t*, float, int, int, int, int, float*, float*, int32_t*,
                          uint16_t*, float*, int32_t*, cudaStream_t);
cudaError_t launch_bf16_decode(const Layout&, const void*, const uint16_t*, const int32_t*, int,
                               const int32_t*, float, int, int, float*, float*, int32_t*,
                               uint16_t*, float*, int32_t*, cudaStream_t);
cudaError_t launch_combine(const float*, const float*, int, int, int, uint16_t*, float*,
                           cudaStream_t);
bool mma_supported(const Layout&);
bool bf16_mma_supported(const Layout&, int);
long long bf16_mma_items(const Layout&, int);
cudaError_t launch_bf16_decode_mma(const Layout&, const void*, const uint16_t*, const int32_t*, int,
                                   const int32_t*, float, float*, float*, int32_t*, int32_t*,
                                   uint16_t*, float*, int32_t*, cudaStream_t);
static int g_decode_kernel = KV4_KERNEL_AUTO;
cudaError_t launch_decode_mma(const Layout&, const void*, const void*, const uint16_t*,
                              const int32_t*, int, const int32_t*, float, int, int, int, int,
                              float*, float*, int32_t*, uint16_t*, float*, int32_t*,
                              cudaStream_t);
bool stream_supported(const Layout&);
long long stream_partials(const Layout&, int);
size_t stream_plan_bytes();
cudaError_t launch_decode_stream(const Layout&, const void*, const void*, const uint16_t*,
                                 const int32_t*, int, const int32_t*, float, float*, float*,
                                 int32_t*, void*, uint16_t*, float*, int32_t*, bool,
                                 cudaStream_t);

// Split planning.  The host does not know the per-sequence lengths (they live
// on the device), so the plan is sized from the block-table capacity: about
// kTargetCtas CTAs in total (16 per SM of a 152-SM GB300), at least
// kMinPagesPerSplit pages per INT4 split, a whole number of 8-page tiles per
// split (the split kernels' page loop), and one protected split per
// kProtChunk side-cache slots.
constexpr int kTargetCtas = 16 * 152;
constexpr int kMinPagesPerSplit = 4;
constexpr int kProtChunk = 256;
constexpr int kTilePagesPlan = 8;

struct Plan {
  int n4, pages_per_split, n8, prot_per_split;
  int total() const { return n4 + n8; }
};

static Plan make_plan(const kv4_layout* lay, int num_seqs, int max_splits, bool with_prot) {
  Plan p;
  const int maxp = lay->max_pages_per_seq;
  const long long units = (long long)(num_seqs > 0 ? num_seqs : 1) * lay->num_kv_heads;
  long long n4 = (kTargetCtas + units - 1) / units;
  if (n4 < 1) n4 = 1;
  if (max_splits > 0) n4 = max_splits;  // caller's choice (still an upper bound below)
  int pps = (int)((maxp + n4 - 1) / n4);
  if (pps < kMinPagesPerSplit) pps = kMinPagesPerSplit;
  if (max_splits > 0 && (maxp + pps - 1) / pps > max_splits) pps = (maxp + max_splits - 1) / max_splits;
  // whole 8-page tiles
  pps = (pps + kTilePagesPlan - 1) / kTilePagesPlan * kTilePagesPlan;
  p.pages_per_split = pps;
  p.n4 = (maxp + pps - 1) / pps;
  const int NS = lay->sink + lay->recent;
  p.prot_per_split = kProtChunk;
  p.n8 = (with_prot && NS > 0) ? (NS + kProtChunk - 1) / kProtChunk : 0;
  return p;
}

static Layout to_layout(const kv4_layout* l) {
  Layout L;
  L.h_q = l->num_q_heads;
  L.h_kv = l->num_kv_heads;
  L.d_h = l->head_dim;
  L.g = l->int4_group;
  L.S = l->sink;
  L.R = l->recent;
  L.max_seqs = l->max_seqs;
  L.num_pages = l->num_pages;
  L.max_pages = l->max_pages_per_seq;
  return L;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Workspace: fp32 partial outputs [rows][n_split][d], their log-normalisers
// [rows][n_split], one int32 completion ticket per (sequence, kv head) and,
// where the work-balanced kernel may run, its plan (the per-CTA start table).
struct Workspace {
  float* part_o;
  float* part_lse;
  int32_t* tickets;
  void* plan;
  size_t ticket_bytes;
  size_t bytes;
};
static size_t round256(size_t x) { return (x + 255) / 256 * 256; }
// Rows of d partial-output values: [query row][split] for the split plan's
// kernels, or (max_splits = 0, a layout the work-balanced kernel serves) at
// least that kernel's partial results x G query heads.
static size_t partial_rows(const kv4_layout* l, int num_seqs, const Plan& p, int max_splits) {
  size_t n = (size_t)num_seqs * l->num_q_heads * (size_t)p.total();
  const Layout L = to_layout(l);
  if (max_splits == 0 && stream_supported(L) && num_seqs > 0) {
    const size_t s =
        (size_t)stream_partials(L, num_seqs) * (size_t)(l->num_q_heads / l->num_kv_heads);
    if (s > n) n = s;
  }
  return n;
}
static Workspace ws_layout(const kv4_layout* l, int num_seqs, const Plan& p, int max_splits,
                           void* base) {
  const size_t prow = partial_rows(l, num_seqs, p, max_splits);
  const size_t o = round256(prow * l->head_dim * sizeof(float));
  const size_t z = round256(prow * sizeof(float));
  const bool stream = max_splits == 0 && stream_supported(to_layout(l)) && num_seqs > 0;
  Workspace w;
  w.ticket_bytes = (size_t)num_seqs * l->num_kv_heads * sizeof(int32_t);
  const size_t tk = round256(w.ticket_bytes);
  w.bytes = o + z + tk + (stream ? round256(stream_plan_bytes()) : 0);
  w.part_o = (float*)base;
  w.part_lse = (float*)((char*)base + o);
  w.tickets = (int32_t*)((char*)base + o + z);
  w.plan = stream ? (void*)((char*)base + o + z + tk) : nullptr;
  return w;
}
static size_t ws_bytes(const kv4_layout* l, int num_seqs, const Plan& p, int max_splits) {
  return ws_layout(l, num_seqs, p, max_splits, nullptr).bytes;
}

}  // namespace kv4

using namespace kv4;

extern "C" {

int kv4_abi_version(void) { return KV4_ABI_VERSION; }

int kv4_set_decode_kernel(int which) {
  const int prev = g_decode_kernel;
  if (which == KV4_KERNEL_AUTO || which == KV4_KERNEL_CUDA_CORE || which == KV4_KERNEL_MMA_SYNC ||
      which == KV4_KERNEL_STREAM)
    g_decode_kernel = which;
  return prev;
}

const char* kv4_status_string(int code) {
  switch (code) {
    case KV4_OK: return "ok";
    case KV4_ERR_INVALID_ARG: return "invalid argument";
    case KV4_ERR_UNSUPPORTED: return "unsupported shape";
    case KV4_ERR_LAUNCH: return "CUDA launch failed";
    case KV4_ERR_WORKSPACE: return "workspace too small";
    default: break;
  }
  return "unknown code";
}

int kv4_check_layout(const kv4_layout* l) {
  if (!l) return KV4_ERR_INVALID_ARG;
  if (l->num_q_heads <= 0 || l->num_kv_heads <= 0 || l->num_q_heads % l->num_kv_heads != 0)
    return KV4_ERR_INVALID_ARG;
  if (l->num_kv_heads > (1 << 16)) return KV4_ERR_INVALID_ARG;  // kernels index heads x chunk in 32 bits
  const int G = l->num_q_heads / l->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KV4_ERR_UNSUPPORTED;
  if (l->head_dim != 64 && l->head_dim != 128) return KV4_ERR_UNSUPPORTED;
  if (l->page_size != 16) return KV4_ERR_UNSUPPORTED;
  const int g = l->int4_group;
  if (g != 32 && g != 64 && g != 128) return KV4_ERR_UNSUPPORTED;
  if (g > l->head_dim) return KV4_ERR_UNSUPPORTED;
  if (l->int8_group != l->head_dim) return KV4_ERR_UNSUPPORTED;
  if (l->sink < 0 || l->recent < 0) return KV4_ERR_INVALID_ARG;
  if ((long long)l->sink + l->recent > (1LL << 30)) return KV4_ERR_INVALID_ARG;
  if (l->max_seqs <= 0 || l->num_pages <= 0 || l->max_pages_per_seq <= 0)
    return KV4_ERR_INVALID_ARG;
  if ((long long)l->max_pages_per_seq * 16 > (1LL << 30)) return KV4_ERR_INVALID_ARG;
  return KV4_OK;
}

size_t kv4_paged_cache_bytes(const kv4_layout* l) {
  if (kv4_check_layout(l) != KV4_OK) return 0;
  return (size_t)l->num_pages * l->num_kv_heads * chunk_bytes(l->head_dim, l->int4_group);
}

size_t kv4_side_cache_bytes(const kv4_layout* l) {
  if (kv4_check_layout(l) != KV4_OK) return 0;
  return (size_t)l->max_seqs * l->num_kv_heads *
         (size_t)side_block_bytes(l->head_dim, l->sink, l->recent);
}

size_t kv4_bf16_cache_bytes(const kv4_layout* l) {
  if (kv4_check_layout(l) != KV4_OK) return 0;
  return (size_t)l->num_pages * l->num_kv_heads * 2 * 16 * l->head_dim * 2;
}

int32_t kv4_num_splits(const kv4_layout* l, int32_t num_seqs, int32_t max_splits) {
  if (kv4_check_layout(l) != KV4_OK || num_seqs < 0) return 0;
  return make_plan(l, num_seqs, max_splits, true).total();
}

size_t kv4_workspace_bytes(const kv4_layout* l, int32_t num_seqs, int32_t max_splits) {
  if (kv4_check_layout(l) != KV4_OK || num_seqs < 0) return 0;
  return ws_bytes(l, num_seqs, make_plan(l, num_seqs, max_splits, true), max_splits);
}

static int quant_append(const kv4_layout* l, void* paged, void* side, const uint16_t* k_new,
                        const uint16_t* v_new, const int32_t* tok_seq, const int32_t* tok_pos,
                        int32_t T, const int32_t* seq_lens, const int32_t* block_table,
                        int32_t* dev_status, bool rotate_k, void* stream) {
  int rc = kv4_check_layout(l);
  if (rc != KV4_OK) return rc;
  if (T < 0) return KV4_ERR_INVALID_ARG;
  if (T == 0) return KV4_OK;
  if (!paged || !k_new || !v_new || !tok_seq || !tok_pos || !seq_lens || !block_table)
    return KV4_ERR_INVALID_ARG;
  if (!side && l->sink + l->recent > 0) return KV4_ERR_INVALID_ARG;
  if (!aligned16(paged) || !aligned16(side) || !aligned16(k_new) || !aligned16(v_new))
    return KV4_ERR_INVALID_ARG;
  cudaError_t e = launch_quant_append(to_layout(l), paged, side, k_new, v_new, tok_seq, tok_pos,
                                      T, seq_lens, block_table, dev_status, rotate_k,
                                      (cudaStream_t)stream);
  return e == cudaSuccess ? KV4_OK : KV4_ERR_LAUNCH;
}

int kv4_quant_append(const kv4_layout* l, void* paged, void* side, const uint16_t* k_new,
                     const uint16_t* v_new, const int32_t* tok_seq, const int32_t* tok_pos,
                     int32_t T, const int32_t* seq_lens, const int32_t* block_table,
                     int32_t* dev_status, void* stream) {
  return quant_append(l, paged, side, k_new, v_new, tok_seq, tok_pos, T, seq_lens, block_table,
                      dev_status, false, stream);
}

int kv4_quant_append_hadamard(const kv4_layout* l, void* paged, void* side,
                              const uint16_t* k_new, const uint16_t* v_new,
                              const int32_t* tok_seq, const int32_t* tok_pos, int32_t T,
                              const int32_t* seq_lens, const int32_t* block_table,
                              int32_t* dev_status, void* stream) {
  return quant_append(l, paged, side, k_new, v_new, tok_seq, tok_pos, T, seq_lens, block_table,
                      dev_status, true, stream);
}

size_t kv4_fp4_cache_bytes(const kv4_layout* l) {
  if (kv4_check_layout(l) != KV4_OK) return 0;
  return (size_t)l->num_pages * l->num_kv_heads * 2 * 16 * (size_t)(l->head_dim / 2 + 16);
}

int kv4_fp4_append(const kv4_layout* l, int32_t format, int32_t rotate_k, void* cache,
                   const uint16_t* k_new, const uint16_t* v_new, const int32_t* tok_seq,
                   const int32_t* tok_pos, int32_t T, const int32_t* seq_lens,
                   const int32_t* block_table, int32_t* dev_status, void* stream) {
  int rc = kv4_check_layout(l);
  if (rc != KV4_OK) return rc;
  if (format != KV4_FP4_NVFP4 && format != KV4_FP4_MXFP4) return KV4_ERR_INVALID_ARG;
  if (T < 0) return KV4_ERR_INVALID_ARG;
  if (T == 0) return KV4_OK;
  if (!cache || !k_new || !v_new || !tok_seq || !tok_pos || !seq_lens || !block_table)
    return KV4_ERR_INVALID_ARG;
  if (!aligned16(cache) || !aligned16(k_new) || !aligned16(v_new)) return KV4_ERR_INVALID_ARG;
  cudaError_t e = launch_fp4_append(to_layout(l), format, rotate_k != 0, cache, k_new, v_new,
                                    tok_seq, tok_pos, T, seq_lens, block_table, dev_status,
                                    (cudaStream_t)stream);
  return e == cudaSuccess ? KV4_OK : KV4_ERR_LAUNCH;
}

int kv4_fp4_to_bf16(const kv4_layout* l, int32_t format, const void* cache, void* bf16_cache,
                    void* stream) {
  int rc = kv4_check_layout(l);
  if (rc != KV4_OK) return rc;
  if (format != KV4_FP4_NVFP4 && format != KV4_FP4_MXFP4) return KV4_ERR_INVALID_ARG;
  if (!cache || !bf16_cache || !aligned16(cache) || !aligned16(bf16_cache)) return KV4_ERR_INVALID_ARG;
  cudaError_t e = launch_fp4_to_bf16(to_layout(l), format, cache, bf16_cache, (cudaStream_t)stream);
  return e == cudaSuccess ? KV4_OK : KV4_ERR_LAUNCH;
}

int kv4_hadamard_bf16(const uint16_t* x, uint16_t* y, int32_t rows, int32_t dim, void* stream) {
  if (rows < 0 || (dim != 64 && dim != 128)) return KV4_ERR_INVALID_ARG;
  if (rows == 0) return KV4_OK;
  if (!x || !y || ((uintptr_t)x & 7u) || ((uintptr_t)y & 7u)) return KV4_ERR_INVALID_ARG;
  const uintptr_t bytes = (uintptr_t)rows * (uintptr_t)dim * 2u;
  if (x != y && (uintptr_t)x < (uintptr_t)y + bytes && (uintptr_t)y < (uintptr_t)x + bytes)
    return KV4_ERR_INVALID_ARG;  // partial overlap
  cudaError_t e = launch_hadamard_bf16(x, y, rows, dim, (cudaStream_t)stream);
  return e == cudaSuccess ? KV4_OK : KV4_ERR_LAUNCH;
}

namespace {
// kv4_decode_attn and kv4_decode_attn_hadamard (rotate_q).
int decode_attn(const kv4_layout* l, const void* paged, const void* side, const uint16_t* q,
                const int32_t* seq_lens, int32_t num_seqs, const int32_t* block_table,
                float sm_scale, int32_t max_splits, void* workspace, size_t workspace_bytes,
                uint16_t* out, float* out_lse, int32_t* dev_status, bool rotate_q, void* stream) {
  int rc = kv4_check_layout(l);
  if (rc != KV4_OK) return rc;
  if (num_seqs < 0 || num_seqs > l->max_seqs || max_splits < 0) return KV4_ERR_INVALID_ARG;
  if (num_seqs == 0) return KV4_OK;
  if (!paged || !q || !seq_lens || !block_table || !workspace || !out) return KV4_ERR_INVALID_ARG;
  if (!side && l->sink + l->recent > 0) return KV4_ERR_INVALID_ARG;
  if (!aligned16(paged) || !aligned16(side) || !aligned16(q) || !aligned16(workspace))
    return KV4_ERR_INVALID_ARG;
  const Plan p = make_plan(l, num_seqs, max_splits, true);
  if (workspace_bytes < ws_bytes(l, num_seqs, p, max_splits)) return KV4_ERR_WORKSPACE;
  const Workspace w = ws_layout(l, num_seqs, p, max_splits, workspace);
  cudaStream_t st = (cudaStream_t)stream;
  const Layout L = to_layout(l);
  // head_dim 128 with 4 query heads per kv head runs a tensor-core kernel:
  // the work-balanced stream kernel, or with a caller-fixed split count the
  // warp-level split kernel; other shapes the CUDA-core kernel.
  int which = g_decode_kernel;
  if (which == KV4_KERNEL_AUTO) which = KV4_KERNEL_STREAM;  // fastest measured on GB300
  if (which == KV4_KERNEL_STREAM && (max_splits > 0 || !stream_supported(L)))
    which = KV4_KERNEL_MMA_SYNC;
  if (!mma_supported(L)) which = KV4_KERNEL_CUDA_CORE;
  // Rotated queries: the stream kernel rotates each pair's query as it sets
  // it up; for the other kernels the rotation runs first, into `out` (same
  // shape as q, written only after every read of the query rows it holds).
  if (rotate_q && which != KV4_KERNEL_STREAM) {
    if (!aligned16(out)) return KV4_ERR_INVALID_ARG;
    const uintptr_t bytes = (uintptr_t)num_seqs * l->num_q_heads * l->head_dim * 2u;
    if ((uintptr_t)q < (uintptr_t)out + bytes && (uintptr_t)out < (uintptr_t)q + bytes)
      return KV4_ERR_INVALID_ARG;
    if (launch_hadamard_bf16(q, out, (long long)num_seqs * l->num_q_heads, l->head_dim, st) !=
        cudaSuccess)
      return KV4_ERR_LAUNCH;
    q = out;
  }
  // Completion tickets for the fused eq. A1 merge start at zero on every call
  // (the stream kernel's launcher clears them itself when it merges in-kernel).
  if (which != KV4_KERNEL_STREAM && cudaMemsetAsync(w.tickets, 0, w.ticket_bytes, st) != cudaSuccess)
    return KV4_ERR_LAUNCH;
  cudaError_t e;
  if (which == KV4_KERNEL_STREAM)
    e = launch_decode_stream(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale,
                             w.part_o, w.part_lse, w.tickets, w.plan, out, out_lse, dev_status,
                             rotate_q, st);
  else if (which == KV4_KERNEL_MMA_SYNC)
    e = launch_decode_mma(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, p.n4,
                          p.pages_per_split, p.n8, p.prot_per_split, w.part_o, w.part_lse,
                          w.tickets, out, out_lse, dev_status, st);
  else
    e = launch_decode(L, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, p.n4,
                      p.pages_per_split, p.n8, p.prot_per_split, w.part_o, w.part_lse,
                      w.tickets, out, out_lse, dev_status, st);
  return e == cudaSuccess ? KV4_OK : KV4_ERR_LAUNCH;
}

}  // namespace

int kv4_decode_attn(const kv4_layout* l, const void* paged, const void* side, const uint16_t* q,
                    const int32_t* seq_lens, int32_t num_seqs, const int32_t* block_table,
                    float sm_scale, int32_t max_splits, void* workspace, size_t workspace_bytes,
                    uint16_t* out, float* out_lse, int32_t* dev_status, void* stream) {
  return decode_attn(l, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, max_splits,
                     workspace, workspace_bytes, out, out_lse, dev_status, false, stream);
}

int kv4_decode_attn_hadamard(const kv4_layout* l, const void* paged, const void* side,
                             const uint16_t* q, const int32_t* seq_lens, int32_t num_seqs,
                             const int32_t* block_table, float sm_scale, int32_t max_splits,
                             void* workspace, size_t workspace_bytes, uint16_t* out,
                             float* out_lse, int32_t* dev_status, void* stream) {
  return decode_attn(l, paged, side, q, seq_lens, num_seqs, block_table, sm_scale, max_splits,
                     workspace, workspace_bytes, out, out_lse, dev_status, true, stream);
}

int kv4_split_combine(const float* part_o, const float* part_lse, int32_t rows, int32_t n_parts,
                      int32_t head_dim, uint16_t* out, float* out_lse, void* stream) {
  if (rows < 0 || n_parts < 0 || (head_dim != 64 && head_dim != 128)) return KV4_ERR_INVALID_ARG;
  if (rows == 0) return KV4_OK;
  if (!out || (n_parts > 0 && (!part_o || !part_lse))) return KV4_ERR_INVALID_ARG;
  cudaError_t e =
      launch_combine(part_o, part_lse, rows, n_parts, head_dim, out, out_lse, (cudaStream_t)stream);
  return e == cudaSuccess ? KV4_OK : KV4_ERR_LAUNCH;
}

int kv4_bf16_append(const kv4_layout* l, void* cache, const uint16_t* k_new, const uint16_t* v_new,
                    const int32_t* tok_seq, const int32_t* tok_pos, int32_t T,
                    const int32_t* seq_lens, const int32_t* block_table, int32_t* dev_status,
                    void* stream) {
  int rc = kv4_check_layout(l);
  if (rc != KV4_OK) return rc;
  if (T < 0) return KV4_ERR_INVALID_ARG;
  if (T == 0) return KV4_OK;
  if (!cache || !k_new || !v_new || !tok_seq || !tok_pos || !seq_lens || !block_table)
    return KV4_ERR_INVALID_ARG;
  if (!aligned16(cache) || !aligned16(k_new) || !aligned16(v_new)) return KV4_ERR_INVALID_ARG;
  cudaError_t e = launch_bf16_append(to_layout(l), cache, k_new, v_new, tok_seq, tok_pos, T,
                                     seq_lens, block_table, dev_status, (cudaStream_t)stream);
  return e == cudaSuccess ? KV4_OK : KV4_ERR_LAUNCH;
}

// Workspace of the bf16 comparator: the split kernel's (as kv4_decode_attn
// with a fixed split count), or for the tensor-core kernel its per-item
// partials, one ticket per pair and the item counter.
static size_t bf16_ws_mma(const kv4_layout* l, int num_seqs) {
  const Layout L = to_layout(l);
  const size_t items = (size_t)bf16_mma_items(L, num_seqs), G = l->num_q_heads / l->num_kv_heads;
  return round256(items * G * l->head_dim * sizeof(float)) + round256(items * G * sizeof(float)) +
         round256(((size_t)num_seqs * l->num_kv_heads + 1) * sizeof(int32_t));
}
static size_t bf16_ws_bytes(const kv4_layout* l, int num_seqs, const Plan& p) {
  size_t n = ws_bytes(l, num_seqs, p, -1);
  if (bf16_mma_supported(to_layout(l), num_seqs)) n = std::max(n, bf16_ws_mma(l, num_seqs));
  return n;
}

size_t kv4_bf16_workspace_bytes(const kv4_layout* l, int32_t num_seqs, int32_t max_splits) {
  if (kv4_check_layout(l) != KV4_OK || num_seqs < 0 || max_splits < 0) return 0;
  return bf16_ws_bytes(l, num_seqs, make_plan(l, num_seqs, max_splits, false));
}

int kv4_bf16_decode_attn(const kv4_layout* l, const void* cache, const uint16_t* q,
                         const int32_t* seq_lens, int32_t num_seqs, const int32_t* block_table,
                         float sm_scale, int32_t max_splits, void* workspace,
                         size_t workspace_bytes, uint16_t* out, float* out_lse,
                         int32_t* dev_status, void* stream) {
  int rc = kv4_check_layout(l);
  if (rc != KV4_OK) return rc;
  if (num_seqs < 0 || num_seqs > l->max_seqs || max_splits < 0) return KV4_ERR_INVALID_ARG;
  if (num_seqs == 0) return KV4_OK;
  if (!cache || !q || !seq_lens || !block_table || !workspace || !out) return KV4_ERR_INVALID_ARG;
  if (!aligned16(cache) || !aligned16(q) || !aligned16(workspace)) return KV4_ERR_INVALID_ARG;
  const Plan p = make_plan(l, num_seqs, max_splits, false);
  if (workspace_bytes < bf16_ws_bytes(l, num_seqs, p)) return KV4_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  const Layout L = to_layout(l);
  cudaError_t e;
  if (max_splits == 0 && bf16_mma_supported(L, num_seqs)) {
    // tensor-core kernel: partials per work item, then the tickets and the
    // item counter, which start at zero
    const size_t items = (size_t)bf16_mma_items(L, num_seqs), G = l->num_q_heads / l->num_kv_heads;
    const size_t o = round256(items * G * l->head_dim * sizeof(float));
    const size_t z = round256(items * G * sizeof(float));
    float* part_o = (float*)workspace;
    float* part_lse = (float*)((char*)workspace + o);
    int32_t* tickets = (int32_t*)((char*)workspace + o + z);
    const size_t n_tk = (size_t)num_seqs * l->num_kv_heads;
    if (cudaMemsetAsync(tickets, 0, (n_tk + 1) * sizeof(int32_t), st) != cudaSuccess)
      return KV4_ERR_LAUNCH;
    e = launch_bf16_decode_mma(L, cache, q, seq_lens, num_seqs, block_table, sm_scale, part_o,
                               part_lse, tickets, tickets + n_tk, out, out_lse, dev_status, st);
  } else {
    // the comparator's split kernel (CUDA cores): sized as for a fixed split count
    const Workspace w = ws_layout(l, num_seqs, p, -1, workspace);
    if (cudaMemsetAsync(w.tickets, 0, w.ticket_bytes, st) != cudaSuccess) return KV4_ERR_LAUNCH;
    e = launch_bf16_decode(L, cache, q, seq_lens, num_seqs, block_table, sm_scale, p.n4,
                           p.pages_per_split, w.part_o, w.part_lse, w.tickets, out, out_lse,
                           dev_status, st);
  }
  return e == cudaSuccess ? KV4_OK : KV4_ERR_LAUNCH;
}

}  // extern "C"
