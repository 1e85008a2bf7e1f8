/*
 * kv4.h -- C ABI of the KV4-RL mixed INT4/INT8 paged KV cache for GB300 (sm_103a).
 *
 * The method ("KV4-RL: Unlocking Faster Asynchronous Rollouts for RLVR with INT4
 * KV Cache Quantization"):
 *   - every cached K/V position is stored as head-wise affine INT4 codes with an
 *     FP16 scale Delta and FP16 offset m per group of channels, x^ = Delta*c + m
 *     (Sec. 3 eq. 3.3; Sec. 5.1; App. A.3 "Encoding and allocation");
 *   - the first S positions (attention sinks) and the most recent R positions
 *     additionally live in an INT8 side cache with one symmetric scale per
 *     token and head, computed from the source vector (Sec. 5.2; App. A.3);
 *   - decode attention reads protected positions from the side cache and all
 *     others from the INT4 pages (disjoint regions, Sec. 5.3) and merges the
 *     regional results with the log-sum-exp identity of App. A.3 eq. A1, which
 *     also merges context splits.
 *
 * Conventions for every entry point
 *   - Memory: the caller owns all memory.  Device pointers are plain CUDA
 *     device addresses (e.g. from cudaMalloc or a PyTorch tensor); host
 *     pointers are noted as such.  The library never allocates, frees or
 *     synchronises; all device work is enqueued on `stream`, a cudaStream_t
 *     passed as void* (NULL = the legacy default stream).
 *   - Return value: KV4_OK, or a KV4_ERR_* code for problems found on the host
 *     (NULL pointers, bad sizes, unsupported shapes, launch failures).  Nothing
 *     is enqueued when an error is returned.
 *   - dev_status: a device int32 that kernels OR KV4_STATUS_* bits into for
 *     data-dependent problems (a block-table entry outside the pool, a position
 *     outside the sequence, a non-finite input).  Kernels never trap: the
 *     offending token / page is skipped.  The caller zeroes it and reads it
 *     back when convenient.  May be NULL (problems are then silently skipped).
 *   - bf16 tensors are passed as const uint16_t* (IEEE bfloat16 bit patterns).
 *   - Stream order and early launch: kv4_quant_append and, when it runs the
 *     work-balanced kernel (max_splits = 0), kv4_decode_attn (and its
 *     _hadamard / _noalloc forms) launch their kernels with programmatic
 *     stream serialisation, so a call's first kernel may start while the
 *     kernel before it on the stream finishes.  Before waiting for that kernel
 *     they read only inputs the library never writes: the append its new K/V
 *     rows, tok_seq, tok_pos, seq_lens and block_table; the decode seq_lens
 *     (and, as L2 prefetches, q and block_table).  Such an input must
 *     therefore be complete when the kernel before the call has completed: an
 *     ordinary kernel, a copy or an event wait before the call all ensure it;
 *     a kernel of the caller's that lets its dependents launch early must not
 *     write them.  Everything else (the caches, the workspace, out) is
 *     touched only after the wait.  In turn the append, and the decode once
 *     each of its CTAs has started, let the next kernel on the stream launch
 *     early: a caller kernel launched with programmatic stream serialisation
 *     after them must call cudaGridDependencySynchronize() before it touches
 *     anything the call reads or writes (ordinary launches are unaffected).
 *
 * Packed layout (bit-exact; the CPU oracle restates it independently)
 *   paged cache  = [num_pages][num_kv_heads][chunk]
 *     chunk      = K codes [16 slots][head_dim/2 bytes]
 *                  V codes [16 slots][head_dim/2 bytes]
 *                  K meta  [16 slots][head_dim/g][2 x fp16: Delta, m]
 *                  V Delta [4 quads][head_dim/g][4 x fp16]
 *                  V m     [4 quads][head_dim/g][4 x fp16]
 *     A byte of a code row holds two consecutive channels, the even one in
 *     its low nibble.
 *     K code row: four quarters q = 0..3 of head_dim/32 four-byte words; word
 *     b of quarter q holds channels 32b + 8q .. 32b + 8q + 7 (block b), so
 *     that one 16-byte read gives a lane one word of every block.
 *     V code row: byte i holds channels 2i and 2i+1, cut into 16-byte pieces
 *     (32 channels each); piece P of slot t is stored at piece position
 *     P ^ ((t >> 1) & (head_dim/32 - 1)), so that transposing shared-memory
 *     reads across consecutive slots hit distinct banks.
 *     V metadata: quad u lists the slots 2u, 2u+1, 2u+8, 2u+9 in that order;
 *     entry (u, group, k) of V Delta / V m holds the Delta / m of the k-th
 *     slot of quad u for that group (the four slots one tensor-core lane
 *     multiplies, read as one 8-byte run per group).
 *     Position p of request slot s lives in page block_table[s][p / 16],
 *     slot p % 16.
 *     chunk bytes = 16*head_dim + 128*head_dim/g  (2560 at d=128, g=32).
 *   side cache   = [max_seqs][num_kv_heads][block], NS = sink + recent,
 *                  NSP = NS rounded up to a multiple of 8
 *     block      = K8 codes [NS][head_dim] int8, V8 codes [NS][head_dim] int8,
 *                  K8 scale [NSP] fp16, V8 scale [NSP] fp16 (entries NS..NSP-1
 *                  are padding, never written), 2*NS*head_dim + 4*NSP bytes;
 *                  every 8-slot run of codes or scales starts 16-byte aligned.
 *     An INT8 code row (one slot) is cut into 16-byte pieces of 16 channels;
 *     piece P of slot t is stored at piece position P ^ (t % (head_dim/16)),
 *     so that reads of one piece across 8 consecutive slots hit distinct banks.
 *     Sink position p < S uses slot p; position p >= S uses ring slot
 *     S + (p mod R).  All multi-byte fields are little-endian.
 *   bf16 comparator cache = [num_pages][num_kv_heads][2 (K,V)][16][head_dim] bf16.
 *
 * Quantization rules (the pages leave rounding open; these readings are fixed):
 *   INT4 group of g channels: m = fp16 rounded down from min(x);
 *     Delta = fp16 rounded up from ((max(x) -up m) /up 15) (fp32, upward);
 *     c = clamp(rne((x -rn m) /rn Delta), 0, 15), and c = 0 when Delta = 0.
 *   INT8 token-head vector: s = fp16 rounded up from (max|x| /up 127);
 *     c = clamp(rne(x /rn s), -127, 127), and c = 0 when s = 0.
 *   A group or vector with a non-finite element (or whose metadata overflows
 *   fp16) is stored as all zeros and sets KV4_STATUS_NONFINITE.
 *
 * Operand range of the tensor-core decode kernels (the default one and the
 * split kernel): their PV products take P' = p * Delta_v (INT4) or p * s_v
 * (INT8) as fp16, with softmax weights p <= 2^8 relative to a lazily moved
 * reference.  They are accurate while every stored Delta_v and s_v is zero or
 * a normal fp16 value of at most 255.875: V group ranges (max - min) from
 * 15 * 2^-14 = 9.2e-4 up to 3838, and max |V| of a protected token-head from
 * 127 * 2^-14 = 7.8e-3 up to 32496 (or exactly zero).  The append encodes
 * other V exactly as the rules above say and sets KV4_STATUS_V_RANGE; a cache
 * holding such V decodes correctly only with the CUDA-core kernel
 * (kv4_set_decode_kernel(KV4_KERNEL_CUDA_CORE)), which computes in fp32.
 * (Measured: V scaled by 2^-6 .. 2^8 stays within the output tolerance on
 * every kernel; at 2^-10 the protected scales are subnormal and the default
 * kernel misses it.)  The INT8 units also take the query as fp16: |q| below
 * 65504, exact for |q| >= 2^-14 (bf16 values below that lose low bits; q
 * scaled by 2^-12 stays within the tolerance).
 */
#ifndef KV4_H_
#define KV4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KV4_ABI_VERSION 3

/* host return codes */
#define KV4_OK 0
#define KV4_ERR_INVALID_ARG 1 /* NULL pointer, negative size, inconsistent layout */
#define KV4_ERR_UNSUPPORTED 2 /* head_dim not in {64,128}, g not in {32,64,128}, ... */
#define KV4_ERR_LAUNCH 3      /* a CUDA launch failed (cudaGetLastError) */
#define KV4_ERR_WORKSPACE 4   /* workspace smaller than kv4_workspace_bytes() */

/* device status bits (ORed into *dev_status) */
#define KV4_STATUS_BAD_PAGE 1  /* block-table entry outside [0, num_pages) */
#define KV4_STATUS_BAD_POS 2   /* position < 0, >= seq_len, or beyond the block table */
#define KV4_STATUS_BAD_SEQ 4   /* request slot outside [0, max_seqs) */
#define KV4_STATUS_NONFINITE 8 /* non-finite input, or metadata overflowing fp16 */
#define KV4_STATUS_BAD_LEN 16  /* decode: seq_len < 0 or beyond the block-table capacity */
#define KV4_STATUS_TIMEOUT 32  /* a bounded wait inside a kernel expired; its outputs are invalid */
#define KV4_STATUS_INTERNAL 64 /* a kernel's internal consistency check failed; outputs invalid */
#define KV4_STATUS_V_RANGE 128 /* append: a V Delta or protected V scale >= 256 or subnormal */

/* Shape of one attention layer's cache.  All fields are host values. */
typedef struct kv4_layout {
  int32_t num_q_heads;       /* h_q (a multiple of num_kv_heads, h_q/h_kv <= 8) */
  int32_t num_kv_heads;      /* h_kv (1 .. 65536) */
  int32_t head_dim;          /* d_h: 64 or 128 */
  int32_t page_size;         /* tokens per page: must be 16 (App. A.2) */
  int32_t int4_group;        /* g: 32, 64 or 128 and g <= head_dim */
  int32_t int8_group;        /* INT8 group: must equal head_dim (per token-head) */
  int32_t sink;              /* S >= 0: protected prefix length */
  int32_t recent;            /* R >= 0: protected recent window */
  int32_t max_seqs;          /* request slots: rows of the block table and side cache */
  int32_t num_pages;         /* pages in the pool */
  int32_t max_pages_per_seq; /* row stride of block_table */
} kv4_layout;

/* ABI version and a static, human-readable name for a return code or status bit. */
int kv4_abi_version(void);
const char* kv4_status_string(int code);

/* Decode kernel selection (process-wide; default KV4_KERNEL_AUTO).  AUTO picks
 * the fastest kernel measured on GB300 for the layout: for head_dim 128 with 4
 * query heads per kv head, the work-balanced persistent tensor-core kernel
 * (STREAM) when max_splits is 0 and the warp-level split kernel (MMA_SYNC)
 * when the caller fixes the split count; the CUDA-core kernel otherwise.
 * STREAM cuts every (sequence, kv head) into two-page INT4 units and 16-slot
 * protected units and gives each CTA of a grid that fills the GPU a share of
 * equal cost; it ignores max_splits, so with max_splits > 0 it runs MMA_SYNC.
 * CUDA_CORE selects the fp32 split kernel.  All compute the same result within
 * the stated tolerance.  A kernel that does not support the layout falls back
 * to the CUDA-core kernel.  Any other value leaves the selection unchanged.
 * Returns the previous value. */
#define KV4_KERNEL_AUTO 0
#define KV4_KERNEL_CUDA_CORE 1
#define KV4_KERNEL_MMA_SYNC 2
#define KV4_KERNEL_STREAM 4
int kv4_set_decode_kernel(int which);

/* Validate a layout; KV4_OK or a KV4_ERR_* code. */
int kv4_check_layout(const kv4_layout* layout);

/* Sizes in bytes of the caller-allocated buffers (0 when the layout is invalid). */
size_t kv4_paged_cache_bytes(const kv4_layout* layout); /* INT4 pages: codes + metadata */
size_t kv4_side_cache_bytes(const kv4_layout* layout);  /* INT8 sink + ring, per slot */
size_t kv4_bf16_cache_bytes(const kv4_layout* layout);  /* comparator pages */

/* Number of context splits per (sequence, kv head) that the split kernels use
 * for `num_seqs` sequences when given `max_splits` (0 = automatic), and the
 * workspace (device scratch: partial outputs, log-normalisers, completion
 * counters and, with max_splits = 0, the work-balanced kernel's start table)
 * kv4_decode_attn needs with that max_splits, for every kernel choice. */
int32_t kv4_num_splits(const kv4_layout* layout, int32_t num_seqs, int32_t max_splits);
size_t kv4_workspace_bytes(const kv4_layout* layout, int32_t num_seqs, int32_t max_splits);

/*
 * kv4_quant_append -- quantize-on-append (KV4-RL Sec. 5.3 and App. A.3
 * "Encoding and allocation": the INT4 entry and, for protected positions, the
 * INT8 entry are both computed from the new token's source K/V).
 *
 * For each of the T new tokens t (request slot tok_seq[t], position
 * tok_pos[t]): writes the INT4 codes and per-group (Delta, m) of K and V into
 * page block_table[slot][pos/16], slot pos%16, for every kv head; and, when
 * the position is protected for the sequence's length after this append --
 * pos < S, or R > 0 and pos >= seq_lens[slot] - R -- writes the INT8 codes and
 * scale into the side cache (sink slot pos, or ring slot S + pos mod R).
 * Multi-token appends (prefill / re-prefill population, App. A.3) may list
 * tokens in any order; tokens must not repeat a (slot, position) pair.
 *
 *   paged, side     device, written in place (layout above)
 *   k_new, v_new    device bf16 [T][num_kv_heads][head_dim]
 *   tok_seq,tok_pos device int32 [T]
 *   seq_lens        device int32 [max_seqs]: lengths after this append
 *   block_table     device int32 [max_seqs][max_pages_per_seq]
 *   T == 0 is a no-op.
 */
int kv4_quant_append(const kv4_layout* layout, void* paged, void* side, const uint16_t* k_new,
                     const uint16_t* v_new, const int32_t* tok_seq, const int32_t* tok_pos,
                     int32_t T, const int32_t* seq_lens, const int32_t* block_table,
                     int32_t* dev_status, void* stream);

/*
 * Hadamard K-rotation (KV4-RL Sec. 3 eq. 3.4: for a normalized Hadamard H with
 * H H^T = I, (qH)(kH)^T = q k^T, so keys may be stored rotated when queries
 * are rotated too; App. A.3 "Encoding and allocation": K and Q rotated after
 * RoPE, V in its original basis; App. D.4 keeps the rotation K-only).
 *
 * H is the normalized Sylvester matrix of order head_dim (H_1 = [1],
 * H_2m = [[H_m, H_m], [H_m, -H_m]], divided by sqrt(head_dim)); no random
 * signs.  It is evaluated in fp32 in one fixed order: butterfly stages
 * h = 1, 2, 4, ..., head_dim/2, each turning the channel pair (i, i+h) with
 * bit h of i clear into (a + b, a - b), then a multiply by the fp32 value
 * nearest 1/sqrt(head_dim); every operation rounds to nearest even.
 *
 * kv4_quant_append_hadamard -- kv4_quant_append with every K vector replaced
 *   by H k (fp32, before both the INT4 and the INT8 encoding); V is encoded
 *   as given.  Same arguments, layout, validation and status bits.  A cache
 *   must be written by one of the two entry points only, and read with
 *   rotated queries when written by this one.
 *
 * kv4_hadamard_bf16 -- the query side: each of `rows` rows of `dim` bf16
 *   values x becomes H x rounded to bf16 (nearest even).  Use it on q before
 *   kv4_decode_attn over a cache written by kv4_quant_append_hadamard (or call
 *   kv4_decode_attn_hadamard, which rotates the query itself); the scores are
 *   then sm_scale * (Hq).(k^ of Hk).
 *     x, y   device bf16 [rows][dim], 8-byte aligned; y == x (in place) is
 *            allowed, any other overlap is KV4_ERR_INVALID_ARG
 *     dim    64 or 128 (the supported head dimensions), else KV4_ERR_INVALID_ARG
 *     rows   >= 0; rows == 0 is a no-op
 *   Non-finite inputs give non-finite outputs (no status word).
 */
int kv4_quant_append_hadamard(const kv4_layout* layout, void* paged, void* side,
                              const uint16_t* k_new, const uint16_t* v_new,
                              const int32_t* tok_seq, const int32_t* tok_pos, int32_t T,
                              const int32_t* seq_lens, const int32_t* block_table,
                              int32_t* dev_status, void* stream);
int kv4_hadamard_bf16(const uint16_t* x, uint16_t* y, int32_t rows, int32_t dim, void* stream);

/*
 * FP4 probe formats (KV4-RL App. D.4, Fig. A4(c)): the pages compare affine
 * INT4 with NVFP4 (E2M1 values, one E4M3 scale per 16 elements and one FP32
 * global scale per token-head vector, 4.75 bits per element) and MXFP4 (E2M1
 * values, one E8M0 scale per 32 elements, 4.25 bits per element) as fidelity
 * probes that reconstruct the stored cache and attend with bf16 operands; no
 * FP4 attention kernel is part of the method.  These entry points write such a
 * cache and reconstruct it into the bf16 comparator layout, so that
 * kv4_bf16_decode_attn computes the probe's attention.
 *
 * Scale rules (one fp32 operation each, rounded to nearest even):
 *   NVFP4  S = max|x| / 2688 over the token-head vector (2688 = 6 * 448);
 *          per block of 16: s_b = E4M3(max|x_b| / (6 S)), e_b = value(s_b) * S,
 *          q = E2M1(x / e_b), q = 0 when e_b = 0
 *   MXFP4  per block of 32: E = floor(log2 max|x_b|) - 2 clamped to
 *          [-127, 127] (-127 for an all-zero block), q = E2M1(x * 2^-E)
 *   E2M1 rounds to the nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6 with ties to the
 *   even code, saturates at 6 and keeps the sign; E4M3 rounds to nearest
 *   even and saturates at 448.  A vector with a non-finite element is stored
 *   as zeros and sets KV4_STATUS_NONFINITE.
 *
 * Probe cache = [num_pages][num_kv_heads][K, V][16 slots][row], row =
 *   head_dim/2 + 16 bytes: the E2M1 codes (byte i: channel 2i in the low
 *   nibble, 2i+1 in the high nibble), then the block scales one byte each
 *   (NVFP4 head_dim/16 E4M3, MXFP4 head_dim/32 E8M0), and for NVFP4 the fp32
 *   S (little-endian) at byte head_dim/2 + 12; other bytes are never written.
 *   Size: kv4_fp4_cache_bytes(layout).
 *
 * kv4_fp4_append -- kv4_quant_append's arguments and validation, writing one
 *   probe row per token, kv head and K/V; rotate_k != 0 rotates K first as
 *   kv4_quant_append_hadamard does (V never).  format: KV4_FP4_NVFP4 or
 *   KV4_FP4_MXFP4, else KV4_ERR_INVALID_ARG.
 * kv4_fp4_to_bf16 -- every row of the pool reconstructed (q times its scale,
 *   rounded to bf16 nearest even) into bf16_cache, a device buffer of
 *   kv4_bf16_cache_bytes(layout) in the comparator layout.
 */
#define KV4_FP4_NVFP4 1
#define KV4_FP4_MXFP4 2
size_t kv4_fp4_cache_bytes(const kv4_layout* layout);
int kv4_fp4_append(const kv4_layout* layout, int32_t format, int32_t rotate_k, void* cache,
                   const uint16_t* k_new, const uint16_t* v_new, const int32_t* tok_seq,
                   const int32_t* tok_pos, int32_t T, const int32_t* seq_lens,
                   const int32_t* block_table, int32_t* dev_status, void* stream);
int kv4_fp4_to_bf16(const kv4_layout* layout, int32_t format, const void* cache, void* bf16_cache,
                    void* stream);

/*
 * kv4_decode_attn -- split-KV GQA decode attention over the mixed cache
 * (KV4-RL Sec. 5.3 and App. A.3: disjoint INT4 and protected regions, each
 * split producing a locally normalised output and log-normaliser, merged by
 * eq. A1).  Query head j reads kv head j / (h_q/h_kv).  For sequence b of
 * length L = seq_lens[b], positions [0, min(S,L)) and [max(S, L-R), L) are read
 * from the side cache, the rest from the INT4 pages.  Scores are
 * sm_scale * q.k^ with the bf16 query used as is; softmax and accumulation in
 * fp32.
 *
 *   q           device bf16 [num_seqs][num_q_heads][head_dim]
 *   seq_lens    device int32 [num_seqs]; row b of block_table / side cache is slot b
 *   max_splits  0 = automatic; else an upper bound on splits per (seq, kv head)
 *   workspace   device, >= kv4_workspace_bytes(layout, num_seqs, max_splits) bytes
 *   out         device bf16 [num_seqs][num_q_heads][head_dim] (round to nearest even)
 *   out_lse     device fp32 [num_seqs][num_q_heads] natural-log normaliser, or NULL
 *   A sequence with L == 0 yields out = 0 and out_lse = -inf.
 */
int kv4_decode_attn(const kv4_layout* layout, const void* paged, const void* side,
                    const uint16_t* q, const int32_t* seq_lens, int32_t num_seqs,
                    const int32_t* block_table, float sm_scale, int32_t max_splits,
                    void* workspace, size_t workspace_bytes, uint16_t* out, float* out_lse,
                    int32_t* dev_status, void* stream);

/*
 * kv4_decode_attn_hadamard -- kv4_decode_attn over a cache written by
 * kv4_quant_append_hadamard, with the query rotation done by the call: each
 * query row q is replaced by H q rounded to bf16, exactly as kv4_hadamard_bf16
 * computes it, and the result equals kv4_hadamard_bf16 followed by
 * kv4_decode_attn on the rotated rows, bit for bit (KV4-RL App. A.3
 * "Encoding and allocation": Q rotated with K).  Same arguments, validation
 * and status bits as kv4_decode_attn; q is not modified.  The default kernel
 * rotates each (sequence, kv head) pair's query rows as it loads them.  On the
 * other kernels (max_splits > 0, or a shape the default kernel does not
 * serve) the rotation runs first into `out` as scratch: out must then be
 * 16-byte aligned and must not overlap q, else KV4_ERR_INVALID_ARG.
 */
int kv4_decode_attn_hadamard(const kv4_layout* layout, const void* paged, const void* side,
                             const uint16_t* q, const int32_t* seq_lens, int32_t num_seqs,
                             const int32_t* block_table, float sm_scale, int32_t max_splits,
                             void* workspace, size_t workspace_bytes, uint16_t* out,
                             float* out_lse, int32_t* dev_status, void* stream);

/*
 * kv4_split_combine -- the regional / split merge of KV4-RL App. A.3 eq. A1
 * on its own: for each of `rows` independent rows,
 *   z = log sum_r exp(z_r),   o = sum_r exp(z_r - z) * o_r,
 * with zero weight for parts whose z_r = -inf (empty splits or regions).
 *
 *   part_o    device fp32 [rows][n_parts][head_dim] (locally normalised outputs)
 *   part_lse  device fp32 [rows][n_parts]
 *   out       device bf16 [rows][head_dim]; out_lse device fp32 [rows] or NULL
 *   A row whose parts are all empty yields out = 0, out_lse = -inf.
 */
int kv4_split_combine(const float* part_o, const float* part_lse, int32_t rows, int32_t n_parts,
                      int32_t head_dim, uint16_t* out, float* out_lse, void* stream);

/*
 * Comparator: the same paged GQA decode over an unquantized bf16 cache
 * (layout above), with the same pages and block table.  Not part of the
 * method; used to report the speed-up of the mixed cache and the drift of its
 * outputs.
 *   kv4_bf16_append writes k_new/v_new [T][h_kv][d_h] into the bf16 pages.
 *   kv4_bf16_decode_attn: with max_splits = 0, head_dim 128, 4 query heads
 *   per kv head and num_seqs <= 2048, a tensor-core kernel (bf16 operands,
 *   fp32 accumulation, softmax weights entered as a bf16 head and tail) whose
 *   warps claim chunks of 64 pages of a (sequence, kv head) pair and merge
 *   the chunks of a pair in order (the result does not depend on which warp
 *   took which chunk); otherwise a CUDA-core split kernel with the split plan
 *   of kv4_decode_attn.  Its workspace is kv4_bf16_workspace_bytes(layout,
 *   num_seqs, max_splits) bytes (KV4_ERR_WORKSPACE if smaller).
 */
size_t kv4_bf16_workspace_bytes(const kv4_layout* layout, int32_t num_seqs, int32_t max_splits);
int kv4_bf16_append(const kv4_layout* layout, void* cache, const uint16_t* k_new,
                    const uint16_t* v_new, const int32_t* tok_seq, const int32_t* tok_pos,
                    int32_t T, const int32_t* seq_lens, const int32_t* block_table,
                    int32_t* dev_status, void* stream);
int kv4_bf16_decode_attn(const kv4_layout* layout, const void* cache, const uint16_t* q,
                         const int32_t* seq_lens, int32_t num_seqs, const int32_t* block_table,
                         float sm_scale, int32_t max_splits, void* workspace,
                         size_t workspace_bytes, uint16_t* out, float* out_lse,
                         int32_t* dev_status, void* stream);

/*
 * kv4_decode_attn_noalloc -- kv4_decode_attn for callers that cannot allocate
 * device memory.  The paper has no counterpart; this is a convenience of this
 * library.
 *
 * Who needs it: kv4_decode_attn takes a caller-allocated workspace.  Some
 * callers cannot provide one -- a plug-in whose host framework has reserved
 * all free device memory for its own pool, a decode loop that must not call
 * cudaMalloc (it synchronises the device and can fail under memory pressure),
 * or a runtime with no device allocator.  This entry point computes exactly
 * what kv4_decode_attn computes, taking its workspace from one fixed scratch
 * array compiled into the library instead.
 *
 * Limits and behaviour:
 *   - The scratch holds kv4_noalloc_scratch_bytes() bytes (16 MiB) on every
 *     GPU that loads the library, for the life of the process.  A call whose
 *     kv4_workspace_bytes(layout, num_seqs, max_splits) exceeds it returns
 *     KV4_ERR_WORKSPACE and enqueues nothing.
 *   - Nothing is allocated or freed: the first call on a device looks up the
 *     scratch's device address (cudaGetSymbolAddress, with that device
 *     current) and caches it, so make that first call before any stream
 *     capture.  The cached address belongs to the device's primary context:
 *     resetting the device (cudaDeviceReset) while the library is loaded is
 *     not supported by this entry point.
 *   - The limit depends on the kernel that runs: test
 *     kv4_workspace_bytes(layout, num_seqs, max_splits) <=
 *     kv4_noalloc_scratch_bytes() before the call (at h_q = 32, h_kv = 8,
 *     head_dim 128 the default kernel fits up to 443 sequences).
 *   - All calls share the one scratch array, which keeps the last call's
 *     contents; the completion counters that must start at zero are cleared on
 *     the stream at the start of every call.  Calls whose work overlaps on the
 *     GPU (different streams, or different host threads) race on the scratch
 *     and must be serialised by the caller.
 *   Arguments are those of kv4_decode_attn without workspace/workspace_bytes.
 */
size_t kv4_noalloc_scratch_bytes(void);
int kv4_decode_attn_noalloc(const kv4_layout* layout, const void* paged, const void* side,
                            const uint16_t* q, const int32_t* seq_lens, int32_t num_seqs,
                            const int32_t* block_table, float sm_scale, int32_t max_splits,
                            uint16_t* out, float* out_lse, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KV4_H_ */
