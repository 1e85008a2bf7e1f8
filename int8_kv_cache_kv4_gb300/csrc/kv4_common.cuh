// kv4_common.cuh -- internal helpers shared by the kv4 CUDA translation units:
// packed-layout offsets, status reporting, and thin inline-PTX wrappers for
// the sm_100-family asynchronous copy engine (mbarrier + cp.async.bulk).
#pragma once
#include <cmath>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "kv4.h"

namespace kv4 {

constexpr int kPage = 16;

// ---------------------------------------------------------------- layout
// Bytes of one (page, kv head) chunk: K codes, V codes, K meta, V meta.
__host__ __device__ inline int chunk_bytes(int d_h, int g) { return 16 * d_h + 128 * (d_h / g); }
__host__ __device__ inline int codes_off_v(int d_h) { return 8 * d_h; }  // 16 rows * d_h/2
__host__ __device__ inline int meta_off_k(int d_h) { return 16 * d_h; }
__host__ __device__ inline int meta_off_v(int d_h, int g) { return 16 * d_h + 64 * (d_h / g); }
// Byte offset inside a V code row of logical byte `b` (channels 2b, 2b + 1)
// for slot `t`: the row's 16-byte pieces (32 channels each) are XOR-permuted
// by (t >> 1) so that transposing 16-byte reads of one piece across 8
// consecutive slots touch distinct banks.
__host__ __device__ inline int row_byte(int b, int t, int d_h) {
  const int np = d_h / 32;
  return 16 * ((b >> 4) ^ ((t >> 1) & (np - 1))) + (b & 15);
}
// Byte offset inside a K code row of the byte holding channels c and c + 1
// (c even).  The row is four quarters q = 0..3 of d_h/32 words each; word b
// of quarter q holds the 8 channels 32 b + 8 q .. 32 b + 8 q + 7 of block b.
// A lane that needs quarter q of every block reads one contiguous run.
__host__ __device__ inline int k_row_byte(int c, int d_h) {
  const int nb = d_h / 32;
  return 4 * (nb * ((c & 31) >> 3) + (c >> 5)) + ((c & 7) >> 1);
}
// V metadata of a chunk: Delta_v for every (slot, group), then m_v, each
// [4 quads][d_h/g groups][4 slots] fp16, quad u holding slots 2u, 2u + 1,
// 2u + 8, 2u + 9 (the slots one tensor-core lane multiplies).
__host__ __device__ inline int v_meta_half(int t, int grp, int ng) {
  return (((t & 7) >> 1) * ng + grp) * 4 + 2 * (t >> 3) + (t & 1);
}
__host__ __device__ inline int v_delta_byte(int t, int grp, int d_h, int g) {
  return 16 * d_h + 64 * (d_h / g) + 2 * v_meta_half(t, grp, d_h / g);
}
__host__ __device__ inline int v_offset_byte(int t, int grp, int d_h, int g) {
  return 16 * d_h + 96 * (d_h / g) + 2 * v_meta_half(t, grp, d_h / g);
}

// Byte offset of channel c inside an INT8 side-cache code row of slot t: the
// row's 16-byte pieces (16 channels each) are XOR-swizzled by the slot.
__host__ __device__ inline int side_byte(int c, int t, int d_h) {
  return 16 * ((c >> 4) ^ (t & (d_h / 16 - 1))) + (c & 15);
}

// Side-cache block of one (slot, kv head): K8 codes [NS][d_h], V8 codes
// [NS][d_h], K8 scales [NSP], V8 scales [NSP] with NSP = NS rounded up to 8,
// so that every 8-slot run of codes or scales starts on a 16-byte boundary.
__host__ __device__ inline int side_scale_entries(int S, int R) { return (S + R + 7) / 8 * 8; }
__host__ __device__ inline long long side_block_bytes(int d_h, int S, int R) {
  return 2LL * (S + R) * d_h + 4LL * side_scale_entries(S, R);
}

// ------------------------------------------------ one-time launch setup
// Per-device, per-kernel host setup (the dynamic shared-memory attribute and,
// for the persistent kernel, its resident-CTA count) costs microseconds of
// host time; it runs once per device and its result is cached.
constexpr int kMaxDevices = 64;
struct OnceSetup {
  std::atomic<int> state[kMaxDevices];  // 1 = done (static storage: zero at start)
  int value[kMaxDevices];
  std::mutex mu;
};
template <class Init>
inline cudaError_t once_per_device(OnceSetup& s, Init init, int* value) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!s.state[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(s.mu);
    if (!s.state[dev].load(std::memory_order_relaxed)) {
      int v = 0;
      if ((e = init(dev, &v)) != cudaSuccess) return e;
      s.value[dev] = v;
      s.state[dev].store(1, std::memory_order_release);
    }
  }
  *value = s.value[dev];
  return cudaSuccess;
}

// Upper bound on the grid of the work-balanced decode kernel (it sizes the
// grid to the resident-CTA capacity of the GPU, 760 on a 152-SM GB300).
constexpr int kMaxStreamCtas = 1024;

struct Layout {
  int h_q, h_kv, d_h, g, S, R;
  int max_seqs, num_pages, max_pages;
};

// Region split of one sequence (KV4-RL Sec. 5.2-5.3): protected positions are
// [0, sink_end) and [rec_start, L); the INT4 region is [sink_end, rec_start).
struct Regions {
  int sink_end, rec_start, n_prot;
};
__host__ __device__ inline Regions regions(int L, int S, int R) {
  Regions r;
  r.sink_end = L < S ? L : S;
  int rs = L - R;
  r.rec_start = rs > r.sink_end ? rs : r.sink_end;
  r.n_prot = r.sink_end + (L - r.rec_start);
  return r;
}
// i-th protected position (0 <= i < n_prot) and its side slot.
__host__ __device__ inline int prot_pos(const Regions& r, int i) {
  return i < r.sink_end ? i : r.rec_start + (i - r.sink_end);
}
__host__ __device__ inline int side_slot(int p, int S, int R) { return p < S ? p : S + (p % R); }

__device__ inline void set_status(int32_t* st, int bits) {
  if (st && bits) atomicOr(st, bits);
}

// ------------------------------------------------- Hadamard rotation (eq. 3.4)
// In-place normalized Hadamard rotation of a head_dim-vector spread over the
// warp: lane l holds channels 4l..4l+3 in x[0..3]; lanes at or past d/4 hold
// zeros and only ever pair among themselves.  The butterfly runs stages
// h = 1, 2, 4, ..., d/2 in that order; at each, the pair of channels (i, i+h)
// with bit h of i clear becomes (a + b, a - b) for a = x_i, b = x_(i+h).
// Stages 1 and 2 stay inside a lane; stage h = 4m pairs lane l with lane
// l ^ m.  A final multiply by c (the fp32 value nearest 1/sqrt(d)) normalizes.
// Every step is an explicitly rounded fp32 operation in this fixed order, so
// the result is reproducible bit for bit by any implementation of the same
// order.  All 32 lanes must call it (full-mask shuffles).
__device__ inline void hadamard_warp(float x[4], int d, float c) {
  const float a0 = __fadd_rn(x[0], x[1]), a1 = __fsub_rn(x[0], x[1]);
  const float a2 = __fadd_rn(x[2], x[3]), a3 = __fsub_rn(x[2], x[3]);
  x[0] = __fadd_rn(a0, a2);
  x[2] = __fsub_rn(a0, a2);
  x[1] = __fadd_rn(a1, a3);
  x[3] = __fsub_rn(a1, a3);
  const int lane = threadIdx.x & 31;
  for (int m = 1; 4 * m < d; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, x[i], m);
      x[i] = upper ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = __fmul_rn(x[i], c);
}

// fp32 value nearest 1/sqrt(d), computed on the host in double precision.
inline float hadamard_scale(int d) { return (float)(1.0 / std::sqrt((double)d)); }

// ------------------------------------------------------------ conversions
__device__ inline float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }
__device__ inline float f16_bits_to_f32(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)h));
}
// float -> bf16 bits, round to nearest even (NaN kept quiet)
__device__ inline uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ------------------------------------------- mbarrier + 1-D bulk async copy
__device__ inline uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ inline void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ inline void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ inline void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

// Bounded wait on an mbarrier phase.  Returns false if the phase did not
// complete within the iteration limit (the caller then reports an error and
// skips the data instead of hanging).
__device__ inline bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iters = 4000000u) {
  uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < max_iters; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned) completing on `bar` via complete_tx.
__device__ inline void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// The same with shared-memory addresses already in the shared window (saves
// the generic-to-shared conversions on a producer's per-copy path).
__device__ inline void mbar_arrive_expect_tx_s(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ inline void mbar_arrive_s(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ inline void bulk_g2s_s(uint32_t smem_dst, const void* gmem_src, uint32_t bytes,
                                  uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_dst),
      "l"(gmem_src), "r"(bytes), "r"(bar)
      : "memory");
}

// ------------------------------------------------------------ reductions
__device__ inline float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ inline float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace kv4
