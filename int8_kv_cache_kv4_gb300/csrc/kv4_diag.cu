// kv4_diag.cu -- a tensor-pipe rate probe behind one diagnostic entry point.
//
// KV4-RL's deployed decode is an integer path (Sec. 5.3 and App. A.3
// "Integer decode path": the query quantized to INT8, an integer QK MMA into
// INT32 accumulators, an 8-bit P operand carrying the value scales).  Whether
// that path can pay on a given GPU rests on its INT8 tensor-core rate next to
// the fp16 rate the float path of this library uses.  This kernel measures
// both with the warp-level MMA form the decode kernels issue: every warp runs
// four independent accumulator chains of back-to-back MMAs on register
// operands, so nothing but the tensor pipe limits it.
#include "kv4_common.cuh"

namespace kv4 {
namespace {

template <int Kind>
__global__ void __launch_bounds__(256) mma_rate_kernel(int iters, uint32_t* sink) {
  // operands: fp16 pairs of 1.0 and 0.5 (kind 0), small int8 values (kind 1);
  // the values do not change the rate, they only keep the results finite
  const uint32_t a = Kind == 0 ? 0x3C003C00u : 0x01010101u;
  const uint32_t b = Kind == 0 ? 0x38003800u : 0x02020202u;
  uint32_t acc = 0;
  if (Kind == 0) {
    float d[4][4] = {};
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[c][0]), "+f"(d[c][1]), "+f"(d[c][2]), "+f"(d[c][3])
            : "r"(a), "r"(a), "r"(a), "r"(a), "r"(b), "r"(b));
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) acc += __float_as_uint(d[c][0] + d[c][1] + d[c][2] + d[c][3]);
  } else {
    int d[4][4] = {};
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+r"(d[c][0]), "+r"(d[c][1]), "+r"(d[c][2]), "+r"(d[c][3])
            : "r"(a), "r"(a), "r"(a), "r"(a), "r"(b), "r"(b));
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) acc += (uint32_t)(d[c][0] + d[c][1] + d[c][2] + d[c][3]);
  }
  if (acc == 0x9E3779B9u) sink[0] = acc;  // keeps the chains live; practically never stored
}

}  // namespace
}  // namespace kv4

extern "C" {

int kv4_diag_mma_rate(int32_t kind, int32_t blocks, int32_t iters, uint32_t* sink, void* stream) {
  if ((kind != 0 && kind != 1) || blocks <= 0 || iters <= 0 || !sink) return KV4_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (kind == 0)
    kv4::mma_rate_kernel<0><<<blocks, 256, 0, st>>>(iters, sink);
  else
    kv4::mma_rate_kernel<1><<<blocks, 256, 0, st>>>(iters, sink);
  return cudaGetLastError() == cudaSuccess ? KV4_OK : KV4_ERR_LAUNCH;
}

}  // extern "C"
