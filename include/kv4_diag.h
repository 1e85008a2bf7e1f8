/*
 * kv4_diag.h -- diagnostics beside the KV4-RL decode library (libkv4_diag.so,
 * a separate library; libkv4.so does not contain or need it).
 *
 * kv4_diag_mma_rate -- tensor-pipe rate probe.  KV4-RL's deployed decode
 * multiplies INT8 operands on the tensor cores (Sec. 5.3 and App. A.3
 * "Integer decode path"); libkv4.so's decode multiplies fp16 ones.  This
 * probe measures both kinds of product in the MMA forms sm_103a offers:
 *   kind 0: warp-level mma.sync m16n8k16, fp16 operands, fp32 accumulation
 *           (4,096 flops each); `blocks` CTAs of 8 warps, each warp issuing
 *           4 x `iters` MMAs on register operands
 *   kind 1: warp-level mma.sync m16n8k32, int8 operands, int32 accumulation
 *           (8,192 ops each); same launch shape
 *   kind 2: tcgen05.mma kind::f16, M = 128, N = 256, K = 16, shared-memory
 *           operands, fp32 accumulator in tensor memory (1,048,576 flops
 *           each); `blocks` CTAs of 128 threads, one thread of each issuing
 *           `iters` MMAs back to back and waiting for their completion
 * *   There is no tcgen05 int8 kind: ptxas rejects tcgen05.mma kind::i8 for
 *   sm_103a ("Feature '.kind::i8' not supported on .target 'sm_103a'").
 * Time the call with events on `stream` to get the rate.
 *   sink    device, 4 bytes.  Kinds 0 and 1 write it only to keep the results
 *           live; kind 2 ORs 1 into it (as an int32 status word) if the
 *           bounded wait for their MMAs expired.  The caller zeroes it.
 *   Returns KV4_DIAG_ERR_INVALID_ARG for another kind, non-positive sizes or
 *   a NULL sink (nothing is launched), KV4_DIAG_ERR_LAUNCH if the launch
 *   failed.  It allocates nothing and does not synchronise.
 */
#ifndef KV4_DIAG_H_
#define KV4_DIAG_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KV4_DIAG_OK 0
#define KV4_DIAG_ERR_INVALID_ARG 1
#define KV4_DIAG_ERR_LAUNCH 3

int kv4_diag_mma_rate(int32_t kind, int32_t blocks, int32_t iters, uint32_t* sink, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KV4_DIAG_H_ */
