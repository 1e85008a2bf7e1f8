// kv4_noalloc.cu -- decode attention for callers that cannot allocate device
// memory.
//
// kv4_decode_attn needs a workspace (the splits' partial outputs, their
// log-normalisers and one completion counter per sequence and kv head) that
// the caller allocates.  Some callers cannot: a plug-in whose host framework
// has already reserved all free device memory for its own pool, a decode loop
// that must not call cudaMalloc because it synchronises the device and can
// fail under memory pressure, or a runtime that exposes no device allocator
// at all.  kv4_decode_attn_noalloc serves them from one fixed scratch array
// that lives in this library's device image: every GPU that loads the library
// holds these kNoAllocScratchBytes until the process exits, and nothing is
// allocated or freed per call.
#include <mutex>

#include "kv4_common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB

// The shared scratch.  Host code cannot use the name as a device address; it
// looks the address up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (set up on first use).
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t kv4_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int kv4_decode_attn_noalloc(const kv4_layout* layout, const void* paged, const void* side,
                            const uint16_t* q, const int32_t* seq_lens, int32_t num_seqs,
                            const int32_t* block_table, float sm_scale, int32_t max_splits,
                            uint16_t* out, float* out_lse, int32_t* dev_status, void* stream) {
  const int rc = kv4_check_layout(layout);
  if (rc != KV4_OK) return rc;
  if (num_seqs < 0 || max_splits < 0) return KV4_ERR_INVALID_ARG;
  if (num_seqs == 0) return KV4_OK;
  const size_t need = kv4_workspace_bytes(layout, num_seqs, max_splits);
  if (need == 0 || need > kNoAllocScratchBytes) return KV4_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return KV4_ERR_LAUNCH;
  return kv4_decode_attn(layout, paged, side, q, seq_lens, num_seqs, block_table, sm_scale,
                         max_splits, scratch, kNoAllocScratchBytes, out, out_lse, dev_status,
                         stream);
}

}  // extern "C"
