// noalloc.cu -- split-KV decode for callers that cannot allocate device memory.
//
// gqa_attn_decode_noalloc() runs the same two kernels as gqa_attn_decode()
// followed by gqa_attn_decode_combine(), but keeps the split partials in a
// fixed scratch array that lives in this library's device image instead of a
// caller-provided workspace.  It exists for callers that must not call
// cudaMalloc at decode time: code running inside a custom allocator's critical
// section (where a nested allocation would deadlock or recurse), or a serving
// process whose device memory pool is sized up front and may not grow.  Such
// callers still pass their own q, K/V cache, seq_lens, out and lse buffers.
#include <mutex>

#include "gqa_attn.h"
#include "internal.h"

// 16 MiB of split partials per device, held for as long as the library is loaded.
static constexpr size_t kNoAllocScratchBytes = 16u << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device with that device current.  In host code the array's name is
// only a host-side stand-in, so the address must come from the runtime.  The
// cached address belongs to the device's current context: after a
// cudaDeviceReset() it is stale (see the header).
gqa_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return GQA_ERR_CUDA;
  if (dev >= kMaxDevices) return GQA_ERR_UNSUPPORTED;  // ordinals past the address table
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return GQA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return GQA_OK;
}

}  // namespace

extern "C" {

gqa_status gqa_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* seq_lens, int B, int S_max, int H_q, int H_kv,
                                   int d, float scale, int n_split, void* out, float* lse,
                                   gqa_stream_t stream) {
  if (n_split < 1) return GQA_ERR_INVALID_ARG;
  if (gqa_attn_decode_workspace_bytes(B, H_q, d, n_split) > kNoAllocScratchBytes)
    return GQA_ERR_INVALID_ARG;  // partials would not fit the fixed scratch array
  void* scratch = nullptr;
  if (n_split > 1) {
    gqa_status st = scratch_for_current_device(&scratch);
    if (st != GQA_OK) return st;
  }
  gqa_status st = gqa_attn_decode(q, k_cache, v_cache, seq_lens, B, S_max, H_q, H_kv, d, scale,
                                  n_split, scratch, out, lse, stream);
  if (st != GQA_OK || n_split == 1) return st;
  return gqa_attn_decode_combine(scratch, B, H_q, d, n_split, out, lse, stream);
}

}  // extern "C"
