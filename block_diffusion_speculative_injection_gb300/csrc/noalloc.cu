// Block attention without any device allocation by the library or the caller.
//
// dflash_block_attention needs a workspace for its split-KV partial results,
// which its caller allocates.  Some callers cannot allocate device memory at
// the point where they run the attention: code inside an inference engine's
// per-request path that must take every buffer from the engine's own pool,
// serving loops that forbid cudaMalloc after start-up because it can
// synchronize the device and fragment memory, and plugin interfaces whose
// execute call has no allocator at all.  This entry point serves them: the
// partials live in a fixed array in device global memory that is part of
// the loaded library image.
#include <cstdio>

#include "internal.cuh"

namespace dflash {

// 16 MiB of split-KV partials.  Every GPU that loads the library holds this
// array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

// Device address of g_attn_scratch, looked up once per device.  Two host
// threads making their first call on one device at the same moment both
// look it up and store the same value.
static std::atomic<void*> g_scratch_ptr[kMaxDevices];

static dflash_status scratch_on_current_device(void** out) {
  const int dev = current_device_slot();
  if (dev < 0) {
    fprintf(stderr, "dflash_block_attention_noalloc: no usable current device\n");
    return DFLASH_E_CUDA;
  }
  void* p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
  if (!p) {
    const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess || !p) {
      fprintf(stderr, "dflash_block_attention_noalloc: cudaGetSymbolAddress failed: %s\n",
              cudaGetErrorString(e));
      return DFLASH_E_CUDA;
    }
    g_scratch_ptr[dev].store(p, std::memory_order_relaxed);
  }
  *out = p;
  return DFLASH_OK;
}

}  // namespace dflash

using namespace dflash;

extern "C" {

dflash_status dflash_block_attention_noalloc(int32_t batch, int32_t n_heads, int32_t n_kv_heads,
                                             int32_t ctx_len, int32_t block, int32_t causal,
                                             const void* q_dev, const void* k_dev,
                                             const void* v_dev, void* out_dev,
                                             dflash_stream_t stream) {
  const int64_t need = block_attention_workspace(batch, n_heads, n_kv_heads, 128, ctx_len, block);
  if (need < 0) return DFLASH_E_INVALID_ARG;
  if (need > (int64_t)kNoAllocScratchBytes) {
    fprintf(stderr,
            "dflash_block_attention_noalloc: these sizes need %lld bytes of split-KV scratch, "
            "more than the fixed %zu bytes; use dflash_block_attention with a workspace\n",
            (long long)need, kNoAllocScratchBytes);
    return DFLASH_E_CAPACITY;
  }
  void* scratch = nullptr;
  if (need > 0) {
    const dflash_status s = scratch_on_current_device(&scratch);
    if (s != DFLASH_OK) return s;
  }
  return block_attention(batch, n_heads, n_kv_heads, 128, ctx_len, block, causal ? 1 : 0, q_dev,
                         k_dev, v_dev, out_dev, scratch, need, (cudaStream_t)stream);
}

}  // extern "C"
