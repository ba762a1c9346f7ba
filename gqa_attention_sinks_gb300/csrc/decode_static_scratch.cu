// attn_sink_decode_static_scratch: decode for callers that cannot allocate
// device memory.  The split-KV partial states go to a library-owned static
// device array instead of a caller-provided workspace; everything else is the
// regular attn_sink_decode path.
#include <mutex>

#include <cuda_runtime.h>

#include "attn_sink.h"

namespace {

// Scratch for split-KV partials (fp32 o and lse).  In host code this name is
// only a host-side stand-in: its device address comes from
// cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_SINK_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (set-up on the
// first call per device), or nullptr on a CUDA error.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" ATTN_SINK_API attn_sink_status attn_sink_decode_static_scratch(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_lens,
    const int32_t* block_table, int32_t block_table_stride, const float* sinks, void* out,
    float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
    int32_t num_pages, float scale, int32_t num_splits, attn_sink_dtype dtype, int32_t* err_flag,
    void* stream) {
  // fp32 with num_splits == 0 runs unsplit and needs no scratch.
  const int32_t splits = (dtype == ATTN_SINK_FP32 && num_splits == 0) ? 1 : num_splits;
  const size_t need =
      attn_sink_decode_workspace_size(B, Hq, Hkv, D, block_table_stride, page_size, splits);
  if (need > ATTN_SINK_STATIC_SCRATCH_BYTES) return ATTN_SINK_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = scratch_on_current_device();
    if (!scratch) return ATTN_SINK_ERR_CUDA;
  }
  return attn_sink_decode(q, k_cache, v_cache, kv_lens, block_table, block_table_stride, sinks,
                          out, lse, B, Hq, Hkv, D, page_size, num_pages, scale, splits, dtype,
                          err_flag, scratch, need > 0 ? ATTN_SINK_STATIC_SCRATCH_BYTES : 0,
                          stream);
}
