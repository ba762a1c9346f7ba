// attn_sink_decode_static_scratch: decode for callers that cannot allocate
// device memory.  The split-KV partial states go to a library-owned static
// device array instead of a caller-provided workspace; everything else is the
// regular attn_sink_decode path.
#include <cudaTypedefs.h>

#include <mutex>

#include <cuda_runtime.h>

#include "attn_sink.h"
#include "kernels.h"

namespace {

// Scratch for split-KV partials (fp32 o and lse).  In host code this name is
// only a host-side stand-in: its device address comes from
// cudaGetSymbolAddress, looked up with the device current.
static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_SINK_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of the array per device, valid for the context it was looked
// up in.  A process that resets the device (cudaDeviceReset) gets a new
// primary context, in which the array has a new address: the context's ID
// (unique for the life of the process) tells the two apart.
struct ScratchAddr {
  void* addr = nullptr;
  unsigned long long ctx_id = 0;
};
ScratchAddr g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

PFN_cuCtxGetCurrent_v4000 ctx_get_current = nullptr;
PFN_cuCtxGetId_v12000 ctx_get_id = nullptr;
std::once_flag g_driver_once;

bool current_ctx_id(unsigned long long* id) {
  std::call_once(g_driver_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!ctx_get_current || !ctx_get_id) return false;
  CUcontext ctx = nullptr;
  if (ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array on the current device and context
// (set-up on the first call there), or nullptr on a CUDA error.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchAddr& e = g_scratch[dev];
  unsigned long long id = 0;
  if (e.addr && current_ctx_id(&id) && id == e.ctx_id) return e.addr;
  // First call on this device, or a new context: look the address up (this
  // also initialises the context if the runtime has not done so yet).
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
  if (!current_ctx_id(&id)) return nullptr;
  e.addr = p;
  e.ctx_id = id;
  return p;
}

}  // namespace

extern "C" ATTN_SINK_API attn_sink_status attn_sink_decode_static_scratch(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_lens,
    const int32_t* block_table, int32_t block_table_stride, const float* sinks, void* out,
    float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
    int32_t num_pages, float scale, int32_t num_splits, attn_sink_dtype dtype, int32_t* err_flag,
    void* stream) {
  // The same argument checks, in the same order, as attn_sink_decode: a bad
  // call gets the same status from both.
  const attn_sink_status st =
      attn_sink::decode_validate(q, k_cache, v_cache, kv_lens, block_table, block_table_stride,
                                 sinks, out, B, Hq, Hkv, D, page_size, num_pages, scale,
                                 num_splits, dtype);
  if (st != ATTN_SINK_OK || B == 0) return st;
  // fp32 with num_splits <= 0 runs unsplit and needs no scratch.
  const int32_t splits = (dtype == ATTN_SINK_FP32 && num_splits <= 0) ? 1 : num_splits;
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
