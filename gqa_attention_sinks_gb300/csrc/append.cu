// KV append for a decode step: the step's key and value of every KV head go
// into the cache slot of the sequence's last position.
//
// "Accelerating Sonar through speculation", section "Inferensi dengan
// Speculative Decoding": before a step runs, pages in the KV cache are
// allocated for each sequence's next token; this writes that token's K/V.
// The bf16 decode fuses the same write into its split kernel; this kernel
// serves the fp32 path.
#include "kernels.h"
#include "ptx.cuh"

namespace attn_sink {
namespace {

// One CTA per sequence; 16-byte copies of the Hkv rows of K and of V.
__global__ void append_kernel(const AppendArgs a) {
  const int b = blockIdx.x;
  const int kv = a.kv_lens[b];
  if (kv < 1) return;
  if (kv > a.bt_stride * a.page_size) {  // the slot lies beyond the table row
    if (threadIdx.x == 0 && a.err_flag) atomicOr(a.err_flag, kFlagBadPage);
    return;
  }
  const int pos = kv - 1;
  const int phys = a.block_table[static_cast<long long>(b) * a.bt_stride + pos / a.page_size];
  if (phys < 0 || phys >= a.num_pages) {
    if (threadIdx.x == 0 && a.err_flag) atomicOr(a.err_flag, kFlagBadPage);
    return;
  }
  const long long row = static_cast<long long>(phys) * a.page_size + pos % a.page_size;
  const int row_chunks = kHeadDim * a.elem_bytes / 16;  // 16-byte pieces of one head's row
  const int per_tensor = a.Hkv * row_chunks;
  for (int i = threadIdx.x; i < 2 * per_tensor; i += blockDim.x) {
    const int t = i / per_tensor, j = i % per_tensor;  // j = head * row_chunks + piece
    const uint4* src = reinterpret_cast<const uint4*>(t ? a.v_new : a.k_new) +
                       static_cast<long long>(b) * per_tensor + j;
    uint4* dst = reinterpret_cast<uint4*>(t ? a.v_cache : a.k_cache) + row * per_tensor + j;
    *dst = *src;
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
  if (a.B <= 0) return cudaSuccess;
  append_kernel<<<a.B, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace attn_sink
