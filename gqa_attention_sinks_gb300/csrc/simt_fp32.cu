// fp32 sink attention (prefill and split-KV decode) on CUDA cores.
//
// The fp32 path serves inputs that must not be rounded to bf16.  One warp owns
// one (query row, chunk) pair; lane l holds head-dim elements 2l and 2l+1.
// Keys are visited in order with the online softmax of "GPT-OSS pada Hari
// ke-0", section "Atensi Sink": the running maximum starts at the head's sink
// (first chunk only) with running sum 1, otherwise at -inf with sum 0.
// All arithmetic is fp32 with correctly rounded exp2f.
#include "kernels.h"
#include "ptx.cuh"

namespace attn_sink {
namespace {

constexpr int kWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ int seq_of_token(const int32_t* cu, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kWarps * 32) simt_fp32_kernel(const SimtArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarps + warp;
  const int chunk = blockIdx.y;
  if (row >= static_cast<long long>(a.total_q) * a.Hq) return;
  const int t = static_cast<int>(row / a.Hq), h = static_cast<int>(row % a.Hq);
  const int b = a.cu_seqlens_q ? seq_of_token(a.cu_seqlens_q, a.B, t) : t;
  const int q_start = a.cu_seqlens_q ? a.cu_seqlens_q[b] : t;
  const int q_len = a.cu_seqlens_q ? a.cu_seqlens_q[b + 1] - q_start : 1;
  const int kv_raw = max(0, a.kv_lens[b]);
  const int kv_len = min(kv_raw, a.bt_stride * a.page_size);  // keys beyond the table row are not read
  const long long pos = static_cast<long long>(kv_len) - q_len + (t - q_start);
  const int g = h / a.group;

  // key range of this chunk (page-aligned split, sink in chunk 0 only)
  long long k0 = 0, k1 = kv_len;
  if (a.num_splits > 1) {
    const long long P = (kv_len + a.page_size - 1) / a.page_size;
    k0 = (chunk * P) / a.num_splits * a.page_size;
    k1 = min(static_cast<long long>(kv_len), ((chunk + 1) * P) / a.num_splits * a.page_size);
  }
  if (a.causal && k1 > pos + 1) k1 = pos + 1;

  const float2 qv = *reinterpret_cast<const float2*>(a.q + row * kHeadDim + 2 * lane);
  const int32_t* bt_row = a.block_table + static_cast<long long>(b) * a.bt_stride;
  float m = chunk == 0 ? a.sinks[h] * kLog2e : -INFINITY;
  float d = chunk == 0 ? 1.f : 0.f;
  float2 o = make_float2(0.f, 0.f);
  bool bad = kv_len < kv_raw;
  for (long long j = k0; j < k1; ++j) {
    const int phys = bt_row[j / a.page_size];
    if (phys < 0 || phys >= a.num_pages) {
      bad = true;
      continue;
    }
    const long long off =
        ((static_cast<long long>(phys) * a.page_size + j % a.page_size) * a.Hkv + g) * kHeadDim + 2 * lane;
    const float2 kv = *reinterpret_cast<const float2*>(a.k_cache + off);
    float dot = qv.x * kv.x + qv.y * kv.y;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, s);
    const float x = dot * a.scale_log2;
    if (x > m) {
      const float alpha = m == -INFINITY ? 0.f : exp2f(m - x);
      d *= alpha;
      o.x *= alpha;
      o.y *= alpha;
      m = x;
    }
    const float p = exp2f(x - m);
    const float2 vv = *reinterpret_cast<const float2*>(a.v_cache + off);
    d += p;
    o.x = fmaf(p, vv.x, o.x);
    o.y = fmaf(p, vv.y, o.y);
  }
  if (bad && lane == 0 && a.err_flag) atomicOr(a.err_flag, kFlagBadPage);

  const bool empty = d <= 0.f || m == -INFINITY;
  const float inv = empty ? 0.f : 1.f / d;
  const float lse = empty ? -INFINITY : (m + log2f(d)) * kLn2;
  o.x *= inv;
  o.y *= inv;
  if (a.num_splits > 1) {
    *reinterpret_cast<float2*>(a.o_part + (row * a.num_splits + chunk) * kHeadDim + 2 * lane) = o;
    if (lane == 0) a.lse_part[row * a.num_splits + chunk] = lse;
  } else {
    *reinterpret_cast<float2*>(a.out + row * kHeadDim + 2 * lane) = o;
    if (a.lse && lane == 0) a.lse[row] = lse;
  }
}

}  // namespace

cudaError_t launch_simt_fp32(const SimtArgs& a, cudaStream_t stream) {
  const long long rows = static_cast<long long>(a.total_q) * a.Hq;
  if (rows == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>((rows + kWarps - 1) / kWarps), a.num_splits > 1 ? a.num_splits : 1);
  simt_fp32_kernel<<<grid, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace attn_sink
