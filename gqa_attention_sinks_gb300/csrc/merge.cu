// Log-sum-exp merge of split-KV partial states.
//
// Each partial c of a row holds o_c (normalised by its own softmax sum) and
// lse_c = ln(sum of its exponentials, the sink included when that chunk
// counted it).  The combined row is
//     L = ln sum_c e^{lse_c},   out = sum_c e^{lse_c - L} o_c.
// No sink is added here: "GPT-OSS pada Hari ke-0", section "Atensi Sink",
// puts the sink in the first chunk only, so it already sits inside partial 0.
//
// One warp per row, two head-dim elements per lane (D = 64); partials are
// read as coalesced 256-byte lines.
#include "kernels.h"
#include "ptx.cuh"

namespace attn_sink {
namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__global__ void __launch_bounds__(kWarps * 32) merge_kernel(const MergeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kWarps + warp;
  if (row >= a.rows) return;

  int n = a.num_parts;
  if (a.kv_lens) {
    const int kv = max(0, a.kv_lens[row / a.Hq]);
    const int units = (kv + kUnitTokens - 1) / kUnitTokens;
    n = max(1, (units + a.chunk_units - 1) / a.chunk_units);
    if (n == 1) return;  // the decode kernel wrote this row directly
    n = min(n, a.s_stride);
  }
  const float* lse_row = a.lse_part + static_cast<long long>(row) * a.s_stride;
  const float* o_row = a.o_part + static_cast<long long>(row) * a.s_stride * kHeadDim;

  float m = -INFINITY;
  for (int c = lane; c < n; c += 32) m = fmaxf(m, lse_row[c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));

  float2 acc = make_float2(0.f, 0.f);
  float den = 0.f;
  if (m != -INFINITY) {
    const float m2 = m * kLog2e;
    for (int c = 0; c < n; ++c) {
      const float l = lse_row[c];
      const float w = l == -INFINITY ? 0.f : exp2f(fmaf(l, kLog2e, -m2));
      const float2 o = *reinterpret_cast<const float2*>(o_row + c * kHeadDim + 2 * lane);
      den += w;
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  acc.x *= inv;
  acc.y *= inv;
  const long long base = static_cast<long long>(row) * kHeadDim + 2 * lane;
  if (a.out_fp32) {
    *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + base) = acc;
  } else {
    *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.out) + base) =
        pack_bf16x2(acc.x, acc.y);
  }
  if (a.lse && lane == 0) a.lse[row] = den > 0.f ? m + log2f(den) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  if (a.rows <= 0) return cudaSuccess;
  const int blocks = (a.rows + kWarps - 1) / kWarps;
  merge_kernel<<<blocks, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace attn_sink
