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
// read as coalesced 256-byte lines, kStep of them in flight at a time.
#include "kernels.h"
#include "ptx.cuh"

namespace attn_sink {
namespace {

constexpr int kWarps = 8;
constexpr int kStep = 8;  // partials whose loads are in flight together
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__global__ void __launch_bounds__(kWarps * 32) merge_kernel(const MergeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kWarps + warp;
  // Launched as a programmatic dependent of the kernel that wrote the
  // partials: wait here until that grid has completed and its writes are
  // visible (returns at once when there is no such grid).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (row >= a.rows) return;

  int n = a.num_parts;
  if (a.stream_start) {
    // Stream-K decode: the row's stream spans the shares c_first..c_last.
    const int b = row / a.Hq, h = row % a.Hq;
    const int s = b * a.n_groups + (h / a.group) / kHeadsPerCta;
    const long long U = a.stream_start[(a.rows / a.Hq) * a.n_groups];
    const long long G = *a.shares;
    const long long x0 = a.stream_start[s], x1 = a.stream_start[s + 1];
    if (x1 == x0) {  // no keys: only the sink (out = 0, lse = sink)
      const long long base = static_cast<long long>(row) * kHeadDim + 2 * lane;
      if (a.out_fp32)
        *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + base) = make_float2(0.f, 0.f);
      else
        *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.out) + base) = 0u;
      if (a.lse && lane == 0) a.lse[row] = a.sinks[h];
      return;
    }
    const long long c_first = ((x0 + 1) * G - 1) / U, c_last = (x1 * G - 1) / U;
    if (c_first == c_last) return;  // written directly by the decode kernel
    n = static_cast<int>(min(c_last - c_first + 1, static_cast<long long>(a.s_stride)));
  } else if (a.kv_lens) {
    int kv = max(0, a.kv_lens[row / a.Hq]);
    if (a.kv_cap > 0) kv = min(kv, a.kv_cap);
    const int units = (kv + kUnitTokens - 1) / kUnitTokens;
    n = max(1, (units + a.chunk_units - 1) / a.chunk_units);
    if (n == 1) return;  // the decode kernel wrote this row directly
    n = min(n, a.s_stride);
    // a ragged batch's decode sequence without a query row has no output row
    if (a.seq_start && a.seq_start[row / a.Hq + 1] <= a.seq_start[row / a.Hq]) return;
  }
  const float* lse_row = a.lse_part + static_cast<long long>(row) * a.s_stride;
  const float* o_row = a.o_part + static_cast<long long>(row) * a.s_stride * kHeadDim;

  // Single pass with a running maximum m (log2 domain).  Each step issues the
  // loads of kStep partials before combining any of them; waiting for each
  // partial before loading the next would cost one memory latency per chunk.
  float m = -INFINITY, den = 0.f;
  float2 acc = make_float2(0.f, 0.f);
  for (int cb = 0; cb < n; cb += kStep) {
    float l[kStep];
    float2 o[kStep];
#pragma unroll
    for (int k = 0; k < kStep; ++k) {
      const bool valid = cb + k < n;
      l[k] = valid ? lse_row[cb + k] : -INFINITY;
      o[k] = valid ? *reinterpret_cast<const float2*>(o_row + (cb + k) * kHeadDim + 2 * lane)
                   : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kStep; ++k) {
      if (l[k] == -INFINITY) continue;
      const float lk = l[k] * kLog2e;
      const float m_new = fmaxf(m, lk);
      const float keep = exp2f(m - m_new);  // 0 while m is -inf
      const float w = exp2f(lk - m_new);
      den = fmaf(den, keep, w);
      acc.x = fmaf(acc.x, keep, w * o[k].x);
      acc.y = fmaf(acc.y, keep, w * o[k].y);
      m = m_new;
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  acc.x *= inv;
  acc.y *= inv;
  const long long orow = a.seq_start ? static_cast<long long>(a.seq_start[row / a.Hq]) * a.Hq + row % a.Hq
                                     : static_cast<long long>(row);
  const long long base = orow * kHeadDim + 2 * lane;
  if (a.out_fp32) {
    *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + base) = acc;
  } else {
    *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.out) + base) =
        pack_bf16x2(acc.x, acc.y);
  }
  if (a.lse && lane == 0) a.lse[orow] = den > 0.f ? (m + log2f(den)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  if (a.rows <= 0) return cudaSuccess;
  const int blocks = (a.rows + kWarps - 1) / kWarps;
  // Programmatic stream serialisation: the merge grid's launch overlaps the end
  // of the previous kernel; griddepcontrol.wait above orders every partial
  // read after that kernel has completed.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel, a);
}

}  // namespace attn_sink
