// Warp-level split-KV decode step shared by the decode kernel and the mixed
// (prefill + decode) kernel: one warp, one KV head, up to 16 packed query heads
// (mma.sync m16n8k16 bf16, fp32 accumulation), one 16-key unit of K and V in
// shared memory as 16 rows of 128 bytes with the 128-byte swizzle TMA writes.
//
// "GPT-OSS pada Hari ke-0", section "Atensi Sink": the online softmax runs
// with the sink as the initial running maximum (first chunk only); this step
// is the per-key-block update of that softmax.
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace attn_sink {
namespace dec {

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a 128B-swizzled tile
// whose base is 1024-byte aligned (the layout TMA writes with SWIZZLE_128B).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Keep the bf16 halves of a B fragment whose key index is below n_valid.
__device__ __forceinline__ uint32_t mask_keys(uint32_t v, int key_lo, int n_valid) {
  uint32_t keep = (key_lo < n_valid ? 0x0000FFFFu : 0u) | (key_lo + 1 < n_valid ? 0xFFFF0000u : 0u);
  return v & keep;
}

// Online-softmax state of one consumer warp for rows r0 = lane/4 and r1 = r0+8.
struct WarpState {
  float m0, m1;   // running max, log2 domain (quad-uniform)
  float d0, d1;   // this thread's share of the running sum of exact p (for lse)
  float w0, w1;   // the same over the bf16-rounded p fed to P*V (normalises O)
  float o[8][4];  // O fragments: [d tile][c0..c3]
};

// One 16-key unit: S = Q K^T, online softmax update, O += P V.
template <bool kTwoRows>
__device__ __forceinline__ void consume_unit(uint32_t k_base, uint32_t v_base, int n_valid,
                                             const uint32_t (&qa)[4][4], float scale_log2,
                                             WarpState& st) {
  const int lane = threadIdx.x & 31;
  float s[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;

  {
    const int mi = lane >> 3, ri = lane & 7;
    const int key = (mi >> 1) * 8 + ri;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t b00, b01, b10, b11;
      ldsm_x4(b00, b01, b10, b11, k_base + swz(key, 2 * ks + (mi & 1)));
      mma_16816(s[0], qa[ks], b00, b01);
      mma_16816(s[1], qa[ks], b10, b11);
    }
  }

  const int kc = 2 * (lane & 3);
  float x[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = nt * 8 + kc + (e & 1);
      const bool row_ok = kTwoRows || e < 2;
      x[nt][e] = (key < n_valid && row_ok) ? s[nt][e] * scale_log2 : -INFINITY;
    }

  float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  const float mn0 = fmaxf(st.m0, mx0);
  const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
  const float al0 = fast_exp2(st.m0 - mu0);
  st.m0 = mn0;

  float mn1 = -INFINITY, mu1 = 0.f, al1 = 1.f;
  if (kTwoRows) {
    float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    mn1 = fmaxf(st.m1, mx1);
    mu1 = mn1 == -INFINITY ? 0.f : mn1;
    al1 = fast_exp2(st.m1 - mu1);
    st.m1 = mn1;
  }

  float p[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    p[nt][0] = fast_exp2(x[nt][0] - mu0);
    p[nt][1] = fast_exp2(x[nt][1] - mu0);
    p[nt][2] = kTwoRows ? fast_exp2(x[nt][2] - mu1) : 0.f;
    p[nt][3] = kTwoRows ? fast_exp2(x[nt][3] - mu1) : 0.f;
  }
  // P is rounded to bf16 for the P*V MMA.  w sums the same rounded values (so a
  // row's weights sum to exactly 1); d sums the exact ones (for the lse).
  uint32_t pa[4];
  pa[0] = pack_bf16x2(p[0][0], p[0][1]);
  pa[1] = kTwoRows ? pack_bf16x2(p[0][2], p[0][3]) : 0u;
  pa[2] = pack_bf16x2(p[1][0], p[1][1]);
  pa[3] = kTwoRows ? pack_bf16x2(p[1][2], p[1][3]) : 0u;
  st.d0 = st.d0 * al0 + (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
  st.w0 = st.w0 * al0 + (bf16_lo(pa[0]) + bf16_hi(pa[0])) + (bf16_lo(pa[2]) + bf16_hi(pa[2]));
  if (kTwoRows) {
    st.d1 = st.d1 * al1 + (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
    st.w1 = st.w1 * al1 + (bf16_lo(pa[1]) + bf16_hi(pa[1])) + (bf16_lo(pa[3]) + bf16_hi(pa[3]));
  }
#pragma unroll
  for (int dn = 0; dn < 8; ++dn) {
    st.o[dn][0] *= al0;
    st.o[dn][1] *= al0;
    if (kTwoRows) {
      st.o[dn][2] *= al1;
      st.o[dn][3] *= al1;
    }
  }

  const int mi = lane >> 3, ri = lane & 7;
  const int vkey = (mi & 1) * 8 + ri;
#pragma unroll
  for (int dp = 0; dp < 4; ++dp) {
    uint32_t v0, v1, v2, v3;
    ldsm_x4_trans(v0, v1, v2, v3, v_base + swz(vkey, 2 * dp + (mi >> 1)));
    if (n_valid < kUnitTokens) {  // unused slots of a last page may hold anything
      v0 = mask_keys(v0, kc, n_valid);
      v1 = mask_keys(v1, 8 + kc, n_valid);
      v2 = mask_keys(v2, kc, n_valid);
      v3 = mask_keys(v3, 8 + kc, n_valid);
    }
    mma_16816(st.o[2 * dp], pa, v0, v1);
    mma_16816(st.o[2 * dp + 1], pa, v2, v3);
  }
}


// A fragments of the warp's packed query heads: rows r0 = lane/4 and r1 = r0 + 8
// of the G heads of one KV head, from q_head0 (bf16 [G, 64], head 0 of the
// group); rows past G (or the whole group when !head_ok) are zero.
__device__ __forceinline__ void load_q_frags(uint32_t (&qa)[4][4], const __nv_bfloat16* q_head0,
                                             int group, bool head_ok) {
  const int lane = threadIdx.x & 31;
  const int r0 = lane >> 2, r1 = r0 + 8;
  const int col = 2 * (lane & 3);
  const bool ok0 = head_ok && r0 < group, ok1 = head_ok && r1 < group;
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    const int d = 16 * ks + col;
    qa[ks][0] = ok0 ? *reinterpret_cast<const uint32_t*>(q_head0 + r0 * kHeadDim + d) : 0u;
    qa[ks][1] = ok1 ? *reinterpret_cast<const uint32_t*>(q_head0 + r1 * kHeadDim + d) : 0u;
    qa[ks][2] = ok0 ? *reinterpret_cast<const uint32_t*>(q_head0 + r0 * kHeadDim + d + 8) : 0u;
    qa[ks][3] = ok1 ? *reinterpret_cast<const uint32_t*>(q_head0 + r1 * kHeadDim + d + 8) : 0u;
  }
}

// Initial online-softmax state.  In the first chunk of a split the sink is the
// initial running max with running sum 1 (one quad lane carries the 1); the
// other chunks start empty.
__device__ __forceinline__ void init_state(WarpState& st, const float* sinks_head0, int group,
                                           bool first_chunk) {
  const int lane = threadIdx.x & 31;
  const int r0 = lane >> 2, r1 = r0 + 8;
  constexpr float kLog2e = 1.4426950408889634f;
  st.m0 = st.m1 = -INFINITY;
  st.d0 = st.d1 = st.w0 = st.w1 = 0.f;
#pragma unroll
  for (int dn = 0; dn < 8; ++dn)
#pragma unroll
    for (int e = 0; e < 4; ++e) st.o[dn][e] = 0.f;
  if (first_chunk) {
    st.m0 = r0 < group ? sinks_head0[r0] * kLog2e : -INFINITY;
    st.m1 = r1 < group ? sinks_head0[r1] * kLog2e : -INFINITY;
    st.d0 = st.w0 = (lane & 3) == 0 ? 1.f : 0.f;
    st.d1 = st.w1 = (lane & 3) == 0 ? 1.f : 0.f;
  }
}

// Reduces the quad-split sums, so that every lane of a quad holds its rows'
// totals.
__device__ __forceinline__ void reduce_sums(WarpState& st) {
#pragma unroll
  for (int x = 1; x <= 2; x <<= 1) {
    st.d0 += __shfl_xor_sync(0xffffffffu, st.d0, x);
    st.d1 += __shfl_xor_sync(0xffffffffu, st.d1, x);
    st.w0 += __shfl_xor_sync(0xffffffffu, st.w0, x);
    st.w1 += __shfl_xor_sync(0xffffffffu, st.w1, x);
  }
}

// Row `half` (0: r0, 1: r1) of the reduced state: the normalised output (O
// over the sum of the rounded p the P*V used) and the natural-log LSE.
// Writes either the final bf16 row (out_row) or an fp32 partial (part_row and
// *part_lse); the lse goes to *lse_out when it is not null.
__device__ __forceinline__ void write_row(const WarpState& st, int half, __nv_bfloat16* out_row,
                                          float* lse_out, float* part_row, float* part_lse) {
  const int lane = threadIdx.x & 31;
  const int col = 2 * (lane & 3);
  constexpr float kLn2 = 0.6931471805599453f;
  const float m = half ? st.m1 : st.m0;
  const float den = half ? st.d1 : st.d0;
  const float wden = half ? st.w1 : st.w0;
  const float inv = wden > 0.f ? 1.f / wden : 0.f;
  const float lse = (den > 0.f && m != -INFINITY) ? (m + __log2f(den)) * kLn2 : -INFINITY;
  if (out_row) {
#pragma unroll
    for (int dn = 0; dn < 8; ++dn)
      *reinterpret_cast<uint32_t*>(out_row + dn * 8 + col) =
          pack_bf16x2(st.o[dn][2 * half] * inv, st.o[dn][2 * half + 1] * inv);
    if (lse_out && (lane & 3) == 0) *lse_out = lse;
  } else {
#pragma unroll
    for (int dn = 0; dn < 8; ++dn)
      *reinterpret_cast<float2*>(part_row + dn * 8 + col) =
          make_float2(st.o[dn][2 * half] * inv, st.o[dn][2 * half + 1] * inv);
    if ((lane & 3) == 0) *part_lse = lse;
  }
}

}  // namespace dec
}  // namespace attn_sink
