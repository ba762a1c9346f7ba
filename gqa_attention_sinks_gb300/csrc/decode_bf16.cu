// Split-KV paged decode for bf16 sink attention on sm_103a.
//
// One CTA owns (chunk c, a group of kHeadsPerCta KV heads, sequence b) and all
// G query heads of each of those KV heads, so every K/V byte of the chunk is
// read from HBM exactly once.
// "GPT-OSS pada Hari ke-0", section "Atensi Sink": attention is parallelised
// over heads and along the KV length; the online softmax starts its running
// maximum at the head's sink value with running sum 1, and only the first
// chunk of a split may do so.
//
// Warp roles (160 threads):
//   warp 4      producer: reads the block table (32 units ahead) and per
//               16-key unit issues one TMA box for K and one for V that cover
//               the unit's 16 rows of all kHeadsPerCta heads (8 KB each; a 4-D
//               tensor map over (dim, token in page, head, page)), into a
//               4-stage shared-memory ring guarded by mbarriers.  A 2 KB box
//               per head and unit occupies the SM's TMA unit about as long as
//               an 8 KB one, so this keeps TMA far from the HBM rate.
//   warps 0..3  consumers: warp w owns KV head g0 + w.  Scores for the G packed
//               query heads (M = 16 rows) come from mma.sync m16n8k16 bf16
//               with fp32 accumulation, the online softmax runs in registers,
//               and P*V reuses the score fragments as the A operand.
// In append mode the producer of the CTA whose chunk holds a sequence's last
// position first writes the step's key and value rows of its heads there
// ("Accelerating Sonar through speculation", section "Inferensi dengan
// Speculative Decoding": pages for each sequence's next token are allocated
// before the step).
// Each warp writes either its head's final output (the sequence has one
// chunk) or an fp32 partial (o, lse) that the merge kernel combines.
//
// The kernel is HBM-bound: per key and KV head it moves 256 B and does
// 2*G*64 MACs, which the tensor-core path hides completely.
#include "kernels.h"
#include "ptx.cuh"

namespace attn_sink {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kStages = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kUnitBytes = kUnitTokens * kHeadDim * 2;              // 2048: one head, one unit
constexpr int kHalfBytes = kHeadsPerCta * kUnitBytes;               // 8 KB: one box
constexpr int kStageBytes = 2 * kHalfBytes;                          // 16 KB (K then V)
constexpr int kRingBytes = kStages * kStageBytes;                    // 64 KB
constexpr int kSmemBytes = kRingBytes + 1024 /*align slack*/ + 128 /*barriers*/;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct alignas(8) Barriers {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint32_t unit_ok[kStages];  // the stage's unit was loaded (its page index is valid)
  int abort_word;
};
static_assert(kConsumerWarps == kHeadsPerCta, "one consumer warp per KV head of the CTA");

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

// kPoll: the waits poll (a test's short wait limit); otherwise they block.
template <bool kTwoRows, bool kPoll>
__global__ void __launch_bounds__(kThreads)
    decode_split_kernel(const __grid_constant__ CUtensorMap k_map,
                        const __grid_constant__ CUtensorMap v_map, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Barriers* bars = reinterpret_cast<Barriers*>(ring + kRingBytes);

  const int c = blockIdx.x, g0 = blockIdx.y * kHeadsPerCta, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- chunk bounds in 16-key units (keys beyond the table row are not read)
  const int kv_raw = a.kv_lens[b] > 0 ? a.kv_lens[b] : 0;
  const int kv_len = min(kv_raw, a.bt_stride * a.page_size);
  if (kv_len < kv_raw && threadIdx.x == 0 && c == 0 && g0 == 0 && a.err_flag)
    atomicOr(a.err_flag, kFlagBadPage);
  const int n_units_seq = (kv_len + kUnitTokens - 1) / kUnitTokens;
  int u0, u1, n_chunks;
  if (a.num_splits > 0) {
    const int units_per_page = a.page_size / kUnitTokens;
    const long long P = (kv_len + a.page_size - 1) / a.page_size;
    const long long pb = (c * P) / a.num_splits, pe = ((c + 1) * P) / a.num_splits;
    u0 = static_cast<int>(pb * units_per_page);
    u1 = min(static_cast<int>(pe * units_per_page), n_units_seq);
    n_chunks = a.num_splits;
  } else {
    n_chunks = max(1, (n_units_seq + a.chunk_units - 1) / a.chunk_units);
    if (c >= n_chunks) return;
    u0 = c * a.chunk_units;
    u1 = min(u0 + a.chunk_units, n_units_seq);
  }
  if (u1 < u0) u1 = u0;
  const int n_iters = u1 - u0;  // one unit per stage

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], kConsumerWarps);
    }
    bars->abort_word = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&k_map);
      tma_prefetch_map(&v_map);
    }
    const uint64_t policy = l2_policy_evict_first();
    const int32_t* bt_row = a.block_table + static_cast<long long>(b) * a.bt_stride;
    const int units_per_page = a.page_size / kUnitTokens;
    // Lane l holds the page and in-page row of unit u0 + 32k + l for the
    // current window of 32 units; the next window is read while this one is
    // used.
    auto fetch = [&](int base, int& phys, int& tok) {
      const int u = u0 + base + lane;
      phys = -1;
      tok = 0;
      if (u < u1) {
        phys = bt_row[u / units_per_page];
        tok = (u % units_per_page) * kUnitTokens;
      }
    };
    if (a.k_new && kv_len >= 1) {
      // Append mode: the CTA whose chunk holds the last position writes the
      // step's key and value rows of its heads there before any copy of that
      // unit is issued; the proxy fences order the generic writes before the
      // TMA reads.
      const int unit_last = (kv_len - 1) / kUnitTokens;
      if (unit_last >= u0 && unit_last < u1) {
        const int pos = kv_len - 1;
        const int phys = bt_row[pos / a.page_size];
        if (phys >= 0 && phys < a.num_pages) {
          const long long row = static_cast<long long>(phys) * a.page_size + pos % a.page_size;
          constexpr int kPieces = kHeadDim * 2 / 16;  // 16-byte pieces of one head's row
          for (int i = lane; i < 2 * kHeadsPerCta * kPieces; i += 32) {
            const int t = i / (kHeadsPerCta * kPieces), h = (i / kPieces) % kHeadsPerCta,
                      piece = i % kPieces;
            const int g = g0 + h;
            if (g < a.Hkv) {
              const uint4* src = reinterpret_cast<const uint4*>(t ? a.v_new : a.k_new) +
                                 (static_cast<long long>(b) * a.Hkv + g) * kPieces + piece;
              uint4* dst = reinterpret_cast<uint4*>(t ? a.v_cache_w : a.k_cache_w) +
                           (row * a.Hkv + g) * kPieces + piece;
              *dst = *src;
            }
          }
          fence_proxy_async_global();
        }
      }
      __syncwarp();
      fence_proxy_async_global();
    }
    int cur_phys, cur_tok, nxt_phys, nxt_tok;
    fetch(0, cur_phys, cur_tok);
    fetch(32, nxt_phys, nxt_tok);
    int issued = 0;
    for (int it = 0; it < n_iters; ++it) {
      if (it > 0 && (it & 31) == 0) {
        cur_phys = nxt_phys;
        cur_tok = nxt_tok;
        fetch(it + 32, nxt_phys, nxt_tok);
      }
      const int stage = it % kStages;
      if (it >= kStages) {
        const bool ready = mbar_wait<kPoll>(&bars->empty[stage], ((it / kStages) + 1) & 1,
                                     &bars->abort_word, a.err_flag, a.wait_limit_ns);
        if (!__all_sync(0xffffffffu, ready)) break;
      }
      const int phys = __shfl_sync(0xffffffffu, cur_phys, it & 31);
      const int tok = __shfl_sync(0xffffffffu, cur_tok, it & 31);
      const bool ok = phys >= 0 && phys < a.num_pages;
      if (lane == 0) {
        if (!ok && a.err_flag) atomicOr(a.err_flag, kFlagBadPage);
        bars->unit_ok[stage] = ok ? 1u : 0u;
        mbar_arrive_expect_tx(&bars->full[stage], ok ? kStageBytes : 0);
        if (ok) {
          uint8_t* st = ring + stage * kStageBytes;
          tma_load_4d_hint(st, &k_map, &bars->full[stage], 0, tok, g0, phys, policy);
          tma_load_4d_hint(st + kHalfBytes, &v_map, &bars->full[stage], 0, tok, g0, phys, policy);
        }
      }
      __syncwarp();
      issued = it + 1;
    }
    // Drain: every issued load lands before the CTA's shared memory goes away.
    if (lane == 0) {
      for (int it = max(0, issued - kStages); it < issued; ++it)
        mbar_wait_drain(&bars->full[it % kStages], (it / kStages) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = g0 + warp;            // this warp's KV head
  const bool head_ok = g < a.Hkv;
  const int r0 = lane >> 2, r1 = r0 + 8;
  const int head0 = g * a.group;
  uint32_t qa[4][4];
  {
    const __nv_bfloat16* qb =
        reinterpret_cast<const __nv_bfloat16*>(a.q) + (static_cast<long long>(b) * a.Hq + head0) * kHeadDim;
    const int col = 2 * (lane & 3);
    const bool ok0 = head_ok && r0 < a.group, ok1 = head_ok && r1 < a.group;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const int d = 16 * ks + col;
      qa[ks][0] = ok0 ? *reinterpret_cast<const uint32_t*>(qb + r0 * kHeadDim + d) : 0u;
      qa[ks][1] = ok1 ? *reinterpret_cast<const uint32_t*>(qb + r1 * kHeadDim + d) : 0u;
      qa[ks][2] = ok0 ? *reinterpret_cast<const uint32_t*>(qb + r0 * kHeadDim + d + 8) : 0u;
      qa[ks][3] = ok1 ? *reinterpret_cast<const uint32_t*>(qb + r1 * kHeadDim + d + 8) : 0u;
    }
  }

  WarpState st;
  st.m0 = st.m1 = -INFINITY;
  st.d0 = st.d1 = st.w0 = st.w1 = 0.f;
#pragma unroll
  for (int dn = 0; dn < 8; ++dn)
#pragma unroll
    for (int e = 0; e < 4; ++e) st.o[dn][e] = 0.f;
  if (c == 0 && head_ok) {
    // The sink enters as the initial running max with running sum 1, in the
    // first chunk only (one quad lane carries the 1).
    st.m0 = r0 < a.group ? a.sinks[head0 + r0] * kLog2e : -INFINITY;
    st.m1 = r1 < a.group ? a.sinks[head0 + r1] * kLog2e : -INFINITY;
    st.d0 = st.w0 = (lane & 3) == 0 ? 1.f : 0.f;
    st.d1 = st.w1 = (lane & 3) == 0 ? 1.f : 0.f;
  }

  for (int it = 0; it < n_iters; ++it) {
    const int stage = it % kStages;
    const bool ready =
        mbar_wait<kPoll>(&bars->full[stage], (it / kStages) & 1, &bars->abort_word, a.err_flag, a.wait_limit_ns);
    if (!__all_sync(0xffffffffu, ready)) break;
    if (head_ok && bars->unit_ok[stage]) {
      const int u = u0 + it;
      const uint32_t k_base = smem_addr(ring + stage * kStageBytes + warp * kUnitBytes);
      const uint32_t v_base = k_base + kHalfBytes;
      const int n_valid = min(kUnitTokens, kv_len - u * kUnitTokens);
      consume_unit<kTwoRows>(k_base, v_base, n_valid, qa, a.scale_log2, st);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->empty[stage]);
  }
  if (!head_ok) return;

  // ---- this warp holds its head's whole state: reduce the quad's sums, write
  st.d0 += __shfl_xor_sync(0xffffffffu, st.d0, 1);
  st.d0 += __shfl_xor_sync(0xffffffffu, st.d0, 2);
  st.d1 += __shfl_xor_sync(0xffffffffu, st.d1, 1);
  st.d1 += __shfl_xor_sync(0xffffffffu, st.d1, 2);
  st.w0 += __shfl_xor_sync(0xffffffffu, st.w0, 1);
  st.w0 += __shfl_xor_sync(0xffffffffu, st.w0, 2);
  st.w1 += __shfl_xor_sync(0xffffffffu, st.w1, 1);
  st.w1 += __shfl_xor_sync(0xffffffffu, st.w1, 2);
  const bool direct = n_chunks == 1;
  const int col = 2 * (lane & 3);
#pragma unroll
  for (int half = 0; half < (kTwoRows ? 2 : 1); ++half) {
    const int row = half ? r1 : r0;
    if (row >= a.group) continue;
    const float m = half ? st.m1 : st.m0;
    const float den = half ? st.d1 : st.d0;
    const float wden = half ? st.w1 : st.w0;
    const float inv = wden > 0.f ? 1.f / wden : 0.f;
    const float lse = (den > 0.f && m != -INFINITY) ? (m + __log2f(den)) * kLn2 : -INFINITY;
    const long long grow = static_cast<long long>(b) * a.Hq + head0 + row;
    if (direct) {
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.out) + grow * kHeadDim;
#pragma unroll
      for (int dn = 0; dn < 8; ++dn)
        *reinterpret_cast<uint32_t*>(orow + dn * 8 + col) =
            pack_bf16x2(st.o[dn][2 * half] * inv, st.o[dn][2 * half + 1] * inv);
      if (a.lse && (lane & 3) == 0) a.lse[grow] = lse;
    } else {
      float* prow = a.o_part + (grow * a.s_stride + c) * kHeadDim;
#pragma unroll
      for (int dn = 0; dn < 8; ++dn)
        *reinterpret_cast<float2*>(prow + dn * 8 + col) =
            make_float2(st.o[dn][2 * half] * inv, st.o[dn][2 * half + 1] * inv);
      if ((lane & 3) == 0) a.lse_part[grow * a.s_stride + c] = lse;
    }
  }
}

}  // namespace

cudaError_t launch_decode_bf16(const DecodeArgs& a, const CUtensorMap& k_map,
                               const CUtensorMap& v_map, cudaStream_t stream) {
  dim3 grid(a.max_chunks, (a.Hkv + kHeadsPerCta - 1) / kHeadsPerCta, a.B);
  const bool poll = a.wait_limit_ns < kPollLimitNs;
  auto kern = a.group > 8 ? (poll ? decode_split_kernel<true, true> : decode_split_kernel<true, false>)
                          : (poll ? decode_split_kernel<false, true> : decode_split_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kSmemBytes, stream>>>(k_map, v_map, a);
  return cudaGetLastError();
}

}  // namespace attn_sink
