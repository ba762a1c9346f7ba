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
#include "decode_unit.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace attn_sink {
namespace {

using namespace dec;

constexpr int kConsumerWarps = 4;
constexpr int kStages = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kUnitBytes = kUnitTokens * kHeadDim * 2;              // 2048: one head, one unit
constexpr int kHalfBytes = kHeadsPerCta * kUnitBytes;               // 8 KB: one box
constexpr int kStageBytes = 2 * kHalfBytes;                          // 16 KB (K then V)
constexpr int kRingBytes = kStages * kStageBytes;                    // 64 KB
constexpr int kSmemBytes = kRingBytes + 1024 /*align slack*/ + 128 /*barriers*/;

struct alignas(8) Barriers {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint32_t unit_ok[kStages];  // the stage's unit was loaded (its page index is valid)
  int abort_word;
};
static_assert(kConsumerWarps == kHeadsPerCta, "one consumer warp per KV head of the CTA");

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
  load_q_frags(qa, reinterpret_cast<const __nv_bfloat16*>(a.q) +
                       (static_cast<long long>(b) * a.Hq + head0) * kHeadDim,
               a.group, head_ok);
  WarpState st;
  init_state(st, a.sinks + head0, a.group, c == 0 && head_ok);

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
  reduce_sums(st);
  const bool direct = n_chunks == 1;
#pragma unroll
  for (int half = 0; half < (kTwoRows ? 2 : 1); ++half) {
    const int row = half ? r1 : r0;
    if (row >= a.group) continue;
    const long long grow = static_cast<long long>(b) * a.Hq + head0 + row;
    if (direct)
      write_row(st, half, reinterpret_cast<__nv_bfloat16*>(a.out) + grow * kHeadDim,
                a.lse ? a.lse + grow : nullptr, nullptr, nullptr);
    else
      write_row(st, half, nullptr, nullptr, a.o_part + (grow * a.s_stride + c) * kHeadDim,
                a.lse_part + grow * a.s_stride + c);
  }
}

// ---------------------------------------------------------------- stream-K
// Share bounds: CTA i of G takes units [floor(i U / G), floor((i+1) U / G)).
__device__ __forceinline__ long long share_lo(long long i, long long U, long long G) { return i * U / G; }
// The CTA whose share holds unit x (0 <= x < U).
__device__ __forceinline__ int share_of(long long x, long long U, long long G) {
  return static_cast<int>(((x + 1) * G - 1) / U);
}

constexpr int kStreamTableBytes = (kStreamMaxStreams + 1) * 4;
constexpr int kStreamSmemBytes = kSmemBytes + kStreamTableBytes;

// kPoll: the waits poll (a test's short wait limit); otherwise they block.
template <bool kTwoRows, bool kPoll>
__global__ void __launch_bounds__(kThreads)
    decode_streamk_kernel(const __grid_constant__ CUtensorMap k_map,
                          const __grid_constant__ CUtensorMap v_map, const DecodeArgs a,
                          const StreamKArgs sk) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Barriers* bars = reinterpret_cast<Barriers*>(ring + kRingBytes);
  int* start = reinterpret_cast<int*>(ring + kRingBytes + 128);  // [n_streams + 1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_streams = a.B * sk.n_groups;
  const int kv_cap = a.bt_stride * a.page_size;  // keys beyond the table row are not read

  // ---- the streams' unit counts and their prefix sums (every CTA the same)
  for (int s = threadIdx.x; s < n_streams; s += blockDim.x) {
    const int kv_raw = max(0, a.kv_lens[s / sk.n_groups]);
    if (blockIdx.x == 0 && s % sk.n_groups == 0 && kv_raw > kv_cap && a.err_flag)
      atomicOr(a.err_flag, kFlagBadPage);
    start[s + 1] = (min(kv_raw, kv_cap) + kUnitTokens - 1) / kUnitTokens;
  }
  if (threadIdx.x == 0) start[0] = 0;
  __syncthreads();
  if (warp == 0) {
    const int per = (n_streams + 31) / 32;
    const int lo = 1 + lane * per, hi = min(n_streams, lo + per - 1);
    int run = 0;
    for (int i = lo; i <= hi; ++i) run += start[i];
    int incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += x;
    }
    int acc = incl - run;
    for (int i = lo; i <= hi; ++i) {
      acc += start[i];
      start[i] = acc;
    }
  }
  __syncthreads();
  const long long U = start[n_streams];
  const long long G = max(1LL, min(static_cast<long long>(gridDim.x), U / kStreamMinShare));
  if (blockIdx.x == 0) {  // the merge reads the same table
    for (int s = threadIdx.x; s <= n_streams; s += blockDim.x) sk.stream_start[s] = start[s];
    if (threadIdx.x == 0) *sk.shares = static_cast<int>(G);
  }
  if (blockIdx.x >= G || U == 0) return;
  const long long x_begin = share_lo(blockIdx.x, U, G), x_end = share_lo(blockIdx.x + 1, U, G);
  // first stream with units in this share
  int s_first = 0;
  {
    int lo = 0, hi = n_streams - 1;  // last s with start[s] <= x_begin
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (start[mid] <= x_begin) lo = mid; else hi = mid - 1;
    }
    s_first = lo;
  }

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&bars->full[st], 1);
      mbar_init(&bars->empty[st], kConsumerWarps);
    }
    bars->abort_word = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // Pieces of the share: stream s, its units [u0, u1).
  auto piece = [&](int s, int& u0, int& u1) {
    u0 = static_cast<int>(max(x_begin, static_cast<long long>(start[s])) - start[s]);
    u1 = static_cast<int>(min(x_end, static_cast<long long>(start[s + 1])) - start[s]);
  };

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&k_map);
      tma_prefetch_map(&v_map);
    }
    const uint64_t policy = l2_policy_evict_first();
    const int units_per_page = a.page_size / kUnitTokens;
    int it = 0;
    bool ok = true;
    for (int s = s_first; ok && s < n_streams && start[s] < x_end; ++s) {
      int u0, u1;
      piece(s, u0, u1);
      if (u1 <= u0) continue;
      const int b = s / sk.n_groups, g0 = (s % sk.n_groups) * kHeadsPerCta;
      const int kv_len = min(max(0, a.kv_lens[b]), kv_cap);
      const int32_t* bt_row = a.block_table + static_cast<long long>(b) * a.bt_stride;
      if (a.k_new && kv_len >= 1) {
        // Append mode: the piece holding the stream's last position writes the
        // step's key and value rows of its heads there before any copy of that
        // unit is issued (the proxy fences order them before the TMA reads).
        const int unit_last = (kv_len - 1) / kUnitTokens;
        if (unit_last >= u0 && unit_last < u1) {
          const int pos = kv_len - 1;
          const int phys = bt_row[pos / a.page_size];
          if (phys >= 0 && phys < a.num_pages) {
            const long long row = static_cast<long long>(phys) * a.page_size + pos % a.page_size;
            constexpr int kPieces = kHeadDim * 2 / 16;
            for (int i = lane; i < 2 * kHeadsPerCta * kPieces; i += 32) {
              const int t = i / (kHeadsPerCta * kPieces), h = (i / kPieces) % kHeadsPerCta,
                        pc = i % kPieces;
              const int g = g0 + h;
              if (g < a.Hkv) {
                const uint4* src = reinterpret_cast<const uint4*>(t ? a.v_new : a.k_new) +
                                   (static_cast<long long>(b) * a.Hkv + g) * kPieces + pc;
                uint4* dst = reinterpret_cast<uint4*>(t ? a.v_cache_w : a.k_cache_w) +
                             (row * a.Hkv + g) * kPieces + pc;
                *dst = *src;
              }
            }
            fence_proxy_async_global();
          }
        }
        __syncwarp();
        fence_proxy_async_global();
      }
      // Lane l holds the page of unit u0 + 32k + l of the current window.
      auto fetch = [&](int base, int& phys, int& tok) {
        const int u = u0 + base + lane;
        phys = -1;
        tok = 0;
        if (u < u1) {
          phys = bt_row[u / units_per_page];
          tok = (u % units_per_page) * kUnitTokens;
        }
      };
      int cur_phys, cur_tok, nxt_phys, nxt_tok;
      fetch(0, cur_phys, cur_tok);
      fetch(32, nxt_phys, nxt_tok);
      for (int k = 0; k < u1 - u0; ++k, ++it) {
        if (k > 0 && (k & 31) == 0) {
          cur_phys = nxt_phys;
          cur_tok = nxt_tok;
          fetch(k + 32, nxt_phys, nxt_tok);
        }
        const int stage = it % kStages;
        if (it >= kStages) {
          const bool ready = mbar_wait<kPoll>(&bars->empty[stage], ((it / kStages) + 1) & 1,
                                              &bars->abort_word, a.err_flag, a.wait_limit_ns);
          ok = __all_sync(0xffffffffu, ready);
          if (!ok) break;
        }
        const int phys = __shfl_sync(0xffffffffu, cur_phys, k & 31);
        const int tok = __shfl_sync(0xffffffffu, cur_tok, k & 31);
        const bool valid = phys >= 0 && phys < a.num_pages;
        if (lane == 0) {
          if (!valid && a.err_flag) atomicOr(a.err_flag, kFlagBadPage);
          bars->unit_ok[stage] = valid ? 1u : 0u;
          mbar_arrive_expect_tx(&bars->full[stage], valid ? kStageBytes : 0);
          if (valid) {
            uint8_t* stp = ring + stage * kStageBytes;
            tma_load_4d_hint(stp, &k_map, &bars->full[stage], 0, tok, g0, phys, policy);
            tma_load_4d_hint(stp + kHalfBytes, &v_map, &bars->full[stage], 0, tok, g0, phys, policy);
          }
        }
        __syncwarp();
      }
    }
    // Drain: every issued load lands before the CTA's shared memory goes away.
    if (lane == 0) {
      for (int i = max(0, it - kStages); i < it; ++i)
        mbar_wait_drain(&bars->full[i % kStages], (i / kStages) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int r0 = lane >> 2, r1 = r0 + 8;
  int it = 0;
  for (int s = s_first; s < n_streams && start[s] < x_end; ++s) {
    int u0, u1;
    piece(s, u0, u1);
    if (u1 <= u0) continue;
    const int b = s / sk.n_groups, g0 = (s % sk.n_groups) * kHeadsPerCta;
    const int kv_len = min(max(0, a.kv_lens[b]), kv_cap);
    const int g = g0 + warp;  // this warp's KV head
    const bool head_ok = g < a.Hkv;
    const int head0 = g * a.group;
    uint32_t qa[4][4];
    load_q_frags(qa, reinterpret_cast<const __nv_bfloat16*>(a.q) +
                         (static_cast<long long>(b) * a.Hq + head0) * kHeadDim,
                 a.group, head_ok);
    WarpState st;
    init_state(st, a.sinks + head0, a.group, u0 == 0 && head_ok);  // the sink: the stream's first piece
    bool ok = true;
    for (int k = 0; k < u1 - u0; ++k, ++it) {
      const int stage = it % kStages;
      const bool ready = mbar_wait<kPoll>(&bars->full[stage], (it / kStages) & 1, &bars->abort_word,
                                          a.err_flag, a.wait_limit_ns);
      ok = __all_sync(0xffffffffu, ready);
      if (!ok) break;
      if (head_ok && bars->unit_ok[stage]) {
        const int u = u0 + k;
        const uint32_t k_base = smem_addr(ring + stage * kStageBytes + warp * kUnitBytes);
        const uint32_t v_base = k_base + kHalfBytes;
        const int n_valid = min(kUnitTokens, kv_len - u * kUnitTokens);
        consume_unit<kTwoRows>(k_base, v_base, n_valid, qa, a.scale_log2, st);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty[stage]);
    }
    if (!ok) return;
    if (!head_ok) continue;
    reduce_sums(st);
    const int units = start[s + 1] - start[s];
    const bool direct = u0 == 0 && u1 == units;
    const int slot = static_cast<int>(blockIdx.x) - share_of(start[s], U, G);
#pragma unroll
    for (int half = 0; half < (kTwoRows ? 2 : 1); ++half) {
      const int row = half ? r1 : r0;
      if (row >= a.group) continue;
      const long long grow = static_cast<long long>(b) * a.Hq + head0 + row;
      if (direct)
        write_row(st, half, reinterpret_cast<__nv_bfloat16*>(a.out) + grow * kHeadDim,
                  a.lse ? a.lse + grow : nullptr, nullptr, nullptr);
      else
        write_row(st, half, nullptr, nullptr, a.o_part + (grow * a.s_stride + slot) * kHeadDim,
                  a.lse_part + grow * a.s_stride + slot);
    }
  }
}

}  // namespace

cudaError_t launch_decode_streamk(const DecodeArgs& a, const StreamKArgs& sk,
                                  const CUtensorMap& k_map, const CUtensorMap& v_map,
                                  unsigned grid, cudaStream_t stream) {
  const bool poll = a.wait_limit_ns < kPollLimitNs;
  auto kern = a.group > 8 ? (poll ? decode_streamk_kernel<true, true> : decode_streamk_kernel<true, false>)
                          : (poll ? decode_streamk_kernel<false, true> : decode_streamk_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kStreamSmemBytes, stream>>>(k_map, v_map, a, sk);
  return cudaGetLastError();
}

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
