// C-ABI entry points declared in include/attn_sink.h: host-side argument
// checks, TMA descriptor encoding, workspace carve-up and kernel dispatch.
// Nothing here allocates, synchronises or reads device memory.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>

#include "attn_sink.h"
#include "kernels.h"

using namespace attn_sink;

namespace {

// SM count the decode split plan assumes when no device can be queried (a
// host without a GPU asking for workspace sizes): a full GB300.
constexpr int kDefaultSms = 152;
constexpr float kLog2e = 1.4426950408889634f;

// Limit of each pipeline wait inside the kernels, read when a call is enqueued.
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// SM count of the current device (cached per device), or kDefaultSms when no
// device can be queried.  The decode split plan and its workspace size use it,
// so both must be asked with the same device current.
int current_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();  // clear the error a missing device leaves behind
    return kDefaultSms;
  }
  int sms = cache[dev].load(std::memory_order_relaxed);
  if (sms > 0) return sms;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    cudaGetLastError();
    return kDefaultSms;
  }
  cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a [rows, cols] row-major matrix, box {64, box_rows},
// 128-byte swizzle (64 bf16 = one 128-byte row per box line).
bool make_map_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                 uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 tensor map over q [total_q, Hq, 64]: box {64, group, tokens}.
bool make_map_q(CUtensorMap* map, const void* base, uint64_t total_q, uint64_t Hq, uint32_t group,
                uint32_t tokens) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, Hq, total_q};
  cuuint64_t strides[2] = {64 * 2, Hq * 64 * 2};
  cuuint32_t box[3] = {64, group, tokens};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D bf16 tensor map over a paged NHD cache [num_pages, page_size, Hkv, 64]
// ordered (dim, token in page, head, page), box {64, 16, box_heads, 1}: one
// copy brings a 16-token slice of box_heads heads, each head's 16 rows
// contiguous (2 KB) in shared memory.  The head stride (128 B) is below the
// token stride; TMA takes each dimension's stride as given.
bool make_map_paged_heads(CUtensorMap* map, const void* base, uint64_t num_pages,
                          uint64_t page_size, uint64_t Hkv, uint32_t box_heads = kHeadsPerCta) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {64, page_size, Hkv, num_pages};
  cuuint64_t strides[3] = {Hkv * 64 * 2, 64 * 2, page_size * Hkv * 64 * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kUnitTokens), box_heads, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

attn_sink_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_SINK_OK;
  if (e == cudaErrorNotSupported) return ATTN_SINK_ERR_UNSUPPORTED;
  return ATTN_SINK_ERR_CUDA;
}

// Shape checks common to prefill and decode.
attn_sink_status check_shapes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                              int32_t num_pages, int32_t bt_stride, attn_sink_dtype dtype) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || page_size <= 0 || num_pages <= 0 || bt_stride <= 0)
    return ATTN_SINK_ERR_INVALID_ARG;
  if (dtype != ATTN_SINK_BF16 && dtype != ATTN_SINK_FP32) return ATTN_SINK_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_SINK_ERR_INVALID_ARG;
  if (D != kHeadDim) return ATTN_SINK_ERR_UNSUPPORTED;
  const int group = Hq / Hkv;
  if (!pow2(group) || group > 16) return ATTN_SINK_ERR_UNSUPPORTED;
  if (dtype == ATTN_SINK_BF16 && (page_size % kUnitTokens != 0 || page_size > 256))
    return ATTN_SINK_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_pages) * page_size > INT_MAX) return ATTN_SINK_ERR_UNSUPPORTED;
  if (static_cast<long long>(bt_stride) * page_size > INT_MAX) return ATTN_SINK_ERR_UNSUPPORTED;
  return ATTN_SINK_OK;
}

// Decode split plan: chunk length in 16-key units and partial slots per row.
struct DecodePlan {
  int num_splits;   // > 0 fixed split count, 0 chunk_units mode
  int chunk_units;
  int max_chunks;   // grid.x
  int s_stride;     // 0: no partials needed
  bool streamk;     // persistent stream-K split (automatic mode)
  int n_groups;     // stream-K: KV-head groups per sequence
};

// num_splits = ATTN_SINK_SPLIT_PERSISTENT runs the persistent stream-K kernel
// (when the prefix table of its (sequence, head group) streams fits in shared
// memory; otherwise the automatic split).  The automatic split stays the
// default: on the gpt-oss decode shape it measured 97-99 us per call against
// 101.5-102 us for stream-K, whose static equal shares cannot absorb the
// per-SM bandwidth differences that the hardware block scheduler absorbs when
// it hands out the chunk CTAs.

DecodePlan plan_decode(int32_t B, int32_t Hkv, int32_t bt_stride, int32_t page_size,
                       int32_t num_splits) {
  DecodePlan p{};
  if (num_splits > 0) {
    p.num_splits = num_splits;
    p.chunk_units = 0;
    p.max_chunks = num_splits;
    p.s_stride = num_splits > 1 ? num_splits : 0;
    return p;
  }
  const bool persistent = num_splits == ATTN_SINK_SPLIT_PERSISTENT;
  const long long max_units =
      (static_cast<long long>(bt_stride) * page_size + kUnitTokens - 1) / kUnitTokens;
  const long long groups = (Hkv + kHeadsPerCta - 1) / kHeadsPerCta;
  if (persistent && static_cast<long long>(B) * groups <= kStreamMaxStreams &&
      static_cast<long long>(B) * groups * max_units <= INT_MAX) {  // (int prefix sums)
    // Shares hold at least kStreamMinShare units, so a stream spans at most
    // ceil(units / kStreamMinShare) + 1 of them: one partial slot each.
    p.num_splits = 0;
    p.streamk = true;
    p.n_groups = static_cast<int>(groups);
    p.s_stride = static_cast<int>((max_units + kStreamMinShare - 1) / kStreamMinShare) + 1;
    return p;
  }
  // A CTA covers kHeadsPerCta KV heads.  Start at 2048 keys per CTA and halve
  // while the grid would have fewer than 8 CTAs per SM; long chunks keep the
  // fp32 partials (and the merge) small.
  int cu = 128;
  const long long target = 8LL * current_sm_count();
  while (cu > 4 && static_cast<long long>(B) * groups * ((max_units + cu - 1) / cu) < target) cu /= 2;
  p.num_splits = 0;
  p.chunk_units = cu;
  p.max_chunks = static_cast<int>(std::max(1LL, (max_units + cu - 1) / cu));
  p.s_stride = p.max_chunks > 1 ? p.max_chunks : 0;
  return p;
}

// Partial slots per decode row of a mixed batch: the decode items of the
// longest sequence the table row can hold.
int mixed_slots(int32_t bt_stride, int32_t page_size) {
  const long long units = (static_cast<long long>(bt_stride) * page_size + kUnitTokens - 1) / kUnitTokens;
  return static_cast<int>(std::max(1LL, (units + kMixedChunkUnits - 1) / kMixedChunkUnits));
}

// Stream-K table in the workspace, after the partials: the streams' prefix
// sums and the number of shares.
size_t streamk_table_bytes(int32_t B, int n_groups) {
  return align_up((static_cast<size_t>(B) * n_groups + 2) * sizeof(int), 256);
}

size_t partial_bytes(long long rows, int s_stride, size_t* o_bytes) {
  const size_t ob = align_up(static_cast<size_t>(rows) * s_stride * kHeadDim * sizeof(float), 256);
  const size_t lb = align_up(static_cast<size_t>(rows) * s_stride * sizeof(float), 256);
  if (o_bytes) *o_bytes = ob;
  return ob + lb;
}

}  // namespace

extern "C" {

ATTN_SINK_API uint64_t attn_sink_set_wait_limit_ns(uint64_t ns) {
  return g_wait_limit_ns.exchange(ns == 0 ? kWaitLimitNs : ns);
}

ATTN_SINK_API const char* attn_sink_status_string(attn_sink_status status) {
  switch (status) {
    case ATTN_SINK_OK: return "ok";
    case ATTN_SINK_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_SINK_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case ATTN_SINK_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case ATTN_SINK_ERR_CUDA: return "CUDA launch or driver error";
  }
  return "unknown status";
}

ATTN_SINK_API size_t attn_sink_decode_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                                     int32_t block_table_stride, int32_t page_size,
                                                     int32_t num_splits) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D != kHeadDim || block_table_stride <= 0 ||
      page_size <= 0 || num_splits < ATTN_SINK_SPLIT_PERSISTENT)
    return 0;
  const DecodePlan p = plan_decode(B, Hkv, block_table_stride, page_size, num_splits);
  if (p.streamk)
    return partial_bytes(static_cast<long long>(B) * Hq, p.s_stride, nullptr) +
           streamk_table_bytes(B, p.n_groups);
  if (p.s_stride == 0) return 0;
  return partial_bytes(static_cast<long long>(B) * Hq, p.s_stride, nullptr);
}

ATTN_SINK_API size_t attn_sink_mixed_workspace_size(int32_t num_decode, int32_t Hq, int32_t Hkv,
                                                    int32_t D, int32_t block_table_stride,
                                                    int32_t page_size) {
  if (num_decode < 0 || Hq <= 0 || Hkv <= 0 || D != kHeadDim || block_table_stride <= 0 ||
      page_size <= 0)
    return 0;
  const int s_stride = mixed_slots(block_table_stride, page_size);
  return kPrefillWorkspaceBytes +
         (s_stride > 1 ? partial_bytes(static_cast<long long>(num_decode) * Hq, s_stride, nullptr) : 0);
}

ATTN_SINK_API size_t attn_sink_prefill_workspace_size(int32_t B, int32_t Hq, int32_t D,
                                                      int32_t max_q_len) {
  if (B <= 0 || Hq <= 0 || D != kHeadDim || max_q_len <= 0) return 0;
  return kPrefillWorkspaceBytes;
}

}  // extern "C"

namespace {

}  // namespace

namespace attn_sink {

// Host-side checks of a decode call that need no workspace (shared with the
// static-scratch entry point, so both report the same status for a bad call).
attn_sink_status decode_validate(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* kv_lens, const int32_t* block_table,
                                 int32_t block_table_stride, const float* sinks, const void* out,
                                 int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                                 int32_t num_pages, float scale, int32_t num_splits,
                                 attn_sink_dtype dtype) {
  attn_sink_status st =
      check_shapes(B, Hq, Hkv, D, page_size, num_pages, block_table_stride, dtype);
  if (st != ATTN_SINK_OK) return st;
  if (!q || !k_cache || !v_cache || !kv_lens || !block_table || !sinks || !out)
    return ATTN_SINK_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return ATTN_SINK_ERR_INVALID_ARG;
  if (num_splits < ATTN_SINK_SPLIT_PERSISTENT || num_splits > 256 || !std::isfinite(scale))
    return ATTN_SINK_ERR_INVALID_ARG;
  return ATTN_SINK_OK;
}

}  // namespace attn_sink

namespace {

// Decode, optionally appending the step's key and value first (k_new != null).
attn_sink_status decode_impl(
    const void* q, const void* k_new, const void* v_new, const void* k_cache, const void* v_cache,
    const int32_t* kv_lens, const int32_t* block_table, int32_t block_table_stride,
    const float* sinks, void* out, float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
    int32_t page_size, int32_t num_pages, float scale, int32_t num_splits, attn_sink_dtype dtype,
    int32_t* err_flag, void* workspace, size_t workspace_bytes, void* stream) {
  const attn_sink_status st =
      decode_validate(q, k_cache, v_cache, kv_lens, block_table, block_table_stride, sinks, out, B,
                      Hq, Hkv, D, page_size, num_pages, scale, num_splits, dtype);
  if (st != ATTN_SINK_OK) return st;
  if (B == 0) return ATTN_SINK_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int group = Hq / Hkv;

  if (dtype == ATTN_SINK_FP32) {
    const int S = num_splits <= 0 ? 1 : num_splits;
    size_t o_bytes = 0;
    const size_t need = S > 1 ? partial_bytes(static_cast<long long>(B) * Hq, S, &o_bytes) : 0;
    if (need && (!workspace || workspace_bytes < need ||
                 (reinterpret_cast<uintptr_t>(workspace) & 255u)))
      return ATTN_SINK_ERR_WORKSPACE;
    if (k_new) {
      AppendArgs ap{};
      ap.k_new = k_new;
      ap.v_new = v_new;
      ap.k_cache = const_cast<void*>(k_cache);
      ap.v_cache = const_cast<void*>(v_cache);
      ap.kv_lens = kv_lens;
      ap.block_table = block_table;
      ap.err_flag = err_flag;
      ap.B = B;
      ap.Hkv = Hkv;
      ap.bt_stride = block_table_stride;
      ap.page_size = page_size;
      ap.num_pages = num_pages;
      ap.elem_bytes = 4;
      cudaError_t e = launch_append(ap, s);
      if (e != cudaSuccess) return from_cuda(e);
    }
    SimtArgs a{};
    a.q = static_cast<const float*>(q);
    a.k_cache = static_cast<const float*>(k_cache);
    a.v_cache = static_cast<const float*>(v_cache);
    a.cu_seqlens_q = nullptr;
    a.kv_lens = kv_lens;
    a.block_table = block_table;
    a.sinks = sinks;
    a.out = static_cast<float*>(out);
    a.lse = lse;
    a.o_part = S > 1 ? static_cast<float*>(workspace) : nullptr;
    a.lse_part = S > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + o_bytes) : nullptr;
    a.err_flag = err_flag;
    a.B = B;
    a.total_q = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.group = group;
    a.bt_stride = block_table_stride;
    a.page_size = page_size;
    a.num_pages = num_pages;
    a.scale_log2 = scale * kLog2e;
    a.causal = 0;
    a.num_splits = S;
    cudaError_t e = launch_simt_fp32(a, s);
    if (e != cudaSuccess || S == 1) return from_cuda(e);
    MergeArgs m{};
    m.o_part = a.o_part;
    m.lse_part = a.lse_part;
    m.out = out;
    m.lse = lse;
    m.rows = B * Hq;
    m.s_stride = S;
    m.num_parts = S;
    m.out_fp32 = 1;
    return from_cuda(launch_merge(m, s));
  }

  const DecodePlan p = plan_decode(B, Hkv, block_table_stride, page_size, num_splits);
  size_t o_bytes = 0;
  size_t need = p.s_stride ? partial_bytes(static_cast<long long>(B) * Hq, p.s_stride, &o_bytes) : 0;
  if (p.streamk) need += streamk_table_bytes(B, p.n_groups);
  if (need && (!workspace || workspace_bytes < need ||
               (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return ATTN_SINK_ERR_WORKSPACE;

  CUtensorMap k_map, v_map;
  if (!make_map_paged_heads(&k_map, k_cache, static_cast<uint64_t>(num_pages),
                            static_cast<uint64_t>(page_size), static_cast<uint64_t>(Hkv)) ||
      !make_map_paged_heads(&v_map, v_cache, static_cast<uint64_t>(num_pages),
                            static_cast<uint64_t>(page_size), static_cast<uint64_t>(Hkv)))
    return ATTN_SINK_ERR_CUDA;

  DecodeArgs a{};
  a.q = q;
  a.kv_lens = kv_lens;
  a.block_table = block_table;
  a.sinks = sinks;
  a.out = out;
  a.lse = lse;
  a.o_part = p.s_stride ? static_cast<float*>(workspace) : nullptr;
  a.lse_part = p.s_stride ? reinterpret_cast<float*>(static_cast<char*>(workspace) + o_bytes) : nullptr;
  a.err_flag = err_flag;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.group = group;
  a.bt_stride = block_table_stride;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.scale_log2 = scale * kLog2e;
  a.num_splits = p.num_splits;
  a.chunk_units = p.chunk_units;
  a.max_chunks = p.max_chunks;
  a.s_stride = p.s_stride;
  a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache_w = k_new ? const_cast<void*>(k_cache) : nullptr;
  a.v_cache_w = k_new ? const_cast<void*>(v_cache) : nullptr;
  if (p.streamk) {
    StreamKArgs sk{};
    sk.n_groups = p.n_groups;
    sk.stream_start = reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                             partial_bytes(static_cast<long long>(B) * Hq, p.s_stride, nullptr));
    sk.shares = sk.stream_start + static_cast<long long>(B) * p.n_groups + 1;
    cudaError_t e = launch_decode_streamk(a, sk, k_map, v_map, 3u * current_sm_count(), s);
    if (e != cudaSuccess) return from_cuda(e);
    MergeArgs m{};
    m.o_part = a.o_part;
    m.lse_part = a.lse_part;
    m.out = out;
    m.lse = lse;
    m.rows = B * Hq;
    m.s_stride = p.s_stride;
    m.num_parts = p.s_stride;
    m.Hq = Hq;
    m.stream_start = sk.stream_start;
    m.shares = sk.shares;
    m.group = group;
    m.n_groups = p.n_groups;
    m.sinks = sinks;
    return from_cuda(launch_merge(m, s));
  }
  cudaError_t e = launch_decode_bf16(a, k_map, v_map, s);
  if (e != cudaSuccess || p.s_stride == 0) return from_cuda(e);

  MergeArgs m{};
  m.o_part = a.o_part;
  m.lse_part = a.lse_part;
  m.out = out;
  m.lse = lse;
  m.rows = B * Hq;
  m.s_stride = p.s_stride;
  m.num_parts = p.num_splits > 0 ? p.num_splits : p.max_chunks;
  m.out_fp32 = 0;
  if (p.num_splits == 0) {
    m.kv_lens = kv_lens;
    m.Hq = Hq;
    m.chunk_units = p.chunk_units;
    m.kv_cap = block_table_stride * page_size;  // as the split kernel clamps kv_len
  }
  return from_cuda(launch_merge(m, s));
}

// Ragged prefill (num_decode < 0) or a mixed batch whose first num_decode
// sequences are single-query decode rows (attn_sink_mixed).
attn_sink_status prefill_impl(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
    const int32_t* kv_lens, const int32_t* block_table, int32_t block_table_stride,
    const float* sinks, void* out, float* lse, int32_t B, int32_t num_decode, int32_t total_q,
    int32_t max_q_len, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages,
    float scale, int32_t causal, attn_sink_dtype dtype, int32_t* err_flag, void* workspace,
    size_t workspace_bytes, void* stream) {
  const bool mixed = num_decode >= 0;
  attn_sink_status st =
      check_shapes(B, Hq, Hkv, D, page_size, num_pages, block_table_stride, dtype);
  if (st != ATTN_SINK_OK) return st;
  if (!q || !k_cache || !v_cache || !cu_seqlens_q || !kv_lens || !block_table || !sinks || !out)
    return ATTN_SINK_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return ATTN_SINK_ERR_INVALID_ARG;
  if (total_q < 0 || max_q_len < 0 || (causal != 0 && causal != 1) || !std::isfinite(scale))
    return ATTN_SINK_ERR_INVALID_ARG;
  if (mixed && dtype == ATTN_SINK_BF16 && (B > kMixedMaxSeqs || Hq > kMixedMaxHeads))
    return ATTN_SINK_ERR_UNSUPPORTED;
  if (B == 0 || total_q == 0) return ATTN_SINK_OK;
  if (max_q_len == 0 && !(mixed && num_decode > 0)) return ATTN_SINK_OK;
  if (static_cast<long long>(total_q) * Hq > INT_MAX) return ATTN_SINK_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int group = Hq / Hkv;

  if (dtype == ATTN_SINK_FP32) {
    // fp32 runs the whole batch (decode rows included) on the SIMT path.
    SimtArgs a{};
    a.q = static_cast<const float*>(q);
    a.k_cache = static_cast<const float*>(k_cache);
    a.v_cache = static_cast<const float*>(v_cache);
    a.cu_seqlens_q = cu_seqlens_q;
    a.kv_lens = kv_lens;
    a.block_table = block_table;
    a.sinks = sinks;
    a.out = static_cast<float*>(out);
    a.lse = lse;
    a.err_flag = err_flag;
    a.B = B;
    a.total_q = total_q;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.group = group;
    a.bt_stride = block_table_stride;
    a.page_size = page_size;
    a.num_pages = num_pages;
    a.scale_log2 = scale * kLog2e;
    a.causal = causal;
    a.num_splits = 1;
    return from_cuda(launch_simt_fp32(a, s));
  }

  const int s_stride = mixed ? mixed_slots(block_table_stride, page_size) : 0;
  const size_t need = mixed ? attn_sink_mixed_workspace_size(num_decode, Hq, Hkv, D,
                                                             block_table_stride, page_size)
                            : kPrefillWorkspaceBytes;
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_SINK_ERR_WORKSPACE;
  CUtensorMap q_map, k_map, v_map, k8_map, v8_map;
  const uint64_t rows = static_cast<uint64_t>(num_pages) * page_size;
  if (!make_map_q(&q_map, q, static_cast<uint64_t>(total_q), static_cast<uint64_t>(Hq),
                  static_cast<uint32_t>(group), static_cast<uint32_t>(128 / group)) ||
      !make_map_2d(&k_map, k_cache, static_cast<uint64_t>(Hkv) * kHeadDim, rows, kUnitTokens) ||
      !make_map_2d(&v_map, v_cache, static_cast<uint64_t>(Hkv) * kHeadDim, rows, kUnitTokens))
    return ATTN_SINK_ERR_CUDA;
  if (mixed &&
      (!make_map_paged_heads(&k8_map, k_cache, static_cast<uint64_t>(num_pages),
                             static_cast<uint64_t>(page_size), static_cast<uint64_t>(Hkv), kMixedBoxHeads) ||
       !make_map_paged_heads(&v8_map, v_cache, static_cast<uint64_t>(num_pages),
                             static_cast<uint64_t>(page_size), static_cast<uint64_t>(Hkv), kMixedBoxHeads)))
    return ATTN_SINK_ERR_CUDA;
  PrefillArgs a{};
  a.cu_seqlens_q = cu_seqlens_q;
  a.kv_lens = kv_lens;
  a.block_table = block_table;
  a.sinks = sinks;
  a.out = out;
  a.lse = lse;
  a.err_flag = err_flag;
  a.B = B;
  a.total_q = total_q;
  a.max_q_len = max_q_len;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.group = group;
  a.bt_stride = block_table_stride;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.scale_log2 = scale * kLog2e;
  a.causal = causal;
  a.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  a.tile_ctr = static_cast<unsigned long long*>(workspace);
  if (!mixed) return from_cuda(launch_prefill_bf16(a, q_map, k_map, v_map, s));

  MixedArgs mx{};
  mx.num_decode = num_decode;
  mx.q = q;
  mx.dec_ctr = a.tile_ctr + 1;
  mx.dec_chunk_units = kMixedChunkUnits;
  size_t o_bytes = 0;
  if (s_stride > 1) {
    partial_bytes(static_cast<long long>(num_decode) * Hq, s_stride, &o_bytes);
    char* parts = static_cast<char*>(workspace) + kPrefillWorkspaceBytes;
    mx.o_part = reinterpret_cast<float*>(parts);
    mx.lse_part = reinterpret_cast<float*>(parts + o_bytes);
    mx.s_stride = s_stride;
  }
  cudaError_t e = launch_mixed_bf16(a, mx, q_map, k_map, v_map, k8_map, v8_map, s);
  if (e != cudaSuccess || s_stride <= 1 || num_decode == 0) return from_cuda(e);
  // Decode rows split into several items: LSE merge of their partials.
  MergeArgs m{};
  m.o_part = mx.o_part;
  m.lse_part = mx.lse_part;
  m.out = out;
  m.lse = lse;
  m.rows = num_decode * Hq;
  m.s_stride = s_stride;
  m.num_parts = s_stride;
  m.out_fp32 = 0;
  m.kv_lens = kv_lens;
  m.Hq = Hq;
  m.chunk_units = kMixedChunkUnits;
  m.kv_cap = block_table_stride * page_size;
  m.seq_start = cu_seqlens_q;
  return from_cuda(launch_merge(m, s));
}

}  // namespace

extern "C" {

ATTN_SINK_API attn_sink_status attn_sink_decode(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_lens,
    const int32_t* block_table, int32_t block_table_stride, const float* sinks, void* out,
    float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
    int32_t num_pages, float scale, int32_t num_splits, attn_sink_dtype dtype, int32_t* err_flag,
    void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(q, nullptr, nullptr, k_cache, v_cache, kv_lens, block_table,
                     block_table_stride, sinks, out, lse, B, Hq, Hkv, D, page_size, num_pages,
                     scale, num_splits, dtype, err_flag, workspace, workspace_bytes, stream);
}

ATTN_SINK_API attn_sink_status attn_sink_decode_append(
    const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
    const int32_t* kv_lens, const int32_t* block_table, int32_t block_table_stride,
    const float* sinks, void* out, float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
    int32_t page_size, int32_t num_pages, float scale, int32_t num_splits, attn_sink_dtype dtype,
    int32_t* err_flag, void* workspace, size_t workspace_bytes, void* stream) {
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return ATTN_SINK_ERR_INVALID_ARG;
  return decode_impl(q, k_new, v_new, k_cache, v_cache, kv_lens, block_table, block_table_stride,
                     sinks, out, lse, B, Hq, Hkv, D, page_size, num_pages, scale, num_splits, dtype,
                     err_flag, workspace, workspace_bytes, stream);
}

ATTN_SINK_API attn_sink_status attn_sink_merge(const float* o_parts, const float* lse_parts,
                                               int32_t rows, int32_t S, int32_t D, void* out,
                                               float* lse_out, attn_sink_dtype dtype,
                                               void* stream) {
  if (rows < 0 || S <= 0 || !o_parts || !lse_parts || !out) return ATTN_SINK_ERR_INVALID_ARG;
  if (dtype != ATTN_SINK_BF16 && dtype != ATTN_SINK_FP32) return ATTN_SINK_ERR_INVALID_ARG;
  if (D != kHeadDim) return ATTN_SINK_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(o_parts) & 7u) || (reinterpret_cast<uintptr_t>(out) & 7u))
    return ATTN_SINK_ERR_INVALID_ARG;
  MergeArgs m{};
  m.o_part = o_parts;
  m.lse_part = lse_parts;
  m.out = out;
  m.lse = lse_out;
  m.rows = rows;
  m.s_stride = S;
  m.num_parts = S;
  m.out_fp32 = dtype == ATTN_SINK_FP32;
  return from_cuda(launch_merge(m, static_cast<cudaStream_t>(stream)));
}

ATTN_SINK_API attn_sink_status attn_sink_prefill(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
    const int32_t* kv_lens, const int32_t* block_table, int32_t block_table_stride,
    const float* sinks, void* out, float* lse, int32_t B, int32_t total_q, int32_t max_q_len,
    int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages, float scale,
    int32_t causal, attn_sink_dtype dtype, int32_t* err_flag, void* workspace,
    size_t workspace_bytes, void* stream) {
  return prefill_impl(q, k_cache, v_cache, cu_seqlens_q, kv_lens, block_table, block_table_stride,
                      sinks, out, lse, B, -1, total_q, max_q_len, Hq, Hkv, D, page_size, num_pages,
                      scale, causal, dtype, err_flag, workspace, workspace_bytes, stream);
}

ATTN_SINK_API attn_sink_status attn_sink_mixed(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
    const int32_t* kv_lens, const int32_t* block_table, int32_t block_table_stride,
    const float* sinks, void* out, float* lse, int32_t B, int32_t num_decode, int32_t total_q,
    int32_t max_q_len, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size, int32_t num_pages,
    float scale, int32_t causal, attn_sink_dtype dtype, int32_t* err_flag, void* workspace,
    size_t workspace_bytes, void* stream) {
  if (num_decode < 0 || num_decode > B) return ATTN_SINK_ERR_INVALID_ARG;
  return prefill_impl(q, k_cache, v_cache, cu_seqlens_q, kv_lens, block_table, block_table_stride,
                      sinks, out, lse, B, num_decode, total_q, max_q_len, Hq, Hkv, D, page_size,
                      num_pages, scale, causal, dtype, err_flag, workspace, workspace_bytes, stream);
}

}  // extern "C"
