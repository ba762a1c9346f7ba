// Internal launch interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn_sink.h"

namespace attn_sink {

// Host-side argument checks of attn_sink_decode (everything but the
// workspace), shared by the decode entry points.
attn_sink_status decode_validate(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* kv_lens, const int32_t* block_table,
                                 int32_t block_table_stride, const float* sinks, const void* out,
                                 int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                                 int32_t num_pages, float scale, int32_t num_splits,
                                 attn_sink_dtype dtype);

constexpr int kHeadDim = 64;     // the only head dimension the kernels are built for
constexpr int kUnitTokens = 16;  // keys per TMA box: one 16-row slice of a page
constexpr int kHeadsPerCta = 4;  // decode: KV heads per CTA (one TMA box covers them)
// Default limit of a pipeline wait inside the kernels, and the fixed limit of
// the drains that let in-flight copies land before a CTA exits.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
// Limits below this (a test setting) run the kernels' polling instantiation.
constexpr uint64_t kPollLimitNs = 1000000ull;  // 1 ms

// ------------------------------------------------------------- bf16 decode
struct DecodeArgs {
  const void* q;               // bf16 [B, Hq, 64]
  const int32_t* kv_lens;      // [B]
  const int32_t* block_table;  // [B, bt_stride]
  const float* sinks;          // [Hq]
  void* out;                   // bf16 [B, Hq, 64]   (rows that need no merge)
  float* lse;                  // [B, Hq] or null
  float* o_part;               // fp32 [B*Hq, s_stride, 64]
  float* lse_part;             // fp32 [B*Hq, s_stride]
  int32_t* err_flag;           // or null
  int B, Hq, Hkv, group;
  int bt_stride, page_size, num_pages;
  float scale_log2;            // scale * log2(e)
  int num_splits;              // > 0: fixed split count; 0: chunk_units mode
  int chunk_units;             // 16-key units per chunk when num_splits == 0
  int max_chunks;              // grid.x
  int s_stride;                // partial slots per row in o_part / lse_part
  uint64_t wait_limit_ns;      // limit of each pipeline wait (drains keep kWaitLimitNs)
  // Append mode (all null otherwise): before its keys are read, the step's
  // k_new / v_new [B, Hkv, 64] go into the slot of position kv_len - 1.
  const void* k_new;
  const void* v_new;
  void* k_cache_w;
  void* v_cache_w;
};

cudaError_t launch_decode_bf16(const DecodeArgs& a, const CUtensorMap& k_map,
                               const CUtensorMap& v_map, cudaStream_t stream);

// Persistent ("stream-K") split decode: every CTA takes an equal, contiguous
// share of all (sequence, group of kHeadsPerCta KV heads) key streams laid end
// to end, split at the streams' boundaries into pieces.  A stream inside one
// CTA's share is written directly; the pieces of a stream that spans CTAs
// c_first..c_last go to partial slots 0..c_last-c_first of its rows for the
// merge.  The shares come from prefix sums every CTA computes from kv_lens, so
// no counter is needed (nothing to zero between calls).
constexpr int kStreamMinShare = 32;      // 16-key units: shares are at least 512 keys
constexpr int kStreamMaxStreams = 2048;  // B * ceil(Hkv / kHeadsPerCta) the prefix table holds
struct StreamKArgs {
  int n_groups;        // ceil(Hkv / kHeadsPerCta)
  int* stream_start;   // workspace [B * n_groups + 1]: prefix sums of units (written by CTA 0)
  int* shares;         // workspace [1]: the number of CTAs with a share (written by CTA 0)
};

cudaError_t launch_decode_streamk(const DecodeArgs& a, const StreamKArgs& sk,
                                  const CUtensorMap& k_map, const CUtensorMap& v_map,
                                  unsigned grid, cudaStream_t stream);

// ------------------------------------------------------------- KV append
// Writes k_new / v_new [B, Hkv, 64] into the cache slot of position
// kv_lens[b] - 1 of every sequence with kv_lens[b] >= 1 (any element size).
struct AppendArgs {
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  const int32_t* kv_lens;
  const int32_t* block_table;
  int32_t* err_flag;
  int B, Hkv, bt_stride, page_size, num_pages, elem_bytes;
};

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);

// ------------------------------------------------------------- merge
struct MergeArgs {
  const float* o_part;    // [rows, s_stride, 64]
  const float* lse_part;  // [rows, s_stride]
  void* out;              // [rows, 64] bf16 or fp32
  float* lse;             // [rows] or null
  int rows, s_stride, num_parts;
  int out_fp32;
  // When kv_lens is set, row r belongs to sequence r / Hq and has
  // max(1, ceil(ceil(kv_len/16) / chunk_units)) parts; rows with one part were
  // written by the decode kernel and are skipped.
  const int32_t* kv_lens;
  int Hq, chunk_units;
  int kv_cap;                  // keys beyond this are not read (0: no cap)
  // When set, row r = b * Hq + h writes output row seq_start[b] * Hq + h (the
  // decode rows of a ragged batch).
  const int32_t* seq_start;
  // Stream-K decode (stream_start set): the parts of row r come from the CTAs
  // whose shares its stream spans (see StreamKArgs); a stream without keys is
  // written here (out = 0, lse = sink).
  const int* stream_start;
  const int* shares;
  int group, n_groups;
  const float* sinks;
};

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);

// ------------------------------------------------------------- fp32 path
struct SimtArgs {
  const float* q;              // [total_q, Hq, D]
  const float* k_cache;        // [num_pages, page_size, Hkv, D]
  const float* v_cache;
  const int32_t* cu_seqlens_q; // [B+1] or null (decode: one query per sequence)
  const int32_t* kv_lens;
  const int32_t* block_table;
  const float* sinks;
  float* out;                  // [total_q, Hq, D] (num_splits == 1)
  float* lse;                  // or null
  float* o_part;               // [rows, num_splits, D]   (num_splits > 1)
  float* lse_part;
  int32_t* err_flag;
  int B, total_q, Hq, Hkv, group;
  int bt_stride, page_size, num_pages;
  float scale_log2;
  int causal;
  int num_splits;
};

cudaError_t launch_simt_fp32(const SimtArgs& a, cudaStream_t stream);

// ------------------------------------------------------------- bf16 prefill
struct PrefillArgs {
  const int32_t* cu_seqlens_q;
  const int32_t* kv_lens;
  const int32_t* block_table;
  const float* sinks;
  void* out;                   // bf16 [total_q, Hq, 64]
  float* lse;                  // [total_q, Hq] or null
  int32_t* err_flag;
  int B, total_q, max_q_len, Hq, Hkv, group;
  int bt_stride, page_size, num_pages;
  float scale_log2;
  int causal;
  uint64_t wait_limit_ns;      // limit of each pipeline wait (drains keep kWaitLimitNs)
  unsigned long long* tile_ctr;  // work-tile claim counter (workspace), zeroed before launch
};

// What the mixed kernel adds (attn_sink_mixed): sequences [0, num_decode) hold
// one query each and run as split-KV decode items instead of query tiles.
// (A separate kernel parameter: growing PrefillArgs measurably changed the
// register allocation, and the speed, of the plain prefill kernel.)
struct MixedArgs {
  int num_decode;
  const void* q;               // bf16 [total_q, Hq, 64]: the decode rows' queries
  unsigned long long* dec_ctr; // decode-item claim counter (workspace), zeroed before launch
  int dec_chunk_units;         // 16-key units per decode item
  float* o_part;               // fp32 [num_decode*Hq, s_stride, 64] decode partials
  float* lse_part;             // fp32 [num_decode*Hq, s_stride]
  int s_stride;                // partial slots per decode row (<= 1: every decode row is unsplit)
};

// Bytes of workspace the bf16 prefill uses (its work-tile claim counter); the
// mixed kernel keeps its decode-item counter in the same block.
constexpr size_t kPrefillWorkspaceBytes = 256;
// Keys per decode item of a mixed batch: 1024 keys of 8 KV heads (2 MB of K/V).
constexpr int kMixedChunkUnits = 64;
constexpr int kMixedBoxHeads = 8;       // KV heads per decode-item TMA box
// The mixed kernel keeps sequence lengths and sinks in shared memory.
constexpr int kMixedMaxSeqs = 1024, kMixedMaxHeads = 256;

cudaError_t launch_prefill_bf16(const PrefillArgs& a, const CUtensorMap& q_map,
                                const CUtensorMap& k_map, const CUtensorMap& v_map,
                                cudaStream_t stream);

// The mixed kernel: the prefill kernel with decode items; k8_map / v8_map view
// the caches as 4-D tensors with boxes of 16 keys x 8 KV heads.
cudaError_t launch_mixed_bf16(const PrefillArgs& a, const MixedArgs& mx, const CUtensorMap& q_map,
                              const CUtensorMap& k_map, const CUtensorMap& v_map,
                              const CUtensorMap& k8_map, const CUtensorMap& v8_map,
                              cudaStream_t stream);

}  // namespace attn_sink
