/*
 * attn_sink.h -- C ABI of the GB300 (sm_103a) library for grouped-query
 * attention with a learned per-head sink logit.
 *
 * The operation ("GPT-OSS pada Hari ke-0", section "Atensi Sink", and the model
 * summary "Atensi: GQA dengan Sink Atensi"): every query head h owns a sink
 * logit sink[h] that joins the softmax as one extra column next to the scaled
 * query-key products,
 *     z   = [ sink[h], scale * q . k_j  for every visible key j ],
 *     out = sum_j softmax(z)[j] * v_j      (the sink column carries no value),
 *     lse = ln( e^sink[h] + sum_j e^{scale q.k_j} ).
 * The sink is a logit in the same units as scale*q.k (it is not scaled);
 * sink = -inf gives ordinary attention.  The same section says that when the
 * key sequence is split into chunks processed in parallel, the sink may be
 * counted only in the first chunk; attn_sink_decode follows that rule and
 * attn_sink_merge combines the chunks.
 *
 * Conventions shared by every call
 *  - Pointers marked "device" are CUDA device addresses; "host" are host
 *    addresses.  The caller owns every buffer.  The library never allocates,
 *    frees, synchronises, or reads device memory back to the host, so every
 *    call can be enqueued on a stream without a host round trip.
 *  - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - Layouts (row-major, innermost last):
 *      q            [total_q, Hq, D]                 ragged by cu_seqlens_q
 *      k_cache/v_cache [num_pages, page_size, Hkv, D]  paged cache
 *      block_table  [B, block_table_stride] int32     logical -> physical page
 *      sinks        [Hq] fp32 (may be -INFINITY; +inf/NaN are undefined)
 *    Query head h reads KV head h / (Hq / Hkv).
 *  - Query i (0-based) of a sequence with q_len queries and kv_len keys sits
 *    at absolute position kv_len - q_len + i; with causal masking it sees keys
 *    0..that position (bottom-right alignment: the queries are the last q_len
 *    tokens of the sequence).  Keys at positions >= kv_len are never read.
 *  - Supported shapes: D = 64; Hq % Hkv == 0 with group size Hq/Hkv a power
 *    of two <= 16; page_size a multiple of 16 and <= 256 (bf16) or any
 *    positive value (fp32).  Other shapes return ATTN_SINK_ERR_UNSUPPORTED.
 *  - q, k_cache, v_cache and out must be 16-byte aligned.
 *  - err_flag (device int32, may be NULL): the kernels OR bits into it and
 *    never trap.  ATTN_SINK_FLAG_BAD_PAGE: a block_table entry outside
 *    [0, num_pages) was met; that page's keys were skipped.
 *    ATTN_SINK_FLAG_TIMEOUT: an internal pipeline wait exceeded its time
 *    limit; the affected outputs are undefined.  The caller clears the flag.
 *  - Errors found on the host return a status before anything is enqueued;
 *    a failed launch returns ATTN_SINK_ERR_CUDA.
 */
#ifndef ATTN_SINK_H
#define ATTN_SINK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_SINK_API __attribute__((visibility("default")))
#else
#define ATTN_SINK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_SINK_OK = 0,
    ATTN_SINK_ERR_INVALID_ARG = 1,
    ATTN_SINK_ERR_UNSUPPORTED = 2,
    ATTN_SINK_ERR_WORKSPACE = 3,
    ATTN_SINK_ERR_CUDA = 4
} attn_sink_status;

typedef enum {
    ATTN_SINK_BF16 = 0, /* q/k/v/out bf16, fp32 accumulation, tensor cores */
    ATTN_SINK_FP32 = 1  /* q/k/v/out fp32, fp32 arithmetic throughout     */
} attn_sink_dtype;

#define ATTN_SINK_FLAG_BAD_PAGE 1
/* num_splits value of attn_sink_decode for the persistent split. */
#define ATTN_SINK_SPLIT_PERSISTENT (-1)
#define ATTN_SINK_FLAG_TIMEOUT 2

/*
 * Causal (or full) ragged prefill over a paged KV cache.
 * ("GPT-OSS pada Hari ke-0", section "Atensi Sink": the prefill kernel
 * template gains the sink parameter.)
 *
 *  q            device [total_q, Hq, D] dtype; sequence b owns rows
 *               cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1.
 *  k_cache, v_cache device [num_pages, page_size, Hkv, D] dtype.
 *  cu_seqlens_q device int32 [B+1], non-decreasing, cu_seqlens_q[0] = 0,
 *               cu_seqlens_q[B] = total_q.
 *  kv_lens      device int32 [B]: keys of sequence b, new tokens included.
 *               Causal rows are bottom-right aligned: row i of a sequence sits
 *               at position kv_len - q_len + i; when kv_len < q_len the rows
 *               before position 0 see no key (out = 0, lse = the sink).
 *  block_table  device int32 [B, block_table_stride]; entries for pages at or
 *               beyond ceil(kv_len / page_size) are never read.
 *  sinks        device fp32 [Hq].
 *  out          device [total_q, Hq, D] dtype (written).
 *  lse          device fp32 [total_q, Hq] natural-log LSE including the sink,
 *               or NULL.
 *  max_q_len    host upper bound of any sequence's q_len (sizes the grid).
 *  scale        softmax scale applied to q.k (typically 1/sqrt(D)).
 *  causal       1 = causal (bottom-right aligned), 0 = every key visible.
 *  workspace    device scratch of at least attn_sink_prefill_workspace_size()
 *               bytes, 256-byte aligned (bf16: required, ATTN_SINK_ERR_WORKSPACE
 *               otherwise; fp32: unused, may be NULL).  It holds the counter
 *               from which the kernel's CTAs claim work tiles at run time
 *               ("Embedding Cepat di GPU", section "Manajemen Grafik CUDA":
 *               per-batch scheduling state lives on the device, so the launch
 *               depends only on host integers).  The call zeroes it on the
 *               stream before the kernel (a memset node under stream capture);
 *               no contents need to be preserved.  Calls that overlap on the
 *               GPU need separate workspaces.
 */
ATTN_SINK_API attn_sink_status attn_sink_prefill(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                   const int32_t* block_table, int32_t block_table_stride,
                                   const float* sinks, void* out, float* lse, int32_t B,
                                   int32_t total_q, int32_t max_q_len, int32_t Hq, int32_t Hkv,
                                   int32_t D, int32_t page_size, int32_t num_pages, float scale,
                                   int32_t causal, attn_sink_dtype dtype, int32_t* err_flag,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes attn_sink_prefill needs for these arguments (0 when the
 * call has nothing to do).  Pure host function. */
ATTN_SINK_API size_t attn_sink_prefill_workspace_size(int32_t B, int32_t Hq, int32_t D,
                                                      int32_t max_q_len);

/*
 * A mixed batch in one launch: decode rows and prefill (or verify) segments
 * of one ragged batch over one page pool.  "Accelerating Sonar through
 * speculation", section "Inferensi dengan Speculative Decoding", puts
 * sequences at different stages into one batch; "GPT-OSS pada Hari ke-0",
 * section "Atensi Sink", gives the attention they all compute.
 *
 * Sequences [0, num_decode) are decode rows: each holds exactly one query
 * (cu_seqlens_q[b+1] - cu_seqlens_q[b] = 1; a sequence with more rows gets
 * only its first row written), at position kv_len - 1, which sees every key.
 * They run as split-KV decode work (chunks of 1024 keys x 8 KV heads, combined
 * by the LSE merge, the sink in the first chunk only) on SMs of their own,
 * while the other SMs run the query tiles of sequences [num_decode, B) as
 * attn_sink_prefill does; one persistent launch claims both kinds of work
 * from two device-side queues, plus the merge.  Results equal
 * attn_sink_prefill over the whole batch (which would run each decode row as
 * a query tile of its own) up to fp32 rounding.
 *
 *  Every argument but the ones below is that of attn_sink_prefill; max_q_len
 *  bounds the q_len of sequences [num_decode, B).
 *  num_decode   host, 0 <= num_decode <= B.
 *  workspace    device scratch of at least attn_sink_mixed_workspace_size()
 *               bytes, 256-byte aligned (bf16: required; fp32: unused).  It
 *               holds the two claim counters (zeroed on the stream before the
 *               kernel) and the decode rows' fp32 partial states; no contents
 *               need to be preserved.  Calls that overlap on the GPU need
 *               separate workspaces.
 * Supported: bf16 with B <= 1024 and Hq <= 256 (else ATTN_SINK_ERR_UNSUPPORTED);
 * fp32 runs the whole batch on the fp32 path.
 */
ATTN_SINK_API attn_sink_status attn_sink_mixed(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                 const int32_t* block_table, int32_t block_table_stride,
                                 const float* sinks, void* out, float* lse, int32_t B,
                                 int32_t num_decode, int32_t total_q, int32_t max_q_len,
                                 int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                                 int32_t num_pages, float scale, int32_t causal,
                                 attn_sink_dtype dtype, int32_t* err_flag, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Workspace bytes attn_sink_mixed needs: the counters plus num_decode * Hq
 * rows of partial states, as many per row as the table row (block_table_stride
 * * page_size keys) holds 1024-key chunks.  Pure host function. */
ATTN_SINK_API size_t attn_sink_mixed_workspace_size(int32_t num_decode, int32_t Hq, int32_t Hkv,
                                                    int32_t D, int32_t block_table_stride,
                                                    int32_t page_size);

/*
 * Paged-KV decode, one query token per sequence, optionally split along the
 * key sequence ("GPT-OSS pada Hari ke-0", section "Atensi Sink": attention is
 * parallelised over heads and along the KV length, and the sink is counted in
 * the first chunk only).
 *
 *  q            device [B, Hq, D] dtype (the query of each sequence sits at
 *               position kv_len - 1 and sees every key 0..kv_len-1).
 *  kv_lens      device int32 [B] (0 allowed: out = 0, lse = sink).
 *  out          device [B, Hq, D] dtype; lse device fp32 [B, Hq] or NULL.
 *  num_splits   0: the library picks a chunk length in keys from B, Hkv,
 *               block_table_stride and the SM count (one CTA per chunk, the
 *               hardware hands the CTAs out); 1: no split; S > 1: chunk c of S
 *               covers pages [floor(c*P/S), floor((c+1)*P/S)) with
 *               P = ceil(kv_len/page_size), S <= 256;
 *               ATTN_SINK_SPLIT_PERSISTENT (-1): persistent CTAs (three per
 *               SM) each take an equal share of all sequences' keys laid end
 *               to end, split at sequence boundaries; the shares come from
 *               prefix sums of kv_lens computed on the device ("Accelerating
 *               Sonar through speculation", section "Inferensi dengan
 *               Speculative Decoding": the per-batch planning the pages do on
 *               the CPU happens on the device).  Used when B * ceil(Hkv/4) <=
 *               2048, otherwise the same as 0.  bf16 only (fp32: as 0).
 *  workspace    device scratch of at least attn_sink_decode_workspace_size()
 *               bytes, 256-byte aligned (may be NULL when that size is 0).
 *               Holds fp32 partial states between the split kernel and the
 *               merge; no contents need to be preserved or initialised.
 * The result does not depend on num_splits beyond fp32 rounding.
 */
ATTN_SINK_API attn_sink_status attn_sink_decode(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* kv_lens, const int32_t* block_table,
                                  int32_t block_table_stride, const float* sinks, void* out,
                                  float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                  int32_t page_size, int32_t num_pages, float scale,
                                  int32_t num_splits, attn_sink_dtype dtype, int32_t* err_flag,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * One decode step that first appends the step's key and value.  "Accelerating
 * Sonar through speculation", section "Inferensi dengan Speculative Decoding":
 * before a step runs, pages in the KV cache are allocated for each sequence's
 * next token.  For every sequence b with kv_lens[b] >= 1, k_new[b] and v_new[b]
 * are written into the cache slot of position kv_lens[b] - 1 (page
 * block_table[b, (kv_lens[b]-1) / page_size], row (kv_lens[b]-1) % page_size,
 * every KV head), then attention runs over keys 0..kv_lens[b]-1 exactly as
 * attn_sink_decode does.  The result equals writing the slot and calling
 * attn_sink_decode; in bf16 the write happens inside the decode launch.
 *
 *  k_new, v_new device [B, Hkv, D] dtype, 16-byte aligned (INVALID_ARG if NULL).
 *  k_cache, v_cache are written (only the B appended slots).
 *  A slot whose page index is outside [0, num_pages), or beyond the table row,
 *  is not written and sets *err_flag |= ATTN_SINK_FLAG_BAD_PAGE.
 * Every other argument, the workspace (attn_sink_decode_workspace_size) and
 * the errors are those of attn_sink_decode.
 */
ATTN_SINK_API attn_sink_status attn_sink_decode_append(const void* q, const void* k_new, const void* v_new,
                                         void* k_cache, void* v_cache, const int32_t* kv_lens,
                                         const int32_t* block_table, int32_t block_table_stride,
                                         const float* sinks, void* out, float* lse, int32_t B,
                                         int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
                                         int32_t num_pages, float scale, int32_t num_splits,
                                         attn_sink_dtype dtype, int32_t* err_flag, void* workspace,
                                         size_t workspace_bytes, void* stream);

/* Workspace bytes attn_sink_decode needs for these arguments (0 when it needs
 * none).  Host function; it reads no device memory.  With num_splits = 0 the
 * chunk length, and so the number of partial states per row, depends on Hkv,
 * the table row length (block_table_stride * page_size keys) and the current
 * device's SM count, so ask with the device current that the call will run
 * on (with no device, a 152-SM GB300 is assumed). */
ATTN_SINK_API size_t attn_sink_decode_workspace_size(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                       int32_t block_table_stride, int32_t page_size,
                                       int32_t num_splits);

/*
 * Log-sum-exp merge of S partial attention states per row.  For row r:
 *     L = ln sum_c e^{lse_parts[r,c]},  out[r] = sum_c e^{lse_parts[r,c] - L} o_parts[r,c].
 * It adds no sink: the sink lives inside whichever partial counted it (the
 * first chunk, per "GPT-OSS pada Hari ke-0", section "Atensi Sink").  Rows
 * whose partials are all -inf give out = 0 and L = -inf.
 *
 *  o_parts   device fp32 [rows, S, D], each partial normalised by its own sum.
 *  lse_parts device fp32 [rows, S] natural-log LSE of each partial.
 *  out       device [rows, D] dtype; lse_out device fp32 [rows] or NULL.
 */
ATTN_SINK_API attn_sink_status attn_sink_merge(const float* o_parts, const float* lse_parts, int32_t rows,
                                 int32_t S, int32_t D, void* out, float* lse_out,
                                 attn_sink_dtype dtype, void* stream);

/*
 * attn_sink_decode without a workspace argument, for callers that cannot
 * allocate device memory: for example a host whose allocator owns all device
 * memory and forbids libraries from calling cudaMalloc, or a latency-critical
 * path that cannot afford cudaMalloc's implicit synchronisation.  (The pages
 * describing the method have no counterpart to this; it is a library
 * convenience.)
 *
 * Arguments, layouts and results are those of attn_sink_decode.  The split-KV
 * partial states live in one library-owned static device array of
 * ATTN_SINK_STATIC_SCRATCH_BYTES bytes, which every GPU that loads this part
 * of the library holds until the process exits.  The caller still passes
 * inputs and outputs; nothing is allocated per call.
 *  - A call whose partials need more than ATTN_SINK_STATIC_SCRATCH_BYTES
 *    (attn_sink_decode_workspace_size reports the need) returns
 *    ATTN_SINK_ERR_WORKSPACE before enqueueing anything.
 *  - Arguments are checked first, exactly as attn_sink_decode checks them, so
 *    a bad call gets the same status from both entry points.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress with that device current), and looks it up again
 *    when the device's context has changed (after cudaDeviceReset); make that
 *    first call, and the first after a reset, before any stream capture on
 *    the device.
 *  - All calls on a device share the array, which keeps the previous call's
 *    contents.  Nothing in it needs clearing: every partial the merge reads is
 *    written earlier in the same call.  Calls that overlap on the GPU (other
 *    streams, or concurrent host threads) race on the array and must be
 *    serialised by the caller.
 */
#define ATTN_SINK_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
ATTN_SINK_API attn_sink_status attn_sink_decode_static_scratch(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_lens,
    const int32_t* block_table, int32_t block_table_stride, const float* sinks, void* out,
    float* lse, int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t page_size,
    int32_t num_pages, float scale, int32_t num_splits, attn_sink_dtype dtype, int32_t* err_flag,
    void* stream);

/* Static description of a status code. */
ATTN_SINK_API const char* attn_sink_status_string(attn_sink_status status);

/*
 * Test hook for the failure path.  Every pipeline wait inside the kernels
 * (on a barrier that a copy, an MMA or another warp completes) gives up after
 * a time limit: the CTA then sets ATTN_SINK_FLAG_TIMEOUT in err_flag, stops
 * its pipeline, lets the copies it issued land (those drains always allow
 * 1 s) and returns, so the CUDA context stays usable; that call's outputs are
 * undefined.  The limit is 1 s.  This sets it, in nanoseconds, for calls
 * enqueued afterwards by any thread of the process (0 restores 1 s), and
 * returns the previous value.  A tiny limit makes a correct call time out,
 * which is how the timeout path is tested without a fault.
 */
ATTN_SINK_API uint64_t attn_sink_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_SINK_H */
