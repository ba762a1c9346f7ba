// Causal ragged prefill for bf16 sink attention on sm_103a: tcgen05 tensor
// cores with TMEM accumulators, operands staged by TMA, persistent CTAs.
//
// "GPT-OSS pada Hari ke-0", section "Atensi Sink": the prefill kernel gains the
// sink parameter; the online softmax starts its running maximum at the head's
// sink value with running sum 1.  A work tile scans every key its query rows
// see, so every row starts from its sink.
//
// Work tile: sequence b, KV head g and a block of 256 query rows = two Q tiles
// of 128 rows.  A Q tile packs 128/G consecutive query tokens x the G query
// heads of KV group g (GQA packing), so each K/V tile is read once per 2*128/G
// tokens of the whole group.  The grid has one CTA per SM.  Work tiles form a
// list ordered longest rows first (the last query block of every sequence,
// then the one before, ...).  CTAs claim tiles from that list at run time
// through a counter in the caller's workspace, so a CTA that drew short tiles
// takes more of them (greedy longest-first assignment).  The Q/K producer warp
// claims each tile, decodes it once and hands it to the other roles through a
// small ring in shared memory; the softmax warps take the next tile from the
// ring before writing the current tile's output.
//
// Warp roles (384 threads):
//   warps 0-3  softmax for Q tile 0, warps 4-7 softmax for Q tile 1: one
//              thread per row; S comes out of TMEM with tcgen05.ld.red, which
//              also returns the row's maximum, exp2 and the sum run in
//              registers, P (bf16) goes back into TMEM in its own columns and
//              feeds P*V as the A operand.  The two warpgroups take turns in
//              the exponential loop.
//   warp 8     tile claims, then TMA producer of Q and K: per work tile the two
//              Q tiles (double-buffered), then per 128-key tile eight 16-row
//              page slices of K into a 4-stage ring.  It runs ahead across work
//              tiles and reads the block-table entries one tile ahead.
//   warps 9-10 one MMA-issuing warp per Q tile (warp 9 also owns TMEM).
//   warp 11    TMA producer of V, in step with warp 8.  A 2 KB page slice
//              occupies the SM's TMA unit for about 90 clocks, so the sixteen
//              slices of a tile take as long as the tile's MMAs; two issuing
//              warps on different SMSPs keep the unit fed while each one
//              computes addresses and waits on barriers.
// Registers: setmaxnreg gives warps 8-11 72 per thread and the two softmax
// warpgroups 216 (the launch allocation is 168 for all 384 threads).
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,320), O1 [320,384),
// P0 [384,448), P1 [448,512) (P as packed bf16 pairs).
//
// Per 128-key tile and Q tile: S = Q K^T is 4 MMAs of 128x128x16 (K-major A
// and B), O += P V is 8 MMAs of 128x64x16 (A in TMEM, V MN-major).  A
// warpgroup hands S back (s_free) as soon as it has loaded it, so S(j+1) is
// computed while the softmax of tile j runs.  Every barrier phase is counted
// across work tiles, so the pipeline never drains between them.
#include "decode_unit.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace attn_sink {
namespace {

constexpr int kRows = 128;
constexpr int kQTiles = 2;
constexpr int kKeys = 128;
constexpr int kStages = 4;
constexpr int kQBufs = 2;
constexpr int kUnitsPerTile = kKeys / kUnitTokens;            // 8
constexpr int kUnitBytes = kUnitTokens * kHeadDim * 2;       // 2 KB
constexpr int kTileBytes = kRows * kHeadDim * 2;             // 16 KB
constexpr int kStageBytes = 2 * kTileBytes;                  // K then V
constexpr int kQBufBytes = kQTiles * kTileBytes;
constexpr int kSoftmaxWarps = 4 * kQTiles;
// The Q/K producer warp, one MMA-issuing warp per Q tile (the first of them
// also allocates TMEM), then the V producer warp.
constexpr int kProducerWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1;
constexpr int kProducerWarpV = kMmaWarp + kQTiles;
constexpr int kThreads = 32 * (kProducerWarpV + 1);
// Registers per thread after the role split: the producer/MMA warpgroup gives
// registers back, the two softmax warpgroups take them.  setmaxnreg.inc draws
// on the block's launch allocation (kThreads x kLaunchRegs), so the split must
// fit in it, or the increase would wait for ever.
constexpr int kLaunchRegs = 168;  // what 65536 / kThreads allows, rounded down to 8
constexpr int kSupportRegs = 72, kSoftmaxRegs = 216;
static_assert(kThreads * kLaunchRegs <= 65536, "launch allocation");
static_assert(128 * kSupportRegs + 256 * kSoftmaxRegs <= kThreads * kLaunchRegs, "register split");
static_assert(kSupportRegs % 8 == 0 && kSoftmaxRegs % 8 == 0, "setmaxnreg granularity");
static_assert(kProducerWarp % 4 == 0 && kProducerWarpV == kProducerWarp + 3, "one support warpgroup");
constexpr uint32_t kTmemCols = 256 * kQTiles;  // S, O and P of every Q tile
__device__ __forceinline__ uint32_t col_s(int q) { return static_cast<uint32_t>(q) * 128u; }
__device__ __forceinline__ uint32_t col_o(int q) { return 128u * kQTiles + static_cast<uint32_t>(q) * 64u; }
__device__ __forceinline__ uint32_t col_p(int q) { return 192u * kQTiles + static_cast<uint32_t>(q) * 64u; }
constexpr int kOffQ = 0;
constexpr int kOffKV = kQBufs * kQBufBytes;
constexpr int kOffBar = kOffKV + kStages * kStageBytes;
// Per-sequence lengths and per-head sinks are copied to shared memory when
// they fit, so that decoding a work tile costs no global-memory round trip.
constexpr int kMetaSeqs = kMixedMaxSeqs, kMetaHeads = kMixedMaxHeads;
constexpr int kBarBytes = 512;
constexpr int kOffMeta = kOffBar + kBarBytes;
constexpr int kMetaBytes = ((2 * kMetaSeqs + 1 + kMetaHeads) * 4 + 255) / 256 * 256;
constexpr int kOffSort = kOffMeta + kMetaBytes;
constexpr int kSortBytes = 2048 * 4;        // the sorted query blocks
constexpr int kOffSched = kOffSort + kSortBytes;
constexpr int kSchedBytes = 256;            // SchedInfo
// Mixed batches: first decode item of every decode sequence (prefix sums).
constexpr int kOffDecItems = kOffSched + kSchedBytes;
constexpr int kDecItemsBytes = ((kMetaSeqs + 1) * 4 + 255) / 256 * 256;
constexpr int kSmemBytes = kOffDecItems + kDecItemsBytes + 1024;
// Decode items: KV heads per item (one consumer warp each, one TMA box).
constexpr int kDecHeads = kMixedBoxHeads;
constexpr int kDecHeadBytes = kUnitTokens * kHeadDim * 2;   // 2 KB: 16 keys of one head
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 64, false, true);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Claimed work tiles in flight between the claiming warp and the other roles.
constexpr int kTileRing = 4;
// Warps that read every claimed tile: the V producer, the MMA warps and the
// softmax warps.
constexpr int kTileReaders = 1 + kQTiles + kSoftmaxWarps;

// A work tile: its sequence b, KV head g, query rows and the key tiles they
// see, derived from its linear index.
struct WorkTile {
  int b, g, q_start, q_len, tok0, kv_raw, kv_len, n_kv;
  int first_pos;  // absolute position of the tile's first query (fits: kv_len, q_len < 2^31)
};

struct alignas(8) Bars {
  uint64_t q_full[kQBufs];
  uint64_t q_empty[kQBufs];   // both Q tiles' MMAs of the buffer's work tile are done
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[kQTiles];   // S is in TMEM, and s_uok holds its stage's unit mask
  uint64_t s_free[kQTiles];   // the warpgroup has loaded S; S may be overwritten
  uint64_t p_ready[kQTiles];  // P is in TMEM (and O rescaled)
  uint64_t pv_done[kQTiles];  // P*V has completed: P may be overwritten, O is current
  uint64_t o_free[kQTiles];   // the warpgroup has read the work tile's final O
  uint64_t exp_turn[kQTiles]; // warpgroup q may run its exponentials (token passed between them)
  uint64_t mma_done;
  uint64_t tile_full[kTileRing];   // the slot holds the next claimed tile
  uint64_t tile_empty[kTileRing];  // every reader has taken the slot's tile
  long long tile_slot[kTileRing];  // claimed tile index, or -1: no tile left
  WorkTile tile_w[kTileRing];      // a claimed query tile, decoded once by the claiming warp
  uint32_t unit_ok[kStages];  // bit u: 16-key unit u of the stage's tile was loaded
  uint32_t s_uok[kQTiles];    // unit_ok of the stage the current S was computed from
  uint32_t tmem_base;
  int abort_word;
};
static_assert(sizeof(Bars) <= kBarBytes, "barrier block");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

// Where the per-sequence lengths and the sinks are read from.
struct Meta {
  const int32_t* cu_seqlens_q;
  const int32_t* kv_lens;
  const float* sinks;
};

// Query block r of sequence b (r = 0 is the last block): its first query
// token and the number of 128-key tiles its rows see.
__device__ __forceinline__ int block_key_tiles(const PrefillArgs& a, int q_len, int kv_len, int n_blocks,
                                               int r, int tok_per_cta, int& tok0) {
  tok0 = (n_blocks - 1 - r) * tok_per_cta;
  const long long last_pos =
      static_cast<long long>(kv_len) - q_len + min(tok0 + tok_per_cta, q_len) - 1;
  long long key_end = kv_len;
  if (a.causal && key_end > last_pos + 1) key_end = last_pos + 1;
  if (key_end < 0) key_end = 0;
  return static_cast<int>((key_end + kKeys - 1) / kKeys);
}

// Work tile t of the row-major list: t = r * (B * Hkv) + b * Hkv + g.
// Returns false when sequence b has no query block r.
template <bool kMixed = false>
__device__ __forceinline__ bool decode_tile(const PrefillArgs& a, const Meta& m, long long t,
                                            int tok_per_cta, WorkTile& w, int num_decode = 0) {
  const long long heads = static_cast<long long>(a.B) * a.Hkv;
  const int r = static_cast<int>(t / heads);  // 0: last query block of each sequence
  const int rem = static_cast<int>(t % heads);
  w.b = rem / a.Hkv;
  w.g = rem % a.Hkv;
  if constexpr (kMixed) {
    if (w.b < num_decode) return false;  // a mixed batch's decode rows run as decode items
  }
  w.q_start = m.cu_seqlens_q[w.b];
  w.q_len = m.cu_seqlens_q[w.b + 1] - w.q_start;
  const int n_blocks = w.q_len > 0 ? (w.q_len + tok_per_cta - 1) / tok_per_cta : 0;
  if (r >= n_blocks) return false;
  w.kv_raw = max(0, m.kv_lens[w.b]);
  w.kv_len = min(w.kv_raw, a.bt_stride * a.page_size);  // keys beyond the table row are not read
  w.n_kv = block_key_tiles(a, w.q_len, w.kv_len, n_blocks, r, tok_per_cta, w.tok0);
  w.first_pos = w.kv_len - w.q_len + w.tok0;
  return true;
}

// The claim order.  Query blocks (b, r) sorted by the key tiles their rows
// see, most first, so that dynamic claims assign the longest work first
// (greedy longest-processing-time).  A sort key packs (2047 - cost, r, b) into
// 21 + 11 + 10 bits; sorting the keys ascending gives cost descending, then
// the row-major order.  Costs above 2047 key tiles compare equal (their order
// is then row-major), which leaves the list valid.
constexpr int kSortMax = 2048;  // query blocks the sorted list holds
constexpr int kAllAlike = -2;   // build_sorted_blocks: every sequence alike
// Batches of alike sequences claim their tiles in groups of this many
// (sequence, KV head) pairs.  On the 8 x 4096 prefill (64 pairs, 67 MB of K/V)
// groups of 32 measured 1.165 ms, 16 1.171, 8 1.181, and all 64 at once 1.175
// (there DRAM reads are 466 MB against 336 with groups: K/V re-read after the
// streamed Q and output evict it); one pair at a time, 1.177 (every CTA of a
// pair reading the same K/V lines at once).
constexpr int kClaimGroup = 32;
__device__ __forceinline__ uint32_t block_sort_key(int cost, int r, int b) {
  return (static_cast<uint32_t>(2047 - min(cost, 2047)) << 21) | (static_cast<uint32_t>(r) << 10) |
         static_cast<uint32_t>(b);
}

// Scheduling facts every CTA derives identically at launch.
struct SchedInfo {
  int sort_count;                 // query blocks placed in the sorted list
  int n_dec_items;                // decode items of a mixed batch
  int dec_first_ctas;             // CTAs that claim decode items before query tiles
  int pad;
  unsigned long long key_tiles;   // query-block key tiles (x Hkv: work of the query tiles)
  unsigned long long dec_units;   // decode units (16 keys x Hkv heads each)
};

// Pads keys[n..) to a power of two and sorts them ascending (bitonic; all
// threads of the CTA).
__device__ __forceinline__ void sort_keys_ascending(uint32_t* keys, int n) {
  int pow2 = 1;
  while (pow2 < n) pow2 <<= 1;
  for (int i = n + threadIdx.x; i < pow2; i += blockDim.x) keys[i] = 0xFFFFFFFFu;
  __syncthreads();
  // bitonic sort, ascending
  for (int k = 2; k <= pow2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < pow2; i += blockDim.x) {
        const int l = i ^ j;
        if (l > i) {
          const uint32_t x = keys[i], y = keys[l];
          if (((i & k) == 0) == (x > y)) {
            keys[i] = y;
            keys[l] = x;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Builds the sorted list in shared memory (all threads of the CTA).  Every
// CTA builds the same list: the keys are distinct, so their sorted order does
// not depend on where each thread placed them.  Returns the number of query
// blocks; kAllAlike when every sequence has the same query and key lengths
// (claims then walk groups of (sequence, KV head) pairs, longest blocks first
// within each group, so a group's K/V stays in L2 while its tiles run, and the
// last claims are short tiles); -1 when the list is not used (more than
// kSortMax blocks, or the metadata is not in shared memory).
__device__ __forceinline__ int build_sorted_blocks(const PrefillArgs& a, const Meta& m, bool meta_in_smem,
                                   int tok_per_cta, uint32_t* keys, int* counter) {
  if (!meta_in_smem || a.B > 1024) return -1;
  if (threadIdx.x == 0) *counter = 0;
  // all sequences alike?
  int differs = 0;
  for (int b = threadIdx.x; b < a.B; b += blockDim.x)
    differs |= (m.cu_seqlens_q[b + 1] - m.cu_seqlens_q[b] != m.cu_seqlens_q[1] - m.cu_seqlens_q[0]) ||
               (m.kv_lens[b] != m.kv_lens[0]);
  if (__syncthreads_or(differs) == 0) return kAllAlike;
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    const int q_len = m.cu_seqlens_q[b + 1] - m.cu_seqlens_q[b];
    const int n_blocks = q_len > 0 ? (q_len + tok_per_cta - 1) / tok_per_cta : 0;
    const int kv_len = min(max(0, m.kv_lens[b]), a.bt_stride * a.page_size);
    for (int r = 0; r < n_blocks; ++r) {
      const int slot = atomicAdd(counter, 1);
      if (slot >= kSortMax) break;
      int tok0;
      keys[slot] = block_sort_key(block_key_tiles(a, q_len, kv_len, n_blocks, r, tok_per_cta, tok0), r, b);
    }
  }
  __syncthreads();
  const int n = *counter;
  if (n > kSortMax) return -1;
  sort_keys_ascending(keys, n);
  return n;
}

// The same for a mixed batch (query tiles of sequences [num_decode, B) only,
// always sorted), also summing the query tiles' key tiles.  The SchedInfo
// fields are zero on entry.
__device__ __forceinline__ int build_sorted_blocks_mixed(const PrefillArgs& a, const MixedArgs& mx,
                                                         const Meta& m, int tok_per_cta, uint32_t* keys,
                                                         SchedInfo* info) {
  unsigned long long tiles = 0;
  for (int b = mx.num_decode + threadIdx.x; b < a.B; b += blockDim.x) {
    const int q_len = m.cu_seqlens_q[b + 1] - m.cu_seqlens_q[b];
    const int n_blocks = q_len > 0 ? (q_len + tok_per_cta - 1) / tok_per_cta : 0;
    const int kv_len = min(max(0, m.kv_lens[b]), a.bt_stride * a.page_size);
    for (int r = 0; r < n_blocks; ++r) {
      int tok0;
      const int cost = block_key_tiles(a, q_len, kv_len, n_blocks, r, tok_per_cta, tok0);
      tiles += static_cast<unsigned long long>(cost);
      const int slot = atomicAdd(&info->sort_count, 1);
      if (slot < kSortMax) keys[slot] = block_sort_key(cost, r, b);
    }
  }
  atomicAdd(&info->key_tiles, tiles);
  __syncthreads();
  const int n = info->sort_count;
  if (n > kSortMax) return -1;
  sort_keys_ascending(keys, n);
  return n;
}

// ---------------------------------------------------------------- decode items
// A mixed batch's decode sequence b (one query at position kv_len - 1, which
// sees every key) runs as decode items: chunk c of kMixedChunkUnits 16-key
// units x a group of kDecHeads KV heads.  Sequence b's items are numbered from
// item_start[b], chunk-major (head group fastest).
struct DecItem {
  int b, hg, c, n_chunks, u0, u1, kv_len;
};

__device__ __forceinline__ int m_kv_raw(const Meta& m, int b) { return max(0, m.kv_lens[b]); }

// Key length of decode sequence b as the kernel reads it, and its chunks.
__device__ __forceinline__ int dec_kv_len(const PrefillArgs& a, const Meta& m, int b) {
  return min(max(0, m.kv_lens[b]), a.bt_stride * a.page_size);
}
__device__ __forceinline__ int dec_chunks(const MixedArgs& mx, int kv_len) {
  const int units = (kv_len + kUnitTokens - 1) / kUnitTokens;
  return max(1, (units + mx.dec_chunk_units - 1) / mx.dec_chunk_units);
}

// Fills item_start[0..num_decode] (all threads of the CTA) and the decode work.
__device__ __forceinline__ void build_decode_items(const PrefillArgs& a, const MixedArgs& mx, const Meta& m,
                                                   int* item_start, SchedInfo* info) {
  const int n_hg = (a.Hkv + kDecHeads - 1) / kDecHeads;
  unsigned long long units = 0;
  for (int b = threadIdx.x; b < mx.num_decode; b += blockDim.x) {
    const int kv = dec_kv_len(a, m, b);
    item_start[b + 1] = dec_chunks(mx, kv) * n_hg;
    units += static_cast<unsigned long long>((kv + kUnitTokens - 1) / kUnitTokens);
  }
  atomicAdd(&info->dec_units, units);
  if (threadIdx.x == 0) item_start[0] = 0;
  __syncthreads();
  // inclusive scan of item_start[1..num_decode] by warp 0: lane l sums a
  // contiguous run, then the runs' totals are scanned across the warp
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (mx.num_decode + 31) / 32;
    const int lo = 1 + lane * per, hi = min(mx.num_decode, lo + per - 1);
    int run = 0;
    for (int i = lo; i <= hi; ++i) run += item_start[i];
    int incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += x;
    }
    int acc = incl - run;
    for (int i = lo; i <= hi; ++i) {
      acc += item_start[i];
      item_start[i] = acc;
    }
    if (lane == 31) info->n_dec_items = incl;
  }
  __syncthreads();
}

// Decode item k: binary search of its sequence in item_start.
__device__ __forceinline__ void decode_item(const PrefillArgs& a, const MixedArgs& mx, const Meta& m,
                                            const int* item_start, int k, DecItem& d) {
  int lo = 0, hi = mx.num_decode - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (item_start[mid] <= k) lo = mid; else hi = mid - 1;
  }
  const int n_hg = (a.Hkv + kDecHeads - 1) / kDecHeads;
  const int within = k - item_start[lo];
  d.b = lo;
  d.hg = within % n_hg;
  d.c = within / n_hg;
  d.kv_len = dec_kv_len(a, m, lo);
  d.n_chunks = dec_chunks(mx, d.kv_len);
  const int units = (d.kv_len + kUnitTokens - 1) / kUnitTokens;
  d.u0 = min(units, d.c * mx.dec_chunk_units);
  d.u1 = min(units, d.u0 + mx.dec_chunk_units);
}

// Claims the next work tile (warp-collective; every lane returns the same
// row-major tile index, or -1 when every tile has been claimed).  With the
// sorted list (n_sorted >= 0) claim k is query block keys[k / Hkv], KV head
// k % Hkv; without it the claims walk the row-major list and pass over the
// indices past a sequence's last block.
template <bool kMixed = false>
__device__ __forceinline__ long long claim_tile(const PrefillArgs& a, const Meta& m, long long n_tiles,
                                                int tok_per_cta, const uint32_t* keys, int n_sorted,
                                                int num_decode = 0) {
  const int lane = threadIdx.x & 31;
  // every sequence alike (never in a mixed batch): n_blocks query blocks each
  const bool alike = !kMixed && n_sorted == kAllAlike;
  const int n_blocks =
      alike ? (m.cu_seqlens_q[1] - m.cu_seqlens_q[0] + tok_per_cta - 1) / tok_per_cta : 1;
  const long long n_claims = n_sorted >= 0 ? static_cast<long long>(n_sorted) * a.Hkv
                             : alike       ? static_cast<long long>(a.B) * a.Hkv * n_blocks
                                           : n_tiles;
  for (;;) {
    unsigned long long c = 0;
    if (lane == 0) c = atomicAdd(a.tile_ctr, 1ull);
    const long long k = static_cast<long long>(__shfl_sync(0xffffffffu, c, 0));
    if (k >= n_claims) return -1;
    if (alike) {
      // Groups of kClaimGroup (sequence, KV head) pairs, one after the other;
      // inside a group the row-major order (every pair's longest block, then
      // the next ...).  A group's K/V stays in L2 while its tiles run.
      const long long pairs = static_cast<long long>(a.B) * a.Hkv;
      const long long span = static_cast<long long>(kClaimGroup) * n_blocks;
      const long long base = (k / span) * kClaimGroup, kin = k % span;
      const long long size = min(static_cast<long long>(kClaimGroup), pairs - base);
      return (kin / size) * pairs + base + kin % size;
    }
    if (n_sorted >= 0) {
      const uint32_t key = keys[k / a.Hkv];
      const int r = static_cast<int>((key >> 10) & 0x7FFu), b = static_cast<int>(key & 0x3FFu);
      return static_cast<long long>(r) * a.B * a.Hkv + static_cast<long long>(b) * a.Hkv + k % a.Hkv;
    }
    WorkTile w;
    if (decode_tile<kMixed>(a, m, k, tok_per_cta, w, num_decode)) return k;
  }
}

// Tile indices handed through the ring: >= 0 a query tile (row-major index),
// -1 no work left, <= -2 decode item -2 - index.
__device__ __forceinline__ bool is_decode_item(long long t) { return t <= -2; }
__device__ __forceinline__ int decode_item_index(long long t) { return static_cast<int>(-2 - t); }

// The claiming warp's view of the two queues of a mixed batch.
struct Claimer {
  bool tiles_done = false, items_done = false;
};

// Next piece of work for this CTA (warp-collective).  CTAs below
// dec_first_ctas take decode items first, the others query tiles first; each
// turns to the other queue when its own runs dry, so HBM-bound decode items
// and tensor-bound query tiles run on different SMs at the same time.
template <bool kMixed>
__device__ __forceinline__ long long claim_work(const PrefillArgs& a, const MixedArgs& mx, const Meta& m,
                                                long long n_tiles, int tok_per_cta, const uint32_t* keys,
                                                int n_sorted, const SchedInfo* info, Claimer& cl) {
  const int lane = threadIdx.x & 31;
  const bool items_first = kMixed && static_cast<int>(blockIdx.x) < info->dec_first_ctas;
  for (int pass = 0; pass < 2; ++pass) {
    const bool items = kMixed && (pass == 0) == items_first;
    if (items) {
      if (cl.items_done) continue;
      unsigned long long c = 0;
      if (lane == 0) c = atomicAdd(mx.dec_ctr, 1ull);
      const long long k = static_cast<long long>(__shfl_sync(0xffffffffu, c, 0));
      if (k < info->n_dec_items) return -2 - k;
      cl.items_done = true;
    } else {
      if (cl.tiles_done) continue;
      const long long t = claim_tile<kMixed>(a, m, n_tiles, tok_per_cta, keys, n_sorted, mx.num_decode);
      if (t >= 0) return t;
      cl.tiles_done = true;
    }
  }
  return -1;
}

// A reader role takes claimed tile number i from the ring (warp-collective),
// and, if w is given, its decoded work tile when it is a query tile.  Returns
// false when the pipeline aborted; t = -1 means no tile is left.
template <bool kPoll>
__device__ __forceinline__ bool take_tile(Bars* bars, int i, long long& t, WorkTile* w,
                                          volatile int* abort_word, const PrefillArgs& a) {
  const int slot = i % kTileRing;
  const bool ready = mbar_wait<kPoll>(&bars->tile_full[slot], (i / kTileRing) & 1, abort_word,
                                      a.err_flag, a.wait_limit_ns);
  if (!__all_sync(0xffffffffu, ready)) return false;
  t = *reinterpret_cast<volatile long long*>(&bars->tile_slot[slot]);
  if (w && t >= 0) *w = bars->tile_w[slot];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&bars->tile_empty[slot]);
  return true;
}

// HBM rate one CTA sustains on decode items (GB/s; measured 47-60 on GB300,
// where the 4-stage ring of one CTA per SM bounds the bytes in flight): the
// mixed kernel sends at most 6.5 TB/s / this many CTAs to decode items first.
constexpr float kDecodeCtaGBs = 60.f;

// kPoll: the waits poll (a test's short wait limit); otherwise they block.
// kMixed: sequences [0, num_decode) run as decode items (attn_sink_mixed).
template <bool kPoll, bool kMixed>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap k_map,
                   const __grid_constant__ CUtensorMap v_map,
                   const __grid_constant__ CUtensorMap k8_map,
                   const __grid_constant__ CUtensorMap v8_map, const PrefillArgs a,
                   const MixedArgs mx, const long long n_tiles) {
  // Arrivals that release a K/V stage: the two P*V commits of a query tile
  // (each issued kKvRelease times in the mixed kernel), or in the mixed kernel
  // the eight consumer warps of a decode item.
  constexpr int kKvRelease = kMixed ? kSoftmaxWarps / kQTiles : 1;
  const int tok_per_tile = kRows / a.group;
  const int tok_per_cta = kQTiles * tok_per_tile;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(base + kOffBar);
  volatile int* abort_word = &bars->abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kQBufs; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], kQTiles);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 2);   // the K and the V producer
      mbar_init(&bars->kv_empty[s], kQTiles * kKvRelease);  // every Q tile's P*V (or decode warp)
    }
    for (int q = 0; q < kQTiles; ++q) {
      mbar_init(&bars->s_full[q], 2);   // the MMA commit and the MMA leader's s_uok arrive
      mbar_init(&bars->s_free[q], 4);   // one arrive per softmax warp
      mbar_init(&bars->p_ready[q], 4);
      mbar_init(&bars->pv_done[q], 1);
      mbar_init(&bars->o_free[q], 4);
      mbar_init(&bars->exp_turn[q], 4);  // one arrive per warp of the other warpgroup
    }
    mbar_init(&bars->mma_done, kQTiles);
    for (int i = 0; i < kTileRing; ++i) {
      mbar_init(&bars->tile_full[i], 1);               // the claiming warp
      mbar_init(&bars->tile_empty[i], kTileReaders);   // one arrive per reader warp
    }
    bars->abort_word = 0;
    if constexpr (kMixed) {
      SchedInfo* si = reinterpret_cast<SchedInfo*>(base + kOffSched);
      si->sort_count = 0;
      si->n_dec_items = 0;
      si->dec_first_ctas = 0;
      si->key_tiles = 0;
      si->dec_units = 0;
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  Meta meta{a.cu_seqlens_q, a.kv_lens, a.sinks};
  if (a.B <= kMetaSeqs && a.Hq <= kMetaHeads) {
    int32_t* cu_s = reinterpret_cast<int32_t*>(base + kOffMeta);
    int32_t* kvl_s = cu_s + kMetaSeqs + 1;
    float* sinks_s = reinterpret_cast<float*>(kvl_s + kMetaSeqs);
    for (int i = threadIdx.x; i <= a.B; i += kThreads) cu_s[i] = a.cu_seqlens_q[i];
    for (int i = threadIdx.x; i < a.B; i += kThreads) kvl_s[i] = a.kv_lens[i];
    for (int i = threadIdx.x; i < a.Hq; i += kThreads) sinks_s[i] = a.sinks[i];
    meta = Meta{cu_s, kvl_s, sinks_s};
  }
  uint32_t* sort_keys = reinterpret_cast<uint32_t*>(base + kOffSort);
  SchedInfo* info = reinterpret_cast<SchedInfo*>(base + kOffSched);
  int* dec_start = reinterpret_cast<int*>(base + kOffDecItems);
  __syncthreads();  // the metadata is in place
  int n_sorted;
  if constexpr (kMixed) {
    n_sorted = build_sorted_blocks_mixed(a, mx, meta, tok_per_cta, sort_keys, info);
    build_decode_items(a, mx, meta, dec_start, info);
    if (threadIdx.x == 0 && info->n_dec_items > 0) {
      // How many CTAs start on decode items: the decode share of the work, at
      // most what saturates HBM (the others start on query tiles).
      const float dec_us = static_cast<float>(info->dec_units) * kUnitTokens * a.Hkv * 256.f / 6.5e6f;
      const float tile_us = static_cast<float>(info->key_tiles) * a.Hkv * 1.15f / gridDim.x;
      int k = static_cast<int>(gridDim.x * dec_us / (dec_us + tile_us) + 0.5f);
      k = min(k, static_cast<int>(6500.f / kDecodeCtaGBs + 0.999f));
      info->dec_first_ctas = info->key_tiles == 0 ? static_cast<int>(gridDim.x) : max(1, k);
    }
  } else {
    n_sorted = build_sorted_blocks(a, meta, a.B <= kMetaSeqs && a.Hq <= kMetaHeads, tok_per_cta,
                                   sort_keys, &info->sort_count);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= kProducerWarp) {
    // Warpgroup 2 (both producers and both MMA warps) runs one setmaxnreg, as
    // the instruction requires of a whole warpgroup.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kSupportRegs));
  if (warp == kProducerWarp || warp == kProducerWarpV) {
    // ---------------------------------------------------------------- TMA
    const bool is_k = warp == kProducerWarp;  // else the V producer
    const CUtensorMap* kv_map = is_k ? &k_map : &v_map;
    const int kv_off = is_k ? 0 : kTileBytes;
    if (lane == 0) {
      if (is_k) tma_prefetch_map(&q_map);
      tma_prefetch_map(kv_map);
      if constexpr (kMixed) tma_prefetch_map(is_k ? &k8_map : &v8_map);
    }
    const uint64_t once = l2_policy_evict_first();   // each Q tile is read by one CTA
    const uint64_t reuse = l2_policy_evict_last();   // K/V tiles serve every later query block
    int qw = 0, kv_it = 0;
    bool ok = true;
    Claimer claimer;
    for (int i = 0; ok; ++i) {
      long long t;
      WorkTile w;
      if (is_k) {
        // Claim the next tile and publish it to the other roles.
        if constexpr (kMixed)
          t = claim_work<kMixed>(a, mx, meta, n_tiles, tok_per_cta, sort_keys, n_sorted, info, claimer);
        else
          t = claim_tile(a, meta, n_tiles, tok_per_cta, sort_keys, n_sorted);
        if (!kMixed && t >= 0)  // a claimed tile always holds query rows
          decode_tile<kMixed>(a, meta, t, tok_per_cta, w, mx.num_decode);
        const int slot = i % kTileRing;
        if (i >= kTileRing) {
          const bool ready = mbar_wait<kPoll>(&bars->tile_empty[slot], ((i / kTileRing) + 1) & 1,
                                              abort_word, a.err_flag, a.wait_limit_ns);
          ok = __all_sync(0xffffffffu, ready);
          if (!ok) break;
        }
        if (lane == 0) {
          if (!kMixed && t >= 0) bars->tile_w[slot] = w;  // (the mixed kernel's readers decode it)
          bars->tile_slot[slot] = t;
          mbar_arrive(&bars->tile_full[slot]);  // release: the slot is written
        }
        __syncwarp();
      } else {
        ok = take_tile<kPoll>(bars, i, t, kMixed ? nullptr : &w, abort_word, a);
        if (!ok) break;
      }
      if constexpr (kMixed) {
      if (t == -1) break;
      if (is_decode_item(t)) {
        // A decode item: per 16-key unit one box of 16 keys x kDecHeads KV
        // heads of K (this warp) or V (the other producer) into the stage.
        DecItem d;
        decode_item(a, mx, meta, dec_start, decode_item_index(t), d);
        const CUtensorMap* map8 = is_k ? &k8_map : &v8_map;
        const int32_t* bt_row = a.block_table + static_cast<long long>(d.b) * a.bt_stride;
        if (is_k && d.c == 0 && lane == 0 && a.err_flag && m_kv_raw(meta, d.b) > d.kv_len)
          atomicOr(a.err_flag, kFlagBadPage);
        const int upp = a.page_size / kUnitTokens;
        // lane l holds the page of unit u0 + 32 * window + l
        auto page_of = [&](int it0) {
          const int u = d.u0 + it0 + lane;
          return u < d.u1 ? bt_row[u / upp] : -1;
        };
        int cur_phys = page_of(0), nxt_phys = page_of(32);
        for (int it = 0; it < d.u1 - d.u0; ++it, ++kv_it) {
          if (it > 0 && (it & 31) == 0) {
            cur_phys = nxt_phys;
            nxt_phys = page_of(it + 32);
          }
          const int st = kv_it % kStages;
          if (kv_it >= kStages) {
            const bool ready = mbar_wait<kPoll>(&bars->kv_empty[st], ((kv_it / kStages) + 1) & 1,
                                                abort_word, a.err_flag, a.wait_limit_ns);
            ok = __all_sync(0xffffffffu, ready);
            if (!ok) break;
          }
          const int phys = __shfl_sync(0xffffffffu, cur_phys, it & 31);
          const int tok = ((d.u0 + it) % upp) * kUnitTokens;
          const bool unit_ok = phys >= 0 && phys < a.num_pages;
          if (lane == 0) {
            if (is_k) {
              bars->unit_ok[st] = unit_ok ? 1u : 0u;  // published by the arrive below
              if (!unit_ok && a.err_flag) atomicOr(a.err_flag, kFlagBadPage);
            }
            mbar_arrive_expect_tx(&bars->kv_full[st], unit_ok ? kDecHeads * kDecHeadBytes : 0);
            if (unit_ok)
              tma_load_4d_hint(base + kOffKV + st * kStageBytes + kv_off, map8, &bars->kv_full[st], 0,
                               tok, d.hg * kDecHeads, phys, once);
          }
          __syncwarp();
        }
        continue;
      }
      } else {
        if (t < 0) break;
      }
      // (The mixed kernel's readers decode the tile themselves: with the
      // decode items' code beside it, the copy measured slower.)
      if constexpr (kMixed) decode_tile<kMixed>(a, meta, t, tok_per_cta, w, mx.num_decode);
      if (is_k && w.kv_len < w.kv_raw && lane == 0 && a.err_flag) atomicOr(a.err_flag, kFlagBadPage);
      if (w.n_kv == 0) continue;
      if (is_k) {
        const int qb = qw % kQBufs;
        if (qw >= kQBufs) {
          const bool ready = mbar_wait<kPoll>(&bars->q_empty[qb], ((qw / kQBufs) + 1) & 1, abort_word, a.err_flag, a.wait_limit_ns);
          ok = __all_sync(0xffffffffu, ready);
          if (!ok) break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->q_full[qb], kQBufBytes);
          for (int q = 0; q < kQTiles; ++q)
            tma_load_3d_hint(base + kOffQ + qb * kQBufBytes + q * kTileBytes, &q_map, &bars->q_full[qb],
                             0, w.g * a.group, w.q_start + w.tok0 + q * tok_per_tile, once);
        }
        ++qw;
      }
      const int32_t* bt_row = a.block_table + static_cast<long long>(w.b) * a.bt_stride;
      // lane u < 8 holds the block-table entry of unit u of a tile (-1 past kv_len)
      auto entry_of = [&](int jj) -> int {
        const int key0 = (jj * kUnitsPerTile + lane) * kUnitTokens;
        return (lane < kUnitsPerTile && jj < w.n_kv && key0 < w.kv_len) ? bt_row[key0 / a.page_size] : -1;
      };
      int next_phys = entry_of(0);
      for (int j = 0; j < w.n_kv; ++j, ++kv_it) {
        const int cur_phys = next_phys;
        next_phys = entry_of(j + 1);
        const int st = kv_it % kStages;
        if (kv_it >= kStages) {
          const bool ready = mbar_wait<kPoll>(&bars->kv_empty[st], ((kv_it / kStages) + 1) & 1, abort_word,
                                       a.err_flag, a.wait_limit_ns);
          ok = __all_sync(0xffffffffu, ready);
          if (!ok) break;
        }
        bool unit_ok = false, bad = false;
        int row = 0;
        if (lane < kUnitsPerTile) {
          const int key0 = (j * kUnitsPerTile + lane) * kUnitTokens;
          if (key0 < w.kv_len) {
            const int phys = cur_phys;
            unit_ok = phys >= 0 && phys < a.num_pages;
            bad = !unit_ok;
            row = phys * a.page_size + key0 % a.page_size;
          }
        }
        // Both producers derive the same mask from the same table entries.
        const uint32_t ok_mask = __ballot_sync(0xffffffffu, unit_ok);
        if (is_k && __ballot_sync(0xffffffffu, bad) && lane == 0 && a.err_flag) atomicOr(a.err_flag, kFlagBadPage);
        if (lane == 0) {
          if (is_k) bars->unit_ok[st] = ok_mask;  // published by the arrive below (release)
          mbar_arrive_expect_tx(&bars->kv_full[st], __popc(ok_mask) * kUnitBytes);
        }
        __syncwarp();
        if (unit_ok)
          tma_load_2d_hint(base + kOffKV + st * kStageBytes + kv_off + lane * kUnitBytes, kv_map,
                           &bars->kv_full[st], w.g * kHeadDim, row, reuse);
      }
    }
    if (lane == 0) {  // every issued copy lands before the CTA leaves
      for (int i = max(0, qw - kQBufs); is_k && i < qw; ++i)
        mbar_wait_drain(&bars->q_full[i % kQBufs], (i / kQBufs) & 1);
      for (int i = max(0, kv_it - kStages); i < kv_it; ++i)
        mbar_wait_drain(&bars->kv_full[i % kStages], (i / kStages) & 1);
    }
  } else if (warp >= kMmaWarp && warp < kMmaWarp + kQTiles) {
    // ---------------------------------------------------------------- MMA
    // Warp kMmaWarp + q issues every MMA of Q tile q, so the two tiles'
    // pipelines never wait on each other.  The whole warp runs the loop (its
    // descriptors stay warp-uniform); one elected lane issues.  A descriptor
    // differs from the stage-0 one only in its start-address field, so each
    // MMA's operands cost one add.
    const int q = warp - kMmaWarp;
    const uint64_t q_desc0 = smem_desc_sw128(smem_addr(base + kOffQ + q * kTileBytes), 16, 1024);
    const uint64_t k_desc0 = smem_desc_sw128(smem_addr(base + kOffKV), 16, 1024);
    const uint64_t v_desc0 = smem_desc_sw128(smem_addr(base + kOffKV + kTileBytes), 8192, 1024);
    constexpr uint32_t kStageDesc = kStageBytes >> 4, kQBufDesc = kQBufBytes >> 4;
    const uint32_t tmem_s = tmem + col_s(q), tmem_o = tmem + col_o(q), tmem_p = tmem + col_p(q);
    const bool leader = elect_one();
    auto issue_s = [&](int qb, int st) {
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk)
          umma_ss(tmem_s, q_desc0 + qb * kQBufDesc + kk * 2, k_desc0 + st * kStageDesc + kk * 2, kIdescS,
                  kk > 0);
        umma_commit(&bars->s_full[q]);
        // The stage's unit mask travels with S: this warp has waited for the
        // stage's kv_full, and the plain arrive releases the copy, so the
        // softmax needs no kv_full wait of its own.  The previous S (and its
        // mask) has been read: this issue followed its s_free.
        bars->s_uok[q] = bars->unit_ok[st];
        mbar_arrive(&bars->s_full[q]);
      }
      __syncwarp();
    };
    auto issue_pv = [&](int st, bool acc) {
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          umma_ts(tmem_o, tmem_p + kk * 8, v_desc0 + st * kStageDesc + kk * 128, kIdescPV, acc || kk > 0);
        umma_commit(&bars->pv_done[q]);
        if constexpr (kMixed) {
#pragma unroll
          for (int k = 0; k < kKvRelease; ++k) umma_commit(&bars->kv_empty[st]);
        } else {
          umma_commit(&bars->kv_empty[st]);
        }
      }
      __syncwarp();
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait<kPoll>(bar, parity, abort_word, a.err_flag, a.wait_limit_ns));
    };
    int qw = 0, kv_it = 0, it = 0, ow = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      long long t;
      WorkTile w;
      ok = take_tile<kPoll>(bars, i, t, kMixed ? nullptr : &w, abort_word, a);
      if constexpr (kMixed) {
        if (!ok || t == -1) break;
        if (is_decode_item(t)) {  // its stages go to the softmax warps
          DecItem d;
          decode_item(a, mx, meta, dec_start, decode_item_index(t), d);
          kv_it += d.u1 - d.u0;
          continue;
        }
      } else {
        if (!ok || t < 0) break;
      }
      if constexpr (kMixed) decode_tile<kMixed>(a, meta, t, tok_per_cta, w, mx.num_decode);
      if (w.n_kv == 0) continue;
      const int qb = qw % kQBufs;
      // Q loaded, the first K/V tile in, and the previous S read out of TMEM.
      ok = wait_all(&bars->q_full[qb], (qw / kQBufs) & 1) &&
           wait_all(&bars->kv_full[kv_it % kStages], (kv_it / kStages) & 1) &&
           (it == 0 || wait_all(&bars->s_free[q], (it - 1) & 1));
      if (!ok) break;
      tc_fence_after_sync();
      issue_s(qb, kv_it % kStages);
      for (int j = 0; j < w.n_kv; ++j) {
        const int cur = kv_it + j, u = it + j;
        if (j + 1 < w.n_kv) {
          ok = wait_all(&bars->kv_full[(cur + 1) % kStages], ((cur + 1) / kStages) & 1) &&
               wait_all(&bars->s_free[q], u & 1);
          if (!ok) break;
          tc_fence_after_sync();
          issue_s(qb, (cur + 1) % kStages);
        }
        // The first P*V of a work tile overwrites O: the previous tile's O must
        // have been read out by then.
        ok = wait_all(&bars->p_ready[q], u & 1) &&
             (j > 0 || ow == 0 || wait_all(&bars->o_free[q], (ow - 1) & 1));
        if (!ok) break;
        tc_fence_after_sync();
        issue_pv(cur % kStages, j > 0);
      }
      if (!ok) break;
      if (leader) umma_commit(&bars->q_empty[qb]);
      __syncwarp();
      ++qw;
      kv_it += w.n_kv;
      it += w.n_kv;
      ++ow;
    }
    if (leader) {
      umma_commit(&bars->mma_done);
      mbar_wait_drain(&bars->mma_done, 0);  // no MMA may still write TMEM at dealloc
    }
    __syncwarp();
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ---------------------------------------------------------------- softmax
    const int q = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const float scale_log2 = a.scale_log2;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_taddr = tmem + lane_off + col_s(q);
    const uint32_t o_taddr = tmem + lane_off + col_o(q);
    const uint32_t p_taddr = tmem + lane_off + col_p(q);
    // The two warpgroups take turns in the MUFU-heavy exponential loop, so that
    // one computes exponentials while the other loads S, reduces and stores P.
    // Warpgroup 1 hands warpgroup 0 the first turn.
    if (kQTiles > 1 && q == 1 && lane == 0) mbar_arrive(&bars->exp_turn[0]);
    // Key tiles consumed so far: every S and P*V this warpgroup has gone
    // through (it), and the K/V stages (kv_it: the same count, plus the
    // decode items' units in the mixed kernel).
    int it = 0, kv_it = 0;
    bool ok = true;
    // The plain kernel takes the next work tile (decoded by the claiming warp)
    // before writing the current one's output: the take then overlaps the wait
    // for the last P*V instead of following the output stores.  (The mixed
    // kernel, whose ring also carries decode items, measured 0.4 % slower with
    // the same early take.)
    long long t_next = 0;
    WorkTile w_next;
    bool have_next = false;
    // This thread's row of a Q tile: its token offset and its query head in the
    // group (the plain kernel keeps them across tiles).
    const int row_tok = q * tok_per_tile + r / a.group, row_head = r % a.group;
    for (int i = 0; ok; ++i) {
      long long t;
      if (!kMixed && have_next)
        t = t_next;
      else
        ok = take_tile<kPoll>(bars, i, t, nullptr, abort_word, a);
      if constexpr (kMixed) {
      if (!ok || t == -1) break;
      if (is_decode_item(t)) {
        // ------------------------------------------------------ decode item
        // Softmax warp w is the consumer of KV head hg * kDecHeads + w: the
        // split-KV decode step on its 2 KB slice of each stage.
        DecItem d;
        decode_item(a, mx, meta, dec_start, decode_item_index(t), d);
        const int g = d.hg * kDecHeads + warp;
        const long long qrow = meta.cu_seqlens_q[d.b];  // the sequence's one query
        // (a decode sequence without a query row has nothing to read or write)
        const bool head_ok = g < a.Hkv && meta.cu_seqlens_q[d.b + 1] > qrow;
        const int head0 = g * a.group;
        uint32_t qa[4][4];
        dec::load_q_frags(qa, reinterpret_cast<const __nv_bfloat16*>(mx.q) + (qrow * a.Hq + head0) * kHeadDim,
                          a.group, head_ok);
        dec::WarpState ds;
        dec::init_state(ds, meta.sinks + head0, a.group, d.c == 0 && head_ok);
        const int n_units = d.u1 - d.u0;
        for (int j = 0; j < n_units; ++j) {
          const int st = (kv_it + j) % kStages;
          const bool ready = mbar_wait<kPoll>(&bars->kv_full[st], ((kv_it + j) / kStages) & 1, abort_word,
                                              a.err_flag, a.wait_limit_ns);
          ok = __all_sync(0xffffffffu, ready);
          if (!ok) break;
          if (head_ok && bars->unit_ok[st]) {
            const uint32_t k_base = smem_addr(base + kOffKV + st * kStageBytes + warp * kDecHeadBytes);
            const uint32_t v_base = k_base + kTileBytes;
            const int n_valid = min(kUnitTokens, d.kv_len - (d.u0 + j) * kUnitTokens);
            if (a.group > 8)
              dec::consume_unit<true>(k_base, v_base, n_valid, qa, scale_log2, ds);
            else
              dec::consume_unit<false>(k_base, v_base, n_valid, qa, scale_log2, ds);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->kv_empty[st]);  // one of kSoftmaxWarps releases
        }
        if (!ok) break;
        kv_it += n_units;
        if (head_ok) {
          dec::reduce_sums(ds);
          const int r0 = lane >> 2;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int row = r0 + 8 * half;
            if (row >= a.group) continue;
            const long long prow = static_cast<long long>(d.b) * a.Hq + head0 + row;
            const long long orow = qrow * a.Hq + head0 + row;
            if (d.n_chunks == 1)
              dec::write_row(ds, half, reinterpret_cast<__nv_bfloat16*>(a.out) + orow * kHeadDim,
                             a.lse ? a.lse + orow : nullptr, nullptr, nullptr);
            else
              dec::write_row(ds, half, nullptr, nullptr, mx.o_part + (prow * mx.s_stride + d.c) * kHeadDim,
                             mx.lse_part + prow * mx.s_stride + d.c);
          }
        }
        continue;
      }
      } else {
        if (!ok || t < 0) break;
      }
      // The first tile (and every tile of the mixed kernel) is decoded here.
      WorkTile w;
      if (!kMixed && have_next)
        w = w_next;
      else
        decode_tile<kMixed>(a, meta, t, tok_per_cta, w, mx.num_decode);
      have_next = false;
      const int tok = w.tok0 + (kMixed ? q * tok_per_tile + r / a.group : row_tok);
      const int head = w.g * a.group + (kMixed ? r % a.group : row_head);
      const bool row_valid = tok < w.q_len;
      const int pos = w.kv_len - w.q_len + tok;  // fits: kv_len, q_len < 2^31
      float m_run = meta.sinks[head] * kLog2e;  // the sink is the initial running max ...
      float d_run = 1.f;                     // ... with running sum e^0 = 1
      for (int j = 0; j < w.n_kv; ++j) {
        const int u = it + j;
        int st;
        if constexpr (kMixed)
          st = (kv_it + j) % kStages;
        else
          st = u % kStages;
        // s_full completes after the MMA warp saw the stage's kv_full: the
        // stage has landed, and s_uok holds its unit mask.
        const bool ready = mbar_wait<kPoll>(&bars->s_full[q], u & 1, abort_word, a.err_flag, a.wait_limit_ns);
        ok = __all_sync(0xffffffffu, ready);
        if (!ok) break;
        const uint32_t uok = bars->s_uok[q];
        tc_fence_after_sync();
        // S comes out of TMEM with its per-row maximum over each 32 columns
        // (tcgen05.ld.red), so a tile whose keys are all visible needs no max
        // arithmetic of its own.
        uint32_t s[4][32];
        float cmax[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_max(s_taddr + 32 * c, s[c], cmax[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tmem_tie(s[c]);
          asm volatile("" : "+f"(cmax[c]));
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[q]);  // the MMA may now write the next S

        const int key_base = j * kKeys;
        const bool full = uok == 0xFFu && key_base + kKeys <= w.kv_len &&
                          (!a.causal || key_base + kKeys - 1 <= w.first_pos);
        if (uok != 0xFFu || key_base + kKeys > w.kv_len) {
          // Keys this tile does not hold (past kv_len, or a skipped page) may sit
          // over stale shared memory: their P is 0, but 0 * NaN is NaN, so thread
          // r clears V row r.  The stage has landed (s_full above) and this
          // warpgroup's P*V is issued only after its p_ready below; each Q tile's
          // P*V waits only for its own warpgroup, so both clear the rows (the same
          // zeros).
          const bool held = key_base + r < w.kv_len && ((uok >> (r / kUnitTokens)) & 1u);
          if (!held) {
            uint4* vrow = reinterpret_cast<uint4*>(base + kOffKV + st * kStageBytes + kTileBytes + r * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) vrow[i] = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
          }
        }
        float mx = fmaxf(max3f(cmax[0], cmax[1], cmax[2]), cmax[3]);
        if (!full) {
          // Some columns are not visible, and the maxima that came with S
          // include them: mask, then take the row max here.  Valid columns
          // form a prefix [0, lim): keys below kv_len and, when causal, not
          // after the row's position.  Skipped pages (rare) are cleared unit
          // by unit.
          int lim = w.kv_len - key_base;
          if (a.causal) lim = min(lim, pos - key_base + 1);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (32 * c + i >= lim) s[c][i] = __float_as_uint(-INFINITY);
          if (uok != 0xFFu) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (!((uok >> ((32 * c + i) / kUnitTokens)) & 1u)) s[c][i] = __float_as_uint(-INFINITY);
          }
          // Row max: eight independent chains of 3-input max.
          float ch[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t* v = &s[k >> 1][(k & 1) * 16];
            float acc = max3f(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
            for (int i = 3; i < 15; i += 2) acc = max3f(acc, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
            ch[k] = fmaxf(acc, __uint_as_float(v[15]));
          }
          mx = max3f(max3f(ch[0], ch[1], ch[2]), max3f(ch[3], ch[4], ch[5]), fmaxf(ch[6], ch[7]));
        }
        const float m_new = fmaxf(m_run, mx * scale_log2);
        // O is rescaled whenever a row's running maximum grows, so the largest p of
        // a row is exactly 1 and its bf16 rounding (for the P*V MMA) is exact.
        const bool resc = m_new > m_run;
        float alpha = 1.f;
        if (resc) {
          alpha = fast_exp2(m_run - m_new);
          d_run *= alpha;
          m_run = m_new;
        }
        const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
        // p = 2^(s*scale*log2e - m), rounded to bf16 for the P*V MMA; the running
        // sum adds the unrounded p.
        const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
        const uint64_t negm2 = f2_pack(neg_m, neg_m);
        uint64_t ex2[4] = {0ull, 0ull, 0ull, 0ull};
        if (kQTiles > 1) {
          const bool turn = mbar_wait<kPoll>(&bars->exp_turn[q], u & 1, abort_word, a.err_flag, a.wait_limit_ns);
          ok = __all_sync(0xffffffffu, turn);
          if (!ok) break;
        }
        uint32_t p[2][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(s[c][i]), __uint_as_float(s[c][i + 1])),
                                       scale2, negm2);
            float x0, x1;
            f2_unpack(x2, x0, x1);
            const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
            const uint32_t pk = pack_bf16x2(e0, e1);
            p[c >> 1][(c & 1) * 16 + i / 2] = pk;
            ex2[(i >> 1) & 3] = f2_add(ex2[(i >> 1) & 3], f2_pack(e0, e1));
          }
        }
        __syncwarp();
        if (kQTiles > 1 && lane == 0) mbar_arrive(&bars->exp_turn[q ^ 1]);  // pass the turn
        if (u > 0) {
          // The previous P*V must have consumed P (and updated O) before this P
          // and any rescale of O go into TMEM.
          const bool done = mbar_wait<kPoll>(&bars->pv_done[q], (u - 1) & 1, abort_word, a.err_flag, a.wait_limit_ns);
          ok = __all_sync(0xffffffffu, done);
          if (!ok) break;
          tc_fence_after_sync();
        }
        tmem_st32(p_taddr, p[0]);
        tmem_st32(p_taddr + 32, p[1]);
        {
          float lo, hi;
          f2_unpack(f2_add(f2_add(ex2[0], ex2[1]), f2_add(ex2[2], ex2[3])), lo, hi);
          d_run += lo + hi;
        }
        tmem_wait_st();
        tmem_keep(p[0]);
        tmem_keep(p[1]);
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          // (At j == 0 the first P*V of the work tile overwrites O instead.)
          uint32_t o[2][32];
          tmem_ld32(o_taddr, o[0]);
          tmem_ld32(o_taddr + 32, o[1]);
          tmem_wait_ld();
          tmem_tie(o[0]);
          tmem_tie(o[1]);
          const uint64_t alpha2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float lo, hi;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(o[h][i]), __uint_as_float(o[h][i + 1])), alpha2), lo, hi);
              o[h][i] = __float_as_uint(lo);
              o[h][i + 1] = __float_as_uint(hi);
            }
          tmem_st32(o_taddr, o[0]);
          tmem_st32(o_taddr + 32, o[1]);
          tmem_wait_st();
          tmem_keep(o[0]);
          tmem_keep(o[1]);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_ready[q]);
      }
      if (!ok) break;
      if constexpr (!kMixed) {
        ok = take_tile<kPoll>(bars, i + 1, t_next, &w_next, abort_word, a);
        if (!ok) break;
        have_next = true;
      }

      // -------------------------------------------------------------- epilogue
      uint32_t o[2][32];
      if (w.n_kv > 0) {
        const bool ready = mbar_wait<kPoll>(&bars->pv_done[q], (it + w.n_kv - 1) & 1, abort_word, a.err_flag, a.wait_limit_ns);
        ok = __all_sync(0xffffffffu, ready);
        if (!ok) break;
        tc_fence_after_sync();
        tmem_ld32(o_taddr, o[0]);
        tmem_ld32(o_taddr + 32, o[1]);
        tmem_wait_ld();
        tmem_tie(o[0]);
        tmem_tie(o[1]);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->o_free[q]);  // the next work tile may overwrite O
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 32; ++i) o[h][i] = 0u;
      }
      if (row_valid) {
        const float inv = d_run > 0.f ? 1.f / d_run : 0.f;
        const long long grow = static_cast<long long>(w.q_start + tok) * a.Hq + head;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.out) + grow * kHeadDim;
        // The output is written once and read by no later tile: evict-first,
        // so it does not push the K/V tiles that later query blocks re-read
        // out of L2.
        const uint64_t out_policy = l2_policy_evict_first();
        if ((reinterpret_cast<uintptr_t>(a.out) & 31u) == 0) {
          // 32-byte stores: whole sectors, four instructions per row.
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int h = v >> 1, i = (v & 1) * 16;
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              pk[e] = pack_bf16x2(__uint_as_float(o[h][i + 2 * e]) * inv, __uint_as_float(o[h][i + 2 * e + 1]) * inv);
            st_global_v8_hint(orow + v * 16, pk, out_policy);
          }
        } else {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const int h = v >> 2, i = (v & 3) * 8;
            uint4 o4;
            o4.x = pack_bf16x2(__uint_as_float(o[h][i + 0]) * inv, __uint_as_float(o[h][i + 1]) * inv);
            o4.y = pack_bf16x2(__uint_as_float(o[h][i + 2]) * inv, __uint_as_float(o[h][i + 3]) * inv);
            o4.z = pack_bf16x2(__uint_as_float(o[h][i + 4]) * inv, __uint_as_float(o[h][i + 5]) * inv);
            o4.w = pack_bf16x2(__uint_as_float(o[h][i + 6]) * inv, __uint_as_float(o[h][i + 7]) * inv);
            st_global_v4_hint(dst + v, o4, out_policy);
          }
        }
        if (a.lse)
          a.lse[grow] = (d_run > 0.f && m_run != -INFINITY) ? (m_run + __log2f(d_run)) * kLn2 : -INFINITY;
      }
      it += w.n_kv;
      if constexpr (kMixed) kv_it += w.n_kv;
    }
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

namespace {

template <bool kMixed>
cudaError_t launch_kernel(const PrefillArgs& a, const MixedArgs& mx, const CUtensorMap& q_map, const CUtensorMap& k_map,
                          const CUtensorMap& v_map, const CUtensorMap& k8_map,
                          const CUtensorMap& v8_map, long long n_tiles, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  auto kern = a.wait_limit_ns < kPollLimitNs ? prefill_kernel<true, kMixed> : prefill_kernel<false, kMixed>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // The register split inside the kernel assumes the launch allocation; a
  // build that launched with fewer registers would make setmaxnreg.inc wait
  // for ever, so it is refused here instead.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
  // A mixed batch's decode items are counted on the device: every SM gets a CTA.
  const unsigned grid = static_cast<unsigned>(kMixed || n_tiles >= sms ? sms : n_tiles);
  // The claim counters start at zero on every launch (a memset node when the
  // stream is being captured).
  e = cudaMemsetAsync(a.tile_ctr, 0, (kMixed ? 2 : 1) * sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kSmemBytes, stream>>>(q_map, k_map, v_map, k8_map, v8_map, a, mx, n_tiles);
  return cudaGetLastError();
}

long long query_tiles(const PrefillArgs& a) {
  const int tok_per_cta = kQTiles * (kRows / a.group);
  const long long blocks = (a.max_q_len + tok_per_cta - 1) / tok_per_cta;
  return blocks * a.B * a.Hkv;
}

}  // namespace

cudaError_t launch_prefill_bf16(const PrefillArgs& a, const CUtensorMap& q_map,
                                const CUtensorMap& k_map, const CUtensorMap& v_map,
                                cudaStream_t stream) {
  const long long n_tiles = query_tiles(a);
  if (n_tiles <= 0) return cudaSuccess;
  // (the decode-item maps are not read by the plain kernel)
  return launch_kernel<false>(a, MixedArgs{}, q_map, k_map, v_map, k_map, v_map, n_tiles, stream);
}

cudaError_t launch_mixed_bf16(const PrefillArgs& a, const MixedArgs& mx, const CUtensorMap& q_map,
                              const CUtensorMap& k_map, const CUtensorMap& v_map,
                              const CUtensorMap& k8_map, const CUtensorMap& v8_map,
                              cudaStream_t stream) {
  return launch_kernel<true>(a, mx, q_map, k_map, v_map, k8_map, v8_map, query_tiles(a), stream);
}

}  // namespace attn_sink
