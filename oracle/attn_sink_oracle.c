/*
 * Plain fp64 CPU oracle for grouped-query attention with a per-head sink logit.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load
 * this file or the library built from it; only the test suite, the smoke check
 * and the benchmark's CPU-baseline leg do.  It shares no code with the CUDA
 * kernels.
 *
 * What it computes ("GPT-OSS pada Hari ke-0", section "Atensi Sink"; and the
 * model summary "Atensi: GQA dengan Sink Atensi" on the same page):
 *   every attention head h owns a learned sink logit sink[h] that enters the
 *   softmax next to the query-key products.  For one query row of head h the
 *   logits are   z = [ sink[h], scale * q . k_j  for every visible key j ],
 *   the softmax is taken over z, and the sink's column is then dropped, so the
 *   output is   out = sum_j softmax(z)_j * v_j   (weights over real keys only)
 *   and the row's log-sum-exp is   lse = ln( e^sink[h] + sum_j e^{s_j} ).
 * The page's formulas were lost in extraction; this is the plainest reading of
 * its prose (a bias term added before the softmax and accumulated with Q.K).
 * The sink is a logit in the same units as scale*q.k and is not scaled.
 *
 * The same page explains that an efficient kernel splits the key sequence into
 * chunks and counts the sink in the first chunk only.  For that, the oracle
 * also computes "partials": the same formula restricted to a key range, with
 * or without the sink term, plus the textbook log-sum-exp merge of partials.
 * A partial over an empty key set without the sink has lse = -inf and o = 0.
 *
 * Data layout (the library's own layout, so the two can be fed the same
 * buffers):
 *   q        [total_q, Hq, D]      rows of a ragged batch, split by cu_seqlens_q
 *   k, v     [num_pages, page_size, Hkv, D]   paged cache
 *   block_table [B, bt_stride]     logical page -> physical page
 *   kv_lens  [B]                   keys per sequence (including new tokens)
 * Query head h reads KV head h / (Hq / Hkv).  Query i of a sequence with q_len
 * queries sits at absolute position kv_len - q_len + i (bottom-right aligned);
 * with causal masking it sees keys 0..position.  Floating inputs are either
 * fp32 or bf16 bit patterns; every value is widened exactly to double.
 * A physical page index outside [0, num_pages) contributes no keys and is
 * counted in the return value.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

static double load_elem(const void* base, int64_t i, int dtype) {
    if (dtype == ORACLE_F32) return (double)((const float*)base)[i];
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

typedef struct {
    const void* q;
    const void* k;
    const void* v;
    int dtype;
    const int32_t* cu_seqlens_q;
    const int32_t* kv_lens;
    const int32_t* block_table;
    int64_t bt_stride;
    const double* sinks;
    int B, Hq, Hkv, D, page_size;
    int64_t num_pages;
    double scale;
    int causal;
} problem_t;

/* Sequence that owns flat query token t (cu_seqlens_q is non-decreasing). */
static int seq_of_token(const problem_t* p, int64_t t) {
    int lo = 0, hi = p->B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (p->cu_seqlens_q[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/* Offset of element 0 of key/value row (sequence b, key j, kv head g), or -1
 * when the page table points outside the pool. */
static int64_t kv_row_offset(const problem_t* p, int b, int64_t j, int g) {
    int64_t logical = j / p->page_size;
    int64_t slot = j % p->page_size;
    int64_t phys = p->block_table[(int64_t)b * p->bt_stride + logical];
    if (phys < 0 || phys >= p->num_pages) return -1;
    return ((phys * p->page_size + slot) * p->Hkv + g) * (int64_t)p->D;
}

/*
 * One query row, one key range [key_begin, key_end), optionally with the sink.
 * Writes the partial's normalised output o[D] and its lse.  Returns the number
 * of invalid page references met.
 */
static int64_t partial_row(const problem_t* p, int64_t row, int64_t key_begin,
                           int64_t key_end, int with_sink, double* s_buf,
                           unsigned char* ok, double* o, double* lse) {
    const int64_t t = row / p->Hq;
    const int h = (int)(row % p->Hq);
    const int b = seq_of_token(p, t);
    const int group = p->Hq / p->Hkv;
    const int g = h / group;
    const int64_t q_len = p->cu_seqlens_q[b + 1] - p->cu_seqlens_q[b];
    const int64_t kv_len = p->kv_lens[b];
    const int64_t pos = kv_len - q_len + (t - p->cu_seqlens_q[b]);
    const int64_t q_off = row * (int64_t)p->D;
    int64_t invalid = 0;

    int64_t end = key_end < kv_len ? key_end : kv_len;
    if (p->causal && end > pos + 1) end = pos + 1;
    int64_t n = end > key_begin ? end - key_begin : 0;

    /* scores s_j = scale * q . k_j ; ok[i] = 0 marks a key skipped for a bad page */
    for (int64_t i = 0; i < n; ++i) {
        int64_t off = kv_row_offset(p, b, key_begin + i, g);
        ok[i] = off >= 0;
        if (!ok[i]) { ++invalid; continue; }
        double dot = 0.0;
        for (int d = 0; d < p->D; ++d)
            dot += load_elem(p->q, q_off + d, p->dtype) * load_elem(p->k, off + d, p->dtype);
        s_buf[i] = p->scale * dot;
    }

    /* M = max over z = [sink (if counted), s_j] */
    double m = -INFINITY;
    if (with_sink) m = p->sinks[h];
    for (int64_t i = 0; i < n; ++i)
        if (ok[i] && s_buf[i] > m) m = s_buf[i];

    for (int d = 0; d < p->D; ++d) o[d] = 0.0;
    if (m == -INFINITY) { *lse = -INFINITY; return invalid; }

    /* Z = e^{sink - M} + sum_j e^{s_j - M};  out = sum_j e^{s_j - M} v_j / Z */
    double z = with_sink ? exp(p->sinks[h] - m) : 0.0;
    for (int64_t i = 0; i < n; ++i) {
        if (!ok[i]) continue;
        double w = exp(s_buf[i] - m);
        z += w;
        int64_t off = kv_row_offset(p, b, key_begin + i, g);
        for (int d = 0; d < p->D; ++d) o[d] += w * load_elem(p->v, off + d, p->dtype);
    }
    for (int d = 0; d < p->D; ++d) o[d] /= z;
    *lse = m + log(z);
    return invalid;
}

static int check_problem(const problem_t* p) {
    if (!p->q || !p->k || !p->v || !p->cu_seqlens_q || !p->kv_lens || !p->block_table || !p->sinks)
        return 0;
    if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->D < 1 || p->page_size < 1) return 0;
    if (p->Hq % p->Hkv != 0) return 0;
    if (p->dtype != ORACLE_F32 && p->dtype != ORACLE_BF16) return 0;
    return 1;
}

/*
 * Partials for a list of query rows.  rows[i] = token * Hq + head (NULL: every
 * row of the batch, n_rows = total_q * Hq).  bounds holds S+1 key boundaries
 * per row (bounds[i*(S+1) + c] .. bounds[i*(S+1) + c + 1] is chunk c); chunk c
 * counts the sink when bit c of sink_mask is set.  Outputs o_parts [n_rows, S,
 * D] and lse_parts [n_rows, S].  Returns the number of invalid page references
 * met, or -1 on bad arguments.
 */
int64_t oracle_partials(const void* q, const void* k_cache, const void* v_cache, int dtype,
                        const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                        const int32_t* block_table, int64_t bt_stride, const double* sinks,
                        int B, int Hq, int Hkv, int D, int page_size, int64_t num_pages,
                        double scale, int causal, const int64_t* rows, int64_t n_rows,
                        const int64_t* bounds, int S, uint64_t sink_mask,
                        double* o_parts, double* lse_parts, int n_threads) {
    problem_t p = {q, k_cache, v_cache, dtype, cu_seqlens_q, kv_lens, block_table, bt_stride,
                   sinks, B, Hq, Hkv, D, page_size, num_pages, scale, causal};
    if (!check_problem(&p) || !bounds || !o_parts || !lse_parts || S < 1 || S > 64 || n_rows < 0)
        return -1;
    int64_t max_kv = 0;
    for (int b = 0; b < B; ++b) if (kv_lens[b] > max_kv) max_kv = kv_lens[b];
    int64_t invalid = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
#pragma omp parallel reduction(+ : invalid)
    {
        size_t cap = (size_t)(max_kv > 0 ? max_kv : 1);
        double* s_buf = (double*)malloc(sizeof(double) * cap);
        unsigned char* ok = (unsigned char*)malloc(cap);
#pragma omp for schedule(dynamic, 4)
        for (int64_t i = 0; i < n_rows; ++i) {
            int64_t row = rows ? rows[i] : i;
            for (int c = 0; c < S; ++c) {
                int64_t kb = bounds[i * (S + 1) + c];
                int64_t ke = bounds[i * (S + 1) + c + 1];
                invalid += partial_row(&p, row, kb, ke, (int)((sink_mask >> c) & 1u), s_buf, ok,
                                       o_parts + (i * S + c) * (int64_t)D, lse_parts + i * S + c);
            }
        }
        free(s_buf);
        free(ok);
    }
    return invalid;
}

/*
 * Log-sum-exp merge of S partial states per row:
 *   L = ln sum_c e^{lse_c},   out = sum_c e^{lse_c - L} o_c.
 * Adds no sink: a sink lives inside whichever partial counted it.
 * All partials at -inf give out = 0 and L = -inf.
 */
void oracle_merge(const double* o_parts, const double* lse_parts, int64_t n_rows, int S, int D,
                  double* out, double* lse_out) {
    for (int64_t r = 0; r < n_rows; ++r) {
        double m = -INFINITY;
        for (int c = 0; c < S; ++c)
            if (lse_parts[r * S + c] > m) m = lse_parts[r * S + c];
        for (int d = 0; d < D; ++d) out[r * D + d] = 0.0;
        if (m == -INFINITY) { lse_out[r] = -INFINITY; continue; }
        double z = 0.0;
        for (int c = 0; c < S; ++c) z += exp(lse_parts[r * S + c] - m);
        double big_l = m + log(z);
        for (int c = 0; c < S; ++c) {
            double w = exp(lse_parts[r * S + c] - big_l);
            for (int d = 0; d < D; ++d) out[r * D + d] += w * o_parts[(r * S + c) * (int64_t)D + d];
        }
        lse_out[r] = big_l;
    }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
