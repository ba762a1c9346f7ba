"""Pins for the fp64 oracle against facts that do not come from the oracle.

Each test fixes the oracle to something independent of its own code: a
pure-Python brute force, closed forms for one key and for n equal keys, the
sink = -inf special case against torch's scaled_dot_product_attention in fp64,
the large-sink limit, the sum rule with V = 1, and the split/merge invariance
that the page "GPT-OSS pada Hari ke-0" (section "Atensi Sink") states: the sink
must be counted in exactly one chunk when the key sequence is split.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as W
from _brute import attention_row


def _problem(batch):
    return oracle.Problem(batch.q, batch.k_cache, batch.v_cache, batch.cu_seqlens_q,
                          batch.kv_lens, batch.block_table, batch.sinks, batch.scale, batch.causal)


def _small_batch(seed, q_lens, kv_lens, Hq=4, Hkv=2, D=8, ps=4, dtype=W.FP32, causal=True,
                 sink_std=1.0, sinks=None):
    rng = np.random.default_rng(seed)
    pool = W.make_pool(rng, kv_lens, Hkv, D, ps, dtype)
    q = W.make_queries(rng, int(np.sum(q_lens)), Hq, D, dtype)
    s = W.sinks_normal(rng, Hq, sink_std) if sinks is None else np.asarray(sinks, np.float32)
    return W.batch_from_pool(pool, np.arange(len(kv_lens)), q_lens, q, s, causal, dtype)


CASES = [
    # (q_lens, kv_lens, Hq, Hkv, D, page_size, dtype, causal)
    ([3, 5], [7, 5], 4, 2, 8, 4, W.FP32, True),
    ([1, 1, 1], [9, 1, 16], 6, 3, 8, 4, W.FP32, True),
    ([4, 2], [10, 19], 4, 4, 16, 16, W.BF16, True),
    ([6], [6], 8, 2, 8, 4, W.BF16, False),
    ([2, 3], [20, 3], 4, 1, 8, 8, W.FP32, False),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_oracle_matches_brute_force(case):
    q_lens, kv_lens, Hq, Hkv, D, ps, dt, causal = CASES[case]
    batch = _small_batch(100 + case, q_lens, kv_lens, Hq, Hkv, D, ps, dt, causal)
    out, lse, bad = _problem(batch).attention()
    assert bad == 0
    for row in range(batch.total_q * Hq):
        ref, ref_lse, _ = attention_row(batch, row)
        np.testing.assert_allclose(out[row], ref, rtol=0, atol=1e-12)
        assert abs(lse[row] - ref_lse) <= 1e-12


def test_single_key_closed_form():
    """One visible key: out = sigmoid(s - sink) * v, lse = ln(e^sink + e^s)."""
    batch = _small_batch(7, [1, 1], [1, 1], Hq=4, Hkv=2, D=8)
    out, lse, _ = _problem(batch).attention()
    for row in range(batch.total_q * batch.Hq):
        t, h = divmod(row, batch.Hq)
        g = h // (batch.Hq // batch.Hkv)
        phys = batch.block_table[t, 0]
        k = batch.k_cache[phys, 0, g].astype(np.float64)
        v = batch.v_cache[phys, 0, g].astype(np.float64)
        s = batch.scale * float(np.dot(batch.q[t, h].astype(np.float64), k))
        sink = float(batch.sinks[h])
        sig = 1.0 / (1.0 + math.exp(sink - s))
        np.testing.assert_allclose(out[row], sig * v, rtol=1e-13, atol=1e-14)
        assert lse[row] == pytest.approx(np.logaddexp(sink, s), abs=1e-13)


def test_identical_keys_closed_form():
    """n equal keys and values: out = n e^s / (e^sink + n e^s) * v."""
    n = 11
    batch = _small_batch(8, [1], [n], Hq=2, Hkv=1, D=8)
    phys0, slot0 = batch.block_table[0, 0], 0
    for j in range(n):
        p, sl = batch.block_table[0, j // batch.page_size], j % batch.page_size
        batch.k_cache[p, sl] = batch.k_cache[phys0, slot0]
        batch.v_cache[p, sl] = batch.v_cache[phys0, slot0]
    out, lse, _ = _problem(batch).attention()
    k = batch.k_cache[phys0, slot0, 0].astype(np.float64)
    v = batch.v_cache[phys0, slot0, 0].astype(np.float64)
    for h in range(batch.Hq):
        s = batch.scale * float(np.dot(batch.q[0, h].astype(np.float64), k))
        sink = float(batch.sinks[h])
        w = n * math.exp(s) / (math.exp(sink) + n * math.exp(s))
        np.testing.assert_allclose(out[h], w * v, rtol=1e-12, atol=1e-14)
        assert lse[h] == pytest.approx(math.log(math.exp(sink) + n * math.exp(s)), abs=1e-12)


def _dense_kv(batch, b):
    """Logical [kv_len, Hkv, D] keys/values of sequence b, read through its table."""
    kv = int(batch.kv_lens[b])
    idx = np.arange(kv)
    phys = batch.block_table[b, idx // batch.page_size]
    k = batch.k_cache[phys, idx % batch.page_size]
    v = batch.v_cache[phys, idx % batch.page_size]
    if batch.dtype == W.BF16:
        k, v = W.bf16_bits_to_f32(k), W.bf16_bits_to_f32(v)
    return k.astype(np.float64), v.astype(np.float64)


@pytest.mark.parametrize("causal", [True, False])
def test_no_sink_reduces_to_sdpa(causal):
    """sink = -inf is plain GQA attention: torch SDPA in fp64 with a bottom-right mask."""
    torch = pytest.importorskip("torch")
    Hq, Hkv = 8, 2
    batch = _small_batch(9, [5, 3], [12, 3], Hq=Hq, Hkv=Hkv, D=16, ps=4, dtype=W.BF16,
                         causal=causal, sinks=[-math.inf] * Hq)
    out, lse, _ = _problem(batch).attention()
    out = out.reshape(batch.total_q, Hq, -1)
    lse = lse.reshape(batch.total_q, Hq)
    qf = W.bf16_bits_to_f32(batch.q).astype(np.float64)
    for b in range(batch.B):
        t0, t1 = batch.cu_seqlens_q[b], batch.cu_seqlens_q[b + 1]
        k, v = _dense_kv(batch, b)
        qt = torch.from_numpy(qf[t0:t1]).permute(1, 0, 2)                 # [Hq, q, D]
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        ql, kl = t1 - t0, k.shape[0]
        mask = None
        if causal:
            pos = torch.arange(kl - ql, kl)[:, None]
            mask = torch.arange(kl)[None, :] <= pos
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt[None], kt[None], vt[None], attn_mask=mask, scale=batch.scale)[0]
        np.testing.assert_allclose(out[t0:t1], ref.permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)
        scores = (qt @ kt.transpose(1, 2)) * batch.scale
        if mask is not None:
            scores = scores.masked_fill(~mask, -math.inf)
        np.testing.assert_allclose(lse[t0:t1], torch.logsumexp(scores, -1).T.numpy(), atol=1e-12)


def test_huge_sink_drives_output_to_zero():
    batch = _small_batch(10, [4], [9], sinks=[1e4] * 4)
    out, lse, _ = _problem(batch).attention()
    assert np.all(np.abs(out) <= 1e-300)
    np.testing.assert_allclose(lse, 1e4, rtol=0, atol=1e-9)


def test_sum_rule_with_unit_values():
    """V = 1 everywhere: attention mass on real keys = 1 - e^{sink - lse}."""
    batch = _small_batch(11, [3, 1, 6], [8, 13, 6], Hq=6, Hkv=3, sink_std=2.0)
    batch.v_cache[:] = 1.0
    out, lse, _ = _problem(batch).attention()
    heads = np.tile(np.arange(batch.Hq), batch.total_q)
    expect = 1.0 - np.exp(batch.sinks[heads].astype(np.float64) - lse)
    np.testing.assert_allclose(out, np.repeat(expect[:, None], batch.D, 1), atol=1e-13)


def _random_bounds(rng, kv, S):
    cuts = np.sort(rng.integers(0, kv + 1, S - 1))
    return np.concatenate([[0], cuts, [kv]])


@pytest.mark.parametrize("S", [1, 2, 3, 32])
def test_split_merge_invariance(S):
    rng = np.random.default_rng(12 + S)
    batch = _small_batch(12, [1] * 4, [1, 17, 40, 64], Hq=4, Hkv=2, D=8, ps=4, sink_std=2.0)
    prob = _problem(batch)
    ref, ref_lse, _ = prob.attention()
    rows = prob.all_rows()
    b = prob.row_seq(rows)
    bounds = np.stack([_random_bounds(rng, batch.kv_lens[x], S) for x in b])
    o, l, _ = prob.partials(rows, bounds, 1)
    out, lse = oracle.merge(o, l)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)
    if S > 1:
        # the sink may sit in any single chunk ...
        o, l, _ = prob.partials(rows, bounds, 1 << (S - 1))
        out, lse = oracle.merge(o, l)
        np.testing.assert_allclose(out, ref, atol=1e-12)
        # ... but counting it in two chunks changes the result
        o, l, _ = prob.partials(rows, bounds, 0b11)
        out, lse = oracle.merge(o, l)
        assert np.max(np.abs(lse - ref_lse)) > 1e-3
    # the page-aligned split rule used by decode gives the same answer
    out, lse, _ = prob.attention_split(num_splits=S)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_split_rule_pages():
    """Chunk c of S covers pages [floor(cP/S), floor((c+1)P/S)), chunk 0 holds key 0."""
    batch = _small_batch(13, [1], [37], ps=4)
    prob = _problem(batch)
    bounds = prob.split_bounds(np.array([0]), 4)[0]
    # P = 10 pages -> page cuts 0, 2, 5, 7, 10 -> keys 0, 8, 20, 28, 37 (clipped)
    assert bounds.tolist() == [0, 8, 20, 28, 37]
    bounds = prob.split_bounds(np.array([0]), 16)[0]
    assert bounds[0] == 0 and bounds[-1] == 37 and np.all(np.diff(bounds) >= 0)


def test_page_table_invariance():
    rng = np.random.default_rng(14)
    a = _small_batch(14, [2, 3], [11, 7], dtype=W.BF16)
    prob_a = _problem(a)
    # same logical contents, different physical placement
    perm = rng.permutation(a.num_pages)
    inv = np.argsort(perm)
    k2, v2 = a.k_cache[perm], a.v_cache[perm]
    bt2 = np.where(a.block_table >= 0, inv[np.maximum(a.block_table, 0)], -1).astype(np.int32)
    prob_b = oracle.Problem(a.q, k2, v2, a.cu_seqlens_q, a.kv_lens, bt2, a.sinks, a.scale)
    oa, la, _ = prob_a.attention()
    ob, lb, _ = prob_b.attention()
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_empty_key_set():
    """kv_len = 0: out = 0 and lse = sink (-inf when the sink is -inf)."""
    batch = _small_batch(15, [1, 1], [0, 5], Hq=2, Hkv=1, sinks=[-math.inf, 0.5], causal=False)
    out, lse, _ = _problem(batch).attention()
    assert np.all(out[:2] == 0)
    assert lse[0] == -math.inf and lse[1] == 0.5


def test_invalid_page_is_skipped_and_counted():
    batch = _small_batch(16, [1], [12], ps=4)
    batch.block_table[0, 1] = batch.num_pages + 3
    out, lse, bad = _problem(batch).attention()
    assert bad == 4 * batch.Hq                  # one page of 4 keys, counted per head row
    for row in range(batch.Hq):
        ref, ref_lse, nbad = attention_row(batch, row)
        assert nbad == 4
        np.testing.assert_allclose(out[row], ref, atol=1e-12)
        assert abs(lse[row] - ref_lse) <= 1e-12


def test_outlier_logits_stay_finite():
    """Keys scaled x20 give logits in the hundreds; max subtraction keeps it finite."""
    batch = _small_batch(17, [1], [30], D=64, Hq=2, Hkv=1, ps=16)
    batch.k_cache *= 20.0
    out, lse, _ = _problem(batch).attention()
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    for row in range(2):
        ref, ref_lse, _ = attention_row(batch, row)
        np.testing.assert_allclose(out[row], ref, atol=1e-12)
        assert abs(lse[row] - ref_lse) <= 1e-9
