"""Host-side checks of the seeded input generator (no GPU)."""
import numpy as np
import pytest

import workloads as W


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(4096).astype(np.float32) * 100,
                        np.array([0.0, -0.0, 1e-40, 3.0e38, np.inf, -np.inf], np.float32)])
    ours = W.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(W.bf16_bits_to_f32(ours),
                          torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_pool_layout():
    rng = np.random.default_rng(1)
    kv = [5, 16, 33]
    pool = W.make_pool(rng, kv, Hkv=2, D=8, page_size=16, dtype=W.FP32)
    need = sum((k + 15) // 16 for k in kv)
    assert pool.k_cache.shape[0] == need + max(1, int(np.ceil(0.1 * need)))
    used = pool.block_table[pool.block_table >= 0]
    assert len(np.unique(used)) == len(used) == need            # distinct pages
    spare = np.setdiff1d(np.arange(pool.k_cache.shape[0]), used)
    assert np.all(np.isnan(pool.k_cache[spare])) and np.all(np.isnan(pool.v_cache[spare]))
    for b, k in enumerate(kv):
        last = pool.block_table[b, (k - 1) // 16]
        assert np.all(np.isnan(pool.k_cache[last, k % 16 or 16:]))      # unused slots
        assert np.all(np.isfinite(pool.k_cache[last, :(k - 1) % 16 + 1]))
        assert np.all(pool.block_table[b, (k + 15) // 16:] == -1)


def test_workloads_are_seeded():
    a = W.gptoss_decode(num_seqs=3, kv_min=16, kv_max=64)
    b = W.gptoss_decode(num_seqs=3, kv_min=16, kv_max=64)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.block_table, b.block_table)
    assert np.array_equal(a.k_cache.view(np.uint16), b.k_cache.view(np.uint16))


def test_mixed_batch_shares_pool():
    m = W.mixed_batch(n_decode=3, decode_kv=(20, 40), n_prefill=2, prefill_new=8, prefix=(0, 30))
    d, p = m["decode"], m["prefill"]
    assert d.k_cache is p.k_cache
    assert np.all(p.q_lens == 8) and np.all(p.kv_lens >= 8)
    assert not set(d.block_table[d.block_table >= 0]) & set(p.block_table[p.block_table >= 0])


def test_tiny_appends_hidden():
    t = W.tiny_prefill_decode()
    pre = t["prefill"]
    assert pre.q.dtype == np.float32 and pre.kv_lens.tolist() == [64, 64]
    for s, step in enumerate(t["steps"]):
        j = 64 + s
        for b in range(2):
            phys = pre.block_table[b, j // 16]
            assert np.all(np.isnan(pre.k_cache[phys, j % 16]))
            assert np.all(np.isfinite(step["new_k"][b]))
