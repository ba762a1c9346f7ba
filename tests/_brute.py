"""Pure-Python brute force for sink attention, used only to pin the C oracle.

No streaming and no vector library: for each query row it lists every logit
z = [sink, scale * q . k_j ...] explicitly, takes the softmax with math.fsum,
drops the sink column and sums the weighted value rows ("GPT-OSS pada Hari
ke-0", section "Atensi Sink").  Meant for inputs of a few hundred keys at most.
"""
import math


def _bf16(bits):
    import struct
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def _val(arr, idx, is_bf16):
    x = arr[idx]
    return _bf16(x) if is_bf16 else float(x)


def attention_row(batch, row, key_range=None, with_sink=True):
    """(out list[D], lse float, n_invalid) for flat row = token * Hq + head."""
    Hq, D = batch.q.shape[1], batch.q.shape[2]
    num_pages, ps, Hkv, _ = batch.k_cache.shape
    is_bf16 = batch.q.dtype.name == "uint16"
    t, h = divmod(int(row), Hq)
    b = 0
    while batch.cu_seqlens_q[b + 1] <= t:
        b += 1
    q_len = int(batch.cu_seqlens_q[b + 1] - batch.cu_seqlens_q[b])
    kv_len = int(batch.kv_lens[b])
    pos = kv_len - q_len + (t - int(batch.cu_seqlens_q[b]))
    g = h // (Hq // Hkv)
    lo, hi = (0, kv_len) if key_range is None else key_range
    hi = min(hi, kv_len)
    if batch.causal:
        hi = min(hi, pos + 1)
    qv = [_val(batch.q, (t, h, d), is_bf16) for d in range(D)]
    logits, values, invalid = [], [], 0
    for j in range(lo, hi):
        phys = int(batch.block_table[b, j // ps])
        if phys < 0 or phys >= num_pages:
            invalid += 1
            continue
        kv = [_val(batch.k_cache, (phys, j % ps, g, d), is_bf16) for d in range(D)]
        vv = [_val(batch.v_cache, (phys, j % ps, g, d), is_bf16) for d in range(D)]
        logits.append(batch.scale * math.fsum(a * c for a, c in zip(qv, kv)))
        values.append(vv)
    z = ([float(batch.sinks[h])] if with_sink else []) + logits
    if not z or max(z) == -math.inf:
        return [0.0] * D, -math.inf, invalid
    m = max(z)
    e = [math.exp(x - m) for x in z]
    total = math.fsum(e)
    w = e[1:] if with_sink else e
    out = [math.fsum(wj * vj[d] for wj, vj in zip(w, values)) / total for d in range(D)]
    return out, m + math.log(total), invalid
