"""Helpers for GPU parity tests: move a workload batch to the device and
compare kernel output with the fp64 oracle under the stated tolerances."""
import numpy as np
import torch

import oracle
import workloads as W

# Tolerances for bf16 inputs with fp32 accumulation (and the fp32 path).
MAX_ABS = 1e-2
MEAN_ABS = 1e-3
LSE_ABS = 1e-3


def to_device(a, dtype):
    """numpy host array -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class DeviceBatch:
    def __init__(self, batch):
        self.b = batch
        self.q = to_device(batch.q, None)
        self.k = to_device(batch.k_cache, None)
        self.v = to_device(batch.v_cache, None)
        self.cu = torch.from_numpy(batch.cu_seqlens_q).cuda()
        self.kv_lens = torch.from_numpy(batch.kv_lens).cuda()
        self.bt = torch.from_numpy(np.ascontiguousarray(batch.block_table)).cuda()
        self.sinks = torch.from_numpy(batch.sinks.astype(np.float32)).cuda()
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")


def oracle_problem(batch):
    return oracle.Problem(batch.q, batch.k_cache, batch.v_cache, batch.cu_seqlens_q,
                          batch.kv_lens, batch.block_table, batch.sinks, batch.scale,
                          batch.causal)


def bf16_half_ulp(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits): the rounding
    error the bf16 output format itself adds to an exact result."""
    ax = np.maximum(np.abs(x), np.float64(2.0 ** -126))
    return np.exp2(np.floor(np.log2(ax)) - 8.0)


def bf16_round(x):
    """Round float64 values to the nearest bf16 value (ties to even), as float64."""
    return W.bf16_bits_to_f32(W.to_bf16_bits(np.asarray(x, np.float32))).astype(np.float64)


# Below this magnitude a bf16 output keeps the bare MAX_ABS bound: half a bf16
# ulp there is at most 2^-8 = 0.0039, well inside 1e-2.  From 2 up, half an ulp
# (>= 0.0078) leaves the kernel's own arithmetic too little of 1e-2, and from 4
# up (>= 0.0156) no bf16 number could meet it, so the bound adds the output
# format's own rounding of the exact value there.
BF16_ROUNDING_FROM = 2.0

LAST_STATS = {}


def compare(out, lse, ref_out, ref_lse, rows=None, what=""):
    """out/lse: kernel tensors ([rows_total, Hq, D] / [rows_total, Hq]); ref: oracle rows.

    Per element: |out - ref| <= MAX_ABS, plus, for bf16 outputs whose exact value
    has |ref| >= BF16_ROUNDING_FROM, half a bf16 ulp of ref (the output format's
    own rounding, which the fp64 oracle does not have).  Mean abs error <=
    MEAN_ABS, lse <= LSE_ABS.  Returns the error statistics (also kept in
    LAST_STATS) and prints them.
    """
    is_bf16 = out.dtype == torch.bfloat16
    o = out.float().reshape(-1, out.shape[-1]).cpu().numpy().astype(np.float64)
    l = lse.reshape(-1).cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l = o[rows], l[rows]
    assert np.all(np.isfinite(o)), "%s: non-finite output" % what
    err = np.abs(o - ref_out)
    big = np.abs(ref_out) >= BF16_ROUNDING_FROM
    bound = MAX_ABS + (np.where(big, bf16_half_ulp(ref_out), 0.0) if is_bf16 else 0.0)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    small_err = float(err[~big].max()) if np.any(~big) else 0.0
    stats = {"what": what, "elements": int(err.size), "max_abs": float(err.max()),
             "mean_abs": float(err.mean()), "max_abs_where_ref_below_2": small_err,
             "big_elements": int(big.sum())}
    if is_bf16:
        # Diagnostic only: how many elements differ from the correctly rounded
        # exact value by more than MAX_ABS (one-ulp straddles of a rounding
        # boundary when |ref| >= 2).
        stats["beyond_1e-2_of_rn_ref"] = int((np.abs(o - bf16_round(ref_out)) > MAX_ABS).sum())
    msg = ("%s: max abs err %.3g (bound there %.3g, |ref| %.3g, kernel %.5g, ref %.5g, row %d), "
           "mean abs err %.3g, max err where |ref|<2: %.3g" %
           (what, err.max(), bound[worst] if np.ndim(bound) else bound, abs(ref_out[worst]),
            o[worst], ref_out[worst], worst[0], err.mean(), small_err))
    assert np.all(err <= bound), msg
    assert err.mean() <= MEAN_ABS, msg
    both_inf = np.isneginf(l) & np.isneginf(ref_lse)
    with np.errstate(invalid="ignore"):
        lerr = np.where(both_inf, 0.0, np.abs(l - ref_lse))
    assert lerr.max() <= LSE_ABS, "%s: lse err %.3g" % (what, lerr.max())
    stats["lse_max_abs"] = float(lerr.max())
    LAST_STATS.clear()
    LAST_STATS.update(stats)
    print("parity %s" % stats)
    return err.max(), err.mean()
