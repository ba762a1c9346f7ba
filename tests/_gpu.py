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


def compare(out, lse, ref_out, ref_lse, rows=None, what=""):
    """out/lse: kernel tensors ([rows_total, Hq, D] / [rows_total, Hq]); ref: oracle rows.

    Bound per element: MAX_ABS on the kernel's arithmetic, plus, for bf16 outputs,
    half a bf16 ulp of the exact value (the output format's own rounding, which
    the fp64 oracle does not have).  Mean abs error <= MEAN_ABS, lse <= LSE_ABS.
    """
    is_bf16 = out.dtype == torch.bfloat16
    o = out.float().reshape(-1, out.shape[-1]).cpu().numpy().astype(np.float64)
    l = lse.reshape(-1).cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l = o[rows], l[rows]
    assert np.all(np.isfinite(o)), "%s: non-finite output" % what
    err = np.abs(o - ref_out)
    bound = MAX_ABS + (bf16_half_ulp(ref_out) if is_bf16 else 0.0)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    msg = ("%s: max abs err %.3g (bound there %.3g, |ref| %.3g, kernel %.5g, ref %.5g, row %d), "
           "mean abs err %.3g, max err where |ref|<1: %.3g" %
           (what, err.max(), bound[worst] if np.ndim(bound) else bound, abs(ref_out[worst]),
            o[worst], ref_out[worst], worst[0], err.mean(),
            err[np.abs(ref_out) < 1].max() if np.any(np.abs(ref_out) < 1) else 0.0))
    assert np.all(err <= bound), msg
    assert err.mean() <= MEAN_ABS, msg
    both_inf = np.isneginf(l) & np.isneginf(ref_lse)
    lerr = np.where(both_inf, 0.0, np.abs(l - ref_lse))
    assert lerr.max() <= LSE_ABS, "%s: lse err %.3g" % (what, lerr.max())
    return err.max(), err.mean()
