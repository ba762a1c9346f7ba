"""The polynomial exp2 of the prefill softmax: its coefficients come from the
committed fit, and the full algorithm (range reduction, cubic, exponent add),
emulated in float32, stays within 1e-4 relative of exp2 (no GPU needed)."""
import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gqa_attention_sinks_gb300", "csrc")
sys.path.insert(0, CSRC)
import exp2_poly  # noqa: E402


def _header_coeffs():
    text = open(os.path.join(CSRC, "exp2_poly.cuh")).read()
    return [float(re.search(r"kExp2C%d = ([-+0-9.e]+)f;" % k, text).group(1)) for k in range(4)]


def _emulate(x):
    """float32 emulation of exp2_poly_pair for one lane."""
    c = [np.float32(v) for v in _header_coeffs()]
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    r = (t - magic).astype(np.float32)
    f = (x - r).astype(np.float32)
    p = (c[3] * f + c[2]).astype(np.float32)
    p = (p * f + c[1]).astype(np.float32)
    p = (p * f + c[0]).astype(np.float32)
    bits = p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.astype(np.uint32).view(np.float32)


def test_header_coefficients_match_fit():
    fit = exp2_poly.fit()
    for h, c in zip(_header_coeffs(), fit):
        assert abs(h - float(np.float32(c))) <= 1e-8 * max(1.0, abs(c))
    assert exp2_poly.max_rel_error(fit) < 1e-4


def test_full_algorithm_accuracy():
    x = np.concatenate([np.linspace(-125.9, 20, 2_000_001), np.arange(-125, 21)]).astype(np.float32)
    y = _emulate(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(y / ref - 1)) < 1e-4


def test_clamp_for_masked_entries():
    y = _emulate(np.array([-np.inf, -1e30, -500.0, -126.0], np.float32))
    assert np.all(np.isfinite(y)) and np.all(y >= 0) and np.all(y <= 2.0 ** -125)
