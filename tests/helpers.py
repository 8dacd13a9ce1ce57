"""Shared comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (floating point; bf16 inputs, fp32 accumulation, bf16 output):
  |gpu - ref|                          <= 1e-2                       for |ref| < 4
                                       <= bf16 spacing / 2 + 2^-8    for |ref| >= 4
  sum |gpu - ref| / sum |ref|          <= 2e-3     on the output (L1 ratio)
  max |lse_gpu - lse_ref|              <= 1e-3     on the natural-log lse

The output is bf16, so even an exact kernel is off by up to half a bf16
spacing after rounding. Below |ref| = 4 half a spacing is at most 2^-7
(about 0.0078, on [2, 4)), under 1e-2, so the 1e-2 bar applies unchanged. From
|ref| = 4 up, half a spacing (2^-6 on [4, 8)) is itself above 1e-2; there the
bar is half a spacing for the final rounding plus an allowance of 2^-8 for
the error before it. That allowance covers P entering the P V product as fp16
(relative rounding at most 2^-11 per term, so at most 2^-11 max|v| on a
weighted mean of V rows, i.e. 2^-8 for |v| < 8, which holds for the normal
inputs used here; tests over larger values pass their max |v|, see
element_bound); fp32 accumulation adds far less.
Rounding the exact output to bf16 alone gives an L1 ratio near 1.35e-3 (a
quarter spacing on average over a significand uniform in [1, 2)); the kernels
keep P at 11 (prefill, fp16) or 16 (decode, bf16 hi+lo) significant bits so
that P adds well under the remaining 0.65e-3.
Rows whose reference sees nothing (lse = -inf) must give out = 0, lse = -inf.

Set SINKATTN_PARITY_LOG=<file> to append one line of error statistics per check.
"""
import json
import os

import numpy as np
import torch

ABS_FLOOR = 1e-2
ABS_FLOOR_UNTIL = 4.0       # |ref| below this: the plain 1e-2 bar
PRE_ROUNDING = 2.0 ** -8    # |ref| from there: half a spacing + this
MEAN_REL = 2e-3
LSE_ABS = 1e-3


def to_np(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().float().cpu().double().numpy()


def bf16_spacing(x):
    """Distance between consecutive bf16 values around |x| (8 significant bits)."""
    a = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.ldexp(1.0, (np.floor(np.log2(a)) - 7).astype(np.int64))


def element_bound(ref, v_absmax=None):
    """Per-element bar on |gpu - ref| for a bf16 output (see the module
    docstring). v_absmax: the largest |v| of the inputs when it may exceed 8
    (unscaled fp8 codes); the pre-rounding allowance is then 2^-11 v_absmax."""
    ref = np.asarray(ref, dtype=np.float64)
    pre = PRE_ROUNDING if v_absmax is None else max(PRE_ROUNDING, 2.0 ** -11 * float(v_absmax))
    return np.where(np.abs(ref) < ABS_FLOOR_UNTIL, ABS_FLOOR, 0.5 * bf16_spacing(ref) + pre)


def check_close(out_gpu, lse_gpu, out_ref, lse_ref, what="", v_absmax=None):
    o = to_np(out_gpu).reshape(out_ref.shape)
    assert np.all(np.isfinite(o)), what + ": non-finite output"
    err = np.abs(o - out_ref)
    bound = element_bound(out_ref, v_absmax)
    max_abs = float(err.max()) if err.size else 0.0
    worst = float((err / bound).max()) if err.size else 0.0
    denom = float(np.abs(out_ref).sum())
    mean_rel = float(err.sum()) / denom if denom > 0 else float(err.sum())
    stats = {"what": what, "max_abs": max_abs, "max_abs_over_bound": worst,
             "mean_rel": mean_rel, "n": int(err.size)}
    if lse_gpu is not None:
        l = to_np(lse_gpu).reshape(lse_ref.shape)
        empty = ~np.isfinite(lse_ref)
        assert np.all(l[empty] == -np.inf), what + ": empty rows must give lse = -inf"
        if np.any(~empty):
            stats["lse_abs"] = float(np.abs(l[~empty] - lse_ref[~empty]).max())
    log = os.environ.get("SINKATTN_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps(stats) + "\n")
    assert worst <= 1.0, "%s: max_abs %.3g exceeds its bound (x%.2f)" % (what, max_abs, worst)
    assert mean_rel <= MEAN_REL, "%s: mean_rel %.3g" % (what, mean_rel)
    if "lse_abs" in stats:
        assert stats["lse_abs"] <= LSE_ABS, "%s: lse err %.3g" % (what, stats["lse_abs"])
    return stats


def check_pair(out_a, lse_a, out_b, lse_b, what=""):
    """Two GPU results of the same definition (different kernels or split
    plans), each bf16-rounded from its own fp32 value. Each is within the
    parity bar of the exact value, so they differ by at most one bf16 spacing
    (the two roundings) plus twice the pre-rounding allowance; below
    |b| = 2 that is under 1e-2 + 2^-7 and the plain 1e-2 bar is kept. L1 ratio
    and lse as in check_close."""
    a = to_np(out_a)
    b = to_np(out_b).reshape(a.shape)
    assert np.all(np.isfinite(a)), what + ": non-finite output"
    err = np.abs(a - b)
    bound = np.where(np.abs(b) < 2.0, ABS_FLOOR, bf16_spacing(b) + 2 * PRE_ROUNDING)
    worst = float((err / bound).max()) if err.size else 0.0
    denom = float(np.abs(b).sum())
    mean_rel = float(err.sum()) / denom if denom > 0 else float(err.sum())
    assert worst <= 1.0, "%s: max diff %.3g over its bound (x%.2f)" % (what, float(err.max()),
                                                                       worst)
    assert mean_rel <= MEAN_REL, "%s: mean_rel %.3g" % (what, mean_rel)
    la, lb = to_np(lse_a), to_np(lse_b).reshape(np.shape(to_np(lse_a)))
    fin = np.isfinite(lb)
    assert np.array_equal(np.isfinite(la), fin), what + ": empty rows differ"
    if np.any(fin):
        assert float(np.abs(la[fin] - lb[fin]).max()) <= LSE_ABS, what + ": lse"


def cuda(t):
    return None if t is None else t.cuda()


# Gradients (backward). The gradient outputs are bf16 like the forward output,
# but their scale differs from tensor to tensor (dq and dk carry `scale`, dv
# sums P-weighted dO over many queries), so the element bound is relative to
# the tensor's own RMS instead of an absolute 1e-2:
#   |gpu - ref|                  <= max(2 bf16 spacings at |ref|, 1e-2 rms(ref))
#   sum |gpu - ref| / sum |ref|  <= GRAD_MEAN_REL
# Beyond the output's own rounding (L1 ratio ~1.35e-3) the kernels add fp16
# rounding of P and dS (11 significant bits) in the second products; D_i is
# formed exactly (fp32 sum of P_ij dP_ij), not from the bf16 forward output,
# whose rounding would be amplified where dP_ij - D_i cancels. So the L1 bar
# is the forward's. dsinks is float32: |gpu - ref| <= 1e-3 (1 + |ref|).
GRAD_SPACINGS = 2.0
GRAD_RMS_FRAC = 1e-2
GRAD_MEAN_REL = 2e-3


def check_grad(gpu, ref, what="", dense=False):
    g = to_np(gpu).reshape(np.shape(ref))
    r = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(g)), what + ": non-finite gradient"
    err = np.abs(g - r)
    stats = {"what": what, "n": int(err.size)}
    if err.size == 0:
        return stats
    if dense:
        bound = 1e-3 * (1.0 + np.abs(r))
    else:
        rms = float(np.sqrt(np.mean(r * r)))
        bound = np.maximum(GRAD_SPACINGS * bf16_spacing(r), GRAD_RMS_FRAC * rms)
        bound = np.maximum(bound, np.finfo(np.float32).tiny)
    worst = float((err / bound).max())
    denom = float(np.abs(r).sum())
    mean_rel = float(err.sum()) / denom if denom > 0 else float(err.sum())
    stats.update({"max_abs": float(err.max()), "max_abs_over_bound": worst,
                  "mean_rel": mean_rel})
    log = os.environ.get("SINKATTN_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps(stats) + "\n")
    assert worst <= 1.0, "%s: max err %.3g over its bound (x%.2f)" % (what, float(err.max()),
                                                                      worst)
    if not dense:
        assert mean_rel <= GRAD_MEAN_REL, "%s: mean_rel %.3g" % (what, mean_rel)
    return stats
