"""Shared helpers for the GPU parity tests (CUDA path vs. the fp64 oracle).

The parity bar.  The stated bar is max |err| <= 1e-2 on BF16 outputs and
<= 1e-3 on FP32 LSE.  An output element may exceed the absolute 1e-2 only by
what the arithmetic the method prescribes can produce, derived here per
element from the oracle's exact result `ref` and absv (the softmax-weighted
mean of |v| in that output column, computed by the oracle):

  * each probability is rounded before the PV product ("Writing Page
    Attention with PyPTO", section 6.3 casts P to BF16 for the matmul): every
    weight moves by at most the format's unit roundoff u_p relative (BF16:
    2^-8; the FP8-cache path rounds P to FP16: 2^-11), which moves the output
    by at most 2 u_p / (1 - u_p) * absv whether the row sum divides by the
    rounded or the unrounded weights;
  * FP32 scores, exp2 and accumulators: an allowance of 2^-12 * absv;
  * the result is rounded to BF16 (round to nearest even): at most half an
    ulp, u_o = 2^-8 relative to the value rounded.

  bound = max(1e-2, d + u_o * (|ref| + d)),  d = (2 u_p / (1 - u_p) + 2^-12) absv

Every comparison is recorded; the session summary reports how many elements
exceeded the absolute 1e-2 and the worst of them.
"""
import functools

import numpy as np
import torch

OUT_TOL = 1e-2
LSE_TOL = 1e-3
BF16_UNIT = 2.0 ** -8          # unit roundoff of BF16 (8 significant bits)
FP16_UNIT = 2.0 ** -11         # unit roundoff of FP16 (11 significant bits)
FP32_ALLOWANCE = 2.0 ** -12

# Session record: elements compared, elements above the absolute bar, the worst
# one above it (ratio err / 1e-2, err, ref, bound, what).
STATS = {"elements": 0, "above_abs": 0, "worst": None}


@functools.lru_cache(maxsize=1)
def built_library():
    from ragged_softmax_attention_gb300 import build
    path = build.build()
    import ragged_softmax_attention_gb300 as fw
    fw.load_library(path)
    return fw


def to_device(inp: dict, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def out_bound(out_ref, absv, p_unit=BF16_UNIT):
    """Per-element bound on |out - ref| (see the module docstring); the plain
    absolute bar where absv is not given."""
    if absv is None:
        return np.full(np.shape(out_ref), OUT_TOL)
    d = (2.0 * p_unit / (1.0 - p_unit) + FP32_ALLOWANCE) * np.asarray(absv, dtype=np.float64)
    return np.maximum(OUT_TOL, d + BF16_UNIT * (np.abs(out_ref) + d))


def _record(diff, ref, bound, what):
    STATS["elements"] += diff.size
    above = diff > OUT_TOL
    n = int(above.sum())
    if n:
        STATS["above_abs"] += n
        i = np.unravel_index(np.argmax(np.where(above, diff, -1.0)), diff.shape)
        worst = (float(diff[i] / OUT_TOL), float(diff[i]), float(ref[i]), float(bound[i]), what)
        if STATS["worst"] is None or worst[0] > STATS["worst"][0]:
            STATS["worst"] = worst


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what="", absv=None, p_unit=BF16_UNIT):
    """Element-wise comparison; rows with -inf LSE must match exactly (zero output, -inf)."""
    o = out_gpu.float().cpu().numpy().reshape(out_ref.shape).astype(np.float64)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    diff = np.abs(o - out_ref)
    err = diff.max() if o.size else 0.0
    if absv is not None:
        absv = np.asarray(absv).reshape(out_ref.shape)
    bound = out_bound(out_ref, absv, p_unit)
    _record(diff, out_ref, bound, what)
    if o.size:
        i = np.unravel_index(np.argmax(diff / bound), diff.shape)
        assert diff[i] <= bound[i], (f"{what}: |out err| {diff[i]:.3e} at ref {out_ref[i]:.4f} exceeds its bound "
                                     f"{bound[i]:.3e} (max |out err| {err:.3e})")
    if lse_gpu is not None:
        l = lse_gpu.float().cpu().numpy().reshape(lse_ref.shape).astype(np.float64)
        ninf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(l), ninf_ref), f"{what}: -inf LSE rows differ"
        if (~ninf_ref).any():
            lerr = np.abs(l[~ninf_ref] - lse_ref[~ninf_ref]).max()
            assert lerr <= LSE_TOL, f"{what}: max |lse err| = {lerr:.3e}"
        return err, (np.abs(l[~ninf_ref] - lse_ref[~ninf_ref]).max() if (~ninf_ref).any() else 0.0)
    return err, None
