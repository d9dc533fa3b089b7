"""Shared helpers for the GPU parity tests (CUDA path vs. the fp64 oracle)."""
import functools

import numpy as np
import torch

# Parity bar: max |err| <= 1e-2 on BF16 outputs and <= 1e-3 on FP32 LSE.
# Above |out| = 1 the output bar scales with the magnitude: a BF16 value in
# [2, 4) has an ulp of 1.56e-2, so a one-ulp rounding difference (fp32 result
# rounded vs. the exact value rounded) cannot meet an absolute 1e-2 there.
OUT_TOL = 1e-2
LSE_TOL = 1e-3


@functools.lru_cache(maxsize=1)
def built_library():
    from ragged_softmax_attention_gb300 import build
    path = build.build()
    import ragged_softmax_attention_gb300 as fw
    fw.load_library(path)
    return fw


def to_device(inp: dict, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    """Element-wise comparison; rows with -inf LSE must match exactly (zero output, -inf)."""
    o = out_gpu.float().cpu().numpy().reshape(out_ref.shape).astype(np.float64)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    diff = np.abs(o - out_ref)
    err = diff.max() if o.size else 0.0
    bound = OUT_TOL * np.maximum(1.0, np.abs(out_ref))
    worst = (diff / bound).max() if o.size else 0.0
    assert worst <= 1.0, f"{what}: max |out err| = {err:.3e} ({worst:.2f} x the magnitude-scaled bar)"
    if lse_gpu is not None:
        l = lse_gpu.float().cpu().numpy().reshape(lse_ref.shape).astype(np.float64)
        ninf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(l), ninf_ref), f"{what}: -inf LSE rows differ"
        if (~ninf_ref).any():
            lerr = np.abs(l[~ninf_ref] - lse_ref[~ninf_ref]).max()
            assert lerr <= LSE_TOL, f"{what}: max |lse err| = {lerr:.3e}"
        return err, (np.abs(l[~ninf_ref] - lse_ref[~ninf_ref]).max() if (~ninf_ref).any() else 0.0)
    return err, None
