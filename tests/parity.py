"""Shared comparison helpers for the GPU parity tests (tests only).

Tolerances (the accuracy bar for bf16 output): attention output max |err| <= 2e-2
and mean |err| <= 2e-3 against the float64 oracle; LSE relative error <= 1e-3
where finite; -inf rows must match exactly.  Integer/index work is bit-exact.
"""

import numpy as np
import torch

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_REL = 1e-3


def assert_attn_close(o_gpu: torch.Tensor, lse_gpu: torch.Tensor, o_ref: np.ndarray, lse_ref: np.ndarray,
                      what: str = ""):
    og = o_gpu.float().cpu().numpy().reshape(o_ref.shape)
    lg = lse_gpu.float().cpu().numpy().reshape(lse_ref.shape)
    ninf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), ninf_ref), f"{what}: -inf rows differ"
    assert np.isfinite(og).all(), f"{what}: non-finite output"
    err = np.abs(og - o_ref)
    assert err.max() <= O_MAX_ABS, f"{what}: max |O err| {err.max():.3e}"
    assert err.mean() <= O_MEAN_ABS, f"{what}: mean |O err| {err.mean():.3e}"
    assert (og[ninf_ref] == 0).all(), f"{what}: empty rows must be 0"
    fin = ~ninf_ref
    if fin.any():
        rel = np.abs(lg[fin] - lse_ref[fin]) / np.maximum(np.abs(lse_ref[fin]), 1e-6)
        assert rel.max() <= LSE_REL, f"{what}: LSE rel err {rel.max():.3e}"
    return float(err.max()), float(err.mean())
