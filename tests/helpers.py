"""Shared test helpers: tolerance checks and small conversions."""

import numpy as np
import torch

# Tolerances of the attention outputs against the fp64 oracle.
BF16_MAX_ABS = 2e-2
BF16_REL_RMS = 1e-2
FP32_MAX_ABS = 1e-4


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    denom = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 1.0
    rel_rms = float(np.sqrt(np.mean(diff ** 2)) / max(denom, 1e-30)) if diff.size else 0.0
    return max_abs, rel_rms


def assert_bf16_close(got, ref, what=""):
    max_abs, rel_rms = errors(got, ref)
    assert max_abs <= BF16_MAX_ABS and rel_rms <= BF16_REL_RMS, (
        f"{what}: max_abs={max_abs:.3e} (<= {BF16_MAX_ABS}), rel_rms={rel_rms:.3e} (<= {BF16_REL_RMS})")
    return max_abs, rel_rms


def assert_fp32_close(got, ref, what=""):
    max_abs, _ = errors(got, ref)
    assert max_abs <= FP32_MAX_ABS, f"{what}: max_abs={max_abs:.3e} (<= {FP32_MAX_ABS})"
    return max_abs


def assert_bf16_close_torch(got, ref, what=""):
    """The bf16 tolerance check evaluated on the GPU (large tensors)."""
    import math
    g = got.float()
    r = ref.float()
    d = g - r
    max_abs = float(d.abs().max())
    rel_rms = float(d.pow(2).mean().sqrt()) / max(float(r.pow(2).mean().sqrt()), 1e-30)
    assert math.isfinite(max_abs) and max_abs <= BF16_MAX_ABS and rel_rms <= BF16_REL_RMS, (
        f"{what}: max_abs={max_abs:.3e} (<= {BF16_MAX_ABS}), rel_rms={rel_rms:.3e} (<= {BF16_REL_RMS})")
    return max_abs, rel_rms
