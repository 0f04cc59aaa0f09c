"""Shared helpers of the GPU parity tests: tolerances and comparisons."""
import numpy as np
import torch

# Tolerance of floating-point outputs and gradients (bf16 inputs, fp32
# accumulation): relative Frobenius error and max-abs error.
REL_FRO = 1e-2
MAX_ABS = 5e-2
# Routing weights: relative error.
W_RTOL = 1e-6


def np64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().double().cpu().numpy()
    return np.asarray(t, dtype=np.float64)


def errors(got, ref):
    g, r = np64(got), np64(ref)
    diff = g - r
    rel = np.linalg.norm(diff) / max(np.linalg.norm(r), 1e-30)
    mabs = float(np.max(np.abs(diff))) if diff.size else 0.0
    return rel, mabs


def assert_close(got, ref, what, rel_fro=REL_FRO, max_abs=MAX_ABS):
    rel, mabs = errors(got, ref)
    assert np.all(np.isfinite(np64(got))), f"{what}: non-finite values"
    assert rel <= rel_fro and mabs <= max_abs, \
        f"{what}: rel Frobenius {rel:.3e} (<= {rel_fro}), max abs {mabs:.3e} (<= {max_abs})"
    return rel, mabs


def cpu(t):
    return t.detach().cpu()
