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


def bf16_ulp(v):
    """Spacing of bf16 values at |v| (8 significant bits)."""
    a = np.maximum(np.abs(np64(v)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def assert_close_rounded(got, ref, what, rel_fro=REL_FRO, max_abs=MAX_ABS, max_flip_frac=1e-3):
    """A bf16 intermediate that both sides round from sums taken in a different
    order (fp32 on the GPU, fp64 in the oracle): where the two sums straddle a
    rounding boundary the values sit one bf16 step apart, which for values of
    magnitude 8 or more exceeds the 5e-2 bound.  Each element must lie within
    max(max_abs, one bf16 step of the reference); at most max_flip_frac of the
    elements may exceed max_abs at all; relative Frobenius as usual."""
    g, r = np64(got), np64(ref)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    diff = np.abs(g - r)
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    bound = np.maximum(max_abs, bf16_ulp(r) * (1 + 1e-6))
    worst = float(np.max(diff / bound)) if diff.size else 0.0
    flips = float(np.mean(diff > max_abs)) if diff.size else 0.0
    assert rel <= rel_fro and worst <= 1.0 and flips <= max_flip_frac, \
        (f"{what}: rel Frobenius {rel:.3e} (<= {rel_fro}), worst |diff| / max({max_abs}, one "
         f"bf16 step) {worst:.3f} (<= 1), elements beyond {max_abs}: {flips:.2e}")
    return rel, float(diff.max()) if diff.size else 0.0


def assert_wgrad_bf16_bound(got, a, b, what):
    """got ~ a^T b, where the GPU rounded b (w h~, or [dg | du]) to bf16 and
    summed in fp32: each entry within 2^-8 sum_r |a_r b_r| of the fp64 sum
    (round to nearest moves each term by at most 2^-9 of itself; the rest
    covers the fp32 sums).  An entry may exceed it only where a clamp
    decision sits within fp32 rounding of the bound (a few in 10^4)."""
    want = a.T @ b
    bound = 2.0 ** -8 * (np.abs(a).T @ np.abs(b)) + 1e-6 * float(np.abs(want).max())
    g = np64(got)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    over = np.abs(g - want) > bound
    rel = np.linalg.norm(g - want) / max(np.linalg.norm(want), 1e-30)
    assert rel <= 1e-2 and over.mean() <= 1e-4, \
        f"{what}: rel Frobenius {rel:.3e}, entries beyond the rounding bound {over.mean():.2e}"
