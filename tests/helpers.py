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


def round_bf16(a):
    """Nearest bf16 values (torch's cast) of a float64 array, as float64."""
    import torch as _t
    return _t.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).to(_t.bfloat16).double().numpy()


def check_mx_wgrad(got_dW2, got_dW13, x, W13e, W2e, dY, row_tok, row_w, clamp, h_gpu, what):
    """An expert's MX weight gradients (operands quantised along its rows):
    stage-wise, dW2 against the oracle's row-quantised matmul of dY and the
    GPU's own MX h (w h~ stored in bf16), which leaves only the fp32 sums
    (tight bound); end to end, dW13 and dW2 against the oracle's MX weight
    gradients, where the ~0.2 % of h~ codes that sit one E4M3 step apart (fp32
    vs fp64 SwiGLU) move dW2's terms (the spec float tolerance), and a
    few [dg|du] elements round to bf16 one step apart (fp32 vs fp64 values),
    where one step can move an E4M3 code or a block's scale: dW13's relative
    Frobenius error stays tight, its entries within 0.5 % of the largest."""
    import oracle
    dyr = dY.double().numpy()[row_tok]
    stage2 = oracle.mx_rows_matmul(dyr, round_bf16(row_w[:, None] * h_gpu))
    tol = lambda ref, f: max(5e-2, f * float(np.abs(ref).max()))
    assert_close(got_dW2, stage2, f"{what} dW2 (stage-wise)", rel_fro=1e-4,
                 max_abs=tol(stage2, 1e-4))
    ref = oracle.expert_wgrad_mx(x, W13e, W2e, dY, row_tok, row_w, clamp)
    assert_close(got_dW13, ref["dW13"], f"{what} dW13", rel_fro=1e-3,
                 max_abs=tol(ref["dW13"], 5e-3))
    assert_close(got_dW2, ref["dW2"], f"{what} dW2", max_abs=tol(ref["dW2"], 1e-2))

