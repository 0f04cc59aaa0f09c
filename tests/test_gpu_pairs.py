"""2-SM pairs of the grouped matmuls (tcgen05.mma.cta_group::2) against the
oracle, and against the single-SM form of the same matmuls.

The cases hold many rows per expert, so every matmul that may pair does:
expert GEMM 1 and 2, dgrad 2, dgrad 1 (row-grouped: pairs of 128-row tiles of
one expert, with ragged last tiles and pairs whose second tile lies past the
expert's rows) and both weight gradients (pairs of 128-row output tiles over
a ragged contraction of each expert's rows).
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_04_gb300 import _lib
from moe_expert_layer_04_gb300 import workloads as W
from moe_expert_layer_04_gb300.layer import Dims, MoELayer
from tests.helpers import assert_close, assert_close_rounded, cpu, np64

pytestmark = pytest.mark.gpu

CASES = {
    # 4 groups (3 routed + shared) of ~2000-3000 rows: odd and even tile counts
    "pairs_E3": W.Workload("pairs_E3", 3000, 256, 3, 2, 256, 2.5, vision_frac=0.3),
    # skewed load, d = 512: two column tiles per row pair in GEMM 2 / dgrad 1
    "pairs_skew": W.Workload("pairs_skew", 2600, 512, 4, 2, 128, 2.5, zipf_s=1.1),
}

OUTPUTS = ("h_perm", "y_perm", "y", "dX", "dW_g", "dW13", "dW2", "dlogits", "dweights")


def run(w, inp, mask, recompute):
    prev = _lib.moe_set_gemm_pairs(mask)
    try:
        layer = MoELayer(Dims(w.T, w.d, w.E, w.k, w.I),
                         dict(W_g=inp["W_g"], W13=inp["W13"], W2=inp["W2"]), w.rho, w.clamp,
                         backward=True, recompute=recompute)
        layer.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"])
        layer.backward(inp["dY"], want_dlogits=True, want_dweights=True)
        torch.cuda.synchronize()
        assert _lib.moe_last_device_status() == _lib.MOE_OK
    finally:
        _lib.moe_set_gemm_pairs(prev)
    return layer


@pytest.mark.parametrize("name,recompute", [("pairs_E3", False), ("pairs_E3", True),
                                            ("pairs_skew", False)])
def test_pairs_against_oracle_and_single_sm(name, recompute):
    w = CASES[name]
    inp = W.make_inputs(w, device="cuda", with_dy=True)
    lp = run(w, inp, _lib.MOE_PAIR_ALL, recompute)
    x, Wg, W13, W2, dY = (cpu(inp[k]) for k in ("x", "W_g", "W13", "W2", "dY"))
    off = None if inp["logit_offset"] is None else cpu(inp["logit_offset"])
    D = lp.dims
    offs = cpu(lp.offsets).numpy()
    counts = np.diff(offs)
    # every group holds several pairs of row tiles, some with a ragged end
    assert counts.min() >= 256 and np.any(counts % 256 != 0)

    # forward rows and the backward against the oracle
    rt = cpu(lp.row_token).numpy().astype(np.int64)
    grp = np.repeat(np.arange(D.E + 1), counts).astype(np.int32)
    rw = np.ones(D.R)
    rw[: D.S] = np64(lp.row_weight)
    h_ref, y_ref = oracle.expert_rows(x, W13, W2, rt, grp, rw, w.clamp)
    if not recompute:
        assert_close_rounded(lp.h_perm, h_ref, f"{name} h")
    assert_close_rounded(lp.y_perm, y_ref, f"{name} y_perm")
    ref = oracle.layer_backward(x, Wg, W13, W2, dY, cpu(inp["bias"]), w.k, w.rho, w.clamp,
                                is_vision=cpu(inp["is_vision"]), offset=off)
    assert_close(lp.dX, ref["dX"], f"{name} dX")
    assert_close(lp.dlogits, ref["dz"], f"{name} dlogits")
    for e in range(D.E + 1):
        rows = np.arange(offs[e], offs[e + 1])
        g = oracle.expert_wgrad(x, W13, W2, dY, e, rt[rows], rw[rows], w.clamp, store_bf16=True)
        assert_close(lp.dW13[e], g["dW13"], f"{name} dW13[{e}]")
        assert_close(lp.dW2[e], g["dW2"], f"{name} dW2[{e}]")

    # the single-SM form of the same matmuls on the same inputs
    l1 = run(w, inp, 0, recompute)
    for k in OUTPUTS:
        a, b = getattr(lp, k), getattr(l1, k)
        if recompute and k == "h_perm":
            continue
        if torch.equal(a, b):
            continue
        ad, bd = a.double(), b.double()
        diff = (ad - bd).abs()
        if a.dtype == torch.bfloat16:
            # a different fp32 summation order may move a rounded output by one
            # bf16 step
            assert bool((diff <= bd.abs() * 2.0 ** -7 + 1e-30).all()), \
                f"{name} {k}: pair vs single-SM differ by more than one bf16 step"
        else:
            d = diff.max().item()
            assert d <= 1e-5 * max(bd.abs().max().item(), 1.0), \
                f"{name} {k}: pair vs single-SM max diff {d:.3e}"
