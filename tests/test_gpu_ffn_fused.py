"""The one-launch expert FFN (moe_expert_ffn_fused) against the two-launch
path and the oracle.

Both paths run the same tiles with the same arithmetic, so h, y_perm, y and
the saved fp32 g|u must agree bit for bit; sampled rows are also checked
against the oracle's fp64 per-row FFN.  The shapes give ragged row tiles,
experts with no rows (their GEMM-2 tiles have nothing to wait for), many
small groups, and more row tiles than SMs (CTAs that run GEMM-1 and GEMM-2
tiles of several row tiles).
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

# name, T, d, E, k, I, experts forced empty
CASES = [
    ("ragged", 300, 256, 6, 2, 256, 0),
    ("empty_experts", 1000, 512, 24, 4, 128, 5),
    ("many_groups", 2048, 256, 64, 6, 384, 3),
    ("many_row_tiles", 20000, 256, 8, 2, 128, 0),
]


def _layers(name, T, d, E, k, I, n_empty, backward=False):
    w = W.Workload(name, T, d, E, k, I, 2.5, vision_frac=0.3)
    inp = W.make_inputs(w, device="cuda")
    if n_empty:
        inp["bias"][:, :n_empty] = -10.0   # these experts get no slot
    weights = dict(W_g=inp["W_g"], W13=inp["W13"], W2=inp["W2"])
    D = Dims(T, d, E, k, I)
    out = []
    for fused in (True, False):
        layer = MoELayer(D, weights, w.rho, w.clamp, backward=backward, fused_ffn=fused)
        if layer.gu_save is not None:
            layer.gu_save.zero_()   # its padding rows (past R in the last block) stay unwritten
        layer.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"])
        out.append(layer)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    return w, inp, out


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_ffn_equals_two_launches(case):
    w, inp, (lf, lu) = _layers(*case)
    assert lf.fused_ffn and not lu.fused_ffn
    if case[6]:
        assert int(cpu(lf.counts)[: case[6]].sum()) == 0
    assert torch.equal(lf.ids, lu.ids)
    for name in ("h_perm", "y_perm", "y"):
        a, b = getattr(lf, name), getattr(lu, name)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name
    # sampled rows against the oracle's per-row FFN
    rng = np.random.default_rng(7)
    R = w.S + w.T
    rows = np.sort(rng.choice(R, size=min(64, R), replace=False)).astype(np.int64)
    rt = cpu(lf.row_token).numpy()[rows].astype(np.int64)
    offs = cpu(lf.offsets).numpy()
    grp = (np.searchsorted(offs, rows, side="right") - 1).astype(np.int32)
    rw = np.ones(len(rows))
    routed = rows < w.S
    rw[routed] = np64(lf.row_weight)[rows[routed]]
    h_ref, y_ref = oracle.expert_rows(cpu(inp["x"]), cpu(inp["W13"]), cpu(inp["W2"]), rt, grp, rw,
                                      w.clamp)
    ridx = torch.from_numpy(rows).cuda()
    assert_close_rounded(lf.h_perm[ridx], h_ref, f"{w.name} h rows")
    assert_close_rounded(lf.y_perm[ridx], y_ref, f"{w.name} y_perm rows")


def test_fused_ffn_saves_the_same_gu_for_the_backward():
    w, inp, (lf, lu) = _layers("gu_save", 700, 256, 8, 2, 256, 1, backward=True)
    assert lf.gu_save is not None
    assert torch.equal(lf.gu_save.view(torch.int32), lu.gu_save.view(torch.int32))
    dY = W.normal_bf16((w.T, w.d), 1.0, 0, "dY_fused", "cuda")
    for layer in (lf, lu):
        layer.backward(dY)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    assert torch.equal(lf.dX.view(torch.int16), lu.dX.view(torch.int16))
    assert torch.equal(lf.dW13, lu.dW13)


@pytest.mark.parametrize("stall", [0, 5])
def test_fused_ffn_wait_times_out_and_context_stays_usable(stall):
    # the GEMM-2 tiles of one row tile wait for a GEMM-1 release that never
    # comes: their bounded waits give up, the call reports MOE_ERR_TIMEOUT,
    # and the next calls on the same context give the usual results
    w, inp, (lf, lu) = _layers("stall", 1000, 256, 6, 2, 256, 0)
    D = lf.dims
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    h = torch.zeros_like(lf.h_perm)
    y = torch.zeros_like(lf.y_perm)
    _lib.moe_selftest_ffn_fused_stall(lf.x_perm, lf.offsets, D.E + 1, D.R, inp["W13"], inp["W2"],
                                      lf.row_weight, D.S, D.d, D.I, lf.clamp, h, y, lf.ws, stall,
                                      1 << 20)
    assert _lib.moe_last_device_status() == _lib.MOE_ERR_TIMEOUT
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    # every GEMM-1 tile ran: h is complete
    assert torch.equal(h.view(torch.int16), lu.h_perm.view(torch.int16))
    # the context is usable: the one-launch call again, bit-identical to the
    # two launches
    lf.experts()
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    assert torch.equal(lf.y_perm.view(torch.int16), lu.y_perm.view(torch.int16))
