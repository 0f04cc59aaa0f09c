"""The MXFP8 training step at the full 64K-token slice (T = 65536, 384
experts top-6 + shared, d = 4096, I = 2048, Zipf load, recompute), in the
launch configuration the bench times (`mx_fwd_bwd`).

Float outputs are compared on seeded samples the oracle computes one by one:
dX, dlogits and dw of sampled tokens against the oracle's MX layer backward
(tokens whose routing the oracle reproduces; a disagreement is allowed only
at a near-tie of the keys); every entry of the weight gradients of three
routed experts (the coldest non-empty one, the median one and a seeded one,
all their rows through the oracle's MX weight gradients, stage-wise and end
to end); dW_g rows as the oracle's reduction of the GPU's logit
gradients; the backward's transposed weight copies of one expert bit for
bit.  Routing and permutation at this size are checked bit for bit in
test_gpu_fullsize.py (the MX layer runs the same kernels for them)."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_04_gb300 import _lib
from moe_expert_layer_04_gb300 import workloads as W
from moe_expert_layer_04_gb300.layer import Dims, MoELayer
from tests.helpers import assert_close, check_mx_wgrad, cpu, np64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N_TOK = 32


def test_long_slice_mx_training_step():
    w = W.WORKLOADS["long_slice_fwd_bwd"]
    full = W.make_inputs(W.WORKLOADS["full_fwd"], device="cuda")
    dev = {k: full[k] for k in ("W_g", "W13", "W2")}
    host = {k: v.cpu() for k, v in dev.items()}
    del full
    inp = W.make_inputs(w, device="cuda", with_weights=False, with_dy=True)
    D = Dims(w.T, w.d, w.E, w.k, w.I)
    layer = MoELayer(D, dev, w.rho, w.clamp, backward=True, recompute=w.recompute, mx=True)
    layer.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"])
    layer.backward(inp["dY"], want_dlogits=True, want_dweights=True)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK

    x, dY = cpu(inp["x"]), cpu(inp["dY"])
    off = cpu(inp["logit_offset"])
    vis = cpu(inp["is_vision"])
    bias = cpu(inp["bias"])
    tok = np.sort(np.random.default_rng(21).choice(w.T, size=N_TOK, replace=False))
    fwd = oracle.layer_forward(x, host["W_g"], host["W13"], host["W2"], bias, w.k, w.rho,
                               w.clamp, is_vision=vis, offset=off, tok=tok)
    same = np.all(fwd["ids"] == cpu(layer.ids).numpy()[tok], axis=1)
    assert np.all(same | (fwd["margin"] < 1e-5)) and same.sum() >= N_TOK - 2
    tok = tok[same]
    ref = oracle.layer_backward_mx(x, host["W_g"], host["W13"], host["W2"], dY, bias, w.k,
                                   w.rho, w.clamp, is_vision=vis, offset=off, tok=tok)
    tt = torch.from_numpy(tok).cuda()
    assert_close(layer.dX[tt], ref["dX"], "MX dX")
    assert_close(layer.dlogits[tt], ref["dz"], "MX dlogits")
    assert_close(layer.dweights[tt], ref["dw"], "MX dw",
                 max_abs=max(5e-2, 5e-3 * np.abs(ref["dw"]).max()))

    counts = cpu(layer.counts).numpy()
    offs = cpu(layer.offsets).numpy()
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    rest = np.setdiff1d(order[: len(order) // 2], [order[0]])
    experts = [int(order[0]), int(order[len(order) // 2]),
               int(np.random.default_rng(22).choice(rest))]
    # dW_g rows: the oracle's reduction of the GPU's logit gradients
    pick = np.array(experts + [int(order[-1])], np.int32)
    dwg_ref = oracle.gate_wgrad_rows(x, np64(layer.dlogits), pick)
    assert_close(layer.dW_g[torch.from_numpy(pick).long().cuda()], dwg_ref, "MX dW_g rows",
                 max_abs=max(5e-2, 1e-3 * np.abs(dwg_ref).max()))
    # whole MX weight gradients of three routed experts
    rt_all = cpu(layer.row_token).numpy().astype(np.int64)
    rw_all = np64(layer.row_weight)
    for e in experts:
        rows = np.arange(offs[e], offs[e + 1])
        ridx = torch.from_numpy(rows).cuda()
        h_gpu = oracle.mx_dequantize(cpu(layer.h_q[ridx]).numpy(),
                                     cpu(layer.h_sf[ridx]).numpy()[:, : w.I // 32])
        check_mx_wgrad(layer.dW2[e], layer.dW13[e], x, host["W13"][e], host["W2"][e], dY,
                       rt_all[rows], rw_all[rows], w.clamp, h_gpu,
                       f"MX expert {e} ({len(rows)} rows)")
    # the backward's weight copies (quantised along d and 2I) of one expert
    e = experts[1]
    q, sf = oracle.mx_quantize(host["W2"][e].t().contiguous())
    assert np.array_equal(cpu(layer.W2t_q[e * w.I:(e + 1) * w.I]).numpy(), q)
    assert np.array_equal(cpu(layer.W2t_sf[e * w.I:(e + 1) * w.I]).numpy()[:, : w.d // 32], sf)
    q, sf = oracle.mx_quantize(host["W13"][e].t().contiguous())
    assert np.array_equal(cpu(layer.W13t_q[e * w.d:(e + 1) * w.d]).numpy(), q)
    assert np.array_equal(cpu(layer.W13t_sf[e * w.d:(e + 1) * w.d]).numpy()[:, : 2 * w.I // 32],
                          sf)
