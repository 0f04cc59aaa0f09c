"""The MXFP8 backward (moe_mx_quantize_t, moe_backward_mx,
moe_expert_ffn_backward_mx) against the oracle.

The transposed weight copies are integer results of the quantisation rule and
must match the oracle's quantiser bit for bit.  The gradients are float
results compared with the oracle's fp64 MX backward: the layer's dX, dw and
dz with oracle.layer_backward_mx, the weight gradients with fp64 sums over
the oracle's MX h and pre-quantisation [dg | du] of the same rows (the GPU
rounds both operands to bf16 and sums in fp32), the expert-level call's rows
with oracle.expert_rows_mx_backward.  The GPU quantises [dg | du] from fp32
values and the oracle from fp64 ones, so a code can sit one E4M3 step apart
where the two straddle a rounding boundary; such flips are rare and move dX
by far less than the tolerance.  Sizes give ragged row tiles, experts without
rows, two scale chunks in dgrad 2's contraction (d = 1024) and a partial one
in dgrad 1's (2I = 512), the 256-wide forward tiles that save g|u, and the
recompute path."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_04_gb300 import _lib
from moe_expert_layer_04_gb300 import workloads as W
from moe_expert_layer_04_gb300.layer import Dims, MoELayer
from tests.helpers import assert_close, check_mx_wgrad, cpu, np64

pytestmark = pytest.mark.gpu

PAD = 0xAA


@pytest.mark.parametrize("G,R,C", [(2, 96, 40), (3, 256, 72), (1, 4096, 64)])
def test_mx_quantize_t_bit_exact(G, R, C):
    g = torch.Generator().manual_seed(G * 131 + R + C)
    x = torch.randn(G, R, C, generator=g, dtype=torch.float64)
    x *= torch.exp(torch.randn(G, 1, C, generator=g, dtype=torch.float64) * 3)
    x[0, :32, 0] = 0.0                                  # a zero block
    x[0, 32:64, 1] = 2.0 ** -131                        # scale clamps at 2^-127
    xb = x.to(torch.bfloat16)
    q = torch.empty(G * C, R, dtype=torch.uint8, device="cuda")
    sf = torch.full((G * C, _lib.moe_mx_sf_pitch(R)), PAD, dtype=torch.uint8, device="cuda")
    _lib.moe_mx_quantize_t(xb.cuda(), G, R, C, q, sf)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    q, sf = cpu(q).numpy(), cpu(sf).numpy()
    for i in range(G):
        q_ref, sf_ref = oracle.mx_quantize(xb[i].t().contiguous())
        assert np.array_equal(q[i * C:(i + 1) * C], q_ref)
        assert np.array_equal(sf[i * C:(i + 1) * C, : R // 32], sf_ref)
    assert np.all(sf[:, R // 32:] == PAD)


@pytest.mark.parametrize("G,R,C", [(1, 128, 128), (2, 256, 384)])
def test_mx_quantize_both_bit_exact(G, R, C):
    """Both orientations in one pass: each equal, bit for bit, to the
    oracle's quantisation of the rows and of the columns."""
    g = torch.Generator().manual_seed(G * 977 + R + C)
    x = torch.randn(G, R, C, generator=g, dtype=torch.float64)
    x *= torch.exp(torch.randn(G, R, 1, generator=g, dtype=torch.float64) * 2)
    x *= torch.exp(torch.randn(G, 1, C, generator=g, dtype=torch.float64) * 2)
    x[0, :32, :32] = 0.0                                # zero blocks both ways
    x[0, 32:64, 0:32] = 2.0 ** -131                     # scales clamp at 2^-127
    x[0, 64, 64:96] = 1.9 * 2.0 ** 3                    # a row block that saturates
    xb = x.to(torch.bfloat16)
    dev = dict(dtype=torch.uint8, device="cuda")
    q = torch.empty(G * R, C, **dev)
    sf = torch.full((G * R, _lib.moe_mx_sf_pitch(C)), PAD, **dev)
    qt = torch.empty(G * C, R, **dev)
    sft = torch.full((G * C, _lib.moe_mx_sf_pitch(R)), PAD, **dev)
    _lib.moe_mx_quantize_both(xb.cuda(), G, R, C, q, sf, qt, sft)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    q_ref, sf_ref = oracle.mx_quantize(xb.reshape(G * R, C))
    assert np.array_equal(cpu(q).numpy(), q_ref)
    assert np.array_equal(cpu(sf).numpy()[:, : C // 32], sf_ref)
    qt_ref, sft_ref = oracle.mx_quantize(xb.transpose(1, 2).reshape(G * C, R))
    assert np.array_equal(cpu(qt).numpy(), qt_ref)
    assert np.array_equal(cpu(sft).numpy()[:, : R // 32], sft_ref)
    assert np.all(cpu(sf).numpy()[:, C // 32:] == PAD)
    assert np.all(cpu(sft).numpy()[:, R // 32:] == PAD)


def _run(name, T, d, E, k, I, n_empty=0, recompute=False):
    w = W.Workload(name, T, d, E, k, I, 2.5, vision_frac=0.3)
    inp = W.make_inputs(w, device="cuda", with_dy=True)
    if n_empty:
        inp["bias"][:, :n_empty] = -10.0
    weights = dict(W_g=inp["W_g"], W13=inp["W13"], W2=inp["W2"])
    layer = MoELayer(Dims(T, d, E, k, I), weights, w.rho, w.clamp, mx=True, backward=True,
                     recompute=recompute)
    layer.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"])
    layer.backward(inp["dY"], want_dlogits=True, want_dweights=True)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    return w, inp, layer


def _rows_meta(layer, w):
    offs = cpu(layer.offsets).numpy()
    rt = cpu(layer.row_token).numpy().astype(np.int64)
    grp = np.repeat(np.arange(w.E + 1), np.diff(offs)).astype(np.int32)
    rw = np.ones(w.S + w.T)
    rw[: w.S] = np64(layer.row_weight)
    return offs, rt, grp, rw


def _check_expert_wgrads(w, inp, layer, experts):
    """Each listed expert's MX weight gradients against the oracle
    (tests.helpers.check_mx_wgrad); an expert without rows gets zeros."""
    offs, rt, grp, rw = _rows_meta(layer, w)
    x, dY = cpu(inp["x"]), cpu(inp["dY"])
    for e in experts:
        rows = np.arange(offs[e], offs[e + 1])
        ex = torch.tensor([e]).cuda()
        if len(rows) == 0:
            assert float(layer.dW13[e].abs().max()) == 0.0
            assert float(layer.dW2[e].abs().max()) == 0.0
            continue
        ridx = torch.from_numpy(rows).cuda()
        h_gpu = oracle.mx_dequantize(cpu(layer.h_q[ridx]).numpy(),
                                     cpu(layer.h_sf[ridx]).numpy()[:, : w.I // 32])
        check_mx_wgrad(layer.dW2[e], layer.dW13[e], x, cpu(inp["W13"][ex][0]),
                       cpu(inp["W2"][ex][0]), dY, rt[rows], rw[rows], w.clamp, h_gpu,
                       f"{w.name} expert {e} ({len(rows)} rows)")


# name, T, d, E, k, I, experts forced empty, recompute, tokens checked (None: all)
CASES = [
    ("ragged", 300, 256, 6, 2, 128, 0, False, None),
    ("ragged_recompute", 300, 256, 6, 2, 128, 0, True, None),
    ("two_scale_chunks", 700, 1024, 5, 2, 256, 0, False, None),
    ("empty_experts", 500, 512, 16, 4, 128, 5, False, None),
    # many rows per expert: the 256-wide forward tiles save g|u
    ("wide_tiles", 6000, 512, 4, 2, 256, 0, False, 64),
    ("wide_tiles_recompute", 6000, 512, 4, 2, 256, 0, True, 64),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_mx_layer_backward_parity(case):
    name, T, d, E, k, I, n_empty, rec, n_tok = case
    w, inp, layer = _run(name, T, d, E, k, I, n_empty, rec)
    x, Wg, W13, W2, dY = (cpu(inp[n]) for n in ("x", "W_g", "W13", "W2", "dY"))
    off = None if inp["logit_offset"] is None else cpu(inp["logit_offset"])
    vis = cpu(inp["is_vision"])
    bias = cpu(inp["bias"])
    fwd = oracle.layer_forward(x, Wg, W13, W2, bias, k, w.rho, w.clamp, is_vision=vis,
                               offset=off)
    np.testing.assert_array_equal(fwd["ids"], cpu(layer.ids).numpy())
    toks = (np.arange(T) if n_tok is None else
            np.sort(np.random.default_rng(5).choice(T, size=n_tok, replace=False)))
    ref = oracle.layer_backward_mx(x, Wg, W13, W2, dY, bias, k, w.rho, w.clamp, is_vision=vis,
                                   offset=off, tok=toks.astype(np.int64))
    tt = torch.from_numpy(toks).cuda()
    assert_close(layer.dX[tt], ref["dX"], f"{name} dX")
    assert_close(layer.dweights[tt], ref["dw"], f"{name} dw",
                 max_abs=5e-2 * max(1, np.abs(ref["dw"]).max() / 10))
    assert_close(layer.dlogits[tt], ref["dz"], f"{name} dlogits")
    if n_tok is None:
        assert_close(layer.dW_g, oracle.gate_wgrad_rows(x, ref["dz"], np.arange(E)),
                     f"{name} dW_g")
    counts = np.diff(cpu(layer.offsets).numpy())
    nonempty = [e for e in range(E) if counts[e] > 0]
    experts = sorted({min(nonempty, key=lambda e: counts[e]), E} |
                     ({max(nonempty, key=lambda e: counts[e])} if T <= 1000 else set()) |
                     ({0} if n_empty else set()))
    _check_expert_wgrads(w, inp, layer, experts)
    # the backward's weight copies, one expert bit for bit
    e = nonempty[0]
    q, sf = oracle.mx_quantize(cpu(inp["W2"][e]).t().contiguous())
    assert np.array_equal(cpu(layer.W2t_q[e * I:(e + 1) * I]).numpy(), q)
    assert np.array_equal(cpu(layer.W2t_sf[e * I:(e + 1) * I]).numpy()[:, : d // 32], sf)
    q, sf = oracle.mx_quantize(cpu(inp["W13"][e]).t().contiguous())
    assert np.array_equal(cpu(layer.W13t_q[e * d:(e + 1) * d]).numpy(), q)
    assert np.array_equal(cpu(layer.W13t_sf[e * d:(e + 1) * d]).numpy()[:, : 2 * I // 32], sf)


@pytest.mark.parametrize("recompute", [False, True])
def test_mx_expert_backward_rows(recompute):
    """moe_expert_ffn_backward_mx on the layer's rows: dX_perm and dw rows
    against the oracle's rows, and the weight gradients equal to the
    layer-level call's bit for bit (the same kernels on the same rows)."""
    T, d, E, k, I = 400, 512, 6, 2, 256
    w, inp, layer = _run("expert_rows", T, d, E, k, I, recompute=recompute)
    D = layer.dims
    G, R = E + 1, D.R
    rtt = layer.row_token.long()
    x_perm = inp["x"][rtt].contiguous()
    dY_perm = inp["dY"][rtt].contiguous()
    dYq = torch.empty(R, d, dtype=torch.uint8, device="cuda")
    dYsf = torch.empty(R, _lib.moe_mx_sf_pitch(d), dtype=torch.uint8, device="cuda")
    _lib.moe_mx_quantize(dY_perm, R, d, dYq, dYsf)
    dX_perm = torch.empty(R, d, dtype=torch.bfloat16, device="cuda")
    dw_rows = torch.empty(D.S, dtype=torch.float32, device="cuda")
    dW13 = torch.empty_like(layer.dW13)
    dW2 = torch.empty_like(layer.dW2)
    ws = torch.empty(_lib.moe_expert_bwd_mx_workspace_size(G, R, d, I, recompute),
                     dtype=torch.uint8, device="cuda")
    _lib.moe_expert_ffn_backward_mx(dict(
        G=G, max_rows=R, S=D.S, d=d, I=I, clamp=w.clamp, offsets=layer.offsets, x_perm=x_perm,
        x_perm_q=layer.x_perm_q, x_perm_sf=layer.x_perm_sf, W13_q=layer.W13_q,
        W13_sf=layer.W13_sf, gu_save=layer.gu_save,
        h_q=None if recompute else layer.h_q, h_sf=None if recompute else layer.h_sf,
        W2t_q=layer.W2t_q, W2t_sf=layer.W2t_sf, W13t_q=layer.W13t_q, W13t_sf=layer.W13t_sf,
        row_weight=layer.row_weight, dY_perm=dY_perm, dY_perm_q=dYq, dY_perm_sf=dYsf,
        dX_perm=dX_perm, dw_rows=dw_rows, dW13=dW13, dW2=dW2, ws=ws))
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    assert torch.equal(dW13, layer.dW13) and torch.equal(dW2, layer.dW2)
    offs, rt, grp, rw = _rows_meta(layer, w)
    ref = oracle.expert_rows_mx_backward(cpu(inp["x"]), cpu(inp["W13"]), cpu(inp["W2"]),
                                         cpu(inp["dY"]), rt, grp, rw, w.clamp)
    assert_close(dX_perm, ref["dx"], "expert rows dX_perm")
    assert_close(dw_rows, ref["dw"][: D.S], "expert rows dw",
                 max_abs=5e-2 * max(1, np.abs(ref["dw"]).max() / 10))
