"""GPU path (through the C ABI) against the CPU oracle on the same seeded inputs.

Index work (expert ids, permutation, counts, offsets) must match bit for bit;
routing weights within 1e-6 relative; float outputs and gradients within
relative Frobenius 1e-2 and max-abs 5e-2.  Routing is checked stage-wise: the
oracle routes the GPU's own fp32 logits, since fp32 GEMM accumulation order
can move a logit by an ulp and legitimately flip a near-tie.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_04_gb300 import _lib
from moe_expert_layer_04_gb300 import workloads as W
from moe_expert_layer_04_gb300.layer import MOE_ROUTE_HASH, MOE_ROUTE_TOPK, Dims, MoELayer
from tests.helpers import W_RTOL, assert_close, assert_close_rounded, cpu, np64

pytestmark = pytest.mark.gpu

# (name, workload) -- several tiles per group and ragged tails
CASES = {
    "tiny": W.WORKLOADS["tiny_fwd"],
    "mid_I192": W.Workload("mid_I192", 320, 256, 24, 4, 192, 2.5, vision_frac=0.25),
    "mid_skew": W.Workload("mid_skew", 520, 384, 12, 3, 256, 2.5, zipf_s=1.1),
    # many rows per expert: the weight gradients run as two-CTA clusters sharing B
    "paired": W.Workload("paired", 2048, 256, 6, 2, 256, 2.5, vision_frac=0.3),
    # the largest expert count: 1025 GEMM groups, most with 0..4 rows
    "max_groups": W.Workload("max_groups", 300, 128, 1024, 8, 64, 2.5, vision_frac=0.3),
    # one token routed to every expert (k = E)
    "one_token_all_experts": W.Workload("one_token_all_experts", 1, 128, 4, 4, 64, 1.0),
}


def make_layer(w, backward=False, recompute=False, seed_inputs=None):
    inp = W.make_inputs(w, device="cuda", with_dy=backward)
    weights = dict(W_g=inp["W_g"], W13=inp["W13"], W2=inp["W2"])
    layer = MoELayer(Dims(w.T, w.d, w.E, w.k, w.I), weights, w.rho, w.clamp, backward=backward,
                     recompute=recompute)
    return layer, inp


def test_gate_logits_and_route_stagewise():
    for name, w in CASES.items():
        layer, inp = make_layer(w)
        vis = inp["is_vision"]
        layer.route(inp["x"], inp["bias"], vis, inp["logit_offset"])
        torch.cuda.synchronize()
        z_ref = oracle.gate_logits(cpu(inp["x"]), cpu(inp["W_g"]),
                                   offset=None if inp["logit_offset"] is None else cpu(inp["logit_offset"]))
        z = np64(layer.logits)
        assert np.max(np.abs(z - z_ref)) < 1e-4 * max(1.0, np.abs(z_ref).max()), name
        ids, wts, s, _ = oracle.route(z, cpu(inp["bias"]), w.k, w.rho, is_vision=cpu(vis))
        np.testing.assert_array_equal(cpu(layer.ids).numpy(), ids, err_msg=name)
        np.testing.assert_array_equal(np64(layer.scores_sel), s, err_msg=name)
        np.testing.assert_allclose(np64(layer.weights), wts, rtol=W_RTOL, atol=0, err_msg=name)


@pytest.mark.parametrize("T,E,k", [(1, 4, 4), (200, 40, 6), (97, 384, 6), (33, 1000, 8),
                                   (64, 16, 1), (50, 32, 32)])
def test_route_logits_exact(T, E, k):
    z = W.random_logits(T, E, 2.0, seed=T * 7 + E).cuda()
    # plant exact ties: equal logits in pairs so equal keys must go to the lower id
    z[:, 1::2] = z[:, 0::2][:, : z[:, 1::2].shape[1]]
    g = torch.Generator().manual_seed(E)
    bias = (torch.rand(2, E, generator=g) * 0.2 - 0.1).cuda()
    bias[:, 1::2] = bias[:, 0::2][:, : bias[:, 1::2].shape[1]]
    vis = (torch.arange(T) % 3 == 0).to(torch.uint8).cuda()
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    wt = torch.empty(T, k, dtype=torch.float32, device="cuda")
    s = torch.empty(T, k, dtype=torch.float32, device="cuda")
    _lib.moe_route_logits(z, bias, vis, None, None, T, E, k, 2.5, MOE_ROUTE_TOPK, ids, wt, s)
    torch.cuda.synchronize()
    r_ids, r_w, r_s, _ = oracle.route(np64(z), cpu(bias), k, 2.5, is_vision=cpu(vis))
    np.testing.assert_array_equal(cpu(ids).numpy(), r_ids)
    np.testing.assert_array_equal(np64(s), r_s)
    np.testing.assert_allclose(np64(wt), r_w, rtol=W_RTOL, atol=0)


def test_route_all_tied_uses_exact_fallback():
    # every key equal: more than 32 experts sit in the exact-key window
    T, E, k = 16, 96, 5
    z = torch.zeros(T, E, device="cuda")
    bias = torch.zeros(2, E, device="cuda")
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    wt = torch.empty(T, k, dtype=torch.float32, device="cuda")
    s = torch.empty(T, k, dtype=torch.float32, device="cuda")
    _lib.moe_route_logits(z, bias, None, None, None, T, E, k, 2.5, MOE_ROUTE_TOPK, ids, wt, s)
    torch.cuda.synchronize()
    assert cpu(ids).tolist() == [list(range(k))] * T
    assert np.all(np64(wt) == np.float32(2.5 / k))


def test_route_hash_exact():
    T, E, k, V = 300, 384, 6, W.VOCAB
    z = W.random_logits(T, E, 1.5, seed=11).cuda()
    tab = W.tid2eid_table(V, E, k, 0, "cuda")
    iid = W.zipf_input_ids(T, V, 1.0, 0, "cuda")
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    wt = torch.empty(T, k, dtype=torch.float32, device="cuda")
    s = torch.empty(T, k, dtype=torch.float32, device="cuda")
    bias = torch.zeros(2, E, device="cuda")
    _lib.moe_route_logits(z, bias, None, iid, tab, T, E, k, 2.5, MOE_ROUTE_HASH, ids, wt, s)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    r_ids, r_w, r_s, _ = oracle.route(np64(z), cpu(bias), k, 2.5, mode=1, input_ids=cpu(iid),
                                      tid2eid=cpu(tab))
    np.testing.assert_array_equal(cpu(ids).numpy(), r_ids)
    np.testing.assert_array_equal(np64(s), r_s)
    np.testing.assert_allclose(np64(wt), r_w, rtol=W_RTOL, atol=0)


# the last case has more than 2048 chunks of 256 slots, so each thread of the
# chunk scan takes more chunks than it holds in registers
@pytest.mark.parametrize("T,E,k,skew,d", [(64, 16, 2, 0.0, 128), (1, 4, 3, 0.0, 8),
                                          (2000, 384, 6, 1.1, 64), (700, 50, 5, 2.5, 128),
                                          (5000, 1000, 8, 0.0, 16), (70000, 64, 8, 1.1, 8)])
def test_permute_exact(T, E, k, skew, d):
    ids = W.random_ids(T, E, k, seed=T + E, skew=skew).cuda()
    wts = torch.rand(T, k, device="cuda")
    x = W.normal_bf16((T, d), 1.0, 0, "xp", "cuda")
    S, R = T * k, T * k + T
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 2, dtype=torch.int32, device="cuda")
    row_token = torch.empty(R, dtype=torch.int32, device="cuda")
    slot_row = torch.empty(S, dtype=torch.int32, device="cuda")
    row_w = torch.empty(S, dtype=torch.float32, device="cuda")
    x_perm = torch.empty(R, d, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(_lib.moe_workspace_size(T, 128, E, k, 64, 0), dtype=torch.uint8,
                     device="cuda")
    _lib.moe_permute(ids, wts, x, T, d, E, k, counts, offsets, row_token, slot_row, row_w,
                     x_perm, ws)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    c, o, rt, sr = oracle.permute(cpu(ids).numpy(), E)
    np.testing.assert_array_equal(cpu(counts).numpy(), c)
    np.testing.assert_array_equal(cpu(offsets).numpy()[: E + 1], o)
    assert cpu(offsets).numpy()[E + 1] == R
    np.testing.assert_array_equal(cpu(row_token).numpy()[:S], rt)
    np.testing.assert_array_equal(cpu(row_token).numpy()[S:], np.arange(T))
    np.testing.assert_array_equal(cpu(slot_row).numpy(), sr)
    np.testing.assert_array_equal(cpu(row_w).numpy()[sr], cpu(wts).numpy().ravel())
    xr = cpu(x).view(torch.int16).numpy()
    np.testing.assert_array_equal(cpu(x_perm).view(torch.int16).numpy(),
                                  xr[cpu(row_token).numpy()])


def _rows_meta(layer, w):
    """Per permuted row: token, expert group and routing weight (from the GPU's own routing)."""
    D = layer.dims
    offs = cpu(layer.offsets).numpy()
    rt = cpu(layer.row_token).numpy().astype(np.int64)
    grp = np.repeat(np.arange(D.E + 1), np.diff(offs)).astype(np.int32)
    rw = np.ones(D.R)
    rw[: D.S] = np64(layer.row_weight)
    return rt, grp, rw


@pytest.mark.parametrize("name", list(CASES))
def test_forward_layer(name):
    w = CASES[name]
    layer, inp = make_layer(w)
    y = layer.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"])
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    x, W13, W2 = cpu(inp["x"]), cpu(inp["W13"]), cpu(inp["W2"])
    rt, grp, rw = _rows_meta(layer, w)
    h_ref, y_ref = oracle.expert_rows(x, W13, W2, rt, grp, rw, w.clamp)
    assert_close_rounded(layer.h_perm, h_ref, f"{name} h")
    assert_close_rounded(layer.y_perm, y_ref, f"{name} y_perm")
    # combine: y[t] = shared row + the token's k routed rows
    sr = cpu(layer.slot_row).numpy().reshape(w.T, w.k)
    y_comb = y_ref[w.S + np.arange(w.T)] + y_ref[sr].sum(1)
    assert_close(y, y_comb, f"{name} y")
    # end to end against the oracle's own routing, where the routing agrees
    full = oracle.layer_forward(x, cpu(inp["W_g"]), W13, W2, cpu(inp["bias"]), w.k, w.rho,
                                w.clamp, is_vision=cpu(inp["is_vision"]),
                                offset=None if inp["logit_offset"] is None else cpu(inp["logit_offset"]))
    same = np.all(full["ids"] == cpu(layer.ids).numpy(), axis=1)
    # a disagreement is only legitimate at a near-tie of the keys
    assert np.all(same | (full["margin"] < 1e-5)), name
    assert_close(np64(y)[same], full["y"][same], f"{name} y end-to-end")


@pytest.mark.parametrize("name,recompute", [("tiny", False), ("mid_I192", False),
                                            ("mid_skew", False), ("mid_skew", True),
                                            ("paired", False), ("max_groups", False),
                                            ("max_groups", True),
                                            ("one_token_all_experts", False)])
def test_backward_layer(name, recompute):
    w = CASES[name]
    layer, inp = make_layer(w, backward=True, recompute=recompute)
    layer.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"])
    layer.backward(inp["dY"], want_dlogits=True, want_dweights=True)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    x, Wg, W13, W2, dY = (cpu(inp[k]) for k in ("x", "W_g", "W13", "W2", "dY"))
    off = None if inp["logit_offset"] is None else cpu(inp["logit_offset"])
    ref = oracle.layer_backward(x, Wg, W13, W2, dY, cpu(inp["bias"]), w.k, w.rho, w.clamp,
                                is_vision=cpu(inp["is_vision"]), offset=off)
    fwd = oracle.layer_forward(x, Wg, W13, W2, cpu(inp["bias"]), w.k, w.rho, w.clamp,
                               is_vision=cpu(inp["is_vision"]), offset=off)
    np.testing.assert_array_equal(fwd["ids"], cpu(layer.ids).numpy())
    assert_close(layer.dX, ref["dX"], f"{name} dX")
    assert_close(layer.dweights, ref["dw"], f"{name} dw", max_abs=5e-2 * max(1, np.abs(ref["dw"]).max() / 10))
    assert_close(layer.dlogits, ref["dz"], f"{name} dlogits")
    assert_close(layer.dW_g, oracle.gate_wgrad_rows(x, ref["dz"], np.arange(w.E)), f"{name} dW_g")
    rt, grp, rw = _rows_meta(layer, w)
    offs = cpu(layer.offsets).numpy()
    counts = np.diff(offs)
    experts = sorted({int(np.argmax(counts[:w.E])), int(np.argmin(counts[:w.E])), 0, w.E})
    for e in experts:
        rows = np.arange(offs[e], offs[e + 1])
        g = oracle.expert_wgrad(x, W13, W2, dY, e, rt[rows], rw[rows], w.clamp, store_bf16=True)
        assert_close(layer.dW13[e], g["dW13"], f"{name} dW13[{e}]")
        assert_close(layer.dW2[e], g["dW2"], f"{name} dW2[{e}]")


@pytest.mark.parametrize("recompute", [False, True])
def test_backward_layer_hash_router(recompute):
    # the backward of the hash router: experts from tid2eid[input_ids], weights
    # from the sigmoid of the gate logits at those experts (bias unused)
    w = W.Workload("mid_hash", 400, 256, 24, 4, 192, 2.5, vision_frac=0.25, hash_variant=True)
    layer, inp = make_layer(w, backward=True, recompute=recompute)
    layer.forward(inp["x"], inp["bias"], inp["is_vision"], None, mode=MOE_ROUTE_HASH,
                  input_ids=inp["input_ids"], tid2eid=inp["tid2eid"])
    layer.backward(inp["dY"], want_dlogits=True, want_dweights=True)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    x, Wg, W13, W2, dY = (cpu(inp[k]) for k in ("x", "W_g", "W13", "W2", "dY"))
    hk = dict(is_vision=cpu(inp["is_vision"]), mode=1, input_ids=cpu(inp["input_ids"]),
              tid2eid=cpu(inp["tid2eid"]))
    fwd = oracle.layer_forward(x, Wg, W13, W2, cpu(inp["bias"]), w.k, w.rho, w.clamp, **hk)
    np.testing.assert_array_equal(fwd["ids"], cpu(layer.ids).numpy())
    np.testing.assert_array_equal(fwd["ids"], cpu(inp["tid2eid"]).numpy()[cpu(inp["input_ids"]).numpy()])
    ref = oracle.layer_backward(x, Wg, W13, W2, dY, cpu(inp["bias"]), w.k, w.rho, w.clamp, **hk)
    assert_close(layer.dX, ref["dX"], "hash dX")
    assert_close(layer.dweights, ref["dw"], "hash dw",
                 max_abs=5e-2 * max(1, np.abs(ref["dw"]).max() / 10))
    assert_close(layer.dlogits, ref["dz"], "hash dlogits")
    assert_close(layer.dW_g, oracle.gate_wgrad_rows(x, ref["dz"], np.arange(w.E)), "hash dW_g")
    rt, grp, rw = _rows_meta(layer, w)
    offs = cpu(layer.offsets).numpy()
    counts = np.diff(offs)
    for e in sorted({int(np.argmax(counts[:w.E])), int(np.argmin(counts[:w.E])), w.E}):
        rows = np.arange(offs[e], offs[e + 1])
        g = oracle.expert_wgrad(x, W13, W2, dY, e, rt[rows], rw[rows], w.clamp, store_bf16=True)
        assert_close(layer.dW13[e], g["dW13"], f"hash dW13[{e}]")
        assert_close(layer.dW2[e], g["dW2"], f"hash dW2[{e}]")


def test_backward_gate_wgrad_chunk_boundaries():
    # dW_g sums each expert's rows in chunks of 256 that never cross an expert:
    # a hash table that gives the experts 256, 257, 127, 512, 127, 1, 0 and 0
    # rows puts groups exactly at, one past and twice the chunk length, a
    # one-row group and empty groups
    T, E, k = 640, 8, 2
    w = W.Workload("gate_chunks", T, 128, E, k, 64, 2.5, vision_frac=0.25)
    layer, inp = make_layer(w, backward=True)
    t = np.arange(T)
    first = np.where(t < 256, 0, np.where(t < 513, 1, 2))
    second = np.where(t < 512, 3, np.where(t < 639, 4, 5))
    tid2eid = torch.tensor(np.stack([first, second], 1), dtype=torch.int32, device="cuda")
    input_ids = torch.arange(T, dtype=torch.int32, device="cuda")
    layer.forward(inp["x"], inp["bias"], inp["is_vision"], None, mode=MOE_ROUTE_HASH,
                  input_ids=input_ids, tid2eid=tid2eid)
    layer.backward(inp["dY"], want_dlogits=True)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    counts = np.diff(cpu(layer.offsets).numpy())[:E]
    np.testing.assert_array_equal(counts, [256, 257, 127, 512, 127, 1, 0, 0])
    x, Wg, W13, W2, dY = (cpu(inp[k_]) for k_ in ("x", "W_g", "W13", "W2", "dY"))
    hk = dict(is_vision=cpu(inp["is_vision"]), mode=1, input_ids=cpu(input_ids),
              tid2eid=cpu(tid2eid))
    ref = oracle.layer_backward(x, Wg, W13, W2, dY, cpu(inp["bias"]), k, w.rho, w.clamp, **hk)
    assert_close(layer.dlogits, ref["dz"], "chunks dlogits")
    assert_close(layer.dW_g, oracle.gate_wgrad_rows(x, ref["dz"], np.arange(E)), "chunks dW_g")
    assert torch.count_nonzero(layer.dW_g[6:]).item() == 0


def test_zero_routed_scaling_gives_zero_routing_gradients():
    # with scaling 0 every routing weight is 0: y is the shared expert alone,
    # and the routing chain passes no gradient (and no NaN) to the logits
    w = W.scaled(CASES["mid_I192"], name="rho0", rho=0.0)
    layer, inp = make_layer(w, backward=True)
    layer.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"])
    layer.backward(inp["dY"], want_dlogits=True, want_dweights=True)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    assert torch.count_nonzero(layer.weights).item() == 0
    assert torch.count_nonzero(layer.dlogits).item() == 0
    assert torch.count_nonzero(layer.dW_g).item() == 0
    assert bool(torch.isfinite(layer.dX).all()) and bool(torch.isfinite(layer.dweights).all())
    x, Wg, W13, W2, dY = (cpu(inp[k]) for k in ("x", "W_g", "W13", "W2", "dY"))
    ref = oracle.layer_backward(x, Wg, W13, W2, dY, cpu(inp["bias"]), w.k, w.rho, w.clamp,
                                is_vision=cpu(inp["is_vision"]))
    assert_close(layer.dX, ref["dX"], "rho0 dX")


def test_empty_expert_gets_zero_grad():
    w = W.Workload("empty", 96, 128, 8, 2, 64, 1.0)
    layer, inp = make_layer(w, backward=True)
    # route every token to experts 0 and 1 only (bias pushes them on top)
    bias = torch.full((2, w.E), -1.0, device="cuda")
    bias[:, :2] = 1.0
    layer.forward(inp["x"], bias)
    layer.backward(inp["dY"])
    torch.cuda.synchronize()
    counts = cpu(layer.counts).numpy()
    assert counts[2:].sum() == 0
    assert torch.count_nonzero(layer.dW13[2:w.E]).item() == 0
    assert torch.count_nonzero(layer.dW2[2:w.E]).item() == 0
    assert torch.count_nonzero(layer.dW_g[2:]).item() == 0


def test_selftest_wait_timeout_reports_status():
    assert _lib.moe_last_device_status() in (_lib.MOE_OK, _lib.MOE_ERR_TIMEOUT)
    _lib.moe_selftest_wait_timeout(200_000)
    assert _lib.moe_last_device_status() == _lib.MOE_ERR_TIMEOUT
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    # the context is still usable
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


def test_abi_rejects_bad_arguments_before_launch():
    T, d, E, k = 8, 128, 4, 2
    x = torch.zeros(T * d + 8, dtype=torch.bfloat16, device="cuda")
    Wg = torch.zeros(E, d, dtype=torch.bfloat16, device="cuda")
    out = [torch.empty(T, E, device="cuda"), torch.empty(T, k, dtype=torch.int32, device="cuda"),
           torch.empty(T, k, device="cuda"), torch.empty(T, k, device="cuda")]
    bias = torch.zeros(2, E, device="cuda")
    with pytest.raises(_lib.MoeError) as ei:   # misaligned x (2-byte offset)
        _lib.moe_route(x[1:1 + T * d], Wg, None, bias, None, None, None, T, d, E, k, 1.0,
                       MOE_ROUTE_TOPK, *out)
    assert ei.value.status == _lib.MOE_ERR_INVALID_ARG
    with pytest.raises(_lib.MoeError) as ei:   # k > E
        _lib.moe_route(x[:T * d], Wg, None, bias, None, None, None, T, d, E, E + 1, 1.0,
                       MOE_ROUTE_TOPK, *out)
    assert ei.value.status == _lib.MOE_ERR_INVALID_ARG
    with pytest.raises(_lib.MoeError) as ei:   # d not a multiple of 128 for the expert FFN
        _lib.moe_expert_ffn(x, out[1], 1, 8, Wg, Wg, None, 0, 96, 64, 7.0, None, x, x)
    assert ei.value.status == _lib.MOE_ERR_UNSUPPORTED
