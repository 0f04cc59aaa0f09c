"""Parity at the full workload sizes, in the launch configuration the bench uses.

Index work is compared on every token (routing from the GPU's own logits,
permutation, counts, offsets: bit-exact; routing weights within 1e-6).  Float
outputs are compared on seeded samples the oracle computes one by one: y, h
and y_perm rows of sampled tokens; dX, dlogits and dw of sampled tokens; and
sampled weight-gradient entries of the hottest, median and coldest non-empty
routed experts and of the shared expert.  dW_g rows of eight experts are
checked against the oracle's reduction of the GPU's logit gradients (which
are themselves checked against the oracle on the sampled tokens).
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_04_gb300 import _lib
from moe_expert_layer_04_gb300 import workloads as W
from moe_expert_layer_04_gb300.layer import MOE_ROUTE_HASH, MOE_ROUTE_TOPK, Dims, MoELayer
from tests.helpers import W_RTOL, assert_close, assert_close_rounded, cpu, np64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# seeded tokens whose outputs (y, h and y_perm rows) and gradients (dX,
# dlogits, dw) are compared, and sampled entries per weight gradient (dW2 and
# dW13 each) of each of the four checked experts
N_TOK = 512
N_ENT = 64


@pytest.fixture(scope="module")
def weights():
    """The full-width expert weights (same seed and shapes for every full-width
    workload), on the device and as host copies for the oracle."""
    w = W.WORKLOADS["full_fwd"]
    inp = W.make_inputs(w, device="cuda")
    dev = {k: inp[k] for k in ("W_g", "W13", "W2")}
    host = {k: v.cpu() for k, v in dev.items()}
    return dev, host


def _sample(n_total, n, seed):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(n_total, size=min(n, n_total), replace=False))


def _run(w, weights, backward=False, mode=MOE_ROUTE_TOPK):
    dev, _ = weights
    inp = W.make_inputs(w, device="cuda", with_weights=False, with_dy=backward)
    layer = MoELayer(Dims(w.T, w.d, w.E, w.k, w.I), dev, w.rho, w.clamp, backward=backward,
                     recompute=w.recompute)
    hash_kw = {}
    if mode == MOE_ROUTE_HASH:
        hash_kw = dict(mode=mode, input_ids=inp["input_ids"], tid2eid=inp["tid2eid"])
    layer.forward(inp["x"], inp["bias"], inp["is_vision"],
                  None if mode == MOE_ROUTE_HASH else inp["logit_offset"], **hash_kw)
    if backward:
        layer.backward(inp["dY"], want_dlogits=True, want_dweights=True)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    return layer, inp


def _check_indices(layer, inp, w, mode):
    z = np64(layer.logits)
    kw = {}
    if mode == MOE_ROUTE_HASH:
        kw = dict(mode=1, input_ids=cpu(inp["input_ids"]), tid2eid=cpu(inp["tid2eid"]))
    ids, wts, s, _ = oracle.route(z, cpu(inp["bias"]), w.k, w.rho, is_vision=cpu(inp["is_vision"]),
                                  **kw)
    g_ids = cpu(layer.ids).numpy()
    np.testing.assert_array_equal(g_ids, ids)
    np.testing.assert_array_equal(np64(layer.scores_sel), s)
    np.testing.assert_allclose(np64(layer.weights), wts, rtol=W_RTOL, atol=0)
    c, o, rt, sr = oracle.permute(g_ids, w.E)
    np.testing.assert_array_equal(cpu(layer.counts).numpy(), c)
    if layer.modality_counts is not None:
        np.testing.assert_array_equal(cpu(layer.modality_counts).numpy(),
                                      oracle.modality_counts(g_ids, cpu(inp["is_vision"]), w.E))
    np.testing.assert_array_equal(cpu(layer.offsets).numpy()[: w.E + 1], o)
    np.testing.assert_array_equal(cpu(layer.row_token).numpy()[: w.S], rt)
    np.testing.assert_array_equal(cpu(layer.slot_row).numpy(), sr)
    return c


def _check_forward_sampled(layer, inp, w, weights, n_tok, mode):
    _, host = weights
    tok = _sample(w.T, n_tok, 1)
    x = cpu(inp["x"])
    if mode == MOE_ROUTE_TOPK:
        off = None if inp["logit_offset"] is None else cpu(inp["logit_offset"])
        z_ref = oracle.gate_logits(x, host["W_g"], offset=off, tok=tok)
        z = np64(layer.logits[torch.from_numpy(tok).cuda()])
        assert np.max(np.abs(z - z_ref)) < 1e-3
    sr = cpu(layer.slot_row).numpy().reshape(w.T, w.k)
    rows = np.concatenate([[w.S + t] + list(sr[t]) for t in tok]).astype(np.int64)
    rt = cpu(layer.row_token).numpy()[rows].astype(np.int64)
    grp = np.concatenate([[w.E] + list(cpu(layer.ids).numpy()[t]) for t in tok]).astype(np.int32)
    rw = np.concatenate([[1.0] + list(np64(layer.weights)[t]) for t in tok])
    h_ref, y_ref = oracle.expert_rows(x, host["W13"], host["W2"], rt, grp, rw, w.clamp)
    ridx = torch.from_numpy(rows).cuda()
    assert_close_rounded(layer.h_perm[ridx], h_ref, f"{w.name} h rows")
    assert_close_rounded(layer.y_perm[ridx], y_ref, f"{w.name} y_perm rows")
    y_tok = y_ref.reshape(len(tok), w.k + 1, -1).sum(1)
    assert_close(layer.y[torch.from_numpy(tok).cuda()], y_tok, f"{w.name} y")


def _check_backward_sampled(layer, inp, w, weights, counts, n_tok, n_ent):
    _, host = weights
    tok = _sample(w.T, n_tok, 2)
    x, dY = cpu(inp["x"]), cpu(inp["dY"])
    off = None if inp["logit_offset"] is None else cpu(inp["logit_offset"])
    ref = oracle.layer_backward(x, host["W_g"], host["W13"], host["W2"], dY, cpu(inp["bias"]),
                                w.k, w.rho, w.clamp, is_vision=cpu(inp["is_vision"]), offset=off,
                                tok=tok)
    fwd = oracle.layer_forward(x, host["W_g"], host["W13"], host["W2"], cpu(inp["bias"]), w.k,
                               w.rho, w.clamp, is_vision=cpu(inp["is_vision"]), offset=off,
                               tok=tok)
    same = np.all(fwd["ids"] == cpu(layer.ids).numpy()[tok], axis=1)
    assert np.all(same | (fwd["margin"] < 1e-5))
    tt = torch.from_numpy(tok[same]).cuda()
    assert_close(layer.dX[tt], ref["dX"][same], f"{w.name} dX")
    assert_close(layer.dlogits[tt], ref["dz"][same], f"{w.name} dlogits")
    # dw = <h, dA>: stage-wise against the oracle's fp64 dA and the GPU's own h
    # (the GEMM + epilogue alone), then end to end, where h's bf16 rounding
    # from fp32 (GPU) or fp64 (oracle) accumulators may differ by one ulp
    sr = cpu(layer.slot_row).numpy().reshape(w.T, w.k)[tok[same]].ravel().astype(np.int64)
    g_ids = cpu(layer.ids).numpy()[tok[same]].ravel().astype(np.int32)
    dA = oracle.rows_dA(dY, host["W2"], np.repeat(tok[same], w.k), g_ids)
    h_gpu = np64(layer.h_perm[torch.from_numpy(sr).cuda()])
    dw_stage = (h_gpu * dA).sum(1).reshape(-1, w.k)
    assert_close(layer.dweights[tt], dw_stage, f"{w.name} dw (stage-wise)", rel_fro=1e-4)
    dw_ref = ref["dw"][same]
    assert_close(layer.dweights[tt], dw_ref, f"{w.name} dw (end to end)",
                 max_abs=max(5e-2, 5e-3 * np.abs(dw_ref).max()))
    # dW_g rows: the oracle's reduction sum_t dz[t, e] x[t] of the GPU's logit
    # gradients (checked above on the sampled tokens) for eight experts: the
    # hottest, the median, the coldest non-empty, an empty one if any, and
    # seeded others.  Each entry sums over the expert's tokens, so the max-abs
    # bound grows with the entries above 5e-2 as for the weight gradients below.
    nz_e = np.nonzero(counts)[0]
    by = nz_e[np.argsort(counts[nz_e], kind="stable")]
    pick = [int(by[-1]), int(by[len(by) // 2]), int(by[0])]
    empty = np.nonzero(counts == 0)[0]
    if len(empty):
        pick.append(int(empty[0]))
    rest = np.setdiff1d(np.arange(w.E), pick)
    pick += [int(e) for e in np.random.default_rng(4).choice(rest, 8 - len(pick), replace=False)]
    dwg_ref = oracle.gate_wgrad_rows(x, np64(layer.dlogits), np.array(pick, np.int32))
    dwg = layer.dW_g[torch.tensor(pick, device="cuda")]
    assert_close(dwg, dwg_ref, f"{w.name} dW_g rows {pick}",
                 max_abs=max(5e-2, 1e-3 * np.abs(dwg_ref).max()))
    if len(empty):
        assert torch.count_nonzero(layer.dW_g[int(empty[0])]).item() == 0
    # sampled weight-gradient entries
    offs = cpu(layer.offsets).numpy()
    rt_all = cpu(layer.row_token).numpy().astype(np.int64)
    rw_all = np.ones(w.S + w.T)
    rw_all[: w.S] = np64(layer.row_weight)
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    experts = [int(order[-1]), int(order[len(order) // 2]), int(order[0]), w.E]
    rng = np.random.default_rng(3)
    for e in experts:
        rows = np.arange(offs[e], offs[e + 1])
        kind = np.repeat(np.array([0, 1], np.int32), n_ent)
        qa = np.concatenate([rng.integers(0, w.d, n_ent), rng.integers(0, 2 * w.I, n_ent)]).astype(np.int32)
        qb = np.concatenate([rng.integers(0, w.I, n_ent), rng.integers(0, w.d, n_ent)]).astype(np.int32)
        got_ref = oracle.expert_wgrad_entries(x, host["W13"], host["W2"], dY, e, rt_all[rows],
                                              rw_all[rows], w.clamp, kind, qa, qb, store_bf16=True)
        g2 = layer.dW2[e][torch.from_numpy(qa[:n_ent]).long().cuda(), torch.from_numpy(qb[:n_ent]).long().cuda()]
        g13 = layer.dW13[e][torch.from_numpy(qa[n_ent:]).long().cuda(), torch.from_numpy(qb[n_ent:]).long().cuda()]
        # stage-wise: the weight-gradient matmul on the GPU's own h rows
        h_rows = layer.h_perm[int(offs[e]):int(offs[e + 1])]
        stage = oracle.wgrad2_entries_given_h(dY, h_rows.cpu(), rt_all[rows], rw_all[rows],
                                              qa[:n_ent], qb[:n_ent], store_bf16=True)
        # the tensor cores' fp32 accumulation over up to 2^16 rows (the shared
        # expert of the 64K-token slice) leaves ~1e-4 of the entries' size
        assert_close(g2, stage, f"{w.name} dW2[{e}] entries (stage-wise)",
                     max_abs=max(5e-2, 2e-4 * np.abs(stage).max()))
        # end to end: over K rows, one-ulp bf16 flips of h (fp32 vs fp64
        # accumulators) add up to ~sqrt(K * 3e-4) ulps; the bound scales with
        # the entries' size above 5e-2
        tol = max(5e-2, 1e-3 * np.abs(got_ref).max())
        assert_close(g2, got_ref[:n_ent], f"{w.name} dW2[{e}] entries", max_abs=tol)
        assert_close(g13, got_ref[n_ent:], f"{w.name} dW13[{e}] entries", max_abs=tol)


def test_full_fwd(weights):
    w = W.WORKLOADS["full_fwd"]
    layer, inp = _run(w, weights)
    _check_indices(layer, inp, w, MOE_ROUTE_TOPK)
    _check_forward_sampled(layer, inp, w, weights, N_TOK, MOE_ROUTE_TOPK)


def test_skewed_multimodal_topk_and_hash(weights):
    w = W.WORKLOADS["skewed_mm_fwd"]
    for mode in (MOE_ROUTE_TOPK, MOE_ROUTE_HASH):
        layer, inp = _run(w, weights, mode=mode)
        counts = _check_indices(layer, inp, w, mode)
        if mode == MOE_ROUTE_TOPK:
            assert counts.max() > 8 * counts.mean()     # the Zipf skew is there
        _check_forward_sampled(layer, inp, w, weights, N_TOK, mode)
        del layer
        torch.cuda.empty_cache()


def test_fwd_bwd(weights):
    w = W.WORKLOADS["fwd_bwd"]
    layer, inp = _run(w, weights, backward=True)
    counts = _check_indices(layer, inp, w, MOE_ROUTE_TOPK)
    _check_forward_sampled(layer, inp, w, weights, N_TOK, MOE_ROUTE_TOPK)
    _check_backward_sampled(layer, inp, w, weights, counts, N_TOK, N_ENT)


def test_long_slice_fwd_bwd_recompute(weights):
    w = W.WORKLOADS["long_slice_fwd_bwd"]
    layer, inp = _run(w, weights, backward=True)
    counts = _check_indices(layer, inp, w, MOE_ROUTE_TOPK)
    assert int(cpu(inp["is_vision"]).sum()) == round(0.3 * w.T)
    _check_forward_sampled(layer, inp, w, weights, N_TOK, MOE_ROUTE_TOPK)
    _check_backward_sampled(layer, inp, w, weights, counts, N_TOK, N_ENT)
