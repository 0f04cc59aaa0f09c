"""The one-kernel gate projection + routing (moe_gate_route) against the oracle.

Stage-wise like the other routing tests: the oracle routes the GPU's own fp32
logits, so expert ids and selected scores must match bit for bit and weights
within 1e-6; the logits themselves are compared with the oracle's fp64
projection.  The per-modality expert load must equal the oracle's count of
the GPU's own ids exactly.  The experts split over a pair of CTAs when E is a
multiple of 64 and stay in one CTA otherwise; the shapes cover both layouts,
one and two MMAs per K step, one and two TMEM accumulators, two to four
operand stages, ragged last tiles, CTAs that loop over several tiles, exact
ties, and the rescan taken when more near-equal keys than the candidate list
holds sit at the k-th place.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_04_gb300 import _lib
from moe_expert_layer_04_gb300 import workloads as W
from moe_expert_layer_04_gb300.layer import MOE_ROUTE_HASH, MOE_ROUTE_TOPK
from tests.helpers import W_RTOL, cpu, np64

pytestmark = pytest.mark.gpu

# name, T, d, E, k, vision fraction, Zipf skew of the load, bias amplitude
CASES = [
    ("E64_ragged", 300, 256, 64, 4, 0.3, 0.0, 0.1),
    ("E384_zipf", 1000, 512, 384, 6, 0.25, 1.1, 0.1),
    ("E512_k8", 129, 128, 512, 8, 0.5, 0.0, 0.1),
    ("E32_k1", 64, 64, 32, 1, 0.0, 0.0, 0.1),
    ("E256_k8", 777, 256, 256, 8, 0.1, 1.1, 0.01),
    ("E96_tiles", 2000, 128, 96, 3, 0.3, 0.0, 0.1),
    # one CTA per tile (E not a multiple of 64) with two MMAs and one accumulator
    ("E288_one_cta", 500, 128, 288, 6, 0.3, 0.0, 0.1),
    # more tiles than SMs: every CTA loops over several tiles
    ("E384_persistent", 152 * 128 * 2 + 77, 64, 384, 6, 0.3, 1.1, 0.01),
    ("E128_persistent", 152 * 128 * 2 + 77, 64, 128, 6, 0.3, 0.0, 0.01),
]

GUARD = 130  # rows of sentinel past T in the logits buffer


def _workload(name, T, d, E, k, vf, zipf, amp, hash_variant=False):
    return W.Workload(name, T, d, E, k, 64, 2.5, vision_frac=vf, zipf_s=zipf, bias_amp=amp,
                      hash_variant=hash_variant)


def _inputs(w):
    inp = W.make_inputs(w, device="cuda", with_weights=False)
    inp["W_g"] = W.normal_bf16((w.E, w.d), 0.02, w.seed, "W_g", "cuda")
    return inp


def _fused(w, inp, mode=MOE_ROUTE_TOPK, counts=True):
    T, E, k = w.T, w.E, w.k
    z_buf = torch.full((T + GUARD, E), float("nan"), device="cuda")
    out = dict(logits=z_buf[:T],
               ids=torch.full((T + 1, k), -7, dtype=torch.int32, device="cuda"),
               weights=torch.empty(T, k, device="cuda"),
               ssel=torch.empty(T, k, device="cuda"),
               counts=torch.full((2, E), -1, dtype=torch.int32, device="cuda") if counts else None)
    hash_kw = (inp["input_ids"], inp["tid2eid"]) if mode == MOE_ROUTE_HASH else (None, None)
    _lib.moe_gate_route(inp["x"], inp["W_g"], None if mode == MOE_ROUTE_HASH else
                        inp["logit_offset"], inp["bias"], inp["is_vision"], *hash_kw, T, w.d, E,
                        k, w.rho, mode, out["logits"], out["ids"], out["weights"], out["ssel"],
                        out["counts"])
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    # nothing past the T rows is written
    assert torch.isnan(z_buf[T:]).all()
    assert (out["ids"][T] == -7).all()
    out["ids"] = out["ids"][:T]
    return out


def _check(w, inp, out, mode=MOE_ROUTE_TOPK):
    z = np64(out["logits"])
    off = None if (mode == MOE_ROUTE_HASH or inp["logit_offset"] is None) \
        else cpu(inp["logit_offset"])
    z_ref = oracle.gate_logits(cpu(inp["x"]), cpu(inp["W_g"]), offset=off)
    assert np.max(np.abs(z - z_ref)) < 1e-4 * max(1.0, np.abs(z_ref).max()), w.name
    kw = {}
    if mode == MOE_ROUTE_HASH:
        kw = dict(mode=1, input_ids=cpu(inp["input_ids"]), tid2eid=cpu(inp["tid2eid"]))
    ids, wts, s, _ = oracle.route(z, cpu(inp["bias"]), w.k, w.rho,
                                  is_vision=cpu(inp["is_vision"]), **kw)
    g_ids = cpu(out["ids"]).numpy()
    np.testing.assert_array_equal(g_ids, ids, err_msg=w.name)
    np.testing.assert_array_equal(np64(out["ssel"]), s, err_msg=w.name)
    np.testing.assert_allclose(np64(out["weights"]), wts, rtol=W_RTOL, atol=0, err_msg=w.name)
    if out["counts"] is not None:
        np.testing.assert_array_equal(cpu(out["counts"]).numpy(),
                                      oracle.modality_counts(g_ids, cpu(inp["is_vision"]), w.E),
                                      err_msg=w.name)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_route_matches_oracle(case):
    w = _workload(*case)
    inp = _inputs(w)
    out = _fused(w, inp)
    _check(w, inp, out)
    # the two-kernel path (projection GEMM, then routing) on the same inputs
    T, E, k = w.T, w.E, w.k
    z2 = torch.empty(T, E, device="cuda")
    ids2 = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w2 = torch.empty(T, k, device="cuda")
    s2 = torch.empty(T, k, device="cuda")
    _lib.moe_route(inp["x"], inp["W_g"], inp["logit_offset"], inp["bias"], inp["is_vision"],
                   None, None, T, w.d, E, k, w.rho, MOE_ROUTE_TOPK, z2, ids2, w2, s2)
    torch.cuda.synchronize()
    zf = np64(out["logits"])
    assert np.max(np.abs(zf - np64(z2))) < 1e-4 * max(1.0, np.abs(zf).max())


def test_fused_route_hash_mode():
    w = _workload("hash_E384", 500, 256, 384, 6, 0.25, 0.0, 0.1, hash_variant=True)
    inp = _inputs(w)
    out = _fused(w, inp, mode=MOE_ROUTE_HASH)
    _check(w, inp, out, mode=MOE_ROUTE_HASH)
    # the experts are the table rows of the token ids
    want = cpu(inp["tid2eid"]).numpy()[cpu(inp["input_ids"]).numpy()]
    np.testing.assert_array_equal(cpu(out["ids"]).numpy(), want)


def test_fused_route_exact_ties_go_to_lower_id():
    # experts in pairs with identical gate rows and identical biases: every key
    # has an exact twin, and the lower id must be taken first
    w = _workload("ties", 400, 128, 64, 5, 0.5, 0.0, 0.1)
    inp = _inputs(w)
    inp["W_g"][1::2] = inp["W_g"][0::2]
    inp["bias"][:, 1::2] = inp["bias"][:, 0::2]
    out = _fused(w, inp)
    _check(w, inp, out)
    ids = cpu(out["ids"]).numpy()
    # a twin pair is taken whole, lower id first, or only its lower member
    for t in range(w.T):
        for j, e in enumerate(ids[t]):
            if e % 2 == 1:
                assert e - 1 in ids[t][:j], (t, ids[t])


@pytest.mark.parametrize("E,k", [(96, 5), (384, 6), (64, 8)])
def test_fused_route_all_keys_equal_rescans(E, k):
    # zero gate and zero bias: every key is sigmoid(0), more experts than the
    # candidate list holds tie at the k-th place, and the ids must be 0..k-1
    w = _workload("all_equal", 260, 64, E, k, 0.5, 0.0, 0.0)
    inp = _inputs(w)
    inp["W_g"].zero_()
    out = _fused(w, inp)
    _check(w, inp, out)
    assert (cpu(out["ids"]).numpy() == np.arange(k)).all()
    np.testing.assert_allclose(np64(out["weights"]), w.rho / k, rtol=W_RTOL)


def test_fused_route_without_counts_and_repeated_calls():
    # counts are optional; a second call overwrites (does not accumulate) them
    w = _workload("repeat", 700, 128, 64, 4, 0.3, 0.0, 0.1)
    inp = _inputs(w)
    _check(w, inp, _fused(w, inp, counts=False))
    out = _fused(w, inp)
    c1 = out["counts"].clone()
    _lib.moe_gate_route(inp["x"], inp["W_g"], None, inp["bias"], inp["is_vision"], None, None,
                        w.T, w.d, w.E, w.k, w.rho, MOE_ROUTE_TOPK, out["logits"], out["ids"],
                        out["weights"], out["ssel"], out["counts"])
    torch.cuda.synchronize()
    assert torch.equal(out["counts"], c1)
    assert int(c1.sum()) == w.T * w.k
