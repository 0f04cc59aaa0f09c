"""Pins of the CPU oracle against what the pages and mathematics fix.

The pages print no worked example for the MoE layer, so the oracle is pinned by
hand-derived cases (tests/golden), brute force, invariants, special cases that
reduce to library routines (torch / scipy), and central finite differences.
Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong index or sign, a transposed weight, the bias leaking into the weights)
fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle
from moe_expert_layer_04_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def f32(a):
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


# ----------------------------------------------------------------- routing

def test_route_hand_cases():
    cases = json.load(open(os.path.join(HERE, "golden", "route_cases.json")))["cases"]
    for c in cases:
        z = np.array([c["z"]], np.float64)
        bias = np.array(c["bias"], np.float32)
        ids, w, s, _ = oracle.route(z, bias, c["k"], c["rho"])
        assert ids[0].tolist() == c["ids"], c["name"]
        np.testing.assert_array_equal(w[0], np.array(c["w"], np.float64), err_msg=c["name"])
        np.testing.assert_array_equal(s[0], 0.5)


def _keys(z, bias_row):
    """fp32 key from the library sigmoid: fp32(fp32(expit(z)) + b)."""
    s = f32(expit(z))
    return f32(s + np.asarray(bias_row, np.float32).astype(np.float64)), s


def test_route_topk_brute_force_tiny():
    w = W.WORKLOADS["tiny_fwd"]
    inp = W.make_inputs(w)
    z = oracle.gate_logits(inp["x"], inp["W_g"])
    vis = np.zeros(w.T, np.uint8)
    vis[::3] = 1
    ids, wt, s, margin = oracle.route(z, inp["bias"], w.k, w.rho, is_vision=vis)
    bias = inp["bias"].numpy()
    subsets = list(itertools.combinations(range(w.E), w.k))
    for t in range(w.T):
        key, sc = _keys(z[t], bias[vis[t]])
        chosen = set(ids[t].tolist())
        assert len(chosen) == w.k
        # every selected key beats every unselected one (ties to the lower id)
        for e in chosen:
            for o in set(range(w.E)) - chosen:
                assert key[e] > key[o] or (key[e] == key[o] and e < o)
        # the chosen set maximises the key sum over all C(E, k) subsets
        best = max(sum(key[list(q)]) for q in subsets)
        assert sum(key[list(ids[t])]) == best
        # output order: descending key, ties by id
        order = sorted(ids[t].tolist(), key=lambda e: (-key[e], e))
        assert ids[t].tolist() == order
        # extraction takes the unbiased score; weights are normalised and scaled
        np.testing.assert_array_equal(s[t], sc[ids[t]])
        np.testing.assert_allclose(wt[t].sum(), w.rho, rtol=1e-6)
        np.testing.assert_allclose(wt[t], f32(w.rho * sc[ids[t]] / sc[ids[t]].sum()), rtol=0)
        kth = sorted(key, reverse=True)
        assert margin[t] == min(kth[j] - kth[j + 1] for j in range(w.k))


def test_route_ties_lowest_id():
    z = np.zeros((2, 8))
    bias = np.zeros(8, np.float32)
    ids, _, _, margin = oracle.route(z, bias, 3, 1.0)
    assert ids.tolist() == [[0, 1, 2], [0, 1, 2]]
    assert margin[0] == 0.0


def test_route_k1_weight_is_scaling():
    z = W.random_logits(50, 32, 1.5, seed=3).numpy().astype(np.float64)
    bias = np.random.default_rng(1).uniform(-0.1, 0.1, 32).astype(np.float32)
    _, w, _, _ = oracle.route(z, bias, 1, 2.5)
    assert np.all(w == 2.5)


def test_route_k_equals_E_matches_library_softnorm():
    z = W.random_logits(20, 12, 2.0, seed=4).numpy().astype(np.float64)
    ids, w, _, _ = oracle.route(z, np.zeros(12, np.float32), 12, 2.5, exact=True)
    s = expit(z)
    ref = 2.5 * s / s.sum(1, keepdims=True)
    got = np.zeros_like(ref)
    np.put_along_axis(got, ids.astype(np.int64), w, axis=1)
    np.testing.assert_allclose(got, ref, rtol=1e-14)


def test_route_vision_bias_row():
    E = 8
    z = np.zeros((4, E))
    bias = np.zeros((2, E), np.float32)
    bias[0, 5] = 0.3   # text favours 5
    bias[1, 2] = 0.3   # vision favours 2
    vis = np.array([0, 1, 0, 1], np.uint8)
    ids, w, _, _ = oracle.route(z, bias, 1, 1.0, is_vision=vis)
    assert ids[:, 0].tolist() == [5, 2, 5, 2]


def test_route_hash_mode():
    rng = np.random.default_rng(5)
    T, E, k, V = 40, 24, 4, 100
    z = rng.normal(size=(T, E))
    tab = np.stack([rng.permutation(E)[:k] for _ in range(V)]).astype(np.int32)
    iid = rng.integers(0, V, T).astype(np.int32)
    b1 = rng.uniform(-0.1, 0.1, (2, E)).astype(np.float32)
    ids, w, s, _ = oracle.route(z, b1, k, 2.5, mode=1, input_ids=iid, tid2eid=tab)
    np.testing.assert_array_equal(ids, tab[iid])
    ids2, w2, _, _ = oracle.route(z, b1 * 0, k, 2.5, mode=1, input_ids=iid, tid2eid=tab)
    np.testing.assert_array_equal(w, w2)          # the bias plays no part in hash mode
    sc = f32(expit(np.take_along_axis(z, tab[iid].astype(np.int64), 1)))
    np.testing.assert_array_equal(s, sc)
    np.testing.assert_allclose(w, f32(2.5 * sc / sc.sum(1, keepdims=True)), rtol=0)


# ----------------------------------------------------------------- permute

@pytest.mark.parametrize("T,E,k,skew", [(64, 16, 2, 0.0), (257, 40, 6, 1.1), (1, 4, 4, 0.0),
                                        (300, 64, 3, 2.0)])
def test_permute_invariants(T, E, k, skew):
    ids = W.random_ids(T, E, k, seed=T + E, skew=skew).numpy()
    counts, offsets, row_token, slot_row = oracle.permute(ids, E)
    np.testing.assert_array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert counts.sum() == T * k
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    # slot_row is a bijection onto rows and row_token is consistent with it
    assert sorted(slot_row.tolist()) == list(range(T * k))
    for t in range(T):
        for j in range(k):
            r = slot_row[t * k + j]
            assert row_token[r] == t
            assert offsets[ids[t, j]] <= r < offsets[ids[t, j] + 1]
    # stable: inside each expert, rows follow (token, slot) order
    slot_of_row = np.empty(T * k, np.int64)
    slot_of_row[slot_row] = np.arange(T * k)
    for e in range(E):
        seg = slot_of_row[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
    # unpermute(permute(x)) is the identity
    x = np.random.default_rng(0).normal(size=(T, 5))
    xp = x[row_token]
    back = xp[slot_row].reshape(T, k, 5)
    for j in range(k):
        np.testing.assert_array_equal(back[:, j], x)


@pytest.mark.parametrize("T,E,k,skew,frac", [(64, 16, 2, 0.0, 0.0), (257, 40, 6, 1.1, 0.3),
                                             (300, 64, 3, 2.0, 1.0), (1, 4, 4, 0.0, 1.0)])
def test_modality_counts_split_the_expert_histogram(T, E, k, skew, frac):
    ids = W.random_ids(T, E, k, seed=T + 2 * E, skew=skew).numpy()
    vis = (np.random.default_rng(T).random(T) < frac).astype(np.uint8)
    c = oracle.modality_counts(ids, vis, E)
    # the two rows add up to the permutation's histogram
    np.testing.assert_array_equal(c.sum(0), oracle.permute(ids, E)[0])
    # each row is the histogram of that modality's tokens alone
    for m in (0, 1):
        sub = ids[vis == m]
        want = oracle.permute(sub, E)[0] if len(sub) else np.zeros(E, np.int32)
        np.testing.assert_array_equal(c[m], want)
        assert c[m].sum() == k * int((vis == m).sum())
    # no modality flags: everything is text
    c0 = oracle.modality_counts(ids, None, E)
    np.testing.assert_array_equal(c0[1], 0)
    np.testing.assert_array_equal(c0[0], c.sum(0))


# --------------------------------------------------------------- expert FFN

def _rand(shape, std, rng):
    return rng.normal(0, std, shape)


def test_expert_unclamped_is_dense_swiglu_ffn():
    rng = np.random.default_rng(7)
    n, d, I, G = 9, 32, 16, 3
    x = _rand((n, d), 1.0, rng)
    W13 = _rand((G, 2 * I, d), 0.2, rng)
    W2 = _rand((G, d, I), 0.2, rng)
    e = rng.integers(0, G, n).astype(np.int32)
    rw = rng.uniform(0.1, 1.0, n)
    h, y = oracle.expert_rows(x, W13, W2, np.arange(n), e, rw, clamp=1e30, exact=True)
    xt = torch.from_numpy(x)
    for r in range(n):
        gu = torch.from_numpy(W13[e[r]]) @ xt[r]
        href = torch.nn.functional.silu(gu[:I]) * gu[I:]
        yref = rw[r] * (torch.from_numpy(W2[e[r]]) @ href)
        np.testing.assert_allclose(h[r], href.numpy(), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(y[r], yref.numpy(), rtol=1e-12, atol=1e-14)


def test_expert_clamp_closed_form_points():
    # one-hot x selects single weight entries, so g and u are set directly
    d, I, c = 4, 2, 7.0
    W13 = np.zeros((1, 2 * I, d))
    W13[0, 0, 0], W13[0, 2, 0] = 10.0, -9.0     # g0 = 10 > c,  u0 = -9 < -c
    W13[0, 1, 0], W13[0, 3, 0] = -3.0, 2.0      # g1 = -3,      u1 = 2 (inside)
    W2 = np.zeros((1, d, I))
    W2[0, 0, 0], W2[0, 1, 1] = 1.0, 1.0
    x = np.array([[1.0, 0, 0, 0]])
    h, y = oracle.expert_rows(x, W13, W2, [0], [0], [1.0], clamp=c, exact=True)
    silu7 = 7.0 / (1.0 + math.exp(-7.0))
    silum3 = -3.0 / (1.0 + math.exp(3.0))
    np.testing.assert_allclose(h[0], [silu7 * -7.0, silum3 * 2.0], rtol=1e-15)
    np.testing.assert_allclose(y[0, :2], h[0], rtol=1e-15)


def test_h_rounding_is_bf16():
    w = W.WORKLOADS["tiny_fwd"]
    inp = W.make_inputs(w)
    n = 16
    e = np.arange(n, dtype=np.int32) % (w.E + 1)
    h_r, _ = oracle.expert_rows(inp["x"], inp["W13"], inp["W2"], np.arange(n), e, None, w.clamp)
    h_x, _ = oracle.expert_rows(inp["x"], inp["W13"], inp["W2"], np.arange(n), e, None, w.clamp,
                                exact=True)
    as_bf = torch.from_numpy(h_r).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(h_r, as_bf)            # representable in bf16
    lib = torch.from_numpy(h_x).float().to(torch.bfloat16).double().numpy()
    ulp = np.abs(h_x) * 2.0 ** -7
    assert np.mean(h_r == lib) > 0.999                    # torch rounds via fp32 (rare double rounding)
    assert np.all(np.abs(h_r - h_x) <= 0.5 * ulp + 1e-300)


# ----------------------------------------------------------- layer forward

def _dense_layer_torch(x, Wg, W13, W2, ids, w, clamp):
    """The layer written densely: every expert on every token, mixed by the
    [T, E] routing matrix (zero off the selection); torch fp64."""
    T, d = x.shape
    E = Wg.shape[0]
    I = W2.shape[-1]
    R = torch.zeros(T, E, dtype=torch.float64)
    R.scatter_(1, torch.from_numpy(ids.astype(np.int64)), torch.from_numpy(w))
    xt = torch.from_numpy(x)
    y = torch.zeros(T, d, dtype=torch.float64)
    for e in range(E + 1):
        gu = xt @ torch.from_numpy(W13[e]).T
        h = torch.nn.functional.silu(gu[:, :I].clamp(max=clamp)) * gu[:, I:].clamp(-clamp, clamp)
        o = h @ torch.from_numpy(W2[e]).T
        y += (R[:, e:e + 1] if e < E else 1.0) * o
    return y.numpy()


@pytest.mark.parametrize("clamp", [7.0, 0.5])
def test_layer_forward_matches_dense_formulation(clamp):
    rng = np.random.default_rng(11)
    T, d, E, k, I = 12, 24, 6, 2, 8
    x = _rand((T, d), 1.0, rng)
    Wg = _rand((E, d), 0.3, rng)
    W13 = _rand((E + 1, 2 * I, d), 0.3, rng)
    W2 = _rand((E + 1, d, I), 0.3, rng)
    bias = rng.uniform(-0.1, 0.1, (2, E)).astype(np.float32)
    out = oracle.layer_forward(x, Wg, W13, W2, bias, k, 2.5, clamp, exact=True)
    np.testing.assert_allclose(out["z"], x @ Wg.T, rtol=1e-13, atol=1e-13)
    ref = _dense_layer_torch(x, Wg, W13, W2, out["ids"], out["w"], clamp)
    np.testing.assert_allclose(out["y"], ref, rtol=1e-12, atol=1e-12)


def test_layer_forward_composes_expert_rows():
    w = W.WORKLOADS["tiny_fwd"]
    inp = W.make_inputs(w)
    tok = np.array([0, 5, 17, 63])
    out = oracle.layer_forward(inp["x"], inp["W_g"], inp["W13"], inp["W2"], inp["bias"], w.k,
                               w.rho, w.clamp, tok=tok)
    n = len(tok)
    rt = np.repeat(tok, w.k + 1)
    re = np.concatenate([np.concatenate([[w.E], out["ids"][i]]) for i in range(n)]).astype(np.int32)
    rw = np.concatenate([np.concatenate([[1.0], out["w"][i]]) for i in range(n)])
    _, yr = oracle.expert_rows(inp["x"], inp["W13"], inp["W2"], rt, re, rw, w.clamp)
    np.testing.assert_allclose(out["y"], yr.reshape(n, w.k + 1, -1).sum(1), rtol=1e-12,
                               atol=1e-12)


def test_layer_hash_mode_uses_table():
    rng = np.random.default_rng(2)
    T, d, E, k, I, V = 10, 16, 8, 2, 8, 30
    x = _rand((T, d), 1.0, rng)
    Wg = _rand((E, d), 0.3, rng)
    W13 = _rand((E + 1, 2 * I, d), 0.3, rng)
    W2 = _rand((E + 1, d, I), 0.3, rng)
    tab = np.stack([rng.permutation(E)[:k] for _ in range(V)]).astype(np.int32)
    iid = rng.integers(0, V, T).astype(np.int32)
    out = oracle.layer_forward(x, Wg, W13, W2, np.zeros(E, np.float32), k, 2.5, 7.0, mode=1,
                               input_ids=iid, tid2eid=tab, exact=True)
    np.testing.assert_array_equal(out["ids"], tab[iid])
    ref = _dense_layer_torch(x, Wg, W13, W2, out["ids"], out["w"], 7.0)
    np.testing.assert_allclose(out["y"], ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------- backward: finite diffs

def _fd_case(seed=3, clamp=7.0, mode=0):
    rng = np.random.default_rng(seed)
    T, d, E, k, I, V = 6, 12, 6, 2, 8, 20
    c = dict(
        x=_rand((T, d), 1.0, rng), Wg=_rand((E, d), 0.5, rng),
        W13=_rand((E + 1, 2 * I, d), 0.4, rng), W2=_rand((E + 1, d, I), 0.4, rng),
        dY=_rand((T, d), 1.0, rng), bias=rng.uniform(-0.1, 0.1, (2, E)).astype(np.float32),
        vis=(rng.random(T) < 0.5).astype(np.uint8), E=E, k=k, I=I, rho=2.5, clamp=clamp,
        mode=mode,
        iid=rng.integers(0, V, T).astype(np.int32),
        tab=np.stack([rng.permutation(E)[:k] for _ in range(V)]).astype(np.int32))
    return c


def _fwd(c, **over):
    a = dict(c)
    a.update(over)
    hash_kw = dict(mode=1, input_ids=a["iid"], tid2eid=a["tab"]) if a["mode"] == 1 else {}
    out = oracle.layer_forward(a["x"], a["Wg"], a["W13"], a["W2"], a["bias"], a["k"], a["rho"],
                               a["clamp"], is_vision=a["vis"], exact=True, **hash_kw)
    return float((out["y"] * a["dY"]).sum()), out["ids"]


def _fd(c, name, idx, h=1e-6):
    base = c[name]
    p = base.copy()
    p[idx] += h
    lp, ip = _fwd(c, **{name: p})
    p[idx] -= 2 * h
    lm, im = _fwd(c, **{name: p})
    _, i0 = _fwd(c)
    assert np.array_equal(ip, i0) and np.array_equal(im, i0), "selection moved under FD"
    return (lp - lm) / (2 * h)


@pytest.mark.parametrize("clamp,mode", [(7.0, 0), (0.6, 0), (7.0, 1)])
def test_backward_finite_differences(clamp, mode):
    c = _fd_case(clamp=clamp, mode=mode)
    hash_kw = dict(mode=1, input_ids=c["iid"], tid2eid=c["tab"]) if mode == 1 else {}
    bwd = oracle.layer_backward(c["x"], c["Wg"], c["W13"], c["W2"], c["dY"], c["bias"], c["k"],
                                c["rho"], c["clamp"], is_vision=c["vis"], exact=True, **hash_kw)
    fwd = oracle.layer_forward(c["x"], c["Wg"], c["W13"], c["W2"], c["bias"], c["k"], c["rho"],
                               c["clamp"], is_vision=c["vis"], exact=True, **hash_kw)
    rng = np.random.default_rng(0)
    T, d = c["x"].shape
    tol = dict(rtol=2e-6, atol=2e-7)
    for _ in range(6):
        idx = (rng.integers(T), rng.integers(d))
        np.testing.assert_allclose(bwd["dX"][idx], _fd(c, "x", idx), **tol)
    # the gate weight gradient from the oracle's own reduction routine
    dWg = oracle.gate_wgrad_rows(c["x"], bwd["dz"], np.arange(c["E"]))
    for _ in range(6):
        idx = (rng.integers(c["E"]), rng.integers(d))
        np.testing.assert_allclose(dWg[idx], _fd(c, "Wg", idx), **tol)
    ids, w = fwd["ids"], fwd["w"]
    for e in list(np.unique(ids)[:3]) + [c["E"]]:
        if e == c["E"]:
            rt, rw = np.arange(T), np.ones(T)
        else:
            tt, jj = np.nonzero(ids == e)
            rt, rw = tt, w[tt, jj]
        g = oracle.expert_wgrad(c["x"], c["W13"], c["W2"], c["dY"], int(e), rt, rw, c["clamp"],
                                exact=True)
        for _ in range(4):
            i13 = (e, rng.integers(2 * c["I"]), rng.integers(d))
            np.testing.assert_allclose(g["dW13"][i13[1:]], _fd(c, "W13", i13), **tol)
            i2 = (e, rng.integers(d), rng.integers(c["I"]))
            np.testing.assert_allclose(g["dW2"][i2[1:]], _fd(c, "W2", i2), **tol)
    # the routing-weight gradient dw equals the derivative of <dY, y> in w_j
    _, dw = bwd["dw"], bwd["dw"]
    rows = np.repeat(np.arange(T), c["k"])
    _, yj = oracle.expert_rows(c["x"], c["W13"], c["W2"], rows, ids.ravel(), None, c["clamp"],
                               exact=True)
    ref = (yj.reshape(T, c["k"], d) * c["dY"][:, None, :]).sum(-1)
    np.testing.assert_allclose(bwd["dw"], ref, rtol=1e-12, atol=1e-12)


def test_gate_wgrad_rows_is_the_transposed_product():
    # dW_g rows = dz^T x (a library matmul), for all tokens and for a listed
    # subset whose dz rows are given in the listed order; bf16 x bits and
    # fp64 x give the same sums
    rng = np.random.default_rng(12)
    T, d, E = 37, 20, 9
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    xd = x.double()
    dz = rng.standard_normal((T, E)) * (rng.random((T, E)) < 0.4)
    rows = np.array([8, 0, 3, 3], np.int32)
    ref = torch.from_numpy(dz).T.matmul(xd).numpy()[rows]
    np.testing.assert_allclose(oracle.gate_wgrad_rows(x, dz, rows), ref, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.gate_wgrad_rows(xd.numpy(), dz, rows), ref, rtol=1e-13,
                               atol=1e-13)
    tok = np.array([30, 2, 11, 5])
    sub = torch.from_numpy(dz[:4]).T.matmul(xd[torch.from_numpy(tok)]).numpy()[rows]
    np.testing.assert_allclose(oracle.gate_wgrad_rows(x, dz[:4], rows, tok=tok), sub,
                               rtol=1e-13, atol=1e-13)


def test_wgrad_entries_match_full_and_bf16_storage():
    w = W.scaled(W.WORKLOADS["tiny_fwd"], T=32)
    inp = W.make_inputs(w, with_dy=True)
    fwd = oracle.layer_forward(inp["x"], inp["W_g"], inp["W13"], inp["W2"], inp["bias"], w.k,
                               w.rho, w.clamp)
    e = int(np.bincount(fwd["ids"].ravel()).argmax())
    tt, jj = np.nonzero(fwd["ids"] == e)
    rw = fwd["w"][tt, jj]
    rng = np.random.default_rng(1)
    q = 24
    kind = rng.integers(0, 2, q).astype(np.int32)
    qa = np.where(kind == 0, rng.integers(0, w.d, q), rng.integers(0, 2 * w.I, q)).astype(np.int32)
    qb = np.where(kind == 0, rng.integers(0, w.I, q), rng.integers(0, w.d, q)).astype(np.int32)
    for sb in (False, True):
        full = oracle.expert_wgrad(inp["x"], inp["W13"], inp["W2"], inp["dY"], e, tt, rw,
                                   w.clamp, store_bf16=sb)
        ent = oracle.expert_wgrad_entries(inp["x"], inp["W13"], inp["W2"], inp["dY"], e, tt, rw,
                                          w.clamp, kind, qa, qb, store_bf16=sb)
        ref = np.where(kind == 0, full["dW2"][qa % w.d, qb % w.I], full["dW13"][qa, qb])
        np.testing.assert_allclose(ent, ref, rtol=1e-12, atol=1e-12)
    a = oracle.expert_wgrad(inp["x"], inp["W13"], inp["W2"], inp["dY"], e, tt, rw, w.clamp)
    b = oracle.expert_wgrad(inp["x"], inp["W13"], inp["W2"], inp["dY"], e, tt, rw, w.clamp,
                            store_bf16=True)
    # bf16 storage changes the sums only at the bf16 level
    for key in ("dW13", "dW2"):
        rel = np.linalg.norm(a[key] - b[key]) / np.linalg.norm(a[key])
        assert 0 < rel < 1e-2


def test_rows_dA_is_the_transposed_product():
    rng = np.random.default_rng(9)
    T, d, I, G = 7, 24, 10, 3
    dY = _rand((T, d), 1.0, rng)
    W2 = _rand((G, d, I), 0.3, rng)
    rt = np.array([0, 3, 3, 6, 1])
    re = np.array([2, 0, 1, 2, 0], np.int32)
    got = oracle.rows_dA(dY, W2, rt, re)
    ref = np.stack([torch.from_numpy(W2[e]).T.matmul(torch.from_numpy(dY[t])).numpy()
                    for t, e in zip(rt, re)])
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-13)


def test_wgrad2_from_given_h_matches_full_wgrad():
    # with h taken from the oracle's own forward, the two routines agree
    w = W.scaled(W.WORKLOADS["tiny_fwd"], T=24)
    inp = W.make_inputs(w, with_dy=True)
    e = 3
    rt = np.arange(0, w.T, 2)
    rw = np.linspace(0.2, 0.9, len(rt))
    h, _ = oracle.expert_rows(inp["x"], inp["W13"], inp["W2"], rt,
                              np.full(len(rt), e, np.int32), None, w.clamp)
    full = oracle.expert_wgrad(inp["x"], inp["W13"], inp["W2"], inp["dY"], e, rt, rw, w.clamp,
                               want=("dW2",), store_bf16=True)["dW2"]
    qa = np.array([0, 5, 77, 127], np.int32)
    qb = np.array([0, 63, 10, 31], np.int32)
    got = oracle.wgrad2_entries_given_h(inp["dY"], h, rt, rw, qa, qb, store_bf16=True)
    np.testing.assert_allclose(got, full[qa, qb], rtol=1e-12, atol=1e-12)
