"""Expert parallelism on CPU ranks (gloo): the exchange plan, the row
exchanges in both directions, the regrouping, the shared expert and the
all-reduced gradients, and a rank that leaves between steps.

The local compute here is a stand-in (StubOps): every expert maps a row to a
per-row function of the row, the expert's own weights and the routing weight,
so a row that reaches the wrong rank, the wrong local expert or the wrong
place on its way back changes the result.  Routing and the permutation come
from the oracle.  An expert-parallel run over W ranks must equal a run of the
same layer with every expert on one rank over all ranks' tokens: per-token
outputs and the owners' weight gradients bit for bit (the owner sums its rows
in the same order), the all-reduced gradients to rounding.
"""
import datetime
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from moe_expert_layer_04_gb300 import workloads as W
from moe_expert_layer_04_gb300.ep import (ExpertParallelMoE, PeerLostError, plan_exchange,
                                          send_counts)
from moe_expert_layer_04_gb300.layer import Dims

# ------------------------------------------------------------- the plan


def test_plan_exchange_regroups_source_major_rows_expert_major():
    # 2 ranks, 4 experts: this rank's offsets over the 4 experts, and the
    # counts the two source ranks send for this rank's 2 experts
    offs = np.array([0, 3, 5, 5, 9, 9 + 12, 21 + 4], np.int32)   # [E + 2]
    sc = send_counts(offs, 2, 4)
    np.testing.assert_array_equal(sc, [[3, 2], [0, 4]])
    rc = np.array([[1, 2], [3, 0]])
    p = plan_exchange(offs, rc, 2, 4)
    assert p.send_splits == [5, 4] and p.recv_splits == [3, 3]
    # received: src0 e0 (row 0), src0 e1 (rows 1, 2), src1 e0 (rows 3, 4, 5)
    np.testing.assert_array_equal(p.regroup, [0, 3, 4, 5, 1, 2])
    np.testing.assert_array_equal(p.local_offsets, [0, 4, 6])
    np.testing.assert_array_equal(p.regroup[p.inverse], np.arange(6))
    np.testing.assert_array_equal(p.inverse[p.regroup], np.arange(6))


@pytest.mark.parametrize("world,E", [(1, 8), (2, 8), (4, 16), (3, 9)])
def test_plan_exchange_random_counts_is_a_permutation(world, E):
    rng = np.random.default_rng(world * 100 + E)
    counts = rng.integers(0, 5, E)
    offs = np.concatenate([[0], np.cumsum(counts)])
    rc = rng.integers(0, 6, (world, E // world))
    p = plan_exchange(offs, rc, world, E)
    n = int(rc.sum())
    assert sorted(p.regroup.tolist()) == list(range(n))
    assert p.local_offsets[-1] == n and sum(p.send_splits) == counts.sum()
    # the regrouped order is expert-major: every row of local expert e comes
    # from a received block of e
    start = np.concatenate([[0], np.cumsum(rc.reshape(-1))])[:-1].reshape(rc.shape)
    for e in range(E // world):
        rows = p.regroup[p.local_offsets[e]:p.local_offsets[e + 1]]
        expect = np.concatenate([np.arange(start[s, e], start[s, e] + rc[s, e])
                                 for s in range(world)])
        np.testing.assert_array_equal(rows, expect)


# -------------------------------------------------------- stand-in compute


def _f64(t):
    return t.double() if t.dtype != torch.bfloat16 else t.float().double()


class StubOps:
    """Local steps of the layer on the CPU: routing and permutation from the
    oracle; experts, combine and backward as simple per-row functions."""

    def __init__(self, dims, rho):
        self.dims, self.rho = dims, rho

    def workspace(self, device):
        return None

    def router_workspace(self, device):
        return None

    def expert_bwd_workspace(self, rows, recompute, device):
        return None

    def route(self, L, x, bias, is_vision, logit_offset, mode, input_ids, tid2eid):
        z = oracle.gate_logits(x, L.W_g)
        ids, w, s, _ = oracle.route(z, bias, L.dims.k, self.rho, is_vision=is_vision)
        L.logits.copy_(torch.from_numpy(z))
        L.ids.copy_(torch.from_numpy(ids))
        L.weights.copy_(torch.from_numpy(w))
        L.scores_sel.copy_(torch.from_numpy(s))

    def permute(self, L, x):
        D = self.dims
        c, o, rt, sr = oracle.permute(L.ids.numpy(), D.E)
        L.counts.copy_(torch.from_numpy(c))
        L.offsets[: D.E + 1] = torch.from_numpy(o)
        L.offsets[D.E + 1] = D.R
        L.row_token[: D.S] = torch.from_numpy(rt)
        L.row_token[D.S:] = torch.arange(D.T, dtype=torch.int32)
        L.slot_row.copy_(torch.from_numpy(sr))
        L.row_weight[torch.from_numpy(sr).long()] = L.weights.reshape(-1)
        L.x_perm.copy_(x[L.row_token.long()])

    def gather_rows(self, src, idx, dst):
        i = idx.long()
        out = src[i.clamp(min=0)] if src.shape[0] else torch.zeros_like(dst)
        out[i < 0] = 0
        dst.copy_(out)

    @staticmethod
    def _a(W2, g):
        return _f64(W2[g][:, 0])    # the stand-in expert g: row -> row * a_g

    def expert_ffn(self, x_rows, offsets, G, W13, W2, row_weight, S, clamp, gu_save, h, y):
        o = offsets.tolist()
        for g in range(G):
            a = self._a(W2, g)
            for r in range(o[g], o[g + 1]):
                w = float(row_weight[r]) if (row_weight is not None and r < S) else 1.0
                y[r] = (w * _f64(x_rows[r]) * a).to(y.dtype)

    def expert_ffn_backward(self, args):
        o = args["offsets"].tolist()
        x, dY, dX = args["x_perm"], args["dY_perm"], args["dX_perm"]
        rw, S, dw = args["row_weight"], args["S"], args["dw_rows"]
        for g in range(args["G"]):
            a = self._a(args["W2"], g)
            g13 = torch.zeros(args["dW13"][g].shape, dtype=torch.float64)
            g2 = torch.zeros(args["dW2"][g].shape, dtype=torch.float64)
            for r in range(o[g], o[g + 1]):
                w = float(rw[r]) if (rw is not None and r < S) else 1.0
                xr, dyr = _f64(x[r]), _f64(dY[r])
                dX[r] = (w * dyr * a).to(dX.dtype)
                if dw is not None and r < S:
                    dw[r] = float((xr * a * dyr).sum())
                g2[:, 0] += w * dyr * xr
                g13[0, :] += dyr * a
            args["dW13"][g] = g13.to(args["dW13"].dtype)
            args["dW2"][g] = g2.to(args["dW2"].dtype)

    def router_backward(self, L, dw_rows, dX_perm, dY, dX):
        D = self.dims
        sr = L.slot_row.long().view(D.T, D.k)
        ids = L.ids.long()
        Wg = _f64(L.W_g)
        g = _f64(dX_perm[D.S:]) + _f64(dX_perm[sr]).sum(1) + \
            (_f64(dw_rows)[sr][..., None] * Wg[ids]).sum(1)
        dX.copy_(g.to(dX.dtype))
        L.dweights.copy_(dw_rows[sr])
        L.dlogits.zero_()
        dwg = torch.zeros(D.E, D.d, dtype=torch.float64)
        o = L.offsets.tolist()
        for e in range(D.E):
            for r in range(o[e], o[e + 1]):
                dwg[e] += float(dw_rows[r]) * _f64(L.x_perm[r])
        L.dW_g.copy_(dwg.to(L.dW_g.dtype))

    def combine(self, L, y_perm, y):
        D = self.dims
        sr = L.slot_row.long().view(D.T, D.k)
        y.copy_((_f64(y_perm[D.S:]) + _f64(y_perm[sr]).sum(1)).to(y.dtype))


# ------------------------------------------------------------ the ranks

CASE = W.Workload("ep_cpu", 24, 64, 8, 2, 64, 2.5, vision_frac=0.25)


def _inputs(T_all):
    w = W.scaled(CASE, T=T_all)
    inp = W.make_inputs(w, with_dy=True)
    return w, inp


def _layer(w, inp, group, store, E_range, T, timeout=30.0):
    D = Dims(T, w.d, w.E, w.k, w.I)
    lo, hi = E_range
    W13 = torch.cat([inp["W13"][lo:hi], inp["W13"][w.E:]])
    W2 = torch.cat([inp["W2"][lo:hi], inp["W2"][w.E:]])
    return ExpertParallelMoE(D, inp["W_g"], W13, W2, w.rho, w.clamp, group=group,
                             ops=StubOps(D, w.rho), store=store, peer_timeout=timeout,
                             device="cpu")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ep_worker(rank, world, port, q):
    store = dist.TCPStore("127.0.0.1", port, world, rank == 0,
                          timeout=datetime.timedelta(seconds=60))
    dist.init_process_group("gloo", store=store, rank=rank, world_size=world)
    try:
        T = CASE.T
        w, inp = _inputs(T * world)
        E_loc = w.E // world
        sl = slice(rank * T, (rank + 1) * T)
        ep = _layer(w, inp, None, store, (rank * E_loc, (rank + 1) * E_loc), T)
        y = ep.forward(inp["x"][sl], inp["bias"], inp["is_vision"][sl], train=True).clone()
        dX = ep.backward(inp["dY"][sl]).clone()
        # the same layer with every expert on this rank alone, all tokens (every
        # rank creates every one-rank group: group creation is collective)
        solos = [dist.new_group([r], backend="gloo") for r in range(world)]
        ref = _layer(w, inp, solos[rank], None, (0, w.E), T * world)
        y_ref = ref.forward(inp["x"], inp["bias"], inp["is_vision"], train=True)[sl]
        dX_ref = ref.backward(inp["dY"])[sl]
        lo, hi = rank * E_loc, (rank + 1) * E_loc
        res = dict(
            y=torch.equal(y, y_ref), dX=torch.equal(dX, dX_ref),
            dW13=torch.equal(ep.dW13[:E_loc], ref.dW13[lo:hi]),
            dW2=torch.equal(ep.dW2[:E_loc], ref.dW2[lo:hi]),
            dW13_sh=torch.allclose(ep.dW13[E_loc:], ref.dW13[w.E:], rtol=1e-6, atol=1e-6),
            dW2_sh=torch.allclose(ep.dW2[E_loc:], ref.dW2[w.E:], rtol=1e-6, atol=1e-6),
            dW_g=torch.allclose(ep.dW_g, ref.dW_g, rtol=1e-6, atol=1e-6),
            recv=int(ep.plan.n_recv), sent=int(sum(ep.plan.send_splits)))
        q.put((rank, res))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_expert_parallel_equals_all_experts_on_one_rank(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ep_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(world))
    for r in range(world):
        for k in ("y", "dX", "dW13", "dW2", "dW13_sh", "dW2_sh", "dW_g"):
            assert res[r][k], f"rank {r}: {k} differs from the single-rank layer"
    # every routed slot went out once and came in once
    assert sum(res[r]["sent"] for r in range(world)) == sum(res[r]["recv"] for r in range(world))
    assert sum(res[r]["sent"] for r in range(world)) == world * CASE.T * CASE.k


def _leaving_worker(rank, world, port, q):
    store = dist.TCPStore("127.0.0.1", port, world, rank == 0,
                          timeout=datetime.timedelta(seconds=60))
    dist.init_process_group("gloo", store=store, rank=rank, world_size=world)
    T = CASE.T
    w, inp = _inputs(T * world)
    E_loc = w.E // world
    sl = slice(rank * T, (rank + 1) * T)
    ep = _layer(w, inp, None, store, (rank * E_loc, (rank + 1) * E_loc), T, timeout=2.0)
    ep.forward(inp["x"][sl], inp["bias"], inp["is_vision"][sl])
    if rank == 1:
        q.put((rank, "left"))
        return           # leaves between steps, with nothing in flight
    try:
        ep.forward(inp["x"][sl], inp["bias"], inp["is_vision"][sl])
        q.put((rank, "no error"))
    except PeerLostError as e:
        q.put((rank, f"PeerLostError: {e}"))


def test_rank_that_leaves_between_steps_is_reported_not_waited_for():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_leaving_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res[1] == "left"
    assert res[0].startswith("PeerLostError") and "[1]" in res[0], res[0]
