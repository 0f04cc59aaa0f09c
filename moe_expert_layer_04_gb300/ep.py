"""Expert parallelism: the routed experts split over the ranks of a process
group, the permuted token rows exchanged with all-to-all.

"Twinkle x 昇腾，率先实现Deepseek-V4系列模型高效训练", FSDP2-4D section:
tokens are dispatched to the rank that owns their expert, computed there,
returned with an all-to-all and combined by routing weight.
"HyperParallel加速DeepSeek-V4.1多模态1M长序列训练" §2.3 MegaMoE: dispatch,
the two expert matmuls and the return.

Partition: E routed experts, W ranks, E % W == 0; rank r owns the contiguous
experts [r E/W, (r+1) E/W) and holds their W13 / W2 plus the shared expert
(replicated, like the gate W_g).  Each rank routes and permutes its own T
tokens; because the permutation is expert-major, the rows bound for rank r'
are one contiguous range of the permuted buffer, so the send sizes come
straight from the per-expert histogram (its prefix sums).

Forward of one step on rank r:
  1. route + permute the local tokens (library calls)
  2. exchange the per-(destination, expert) row counts (all-to-all of W x E/W
     ints), then the routed rows and their routing weights
  3. regroup the received rows from source-major to expert-major order
     (moe_gather_rows) and run the local experts (moe_expert_ffn)
  4. regroup back, return the rows to their sources (all-to-all); the shared
     expert runs locally on the rank's own tokens; combine (moe_combine)
Backward mirrors it: dY rows go to the owners, moe_expert_ffn_backward runs
there (weight gradients stay with the owner), the input gradients and the
routing-weight gradients come back, and moe_router_backward finishes on the
source.  The shared expert's and the gate's weight gradients are sums over
all ranks' tokens: one all-reduce each.

The collectives are torch.distributed (NCCL between GPUs, gloo on CPU); rows
travel as raw bytes.  Before each step every rank records itself in the
process group's key-value store and waits, bounded, for the others: a rank
that left between steps is reported as PeerLostError instead of a
collective that never returns.

`ops` supplies the local compute.  The default, LibMoeOps, is the CUDA
library; tests on CPU ranks pass their own stand-ins to check the exchange
plan without a GPU.
"""
from __future__ import annotations

import datetime
from dataclasses import dataclass

import numpy as np
import torch
import torch.distributed as dist

from . import _lib
from .layer import Dims, gate_route_supported


class PeerLostError(RuntimeError):
    """A rank of the group did not reach the current step in time."""


# ------------------------------------------------------------ the plan

@dataclass
class ExchangePlan:
    """Host-side plan of one step's exchange on one rank."""
    send_splits: list          # rows this rank sends to each rank
    recv_counts: np.ndarray    # [W, E_loc]: rows from each source rank for each local expert
    recv_splits: list          # rows this rank receives from each rank
    regroup: np.ndarray        # int32: expert-major row j <- received row regroup[j]
    inverse: np.ndarray        # int32: received row i <- expert-major row inverse[i]
    local_offsets: np.ndarray  # int32 [E_loc + 1]: the local experts' row ranges

    @property
    def n_recv(self):
        return int(self.regroup.shape[0])


def send_counts(offsets, world: int, E: int) -> np.ndarray:
    """Rows this rank sends to each (destination rank, local expert of it):
    [W, E/W], from the expert-major permutation's offsets [>= E+1]."""
    o = np.asarray(offsets, dtype=np.int64)[: E + 1]
    return np.diff(o).reshape(world, E // world)


def plan_exchange(offsets, recv_counts, world: int, E: int) -> ExchangePlan:
    """The exchange plan from this rank's offsets (expert-major, [>= E+1])
    and the counts the other ranks will send it (recv_counts [W, E/W])."""
    E_loc = E // world
    o = np.asarray(offsets, dtype=np.int64)[: E + 1]
    bounds = o[:: E_loc]                       # [W + 1]: range of each destination's rows
    send_splits = np.diff(bounds).tolist()
    rc = np.asarray(recv_counts, dtype=np.int64).reshape(world, E_loc)
    recv_splits = rc.sum(1).tolist()
    # received order: source-major, then expert, then the source's row order
    start = np.concatenate([[0], np.cumsum(rc.reshape(-1))])[:-1].reshape(world, E_loc)
    parts = [np.arange(start[s, e], start[s, e] + rc[s, e]) for e in range(E_loc)
             for s in range(world)]
    regroup = (np.concatenate(parts) if parts else np.zeros(0, np.int64)).astype(np.int32)
    inverse = np.empty_like(regroup)
    inverse[regroup] = np.arange(regroup.shape[0], dtype=np.int32)
    local_offsets = np.concatenate([[0], np.cumsum(rc.sum(0))]).astype(np.int32)
    return ExchangePlan(send_splits, rc, recv_splits, regroup, inverse, local_offsets)


# ------------------------------------------------------- local compute

class LibMoeOps:
    """The local steps of an expert-parallel layer on the CUDA library."""

    def __init__(self, dims: Dims, fused_route=None):
        self.dims = dims
        ok = gate_route_supported(dims.d, dims.E, dims.k)
        self.fused_route = ok if fused_route is None else bool(fused_route)

    def route(self, L, x, bias, is_vision, logit_offset, mode, input_ids, tid2eid):
        D = self.dims
        if self.fused_route:
            _lib.moe_gate_route(x, L.W_g, logit_offset, bias, is_vision, input_ids, tid2eid, D.T,
                                D.d, D.E, D.k, L.scaling, mode, L.logits, L.ids, L.weights,
                                L.scores_sel, L.modality_counts)
        else:
            _lib.moe_route(x, L.W_g, logit_offset, bias, is_vision, input_ids, tid2eid, D.T, D.d,
                           D.E, D.k, L.scaling, mode, L.logits, L.ids, L.weights, L.scores_sel)

    def permute(self, L, x):
        D = self.dims
        _lib.moe_permute(L.ids, L.weights, x, D.T, D.d, D.E, D.k, L.counts, L.offsets,
                         L.row_token, L.slot_row, L.row_weight, L.x_perm, L.ws)

    def gather_rows(self, src, idx, dst):
        _lib.moe_gather_rows(src, idx, dst)

    def expert_ffn(self, x_rows, offsets, G, W13, W2, row_weight, S, clamp, gu_save, h, y):
        _lib.moe_expert_ffn(x_rows, offsets, G, int(x_rows.shape[0]), W13, W2, row_weight, S,
                            self.dims.d, self.dims.I, clamp, gu_save, h, y, None)

    def expert_ffn_backward(self, args):
        _lib.moe_expert_ffn_backward(args)

    def expert_bwd_workspace(self, rows, recompute, device):
        n = _lib.moe_expert_bwd_workspace_size(max(rows, 1), self.dims.d, self.dims.I, recompute)
        return torch.empty(n, dtype=torch.uint8, device=device)

    def router_backward(self, L, dw_rows, dX_perm, dY_unused, dX):
        D = self.dims
        _lib.moe_router_backward(dw_rows, dX_perm, L.x_perm, L.offsets, L.ids, L.weights,
                                 L.scores_sel, L.slot_row, L.W_g, D.T, D.d, D.E, D.k, L.scaling,
                                 dX, L.dlogits, L.dweights, L.dW_g, L.ws_router)

    def combine(self, L, y_perm, y):
        D = self.dims
        _lib.moe_combine(y_perm, L.slot_row, D.T, D.d, D.k, 1, y)

    def router_workspace(self, device):
        D = self.dims
        return torch.empty(_lib.moe_router_bwd_workspace_size(D.T, D.d, D.E, D.k),
                           dtype=torch.uint8, device=device)

    def workspace(self, device):
        D = self.dims
        return torch.empty(_lib.moe_workspace_size(D.T, D.d, D.E, D.k, D.I, 0), dtype=torch.uint8,
                           device=device)


# ------------------------------------------------------------ the layer

def _bytes(t):
    """A [n, ...] tensor as [n, bytes per row] uint8 (rows travel as bytes)."""
    rb = int(np.prod(t.shape[1:], dtype=np.int64)) * t.element_size()
    return t.contiguous().view(torch.uint8).view(t.shape[0], rb)


class ExpertParallelMoE:
    """One MoE layer whose routed experts are split over the ranks of
    `group` (the default group when None).

    dims: per-rank sizes (T = this rank's tokens; E = all routed experts).
    W_g [E,d]; W13 [E/W + 1, 2I, d] and W2 [E/W + 1, d, I]: this rank's routed
    experts in order, then the shared expert.  store: the group's key-value
    store for the step check (None: no check); peer_timeout in seconds.
    recompute: the backward recomputes the local experts' g|u instead of
    keeping it from the forward.
    """

    def __init__(self, dims: Dims, W_g, W13, W2, scaling: float, clamp: float = 7.0, group=None,
                 ops=None, store=None, peer_timeout: float = 60.0, recompute: bool = False,
                 device=None):
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if dims.E % self.world:
            raise ValueError(f"E = {dims.E} experts do not split over {self.world} ranks")
        self.dims, self.group, self.store = dims, group, store
        self.E_loc = dims.E // self.world
        if W13.shape[0] != self.E_loc + 1 or W2.shape[0] != self.E_loc + 1:
            raise ValueError("W13 / W2 must hold this rank's routed experts and the shared one")
        self.W_g, self.W13, self.W2 = W_g, W13, W2
        self.scaling, self.clamp = float(scaling), float(clamp)
        self.recompute = recompute
        self.peer_timeout = float(peer_timeout)
        self.ops = ops if ops is not None else LibMoeOps(dims)
        self.step = 0
        dev = torch.device(device) if device is not None else W_g.device
        self.device = dev
        D = dims
        e = dict(device=dev)
        self.logits = torch.empty(D.T, D.E, dtype=torch.float32, **e)
        self.ids = torch.empty(D.T, D.k, dtype=torch.int32, **e)
        self.weights = torch.empty(D.T, D.k, dtype=torch.float32, **e)
        self.scores_sel = torch.empty(D.T, D.k, dtype=torch.float32, **e)
        self.modality_counts = torch.empty(2, D.E, dtype=torch.int32, **e)
        self.counts = torch.empty(D.E, dtype=torch.int32, **e)
        self.offsets = torch.empty(D.E + 2, dtype=torch.int32, **e)
        self.row_token = torch.empty(D.R, dtype=torch.int32, **e)
        self.slot_row = torch.empty(D.S, dtype=torch.int32, **e)
        self.row_weight = torch.empty(D.S, dtype=torch.float32, **e)
        self.x_perm = torch.empty(D.R, D.d, dtype=torch.bfloat16, **e)
        self.y_perm = torch.empty(D.R, D.d, dtype=torch.bfloat16, **e)
        self.h_sh = torch.empty(D.T, D.I, dtype=torch.bfloat16, **e)
        self.y = torch.empty(D.T, D.d, dtype=torch.bfloat16, **e)
        self.ws = self.ops.workspace(dev)
        self.ws_router = None
        self.sh_offsets = torch.tensor([0, D.T], dtype=torch.int32, device=dev)
        self.dX = self.dW_g = self.dW13 = self.dW2 = None
        self.dlogits = self.dweights = None

    # -------------------------------------------------------- step check
    def _check_peers(self):
        """Every rank records that it reached this step; wait (bounded) for
        all of them before the step's first collective."""
        self.step += 1
        if self.store is None:
            return
        key = f"moe_ep/step{self.step}/rank"
        self.store.set(f"{key}{self.rank}", "1")
        keys = [f"{key}{r}" for r in range(self.world)]
        try:
            self.store.wait(keys, datetime.timedelta(seconds=self.peer_timeout))
        except Exception as e:  # the store raises on timeout
            missing = [r for r in range(self.world) if not self.store.check([f"{key}{r}"])]
            raise PeerLostError(f"rank(s) {missing} did not reach step {self.step} within "
                                f"{self.peer_timeout:g} s") from e

    # ------------------------------------------------------- exchanges
    def _a2a(self, out, inp, out_splits, in_splits):
        dist.all_to_all_single(_bytes(out), _bytes(inp), out_splits, in_splits, group=self.group)

    def _exchange_counts(self):
        """The per-(destination, expert) counts out, the per-(source, expert)
        counts in; the offsets come to the host once per step."""
        offs = self.offsets.cpu().numpy()
        sc = send_counts(offs, self.world, self.dims.E)
        send = torch.from_numpy(np.ascontiguousarray(sc.astype(np.int64))).to(self.device)
        recv = torch.empty_like(send)
        dist.all_to_all_single(recv, send, group=self.group)
        return plan_exchange(offs, recv.cpu().numpy(), self.world, self.dims.E)

    def _rows(self, n, width, dtype):
        return torch.empty(n, width, dtype=dtype, device=self.device)

    # ---------------------------------------------------------- forward
    def forward(self, x, bias, is_vision=None, logit_offset=None, mode=_lib.MOE_ROUTE_TOPK,
                input_ids=None, tid2eid=None, train=False):
        self._check_peers()
        D, ops = self.dims, self.ops
        self.x = x
        ops.route(self, x, bias, is_vision, logit_offset, mode, input_ids, tid2eid)
        ops.permute(self, x)
        plan = self._exchange_counts()
        self.plan = plan
        n = plan.n_recv
        S = D.S
        # dispatch: routed rows and their routing weights to the experts' owners
        x_recv = self._rows(n, D.d, torch.bfloat16)
        w_recv = torch.empty(n, dtype=torch.float32, device=self.device)
        self._a2a(x_recv, self.x_perm[:S], plan.recv_splits, plan.send_splits)
        self._a2a(w_recv, self.row_weight, plan.recv_splits, plan.send_splits)
        idx = torch.from_numpy(plan.regroup).to(self.device)
        inv = torch.from_numpy(plan.inverse).to(self.device)
        self.regroup_idx, self.inverse_idx = idx, inv
        self.x_loc = self._rows(n, D.d, torch.bfloat16)
        self.w_loc = torch.empty(n, dtype=torch.float32, device=self.device)
        ops.gather_rows(x_recv, idx, self.x_loc)
        ops.gather_rows(w_recv, idx, self.w_loc)
        self.loc_offsets = torch.from_numpy(plan.local_offsets).to(self.device)
        keep_gu = train and not self.recompute
        self.gu_loc = (torch.empty((max(n, 1) + 31) // 32 * 32, 2 * D.I, dtype=torch.float32,
                                   device=self.device) if keep_gu else None)
        self.gu_sh = (torch.empty((D.T + 31) // 32 * 32, 2 * D.I, dtype=torch.float32,
                                  device=self.device) if keep_gu else None)
        y_loc = self._rows(n, D.d, torch.bfloat16)
        if n:
            h_loc = self._rows(n, D.I, torch.bfloat16)
            ops.expert_ffn(self.x_loc, self.loc_offsets, self.E_loc, self.W13[: self.E_loc],
                           self.W2[: self.E_loc], self.w_loc, n, self.clamp, self.gu_loc, h_loc,
                           y_loc)
        # return: back to received order, then to the sources
        y_recv = self._rows(n, D.d, torch.bfloat16)
        ops.gather_rows(y_loc, inv, y_recv)
        self._a2a(self.y_perm[:S], y_recv, plan.send_splits, plan.recv_splits)
        # the shared expert on this rank's own tokens (its rows S.. of x_perm)
        ops.expert_ffn(self.x_perm[S:], self.sh_offsets, 1, self.W13[self.E_loc:],
                       self.W2[self.E_loc:], None, 0, self.clamp, self.gu_sh, self.h_sh,
                       self.y_perm[S:])
        ops.combine(self, self.y_perm, self.y)
        return self.y

    # --------------------------------------------------------- backward
    def backward(self, dY):
        """Backward of the last forward (run with train=True unless the layer
        recomputes).  Returns dX; fills dW13 / dW2 (this rank's experts and
        the shared one, the latter summed over the ranks), dW_g (summed over
        the ranks), dlogits, dweights."""
        self._check_peers()
        D, ops, plan = self.dims, self.ops, self.plan
        S, n = D.S, plan.n_recv
        dev = self.device
        if self.dX is None:
            self.dX = torch.empty(D.T, D.d, dtype=torch.bfloat16, device=dev)
            self.dW_g = torch.empty(D.E, D.d, dtype=torch.float32, device=dev)
            self.dW13 = torch.empty(self.E_loc + 1, 2 * D.I, D.d, dtype=torch.float32, device=dev)
            self.dW2 = torch.empty(self.E_loc + 1, D.d, D.I, dtype=torch.float32, device=dev)
            self.dlogits = torch.empty(D.T, D.E, dtype=torch.float32, device=dev)
            self.dweights = torch.empty(D.T, D.k, dtype=torch.float32, device=dev)
            self.ws_router = ops.router_workspace(dev)
        # dY of every permuted row, then the routed ones to the owners
        dY_perm = self._rows(D.R, D.d, torch.bfloat16)
        ops.gather_rows(dY, self.row_token, dY_perm)
        dY_recv = self._rows(n, D.d, torch.bfloat16)
        self._a2a(dY_recv, dY_perm[:S], plan.recv_splits, plan.send_splits)
        dY_loc = self._rows(n, D.d, torch.bfloat16)
        ops.gather_rows(dY_recv, self.regroup_idx, dY_loc)
        dX_loc = self._rows(n, D.d, torch.bfloat16)
        dw_loc = torch.empty(n, dtype=torch.float32, device=dev)
        if n:
            ops.expert_ffn_backward(dict(
                G=self.E_loc, max_rows=n, S=n, d=D.d, I=D.I, clamp=self.clamp,
                offsets=self.loc_offsets, x_perm=self.x_loc, W13=self.W13[: self.E_loc],
                W2=self.W2[: self.E_loc], row_weight=self.w_loc, gu_save=self.gu_loc,
                dY_perm=dY_loc, dX_perm=dX_loc, dw_rows=dw_loc, dW13=self.dW13[: self.E_loc],
                dW2=self.dW2[: self.E_loc],
                ws=ops.expert_bwd_workspace(n, self.gu_loc is None, dev)))
        else:
            self.dW13[: self.E_loc].zero_()
            self.dW2[: self.E_loc].zero_()
        # back to received order, then to the sources
        dX_recv = self._rows(n, D.d, torch.bfloat16)
        dw_recv = torch.empty(n, dtype=torch.float32, device=dev)
        ops.gather_rows(dX_loc, self.inverse_idx, dX_recv)
        ops.gather_rows(dw_loc, self.inverse_idx, dw_recv)
        dX_perm = self._rows(D.R, D.d, torch.bfloat16)
        dw_rows = torch.empty(S, dtype=torch.float32, device=dev)
        self._a2a(dX_perm[:S], dX_recv, plan.send_splits, plan.recv_splits)
        self._a2a(dw_rows, dw_recv, plan.send_splits, plan.recv_splits)
        # the shared expert on this rank's tokens
        ops.expert_ffn_backward(dict(
            G=1, max_rows=D.T, S=0, d=D.d, I=D.I, clamp=self.clamp, offsets=self.sh_offsets,
            x_perm=self.x_perm[S:], W13=self.W13[self.E_loc:], W2=self.W2[self.E_loc:],
            row_weight=None, gu_save=self.gu_sh, dY_perm=dY_perm[S:], dX_perm=dX_perm[S:],
            dw_rows=None, dW13=self.dW13[self.E_loc:], dW2=self.dW2[self.E_loc:],
            ws=ops.expert_bwd_workspace(D.T, self.gu_sh is None, dev)))
        ops.router_backward(self, dw_rows, dX_perm, dY, self.dX)
        # replicated parameters: sum their gradients over the ranks
        if self.world > 1:
            for g in (self.dW_g, self.dW13[self.E_loc:], self.dW2[self.E_loc:]):
                dist.all_reduce(g, group=self.group)
        return self.dX


__all__ = ["ExpertParallelMoE", "ExchangePlan", "LibMoeOps", "PeerLostError", "plan_exchange",
           "send_counts"]
