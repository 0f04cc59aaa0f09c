"""The routed MoE layer on one GPU, as a sequence of C-ABI calls.

This module only allocates device memory (through PyTorch) and calls the
library in order; every step of the layer runs in the library's kernels:

  forward   moe_gate_route (or moe_route) -> moe_permute -> moe_expert_ffn
            (or the one-launch moe_expert_ffn_fused) -> moe_combine
  backward  moe_backward

("HyperParallel加速DeepSeek-V4.1多模态1M长序列训练" §2.3: MegaGate routing
pipeline, then MegaMoE dispatch, two expert matmuls around the clamped
SwiGLU, and result return; the shared expert of "MindSpore HyperParallel
一键开箱DeepSeek-V4.1-Flash" §01 runs as expert group E on every token.)
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib
from ._lib import MOE_FLAG_BACKWARD, MOE_FLAG_RECOMPUTE, MOE_ROUTE_HASH, MOE_ROUTE_TOPK


def gate_route_supported(d: int, E: int, k: int) -> bool:
    """Shapes the one-kernel gate projection + routing (moe_gate_route) takes:
    the logits of 128 tokens for all E experts must fit in tensor memory."""
    return d % 64 == 0 and E % 32 == 0 and 32 <= E <= 512 and 1 <= k <= min(8, E)


def mx_supported(d: int, I: int) -> bool:
    """Shapes the MXFP8 expert matmuls (moe_expert_ffn_mx) take."""
    return d % 256 == 0 and I % 128 == 0


def ffn_fused_supported(d: int, I: int) -> bool:
    """Shapes the one-launch expert FFN (moe_expert_ffn_fused) takes: 256-wide
    tiles in both matmuls."""
    return I % 128 == 0 and d % 256 == 0


@dataclass(frozen=True)
class Dims:
    T: int
    d: int
    E: int
    k: int
    I: int

    @property
    def S(self):
        return self.T * self.k

    @property
    def R(self):
        return self.T * self.k + self.T


class MoELayer:
    """Preallocated buffers for one layer shape, reused across calls.

    weights: dict with W_g [E,d], W13 [E+1,2I,d], W2 [E+1,d,I] (bf16, CUDA).
    fused_route: route with the one-kernel gate projection + routing, which
    also counts the expert load per modality (None: whenever the shape allows).
    fused_ffn: run both expert matmuls in one persistent launch
    (moe_expert_ffn_fused).  Off by default: it is bit-identical to the two
    launches and measures the same on one GPU, and its waits assume that no
    other work shares the GPU's SMs.
    mx: the low-precision variant -- the expert weights are quantised to MXFP8
    here (moe_mx_quantize; again with quantize_weights() after they change),
    each step's token rows are quantised in the dispatch (moe_mx_gather) and
    both expert matmuls take MXFP8 operands (moe_expert_ffn_mx); h between them
    is MXFP8 too.  With backward, the weights also get copies quantised along
    their other axis (moe_mx_quantize_t) and the backward runs the MX dgrad
    matmuls (moe_backward_mx).  Two launches (not fused_ffn).
    """

    def __init__(self, dims: Dims, weights: dict, scaling: float, clamp: float = 7.0,
                 backward: bool = False, recompute: bool = False, device="cuda",
                 fused_route: bool | None = None, fused_ffn: bool = False, mx: bool = False):
        self.dims = dims
        if mx and (fused_ffn or not mx_supported(dims.d, dims.I)):
            raise ValueError(f"the MXFP8 layer runs two launches and needs "
                             f"d % 256 == 0, I % 128 == 0 (got {dims})")
        self.mx = bool(mx)
        ok = gate_route_supported(dims.d, dims.E, dims.k)
        if fused_route and not ok:
            raise ValueError(f"moe_gate_route does not take the shape {dims}")
        self.fused_route = ok if fused_route is None else bool(fused_route)
        if fused_ffn and not ffn_fused_supported(dims.d, dims.I):
            raise ValueError(f"moe_expert_ffn_fused does not take the shape {dims}")
        self.fused_ffn = bool(fused_ffn)
        self.w = weights
        self.scaling = float(scaling)
        self.clamp = float(clamp)
        self.recompute = recompute
        self.backward_enabled = backward
        D = dims
        dev = torch.device(device)
        e = dict(device=dev)
        self.logits = torch.empty(D.T, D.E, dtype=torch.float32, **e)
        self.ids = torch.empty(D.T, D.k, dtype=torch.int32, **e)
        self.weights = torch.empty(D.T, D.k, dtype=torch.float32, **e)
        self.scores_sel = torch.empty(D.T, D.k, dtype=torch.float32, **e)
        self.counts = torch.empty(D.E, dtype=torch.int32, **e)
        # slots per (modality, expert), row 0 text, row 1 vision (fused routing)
        self.modality_counts = (torch.empty(2, D.E, dtype=torch.int32, **e)
                                if self.fused_route else None)
        self.offsets = torch.empty(D.E + 2, dtype=torch.int32, **e)
        self.row_token = torch.empty(D.R, dtype=torch.int32, **e)
        self.slot_row = torch.empty(D.S, dtype=torch.int32, **e)
        self.row_weight = torch.empty(D.S, dtype=torch.float32, **e)
        if self.mx:
            self._init_mx(weights, e)
        else:
            self.x_perm = torch.empty(D.R, D.d, dtype=torch.bfloat16, **e)
            self.h_perm = torch.empty(D.R, D.I, dtype=torch.bfloat16, **e)
        self.y_perm = torch.empty(D.R, D.d, dtype=torch.bfloat16, **e)
        # fp32 g|u, row-block interleaved in blocks of 32 rows (see moe.h)
        self.gu_save = (torch.empty((D.R + 31) // 32 * 32, 2 * D.I, dtype=torch.float32, **e)
                        if backward and not recompute else None)
        self.y = torch.empty(D.T, D.d, dtype=torch.bfloat16, **e)
        flags = (MOE_FLAG_BACKWARD if backward else 0) | (MOE_FLAG_RECOMPUTE if recompute else 0)
        # the MX backward has a workspace of its own
        ws = _lib.moe_workspace_size(D.T, D.d, D.E, D.k, D.I, 0 if self.mx else flags)
        if ws == 0:
            raise ValueError(f"unsupported layer shape {D}")
        self.ws = torch.empty(ws, dtype=torch.uint8, **e)
        if self.mx and backward:
            wsb = _lib.moe_backward_mx_workspace_size(D.T, D.d, D.E, D.k, D.I, recompute)
            if wsb == 0:
                raise ValueError(f"unsupported layer shape {D}")
            self.ws_bwd = torch.empty(wsb, dtype=torch.uint8, **e)
        if backward:
            self.dX = torch.empty(D.T, D.d, dtype=torch.bfloat16, **e)
            self.dW_g = torch.empty(D.E, D.d, dtype=torch.float32, **e)
            self.dW13 = torch.empty(D.E + 1, 2 * D.I, D.d, dtype=torch.float32, **e)
            self.dW2 = torch.empty(D.E + 1, D.d, D.I, dtype=torch.float32, **e)
            self.dlogits = None
            self.dweights = None

    def _init_mx(self, weights, e):
        D = self.dims
        u8 = dict(dtype=torch.uint8, **e)
        pd, pi = _lib.moe_mx_sf_pitch(D.d), _lib.moe_mx_sf_pitch(D.I)
        G = D.E + 1
        self.W13_q = torch.empty(G * 2 * D.I, D.d, **u8)
        self.W13_sf = torch.empty(G * 2 * D.I, pd, **u8)
        self.W2_q = torch.empty(G * D.d, D.I, **u8)
        self.W2_sf = torch.empty(G * D.d, pi, **u8)
        if self.backward_enabled:
            # the dgrad matmuls contract over d (W2) and 2I (W13)
            self.W2t_q = torch.empty(G * D.I, D.d, **u8)
            self.W2t_sf = torch.empty(G * D.I, pd, **u8)
            self.W13t_q = torch.empty(G * D.d, 2 * D.I, **u8)
            self.W13t_sf = torch.empty(G * D.d, _lib.moe_mx_sf_pitch(2 * D.I), **u8)
        self.quantize_weights()
        self.x_perm_q = torch.empty(D.R, D.d, **u8)
        self.x_perm_sf = torch.empty(D.R, pd, **u8)
        self.h_q = torch.empty(D.R, D.I, **u8)
        self.h_sf = torch.empty(D.R, pi, **u8)

    def quantize_weights(self, stream=None):
        """(MX layer) Quantise the expert weights from self.w into the MX
        copies the matmuls read: along d and I for the forward, and with
        backward also along d (W2) and 2I (W13) for the dgrad matmuls."""
        D = self.dims
        G = D.E + 1
        W13, W2 = self.w["W13"], self.w["W2"]
        if self.backward_enabled:
            # one pass over each weight for both copies
            _lib.moe_mx_quantize_both(W13, G, 2 * D.I, D.d, self.W13_q, self.W13_sf,
                                      self.W13t_q, self.W13t_sf, stream)
            _lib.moe_mx_quantize_both(W2, G, D.d, D.I, self.W2_q, self.W2_sf, self.W2t_q,
                                      self.W2t_sf, stream)
            return
        _lib.moe_mx_quantize(W13, G * 2 * D.I, D.d, self.W13_q, self.W13_sf, stream)
        _lib.moe_mx_quantize(W2, G * D.d, D.I, self.W2_q, self.W2_sf, stream)

    # ------------------------------------------------------------ forward
    def route(self, x, bias, is_vision=None, logit_offset=None, mode=MOE_ROUTE_TOPK,
              input_ids=None, tid2eid=None, stream=None):
        D = self.dims
        self.x = x       # the backward reads the forward's input
        if self.fused_route:
            _lib.moe_gate_route(x, self.w["W_g"], logit_offset, bias, is_vision, input_ids,
                                tid2eid, D.T, D.d, D.E, D.k, self.scaling, mode, self.logits,
                                self.ids, self.weights, self.scores_sel, self.modality_counts,
                                stream)
        else:
            _lib.moe_route(x, self.w["W_g"], logit_offset, bias, is_vision, input_ids, tid2eid,
                           D.T, D.d, D.E, D.k, self.scaling, mode, self.logits, self.ids,
                           self.weights, self.scores_sel, stream)

    def dispatch(self, x, stream=None):
        D = self.dims
        _lib.moe_permute(self.ids, self.weights, None if self.mx else x, D.T, D.d, D.E, D.k,
                         self.counts, self.offsets, self.row_token, self.slot_row,
                         self.row_weight, None if self.mx else self.x_perm, self.ws, stream)
        if self.mx:
            _lib.moe_mx_gather(x, self.slot_row, D.T, D.d, D.k, self.x_perm_q, self.x_perm_sf,
                               stream)

    def experts(self, stream=None):
        D = self.dims
        if self.mx:
            _lib.moe_expert_ffn_mx(self.x_perm_q, self.x_perm_sf, self.offsets, D.E + 1, D.R,
                                   self.W13_q, self.W13_sf, self.W2_q, self.W2_sf,
                                   self.row_weight, D.S, D.d, D.I, self.clamp, self.h_q,
                                   self.h_sf, self.y_perm, self.gu_save, stream)
            return
        if self.fused_ffn:
            _lib.moe_expert_ffn_fused(self.x_perm, self.offsets, D.E + 1, D.R, self.w["W13"],
                                      self.w["W2"], self.row_weight, D.S, D.d, D.I, self.clamp,
                                      self.gu_save, self.h_perm, self.y_perm, self.ws, stream)
            return
        _lib.moe_expert_ffn(self.x_perm, self.offsets, D.E + 1, D.R, self.w["W13"], self.w["W2"],
                            self.row_weight, D.S, D.d, D.I, self.clamp, self.gu_save,
                            self.h_perm, self.y_perm, None, stream)

    def expert_gemm1(self, stream=None):
        D = self.dims
        if self.mx:
            _lib.moe_expert_gemm1_mx(self.x_perm_q, self.x_perm_sf, self.offsets, D.E + 1, D.R,
                                     self.W13_q, self.W13_sf, D.d, D.I, self.clamp, self.h_q,
                                     self.h_sf, self.gu_save, stream)
            return
        _lib.moe_expert_gemm1(self.x_perm, self.offsets, D.E + 1, D.R, self.w["W13"], D.d, D.I,
                              self.clamp, self.gu_save, self.h_perm, stream)

    def expert_gemm2(self, stream=None):
        D = self.dims
        if self.mx:
            _lib.moe_expert_gemm2_mx(self.h_q, self.h_sf, self.offsets, D.E + 1, D.R, self.W2_q,
                                     self.W2_sf, self.row_weight, D.S, D.d, D.I, self.y_perm,
                                     stream)
            return
        _lib.moe_expert_gemm2(self.h_perm, self.offsets, D.E + 1, D.R, self.w["W2"],
                              self.row_weight, D.S, D.d, D.I, self.y_perm, stream)

    def combine(self, stream=None, y=None):
        D = self.dims
        _lib.moe_combine(self.y_perm, self.slot_row, D.T, D.d, D.k, 1,
                         self.y if y is None else y, stream)

    def forward(self, x, bias, is_vision=None, logit_offset=None, mode=MOE_ROUTE_TOPK,
                input_ids=None, tid2eid=None, stream=None, y=None):
        """One forward pass; the output goes to self.y, or to `y` ([T, d] bf16)
        when given."""
        self.x = x
        self.route(x, bias, is_vision, logit_offset, mode, input_ids, tid2eid, stream)
        self.dispatch(x, stream)
        self.experts(stream)
        self.combine(stream, y)
        return self.y if y is None else y

    # ----------------------------------------------------------- backward
    def backward(self, dY, want_dlogits=False, want_dweights=False, stream=None,
                 stage_events=None):
        """Backward of the last forward; returns dX.  stage_events: optional
        list of MOE_BWD_STAGES + 1 torch.cuda.Event (recorded once before) that
        the library records around each of its stages."""
        D = self.dims
        if not self.backward_enabled:
            raise RuntimeError("layer built without backward buffers")
        if want_dlogits and self.dlogits is None:
            self.dlogits = torch.empty(D.T, D.E, dtype=torch.float32, device=dY.device)
        if want_dweights and self.dweights is None:
            self.dweights = torch.empty(D.T, D.k, dtype=torch.float32, device=dY.device)
        if self.mx:
            _lib.moe_backward_mx(dict(
                T=D.T, d=D.d, E=D.E, k=D.k, I=D.I, scaling=self.scaling, clamp=self.clamp,
                x=self.x, W_g=self.w["W_g"], W13_q=self.W13_q, W13_sf=self.W13_sf,
                W2t_q=self.W2t_q, W2t_sf=self.W2t_sf, W13t_q=self.W13t_q, W13t_sf=self.W13t_sf,
                ids=self.ids, weights=self.weights, scores_sel=self.scores_sel,
                row_weight=self.row_weight, offsets=self.offsets, row_token=self.row_token,
                slot_row=self.slot_row, x_perm_q=self.x_perm_q, x_perm_sf=self.x_perm_sf, gu_save=self.gu_save,
                h_q=None if self.recompute else self.h_q,
                h_sf=None if self.recompute else self.h_sf,
                dY=dY, dX=self.dX, dW_g=self.dW_g, dW13=self.dW13, dW2=self.dW2,
                dlogits=self.dlogits if want_dlogits else None,
                dweights=self.dweights if want_dweights else None, ws=self.ws_bwd,
                stage_events=stage_events), stream)
            return self.dX
        args = dict(T=D.T, d=D.d, E=D.E, k=D.k, I=D.I, scaling=self.scaling, clamp=self.clamp,
                    flags=MOE_FLAG_RECOMPUTE if self.recompute else 0,
                    x=self.x, W_g=self.w["W_g"], W13=self.w["W13"], W2=self.w["W2"],
                    ids=self.ids, weights=self.weights, scores_sel=self.scores_sel,
                    row_weight=self.row_weight, offsets=self.offsets, row_token=self.row_token,
                    slot_row=self.slot_row,
                    x_perm=None if self.recompute else self.x_perm,
                    gu_save=None if self.recompute else self.gu_save,
                    dY=dY, dX=self.dX, dW_g=self.dW_g, dW13=self.dW13, dW2=self.dW2,
                    dlogits=self.dlogits if want_dlogits else None,
                    dweights=self.dweights if want_dweights else None, ws=self.ws,
                    stage_events=stage_events)
        _lib.moe_backward(args, stream)
        return self.dX


    # ------------------------------------------------- steps from host memory
    def step_host(self, x_host, y_host, dY_host=None, dX_host=None, bias=None, is_vision=None,
                  logit_offset=None, mode=MOE_ROUTE_TOPK, input_ids=None, tid2eid=None,
                  stream=None, copy_stream=None):
        """One step from and to host memory through moe_layer_step_host: x_host
        ([T,d] bf16, pinned CPU) in, y_host out; with dY_host / dX_host also the
        backward (dX out, weight gradients in self.dW13 / dW2 / dW_g).  The
        routing inputs are device tensors as for forward()."""
        self._ensure_host_struct(dY_host is not None, bias, is_vision, logit_offset, mode,
                                 input_ids, tid2eid)
        self.x = self.x_dev
        _lib.moe_layer_step_host(self._host_struct, x_host, dY_host, y_host, dX_host, stream,
                                 copy_stream)

    def steps_host(self, x_hosts, y_hosts, dY_hosts=None, dX_hosts=None, bias=None,
                   is_vision=None, logit_offset=None, mode=MOE_ROUTE_TOPK, input_ids=None,
                   tid2eid=None, stream=None, copy_in_stream=None, copy_out_stream=None):
        """len(x_hosts) steps from and to host memory through
        moe_layer_steps_host, pipelined: the next step's uploads and the last
        step's downloads overlap the compute (lists of pinned CPU [T,d] bf16
        tensors; dY_hosts / dX_hosts for training steps)."""
        D = self.dims
        self._ensure_host_struct(dY_hosts is not None, bias, is_vision, logit_offset, mode,
                                 input_ids, tid2eid)
        if getattr(self, "_io2", None) is None:
            mk = lambda: torch.empty(D.T, D.d, dtype=torch.bfloat16, device=self.y.device)
            self._io2 = dict(x=mk(), y=mk(), dY=mk() if self.backward_enabled else None,
                             dX=mk() if self.backward_enabled else None)
        _lib.moe_layer_steps_host(self._host_struct, self._io2, x_hosts, dY_hosts, y_hosts,
                                  dX_hosts, stream, copy_in_stream, copy_out_stream)

    def _ensure_host_struct(self, train, bias, is_vision, logit_offset, mode, input_ids,
                            tid2eid):
        D = self.dims
        if self.mx:
            raise RuntimeError("the host-memory steps run the bf16 layer")
        if train and not self.backward_enabled:
            raise RuntimeError("layer built without backward buffers")
        key = (id(bias), id(is_vision), id(logit_offset), mode, id(input_ids), id(tid2eid))
        if getattr(self, "_host_key", None) != key:
            dev = self.y.device
            if getattr(self, "x_dev", None) is None:
                self.x_dev = torch.empty(D.T, D.d, dtype=torch.bfloat16, device=dev)
            if self.backward_enabled and getattr(self, "dY_dev", None) is None:
                self.dY_dev = torch.empty(D.T, D.d, dtype=torch.bfloat16, device=dev)
            self._host_refs = (bias, is_vision, logit_offset, input_ids, tid2eid)
            self._host_struct = _lib.layer_buffers(dict(
                T=D.T, d=D.d, E=D.E, k=D.k, I=D.I, scaling=self.scaling, clamp=self.clamp,
                flags=MOE_FLAG_RECOMPUTE if self.recompute else 0, mode=int(mode),
                W_g=self.w["W_g"], W13=self.w["W13"], W2=self.w["W2"],
                logit_offset=logit_offset, bias=bias, is_vision=is_vision, input_ids=input_ids,
                tid2eid=tid2eid, vocab=0 if tid2eid is None else int(tid2eid.shape[0]),
                x=self.x_dev, y=self.y,
                dY=self.dY_dev if self.backward_enabled else None,
                dX=self.dX if self.backward_enabled else None,
                logits=self.logits, ids=self.ids, weights=self.weights,
                scores_sel=self.scores_sel, modality_counts=self.modality_counts,
                counts=self.counts, offsets=self.offsets, row_token=self.row_token,
                slot_row=self.slot_row, row_weight=self.row_weight, x_perm=self.x_perm,
                h_perm=self.h_perm, y_perm=self.y_perm, gu_save=self.gu_save,
                dW_g=getattr(self, "dW_g", None), dW13=getattr(self, "dW13", None),
                dW2=getattr(self, "dW2", None), ws=self.ws))
            self._host_key = key


__all__ = ["Dims", "MoELayer", "MOE_ROUTE_TOPK", "MOE_ROUTE_HASH"]


class HostPipeline:
    """Forward passes over batches that live in pinned host memory.

    Each batch is copied to the device, run through the layer, and its output
    copied back.  Two device buffers each way and one copy stream per
    direction let batch i+1's host-to-device copy and batch i-1's
    device-to-host copy run while the layer computes batch i, so a sequence
    of batches costs about the compute alone; every batch still makes both
    copies.  Batches run in order on the caller's current stream, which
    afterwards also waits for the last copy back.
    """

    def __init__(self, layer: MoELayer):
        D = layer.dims
        dev = layer.y.device
        self.layer = layer
        self.x_dev = [torch.empty(D.T, D.d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.y_dev = [torch.empty(D.T, D.d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.x_ready = [torch.cuda.Event() for _ in range(2)]
        self.x_free = [torch.cuda.Event() for _ in range(2)]
        self.y_ready = [torch.cuda.Event() for _ in range(2)]
        self.y_free = [torch.cuda.Event() for _ in range(2)]

    def _copy_in(self, i, x_host):
        b = i % 2
        with torch.cuda.stream(self.h2d):
            self.h2d.wait_event(self.x_free[b])      # batch i-2 no longer reads x_dev[b]
            self.x_dev[b].copy_(x_host, non_blocking=True)
            self.x_ready[b].record(self.h2d)

    def run(self, xs_host, ys_host, bias, is_vision=None, logit_offset=None, **route_kw):
        """xs_host[i] ([T, d] bf16, pinned) -> layer -> ys_host[i] (pinned)."""
        comp = torch.cuda.current_stream(self.layer.y.device)
        # the copies start after everything the caller queued before
        self.h2d.wait_stream(comp)
        self.d2h.wait_stream(comp)
        n = len(xs_host)
        if n:
            self._copy_in(0, xs_host[0])
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                self._copy_in(i + 1, xs_host[i + 1])
            comp.wait_event(self.x_ready[b])
            comp.wait_event(self.y_free[b])          # batch i-2's output has left y_dev[b]
            self.layer.forward(self.x_dev[b], bias, is_vision, logit_offset, y=self.y_dev[b],
                               **route_kw)
            self.x_free[b].record(comp)
            self.y_ready[b].record(comp)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(self.y_ready[b])
                ys_host[i].copy_(self.y_dev[b], non_blocking=True)
                self.y_free[b].record(self.d2h)
        comp.wait_stream(self.d2h)
