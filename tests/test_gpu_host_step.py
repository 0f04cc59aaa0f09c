"""The whole-layer step from host memory (moe_layer_step_host) against the
same step through the individual calls on device buffers: forward-only and
training steps, with and without a second stream for the copies, in both
routing modes.  Same kernels on the same inputs, so every output and gradient
must agree bit for bit."""
import pytest
import torch

from moe_expert_layer_04_gb300 import _lib
from moe_expert_layer_04_gb300 import workloads as W
from moe_expert_layer_04_gb300.layer import MOE_ROUTE_HASH, MOE_ROUTE_TOPK, Dims, MoELayer

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


@pytest.mark.parametrize("mode,recompute,overlap", [(MOE_ROUTE_TOPK, False, False),
                                                    (MOE_ROUTE_TOPK, True, True),
                                                    (MOE_ROUTE_HASH, False, True)])
def test_host_step_equals_device_calls(mode, recompute, overlap):
    w = W.Workload("host_step", 700, 256, 24, 4, 128, 2.5, vision_frac=0.3,
                   hash_variant=mode == MOE_ROUTE_HASH)
    inp = W.make_inputs(w, device="cuda", with_dy=True)
    weights = dict(W_g=inp["W_g"], W13=inp["W13"], W2=inp["W2"])
    D = Dims(w.T, w.d, w.E, w.k, w.I)
    rk = dict(mode=mode, input_ids=inp.get("input_ids"), tid2eid=inp.get("tid2eid"))
    off = None if mode == MOE_ROUTE_HASH else inp["logit_offset"]
    ref = MoELayer(D, weights, w.rho, w.clamp, backward=True, recompute=recompute)
    ref.forward(inp["x"], inp["bias"], inp["is_vision"], off, **rk)
    ref.backward(inp["dY"])

    lay = MoELayer(D, weights, w.rho, w.clamp, backward=True, recompute=recompute)
    x_h, dY_h = inp["x"].cpu().pin_memory(), inp["dY"].cpu().pin_memory()
    y_h = torch.empty_like(x_h).pin_memory()
    dX_h = torch.empty_like(x_h).pin_memory()
    cs = torch.cuda.Stream() if overlap else None
    for _ in range(2):      # the second step reuses every buffer of the first
        lay.step_host(x_h, y_h, dY_h, dX_h, inp["bias"], inp["is_vision"], off, copy_stream=cs,
                      **rk)
    torch.cuda.current_stream().synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    assert torch.equal(_bits(y_h), _bits(ref.y.cpu()))
    assert torch.equal(_bits(dX_h), _bits(ref.dX.cpu()))
    for name in ("ids", "weights", "dW_g", "dW13", "dW2"):
        assert torch.equal(getattr(lay, name), getattr(ref, name)), name
    # forward only
    y2 = torch.empty_like(x_h).pin_memory()
    lay.step_host(x_h, y2, bias=inp["bias"], is_vision=inp["is_vision"], logit_offset=off, **rk)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(_bits(y2), _bits(ref.y.cpu()))


def test_host_step_rejects_half_a_backward():
    w = W.Workload("host_step_bad", 64, 128, 8, 2, 64, 1.0)
    inp = W.make_inputs(w, device="cuda", with_dy=True)
    lay = MoELayer(Dims(w.T, w.d, w.E, w.k, w.I),
                   dict(W_g=inp["W_g"], W13=inp["W13"], W2=inp["W2"]), w.rho, w.clamp,
                   backward=True)
    x_h = inp["x"].cpu().pin_memory()
    with pytest.raises(_lib.MoeError) as ei:
        lay.step_host(x_h, torch.empty_like(x_h), dY_host=x_h, dX_host=None, bias=inp["bias"])
    assert ei.value.status == _lib.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("train,n", [(True, 4), (False, 3), (True, 1)])
def test_pipelined_host_steps_equal_single_steps(train, n):
    """moe_layer_steps_host over n steps with different inputs: each step's y
    (and dX) and the last step's weight gradients bit for bit those of the
    same steps through moe_layer_step_host one at a time."""
    w = W.Workload("host_steps", 600, 256, 16, 4, 128, 2.5, vision_frac=0.3)
    inp = W.make_inputs(w, device="cuda", with_dy=True)
    weights = dict(W_g=inp["W_g"], W13=inp["W13"], W2=inp["W2"])
    D = Dims(w.T, w.d, w.E, w.k, w.I)
    g = torch.Generator().manual_seed(n)
    xs = [(torch.randn(w.T, w.d, generator=g) * (1 + i)).to(torch.bfloat16).pin_memory()
          for i in range(n)]
    dys = [torch.randn(w.T, w.d, generator=g).to(torch.bfloat16).pin_memory()
           for _ in range(n)] if train else None
    route = dict(bias=inp["bias"], is_vision=inp["is_vision"], logit_offset=inp["logit_offset"])
    ref = MoELayer(D, weights, w.rho, w.clamp, backward=True)
    ref_y, ref_dx = [], []
    for i in range(n):
        y_h = torch.empty_like(xs[i]).pin_memory()
        dx_h = torch.empty_like(xs[i]).pin_memory() if train else None
        ref.step_host(xs[i], y_h, dys[i] if train else None, dx_h, **route)
        torch.cuda.current_stream().synchronize()
        ref_y.append(y_h)
        ref_dx.append(dx_h)
    lay = MoELayer(D, weights, w.rho, w.clamp, backward=True)
    ys = [torch.empty_like(x).pin_memory() for x in xs]
    dxs = [torch.empty_like(x).pin_memory() for x in xs] if train else None
    lay.steps_host(xs, ys, dys, dxs, copy_in_stream=torch.cuda.Stream(),
                   copy_out_stream=torch.cuda.Stream(), **route)
    torch.cuda.current_stream().synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    for i in range(n):
        assert torch.equal(_bits(ys[i]), _bits(ref_y[i])), i
        if train:
            assert torch.equal(_bits(dxs[i]), _bits(ref_dx[i])), i
    if train:
        for name in ("dW_g", "dW13", "dW2"):
            assert torch.equal(getattr(lay, name), getattr(ref, name)), name
