"""HostPipeline: forward passes over batches in pinned host memory with the
copies overlapped, against one forward per batch on the device."""
import pytest
import torch

from moe_expert_layer_04_gb300 import _lib
from moe_expert_layer_04_gb300 import workloads as W
from moe_expert_layer_04_gb300.layer import Dims, HostPipeline, MoELayer

pytestmark = pytest.mark.gpu


def test_pipeline_outputs_equal_plain_forwards():
    w = W.Workload("pipe", 700, 256, 64, 4, 128, 2.5, vision_frac=0.3)
    inp = W.make_inputs(w, device="cuda")
    weights = dict(W_g=inp["W_g"], W13=inp["W13"], W2=inp["W2"])
    layer = MoELayer(Dims(w.T, w.d, w.E, w.k, w.I), weights, w.rho, w.clamp)
    # five different batches: ping-pong buffers are reused and must not mix
    xs = [W.normal_bf16((w.T, w.d), 1.0, 0, f"pipe_x{i}", "cuda") for i in range(5)]
    args = (inp["bias"], inp["is_vision"], inp["logit_offset"])
    want = []
    for x in xs:
        want.append(layer.forward(x, *args).clone())
    xs_host = [x.cpu().pin_memory() for x in xs]
    ys_host = [torch.empty(w.T, w.d, dtype=torch.bfloat16).pin_memory() for _ in xs]
    HostPipeline(layer).run(xs_host, ys_host, *args)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    for i, (y, ref) in enumerate(zip(ys_host, want)):
        assert torch.equal(y.view(torch.int16), ref.cpu().view(torch.int16)), i
