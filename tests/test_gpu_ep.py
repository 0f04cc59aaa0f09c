"""The expert-parallel layer on the GPU with the CUDA library (one rank over
NCCL): its exchange degenerates to copies, and every output and gradient must
equal the single-GPU layer's bit for bit -- the same kernels on the same rows
(the routed experts and the shared expert run as separate calls, whose per-row
arithmetic and per-expert row order are those of the one grouped call).
The multi-rank exchange itself is checked on CPU ranks (test_ep_cpu.py)."""
import datetime
import socket

import pytest
import torch
import torch.distributed as dist

from moe_expert_layer_04_gb300 import _lib
from moe_expert_layer_04_gb300 import workloads as W
from moe_expert_layer_04_gb300.ep import ExpertParallelMoE
from moe_expert_layer_04_gb300.layer import Dims, MoELayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nccl_one_rank():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    store = dist.TCPStore("127.0.0.1", port, 1, True, timeout=datetime.timedelta(seconds=60))
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    yield store
    dist.destroy_process_group()


@pytest.mark.parametrize("recompute", [False, True])
def test_ep_one_rank_equals_single_gpu_layer(nccl_one_rank, recompute):
    w = W.Workload("ep_gpu", 600, 256, 32, 4, 128, 2.5, vision_frac=0.3, zipf_s=1.1)
    inp = W.make_inputs(w, device="cuda", with_dy=True)
    D = Dims(w.T, w.d, w.E, w.k, w.I)
    ref = MoELayer(D, dict(W_g=inp["W_g"], W13=inp["W13"], W2=inp["W2"]), w.rho, w.clamp,
                   backward=True, recompute=recompute)
    ref.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"])
    ref.backward(inp["dY"], want_dlogits=True, want_dweights=True)
    ep = ExpertParallelMoE(D, inp["W_g"], inp["W13"], inp["W2"], w.rho, w.clamp,
                           store=nccl_one_rank, peer_timeout=30.0, recompute=recompute)
    for _ in range(2):      # the second step reuses the layer's buffers
        ep.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"], train=True)
        ep.backward(inp["dY"])
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    for name in ("ids", "weights", "y", "dX", "dW_g", "dlogits", "dweights"):
        a, b = getattr(ep, name), getattr(ref, name)
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), name
    E = w.E
    assert torch.equal(ep.dW13[:E], ref.dW13[:E]) and torch.equal(ep.dW2[:E], ref.dW2[:E])
    # the shared expert's weight gradients come from a call of their own, whose
    # tile shape may differ from the one grouped call's (fp32 sums over the
    # same rows in the same order, up to the tensor cores' internal grouping)
    for name in ("dW13", "dW2"):
        a, b = getattr(ep, name)[E], getattr(ref, name)[E]
        assert torch.allclose(a, b, rtol=1e-5, atol=1e-5 * b.abs().max().item()), name


def test_gather_rows_moves_rows_and_zero_fills():
    src = torch.randn(50, 96, device="cuda").to(torch.bfloat16)
    idx = torch.tensor([3, -1, 49, 0, 3], dtype=torch.int32, device="cuda")
    dst = torch.empty(5, 96, dtype=torch.bfloat16, device="cuda")
    _lib.moe_gather_rows(src, idx, dst)
    vals = torch.randn(7, device="cuda")
    out = torch.empty(3, device="cuda")
    _lib.moe_gather_rows(vals, torch.tensor([6, 0, 2], dtype=torch.int32, device="cuda"), out)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    assert torch.equal(dst[0], src[3]) and torch.equal(dst[2], src[49])
    assert torch.equal(dst[3], src[0]) and torch.equal(dst[4], src[3])
    assert torch.count_nonzero(dst[1]).item() == 0
    assert torch.equal(out, vals[[6, 0, 2]])
