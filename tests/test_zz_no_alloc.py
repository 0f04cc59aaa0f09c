"""The allocation-free dispatch entry point, checked against the usual one.

moe_permute_noalloc is for callers that cannot allocate device memory, such as
a plugin whose host program owns every device allocation, or a runtime that
forbids allocating once it runs.  It keeps its scratch in one fixed array
inside the library instead of a caller-provided workspace.  Its results must
equal moe_permute's on the same inputs, and must stay equal on a second call
that reuses the array the first call left behind.
"""
import pytest
import torch

from moe_expert_layer_04_gb300 import _lib
from moe_expert_layer_04_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _dispatch(noalloc, ids, wts, x, T, d, E, k):
    S, R = T * k, T * k + T
    out = dict(counts=torch.empty(E, dtype=torch.int32, device="cuda"),
               offsets=torch.empty(E + 2, dtype=torch.int32, device="cuda"),
               row_token=torch.empty(R, dtype=torch.int32, device="cuda"),
               slot_row=torch.empty(S, dtype=torch.int32, device="cuda"),
               row_weight=torch.empty(S, dtype=torch.float32, device="cuda"),
               x_perm=torch.empty(R, d, dtype=torch.bfloat16, device="cuda"))
    args = (ids, wts, x, T, d, E, k, out["counts"], out["offsets"], out["row_token"],
            out["slot_row"], out["row_weight"], out["x_perm"])
    if noalloc:
        _lib.moe_permute_noalloc(*args)
    else:
        ws = torch.empty(_lib.moe_workspace_size(T, 128, E, k, 64, 0), dtype=torch.uint8,
                         device="cuda")
        _lib.moe_permute(*args, ws)
    torch.cuda.synchronize()
    return out


def test_noalloc_dispatch_equals_workspace_dispatch_on_two_calls():
    # two calls in a row with different shapes: the second one runs on the
    # array the first left behind
    for T, E, k, skew, d in [(3000, 384, 6, 1.1, 256), (1100, 97, 4, 0.0, 128)]:
        ids = W.random_ids(T, E, k, seed=T + E, skew=skew).cuda()
        wts = torch.rand(T, k, device="cuda")
        x = W.normal_bf16((T, d), 1.0, 0, f"noalloc{T}", "cuda")
        got = _dispatch(True, ids, wts, x, T, d, E, k)
        assert _lib.moe_last_device_status() == _lib.MOE_OK
        ref = _dispatch(False, ids, wts, x, T, d, E, k)
        for name in ref:
            a, b = got[name], ref[name]
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), f"{name} differs (T={T}, E={E}, k={k})"


def test_noalloc_rejects_sizes_beyond_its_array():
    small = torch.zeros(16, dtype=torch.int32, device="cuda")
    # ceil(70000 * 8 / 256) * 1024 ints > 2^20
    with pytest.raises(_lib.MoeError) as ei:
        _lib.moe_permute_noalloc(small, None, None, 70000, 128, 1024, 8, small, small, small,
                                 small, None, None)
    assert ei.value.status == _lib.MOE_ERR_UNSUPPORTED


def test_noalloc_at_its_size_limit():
    # ceil(32768 * 8 / 256) * 1024 = 2^20 histogram entries: exactly the whole
    # array; one more token is one chunk too many
    T, E, k, d = 32768, 1024, 8, 8
    ids = W.random_ids(T, E, k, seed=5).cuda()
    wts = torch.rand(T, k, device="cuda")
    x = W.normal_bf16((T, d), 1.0, 0, "noalloc_limit", "cuda")
    got = _dispatch(True, ids, wts, x, T, d, E, k)
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    ref = _dispatch(False, ids, wts, x, T, d, E, k)
    for name in ref:
        a, b = got[name], ref[name]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), f"{name} differs at the size limit"
    ids1 = torch.zeros(T + 1, k, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.MoeError) as ei:
        _lib.moe_permute_noalloc(ids1, None, None, T + 1, d, E, k, *[torch.zeros(
            16, dtype=torch.int32, device="cuda") for _ in range(4)], None, None)
    assert ei.value.status == _lib.MOE_ERR_UNSUPPORTED
