"""The C ABI library on the host: it builds, loads, exports every function that
include/moe.h declares, its argument struct matches the header, and its
host-side validation answers without touching a GPU."""
import ctypes
import os
import re

import pytest

from moe_expert_layer_04_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = open(os.path.join(ROOT, "include", "moe.h")).read()


def declared_functions():
    body = re.sub(r"/\*.*?\*/", "", HEADER, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s+\*?\s*(moe_\w+)\s*\(", body, flags=re.M)))


def test_library_builds_and_exports_every_declared_symbol():
    lib = _lib.load()
    names = declared_functions()
    assert "moe_route" in names and "moe_backward" in names and len(names) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in moe.h but not exported"
    assert sorted(_lib.EXPORTS) == names


@pytest.mark.parametrize("struct,mirror", [("moe_bwd_args", _lib.BwdArgs),
                                           ("moe_layer_buffers", _lib.LayerBuffers),
                                           ("moe_expert_bwd_args", _lib.ExpertBwdArgs),
                                           ("moe_expert_bwd_mx_args", _lib.ExpertBwdMxArgs),
                                           ("moe_bwd_mx_args", _lib.BwdMxArgs),
                                           ("moe_layer_io", _lib.LayerIo)])
def test_structs_match_header(struct, mirror):
    m = re.search(r"typedef struct \{((?:(?!typedef struct).)*?)\} " + struct + ";", HEADER,
                  flags=re.S)
    body = re.sub(r"/\*.*?\*/", "", m.group(1), flags=re.S)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        names = decl.split()[-1] if "," not in decl else decl
        # "int T, d, E, k, I" / "float scaling, clamp" / "const float *weights"
        parts = re.sub(r"^(const\s+)?\w+\s*", "", decl)
        for p in parts.split(","):
            fields.append(re.findall(r"\w+", p)[-1])    # the declarator's name
    assert [f for f, _ in mirror._fields_] == fields


def test_workspace_size_host_logic():
    ws = _lib.moe_workspace_size
    assert ws(4096, 4096, 384, 6, 2048, 0) > 0
    assert ws(4096, 4096, 384, 6, 2048, 1) > ws(4096, 4096, 384, 6, 2048, 0)
    assert ws(4096, 4096, 384, 6, 2048, 3) > ws(4096, 4096, 384, 6, 2048, 1)
    # backward needs at least the permuted dY, dX, [dg|du] and w h buffers
    R = 4096 * 7
    assert ws(4096, 4096, 384, 6, 2048, 1) >= R * (4096 * 2 * 2 + 4096 * 2 + 2048 * 2)
    # unsupported shapes report 0
    assert ws(4096, 4000, 384, 6, 2048, 0) == 0      # d % 128
    assert ws(4096, 4096, 384, 6, 2000, 0) == 0      # I % 64
    assert ws(4096, 4096, 2048, 6, 2048, 0) == 0     # E > 1024
    assert ws(4096, 4096, 384, 33, 2048, 0) == 0     # k > 32
    assert ws(4096, 4096, 4, 6, 2048, 0) == 0        # k > E


def test_validation_rejects_before_any_launch():
    lib = _lib.load()
    nul = None
    # moe_route: null x
    st = lib.moe_route(nul, nul, nul, nul, nul, nul, nul, 0, 8, 128, 4, 2, 1.0, 0, nul, nul, nul,
                       nul, nul)
    assert st == _lib.MOE_ERR_INVALID_ARG
    # bad mode
    st = lib.moe_route_logits(ctypes.c_void_p(16), ctypes.c_void_p(16), nul, nul, nul, 0, 8, 4, 2,
                              1.0, 7, ctypes.c_void_p(16), ctypes.c_void_p(16),
                              ctypes.c_void_p(16), nul)
    assert st == _lib.MOE_ERR_INVALID_ARG
    # moe_gate_route: shapes whose logits tile does not fit in tensor memory,
    # or k above 8, are unsupported (moe_route takes them)
    a = ctypes.c_void_p(4096)
    for (d, E, k) in [(128, 16, 2), (128, 1024, 6), (128, 384, 9), (96, 384, 6), (128, 100, 4)]:
        st = lib.moe_gate_route(a, a, nul, a, nul, nul, nul, 0, 256, d, E, k, 1.0, 0, a, a, a,
                                a, nul, nul)
        assert st == _lib.MOE_ERR_UNSUPPORTED, (d, E, k)
    # ... and a misaligned logits pointer is an invalid argument
    st = lib.moe_gate_route(a, a, nul, a, nul, nul, nul, 0, 256, 128, 64, 4, 1.0, 0,
                            ctypes.c_void_p(4100), a, a, a, nul, nul)
    assert st == _lib.MOE_ERR_INVALID_ARG
    # moe_permute without a workspace
    p = ctypes.c_void_p(256)
    st = lib.moe_permute(p, nul, nul, 8, 128, 4, 2, p, p, p, p, nul, nul, nul, 0, nul)
    assert st == _lib.MOE_ERR_WORKSPACE
    # moe_expert_ffn: unsupported d
    st = lib.moe_expert_ffn(p, p, 2, 64, p, p, nul, 0, 96, 64, 7.0, nul, p, p, nul, 0, nul)
    assert st == _lib.MOE_ERR_UNSUPPORTED
    # moe_expert_ffn: misaligned pointer
    q = ctypes.c_void_p(258)
    st = lib.moe_expert_ffn(q, p, 2, 64, p, p, nul, 0, 128, 64, 7.0, nul, p, p, nul, 0, nul)
    assert st == _lib.MOE_ERR_INVALID_ARG
    # moe_expert_ffn_fused: tiles must be 256 wide in both matmuls, and the
    # readiness counters need a workspace of 4 * (ceil(max_rows/128) + G) bytes
    big = 1 << 20
    assert lib.moe_expert_ffn_fused(p, p, 2, 64, p, p, nul, 0, 384, 128, 7.0, nul, p, p, p, big,
                                    nul) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_expert_ffn_fused(p, p, 2, 64, p, p, nul, 0, 256, 192, 7.0, nul, p, p, p, big,
                                    nul) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_expert_ffn_fused(p, p, 2, 64, p, p, nul, 0, 256, 128, 7.0, nul, p, p, nul, 0,
                                    nul) == _lib.MOE_ERR_WORKSPACE
    assert lib.moe_expert_ffn_fused(p, p, 2, 300, p, p, nul, 0, 256, 128, 7.0, nul, p, p, p, 16,
                                    nul) == _lib.MOE_ERR_WORKSPACE
    # moe_backward: null args, and missing saved state without recompute
    assert lib.moe_backward(None, nul) == _lib.MOE_ERR_INVALID_ARG
    a = _lib.BwdArgs(T=8, d=128, E=4, k=2, I=64, scaling=1.0, clamp=7.0, flags=0)
    assert lib.moe_backward(ctypes.byref(a), nul) == _lib.MOE_ERR_INVALID_ARG
    # non-positive clamp and bad timeout limits
    assert lib.moe_selftest_wait_timeout(0, nul) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_wait_timeout(1 << 40, nul) == _lib.MOE_ERR_INVALID_ARG


def test_mx_calls_host_logic():
    lib = _lib.load()
    # scale rows: K/32 codes padded to 16 bytes
    assert [lib.moe_mx_sf_pitch(K) for K in (32, 64, 512, 544, 2048, 4096)] == [16, 16, 16, 32,
                                                                                 64, 128]
    nul = None
    p = ctypes.c_void_p(256)
    q = ctypes.c_void_p(264)                       # 8-byte aligned only
    # moe_mx_quantize: K a multiple of 32, aligned arrays; zero rows launch nothing
    assert lib.moe_mx_quantize(p, 4, 48, p, p, nul) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_mx_quantize(p, 4, 64, q, p, nul) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_mx_quantize(nul, 4, 64, p, p, nul) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_mx_quantize(p, 0, 64, p, p, nul) == _lib.MOE_OK
    # moe_mx_gather
    assert lib.moe_mx_gather(p, p, 8, 48, 2, p, p, nul) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_mx_gather(p, nul, 8, 64, 2, p, p, nul) == _lib.MOE_ERR_INVALID_ARG
    # moe_expert_ffn_mx: 256-wide tiles in both matmuls, aligned arrays, clamp > 0
    args = lambda d, I, clamp=7.0, hq=p: (p, p, p, 2, 64, p, p, p, p, nul, 0, d, I, clamp, nul,
                                          hq, p, p, nul)
    assert lib.moe_expert_ffn_mx(*args(128, 128)) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_expert_ffn_mx(*args(256, 64)) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_expert_ffn_mx(*args(256, 128, hq=q)) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_ffn_mx(*args(256, 128, clamp=0.0)) == _lib.MOE_ERR_INVALID_ARG
    # moe_mx_quantize_t: R a multiple of 32, G and C at least 1, aligned arrays
    assert lib.moe_mx_quantize_t(p, 2, 48, 8, p, p, nul) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_mx_quantize_t(p, 0, 64, 8, p, p, nul) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_mx_quantize_t(p, 2, 64, 8, q, p, nul) == _lib.MOE_ERR_INVALID_ARG
    # moe_mx_quantize_both: 128 x 128 tiles
    assert lib.moe_mx_quantize_both(p, 1, 96, 128, p, p, p, p, nul) == _lib.MOE_ERR_UNSUPPORTED
    assert lib.moe_mx_quantize_both(p, 1, 128, 128, p, p, q, p, nul) == _lib.MOE_ERR_INVALID_ARG
    # the MX backward: shapes, workspace sizes, missing saved state
    assert lib.moe_backward_mx_workspace_size(64, 128, 8, 2, 128, 0) == 0    # d % 256
    assert lib.moe_backward_mx_workspace_size(64, 256, 8, 2, 64, 0) == 0     # I % 128
    ws0 = lib.moe_backward_mx_workspace_size(64, 256, 8, 2, 128, 0)
    ws1 = lib.moe_backward_mx_workspace_size(64, 256, 8, 2, 128, 1)
    assert 0 < ws0 < ws1
    assert 0 < lib.moe_expert_bwd_mx_workspace_size(3, 300, 256, 128, 0) < \
        lib.moe_expert_bwd_mx_workspace_size(3, 300, 256, 128, 1)
    a = _lib.BwdMxArgs()
    a.T, a.d, a.E, a.k, a.I, a.scaling, a.clamp = 64, 256, 8, 2, 128, 2.5, 7.0
    for name, _ in _lib.BwdMxArgs._fields_[7:]:
        if name not in ("ws_bytes", "stage_events", "dlogits", "dweights"):
            setattr(a, name, 256)
    a.ws_bytes = ws0
    a.gu_save = None                                  # recompute: needs ws1 bytes
    assert lib.moe_backward_mx(ctypes.byref(a), nul) == _lib.MOE_ERR_WORKSPACE
    a.x_perm_q = None                                 # ... and the forward's MX rows
    a.ws_bytes = ws1
    assert lib.moe_backward_mx(ctypes.byref(a), nul) == _lib.MOE_ERR_INVALID_ARG
    a.x_perm_q, a.gu_save, a.h_q = 256, 256, None     # saved g|u without the MX h
    assert lib.moe_backward_mx(ctypes.byref(a), nul) == _lib.MOE_ERR_INVALID_ARG
    a.I = 64
    assert lib.moe_backward_mx(ctypes.byref(a), nul) == _lib.MOE_ERR_UNSUPPORTED
    e = _lib.ExpertBwdMxArgs()
    e.G, e.max_rows, e.S, e.d, e.I, e.clamp = 3, 300, 200, 256, 128, 7.0
    for name, _ in _lib.ExpertBwdMxArgs._fields_[6:]:
        if name not in ("ws_bytes", "dw_rows"):
            setattr(e, name, 256)
    e.ws_bytes = lib.moe_expert_bwd_mx_workspace_size(3, 300, 256, 128, 0) - 1
    assert lib.moe_expert_ffn_backward_mx(ctypes.byref(e), nul) == _lib.MOE_ERR_WORKSPACE
    e.dY_perm_q = 264                                 # 8-byte aligned only
    assert lib.moe_expert_ffn_backward_mx(ctypes.byref(e), nul) == _lib.MOE_ERR_INVALID_ARG


def test_status_strings():
    for s in range(6):
        assert _lib.status_string(s) and _lib.status_string(s) != "unknown status"
    assert _lib.status_string(99) == "unknown status"


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        _lib.moe_combine(x, torch.zeros(16, dtype=torch.int32), 8, 128, 2, 1, x)
