"""Build, load and bind libmoe.so -- the C ABI of include/moe.h.

The binding only marshals arguments: every function here takes torch tensors
(or ints / floats), checks dtype, device and contiguity, and passes raw device
pointers to the C entry point of the same name.  All arithmetic happens in the
CUDA kernels behind the ABI; there is no fallback.  A missing or unbuildable
library raises.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD, "libmoe.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, \
    MOE_ERR_WORKSPACE = range(6)
MOE_ROUTE_TOPK, MOE_ROUTE_HASH = 0, 1
MOE_FLAG_BACKWARD, MOE_FLAG_RECOMPUTE = 1, 2
MOE_PAIR_EXPERT_GEMM1, MOE_PAIR_EXPERT_GEMM2, MOE_PAIR_DGRAD2, MOE_PAIR_DGRAD1, MOE_PAIR_WGRAD = \
    1 << 1, 1 << 2, 1 << 3, 1 << 4, 1 << 5
MOE_PAIR_ALL = (MOE_PAIR_EXPERT_GEMM1 | MOE_PAIR_EXPERT_GEMM2 | MOE_PAIR_DGRAD2 | MOE_PAIR_DGRAD1
                | MOE_PAIR_WGRAD)

EXPORTS = ["moe_workspace_size", "moe_route", "moe_route_logits", "moe_gate_route", "moe_permute",
           "moe_permute_noalloc",
           "moe_expert_ffn", "moe_expert_ffn_fused", "moe_expert_gemm1", "moe_expert_gemm2", "moe_combine", "moe_backward", "moe_status_string",
           "moe_last_device_status", "moe_selftest_wait_timeout", "moe_selftest_ffn_fused_stall",
           "moe_layer_step_host", "moe_layer_steps_host", "moe_gather_rows", "moe_expert_bwd_workspace_size",
           "moe_expert_ffn_backward", "moe_router_bwd_workspace_size", "moe_router_backward",
           "moe_set_gemm_pairs", "moe_mx_sf_pitch", "moe_mx_quantize", "moe_mx_gather", "moe_expert_ffn_mx",
           "moe_expert_gemm1_mx", "moe_expert_gemm2_mx", "moe_mx_quantize_t",
           "moe_expert_bwd_mx_workspace_size", "moe_expert_ffn_backward_mx",
           "moe_backward_mx_workspace_size", "moe_backward_mx", "moe_mx_quantize_both"]


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: status {status} ({status_string(status)})")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs + [os.path.join(INCLUDE, "moe.h")]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a (in parallel) and link libmoe.so."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    newest = max(os.path.getmtime(p) for p in srcs + _headers())
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    nvcc = _nvcc()
    flags = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
             "-Xptxas", "-v"] if verbose else [ARCH, "-O3", "-lineinfo", "-std=c++17",
                                                "-Xcompiler", "-fPIC", "-I", INCLUDE]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        r = subprocess.run([nvcc, *flags, "-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, ARCH, "-shared", "--cudart=static", "-o", tmp, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_P, _I, _F, _Z, _LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, \
    ctypes.c_longlong


class BwdArgs(ctypes.Structure):
    """Mirror of moe_bwd_args."""
    _fields_ = [("T", _I), ("d", _I), ("E", _I), ("k", _I), ("I", _I),
                ("scaling", _F), ("clamp", _F), ("flags", _I),
                ("x", _P), ("W_g", _P), ("W13", _P), ("W2", _P),
                ("ids", _P), ("weights", _P), ("scores_sel", _P), ("row_weight", _P),
                ("offsets", _P), ("row_token", _P), ("slot_row", _P),
                ("x_perm", _P), ("gu_save", _P), ("dY", _P),
                ("dX", _P), ("dW_g", _P), ("dW13", _P), ("dW2", _P),
                ("dlogits", _P), ("dweights", _P), ("ws", _P), ("ws_bytes", _Z),
                ("stage_events", ctypes.POINTER(_P))]


class ExpertBwdArgs(ctypes.Structure):
    """Mirror of moe_expert_bwd_args."""
    _fields_ = [("G", _I), ("max_rows", _I), ("S", _I), ("d", _I), ("I", _I), ("clamp", _F),
                ("offsets", _P), ("x_perm", _P), ("W13", _P), ("W2", _P), ("row_weight", _P),
                ("gu_save", _P), ("dY_perm", _P), ("dX_perm", _P), ("dw_rows", _P),
                ("dW13", _P), ("dW2", _P), ("ws", _P), ("ws_bytes", _Z)]


class LayerBuffers(ctypes.Structure):
    """Mirror of moe_layer_buffers."""
    _fields_ = [("T", _I), ("d", _I), ("E", _I), ("k", _I), ("I", _I),
                ("scaling", _F), ("clamp", _F), ("flags", _I), ("mode", _I),
                ("W_g", _P), ("W13", _P), ("W2", _P),
                ("logit_offset", _P), ("bias", _P), ("is_vision", _P), ("input_ids", _P),
                ("tid2eid", _P), ("vocab", _I),
                ("x", _P), ("y", _P), ("dY", _P), ("dX", _P),
                ("logits", _P), ("ids", _P), ("weights", _P), ("scores_sel", _P),
                ("modality_counts", _P), ("counts", _P), ("offsets", _P), ("row_token", _P),
                ("slot_row", _P), ("row_weight", _P), ("x_perm", _P), ("h_perm", _P),
                ("y_perm", _P), ("gu_save", _P), ("dW_g", _P), ("dW13", _P), ("dW2", _P),
                ("ws", _P), ("ws_bytes", _Z)]


class LayerIo(ctypes.Structure):
    """Mirror of moe_layer_io."""
    _fields_ = [("x", _P), ("dY", _P), ("y", _P), ("dX", _P)]


class ExpertBwdMxArgs(ctypes.Structure):
    """Mirror of moe_expert_bwd_mx_args."""
    _fields_ = [("G", _I), ("max_rows", _I), ("S", _I), ("d", _I), ("I", _I), ("clamp", _F),
                ("offsets", _P), ("x_perm", _P), ("x_perm_q", _P), ("x_perm_sf", _P),
                ("W13_q", _P), ("W13_sf", _P), ("gu_save", _P), ("h_q", _P), ("h_sf", _P),
                ("W2t_q", _P), ("W2t_sf", _P), ("W13t_q", _P), ("W13t_sf", _P),
                ("row_weight", _P), ("dY_perm", _P), ("dY_perm_q", _P), ("dY_perm_sf", _P),
                ("dX_perm", _P), ("dw_rows", _P), ("dW13", _P), ("dW2", _P),
                ("ws", _P), ("ws_bytes", _Z)]


class BwdMxArgs(ctypes.Structure):
    """Mirror of moe_bwd_mx_args."""
    _fields_ = [("T", _I), ("d", _I), ("E", _I), ("k", _I), ("I", _I),
                ("scaling", _F), ("clamp", _F),
                ("x", _P), ("W_g", _P), ("W13_q", _P), ("W13_sf", _P), ("W2t_q", _P),
                ("W2t_sf", _P), ("W13t_q", _P), ("W13t_sf", _P),
                ("ids", _P), ("weights", _P), ("scores_sel", _P), ("row_weight", _P),
                ("offsets", _P), ("row_token", _P), ("slot_row", _P), ("x_perm_q", _P),
                ("x_perm_sf", _P), ("gu_save", _P), ("h_q", _P), ("h_sf", _P), ("dY", _P),
                ("dX", _P), ("dW_g", _P), ("dW13", _P), ("dW2", _P),
                ("dlogits", _P), ("dweights", _P), ("ws", _P), ("ws_bytes", _Z),
                ("stage_events", ctypes.POINTER(_P))]


MOE_BWD_STAGE_NAMES = ["recompute_gather", "recompute_gemm1", "gather_dY", "dgrad2", "wgrad2",
                       "dgrad1", "wgrad1", "router_bwd", "dX", "dW_g"]
MOE_BWD_STAGES = len(MOE_BWD_STAGE_NAMES)


_SIGS = {
    "moe_workspace_size": ([_I, _I, _I, _I, _I, _I], _Z),
    "moe_route": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P, _P],
                  _I),
    "moe_route_logits": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P], _I),
    "moe_gate_route": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P, _P,
                        _P, _P], _I),
    "moe_permute": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _Z, _P], _I),
    "moe_permute_noalloc": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_expert_ffn": ([_P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _F, _P, _P, _P, _P, _Z, _P], _I),
    "moe_expert_ffn_fused": ([_P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _F, _P, _P, _P, _P, _Z, _P],
                             _I),
    "moe_expert_gemm1": ([_P, _P, _I, _I, _P, _I, _I, _F, _P, _P, _P], _I),
    "moe_expert_gemm2": ([_P, _P, _I, _I, _P, _P, _I, _I, _I, _P, _P], _I),
    "moe_combine": ([_P, _P, _I, _I, _I, _I, _P, _P], _I),
    "moe_backward": ([ctypes.POINTER(BwdArgs), _P], _I),
    "moe_status_string": ([_I], ctypes.c_char_p),
    "moe_last_device_status": ([_P], _I),
    "moe_selftest_wait_timeout": ([_LL, _P], _I),
    "moe_set_gemm_pairs": ([_I], _I),
    "moe_gather_rows": ([_P, _P, _LL, _LL, _I, _P, _P], _I),
    "moe_expert_bwd_workspace_size": ([_I, _I, _I, _I], _Z),
    "moe_expert_ffn_backward": ([ctypes.POINTER(ExpertBwdArgs), _P], _I),
    "moe_router_bwd_workspace_size": ([_I, _I, _I, _I], _Z),
    "moe_router_backward": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P,
                             _P, _P, _Z, _P], _I),
    "moe_layer_step_host": ([ctypes.POINTER(LayerBuffers), _P, _P, _P, _P, _P, _P], _I),
    "moe_layer_steps_host": ([ctypes.POINTER(LayerBuffers), ctypes.POINTER(LayerIo), _I,
                              ctypes.POINTER(_P), ctypes.POINTER(_P), ctypes.POINTER(_P),
                              ctypes.POINTER(_P), _P, _P, _P], _I),
    "moe_selftest_ffn_fused_stall": ([_P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _F, _P, _P, _P, _Z,
                                      _I, _LL, _P], _I),
    "moe_mx_sf_pitch": ([_I], _I),
    "moe_mx_quantize": ([_P, _LL, _I, _P, _P, _P], _I),
    "moe_mx_gather": ([_P, _P, _I, _I, _I, _P, _P, _P], _I),
    "moe_expert_ffn_mx": ([_P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _I, _I, _I, _F, _P, _P, _P,
                           _P, _P], _I),
    "moe_expert_gemm1_mx": ([_P, _P, _P, _I, _I, _P, _P, _I, _I, _F, _P, _P, _P, _P], _I),
    "moe_mx_quantize_t": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "moe_mx_quantize_both": ([_P, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "moe_expert_bwd_mx_workspace_size": ([_I, _I, _I, _I, _I], _Z),
    "moe_expert_ffn_backward_mx": ([ctypes.POINTER(ExpertBwdMxArgs), _P], _I),
    "moe_backward_mx_workspace_size": ([_I, _I, _I, _I, _I, _I], _Z),
    "moe_backward_mx": ([ctypes.POINTER(BwdMxArgs), _P], _I),
    "moe_expert_gemm2_mx": ([_P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _I, _P, _P], _I),
}

_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load (building first if needed) and bind the library."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or build()
            lib = ctypes.CDLL(p)
            for name, (args, res) in _SIGS.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def lib_path() -> str:
    return LIB_PATH


# ----------------------------------------------------------- marshalling

def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, st):
    if st != MOE_OK:
        raise MoeError(fn, st)


BF16, F32, I32, U8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8


def status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_workspace_size(T, d, E, k, I, flags=0) -> int:
    return int(load().moe_workspace_size(T, d, E, k, I, flags))


def moe_route(x, W_g, logit_offset, bias, is_vision, input_ids, tid2eid, T, d, E, k, scaling,
              mode, logits, ids, weights, scores_sel, stream=None):
    vocab = 0 if tid2eid is None else int(tid2eid.shape[0])
    st = load().moe_route(_ptr(x, BF16, "x"), _ptr(W_g, BF16, "W_g"),
                          _ptr(logit_offset, F32, "logit_offset"), _ptr(bias, F32, "bias"),
                          _ptr(is_vision, U8, "is_vision"), _ptr(input_ids, I32, "input_ids"),
                          _ptr(tid2eid, I32, "tid2eid"), vocab, T, d, E, k, float(scaling),
                          int(mode), _ptr(logits, F32, "logits"), _ptr(ids, I32, "ids"),
                          _ptr(weights, F32, "weights"), _ptr(scores_sel, F32, "scores_sel"),
                          _stream(stream))
    _check("moe_route", st)


def moe_route_logits(logits, bias, is_vision, input_ids, tid2eid, T, E, k, scaling, mode, ids,
                     weights, scores_sel, stream=None):
    vocab = 0 if tid2eid is None else int(tid2eid.shape[0])
    st = load().moe_route_logits(_ptr(logits, F32, "logits"), _ptr(bias, F32, "bias"),
                                 _ptr(is_vision, U8, "is_vision"),
                                 _ptr(input_ids, I32, "input_ids"), _ptr(tid2eid, I32, "tid2eid"),
                                 vocab, T, E, k, float(scaling), int(mode),
                                 _ptr(ids, I32, "ids"), _ptr(weights, F32, "weights"),
                                 _ptr(scores_sel, F32, "scores_sel"), _stream(stream))
    _check("moe_route_logits", st)


def moe_gate_route(x, W_g, logit_offset, bias, is_vision, input_ids, tid2eid, T, d, E, k,
                   scaling, mode, logits, ids, weights, scores_sel, modality_counts=None,
                   stream=None):
    vocab = 0 if tid2eid is None else int(tid2eid.shape[0])
    st = load().moe_gate_route(_ptr(x, BF16, "x"), _ptr(W_g, BF16, "W_g"),
                               _ptr(logit_offset, F32, "logit_offset"), _ptr(bias, F32, "bias"),
                               _ptr(is_vision, U8, "is_vision"), _ptr(input_ids, I32, "input_ids"),
                               _ptr(tid2eid, I32, "tid2eid"), vocab, T, d, E, k, float(scaling),
                               int(mode), _ptr(logits, F32, "logits"), _ptr(ids, I32, "ids"),
                               _ptr(weights, F32, "weights"), _ptr(scores_sel, F32, "scores_sel"),
                               _ptr(modality_counts, I32, "modality_counts"), _stream(stream))
    _check("moe_gate_route", st)


def moe_permute(ids, weights, x, T, d, E, k, counts, offsets, row_token, slot_row, row_weight,
                x_perm, ws, stream=None):
    st = load().moe_permute(_ptr(ids, I32, "ids"), _ptr(weights, F32, "weights"),
                            _ptr(x, BF16, "x"), T, d, E, k, _ptr(counts, I32, "counts"),
                            _ptr(offsets, I32, "offsets"), _ptr(row_token, I32, "row_token"),
                            _ptr(slot_row, I32, "slot_row"), _ptr(row_weight, F32, "row_weight"),
                            _ptr(x_perm, BF16, "x_perm"), _ptr(ws, U8, "ws"),
                            0 if ws is None else ws.numel(), _stream(stream))
    _check("moe_permute", st)


def moe_permute_noalloc(ids, weights, x, T, d, E, k, counts, offsets, row_token, slot_row,
                        row_weight, x_perm, stream=None):
    """moe_permute with the library's fixed scratch array instead of a workspace."""
    st = load().moe_permute_noalloc(_ptr(ids, I32, "ids"), _ptr(weights, F32, "weights"),
                                    _ptr(x, BF16, "x"), T, d, E, k, _ptr(counts, I32, "counts"),
                                    _ptr(offsets, I32, "offsets"),
                                    _ptr(row_token, I32, "row_token"),
                                    _ptr(slot_row, I32, "slot_row"),
                                    _ptr(row_weight, F32, "row_weight"),
                                    _ptr(x_perm, BF16, "x_perm"), _stream(stream))
    _check("moe_permute_noalloc", st)


def moe_expert_ffn(x_perm, offsets, G, max_rows, W13, W2, row_weight, S, d, I, clamp, gu_save,
                   h_perm, y_perm, ws=None, stream=None):
    st = load().moe_expert_ffn(_ptr(x_perm, BF16, "x_perm"), _ptr(offsets, I32, "offsets"), G,
                               max_rows, _ptr(W13, BF16, "W13"), _ptr(W2, BF16, "W2"),
                               _ptr(row_weight, F32, "row_weight"), S, d, I, float(clamp),
                               _ptr(gu_save, F32, "gu_save"), _ptr(h_perm, BF16, "h_perm"),
                               _ptr(y_perm, BF16, "y_perm"), _ptr(ws, U8, "ws"),
                               0 if ws is None else ws.numel(), _stream(stream))
    _check("moe_expert_ffn", st)


def moe_expert_ffn_fused(x_perm, offsets, G, max_rows, W13, W2, row_weight, S, d, I, clamp,
                         gu_save, h_perm, y_perm, ws, stream=None):
    st = load().moe_expert_ffn_fused(_ptr(x_perm, BF16, "x_perm"), _ptr(offsets, I32, "offsets"),
                                     G, max_rows, _ptr(W13, BF16, "W13"), _ptr(W2, BF16, "W2"),
                                     _ptr(row_weight, F32, "row_weight"), S, d, I, float(clamp),
                                     _ptr(gu_save, F32, "gu_save"), _ptr(h_perm, BF16, "h_perm"),
                                     _ptr(y_perm, BF16, "y_perm"), _ptr(ws, U8, "ws"),
                                     0 if ws is None else ws.numel(), _stream(stream))
    _check("moe_expert_ffn_fused", st)


def moe_mx_sf_pitch(K):
    return load().moe_mx_sf_pitch(int(K))


def moe_mx_quantize(src, rows, K, q, sf, stream=None):
    st = load().moe_mx_quantize(_ptr(src, BF16, "src"), int(rows), int(K), _ptr(q, U8, "q"),
                                _ptr(sf, U8, "sf"), _stream(stream))
    _check("moe_mx_quantize", st)


def moe_mx_gather(x, slot_row, T, d, k, x_perm_q, x_perm_sf, stream=None):
    st = load().moe_mx_gather(_ptr(x, BF16, "x"), _ptr(slot_row, I32, "slot_row"), T, d, k,
                              _ptr(x_perm_q, U8, "x_perm_q"), _ptr(x_perm_sf, U8, "x_perm_sf"),
                              _stream(stream))
    _check("moe_mx_gather", st)


def moe_expert_ffn_mx(x_perm_q, x_perm_sf, offsets, G, max_rows, W13_q, W13_sf, W2_q, W2_sf,
                      row_weight, S, d, I, clamp, h_q, h_sf, y_perm, gu_save=None, stream=None):
    st = load().moe_expert_ffn_mx(_ptr(x_perm_q, U8, "x_perm_q"), _ptr(x_perm_sf, U8, "x_perm_sf"),
                                  _ptr(offsets, I32, "offsets"), G, max_rows,
                                  _ptr(W13_q, U8, "W13_q"), _ptr(W13_sf, U8, "W13_sf"),
                                  _ptr(W2_q, U8, "W2_q"), _ptr(W2_sf, U8, "W2_sf"),
                                  _ptr(row_weight, F32, "row_weight"), S, d, I, float(clamp),
                                  _ptr(gu_save, F32, "gu_save"), _ptr(h_q, U8, "h_q"),
                                  _ptr(h_sf, U8, "h_sf"), _ptr(y_perm, BF16, "y_perm"),
                                  _stream(stream))
    _check("moe_expert_ffn_mx", st)


def moe_expert_gemm1_mx(x_perm_q, x_perm_sf, offsets, G, max_rows, W13_q, W13_sf, d, I, clamp,
                        h_q, h_sf, gu_save=None, stream=None):
    st = load().moe_expert_gemm1_mx(_ptr(x_perm_q, U8, "x_perm_q"),
                                    _ptr(x_perm_sf, U8, "x_perm_sf"),
                                    _ptr(offsets, I32, "offsets"), G, max_rows,
                                    _ptr(W13_q, U8, "W13_q"), _ptr(W13_sf, U8, "W13_sf"), d, I,
                                    float(clamp), _ptr(gu_save, F32, "gu_save"),
                                    _ptr(h_q, U8, "h_q"), _ptr(h_sf, U8, "h_sf"), _stream(stream))
    _check("moe_expert_gemm1_mx", st)


def moe_expert_gemm2_mx(h_q, h_sf, offsets, G, max_rows, W2_q, W2_sf, row_weight, S, d, I,
                        y_perm, stream=None):
    st = load().moe_expert_gemm2_mx(_ptr(h_q, U8, "h_q"), _ptr(h_sf, U8, "h_sf"),
                                    _ptr(offsets, I32, "offsets"), G, max_rows,
                                    _ptr(W2_q, U8, "W2_q"), _ptr(W2_sf, U8, "W2_sf"),
                                    _ptr(row_weight, F32, "row_weight"), S, d, I,
                                    _ptr(y_perm, BF16, "y_perm"), _stream(stream))
    _check("moe_expert_gemm2_mx", st)


def moe_mx_quantize_t(src, G, R, C, q, sf, stream=None):
    st = load().moe_mx_quantize_t(_ptr(src, BF16, "src"), int(G), int(R), int(C),
                                  _ptr(q, U8, "q"), _ptr(sf, U8, "sf"), _stream(stream))
    _check("moe_mx_quantize_t", st)


def moe_mx_quantize_both(src, G, R, C, q, sf, qt, sft, stream=None):
    st = load().moe_mx_quantize_both(_ptr(src, BF16, "src"), int(G), int(R), int(C),
                                     _ptr(q, U8, "q"), _ptr(sf, U8, "sf"), _ptr(qt, U8, "qt"),
                                     _ptr(sft, U8, "sft"), _stream(stream))
    _check("moe_mx_quantize_both", st)


def moe_expert_bwd_mx_workspace_size(G, max_rows, d, I, recompute) -> int:
    return int(load().moe_expert_bwd_mx_workspace_size(G, max_rows, d, I, int(bool(recompute))))


def moe_backward_mx_workspace_size(T, d, E, k, I, recompute) -> int:
    return int(load().moe_backward_mx_workspace_size(T, d, E, k, I, int(bool(recompute))))


_MX_BWD_TYPES = dict(offsets=I32, x_perm=BF16, x_perm_q=U8, x_perm_sf=U8, W13_q=U8, W13_sf=U8,
                     gu_save=F32, h_q=U8, h_sf=U8, W2t_q=U8, W2t_sf=U8, W13t_q=U8, W13t_sf=U8,
                     row_weight=F32, dY_perm=BF16, dY_perm_q=U8, dY_perm_sf=U8, dX_perm=BF16,
                     dw_rows=F32, dW13=F32, dW2=F32, ws=U8, x=BF16, W_g=BF16, ids=I32,
                     weights=F32, scores_sel=F32, slot_row=I32, row_token=I32, dY=BF16,
                     dX=BF16, dW_g=F32,
                     dlogits=F32, dweights=F32)


def _fill_args(a, args: dict):
    for name, _ in a._fields_:
        if name in ("ws_bytes", "stage_events"):
            continue
        v = args.get(name)
        setattr(a, name, _ptr(v, _MX_BWD_TYPES[name], name) if name in _MX_BWD_TYPES else v)
    a.ws_bytes = 0 if args.get("ws") is None else args["ws"].numel()


def moe_expert_ffn_backward_mx(args: dict, stream=None):
    """args: the fields of moe_expert_bwd_mx_args (tensors for pointers)."""
    a = ExpertBwdMxArgs()
    _fill_args(a, args)
    st = load().moe_expert_ffn_backward_mx(ctypes.byref(a), _stream(stream))
    _check("moe_expert_ffn_backward_mx", st)


def moe_backward_mx(args: dict, stream=None):
    """args: the fields of moe_bwd_mx_args (tensors for pointers)."""
    a = BwdMxArgs()
    _fill_args(a, args)
    a.stage_events = _stage_events(args.get("stage_events"))
    st = load().moe_backward_mx(ctypes.byref(a), _stream(stream))
    _check("moe_backward_mx", st)


def moe_expert_gemm1(x_perm, offsets, G, max_rows, W13, d, I, clamp, gu_save, h_perm,
                     stream=None):
    st = load().moe_expert_gemm1(_ptr(x_perm, BF16, "x_perm"), _ptr(offsets, I32, "offsets"), G,
                                 max_rows, _ptr(W13, BF16, "W13"), d, I, float(clamp),
                                 _ptr(gu_save, F32, "gu_save"), _ptr(h_perm, BF16, "h_perm"),
                                 _stream(stream))
    _check("moe_expert_gemm1", st)


def moe_expert_gemm2(h_perm, offsets, G, max_rows, W2, row_weight, S, d, I, y_perm, stream=None):
    st = load().moe_expert_gemm2(_ptr(h_perm, BF16, "h_perm"), _ptr(offsets, I32, "offsets"), G,
                                 max_rows, _ptr(W2, BF16, "W2"), _ptr(row_weight, F32, "row_weight"),
                                 S, d, I, _ptr(y_perm, BF16, "y_perm"), _stream(stream))
    _check("moe_expert_gemm2", st)


def moe_combine(y_perm, slot_row, T, d, k, with_shared, y, stream=None):
    st = load().moe_combine(_ptr(y_perm, BF16, "y_perm"), _ptr(slot_row, I32, "slot_row"), T, d,
                            k, int(with_shared), _ptr(y, BF16, "y"), _stream(stream))
    _check("moe_combine", st)


def _stage_events(ev):
    """torch.cuda.Event objects (recorded at least once, so that their CUDA
    events exist) or None entries -> a C array of cudaEvent_t (or NULL)."""
    if ev is None:
        return None
    if len(ev) != MOE_BWD_STAGES + 1:
        raise ValueError(f"stage_events: {MOE_BWD_STAGES + 1} entries expected")
    handles = (_P * len(ev))(*[None if e is None else e.cuda_event for e in ev])
    _stage_events.keep = handles   # alive until the call returns
    return ctypes.cast(handles, ctypes.POINTER(_P))


def moe_backward(args: dict, stream=None):
    """args: the fields of moe_bwd_args (tensors for pointers)."""
    a = BwdArgs()
    types = dict(x=BF16, W_g=BF16, W13=BF16, W2=BF16, ids=I32, weights=F32, scores_sel=F32,
                 row_weight=F32, offsets=I32, row_token=I32, slot_row=I32, x_perm=BF16,
                 gu_save=F32, dY=BF16, dX=BF16, dW_g=F32, dW13=F32, dW2=F32, dlogits=F32,
                 dweights=F32, ws=U8)
    for name, _ in BwdArgs._fields_:
        if name in ("ws_bytes", "stage_events"):
            continue
        v = args.get(name)
        if name in types:
            setattr(a, name, _ptr(v, types[name], name))
        else:
            setattr(a, name, v)
    a.ws_bytes = 0 if args.get("ws") is None else args["ws"].numel()
    a.stage_events = _stage_events(args.get("stage_events"))
    st = load().moe_backward(ctypes.byref(a), _stream(stream))
    _check("moe_backward", st)


def moe_last_device_status(stream=None) -> int:
    return int(load().moe_last_device_status(_stream(stream)))


def moe_selftest_wait_timeout(limit_cycles, stream=None):
    st = load().moe_selftest_wait_timeout(int(limit_cycles), _stream(stream))
    _check("moe_selftest_wait_timeout", st)


def moe_set_gemm_pairs(mask: int) -> int:
    """Which grouped matmuls may run as 2-SM pairs (MOE_PAIR_* bits); returns
    the previous mask."""
    return int(load().moe_set_gemm_pairs(int(mask)))


def moe_selftest_ffn_fused_stall(x_perm, offsets, G, max_rows, W13, W2, row_weight, S, d, I,
                                 clamp, h_perm, y_perm, ws, stall_row_tile, limit_cycles,
                                 stream=None):
    """moe_expert_ffn_fused with one row tile's GEMM-2 wait made unreachable
    (test hook of the bounded wait)."""
    st = load().moe_selftest_ffn_fused_stall(
        _ptr(x_perm, BF16, "x_perm"), _ptr(offsets, I32, "offsets"), G, max_rows,
        _ptr(W13, BF16, "W13"), _ptr(W2, BF16, "W2"), _ptr(row_weight, F32, "row_weight"), S, d,
        I, clamp, _ptr(h_perm, BF16, "h_perm"), _ptr(y_perm, BF16, "y_perm"), _ptr(ws, U8, "ws"),
        0 if ws is None else ws.numel(), int(stall_row_tile), int(limit_cycles), _stream(stream))
    _check("moe_selftest_ffn_fused_stall", st)


_LAYER_TYPES = dict(W_g=BF16, W13=BF16, W2=BF16, logit_offset=F32, bias=F32, is_vision=U8,
                    input_ids=I32, tid2eid=I32, x=BF16, y=BF16, dY=BF16, dX=BF16, logits=F32,
                    ids=I32, weights=F32, scores_sel=F32, modality_counts=I32, counts=I32,
                    offsets=I32, row_token=I32, slot_row=I32, row_weight=F32, x_perm=BF16,
                    h_perm=BF16, y_perm=BF16, gu_save=F32, dW_g=F32, dW13=F32, dW2=F32, ws=U8)


def layer_buffers(fields: dict) -> LayerBuffers:
    """A moe_layer_buffers from a dict of ints / floats / CUDA tensors (None
    for NULL).  The caller keeps the tensors alive while the struct is used."""
    L = LayerBuffers()
    for name, _ in LayerBuffers._fields_:
        if name == "ws_bytes":
            continue
        v = fields.get(name)
        if name in _LAYER_TYPES:
            setattr(L, name, _ptr(v, _LAYER_TYPES[name], name))
        else:
            setattr(L, name, 0 if v is None else v)
    L.ws_bytes = 0 if fields.get("ws") is None else fields["ws"].numel()
    return L


def _host_ptr(t, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu" or not t.is_contiguous():
        raise ValueError(f"{name}: must be a contiguous CPU tensor")
    if t.dtype != BF16:
        raise TypeError(f"{name}: expected {BF16}, got {t.dtype}")
    return t.data_ptr()


def moe_layer_step_host(L: LayerBuffers, x_host, dY_host, y_host, dX_host, stream=None,
                        copy_stream=None):
    """One layer step from and to host memory (pinned CPU tensors, [T,d] bf16)."""
    cs = None if copy_stream is None else ctypes.c_void_p(copy_stream.cuda_stream)
    st = load().moe_layer_step_host(ctypes.byref(L), _host_ptr(x_host, "x_host"),
                                    _host_ptr(dY_host, "dY_host"), _host_ptr(y_host, "y_host"),
                                    _host_ptr(dX_host, "dX_host"), _stream(stream), cs)
    _check("moe_layer_step_host", st)


def moe_layer_steps_host(L: LayerBuffers, second: dict, x_host, dY_host, y_host, dX_host,
                         stream=None, copy_in_stream=None, copy_out_stream=None):
    """len(x_host) pipelined layer steps from and to host memory: lists of
    pinned CPU [T,d] bf16 tensors (dY_host / dX_host None for forward-only
    steps); `second` holds the second set of device rows (x, dY, y, dX CUDA
    tensors)."""
    n = len(x_host)
    io = LayerIo(_ptr(second.get("x"), BF16, "x"), _ptr(second.get("dY"), BF16, "dY"),
                 _ptr(second.get("y"), BF16, "y"), _ptr(second.get("dX"), BF16, "dX"))

    def arr(ts, name):
        if ts is None:
            return None
        if len(ts) != n:
            raise ValueError(f"{name}: {n} tensors expected")
        return (_P * n)(*[_host_ptr(t, name) for t in ts])
    xs, dys, ys, dxs = arr(x_host, "x_host"), arr(dY_host, "dY_host"), arr(y_host, "y_host"), \
        arr(dX_host, "dX_host")
    cast = lambda a: None if a is None else ctypes.cast(a, ctypes.POINTER(_P))
    ci = None if copy_in_stream is None else ctypes.c_void_p(copy_in_stream.cuda_stream)
    co = None if copy_out_stream is None else ctypes.c_void_p(copy_out_stream.cuda_stream)
    st = load().moe_layer_steps_host(ctypes.byref(L), ctypes.byref(io), n, cast(xs), cast(dys),
                                     cast(ys), cast(dxs), _stream(stream), ci, co)
    _check("moe_layer_steps_host", st)


def moe_gather_rows(src, idx, dst, stream=None):
    """dst[i] = src[idx[i]] row by row (negative index: zero row).  src and dst
    CUDA tensors with equal row sizes (any dtype, rows a multiple of 4 bytes)."""
    if src.dim() == 1:
        src, dst = src.view(-1, 1), dst.view(-1, 1)
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else \
        dst[0].numel() * dst.element_size()
    n = int(idx.numel())
    if dst.shape[0] != n:
        raise ValueError("dst rows must equal the index count")
    st = load().moe_gather_rows(_ptr(src, None, "src") if src.shape[0] else None,
                                _ptr(idx, I32, "idx"), n, int(src.shape[0]), int(row_bytes),
                                _ptr(dst, None, "dst"), _stream(stream))
    _check("moe_gather_rows", st)


def moe_expert_bwd_workspace_size(max_rows, d, I, recompute) -> int:
    return int(load().moe_expert_bwd_workspace_size(max_rows, d, I, int(bool(recompute))))


def moe_expert_ffn_backward(args: dict, stream=None):
    """args: the fields of moe_expert_bwd_args (tensors for pointers)."""
    a = ExpertBwdArgs()
    types = dict(offsets=I32, x_perm=BF16, W13=BF16, W2=BF16, row_weight=F32, gu_save=F32,
                 dY_perm=BF16, dX_perm=BF16, dw_rows=F32, dW13=F32, dW2=F32, ws=U8)
    for name, _ in ExpertBwdArgs._fields_:
        if name == "ws_bytes":
            continue
        v = args.get(name)
        setattr(a, name, _ptr(v, types[name], name) if name in types else v)
    a.ws_bytes = 0 if args.get("ws") is None else args["ws"].numel()
    st = load().moe_expert_ffn_backward(ctypes.byref(a), _stream(stream))
    _check("moe_expert_ffn_backward", st)


def moe_router_bwd_workspace_size(T, d, E, k) -> int:
    return int(load().moe_router_bwd_workspace_size(T, d, E, k))


def moe_router_backward(dw_rows, dX_perm, x_perm, offsets, ids, weights, scores_sel, slot_row,
                        W_g, T, d, E, k, scaling, dX, dlogits, dweights, dW_g, ws, stream=None):
    st = load().moe_router_backward(
        _ptr(dw_rows, F32, "dw_rows"), _ptr(dX_perm, BF16, "dX_perm"), _ptr(x_perm, BF16, "x_perm"),
        _ptr(offsets, I32, "offsets"), _ptr(ids, I32, "ids"), _ptr(weights, F32, "weights"),
        _ptr(scores_sel, F32, "scores_sel"), _ptr(slot_row, I32, "slot_row"),
        _ptr(W_g, BF16, "W_g"), T, d, E, k, scaling, _ptr(dX, BF16, "dX"),
        _ptr(dlogits, F32, "dlogits"), _ptr(dweights, F32, "dweights"), _ptr(dW_g, F32, "dW_g"),
        _ptr(ws, U8, "ws"), 0 if ws is None else ws.numel(), _stream(stream))
    _check("moe_router_backward", st)
