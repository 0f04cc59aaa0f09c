"""Plain fp64 CPU oracle for the routed MoE layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does: it
shares no code, headers or helpers with this oracle.

The arithmetic lives in ``moe_oracle.c`` (plain loops, fp64, one token at a
time, OpenMP over tokens only).  This module compiles it with gcc, loads it
with ctypes and converts numpy / torch-CPU arrays to the C calling
convention.  Float tensors may be bfloat16 (passed as raw 16-bit patterns,
converted exactly inside C) or float64; one call uses one or the other.

Page references (title, section):
  "HyperParallel加速DeepSeek-V4.1多模态1M长序列训练", §2.3 MegaKernel
      (MegaGate, MegaMoE bullets) -- routing, dispatch, expert FFN, return;
  "MindSpore HyperParallel一键开箱DeepSeek-V4.1-Flash", §01 -- shared expert;
  "Twinkle x 昇腾，率先实现Deepseek-V4系列模型高效训练", FSDP2-4D section --
      TopKRouter / HashRouter outputs and the combine by routing weight.

Parity pins: see tests/test_oracle_*.py.  None of the functions is pinned by
a value printed on the pages (they print none); all are pinned by brute
force, closed forms, invariants, library routines and finite differences.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp contraction off so x86 and Arm agree)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int
_D = ctypes.c_double


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            sig = {
                "orc_num_threads": ([], _I),
                "orc_set_num_threads": ([_I], None),
                "orc_gate_logits": ([_P, _P, _I, _P, _I, _P, _I, _I, _I, _P], None),
                "orc_route": ([_P, _P, _P, _I, _P, _P, _I, _I, _P, _I, _I, _D, _I,
                               _P, _P, _P, _P], None),
                "orc_permute": ([_P, _I, _I, _I, _P, _P, _P, _P], None),
                "orc_modality_counts": ([_P, _P, _I, _I, _I, _P], None),
                "orc_expert_rows": ([_P, _P, _P, _I, _I, _P, _P, _P, _I, _I, _D, _I,
                                     _P, _P], None),
                "orc_layer_forward": ([_P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _I,
                                       _I, _P, _I, _I, _I, _I, _D, _D, _I,
                                       _P, _P, _P, _P, _P, _P], None),
                "orc_layer_backward": ([_P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P,
                                        _I, _I, _P, _I, _I, _I, _I, _D, _D, _I,
                                        _P, _P, _P], None),
                "orc_rows_dA": ([_P, _P, _I, _I, _P, _P, _I, _I, _P], None),
                "orc_gate_wgrad_rows": ([_P, _I, _P, _I, _P, _I, _I, _I, _P, _P], None),
                "orc_wgrad2_entries_given_h": ([_P, _P, _I, _I, _P, _P, _I, _I, _I, _I, _P, _P,
                                                _P], None),
                "orc_expert_wgrad": ([_P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I, _D, _I,
                                      _I, _P, _P], None),
                "orc_expert_wgrad_entries": ([_P, _P, _P, _P, _I, _I, _I, _P, _P, _I, _I,
                                              _D, _I, _I, _I, _P, _P, _P, _P], None),
                "orc_mx_quantize": ([_P, _I, _I, _I, _I, _P, _P], None),
                "orc_mx_dequantize": ([_P, _P, _I, _I, _I, _P], None),
                "orc_e4m3_decode_all": ([_P], None),
                "orc_e4m3_encode": ([_P, _I, _P], None),
                "orc_expert_rows_mx": ([_P, _P, _P, _I, _P, _P, _P, _I, _I, _D, _P, _P], None),
                "orc_expert_rows_mx_backward": ([_P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _D,
                                                 _P, _P, _P, _P], None),
                "orc_mx_rows_matmul": ([_P, _P, _I, _I, _I, _P], None),
                "orc_expert_wgrad_mx": ([_P, _P, _P, _P, _I, _P, _P, _I, _I, _D, _P, _P], None),
                "orc_layer_backward_mx": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I,
                                           _I, _P, _I, _I, _I, _I, _D, _D, _P, _P, _P], None),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


# --------------------------------------------------------------- helpers

def _to_np(a):
    """torch tensor or numpy array -> contiguous numpy array (bf16 -> uint16 bits)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                return a.view(torch.int16).numpy().view(np.uint16)
            return a.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a)


def _floats(*arrays):
    """Convert the float tensors of one call to a common C form: all bf16 bit
    patterns (flag 1) or all float64 (flag 0)."""
    conv = [_to_np(a) for a in arrays]
    if all(c.dtype == np.uint16 for c in conv):
        return conv, 1
    return [np.ascontiguousarray(c, dtype=np.float64) if c.dtype != np.uint16 else
            _bf16_bits_to_f64(c) for c in conv], 0


def _bf16_bits_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _opt(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(_to_np(a), dtype=dtype)


def _tok(tok, n_default):
    if tok is None:
        return None, n_default
    t = np.ascontiguousarray(_to_np(tok), dtype=np.int64)
    return t, int(t.shape[0])


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


# ------------------------------------------------------------- the steps

def gate_logits(x, W_g, offset=None, tok=None, exact=False):
    """z = x W_g^T (+ offset), fp64 accumulation, rounded to fp32 unless exact."""
    (xn, wn), bf = _floats(x, W_g)
    E, d = wn.shape
    tk, n = _tok(tok, xn.shape[0])
    off = _opt(offset, np.float32)
    z = np.empty((n, E), np.float64)
    _load().orc_gate_logits(_ptr(xn), _ptr(wn), bf, _ptr(off), n, _ptr(tk), d, E, int(exact),
                            _ptr(z))
    return z


def route(z, bias, k, rho, is_vision=None, mode=0, input_ids=None, tid2eid=None, tok=None,
          exact=False):
    """Routing of tokens from their logits z [n, E].

    Returns ids int32 [n,k], w [n,k], s_sel [n,k], margin [n] (fp64 arrays holding
    fp32 values unless exact)."""
    zn = np.ascontiguousarray(_to_np(z), dtype=np.float64)
    n, E = zn.shape
    tk, _ = _tok(tok, n)
    b = np.ascontiguousarray(_to_np(bias), dtype=np.float32).reshape(-1)
    if b.shape[0] == E:
        b = np.concatenate([b, b])
    vis = _opt(is_vision, np.uint8)
    ii = _opt(input_ids, np.int32)
    tab = _opt(tid2eid, np.int32)
    vocab = 0 if tab is None else int(tab.shape[0])
    ids = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    s = np.empty((n, k), np.float64)
    m = np.empty((n,), np.float64)
    _load().orc_route(_ptr(zn), _ptr(b), _ptr(vis), int(mode), _ptr(ii), _ptr(tab), vocab, n,
                      _ptr(tk), E, k, float(rho), int(exact), _ptr(ids), _ptr(w), _ptr(s),
                      _ptr(m))
    return ids, w, s, m


def permute(ids, E):
    """Stable expert-major permutation: counts, offsets [E+1], row_token, slot_row."""
    idn = np.ascontiguousarray(_to_np(ids), dtype=np.int32)
    T, k = idn.shape
    counts = np.empty((E,), np.int32)
    offsets = np.empty((E + 1,), np.int32)
    row_token = np.empty((T * k,), np.int32)
    slot_row = np.empty((T * k,), np.int32)
    _load().orc_permute(_ptr(idn), T, E, k, _ptr(counts), _ptr(offsets), _ptr(row_token),
                        _ptr(slot_row))
    return counts, offsets, row_token, slot_row


def modality_counts(ids, is_vision, E):
    """Slots per (modality, expert): [2, E], row 0 text, row 1 vision."""
    idn = np.ascontiguousarray(_to_np(ids), dtype=np.int32)
    T, k = idn.shape
    vis = None if is_vision is None else np.ascontiguousarray(_to_np(is_vision), dtype=np.uint8)
    counts = np.empty((2, E), np.int32)
    _load().orc_modality_counts(_ptr(idn), None if vis is None else _ptr(vis), T, E, k,
                                _ptr(counts))
    return counts


def expert_rows(x, W13, W2, row_tok, row_exp, row_w, clamp, exact=False):
    """Per-row expert FFN: y[r] = row_w[r] * W2[e] h(x[row_tok[r]]); returns (h, y)."""
    (xn, w13, w2), bf = _floats(x, W13, W2)
    d = xn.shape[1]
    I = w2.shape[-1]
    rt = np.ascontiguousarray(_to_np(row_tok), dtype=np.int64)
    re = np.ascontiguousarray(_to_np(row_exp), dtype=np.int32)
    rw = _opt(row_w, np.float64)
    n = rt.shape[0]
    h = np.empty((n, I), np.float64)
    y = np.empty((n, d), np.float64)
    _load().orc_expert_rows(_ptr(xn), _ptr(w13), _ptr(w2), bf, n, _ptr(rt), _ptr(re), _ptr(rw),
                            d, I, float(clamp), int(exact), _ptr(h), _ptr(y))
    return h, y


def _route_args(bias, E, is_vision, input_ids, tid2eid, offset):
    b = np.ascontiguousarray(_to_np(bias), dtype=np.float32).reshape(-1)
    if b.shape[0] == E:
        b = np.concatenate([b, b])
    tab = _opt(tid2eid, np.int32)
    return (b, _opt(is_vision, np.uint8), _opt(input_ids, np.int32), tab,
            0 if tab is None else int(tab.shape[0]), _opt(offset, np.float32))


def layer_forward(x, W_g, W13, W2, bias, k, rho, clamp, is_vision=None, mode=0,
                  input_ids=None, tid2eid=None, offset=None, tok=None, exact=False):
    """Forward of the layer for the listed tokens (all when tok is None).

    Returns dict(z, ids, w, s_sel, margin, y)."""
    (xn, wg, w13, w2), bf = _floats(x, W_g, W13, W2)
    E, d = wg.shape
    I = w2.shape[-1]
    b, vis, ii, tab, vocab, off = _route_args(bias, E, is_vision, input_ids, tid2eid, offset)
    tk, n = _tok(tok, xn.shape[0])
    z = np.empty((n, E), np.float64)
    ids = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    s = np.empty((n, k), np.float64)
    m = np.empty((n,), np.float64)
    y = np.empty((n, d), np.float64)
    _load().orc_layer_forward(_ptr(xn), _ptr(wg), _ptr(w13), _ptr(w2), bf, _ptr(off), _ptr(b),
                              _ptr(vis), int(mode), _ptr(ii), _ptr(tab), vocab, n, _ptr(tk),
                              d, E, k, I, float(rho), float(clamp), int(exact), _ptr(z),
                              _ptr(ids), _ptr(w), _ptr(s), _ptr(m), _ptr(y))
    return dict(z=z, ids=ids, w=w, s_sel=s, margin=m, y=y)


def layer_backward(x, W_g, W13, W2, dY, bias, k, rho, clamp, is_vision=None, mode=0,
                   input_ids=None, tid2eid=None, offset=None, tok=None, exact=False):
    """Token-local backward for the listed tokens: dict(dX [n,d], dz [n,E], dw [n,k])."""
    (xn, wg, w13, w2, dy), bf = _floats(x, W_g, W13, W2, dY)
    E, d = wg.shape
    I = w2.shape[-1]
    b, vis, ii, tab, vocab, off = _route_args(bias, E, is_vision, input_ids, tid2eid, offset)
    tk, n = _tok(tok, xn.shape[0])
    dX = np.empty((n, d), np.float64)
    dz = np.empty((n, E), np.float64)
    dw = np.empty((n, k), np.float64)
    _load().orc_layer_backward(_ptr(xn), _ptr(wg), _ptr(w13), _ptr(w2), _ptr(dy), bf, _ptr(off),
                               _ptr(b), _ptr(vis), int(mode), _ptr(ii), _ptr(tab), vocab, n,
                               _ptr(tk), d, E, k, I, float(rho), float(clamp), int(exact),
                               _ptr(dX), _ptr(dz), _ptr(dw))
    return dict(dX=dX, dz=dz, dw=dw)


def gate_wgrad_rows(x, dz, rows, tok=None):
    """Rows of the gate weight gradient, dW_g[e] = sum_t dz[t, e] x[t] for each
    expert e in `rows`, over the tokens of dz [n, E] (x rows tok, or 0..n-1)."""
    (xn,), bf = _floats(x)
    d = xn.shape[1]
    dzn = np.ascontiguousarray(_to_np(dz), dtype=np.float64)
    n, E = dzn.shape
    tk, _ = _tok(tok, n)
    rr = np.ascontiguousarray(rows, dtype=np.int32)
    out = np.empty((rr.shape[0], d), np.float64)
    _load().orc_gate_wgrad_rows(_ptr(xn), bf, _ptr(dzn), n, _ptr(tk), d, E, rr.shape[0], _ptr(rr),
                                _ptr(out))
    return out


def rows_dA(dY, W2, row_tok, row_exp):
    """dA[r] = dY[row_tok[r]] W2[row_exp[r]] (length I): the gradient at the
    SwiGLU output of each listed expert row, before the routing weight."""
    (dy, w2), bf = _floats(dY, W2)
    d = dy.shape[1]
    I = w2.shape[-1]
    rt = np.ascontiguousarray(_to_np(row_tok), dtype=np.int64)
    re = np.ascontiguousarray(_to_np(row_exp), dtype=np.int32)
    out = np.empty((rt.shape[0], I), np.float64)
    _load().orc_rows_dA(_ptr(dy), _ptr(w2), bf, rt.shape[0], _ptr(rt), _ptr(re), d, I, _ptr(out))
    return out


def wgrad2_entries_given_h(dY, h_rows, row_tok, row_w, qa, qb, store_bf16=True):
    """dW2 entries sum_r dY[row_tok[r], qa] * (row_w[r] h_rows[r, qb]) from given
    intermediate rows (checks the weight-gradient matmul on its own)."""
    (dy, h), bf = _floats(dY, h_rows)
    d = dy.shape[1]
    I = h.shape[1]
    rt = np.ascontiguousarray(_to_np(row_tok), dtype=np.int64)
    rw = np.ascontiguousarray(_to_np(row_w), dtype=np.float64)
    a = np.ascontiguousarray(qa, dtype=np.int32)
    b = np.ascontiguousarray(qb, dtype=np.int32)
    out = np.empty((a.shape[0],), np.float64)
    _load().orc_wgrad2_entries_given_h(_ptr(dy), _ptr(h), bf, rt.shape[0], _ptr(rt), _ptr(rw), d,
                                       I, int(store_bf16), a.shape[0], _ptr(a), _ptr(b),
                                       _ptr(out))
    return out


def expert_wgrad(x, W13, W2, dY, e, row_tok, row_w, clamp, exact=False, want=("dW13", "dW2"),
                 store_bf16=False):
    """Full weight gradients of expert e from its rows: dict(dW13 [2I,d], dW2 [d,I]).

    store_bf16 rounds the stored per-row factors [dg|du] and w*h to bf16."""
    (xn, w13, w2, dy), bf = _floats(x, W13, W2, dY)
    d = xn.shape[1]
    I = w2.shape[-1]
    rt = np.ascontiguousarray(_to_np(row_tok), dtype=np.int64)
    rw = np.ascontiguousarray(_to_np(row_w), dtype=np.float64)
    out = {}
    g13 = np.empty((2 * I, d), np.float64) if "dW13" in want else None
    g2 = np.empty((d, I), np.float64) if "dW2" in want else None
    _load().orc_expert_wgrad(_ptr(xn), _ptr(w13), _ptr(w2), _ptr(dy), bf, int(e), rt.shape[0],
                             _ptr(rt), _ptr(rw), d, I, float(clamp), int(exact),
                             int(store_bf16), _ptr(g13), _ptr(g2))
    if g13 is not None:
        out["dW13"] = g13
    if g2 is not None:
        out["dW2"] = g2
    return out


def expert_wgrad_entries(x, W13, W2, dY, e, row_tok, row_w, clamp, kind, qa, qb, exact=False,
                         store_bf16=False):
    """Sampled weight-gradient entries of expert e (kind 0: dW2[qa,qb]; 1: dW13[qa,qb])."""
    (xn, w13, w2, dy), bf = _floats(x, W13, W2, dY)
    d = xn.shape[1]
    I = w2.shape[-1]
    rt = np.ascontiguousarray(_to_np(row_tok), dtype=np.int64)
    rw = np.ascontiguousarray(_to_np(row_w), dtype=np.float64)
    kd = np.ascontiguousarray(kind, dtype=np.int32)
    a = np.ascontiguousarray(qa, dtype=np.int32)
    b = np.ascontiguousarray(qb, dtype=np.int32)
    out = np.empty((kd.shape[0],), np.float64)
    _load().orc_expert_wgrad_entries(_ptr(xn), _ptr(w13), _ptr(w2), _ptr(dy), bf, int(e),
                                     rt.shape[0], _ptr(rt), _ptr(rw), d, I, float(clamp),
                                     int(exact), int(store_bf16), kd.shape[0], _ptr(kd),
                                     _ptr(a), _ptr(b), _ptr(out))
    return out


# ------------------------------------------------------------------ MXFP8
# OCP Microscaling (MX) v1.0 with E4M3 elements: blocks of 32 along the
# contraction, one E8M0 scale per block (see moe_oracle.c for the reading).

def e4m3_decode_all():
    """Value of every E4M3 code 0..255 (NaN for 0x7F and 0xFF)."""
    out = np.empty(256, np.float64)
    _load().orc_e4m3_decode_all(_ptr(out))
    return out


def e4m3_encode(y):
    """Nearest E4M3 code of each value (ties to even, saturating at 448)."""
    yv = np.ascontiguousarray(np.asarray(y, dtype=np.float64).reshape(-1))
    out = np.empty(yv.shape[0], np.uint8)
    _load().orc_e4m3_encode(_ptr(yv), int(yv.shape[0]), _ptr(out))
    return out.reshape(np.shape(y))


def mx_quantize(src, sf_pitch=None):
    """MX quantisation of a [rows, K] matrix (torch bf16 or float64, K % 32 ==
    0) along K.  Returns (q uint8 [rows, K], sf uint8 [rows, sf_pitch]);
    sf_pitch defaults to K // 32 (padding bytes are zero)."""
    (a,), bf = _floats(src)
    rows, K = a.shape
    assert K % 32 == 0
    pitch = K // 32 if sf_pitch is None else int(sf_pitch)
    q = np.empty((rows, K), np.uint8)
    sf = np.zeros((rows, pitch), np.uint8)
    _load().orc_mx_quantize(_ptr(a), bf, rows, K, pitch, _ptr(q), _ptr(sf))
    return q, sf


def mx_dequantize(q, sf, K=None):
    """Values (float64 [rows, K]) of a quantised matrix."""
    qn = np.ascontiguousarray(_to_np(q), dtype=np.uint8)
    sn = np.ascontiguousarray(_to_np(sf), dtype=np.uint8)
    rows, K = qn.shape
    out = np.empty((rows, K), np.float64)
    _load().orc_mx_dequantize(_ptr(qn), _ptr(sn), rows, K, int(sn.shape[1]), _ptr(out))
    return out


def expert_rows_mx(x, W13, W2, row_tok, row_exp, row_w, clamp):
    """MXFP8 expert FFN per row (x, W13, W2 bf16): returns (h, y) with h the
    dequantised MX h [n, I] and y = row_w * W2~[e] h [n, d]."""
    (xn, w13, w2), bf = _floats(x, W13, W2)
    assert bf == 1, "the MX oracle takes bf16 inputs"
    d = xn.shape[1]
    I = w2.shape[-1]
    rt = np.ascontiguousarray(_to_np(row_tok), dtype=np.int64)
    re = np.ascontiguousarray(_to_np(row_exp), dtype=np.int32)
    rw = _opt(row_w, np.float64)
    n = rt.shape[0]
    h = np.empty((n, I), np.float64)
    y = np.empty((n, d), np.float64)
    _load().orc_expert_rows_mx(_ptr(xn), _ptr(w13), _ptr(w2), n, _ptr(rt), _ptr(re), _ptr(rw),
                               d, I, float(clamp), _ptr(h), _ptr(y))
    return h, y


def expert_rows_mx_backward(x, W13, W2, dY, row_tok, row_exp, row_w, clamp):
    """Backward of the MXFP8 expert FFN per row (training form: each matmul's
    operands MX along its own contraction).  Returns dict(dw [n], dgu [n, 2I]
    (before quantisation), h [n, I] (the forward's MX h), dx [n, d])."""
    (xn, w13, w2, dy), bf = _floats(x, W13, W2, dY)
    assert bf == 1, "the MX oracle takes bf16 inputs"
    d = xn.shape[1]
    I = w2.shape[-1]
    rt = np.ascontiguousarray(_to_np(row_tok), dtype=np.int64)
    re = np.ascontiguousarray(_to_np(row_exp), dtype=np.int32)
    rw = _opt(row_w, np.float64)
    n = rt.shape[0]
    dw = np.empty((n,), np.float64)
    dgu = np.empty((n, 2 * I), np.float64)
    h = np.empty((n, I), np.float64)
    dx = np.empty((n, d), np.float64)
    _load().orc_expert_rows_mx_backward(_ptr(xn), _ptr(w13), _ptr(w2), _ptr(dy), n, _ptr(rt),
                                        _ptr(re), _ptr(rw), d, I, float(clamp), _ptr(dw),
                                        _ptr(dgu), _ptr(h), _ptr(dx))
    return dict(dw=dw, dgu=dgu, h=h, dx=dx)


def layer_backward_mx(x, W_g, W13, W2, dY, bias, k, rho, clamp, is_vision=None, mode=0,
                      input_ids=None, tid2eid=None, offset=None, tok=None):
    """Token-local backward of the layer with the MXFP8 expert matmuls for the
    listed tokens (bf16 inputs): dict(dX [n,d], dz [n,E], dw [n,k])."""
    (xn, wg, w13, w2, dy), bf = _floats(x, W_g, W13, W2, dY)
    assert bf == 1, "the MX oracle takes bf16 inputs"
    E, d = wg.shape
    I = w2.shape[-1]
    b, vis, ii, tab, vocab, off = _route_args(bias, E, is_vision, input_ids, tid2eid, offset)
    tk, n = _tok(tok, xn.shape[0])
    dX = np.empty((n, d), np.float64)
    dz = np.empty((n, E), np.float64)
    dw = np.empty((n, k), np.float64)
    _load().orc_layer_backward_mx(_ptr(xn), _ptr(wg), _ptr(w13), _ptr(w2), _ptr(dy), _ptr(off),
                                  _ptr(b), _ptr(vis), int(mode), _ptr(ii), _ptr(tab), vocab, n,
                                  _ptr(tk), d, E, k, I, float(rho), float(clamp), _ptr(dX),
                                  _ptr(dz), _ptr(dw))
    return dict(dX=dX, dz=dz, dw=dw)


def mx_rows_matmul(A, B):
    """A^T B (A [K, M], B [K, N], float64) with both operands MX-quantised
    along their rows in blocks of 32 from row 0 (the last block zero-padded):
    float64 [M, N]."""
    a = np.ascontiguousarray(np.asarray(A, dtype=np.float64))
    b = np.ascontiguousarray(np.asarray(B, dtype=np.float64))
    K, M = a.shape
    assert b.shape[0] == K
    N = b.shape[1]
    out = np.empty((M, N), np.float64)
    _load().orc_mx_rows_matmul(_ptr(a), _ptr(b), K, M, N, _ptr(out))
    return out


def expert_wgrad_mx(x, W13e, W2e, dY, row_tok, row_w, clamp):
    """Weight gradients of one expert in the MX training form over its rows in
    the given order (bf16 inputs; W13e [2I, d], W2e [d, I] that expert's
    weights): dict(dW13 [2I, d], dW2 [d, I])."""
    (xn, w13, w2, dy), bf = _floats(x, W13e, W2e, dY)
    assert bf == 1, "the MX oracle takes bf16 inputs"
    d = xn.shape[1]
    I = w2.shape[-1]
    rt = np.ascontiguousarray(_to_np(row_tok), dtype=np.int64)
    rw = _opt(row_w, np.float64)
    n = rt.shape[0]
    dW13 = np.empty((2 * I, d), np.float64)
    dW2 = np.empty((d, I), np.float64)
    _load().orc_expert_wgrad_mx(_ptr(xn), _ptr(w13), _ptr(w2), _ptr(dy), n, _ptr(rt), _ptr(rw),
                                d, I, float(clamp), _ptr(dW13), _ptr(dW2))
    return dict(dW13=dW13, dW2=dW2)

