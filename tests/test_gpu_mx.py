"""The MXFP8 path (moe_mx_quantize, moe_mx_gather, moe_expert_ffn_mx) against
the oracle.

Codes and scale codes are integer results of a fixed rounding rule, so the
quantiser and the quantising dispatch gather must match the oracle bit for
bit, including zero blocks, ties between E4M3 neighbours, saturation, signed
zeros, and blocks whose scale clamps at 2^-127.  The MX expert FFN is a float
result: y_perm and the dequantised MX h are compared with the oracle's fp64
MX FFN (its h is quantised from fp64 SwiGLU values, the GPU's from fp32 ones,
so a code may sit one step apart where the two straddle a rounding boundary;
such codes must stay rare).  Sizes give ragged row tiles, experts without
rows, two scale chunks per contraction (d = 1024), a partial chunk (I = 256),
more row tiles than SMs, and the full-width layer on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_04_gb300 import _lib
from moe_expert_layer_04_gb300 import workloads as W
from moe_expert_layer_04_gb300.layer import Dims, MoELayer
from tests.helpers import MAX_ABS, assert_close, cpu, np64

pytestmark = pytest.mark.gpu

PAD = 0xAA   # fill of the scale rows' padding bytes, which no call may write


def _special_blocks(x):
    """Overwrites the first blocks of x (float64 [rows, K], K >= 256) with the
    edge cases of the rounding rule."""
    tab = oracle.e4m3_decode_all()
    grid = tab[:0x7F]
    X = 2.0 ** -5
    x[0, 0:32] = 0.0
    x[0, 0:32:2] = -0.0                                    # a block of signed zeros
    ties = (grid[:-1] + grid[1:]) / 2                      # every tie between neighbours
    x[0, 32] = 256 * X                                     # block max fixes X
    x[0, 33:64] = ties[np.linspace(0, len(ties) - 1, 31).astype(int)] * X
    x[0, 64] = 256 * X
    x[0, 65:96] = -ties[np.linspace(0, len(ties) - 1, 31).astype(int)] * X
    x[0, 96] = 1.9 * 2.0 ** 3                              # scaled 486.4: saturates to 448
    x[0, 97:128] = np.linspace(-15, 15, 31)
    x[0, 128:160] = 2.0 ** -131                            # scale clamps at 2^-127
    x[0, 160] = 256 * X
    x[0, 161:192] = -(2.0 ** -12) * X                      # negative values rounding to -0
    x[0, 192] = 2.0 ** 120                                 # large scale
    x[0, 193:224] = np.linspace(-(2.0 ** 118), 2.0 ** 118, 31)
    return x


def _quantize_gpu(xb):
    rows, K = xb.shape
    q = torch.empty(rows, K, dtype=torch.uint8, device="cuda")
    sf = torch.full((rows, _lib.moe_mx_sf_pitch(K)), PAD, dtype=torch.uint8, device="cuda")
    _lib.moe_mx_quantize(xb, rows, K, q, sf)
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    return cpu(q).numpy(), cpu(sf).numpy()


@pytest.mark.parametrize("rows,K", [(1, 32), (300, 96), (7, 256), (257, 4096)])
def test_mx_quantize_bit_exact(rows, K):
    g = torch.Generator().manual_seed(rows * 7919 + K)
    x = torch.randn(rows, K, generator=g, dtype=torch.float64)
    x *= torch.exp(torch.randn(rows, 1, generator=g, dtype=torch.float64) * 3)
    x = x.numpy()
    if K >= 256:
        x = _special_blocks(x)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    q, sf = _quantize_gpu(xb.cuda())
    q_ref, sf_ref = oracle.mx_quantize(xb)
    assert np.array_equal(sf[:, : K // 32], sf_ref)
    assert np.array_equal(q, q_ref)
    assert np.all(sf[:, K // 32:] == PAD)


def _mx_layer(name, T, d, E, k, I, n_empty=0, big=False):
    w = W.Workload(name, T, d, E, k, I, 2.5, vision_frac=0.3)
    inp = W.make_inputs(w, device="cuda")
    if n_empty:
        inp["bias"][:, :n_empty] = -10.0   # these experts get no slot
    if big:
        # block scales above 2^7 (the expansion's second multiply): x and one
        # expert's W13 rows times 2^16; the clamp keeps h, and so y, bounded
        inp["x"] *= 2.0 ** 16
        inp["W13"][1] *= 2.0 ** 16
    weights = dict(W_g=inp["W_g"], W13=inp["W13"], W2=inp["W2"])
    layer = MoELayer(Dims(T, d, E, k, I), weights, w.rho, w.clamp, mx=True)
    layer.h_sf.fill_(PAD)
    layer.x_perm_sf.fill_(PAD)
    layer.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"])
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    return w, inp, layer


def _row_groups(layer, rows):
    offs = cpu(layer.offsets).numpy()
    return (np.searchsorted(offs, rows, side="right") - 1).astype(np.int32)


def _check_rows(w, inp, layer, rows, scale_abs=False):
    """y_perm and the MX h of the given rows against the oracle's MX FFN.
    scale_abs: the max-abs bound is relative to the largest |value| (outputs
    far from unit magnitude, where one h code step moves y by more than the
    absolute bound)."""
    rt = cpu(layer.row_token).numpy()[rows].astype(np.int64)
    grp = _row_groups(layer, rows)
    rw = np.ones(len(rows))
    routed = rows < w.S
    rw[routed] = np64(layer.row_weight)[rows[routed]]
    # only the weights of the groups these rows belong to go to the host
    uniq, inv = np.unique(grp, return_inverse=True)
    sel = torch.from_numpy(uniq.astype(np.int64)).cuda()
    h_ref, y_ref = oracle.expert_rows_mx(cpu(inp["x"]), cpu(inp["W13"][sel]), cpu(inp["W2"][sel]),
                                         rt, inv.astype(np.int32), rw, w.clamp)
    ridx = torch.from_numpy(rows).cuda()
    ay = MAX_ABS * max(1.0, float(np.abs(y_ref).max())) if scale_abs else MAX_ABS
    assert_close(layer.y_perm[ridx], y_ref, f"{w.name} MX y_perm rows", max_abs=ay)
    hq = cpu(layer.h_q[ridx]).numpy()
    hsf = cpu(layer.h_sf[ridx]).numpy()
    assert np.all(hsf[:, w.I // 32:] == PAD)
    h_gpu = oracle.mx_dequantize(hq, hsf[:, : w.I // 32])
    ah = MAX_ABS * max(1.0, float(np.abs(h_ref).max())) if scale_abs else MAX_ABS
    assert_close(h_gpu, h_ref, f"{w.name} MX h rows", max_abs=ah)
    # codes: the oracle's MX h re-encoded from its values
    q_ref, sf_ref = oracle.mx_quantize(h_ref)
    assert np.array_equal(oracle.mx_dequantize(q_ref, sf_ref), h_ref)
    mism = np.mean(hq != q_ref)
    assert mism <= 2e-3, f"{w.name}: {mism:.2e} of the h codes differ"
    return rt


# name, T, d, E, k, I, experts forced empty, rows checked (None: all), large scales
CASES = [
    ("ragged", 300, 256, 6, 2, 128, 0, None, False),
    ("two_scale_chunks", 700, 1024, 5, 2, 256, 0, None, False),
    ("empty_experts", 500, 512, 16, 4, 128, 5, None, False),
    ("many_row_tiles", 12000, 256, 4, 2, 128, 0, 384, False),
    # many rows per expert: the 256-wide tiles, several column tiles each way
    ("wide_tiles", 6000, 512, 4, 2, 256, 0, 384, False),
    ("scales_above_2e7", 400, 256, 4, 2, 128, 0, None, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_mx_ffn_parity(case):
    name, T, d, E, k, I, n_empty, n_rows, big = case
    w, inp, layer = _mx_layer(name, T, d, E, k, I, n_empty, big)
    if big:
        sf = cpu(layer.x_perm_sf).numpy()[:, : d // 32]
        assert (sf.astype(int) - 127 > 7).all()            # every x block takes the second multiply
    if n_empty:
        assert int(cpu(layer.counts)[:n_empty].sum()) == 0
    R = w.S + w.T
    # the dispatch gather: every row holds its token's MX row, bit for bit
    q_ref, sf_ref = oracle.mx_quantize(cpu(inp["x"]))
    row_token = cpu(layer.row_token).numpy()
    assert np.array_equal(cpu(layer.x_perm_q).numpy(), q_ref[row_token])
    xsf = cpu(layer.x_perm_sf).numpy()
    assert np.array_equal(xsf[:, : d // 32], sf_ref[row_token])
    assert np.all(xsf[:, d // 32:] == PAD)
    # the weights, quantised once by the layer
    q13, sf13 = oracle.mx_quantize(cpu(inp["W13"]).reshape(-1, d))
    assert np.array_equal(cpu(layer.W13_q).numpy(), q13)
    assert np.array_equal(cpu(layer.W13_sf).numpy()[:, : d // 32], sf13)
    rows = (np.arange(R) if n_rows is None else
            np.sort(np.random.default_rng(11).choice(R, size=n_rows, replace=False)))
    # with x and W13 times 2^16, g is a sum of ~1e3-sized terms whose fp32
    # rounding (~1e-2) can move an unclamped h across an E4M3 boundary; one h
    # code step then moves y by ~0.2 on outputs of magnitude ~10
    _check_rows(w, inp, layer, rows.astype(np.int64), scale_abs=big)
    # the combine of the MX rows: y of sampled tokens
    toks = np.sort(np.random.default_rng(12).choice(T, size=min(T, 48), replace=False))
    slot_row = cpu(layer.slot_row).numpy().reshape(T, k)
    yp = np64(layer.y_perm)
    y_ref = yp[w.S + toks] + yp[slot_row[toks]].sum(axis=1)
    ay = MAX_ABS * max(1.0, float(np.abs(y_ref).max())) if big else MAX_ABS
    assert_close(layer.y[torch.from_numpy(toks).cuda()], y_ref, f"{name} MX y", max_abs=ay)


@pytest.mark.slow
def test_mx_full_width_sampled_rows():
    """The full-width layer (T = 4096, 384 experts top-6 + shared, d = 4096,
    I = 2048) in MXFP8, on rows of the hottest, median and coldest routed
    experts and of the shared expert."""
    w = W.WORKLOADS["full_fwd"]
    inp = W.make_inputs(w, device="cuda")
    weights = dict(W_g=inp["W_g"], W13=inp["W13"], W2=inp["W2"])
    layer = MoELayer(Dims(w.T, w.d, w.E, w.k, w.I), weights, w.rho, w.clamp, mx=True)
    layer.h_sf.fill_(PAD)
    layer.forward(inp["x"], inp["bias"], inp["is_vision"], inp["logit_offset"])
    torch.cuda.synchronize()
    assert _lib.moe_last_device_status() == _lib.MOE_OK
    counts = cpu(layer.counts).numpy()
    offs = cpu(layer.offsets).numpy()
    order = np.argsort(counts, kind="stable")
    nonempty = order[counts[order] > 0]
    picks = [nonempty[-1], nonempty[len(nonempty) // 2], nonempty[0], w.E]
    rows = []
    for e in picks:
        lo, hi = offs[e], offs[e + 1]
        rows += [lo, hi - 1] if hi - lo > 1 else [lo]
    rows = np.array(sorted(set(rows)), np.int64)
    _check_rows(w, inp, layer, rows)
    # one routed expert's quantised weights, bit for bit
    e = int(picks[0])
    span = slice(e * 2 * w.I, (e + 1) * 2 * w.I)
    q13, sf13 = oracle.mx_quantize(cpu(inp["W13"][e]))
    assert np.array_equal(cpu(layer.W13_q[span]).numpy(), q13)
    assert np.array_equal(cpu(layer.W13_sf[span]).numpy()[:, : w.d // 32], sf13)
