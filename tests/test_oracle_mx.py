"""Pins of the MXFP8 part of the oracle (OCP MX v1.0 with E4M3 elements).

The pages name MxFP8 as the next low-precision step and define no format, so
the pins come from the format's published definition (values in
tests/golden/ocp_mx_e4m3.txt), from a library routine (PyTorch's float8_e4m3fn
cast, round-to-nearest-even), from closed forms of the scale selection, from
the quantisation error bound, and from the reduction of the MX expert FFN to
the plain expert FFN oracle (itself pinned in test_oracle_pins.py) on
dequantised inputs."""
import math
import os

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ocp_mx_e4m3.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            kind, code, val = line.split()
            rows.append((kind, int(code, 16), float(val)))
    return rows


def _same(a, b):
    return (math.isnan(a) and math.isnan(b)) or (a == b and math.copysign(1, a) == math.copysign(1, b))


def test_e4m3_values_from_spec():
    tab = oracle.e4m3_decode_all()
    for kind, code, val in _golden():
        if kind == "e4m3":
            assert _same(tab[code], val), (hex(code), tab[code], val)


def test_e4m3_table_matches_torch():
    tab = oracle.e4m3_decode_all()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        assert _same(tab[c], ref[c]), hex(c)
    # strictly increasing over the finite non-negative codes
    assert np.all(np.diff(tab[:0x7F]) > 0)


def _torch_codes(y):
    return torch.tensor(y, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_in_range():
    tab = oracle.e4m3_decode_all()
    grid = tab[:0x7F]                        # 0 .. 448
    mids = (grid[:-1] + grid[1:]) / 2        # every tie between neighbours
    rng = np.random.default_rng(0)
    rand = rng.uniform(-448, 448, 20000)
    small = rng.uniform(-0.03, 0.03, 20000)  # subnormal and smallest normals
    y = np.concatenate([grid, -grid, mids, -mids, rand, small]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(y.astype(np.float64)), _torch_codes(y))


def test_e4m3_encode_saturates():
    codes = oracle.e4m3_encode(np.array([448.0, 449.0, 464.0, 480.0, 511.0, 1e6, -470.0, -1e30]))
    assert list(codes) == [0x7E] * 6 + [0xFE, 0xFE]


def test_e4m3_encode_signed_zero():
    codes = oracle.e4m3_encode(np.array([0.0, -0.0, 1e-9, -1e-9, 2.0 ** -10, -(2.0 ** -10)]))
    # 2^-10 is the tie between 0 and the smallest subnormal: ties to even -> 0
    assert list(codes) == [0x00, 0x80, 0x00, 0x80, 0x00, 0x80]


def _block(vals):
    v = np.zeros((1, 32))
    v[0, :len(vals)] = vals
    return v


def test_mx_scale_closed_forms():
    for p in range(-30, 31):
        q, sf = oracle.mx_quantize(_block([2.0 ** p, 0.5 * 2.0 ** p, -(2.0 ** p)]))
        assert sf[0, 0] == p - 8 + 127
        assert list(q[0, :3]) == [0x78, 0x70, 0xF8]       # 256, 128, -256 after scaling
        q, sf = oracle.mx_quantize(_block([1.75 * 2.0 ** p]))
        assert sf[0, 0] == p - 8 + 127 and q[0, 0] == 0x7E
        q, sf = oracle.mx_quantize(_block([1.9 * 2.0 ** p]))   # 486.4 -> saturates to 448
        assert sf[0, 0] == p - 8 + 127 and q[0, 0] == 0x7E
    q, sf = oracle.mx_quantize(np.zeros((2, 64)))
    assert not q.any() and not sf.any()
    q, sf = oracle.mx_quantize(_block([2.0 ** -130]))        # scale exponent clamps at -127
    assert sf[0, 0] == 0 and q[0, 0] == 0x20                 # 2^-130 / 2^-127 = 2^-3
    q, sf = oracle.mx_quantize(_block([2.0 ** 140]))         # clamps at +127, element saturates
    assert sf[0, 0] == 254 and q[0, 0] == 0x7E


def test_mx_roundtrip_on_grid():
    rng = np.random.default_rng(1)
    tab = oracle.e4m3_decode_all()
    rows, K = 16, 256
    codes = rng.integers(0, 0x7F, size=(rows, K)) | (rng.integers(0, 2, size=(rows, K)) << 7)
    codes = codes.astype(np.uint8)
    codes[:, ::32] = rng.integers(0x78, 0x7F, size=(rows, K // 32))  # block max in the top binade
    se = rng.integers(-40, 40, size=(rows, K // 32))
    v = tab[codes] * np.repeat(2.0 ** se, 32, axis=1)
    q, sf = oracle.mx_quantize(v)
    assert np.array_equal(sf.astype(np.int64) - 127, se)
    assert np.array_equal(q, codes)
    assert np.array_equal(oracle.mx_dequantize(q, sf), v)


def test_mx_error_bound_and_bf16_path():
    g = torch.Generator().manual_seed(2)
    x = torch.randn(64, 512, generator=g, dtype=torch.float64)
    x[:, 64:96] *= 1e-3                         # blocks of very different magnitude
    x[3, 100] = 40.0                            # an outlier inside a block
    xb = x.to(torch.bfloat16)
    q, sf = oracle.mx_quantize(xb)
    q2, sf2 = oracle.mx_quantize(xb.double().numpy())
    assert np.array_equal(q, q2) and np.array_equal(sf, sf2)
    v = xb.double().numpy()
    dq = oracle.mx_dequantize(q, sf)
    X = np.repeat(2.0 ** (sf.astype(np.float64) - 127), 32, axis=1)
    # half a quantum (2^-4 relative in the normal range, 2^-10 X below it), or
    # the saturation of a scaled magnitude in (448, 512) to 448
    bound = np.maximum(np.maximum(np.abs(v) * 2.0 ** -4, X * 2.0 ** -10), np.abs(v) - 448 * X)
    assert np.all(np.abs(dq - v) <= bound)
    # the block maximum lands in E4M3's top binade [256, 448]
    bmax = np.abs(v).reshape(64, 16, 32).max(axis=2)
    r = bmax / 2.0 ** (sf.astype(np.float64) - 127)
    assert np.all((r >= 256) & (r < 512))


def _bf16(a):
    t = torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)
    assert np.array_equal(t.double().numpy(), a)   # MX values are exact in bf16
    return t


def test_expert_rows_mx_reduces_to_plain_oracle():
    d, I, G = 128, 64, 3
    g = torch.Generator().manual_seed(3)
    x = torch.randn(6, d, generator=g).to(torch.bfloat16)
    W13 = (torch.randn(G, 2 * I, d, generator=g) * 0.05).to(torch.bfloat16)
    W2 = (torch.randn(G, d, I, generator=g) * 0.05).to(torch.bfloat16)
    tok = np.array([0, 1, 2, 3, 4, 5, 1, 0])
    exp_ = np.array([0, 2, 1, 1, 0, 2, 0, 1], np.int32)
    rw = np.linspace(0.2, 1.4, 8)
    clamp = 0.8                              # some g and u clamp
    h_mx, y_mx = oracle.expert_rows_mx(x, W13, W2, tok, exp_, rw, clamp)
    # the same FFN on the dequantised operands, exactly, through the plain oracle
    xd = _bf16(oracle.mx_dequantize(*oracle.mx_quantize(x)))
    w13d = _bf16(oracle.mx_dequantize(*oracle.mx_quantize(W13.reshape(-1, d))).reshape(G, 2 * I, d))
    w2d = _bf16(oracle.mx_dequantize(*oracle.mx_quantize(W2.reshape(-1, I))).reshape(G, d, I))
    h_ex, _ = oracle.expert_rows(xd, w13d, w2d, tok, exp_, rw, clamp, exact=True)
    assert np.array_equal(h_mx, oracle.mx_dequantize(*oracle.mx_quantize(h_ex)))
    y_lib = np.stack([rw[r] * (w2d[exp_[r]].double().numpy() @ h_mx[r]) for r in range(8)])
    assert np.allclose(y_mx, y_lib, rtol=1e-12, atol=1e-15)
    # MXFP8 is a few percent away from the bf16 FFN, never identical to it
    _, y_bf = oracle.expert_rows(x, W13, W2, tok, exp_, rw, clamp, exact=True)
    rel = np.linalg.norm(y_mx - y_bf) / np.linalg.norm(y_bf)
    assert 1e-3 < rel < 0.1, rel


# ------------------------------------------------------- the MX backward


def _deq(q, sf):
    return oracle.mx_dequantize(q, sf)


def _mx(a):
    """Values of a [rows, K] matrix after MX quantisation along K (the
    quantiser itself is pinned above)."""
    q, sf = oracle.mx_quantize(np.ascontiguousarray(a, dtype=np.float64))
    return _deq(q, sf)


def _bwd_case(grid, seed=5):
    rng = np.random.default_rng(seed)
    n, d, I, E = 10, 64, 64, 3
    if grid:
        # powers of two in [1/2, 2] (and zeros): every block of 32 along any
        # axis is exactly on the MX grid, so every quantisation of an input
        # operand is the identity
        def pick(shape):
            v = rng.choice([0.0, 0.5, 1.0, 2.0, -0.5, -1.0, -2.0], size=shape)
            return torch.from_numpy(v).to(torch.bfloat16)
        x, dY = pick((n, d)), pick((n, d))
        W13 = torch.from_numpy(rng.choice([0.0, 0.5, -0.5, 1.0 / 64, -1.0 / 64],
                                          size=(E, 2 * I, d))).to(torch.bfloat16)
        W2 = torch.from_numpy(rng.choice([0.0, 0.5, -0.5, 1.0 / 64, -1.0 / 64],
                                         size=(E, d, I))).to(torch.bfloat16)
    else:
        x = torch.randn(n, d, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
        dY = torch.randn(n, d, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16)
        W13 = (torch.randn(E, 2 * I, d, generator=torch.Generator().manual_seed(seed + 2)) *
               0.1).to(torch.bfloat16)
        W2 = (torch.randn(E, d, I, generator=torch.Generator().manual_seed(seed + 3)) *
              0.1).to(torch.bfloat16)
    rt = np.arange(n, dtype=np.int64)
    re = (np.arange(n) % E).astype(np.int32)
    rw = np.linspace(0.3, 1.7, n)
    return x, dY, W13, W2, rt, re, rw


@pytest.mark.parametrize("clamp", [7.0, 1.5])
def test_mx_backward_on_grid_inputs_is_the_autograd_chain(clamp):
    # inputs on the MX grid along every axis: the only quantisations left are
    # those of h (the forward's GEMM-2 input) and of [dg | du] (dgrad 1's
    # input); everything else must be the exact chain rule, which torch's
    # autograd differentiates independently of the oracle's formulas
    x, dY, W13, W2, rt, re, rw = _bwd_case(grid=True)
    out = oracle.expert_rows_mx_backward(x, W13, W2, dY, rt, re, rw, clamp)
    xd, dyd = x.double(), dY.double()
    I = W2.shape[-1]
    for r in range(len(rt)):
        e = int(re[r])
        w13, w2 = W13[e].double(), W2[e].double()
        gu = (w13 @ xd[r]).clone().requires_grad_(True)
        g, u = gu[:I], gu[I:]
        h = torch.nn.functional.silu(torch.clamp(g, max=clamp)) * torch.clamp(u, -clamp, clamp)
        hq = torch.from_numpy(_mx(h.detach().numpy()[None])[0])
        np.testing.assert_array_equal(out["h"][r], hq.numpy())
        dA = w2.T @ dyd[r]
        np.testing.assert_allclose(out["dw"][r], float(hq @ dA), rtol=1e-12, atol=1e-12)
        (h * (rw[r] * dA)).sum().backward()
        np.testing.assert_allclose(out["dgu"][r], gu.grad.numpy(), rtol=1e-12, atol=1e-12)
        dgq = torch.from_numpy(_mx(gu.grad.numpy()[None])[0])
        np.testing.assert_allclose(out["dx"][r], (w13.T @ dgq).numpy(), rtol=1e-12, atol=1e-12)


def test_mx_backward_quantises_each_matmul_along_its_contraction():
    # general inputs: dA uses W2 quantised along d (its columns) and dY along
    # d; dX uses W13 quantised along 2I (its columns) and [dg | du] along 2I
    x, dY, W13, W2, rt, re, rw = _bwd_case(grid=False)
    out = oracle.expert_rows_mx_backward(x, W13, W2, dY, rt, re, rw, 7.0)
    dyq = _mx(dY.double().numpy())
    for r in range(len(rt)):
        e = int(re[r])
        w2t = _mx(W2[e].double().numpy().T)          # [I, d]: along d
        w13t = _mx(W13[e].double().numpy().T)        # [d, 2I]: along 2I
        dA = w2t @ dyq[r]
        np.testing.assert_allclose(out["dw"][r], out["h"][r] @ dA, rtol=1e-12, atol=1e-12)
        dgq = _mx(out["dgu"][r][None])[0]
        np.testing.assert_allclose(out["dx"][r], w13t @ dgq, rtol=1e-12, atol=1e-12)
        # quantising W2 along I instead (a plausible mistake) changes dw
        wrong = _mx(W2[e].double().numpy()).T @ dyq[r]
        assert abs(out["h"][r] @ wrong - out["dw"][r]) > 1e-9 * max(1.0, abs(out["dw"][r]))
    # and the MX h is the forward's (orc_expert_rows_mx)
    h_fwd, _ = oracle.expert_rows_mx(x, W13, W2, rt, re, rw, 7.0)
    np.testing.assert_array_equal(out["h"], h_fwd)


def test_mx_backward_stays_near_the_exact_backward():
    # the MX chain approximates the exact gradients: against the plain
    # per-row forward's h and the exact dA (fp64 on the bf16 operands), the
    # MX dw and [dg | du] differ by no more than the E4M3 rounding allows
    x, dY, W13, W2, rt, re, rw = _bwd_case(grid=False, seed=9)
    out = oracle.expert_rows_mx_backward(x, W13, W2, dY, rt, re, rw, 7.0)
    h_plain, _ = oracle.expert_rows(x, W13, W2, rt, re, rw, 7.0, exact=True)
    dA = oracle.rows_dA(dY, W2, rt, re)
    dw_exact = (h_plain * dA).sum(1)
    # each product carries at most a few E4M3 steps (2^-3 relative at most per
    # factor), so the error is bounded by a fraction of the sum of |products|
    mag = np.abs(h_plain * dA).sum(1)
    assert np.all(np.abs(out["dw"] - dw_exact) <= 0.15 * mag), \
        np.max(np.abs(out["dw"] - dw_exact) / mag)
    # over the rows the MX dw follows the exact one; a sign slip would not
    nrm = np.linalg.norm(dw_exact)
    assert np.linalg.norm(out["dw"] - dw_exact) < 0.2 * nrm
    assert np.linalg.norm(-out["dw"] - dw_exact) > 1.5 * nrm


# ----------------------------------------------- the MX layer backward


def _layer_case(seed=21):
    g = torch.Generator().manual_seed(seed)
    T, d, E, k, I = 12, 64, 5, 2, 64
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    dY = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W_g = (torch.randn(E, d, generator=g) * 0.2).to(torch.bfloat16)
    W13 = (torch.randn(E + 1, 2 * I, d, generator=g) * 0.1).to(torch.bfloat16)
    W2 = (torch.randn(E + 1, d, I, generator=g) * 0.1).to(torch.bfloat16)
    bias = torch.zeros(E)
    is_vision = (torch.arange(T) % 3 == 0).to(torch.uint8)
    return T, d, E, k, I, x, dY, W_g, W13, W2, bias, is_vision


def test_mx_layer_backward_assembles_the_token_rows():
    # dw is the routed rows' <h~, dA>, and dX is the sum of the token's k + 1
    # MX rows (shared expert included) plus the gate term dz W_g
    T, d, E, k, I, x, dY, W_g, W13, W2, bias, vis = _layer_case()
    rho, clamp = 2.5, 7.0
    out = oracle.layer_backward_mx(x, W_g, W13, W2, dY, bias, k, rho, clamp, is_vision=vis)
    fwd = oracle.layer_forward(x, W_g, W13, W2, bias, k, rho, clamp, is_vision=vis)
    rt = np.repeat(np.arange(T), k + 1).astype(np.int64)
    re = np.concatenate([np.full((T, 1), E, np.int32), fwd["ids"]], axis=1).reshape(-1)
    rw = np.concatenate([np.ones((T, 1)), fwd["w"]], axis=1).reshape(-1)
    rows = oracle.expert_rows_mx_backward(x, W13, W2, dY, rt, re.astype(np.int32), rw, clamp)
    np.testing.assert_allclose(out["dw"], rows["dw"].reshape(T, k + 1)[:, 1:], rtol=1e-12,
                               atol=1e-14)
    dx_rows = rows["dx"].reshape(T, k + 1, d).sum(1)
    gate = out["dz"] @ W_g.double().numpy()
    np.testing.assert_allclose(out["dX"], dx_rows + gate, rtol=1e-10, atol=1e-12)
    # dz lives on the selection only, and the gate term is not negligible
    sel = np.zeros((T, E), bool)
    np.put_along_axis(sel, fwd["ids"].astype(np.int64), True, axis=1)
    assert np.all(out["dz"][~sel] == 0.0) and np.abs(out["dz"][sel]).min() > 0.0
    assert np.linalg.norm(gate) > 1e-3 * np.linalg.norm(out["dX"])


def test_mx_layer_backward_logit_gradient_by_finite_differences():
    # dz is the derivative of sum_j dw_j w_j(z) at the fp32 logits the layer
    # routes with, with dw held fixed: central differences of the oracle's
    # own forward routing (exact weights, fixed selection)
    T, d, E, k, I, x, dY, W_g, W13, W2, bias, vis = _layer_case(seed=22)
    rho = 2.5
    out = oracle.layer_backward_mx(x, W_g, W13, W2, dY, bias, k, rho, 7.0, is_vision=vis)
    z = oracle.gate_logits(x, W_g)
    ids0, _, _, margin = oracle.route(z, bias, k, rho, is_vision=vis, exact=True)
    assert margin.min() > 1e-3
    eps = 1e-6
    for m in range(E):
        zp, zm = z.copy(), z.copy()
        zp[:, m] += eps
        zm[:, m] -= eps
        idp, wp, _, _ = oracle.route(zp, bias, k, rho, is_vision=vis, exact=True)
        idm, wm, _, _ = oracle.route(zm, bias, k, rho, is_vision=vis, exact=True)
        assert np.array_equal(idp, ids0) and np.array_equal(idm, ids0)
        fd = ((wp - wm) / (2 * eps) * out["dw"]).sum(1)
        np.testing.assert_allclose(out["dz"][:, m], fd, rtol=1e-5, atol=1e-8)


# ----------------------------------------- MX weight gradients (rows)


def _grid(rng, shape):
    # powers of two in [1/2, 2] and zeros: every block of 32, along any axis,
    # is on the MX grid, so its quantisation is the identity
    return rng.choice([0.0, 0.5, 1.0, 2.0, -0.5, -1.0, -2.0], size=shape)


@pytest.mark.parametrize("K", [32, 70, 5])
def test_mx_rows_matmul_on_grid_is_the_matmul(K):
    rng = np.random.default_rng(K)
    A, B = _grid(rng, (K, 40)), _grid(rng, (K, 24))
    np.testing.assert_array_equal(oracle.mx_rows_matmul(A, B), A.T @ B)


def test_mx_rows_matmul_error_bound():
    # each operand element moves by at most 2^-4 of itself (E4M3 rounding of
    # a normal value) plus half the subnormal quantum of its block, 2^-10 X
    # with X <= 2^-8 of the block's largest magnitude
    rng = np.random.default_rng(7)
    K, M, N = 100, 48, 40
    A = rng.standard_normal((K, M)) * np.exp(rng.standard_normal((K, 1)))
    B = rng.standard_normal((K, N)) * np.exp(rng.standard_normal((1, N)))
    out = oracle.mx_rows_matmul(A, B)
    exact = A.T @ B
    ea = 2.0 ** -4 * np.abs(A) + 2.0 ** -18 * np.abs(A).max()
    eb = 2.0 ** -4 * np.abs(B) + 2.0 ** -18 * np.abs(B).max()
    bound = ea.T @ np.abs(B) + np.abs(A).T @ eb + ea.T @ eb
    assert np.all(np.abs(out - exact) <= bound * (1 + 1e-12))
    assert np.linalg.norm(out - exact) < 0.05 * np.linalg.norm(exact)
    # quantising along the columns instead (a plausible mistake) differs
    qa = oracle.mx_dequantize(*oracle.mx_quantize(A[:, :32].copy()))
    qb = oracle.mx_dequantize(*oracle.mx_quantize(B[:, :32].copy()))
    assert np.abs(qa.T @ qb - out[:32, :32]).max() > 1e-6 * np.abs(out).max()


def test_mx_rows_matmul_blocks_start_at_row_zero():
    rng = np.random.default_rng(9)
    A, B = rng.standard_normal((96, 16)), rng.standard_normal((96, 8))
    # independent blocks of 32 rows from row 0
    parts = sum(oracle.mx_rows_matmul(A[i:i + 32], B[i:i + 32]) for i in (0, 32, 64))
    np.testing.assert_allclose(oracle.mx_rows_matmul(A, B), parts, rtol=1e-12, atol=1e-12)
    # moving the rows across block boundaries (a plausible alignment mistake:
    # blocks counted from a global row, not the group's first) changes it
    Z = np.zeros((5, 16)), np.zeros((5, 8))
    shifted = oracle.mx_rows_matmul(np.vstack([Z[0], A]), np.vstack([Z[1], B]))
    assert np.abs(shifted - oracle.mx_rows_matmul(A, B)).max() > 1e-6


def _round_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


def test_expert_wgrad_mx_assembles_the_rows():
    # dW2 = rows-MX(dY rows, bf16(w h~)) and dW13 = rows-MX(bf16([dg|du]), x
    # rows), with h~ and [dg|du] the MX backward's (stored in bf16 like the
    # bf16 layer's weight-gradient operands; torch's cast is the rounding
    # routine), and both near the exact gradients
    x, dY, W13, W2, rt, re, rw = _bwd_case(grid=False, seed=13)
    e = 1
    sel = re == e
    rt_e, rw_e = rt[sel], rw[sel]
    out = oracle.expert_wgrad_mx(x, W13[e], W2[e], dY, rt_e, rw_e, 7.0)
    rows = oracle.expert_rows_mx_backward(x, W13[e:e + 1], W2[e:e + 1], dY, rt_e,
                                          np.zeros(len(rt_e), np.int32), rw_e, 7.0)
    xr, dyr = x.double().numpy()[rt_e], dY.double().numpy()[rt_e]
    np.testing.assert_array_equal(out["dW2"],
                                  oracle.mx_rows_matmul(dyr, _round_bf16(rw_e[:, None] * rows["h"])))
    np.testing.assert_array_equal(out["dW13"], oracle.mx_rows_matmul(_round_bf16(rows["dgu"]), xr))
    ex = oracle.expert_wgrad(x, W13, W2, dY, e, rt_e, rw_e, 7.0, exact=True)
    for k in ("dW2", "dW13"):
        rel = np.linalg.norm(out[k] - ex[k]) / np.linalg.norm(ex[k])
        assert 1e-3 < rel < 0.15, (k, rel)
