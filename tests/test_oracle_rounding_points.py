"""Pins of the oracle's rounding points (mirror mode), on hand-picked bf16
cases where rounding at a different point changes a value the test asserts.

The layer stores its activations in bf16 and the oracle's mirror mode rounds
where the layer stores one (G|U, H, Yp, out, dYp, dA; fp32 for dXp, dx and
the weight gradients). Which value gets rounded, and when, is a reading of
the pages (they fix no precision), and these cases fix the reading:
  forward   A = bf16(G|U) with G, U exact sums of products;
            H = bf16(silu(G) U) from the UNROUNDED G and U;
            Yp = bf16(H W_down^T) from the ROUNDED H;
  backward  dH = dYp W_down unrounded; G, U come from the stored bf16 A;
            dA = bf16([dG | dU]); dXp = fp32(dA W_gu) from the ROUNDED dA;
  combine   out = bf16(sum_k w_k Yp_k): one rounding after the sum;
  dYp       = bf16(w dout);  dx = fp32(sum_k dXp_k + dx_add).
The inputs are bf16 values (as the layer receives them); the expected values
are recomputed here from the formulas with Python floats (math.exp) and the
oracle's bf16 rounding, which test_oracle_values.py pins against torch. For
each case the test also checks that the alternative rounding point gives a
different value, and that every value before rounding lies well away from a
rounding midpoint, so that the last-bit behaviour of exp cannot decide it.
"""
import math

import numpy as np

from oracle import moe_oracle as O


def rb(v: float) -> float:
    return float(O.round_bf16(np.float64(v)))


def f32(v: float) -> float:
    return float(np.float32(v))


def is_bf16(v: float) -> bool:
    return rb(v) == v


def clear_of_midpoint(v: float, bits: int = 8) -> bool:
    """v is at least 2^-16 of a unit in the last place away from the
    midpoint between two neighbouring values of `bits` significant bits."""
    if v == 0.0:
        return True
    m, _ = math.frexp(abs(v))          # m in [0.5, 1)
    s = m * 2.0 ** bits
    return abs((s - math.floor(s)) - 0.5) > 2.0 ** -16


def silu(g: float) -> float:
    return g / (1.0 + math.exp(-g))


def sigmoid(g: float) -> float:
    return 1.0 / (1.0 + math.exp(-g))


# one token, d = 2, one expert with F = 1
x = [0.0177001953125, -0.61328125]
wg = [-0.6328125, -0.9921875]
wu = [0.048095703125, 1.0703125]
wd = [-0.32421875, 0.5]     # W_down [d=2, F=1]
dy = [0.419921875, 0.0]     # upstream gradient of Yp


def _arrays():
    X = np.array([x])
    Wgu = np.array([wg, wu])
    Wd = np.array([[wd[0]], [wd[1]]])
    return X, Wgu, Wd


def test_inputs_are_bf16_values():
    assert all(is_bf16(v) for v in x + wg + wu + wd + dy)


def test_forward_rounding_points():
    G = x[0] * wg[0] + x[1] * wg[1]          # exact: products of 8-bit significands
    U = x[0] * wu[0] + x[1] * wu[1]
    assert not is_bf16(G) and not is_bf16(U)
    h = silu(G) * U
    H = rb(h)
    Y = [rb(H * wd[0]), rb(H * wd[1])]
    for v in (G, U, h, H * wd[0]):
        assert clear_of_midpoint(v)
    A, H_o, Y_o = O.swiglu_group(*_arrays(), O.round_bf16)
    assert A.tolist() == [[rb(G), rb(U)]]
    assert H_o.tolist() == [[H]]
    assert Y_o.tolist() == [Y]
    # the alternatives differ: H from bf16-rounded G and U, Yp from unrounded H
    assert clear_of_midpoint(silu(rb(G)) * rb(U)) and clear_of_midpoint(h * wd[0])
    assert rb(silu(rb(G)) * rb(U)) != H
    assert rb(h * wd[0]) != Y[0]


def test_backward_rounding_points():
    X, Wgu, Wd = _arrays()
    A, H, _ = O.swiglu_group(X, Wgu, Wd, O.round_bf16)
    Gb, Ub = float(A[0, 0]), float(A[0, 1])
    dH = dy[0] * wd[0] + dy[1] * wd[1]
    assert not is_bf16(dH)
    sg = sigmoid(Gb)
    dG = dH * Ub * sg * (1.0 + Gb * (1.0 - sg))
    dU = dH * Gb * sg
    for v in (dG, dU):
        assert clear_of_midpoint(v)
    dA = [rb(dG), rb(dU)]
    dX = [f32(dA[0] * wg[j] + dA[1] * wu[j]) for j in range(2)]
    dWd = [[f32(dy[0] * float(H[0, 0]))], [f32(dy[1] * float(H[0, 0]))]]
    dWgu = [[f32(dA[0] * x[j]) for j in range(2)], [f32(dA[1] * x[j]) for j in range(2)]]
    dX_o, dWd_o, dWgu_o, dA_o = O.swiglu_group_bwd(np.array([dy]), X, A, H, Wgu, Wd,
                                                   O.round_bf16, O.round_f32)
    assert dA_o.tolist() == [dA]
    assert dX_o.tolist() == [dX]
    assert dWd_o.tolist() == dWd
    assert dWgu_o.tolist() == dWgu
    # the alternatives differ: dA from a bf16-rounded dH, dXp from the unrounded dA
    dHb = rb(dH)
    alt = [rb(dHb * Ub * sg * (1.0 + Gb * (1.0 - sg))), rb(dHb * Gb * sg)]
    assert alt != dA
    assert [f32(dG * wg[j] + dU * wu[j]) for j in range(2)] != dX


def test_combine_rounds_once_after_the_sum():
    y = [1.875, -1.2109375]                          # bf16 rows of Yp (d = 1)
    w = [0.7936545014381409, 0.3989872634410858]     # fp32 combine weights
    assert all(is_bf16(v) for v in y) and all(f32(v) == v for v in w)
    s = w[0] * y[0] + w[1] * y[1]
    assert clear_of_midpoint(s)
    row_of = np.array([[0, 1]], np.int32)
    out = O.unpermute(np.array([[y[0]], [y[1]]]), row_of, np.array([w]), dtype="bf16")
    assert out.tolist() == [[rb(s)]]
    assert rb(rb(w[0] * y[0]) + rb(w[1] * y[1])) != rb(s)   # per-term rounding differs


def test_unpermute_bwd_rounds_dyp_to_bf16_and_keeps_dw_fp32():
    g, w, yp = 0.419921875, 0.7936545014381409, 1.875
    r = O.unpermute_bwd(np.array([[g]]), np.array([[yp]]), np.array([[0]], np.int32),
                        np.array([[w]]), dtype="bf16")
    assert clear_of_midpoint(w * g)
    assert r["dYp"].tolist() == [[rb(w * g)]] and rb(w * g) != w * g
    assert r["dw"].tolist() == [[f32(g * yp)]]


def test_permute_bwd_sums_in_fp32():
    dXp = np.array([[1.0 + 2.0 ** -20], [2.0 ** -10]])
    r = O.permute_bwd(dXp, np.array([[0, 1]], np.int32), np.array([[3.0 ** -5]]))
    v = (1.0 + 2.0 ** -20) + 2.0 ** -10 + 3.0 ** -5
    assert r.tolist() == [[f32(v)]]
    assert f32(v) != rb(v)   # an fp32 value, not a bf16 one
