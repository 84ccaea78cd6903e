"""Pins of the oracle's SwiGLU epilogue ("Piper Kernels", section "ConvRot
INT8": SwiGLU of a raw [up | gate] tensor; here the halves interleave, up f in
column 2f and gate f in column 2f + 1).  The pins use facts of the logistic
function, not its formula: sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4,
sigmoid(-ln 3) = 1/4, sigmoid(ln 7) = 7/8, and e^-x - e^-2x < sigmoid(-x) <
e^-x; planted mistakes (halves swapped, the exponent's sign, the pairing)
each fail one of them."""

import math

import numpy as np
import pytest

import oracle
from oracle import w4a16_oracle as base

LN3, LN7 = math.log(3.0), math.log(7.0)


def _rational_points(swiglu):
    # pairs (up, gate) with gates whose logistic value is rational
    y = np.array([[2.0, 0.0, -3.0, LN3, 0.5, -LN3, 4.0, LN7]])
    h = swiglu(y)
    want = np.array([[0.0, -3.0 * LN3 * 0.75, 0.5 * -LN3 * 0.25, 4.0 * LN7 * 0.875]])
    return h.shape == want.shape and np.allclose(h, want, rtol=1e-14, atol=1e-15)


def _hand_gemm(gemm_swiglu):
    # K = 128, A = [1, 2, 0, ...]; rows up0 = 7 e0, gate0 = 7 e1, up1 = 7 e1,
    # gate1 = -7 e0 (amax 7: scale 1, codes = values), so y = [7, 14, 14, -7]
    w = np.zeros((4, 128), np.float32)
    w[0, 0], w[1, 1], w[2, 1], w[3, 0] = 7.0, 7.0, 7.0, -7.0
    a = np.zeros((1, 128), np.float32)
    a[0, 0], a[0, 1] = 1.0, 2.0
    packed, scales = oracle.quantize_f32(w)
    a_bits = (a.view(np.uint32) >> 16).astype(np.uint16)
    h = gemm_swiglu(a_bits, packed, scales)
    if h.shape != (1, 2):
        return False
    e7, e14 = math.exp(-7.0), math.exp(-14.0)
    h0_ok = 98.0 * (1.0 - e14) < h[0, 0] < 98.0          # 7 * silu(14), sigmoid(14) = 1 - sigmoid(-14)
    h1_ok = -98.0 * e7 < h[0, 1] < -98.0 * (e7 - e14)    # 14 * silu(-7)
    return bool(h0_ok and h1_ok)


def test_rational_sigmoid_points():
    assert _rational_points(oracle.swiglu)


def test_hand_worked_gemm():
    assert _hand_gemm(oracle.gemm_swiglu)


def test_large_magnitudes_are_finite():
    h = oracle.swiglu(np.array([[3.0, -1000.0, 3.0, 1000.0]]))
    assert h[0, 0] == 0.0 and h[0, 1] == 3000.0


def test_odd_width_is_rejected():
    with pytest.raises(ValueError):
        oracle.swiglu(np.zeros((1, 3)))


def _swapped(y):
    y = np.asarray(y, np.float64)
    up, gate = y[:, 1::2], y[:, 0::2]
    with np.errstate(over="ignore"):
        return gate / (1.0 + np.exp(-gate)) * up


def _exp_sign(y):
    y = np.asarray(y, np.float64)
    up, gate = y[:, 0::2], y[:, 1::2]
    with np.errstate(over="ignore"):
        return gate / (1.0 + np.exp(gate)) * up


def _halves(y):
    # the halves layout instead of the interleaved one
    y = np.asarray(y, np.float64)
    F = y.shape[1] // 2
    up, gate = y[:, :F], y[:, F:]
    with np.errstate(over="ignore"):
        return gate / (1.0 + np.exp(-gate)) * up


@pytest.mark.parametrize("mutant", [_swapped, _exp_sign, _halves], ids=["swapped", "exp_sign", "halves"])
def test_planted_mistakes_fail_a_pin(mutant):
    gemm_mutant = lambda a_bits, packed, scales: mutant(base.gemm(a_bits, packed, scales))
    assert not (_rational_points(mutant) and _hand_gemm(gemm_mutant))


def _bias_only(gemm_swiglu):
    # A = 0, so the pre-activation is the bias: (up0, gate0, up1, gate1) =
    # (2, ln 3, 5, 0) gives h = (2 ln 3 * 3/4, 0)
    w = np.zeros((4, 128), np.float32)
    w[:, 0] = 7.0
    packed, scales = oracle.quantize_f32(w)
    a_bits = np.zeros((1, 128), np.uint16)
    bias = np.array([2.0, LN3, 5.0, 0.0], np.float32)
    bias_bits = (bias.view(np.uint32) >> 16).astype(np.uint16)     # bf16 (truncation)
    b = (bias_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    h = gemm_swiglu(a_bits, packed, scales, bias_bits)
    want = np.array([[b[0] * b[1] / (1.0 + math.exp(-b[1])), 0.0]])
    return h.shape == want.shape and np.allclose(h, want, rtol=1e-6, atol=1e-12)


def test_bias_enters_before_swiglu():
    assert _bias_only(oracle.gemm_swiglu)
    # sigmoid(bf16(ln 3)) is within 1e-2 of 3/4: the bias pair is (up, gate)
    b1 = float(((np.array([LN3], np.float32).view(np.uint32) >> 16) << 16).view(np.float32)[0])
    assert abs(1.0 / (1.0 + math.exp(-b1)) - 0.75) < 1e-2


@pytest.mark.parametrize("where", ["after", "halves"])
def test_bias_mistakes_fail_the_pin(where):
    def mutant(a_bits, packed, scales, bias_bits=None):
        y = base.gemm(a_bits, packed, scales)
        b = base.act_bits_to_f32(bias_bits, "bf16").astype(np.float64)
        if where == "after":       # bias added to h instead of to y
            return oracle.swiglu(y) + b[0::2][None, :]
        F = b.size // 2            # bias read as [up | gate] halves
        return oracle.swiglu(y + np.stack([b[:F], b[F:]], axis=1).reshape(-1)[None, :])
    assert not _bias_only(mutant)
