"""Checks that pin the CPU oracle to facts that do not come from the oracle.

Each ``check_*`` takes an oracle-like namespace (``quantize_f32``,
``quantize``, ``dequantize``, ``gemm``, ``unpack_codes``) and raises
``AssertionError`` when it disagrees with:

* the hand-worked examples in ``golden/rtn_hand_examples.txt``;
* exact rational arithmetic (``fractions.Fraction``) for the scale formula,
  i.e. fp16(fp32(amax / 7)) with IEEE round-to-nearest-even implemented here
  from its definition (not by a float cast);
* brute force over all 16 codes for the code choice;
* exact dot products (``math.fsum`` of exact products) with the standard
  floating-point summation error bound for the GEMM;
* closed forms: one-hot activation rows, power-of-two scales with integer
  activations (exact integer sums).

``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutants.py``
plants plausible mistakes in copies of the oracle and shows each is caught.
"""

from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "rtn_hand_examples.txt")

FP32 = (24, -126)   # significand bits (with the hidden bit), min normal exponent
FP16 = (11, -14)


# --------------------------------------------------------------------------
# exact IEEE rounding from the definition
# --------------------------------------------------------------------------
def round_binary(v: Fraction, fmt) -> Fraction:
    """Round ``v`` to the nearest value of a binary format with ``p``-bit
    significand and minimum normal exponent ``emin`` (subnormals kept, no
    overflow), ties to the even significand."""
    p, emin = fmt
    if v == 0:
        return Fraction(0)
    sign = 1 if v > 0 else -1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    ulp = Fraction(2) ** (e - p + 1)
    m = a / ulp
    n = m.numerator // m.denominator
    r = m - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def expected_scale(group_vals) -> Fraction:
    """fp16(fp32(amax / 7)), zero -> 1, all in exact arithmetic."""
    amax = max(abs(Fraction(float(v))) for v in group_vals)
    s32 = round_binary(amax / 7, FP32)
    s16 = round_binary(s32, FP16)
    return Fraction(1) if s16 == 0 else s16


def brute_force_code(x: Fraction, s: Fraction) -> int:
    """argmin over c in [-8, 7] of |x - c*s|, ties to the even c."""
    best = None
    for c in range(-8, 8):
        d = abs(x - c * s)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


# --------------------------------------------------------------------------
# golden fixture
# --------------------------------------------------------------------------
def load_golden():
    rows, gemms = {}, []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [p.strip() for p in line.split("|")]
            if parts[0].startswith("gemm"):
                gemms.append((parts[0], parts[1].split(), [float(v) for v in parts[2].split()]))
                continue
            name, xs, shex, codes, pbytes = parts
            rows[name] = dict(
                x=[float(v) for v in xs.split()],
                scale_bits=int(shex, 16),
                codes=[int(v) for v in codes.split()],
                packed=[int(v, 16) for v in pbytes.split()],
            )
    return rows, gemms


def golden_row_values(row) -> np.ndarray:
    x = np.zeros(128, dtype=np.float32)
    x[: len(row["x"])] = row["x"]
    return x


def check_hand_examples(orc):
    rows, gemms = load_golden()
    names = list(rows)
    x = np.stack([golden_row_values(rows[n]) for n in names])
    packed, sbits = orc.quantize_f32(x)
    codes = orc.unpack_codes(packed)
    for i, n in enumerate(names):
        r = rows[n]
        assert int(sbits[0, i]) == r["scale_bits"], (n, hex(int(sbits[0, i])))
        assert list(codes[i, :8]) == r["codes"], (n, list(codes[i, :8]))
        assert list(packed[i, :4]) == r["packed"], (n, list(packed[i, :4]))
        assert not codes[i, 8:].any()
        # the scale also re-derived exactly from the row
        assert Fraction(float(np.uint16(sbits[0, i]).view(np.float16))) == expected_scale(x[i])
    for _, wnames, yexp in gemms:
        w = np.stack([golden_row_values(rows[n]) for n in wnames])
        pk, sb = orc.quantize_f32(w)
        ones = np.full((1, 128), 0x3F80, dtype=np.uint16)      # bf16 1.0
        y = orc.gemm(ones, pk, sb)
        assert y.shape == (1, len(wnames))
        assert [float(v) for v in y[0]] == yexp, (list(y[0]), yexp)


# --------------------------------------------------------------------------
# quantize
# --------------------------------------------------------------------------
def scale_values(sbits: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(sbits, dtype=np.uint16).view(np.float16).astype(np.float64)


def check_scales_exact(orc, x: np.ndarray):
    """Every scale equals the exact-arithmetic fp16(fp32(amax/7)) (zero->1),
    stored at scales[g, n]."""
    _, sbits = orc.quantize_f32(x)
    N, K = x.shape
    G = K // 128
    assert sbits.shape == (G, N), sbits.shape
    sv = scale_values(sbits)
    for n in range(N):
        for g in range(G):
            exp = expected_scale(x[n, 128 * g: 128 * (g + 1)])
            assert Fraction(float(sv[g, n])) == exp, (n, g, float(sv[g, n]), float(exp))


def check_codes_bruteforce(orc, x: np.ndarray):
    """Every code equals the brute-force argmin over the 16 codes (exact
    rationals, ties to even) using the exact-arithmetic scale."""
    packed, _ = orc.quantize_f32(x)
    codes = orc.unpack_codes(packed)
    N, K = x.shape
    for n in range(N):
        for g in range(K // 128):
            s = expected_scale(x[n, 128 * g: 128 * (g + 1)])
            for k in range(128 * g, 128 * (g + 1)):
                c = brute_force_code(Fraction(float(x[n, k])), s)
                assert int(codes[n, k]) == c, (n, k, float(x[n, k]), float(s), int(codes[n, k]), c)


def check_codes_local_optimal(orc, x: np.ndarray):
    """Vectorised form of the brute force for large samples.  With x a bf16
    or fp32 value and s an fp16 value, every difference x - c*s that can
    decide between two neighbouring codes is exact in float64 (both operands
    lie within 2^30 of each other's scale), so comparing |x - q s| against
    |x - (q +- 1) s| in float64 is an exact local-optimality test; |x - c s|
    is convex in c, so local optimality over [-8, 7] is global."""
    packed, sbits = orc.quantize_f32(x)
    codes = orc.unpack_codes(packed).astype(np.float64)
    N, K = x.shape
    s = np.repeat(scale_values(sbits).T, 128, axis=1)    # [N, K]
    xd = x.astype(np.float64)
    d0 = np.abs(xd - codes * s)
    even = (codes % 2) == 0
    for step in (1.0, -1.0):
        nb = codes + step
        valid = (nb >= -8) & (nb <= 7)
        dn = np.abs(xd - nb * s)
        ok = (d0 < dn) | ((d0 == dn) & even) | ~valid
        assert ok.all(), np.argwhere(~ok)[:5]
    assert codes.min() >= -8 and codes.max() <= 7


def check_invariants(orc, x: np.ndarray):
    """(i) codes in [-8,7]; (ii) dequantize then requantize reproduces codes
    and scales for groups with a normal fp16 scale; (iii) |x - q s| <= s/2 for
    normal scales; (iv) every group with a normal, non-rescued scale holds a
    +-7 code; (v) all-zero groups get scale 1 and codes 0."""
    packed, sbits = orc.quantize_f32(x)
    codes = orc.unpack_codes(packed)
    N, K = x.shape
    G = K // 128
    sv = scale_values(sbits)                                      # [G, N]
    assert codes.min() >= -8 and codes.max() <= 7                 # (i)
    normal = sv >= 2.0 ** -14                                     # [G, N]
    amax = np.abs(x.reshape(N, G, 128)).max(axis=2).T             # [G, N]
    rescued = (sv == 1.0) & (amax < 7 * 2.0 ** -25)               # zero rule applied
    wd = orc.dequantize(packed, sbits)
    p2, s2 = orc.quantize_f32(wd)
    c2 = orc.unpack_codes(p2)
    for g in range(G):
        sl = slice(128 * g, 128 * (g + 1))
        for n in range(N):
            if normal[g, n] and not rescued[g, n]:
                assert s2[g, n] == sbits[g, n], (n, g)            # (ii)
                assert (c2[n, sl] == codes[n, sl]).all(), (n, g)
                err = np.abs(x[n, sl].astype(np.float64) - codes[n, sl] * sv[g, n])
                assert (err <= sv[g, n] / 2).all(), (n, g)        # (iii)
                assert np.abs(codes[n, sl]).max() == 7, (n, g)     # (iv)
            if amax[g, n] == 0:
                assert sv[g, n] == 1.0 and not codes[n, sl].any()  # (v)


def check_dequantize(orc, x: np.ndarray):
    """dequantize(quantize(x)) is within half an exactly-derived scale of x,
    element by element (catches a wrong group index or scale layout)."""
    packed, sbits = orc.quantize_f32(x)
    wd = orc.dequantize(packed, sbits)
    assert wd.shape == x.shape and wd.dtype == np.float32
    N, K = x.shape
    for n in range(N):
        for g in range(K // 128):
            s = float(expected_scale(x[n, 128 * g: 128 * (g + 1)]))
            err = np.abs(wd[n, 128 * g: 128 * (g + 1)].astype(np.float64) - x[n, 128 * g: 128 * (g + 1)])
            if s >= 2.0 ** -14 and np.abs(x[n, 128 * g: 128 * (g + 1)]).max() <= 7.5 * s:
                assert (err <= s / 2).all(), (n, g)
            # every dequantized value is an integer multiple (-8..7) of s
            m = wd[n, 128 * g: 128 * (g + 1)].astype(np.float64) / s
            assert (m == np.round(m)).all() and m.min() >= -8 and m.max() <= 7


# --------------------------------------------------------------------------
# GEMM
# --------------------------------------------------------------------------
U32 = 2.0 ** -24


def exact_gemm(a: np.ndarray, wd: np.ndarray, bias=None) -> np.ndarray:
    """Correctly rounded float64 value of A @ Wd^T (+bias): each product of a
    bf16 and an (int4 x fp16) value is exact in float64 and math.fsum sums
    exactly before one rounding."""
    M, N = a.shape[0], wd.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    for m in range(M):
        for n in range(N):
            terms = [float(a[m, k]) * float(wd[n, k]) for k in range(a.shape[1])]
            if bias is not None:
                terms.append(float(bias[n]))
            y[m, n] = math.fsum(terms)
    return y


def check_gemm_exact_bound(orc, a_bits, w_bits, bias_bits=None, act="bf16"):
    """|Y_oracle - Y_exact| <= gamma_{K+1} * (sum |a w| + |b|): the a-priori
    bound of any FP32 summation order.  ``act``: type of the activation and
    bias bit patterns ("bf16" or "f16")."""
    packed, sbits = orc.quantize(w_bits)
    wd = orc.dequantize(packed, sbits).astype(np.float64)
    a = _bits_f64(a_bits, act)
    b = None if bias_bits is None else _bits_f64(bias_bits, act)
    y = (orc.gemm(a_bits, packed, sbits, bias_bits) if act == "bf16" else
         orc.gemm(a_bits, packed, sbits, bias_bits, act=act)).astype(np.float64)
    ye = exact_gemm(a, wd, b)
    K = a.shape[1]
    gamma = (K + 1) * U32 / (1 - (K + 1) * U32)
    mag = np.abs(a) @ np.abs(wd).T + (0 if b is None else np.abs(b)[None, :])
    assert y.shape == ye.shape
    assert (np.abs(y - ye) <= gamma * mag + 1e-45).all(), np.max(np.abs(y - ye) - gamma * mag)


def check_gemm_one_hot(orc, w_bits, act="bf16"):
    """A row of A equal to e_k (1.0 at k: bf16 0x3F80, fp16 0x3C00) returns
    column k of the dequantized weight exactly: Y[m, n] = Wd[n, k_m]."""
    packed, sbits = orc.quantize(w_bits)
    wd = orc.dequantize(packed, sbits)
    N, K = wd.shape
    ks = [0, 1, 127, 128, K // 2 + 3, K - 1]
    a = np.zeros((len(ks), K), dtype=np.uint16)
    for m, k in enumerate(ks):
        a[m, k] = 0x3F80 if act == "bf16" else 0x3C00
    y = orc.gemm(a, packed, sbits) if act == "bf16" else orc.gemm(a, packed, sbits, act=act)
    for m, k in enumerate(ks):
        assert (y[m] == wd[:, k]).all(), (m, k)


def check_gemm_integer_exact(orc, seed=7):
    """Power-of-two scales with small-integer activations: every partial sum
    is an exactly representable fp32 value, so the result equals the integer
    closed form exactly.  Rows use scale 2^j by making amax = 7 * 2^j."""
    rng = np.random.default_rng(seed)
    N, K, M = 24, 384, 5
    G = K // 128
    codes = rng.integers(-7, 8, size=(N, K))
    exps = rng.integers(-4, 3, size=(N, G))
    for n in range(N):
        for g in range(G):
            codes[n, 128 * g + rng.integers(0, 128)] = 7 * (1 if rng.random() < 0.5 else -1)
    x = (codes * np.repeat(2.0 ** exps, 128, axis=1)).astype(np.float32)
    a_int = rng.integers(-3, 4, size=(M, K))
    a_bits = (a_int.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # small ints are bf16-exact
    packed, sbits = orc.quantize_f32(x)
    y = orc.gemm(a_bits, packed, sbits)
    exact = a_int.astype(np.float64) @ x.astype(np.float64).T
    assert (y.astype(np.float64) == exact).all()
    # bias added once, in fp32 (exact here: small dyadic values)
    bias = (rng.integers(-8, 9, size=N).astype(np.float32) * np.float32(0.25))
    b_bits = (bias.view(np.uint32) >> 16).astype(np.uint16)
    yb = orc.gemm(a_bits, packed, sbits, b_bits)
    assert (yb.astype(np.float64) == exact + bias[None, :].astype(np.float64)).all()


def _bits_f64(bits, act="bf16"):
    if act == "f16":
        return f16_values(bits)
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f16_values(bits) -> np.ndarray:
    """IEEE binary16 bit patterns -> float64 values from the format's
    definition (sign, 5-bit biased exponent, 10-bit fraction; exponent 0 is
    subnormal), not through any library conversion."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    normal = sign * np.ldexp(1.0 + f / 1024.0, (e - 15).astype(np.int64))
    sub = sign * np.ldexp(f / 1024.0, -14)
    return np.where(e == 0, sub, normal)


def check_f16_widening(orc):
    """Every finite fp16 bit pattern widens to its defined value exactly."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = ((bits.astype(np.int64) >> 10) & 0x1F) != 0x1F
    got = orc.f16_bits_to_f32(bits[finite]).astype(np.float64)
    want = f16_values(bits[finite])
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------
# input sets used by the pins
# --------------------------------------------------------------------------
def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 values (returned as float32) with
    nearest-even, using integer arithmetic on the bit pattern."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) >> 16 << 16
    return u.astype(np.uint32).view(np.float32)


def special_groups(n_rows: int = 16) -> np.ndarray:
    """Rows of crafted 128-wide groups: zero, spikes, constants, exact ties,
    subnormal and underflowing scales, large values, bf16 extremes."""
    rng = np.random.default_rng(1234)
    rows = []
    z = np.zeros(128, np.float32)
    rows.append(z.copy())                                           # all zero
    r = z.copy(); r[17] = 3.0; rows.append(r)                       # single spike
    r = z.copy(); r[90] = -5.5; r[3] = 1.0; rows.append(r)          # negative spike sets amax
    rows.append(np.full(128, 0.3, np.float32))                      # constant
    r = (np.arange(128) % 16 - 7.5).astype(np.float32); r[0] = 7.0  # s = 1: x = k + 0.5 ties
    rows.append(r)
    r = (np.arange(128) % 29 - 14).astype(np.float32) / 2           # s = 1, halves: ties
    rows.append(r)
    r = bf16_round(rng.standard_normal(128).astype(np.float32) * 3e-5)  # subnormal fp16 scale
    rows.append(r)
    r = bf16_round(rng.standard_normal(128).astype(np.float32) * 1e-8)  # scale underflows -> 1
    rows.append(r)
    r = bf16_round(rng.standard_normal(128).astype(np.float32) * 1e5); r[5] = 4.0e5  # large
    rows.append(r)
    r = z.copy(); r[0] = 1e-38; r[1] = -2e-39; rows.append(bf16_round(r))  # tiny bf16 values
    r = bf16_round(rng.standard_t(4, 128).astype(np.float32) * 0.02)  # heavy tails
    rows.append(r)
    while len(rows) < n_rows:
        rows.append(bf16_round(rng.standard_normal(128).astype(np.float32) * 0.02))
    return np.stack(rows[:n_rows]).astype(np.float32)


def random_weights(N, K, seed, dist="normal") -> np.ndarray:
    rng = np.random.default_rng(seed)
    if dist == "normal":
        x = rng.standard_normal((N, K)).astype(np.float32) * np.float32(0.02)
    else:
        x = (rng.standard_t(4, (N, K)) * 0.02).astype(np.float32)
    return bf16_round(x)


def to_bits(x: np.ndarray) -> np.ndarray:
    """float32 values that are already bf16-exact -> uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert ((u & 0xFFFF) == 0).all()
    return (u >> 16).astype(np.uint16)
