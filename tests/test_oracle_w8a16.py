"""Pins of the INT8 weight-only (W8A16) oracle (CPU only).

"Kernel dispatch and Humming quantization in PhyAI": INT8 is one of the
Humming weight schemes (section "Choose precision by layer and hardware");
round to nearest at load, group 128 (section "Humming makes the separation
useful"), read as the INT4 method with 8-bit codes: fp16(fp32 absmax / 127),
codes clamp(rint(x / s), -128, 127).

Each check takes a namespace of oracle functions, so that the mutant tests at
the end can run the same pins on planted mistakes."""

import os
import types
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import w8a16_oracle as o8
import pins

HERE = os.path.dirname(os.path.abspath(__file__))


def real_ns():
    return types.SimpleNamespace(quantize8_f32=o8.quantize8_f32, quantize8=o8.quantize8,
                                 dequantize8=o8.dequantize8, gemm8=o8.gemm8,
                                 to_tile_layout8=o8.to_tile_layout8,
                                 from_tile_layout8=o8.from_tile_layout8)


def expected_scale8(group_vals) -> Fraction:
    """fp16(fp32(amax / 127)), zero -> 1, in exact arithmetic."""
    amax = max(abs(Fraction(float(v))) for v in group_vals)
    s16 = pins.round_binary(pins.round_binary(amax / 127, pins.FP32), pins.FP16)
    return Fraction(1) if s16 == 0 else s16


def brute_force_code8(x: Fraction, s: Fraction) -> int:
    """argmin over all 256 codes c of |x - c s|, ties to the even c."""
    best = None
    for c in range(-128, 128):
        d = abs(x - c * s)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


def load_golden8():
    rows = {}
    with open(os.path.join(HERE, "golden", "rtn8_hand_examples.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, xs, sc, codes, by = (p.strip() for p in line.split("|"))
            rows[name] = ([float(v) for v in xs.split()], int(sc, 16),
                          [int(v) for v in codes.split()], [int(v, 16) for v in by.split()])
    return rows


# ------------------------------------------------------------------- pins
def check_hand_examples(ns):
    rows = load_golden8()
    assert set(rows) == {"r0", "r1", "r2", "r3"}
    x = np.zeros((4, 128), np.float32)
    for i, n in enumerate(["r0", "r1", "r2", "r3"]):
        xs = rows[n][0]
        x[i, :len(xs)] = xs
    codes, sbits = ns.quantize8_f32(x)
    for i, n in enumerate(["r0", "r1", "r2", "r3"]):
        _, sc, cs, by = rows[n]
        assert int(sbits[0, i]) == sc, (n, hex(int(sbits[0, i])))
        assert list(codes[i, :len(cs)].view(np.int8)) == cs, n
        assert list(codes[i, :len(by)]) == by, n
        assert not codes[i, max(len(cs), len(by)):].any(), n


def check_scales_and_codes_exact(ns, x):
    codes, sbits = ns.quantize8_f32(x)
    q = codes.view(np.int8)
    sv = pins.scale_values(sbits)
    N, K = x.shape
    for n in range(N):
        for g in range(K // 128):
            grp = x[n, 128 * g:128 * (g + 1)]
            s = expected_scale8(grp)
            assert Fraction(float(sv[g, n])) == s, (n, g)
            for k in range(128):
                assert int(q[n, 128 * g + k]) == brute_force_code8(Fraction(float(grp[k])), s), (n, g, k)


def check_local_optimal(ns, x):
    """Vectorised brute force for a large sample: |x - q s| against the
    neighbouring codes in float64 (exact for these magnitudes; |x - c s| is
    convex in c)."""
    codes, sbits = ns.quantize8_f32(x)
    q = codes.view(np.int8).astype(np.float64)
    s = np.repeat(pins.scale_values(sbits).T, 128, axis=1)
    xd = x.astype(np.float64)
    d0 = np.abs(xd - q * s)
    even = (q % 2) == 0
    for step in (1.0, -1.0):
        nb = q + step
        valid = (nb >= -128) & (nb <= 127)
        dn = np.abs(xd - nb * s)
        assert (((d0 < dn) | ((d0 == dn) & even)) | ~valid).all()


def check_invariants(ns, x):
    codes, sbits = ns.quantize8_f32(x)
    q = codes.view(np.int8)
    N, K = x.shape
    G = K // 128
    sv = pins.scale_values(sbits)
    normal = sv >= 2.0 ** -14
    amax = np.abs(x.reshape(N, G, 128)).max(axis=2).T
    rescued = (sv == 1.0) & (amax < 127 * 2.0 ** -25)
    wd = ns.dequantize8(codes, sbits)
    c2, s2 = ns.quantize8_f32(wd)
    for g in range(G):
        sl = slice(128 * g, 128 * (g + 1))
        for n in range(N):
            if normal[g, n] and not rescued[g, n]:
                assert s2[g, n] == sbits[g, n] and (c2[n, sl] == codes[n, sl]).all(), (n, g)
                err = np.abs(x[n, sl].astype(np.float64) - q[n, sl] * sv[g, n])
                assert (err <= sv[g, n] / 2).all(), (n, g)
                assert np.abs(q[n, sl].astype(np.int32)).max() == 127, (n, g)
                assert q[n, sl].min() >= -127, (n, g)       # -128 never for a normal scale
            if amax[g, n] == 0:
                assert sv[g, n] == 1.0 and not q[n, sl].any()


def check_tile_layout(ns):
    rng = np.random.default_rng(3)
    N, K = 200, 384
    b = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    t = ns.to_tile_layout8(b)
    assert t.size == 256 * K
    G = K // 128
    for (n, k) in [(0, 0), (5, 130), (127, 383), (128, 0), (199, 255)]:
        tn, g, r, c = n // 128, k // 128, n % 128, k % 128
        assert t[(tn * G + g) * 16384 + r * 128 + c] == b[n, k], (n, k)
    assert not t.reshape(2, G, 128, 128)[1, :, 72:, :].any()      # padding rows
    assert np.array_equal(ns.from_tile_layout8(t, N, K), b)


def check_gemm(ns):
    x = pins.random_weights(10, 256, 9, "t4")
    rng = np.random.default_rng(10)
    a = pins.bf16_round(rng.standard_normal((3, 256)).astype(np.float32))
    bias = pins.bf16_round(rng.standard_normal(10).astype(np.float32))
    codes, sbits = ns.quantize8(pins.to_bits(x))
    wd = ns.dequantize8(codes, sbits).astype(np.float64)
    # dequantize is q * s exactly
    q = codes.view(np.int8).astype(np.float64)
    assert np.array_equal(wd, q * np.repeat(pins.scale_values(sbits).T, 128, axis=1))
    y = ns.gemm8(pins.to_bits(a), codes, sbits, pins.to_bits(bias)).astype(np.float64)
    ye = pins.exact_gemm(a.astype(np.float64), wd, bias.astype(np.float64))
    gamma = 257 * 2.0 ** -24 / (1 - 257 * 2.0 ** -24)
    mag = np.abs(a.astype(np.float64)) @ np.abs(wd).T + np.abs(bias.astype(np.float64))[None, :]
    assert (np.abs(y - ye) <= gamma * mag + 1e-45).all()
    # one-hot rows of A return columns of the dequantized weight exactly
    ks = [0, 1, 127, 128, 255]
    oh = np.zeros((len(ks), 256), np.uint16)
    for m, k in enumerate(ks):
        oh[m, k] = 0x3F80
    yo = ns.gemm8(oh, codes, sbits)
    for m, k in enumerate(ks):
        assert (yo[m] == wd[:, k]).all()


def check_gemm_integer_exact(ns):
    # power-of-two scales and small integer activations: every product and
    # partial sum is exact in fp32, so the result is the exact integer sum
    rng = np.random.default_rng(17)
    N, K, M = 16, 512, 4
    e = rng.integers(-3, 0, size=(N, K // 128))
    c = rng.integers(-60, 61, size=(N, K))
    c[:, ::128] = 127
    x = (c * np.repeat(2.0 ** e, 128, axis=1)).astype(np.float32)
    a = rng.integers(-2, 3, size=(M, K)).astype(np.float32)
    codes, sbits = ns.quantize8_f32(x)
    y = ns.gemm8(pins.to_bits(a), codes, sbits)
    assert np.array_equal(y.astype(np.float64), a.astype(np.float64) @ x.astype(np.float64).T)


def _all(ns):
    check_hand_examples(ns)
    check_scales_and_codes_exact(ns, pins.special_groups(6).reshape(3, 256))
    check_local_optimal(ns, pins.random_weights(512, 1024, 4, "t4"))
    check_invariants(ns, np.concatenate([pins.special_groups(16).reshape(4, 512),
                                         pins.random_weights(12, 512, 6, "normal")]))
    check_tile_layout(ns)
    check_gemm(ns)
    check_gemm_integer_exact(ns)


ALL = [check_hand_examples, check_tile_layout, check_gemm, check_gemm_integer_exact]


def test_hand_examples():
    check_hand_examples(real_ns())


def test_scales_and_codes_exact():
    check_scales_and_codes_exact(real_ns(), pins.special_groups(6).reshape(3, 256))


def test_local_optimal_and_invariants():
    ns = real_ns()
    check_local_optimal(ns, pins.random_weights(512, 1024, 4, "t4"))
    check_invariants(ns, np.concatenate([pins.special_groups(16).reshape(4, 512),
                                         pins.random_weights(12, 512, 6, "normal")]))


def test_tile_layout():
    check_tile_layout(real_ns())


def test_gemm():
    check_gemm(real_ns())
    check_gemm_integer_exact(real_ns())


# ---------------------------------------------------------------- mutants
def _q8_variant(div_by=127.0, fp32_scale=False, ties_away=False):
    def q(x, group=128):
        x = np.ascontiguousarray(x, np.float32)
        N, K = x.shape
        xg = x.reshape(N, K // group, group)
        s32 = np.max(np.abs(xg), axis=2) / np.float32(div_by)
        s16 = s32.astype(np.float16)
        s16 = np.where(s16 == 0, np.float16(1.0), s16)
        sd = np.where(s32 == 0, np.float32(1.0), s32) if fp32_scale else s16.astype(np.float32)
        r = xg / sd[:, :, None]
        r = np.floor(r + np.float32(0.5)) if ties_away else np.rint(r)
        qq = np.clip(r, -128, 127).astype(np.int8).reshape(N, K)
        return qq.view(np.uint8), np.ascontiguousarray(s16.T).view(np.uint16)
    return q


def _tile_transposed(codes):
    codes = np.ascontiguousarray(codes, np.uint8)
    N, K = codes.shape
    nt = (N + 127) // 128
    p = np.zeros((nt * 128, K), np.uint8)
    p[:N] = codes
    return np.ascontiguousarray(p.reshape(nt, 128, K // 128, 128).transpose(2, 0, 1, 3)).reshape(-1)


MUTANTS = {
    "div_by_128": dict(quantize8_f32=_q8_variant(div_by=128.0)),
    "fp32_scale_codes": dict(quantize8_f32=_q8_variant(fp32_scale=True)),
    "ties_away": dict(quantize8_f32=_q8_variant(ties_away=True)),
    "tile_order": dict(to_tile_layout8=_tile_transposed),
    "gemm_drop_bias": dict(gemm8=lambda a, c, s, b=None, group=128, rows=None, act="bf16":
                           o8.gemm8(a, c, s, None, group, rows, act)),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_w8_mutant_is_caught(name):
    ns = real_ns()
    for k, v in MUTANTS[name].items():
        setattr(ns, k, v)
    if "quantize8_f32" in MUTANTS[name]:
        ns.quantize8 = lambda w, group=128: ns.quantize8_f32(oracle.bf16_bits_to_f32(w), group)
    with pytest.raises(AssertionError):
        _all(ns)


def test_unmutated_copy_passes():
    _all(real_ns())
