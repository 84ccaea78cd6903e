"""Pins of the FP4 weight-only oracle (MXFP4 and NVFP4), CPU only.

"Kernel dispatch and Humming quantization in PhyAI", section "Choose
precision by layer and hardware": MXFP4 and NVFP4 weights with BF16
activations.  "Piper Kernels", section "NVFP4 construction": blocks of 16 and
a global per-tensor scale; the global scale and bias are applied in FP32 in
the GEMM epilogue.  Element format E2M1; MXFP4 per the OCP MX v1.0
specification (32-value blocks, E8M0 scales).

The pins compare the oracle with facts it does not compute itself:

* the E2M1 and E4M3 value sets written from their bit-level definitions, and
  rounding to them by exact rational arithmetic (``pins.round_binary``) with
  saturation, not by the oracle's tables and thresholds;
* the E4M3 value table of PyTorch's ``float8_e4m3fn`` type and its
  round-to-nearest cast (an independent library routine);
* the MX shared exponent by exact comparisons with powers of two;
* hand-worked blocks in ``golden/fp4_hand_examples.txt``;
* the whole quantize of small tensors recomputed element by element in
  ``fractions.Fraction`` arithmetic;
* dequantize and GEMM against exact products and sums (one-hot rows, the
  fp32 summation error bound).

Every check takes a namespace of oracle functions so that the mutant tests at
the end can run the same pins on planted mistakes."""

import math
import os
import types
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import fp4_oracle as f4
import pins

HERE = os.path.dirname(os.path.abspath(__file__))
E2M1 = (2, 0)      # significand bits with the hidden bit, minimum normal exponent
E4M3 = (4, -6)
F32 = pins.FP32


def real_ns():
    names = ["e2m1_decode", "e2m1_encode", "e4m3_encode", "e4m3_decode", "mx_exponent",
             "quantize_mxfp4_f32", "dequantize_mxfp4", "quantize_nvfp4_f32",
             "dequantize_nvfp4", "pack_codes_fp4", "unpack_codes_fp4", "gemm_fp4"]
    return types.SimpleNamespace(**{n: getattr(f4, n) for n in names})


# ----------------------------------------------------- format definitions
def e2m1_value(code: int) -> Fraction:
    """Value of a 4-bit E2M1 code from its fields: sign, 2 exponent bits
    (bias 1), 1 mantissa bit; exponent field 0 is subnormal."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return -v if s else v


def e4m3_value(code: int) -> Fraction:
    """Value of a non-negative E4M3 code (bias 7, 3 mantissa bits)."""
    e, m = (code >> 3) & 15, code & 7
    return Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else \
        (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


_E2M1_CODE = {e2m1_value(c): c for c in range(8)}
_E4M3_CODE = {e4m3_value(c): c for c in range(127)}


def e2m1_round(v: Fraction) -> int:
    """Code of v: nearest E2M1 value, ties to the even significand,
    saturating at 6; a result of 0 has no sign."""
    r = min(pins.round_binary(abs(v), E2M1), Fraction(6))
    c = _E2M1_CODE[r]
    return c | 8 if (v < 0 and c != 0) else c


def e4m3_round(v: Fraction) -> int:
    r = min(pins.round_binary(v, E4M3), Fraction(448))
    return _E4M3_CODE[r]


def f32(v: Fraction) -> Fraction:
    return pins.round_binary(v, F32)


# ------------------------------------------------------------------- pins
def check_e2m1_format(ns):
    assert [Fraction(float(v)) for v in ns.e2m1_decode(np.arange(16, dtype=np.uint8))] == \
        [e2m1_value(c) for c in range(16)]
    # every multiple of 1/16 in [-8, 8] (all midpoints included), random
    # values, values past the largest magnitude
    rng = np.random.default_rng(3)
    xs = np.concatenate([np.arange(-128, 129) / 16.0, rng.uniform(-7, 7, 400),
                         [6.5, -6.01, 100.0, -1e30, 1e-30, -1e-30]]).astype(np.float32)
    got = ns.e2m1_encode(xs)
    want = [e2m1_round(Fraction(float(x))) for x in xs]
    assert [int(g) for g in got] == want


def check_e4m3_format(ns):
    # the value table against PyTorch's float8_e4m3fn type
    codes = torch.arange(127, dtype=torch.uint8)
    tv = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ns.e4m3_decode(np.arange(127, dtype=np.uint8)).astype(np.float64), tv)
    assert [Fraction(float(v)) for v in tv] == [e4m3_value(c) for c in range(127)]
    # rounding: every midpoint between neighbours, random values, subnormals
    vals = np.array([float(e4m3_value(c)) for c in range(127)])
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(4)
    xs = np.concatenate([vals, mids, rng.uniform(0, 448, 300), rng.uniform(0, 2.0 ** -6, 100),
                         np.exp2(rng.uniform(-12, 8, 300))]).astype(np.float32)
    got = ns.e4m3_encode(xs)
    assert [int(g) for g in got] == [e4m3_round(Fraction(float(x))) for x in xs]
    # in range, the same as PyTorch's round-to-nearest cast
    inr = xs[xs <= 448]
    tc = torch.from_numpy(inr).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ns.e4m3_encode(inr), tc)
    # saturation
    assert [int(c) for c in ns.e4m3_encode(np.array([449, 464, 480, 1e6], np.float32))] == [126] * 4


def check_mx_exponent(ns):
    rng = np.random.default_rng(5)
    a = np.exp2(rng.uniform(-149, 127.9, 2000)).astype(np.float32)
    a = np.concatenate([a, np.float32([1, 2, 4, 6, 7.99, 8, 2.0 ** -126, 2.0 ** -149,
                                       3.4e38, 1e-45])])
    e = ns.mx_exponent(a).astype(int)
    for amax, code in zip(a.tolist(), e.tolist()):
        fa = Fraction(amax)
        if fa == 0:
            assert code == 127
            continue
        fl = math.floor(math.log2(amax))
        while Fraction(2) ** fl > fa:
            fl -= 1
        while Fraction(2) ** (fl + 1) <= fa:
            fl += 1
        assert code == min(max(fl - 2 + 127, 0), 254), amax
    assert int(ns.mx_exponent(np.float32([0.0]))[0]) == 127


def load_golden():
    rows = []
    with open(os.path.join(HERE, "golden", "fp4_hand_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            sch, t, b, xs, sc, cs = (p.strip() for p in line.split("|"))
            rows.append((sch, t, int(b), [float(v) for v in xs.split()], int(sc, 16),
                         [int(c, 16) for c in cs.split()]))
    return rows


def check_hand_examples(ns):
    rows = load_golden()
    assert len(rows) == 9
    for sch in ("mx", "nv"):
        bs = 32 if sch == "mx" else 16
        for t in sorted({r[1] for r in rows if r[0] == sch}):
            mine = [r for r in rows if r[0] == sch and r[1] == t]
            x = np.zeros((1, 128), np.float32)
            want_codes = np.zeros(128, np.uint8)
            want_sc = np.full(128 // bs, 0x7F if sch == "mx" else 0x00, np.uint8)
            for _, _, b, xs, sc, cs in mine:
                x[0, b * bs: b * bs + len(xs)] = xs
                want_codes[b * bs: b * bs + len(cs)] = cs
                want_sc[b] = sc
            if sch == "mx":
                packed, sc = ns.quantize_mxfp4_f32(x)
            else:
                packed, sc, _ = ns.quantize_nvfp4_f32(x)
            assert np.array_equal(sc[:, 0], want_sc), (sch, t)
            assert np.array_equal(ns.unpack_codes_fp4(packed)[0], want_codes), (sch, t)


def check_mx_exact(ns, x):
    """The whole MXFP4 quantize, element by element in exact arithmetic."""
    packed, sc = ns.quantize_mxfp4_f32(x)
    codes = ns.unpack_codes_fp4(packed)
    N, K = x.shape
    for n in range(N):
        for b in range(K // 32):
            blk = [Fraction(float(v)) for v in x[n, 32 * b: 32 * b + 32]]
            amax = max(abs(v) for v in blk)
            if amax == 0:
                e = 127
            else:
                fl = 0
                while Fraction(2) ** fl > amax:
                    fl -= 1
                while Fraction(2) ** (fl + 1) <= amax:
                    fl += 1
                e = min(max(fl - 2 + 127, 0), 254)
            assert int(sc[b, n]) == e, (n, b)
            scale = Fraction(2) ** (e - 127)
            for j, v in enumerate(blk):
                assert int(codes[n, 32 * b + j]) == e2m1_round(f32(v / scale)), (n, b, j)


def check_nv_exact(ns, x):
    """The whole NVFP4 quantize in exact arithmetic (every fp32 operation
    rounded from its exact value)."""
    packed, sc, g = ns.quantize_nvfp4_f32(x)
    codes = ns.unpack_codes_fp4(packed)
    N, K = x.shape
    amax_t = max(abs(Fraction(float(v))) for v in x.reshape(-1))
    g_want = Fraction(1) if amax_t == 0 else f32(amax_t / 2688)
    assert Fraction(float(g)) == g_want
    for n in range(N):
        for b in range(K // 16):
            blk = [Fraction(float(v)) for v in x[n, 16 * b: 16 * b + 16]]
            amax = max(abs(v) for v in blk)
            code = e4m3_round(f32(f32(amax / 6) / g_want))
            assert int(sc[b, n]) == code, (n, b)
            step = f32(e4m3_value(code) * g_want)
            for j, v in enumerate(blk):
                want = 0 if step == 0 else e2m1_round(f32(v / step))
                assert int(codes[n, 16 * b + j]) == want, (n, b, j)


def check_packing(ns):
    c = np.array([[1, 2, 3, 4, 15, 8, 0, 7]], np.uint8)
    p = ns.pack_codes_fp4(c)
    assert [int(v) for v in p[0]] == [0x21, 0x43, 0x8F, 0x70]   # low nibble = even k
    rng = np.random.default_rng(6)
    c = rng.integers(0, 16, (5, 64)).astype(np.uint8)
    assert np.array_equal(ns.unpack_codes_fp4(ns.pack_codes_fp4(c)), c)


def check_dequantize(ns, x):
    packed, sc = ns.quantize_mxfp4_f32(x)
    codes = ns.unpack_codes_fp4(packed)
    wd = ns.dequantize_mxfp4(packed, sc)
    for (n, k) in [(0, 0), (0, 31), (1, 32), (2, 127), (3, 200), (x.shape[0] - 1, x.shape[1] - 1)]:
        want = e2m1_value(int(codes[n, k])) * Fraction(2) ** (int(sc[k // 32, n]) - 127)
        assert Fraction(float(wd[n, k])) == want, (n, k)
    packed, sc, g = ns.quantize_nvfp4_f32(x)
    codes = ns.unpack_codes_fp4(packed)
    wd = ns.dequantize_nvfp4(packed, sc, g)
    for (n, k) in [(0, 0), (0, 15), (1, 16), (2, 127), (3, 200), (x.shape[0] - 1, x.shape[1] - 1)]:
        want = f32(e2m1_value(int(codes[n, k])) * e4m3_value(int(sc[k // 16, n])) *
                   Fraction(float(g)))
        assert Fraction(float(wd[n, k])) == want, (n, k)


def check_invariants(ns, x):
    # MXFP4: x * 2^j has the same codes and exponent + j; NVFP4: the same
    # codes and block scales, g * 2^j; negation flips the nonzero signs
    p0, s0 = ns.quantize_mxfp4_f32(x)
    p1, s1 = ns.quantize_mxfp4_f32(x * np.float32(8.0))
    assert np.array_equal(p0, p1)
    nz = s0 != 127    # all-zero blocks keep the zero rule's code
    assert np.array_equal(s1.astype(int)[nz], s0.astype(int)[nz] + 3)
    q0, t0, g0 = ns.quantize_nvfp4_f32(x)
    q1, t1, g1 = ns.quantize_nvfp4_f32(x * np.float32(0.25))
    assert np.array_equal(q0, q1) and np.array_equal(t0, t1) and g1 == g0 * np.float32(0.25)
    c0 = ns.unpack_codes_fp4(p0)
    cn = ns.unpack_codes_fp4(ns.quantize_mxfp4_f32(-x)[0])
    assert np.array_equal(cn, np.where(c0 & 7, c0 ^ 8, c0))
    # MXFP4 error bound: half a spacing of the code grid inside the range
    wd = ns.dequantize_mxfp4(p0, s0).astype(np.float64)
    sc = np.repeat(np.exp2(s0.astype(np.float64).T - 127), 32, axis=1)
    r = np.abs(x.astype(np.float64)) / sc
    spacing = np.where(r < 2, 0.5, np.where(r < 4, 1.0, 2.0))
    inside = r <= 6
    assert (np.abs(wd - x)[inside] <= (spacing * sc / 2)[inside]).all()
    assert (np.abs(wd)[~inside] == 6 * sc[~inside]).all()


def check_gemm(ns):
    x = pins.random_weights(12, 256, 9, "t4")
    rng = np.random.default_rng(10)
    a = pins.bf16_round(rng.standard_normal((3, 256)).astype(np.float32))
    bias = pins.bf16_round(rng.standard_normal(12).astype(np.float32))
    for wd in (ns.dequantize_mxfp4(*ns.quantize_mxfp4_f32(x)),
               ns.dequantize_nvfp4(*ns.quantize_nvfp4_f32(x))):
        wd = wd.astype(np.float64)
        y = ns.gemm_fp4(pins.to_bits(a), wd.astype(np.float32), pins.to_bits(bias)).astype(np.float64)
        ye = pins.exact_gemm(a.astype(np.float64), wd, bias.astype(np.float64))
        gamma = 257 * 2.0 ** -24 / (1 - 257 * 2.0 ** -24)
        mag = np.abs(a.astype(np.float64)) @ np.abs(wd).T + np.abs(bias.astype(np.float64))[None, :]
        assert (np.abs(y - ye) <= gamma * mag + 1e-45).all()
        ks = [0, 1, 31, 32, 255]
        oh = np.zeros((len(ks), 256), np.uint16)
        for m, k in enumerate(ks):
            oh[m, k] = 0x3F80
        yo = ns.gemm_fp4(oh, wd.astype(np.float32))
        for m, k in enumerate(ks):
            assert (yo[m] == wd[:, k]).all()


def small_weights():
    x = np.concatenate([pins.special_groups(8).reshape(4, 256),
                        pins.random_weights(4, 256, 11, "t4")])
    x[2, 40:48] = [0.25, -0.75, 1.25, 5.0, -2.5, 3.5, 1.75, 0.0]   # ties at scale 1 (amax 6)
    x[2, 32] = 6.0
    return x


def _all(ns):
    check_e2m1_format(ns)
    check_e4m3_format(ns)
    check_mx_exponent(ns)
    check_hand_examples(ns)
    x = small_weights()
    check_mx_exact(ns, x)
    check_nv_exact(ns, x)
    check_packing(ns)
    check_dequantize(ns, x)
    check_invariants(ns, np.concatenate([x, pins.random_weights(8, 256, 12, "normal")]))
    check_gemm(ns)


def test_formats():
    ns = real_ns()
    check_e2m1_format(ns)
    check_e4m3_format(ns)
    check_mx_exponent(ns)


def test_hand_examples():
    check_hand_examples(real_ns())


def test_quantize_exact():
    ns = real_ns()
    x = small_weights()
    check_mx_exact(ns, x)
    check_nv_exact(ns, x)


def test_nv_zero_tensor():
    packed, sc, g = f4.quantize_nvfp4_f32(np.zeros((2, 128), np.float32))
    assert g == np.float32(1.0) and not packed.any() and not sc.any()


def test_packing_dequantize_invariants():
    ns = real_ns()
    check_packing(ns)
    x = small_weights()
    check_dequantize(ns, x)
    check_invariants(ns, np.concatenate([x, pins.random_weights(8, 256, 12, "normal")]))


def test_gemm():
    check_gemm(real_ns())


# ---------------------------------------------------------------- mutants
def _e2m1_ties_away(x):
    a = np.abs(np.asarray(x, np.float32))
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    idx = np.zeros(a.shape, np.uint8)
    for i, m in enumerate(mids):
        idx = np.where(a >= m, np.uint8(i + 1), idx)
    neg = np.signbit(np.asarray(x, np.float32)) & (idx != 0)
    return (idx | (neg.astype(np.uint8) << 3)).astype(np.uint8)


def _e2m1_signed_zero(x):
    c = f4.e2m1_encode(x)
    return np.where(np.signbit(np.asarray(x, np.float32)), c | 8, c).astype(np.uint8)


def _mx_no_emax(amax):
    return np.clip(f4.mx_exponent(amax).astype(int) + 2, 0, 254).astype(np.uint8)


def _e4m3_bias8_decode(codes):
    return (f4.e4m3_decode(codes) * np.float32(0.5)).astype(np.float32)


def _pack_swapped(codes):
    c = np.asarray(codes, np.uint8)
    return (c[:, 1::2] | (c[:, 0::2] << 4)).astype(np.uint8)


def _nv_quant_variant(den=2688.0, block=16, one_step=False):
    def q(x, tensor_scale=None):
        x = np.ascontiguousarray(x, np.float32)
        n, k = x.shape
        am = np.float32(np.max(np.abs(x)))
        g = np.float32(1.0) if am == 0 else np.float32(am / np.float32(den))
        xb = x.reshape(n, k // block, block)
        amax = np.max(np.abs(xb), axis=2)
        if one_step:
            sb_code = f4.e4m3_encode((amax / np.float32(np.float32(6.0) * g)).astype(np.float32))
        else:
            sb_code = f4.e4m3_encode(((amax / np.float32(6.0)).astype(np.float32) / g).astype(np.float32))
        step = (f4.e4m3_decode(sb_code) * g).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            r = np.where(step[:, :, None] > 0, xb / step[:, :, None], 0).astype(np.float32)
        codes = f4.e2m1_encode(r).reshape(n, k)
        sb = np.repeat(sb_code, block // 16, axis=1)      # one code per 16 values
        return f4.pack_codes_fp4(codes), np.ascontiguousarray(sb.T), g
    return q


MUTANTS = {
    "e2m1_ties_away": dict(e2m1_encode=_e2m1_ties_away),
    "e2m1_signed_zero": dict(e2m1_encode=_e2m1_signed_zero),
    "mx_no_emax": dict(mx_exponent=_mx_no_emax),
    "e4m3_bias8": dict(e4m3_decode=_e4m3_bias8_decode),
    "nibble_order": dict(pack_codes_fp4=_pack_swapped),
    "nv_global_over_6": dict(quantize_nvfp4_f32=_nv_quant_variant(den=6.0)),
    "nv_block_32": dict(quantize_nvfp4_f32=_nv_quant_variant(block=32)),
    "nv_dequant_no_global": dict(dequantize_nvfp4=lambda p, s, g: f4.dequantize_nvfp4(p, s, 1.0)),
    "gemm_drop_bias": dict(gemm_fp4=lambda a, wd, b=None, rows=None: f4.gemm_fp4(a, wd, None, rows)),
}


def _mutant_ns(name):
    ns = real_ns()
    for k, v in MUTANTS[name].items():
        setattr(ns, k, v)
    # the quantizers call the module's helpers: route them through the namespace
    if any(k in MUTANTS[name] for k in ("e2m1_encode", "mx_exponent", "pack_codes_fp4")):
        def q_mx(x):
            x = np.ascontiguousarray(x, np.float32)
            n, k = x.shape
            xb = x.reshape(n, k // 32, 32)
            e = ns.mx_exponent(np.max(np.abs(xb), axis=2))
            scale = np.ldexp(np.float32(1.0), e.astype(np.int32) - 127).astype(np.float32)
            codes = ns.e2m1_encode(xb / scale[:, :, None]).reshape(n, k)
            return ns.pack_codes_fp4(codes), np.ascontiguousarray(e.T)
        ns.quantize_mxfp4_f32 = q_mx
    return ns


@pytest.mark.parametrize("name", list(MUTANTS))
def test_fp4_mutant_is_caught(name):
    with pytest.raises(AssertionError):
        _all(_mutant_ns(name))


def test_unmutated_copy_passes():
    _all(real_ns())
