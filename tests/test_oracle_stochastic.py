"""Pins of the stochastic-rounding quantize oracle (CPU only).

"Piper Kernels", section "Stochastic quantization": one of the two adjacent
codes is chosen with probability proportional to the distance, so the
expected value is the unrounded one; values outside the code range and exact
hits are never perturbed; draws come from a seeded generator indexed by the
logical element offset.  Section "ConvRot INT8" (add_/addmm_): the seeded
selection keeps the deterministic scales.  The generator is Philox4x32-10
(Salmon et al., "Parallel random numbers: as easy as 1, 2, 3").

Every check below takes a namespace of oracle functions, so that
test_oracle_mutants_stochastic can run the same pins on planted mistakes."""

import os
import types

import numpy as np
import pytest

import oracle
from oracle import stochastic as sr
import pins

HERE = os.path.dirname(os.path.abspath(__file__))


def real_ns():
    return types.SimpleNamespace(philox4x32_10=sr.philox4x32_10, uniform_at=sr.uniform_at,
                                 uniform_block=sr.uniform_block,
                                 stochastic_code=sr.stochastic_code,
                                 quantize_sr_f32=sr.quantize_sr_f32)


def load_kat():
    rows = []
    with open(os.path.join(HERE, "golden", "philox4x32_10_kat.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            ctr, key, out = (tuple(int(w, 16) for w in part.split()) for part in line.split("|"))
            rows.append((ctr, key, out))
    return rows


# ------------------------------------------------------------------- pins
def check_philox_kat(ns):
    rows = load_kat()
    assert len(rows) == 3
    for ctr, key, out in rows:
        got = ns.philox4x32_10([np.uint32(c) for c in ctr], [np.uint32(k) for k in key])
        assert tuple(int(g) for g in got) == out, (ctr, key)


def check_uniform_definition(ns):
    # reading SR3 on a hand-listed example: K = 8, elements (0,0), (0,5), (1,2)
    # have offsets 0, 5, 10: counters 0, 1, 2 and words 0, 1, 2
    seed = 0x0123456789ABCDEF
    key = (np.uint32(seed & 0xFFFFFFFF), np.uint32(seed >> 32))
    z = np.uint32(0)
    want = []
    for c, w in ((0, 0), (1, 1), (2, 2)):
        words = ns.philox4x32_10([np.uint32(c), z, z, z], key)
        want.append(np.float32(int(words[w]) >> 8) * np.float32(2.0 ** -24))
    u = ns.uniform_block(seed, 8, slice(0, 2), slice(0, 8))
    assert u[0, 0] == want[0] and u[0, 5] == want[1] and u[1, 2] == want[2]


def check_uniform_geometry(ns):
    # the draw depends on (seed, logical offset) only: any block of the
    # logical weight sees the same values as the whole
    seed = 77
    full = ns.uniform_block(seed, 256, slice(0, 40), slice(0, 256))
    part = ns.uniform_block(seed, 256, slice(13, 29), slice(37, 141))
    assert np.array_equal(part, full[13:29, 37:141])
    assert np.array_equal(ns.uniform_at(seed, np.array([13 * 256 + 37])), full[13:14, 37])


def check_uniform_values(ns):
    u = ns.uniform_block(2024, 4096, slice(0, 256), slice(0, 4096)).ravel()
    assert u.dtype == np.float32 and u.min() >= 0.0 and u.max() < 1.0
    assert np.all(u * np.float32(2.0 ** 24) == np.floor(u * np.float32(2.0 ** 24)))
    n = u.size
    # mean 1/2 and variance 1/12 of U[0, 1), within 6 standard errors
    assert abs(u.mean() - 0.5) < 6 * np.sqrt(1 / 12 / n)
    assert abs(u.var() - 1 / 12) < 6 * np.sqrt(1 / 180 / n)
    # 16 equal bins, chi-square with 15 degrees of freedom well inside its tail
    counts = np.bincount((u * 16).astype(np.int64), minlength=16)
    chi2 = ((counts - n / 16) ** 2 / (n / 16)).sum()
    assert chi2 < 60.0
    # different seeds give different streams; the high key word matters
    a = ns.uniform_block(1, 64, slice(0, 1), slice(0, 64))
    b = ns.uniform_block(1 + (1 << 32), 64, slice(0, 1), slice(0, 64))
    assert not np.array_equal(a, b)


def check_code_rule_bruteforce(ns):
    # expected value over a complete grid of draws u = i / 4096: for a
    # fraction that is a multiple of 1/4096 the mean code equals r exactly
    u = (np.arange(4096, dtype=np.float32) / np.float32(4096.0))
    for r in (2.25, -3.75, -7.5, 6.0009765625, 0.5, -0.25, 1.0 - 1.0 / 4096):
        q = ns.stochastic_code(np.full(4096, r, np.float32), u).astype(np.float64)
        assert set(np.unique(q)) <= {np.floor(r), np.floor(r) + 1}, r
        assert q.mean() == r, (r, q.mean())
    # exact hits: never perturbed
    for r in (-8.0, -3.0, 0.0, 5.0, 7.0):
        q = ns.stochastic_code(np.full(4096, r, np.float32), u)
        assert np.all(q == r), r
    # outside the code range: the deterministic (clamped nearest) code
    for r, want in ((7.25, 7), (7.5, 7), (7.75, 7), (-8.25, -8), (-9.5, -8), (100.0, 7)):
        q = ns.stochastic_code(np.full(4096, r, np.float32), u)
        assert np.all(q == want), r
    # u = 0 rounds up any positive fraction; the largest draw rounds up
    # exactly the fractions above it
    top = np.float32(1.0 - 2.0 ** -24)
    assert ns.stochastic_code(np.float32([2.125]), np.float32([0.0]))[0] == 3
    assert ns.stochastic_code(np.float32([2.125]), np.float32([top]))[0] == 2


def _ratio_weights(ratio, rows, group=128):
    # rows of groups whose first element is 7 (scale exactly 1) and whose
    # other elements are `ratio`, so x / s = ratio exactly
    x = np.full((rows, group), np.float32(ratio), np.float32)
    x[:, 0] = 7.0
    return x


def check_unbiased(ns):
    # frequency of rounding up = fractional part, within 6 standard errors,
    # for several seeds and fractions
    for ratio in (2.25, -5.625, 0.875):
        frac = ratio - np.floor(ratio)
        x = _ratio_weights(ratio, 512)
        for seed in (0, 1, 0xFFFFFFFFFFFFFFFF):
            packed, _ = ns.quantize_sr_f32(x, seed)
            codes = oracle.unpack_codes(packed)[:, 1:].astype(np.float64)
            up = (codes == np.floor(ratio) + 1).mean()
            n = codes.size
            assert np.all((codes == np.floor(ratio)) | (codes == np.floor(ratio) + 1))
            assert abs(up - frac) < 6 * np.sqrt(frac * (1 - frac) / n), (ratio, seed, up)


def check_against_rtn(ns):
    # scales are the round-to-nearest scales; every code is one of the two
    # integers adjacent to the exact ratio (either one when the ratio is
    # within fp32 rounding of an integer); outside [-8, 7] the RTN code
    x = np.concatenate([pins.random_weights(64, 512, 41, "t4"),
                        pins.special_groups(16).reshape(4, 512)])
    for seed in (5, 6):
        packed, sbits = ns.quantize_sr_f32(x, seed)
        rp, rs = oracle.quantize_f32(x)
        assert np.array_equal(sbits, rs)
        s = np.repeat(oracle.scales_f32(rs).T.astype(np.float64), 128, axis=1)
        exact = x.astype(np.float64) / s
        q = oracle.unpack_codes(packed).astype(np.float64)
        q_rtn = oracle.unpack_codes(rp).astype(np.float64)
        inside = (exact >= -8) & (exact <= 7)
        near_int = np.abs(exact - np.rint(exact)) < 1e-6
        lo, hi = np.floor(exact), np.ceil(exact)
        ok = (q == lo) | (q == hi) | (near_int & (np.abs(q - np.rint(exact)) <= 1))
        assert np.all(ok[inside])
        assert np.array_equal(q[~inside & ~near_int], q_rtn[~inside & ~near_int])
        # exact multiples of the scale are never perturbed
        assert np.array_equal(q[near_int & inside], q_rtn[near_int & inside])


def check_seeds(ns):
    x = pins.random_weights(32, 256, 43, "normal")
    a = ns.quantize_sr_f32(x, 9)
    b = ns.quantize_sr_f32(x, 9)
    c = ns.quantize_sr_f32(x, 10)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert not np.array_equal(a[0], c[0]) and np.array_equal(a[1], c[1])


ALL_PINS = [check_philox_kat, check_uniform_definition, check_uniform_geometry, check_uniform_values,
            check_code_rule_bruteforce, check_unbiased, check_against_rtn, check_seeds]


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_stochastic_oracle_pin(pin):
    pin(real_ns())


def test_seed_range():
    with pytest.raises(ValueError):
        sr.seed_key(-1)
    with pytest.raises(ValueError):
        sr.seed_key(1 << 64)
