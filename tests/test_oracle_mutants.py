"""Plants plausible mistakes in copies of the oracle (on the CPU) and checks
that at least one pin fails for each: the pins are strong enough to catch a
dropped term, a wrong sign or index, a transposed operand, the wrong
rounding or the wrong packing."""

import types

import numpy as np
import pytest

import oracle
import pins
from oracle import w4a16_oracle as base


def _namespace(**overrides):
    ns = types.SimpleNamespace(
        quantize_f32=base.quantize_f32,
        quantize=None,
        dequantize=base.dequantize,
        gemm=base.gemm,
        unpack_codes=base.unpack_codes,
    )
    for k, v in overrides.items():
        setattr(ns, k, v)
    if "quantize" not in overrides:
        ns.quantize = lambda w_bits, group=128: ns.quantize_f32(base.bf16_bits_to_f32(w_bits), group)
    return ns


def _quantize_variant(*, recip=False, fp32_scale_codes=False, zero_rule_before=False,
                      ties_away=False, no_abs=False, nibble_swap=False, scales_nk=False,
                      div_by=7.0):
    def q(x, group=128):
        x = np.ascontiguousarray(x, dtype=np.float32)
        N, K = x.shape
        G = K // group
        xg = x.reshape(N, G, group)
        amax = np.max(xg if no_abs else np.abs(xg), axis=2)
        s32 = amax / np.float32(div_by)
        if zero_rule_before:
            s32 = np.where(amax == 0, np.float32(1.0), s32)
            s16 = s32.astype(np.float16)
        else:
            s16 = s32.astype(np.float16)
            s16 = np.where(s16 == 0, np.float16(1.0), s16)
        sdiv = s32 if fp32_scale_codes else s16.astype(np.float32)
        with np.errstate(all="ignore"):
            if recip:
                ratio = xg * (np.float32(1.0) / sdiv)[:, :, None]
            else:
                ratio = xg / sdiv[:, :, None]
            r = np.floor(ratio + np.float32(0.5)) if ties_away else np.rint(ratio)
            r = np.nan_to_num(r, nan=0.0)
        codes = np.clip(r, -8, 7).astype(np.int8).reshape(N, K)
        c = codes.astype(np.int16)
        lo = (c[:, 0::2] & 0xF).astype(np.uint8)
        hi = (c[:, 1::2] & 0xF).astype(np.uint8)
        packed = (hi | (lo << 4)) if nibble_swap else (lo | (hi << 4))
        sb = s16 if scales_nk else s16.T
        return packed.astype(np.uint8), np.ascontiguousarray(sb).view(np.uint16)
    return q


def _gemm_variant(*, transpose=False, drop_bias=False, neg=False, group_shift=False,
                  f16_as_bf16=False):
    def g(a_bits, packed, scale_bits, bias_bits=None, group=128, rows=None, act="bf16"):
        widen = (lambda b: base.act_bits_to_f32(b, "bf16" if f16_as_bf16 else act))
        a = widen(a_bits)
        if group_shift:
            codes = base.unpack_codes(packed).astype(np.float32)
            s = base.scales_f32(scale_bits)
            wd = codes * np.repeat(np.roll(s, 1, axis=0).T, group, axis=1)
        else:
            wd = base.dequantize(packed, scale_bits, group)
        y = a @ (wd if transpose else wd.T)
        if neg:
            y = -y
        if bias_bits is not None and not drop_bias:
            y = y + widen(bias_bits)[None, :]
        return y.astype(np.float32)
    return g


def _all_quantize_pins(ns):
    pins.check_hand_examples(ns)
    pins.check_scales_exact(ns, pins.special_groups(16).reshape(8, 256))
    pins.check_scales_exact(ns, pins.random_weights(6, 512, 0, "t4"))
    pins.check_codes_bruteforce(ns, pins.special_groups(16).reshape(8, 256))
    pins.check_codes_local_optimal(ns, pins.random_weights(1024, 2048, 4, "normal"))
    pins.check_invariants(ns, pins.special_groups(32).reshape(16, 256))
    pins.check_dequantize(ns, pins.random_weights(16, 384, 8, "t4"))


def _all_gemm_pins(ns):
    x = pins.random_weights(10, 256, 9)
    rng = np.random.default_rng(10)
    a = pins.bf16_round(rng.standard_normal((3, 256)).astype(np.float32))
    b = pins.bf16_round(rng.standard_normal(10).astype(np.float32))
    pins.check_hand_examples(ns)
    pins.check_gemm_exact_bound(ns, pins.to_bits(a), pins.to_bits(x), pins.to_bits(b))
    pins.check_gemm_one_hot(ns, pins.to_bits(pins.random_weights(256, 256, 11, "t4")))
    pins.check_gemm_integer_exact(ns)
    # fp16 activations
    a16 = rng.standard_normal((3, 256)).astype(np.float16).view(np.uint16)
    b16 = rng.standard_normal(10).astype(np.float16).view(np.uint16)
    pins.check_gemm_exact_bound(ns, a16, pins.to_bits(x), b16, act="f16")
    pins.check_gemm_one_hot(ns, pins.to_bits(pins.random_weights(256, 256, 12, "t4")), act="f16")


def test_unmutated_copy_passes():
    ns = _namespace(quantize_f32=_quantize_variant(), gemm=_gemm_variant())
    _all_quantize_pins(ns)
    _all_gemm_pins(ns)


@pytest.mark.parametrize("mutation", [
    "recip", "fp32_scale_codes", "zero_rule_before", "ties_away", "no_abs",
    "nibble_swap", "scales_nk", "div_by_8",
])
def test_quantize_mutant_is_caught(mutation):
    kw = {"div_by": 8.0} if mutation == "div_by_8" else {mutation: True}
    ns = _namespace(quantize_f32=_quantize_variant(**kw))
    with pytest.raises((AssertionError, ValueError, IndexError)):
        _all_quantize_pins(ns)


@pytest.mark.parametrize("mutation", ["transpose", "drop_bias", "neg", "group_shift", "f16_as_bf16"])
def test_gemm_mutant_is_caught(mutation):
    ns = _namespace(gemm=_gemm_variant(**{mutation: True}))
    with pytest.raises((AssertionError, ValueError)):
        _all_gemm_pins(ns)


def test_real_oracle_is_what_the_pins_saw():
    # guard: the namespace used above wraps the very functions the package exports
    assert oracle.quantize_f32 is base.quantize_f32 and oracle.gemm is base.gemm
