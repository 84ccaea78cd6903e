"""The CPU oracle against facts that do not come from it (see pins.py)."""

import numpy as np
import pytest

import oracle
import pins


def test_hand_worked_examples():
    pins.check_hand_examples(oracle)


@pytest.mark.parametrize("dist,seed", [("normal", 0), ("t4", 1)])
def test_scales_exact_rational(dist, seed):
    pins.check_scales_exact(oracle, pins.random_weights(12, 512, seed, dist))


def test_scales_exact_rational_special_groups():
    pins.check_scales_exact(oracle, pins.special_groups(16).reshape(8, 256))


@pytest.mark.parametrize("dist,seed", [("normal", 2), ("t4", 3)])
def test_codes_brute_force(dist, seed):
    pins.check_codes_bruteforce(oracle, pins.random_weights(4, 256, seed, dist))


def test_codes_brute_force_special_groups():
    pins.check_codes_bruteforce(oracle, pins.special_groups(16).reshape(8, 256))


@pytest.mark.parametrize("dist,seed", [("normal", 4), ("t4", 5)])
def test_codes_locally_optimal_large(dist, seed):
    # 2M elements: enough that a reciprocal-multiply quantizer is caught
    pins.check_codes_local_optimal(oracle, pins.random_weights(1024, 2048, seed, dist))


def test_codes_locally_optimal_special_groups():
    pins.check_codes_local_optimal(oracle, pins.special_groups(32).reshape(8, 512))


@pytest.mark.parametrize("dist,seed", [("normal", 6), ("t4", 7)])
def test_invariants(dist, seed):
    pins.check_invariants(oracle, pins.random_weights(64, 1024, seed, dist))


def test_invariants_special_groups():
    pins.check_invariants(oracle, pins.special_groups(32).reshape(16, 256))


def test_dequantize():
    pins.check_dequantize(oracle, pins.random_weights(16, 384, 8, "t4"))
    pins.check_dequantize(oracle, pins.special_groups(16).reshape(4, 512))


def test_gemm_exact_bound():
    x = pins.random_weights(10, 256, 9)
    rng = np.random.default_rng(10)
    a = pins.bf16_round(rng.standard_normal((3, 256)).astype(np.float32))
    b = pins.bf16_round(rng.standard_normal(10).astype(np.float32))
    pins.check_gemm_exact_bound(oracle, pins.to_bits(a), pins.to_bits(x))
    pins.check_gemm_exact_bound(oracle, pins.to_bits(a), pins.to_bits(x), pins.to_bits(b))


def test_f16_widening_matches_format_definition():
    pins.check_f16_widening(oracle)


def test_gemm_f16_activations_exact_bound_and_one_hot():
    x = pins.random_weights(10, 256, 9)
    rng = np.random.default_rng(13)
    a = rng.standard_normal((3, 256)).astype(np.float16).view(np.uint16)
    b = rng.standard_normal(10).astype(np.float16).view(np.uint16)
    pins.check_gemm_exact_bound(oracle, a, pins.to_bits(x), act="f16")
    pins.check_gemm_exact_bound(oracle, a, pins.to_bits(x), b, act="f16")
    pins.check_gemm_one_hot(oracle, pins.to_bits(pins.random_weights(256, 256, 11, "t4")), act="f16")


def test_gemm_one_hot_square():
    # N == K so that a transposed operand would not raise a shape error
    pins.check_gemm_one_hot(oracle, pins.to_bits(pins.random_weights(256, 256, 11, "t4")))


def test_gemm_integer_exact():
    pins.check_gemm_integer_exact(oracle)


def test_pack_unpack_roundtrip():
    rng = np.random.default_rng(12)
    c = rng.integers(-8, 8, size=(5, 256)).astype(np.int8)
    p = oracle.pack_codes(c)
    assert p.shape == (5, 128) and p.dtype == np.uint8
    assert (oracle.unpack_codes(p) == c).all()
    # byte layout: low nibble is the even index
    assert oracle.pack_codes(np.array([[1, -2]], np.int8))[0, 0] == 0xE1


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.quantize_f32(np.zeros((2, 100), np.float32))
    with pytest.raises(ValueError):
        oracle.quantize_f32(np.zeros((2, 256), np.float32), group=64)


def test_tile_layout_closed_form():
    # every byte lands at the offset the layout formula gives, by brute force
    rng = np.random.default_rng(13)
    N, K = 136, 384
    p = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    t = oracle.to_tile_layout(p)
    assert t.size == oracle.tiled_bytes(N, K) == 256 * K // 2
    G = K // 128
    for n in range(N):
        for j in range(K // 2):
            off = ((n // 128) * G + j // 64) * 8192 + (n % 128) * 64 + j % 64
            assert t[off] == p[n, j]
    # padding rows are zero, and the inverse recovers the row-major bytes
    pad = np.ones(t.size, bool)
    for n in range(N):
        for g in range(G):
            base = ((n // 128) * G + g) * 8192 + (n % 128) * 64
            pad[base:base + 64] = False
    assert not t[pad].any()
    assert (oracle.from_tile_layout(t, N, K) == p).all()


def test_scale_overflow_follows_ieee():
    # Outside the method's preconditions (|w| small enough that amax / 7 fits
    # fp16), the oracle's steps still have one IEEE reading, worked by hand:
    # amax = 2^19 = 524288 (bf16-exact); fl32(524288 / 7) = 74898.28...,
    # above fp16's largest finite value 65504 and above the rounding boundary
    # 65520, so fp16 round-to-nearest gives +inf (0x7C00), which is not 0, so
    # the zero rule does not apply; every x / inf is +-0 and rounds to code 0.
    x = np.zeros((1, 128), dtype=np.float32)
    x[0, :3] = [524288.0, 3.0, -3.0]
    with np.errstate(over="ignore"):
        packed, sbits = oracle.quantize_f32(x)
    assert int(sbits[0, 0]) == 0x7C00
    assert not oracle.unpack_codes(packed).any()
    assert not packed.any()
