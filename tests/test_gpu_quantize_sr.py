"""Stochastic-rounding quantize on the GPU against the oracle: codes and
scales bit-exact for the same seed ("Piper Kernels", section "Stochastic
quantization"; draws from Philox4x32-10 by logical element offset)."""

import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_helpers import bits, check_quantize_exact
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu

SEEDS = [0, 1, (1 << 64) - 1, 0x123456789ABCDEF0]


def check_sr_exact(W_cpu, seed, packed, scales, row0=0, rows=None):
    """Codes and scales of rows row0 .. row0 + rows - 1 (whole 128-row tiles)
    against the oracle."""
    wb = bits(W_cpu)
    N, K = wb.shape
    rows = N if rows is None else rows
    p_rm, s_ref = oracle.quantize_sr(wb[row0:row0 + rows], seed, row0=row0)
    G = K // 128
    p = packed.cpu().numpy().reshape(-1)
    if row0 == 0 and rows == N:
        p_ref = oracle.to_tile_layout(p_rm)
        got = p
    else:
        assert row0 % 128 == 0 and rows % 128 == 0
        t0, t1 = row0 // 128, (row0 + rows) // 128
        got = p[t0 * G * 8192:t1 * G * 8192]
        p_ref = oracle.to_tile_layout(p_rm)
    s = scales.cpu().view(torch.int16).numpy().view(np.uint16)[:, row0:row0 + rows]
    assert np.array_equal(s, s_ref), "scale mismatch"
    bad = np.argwhere(got != p_ref)
    assert bad.size == 0, f"seed {seed}: {len(bad)} packed-byte mismatches, first {bad[:4].tolist()}"


@pytest.mark.parametrize("seed", SEEDS)
def test_tiny_and_special_groups(w4, seed):
    for x in (pins.special_groups(64).reshape(16, 512), pins.random_weights(24, 384, 3, "t4")):
        W = synthetic.to_bf16(x)
        packed, scales = w4.w4a16_quantize(W.cuda(), seed=seed)
        torch.cuda.synchronize()
        check_sr_exact(W, seed, packed, scales)


def test_ties_and_exact_hits(w4):
    # power-of-two scales: exact multiples are never perturbed, half-integers
    # go either way
    rng = np.random.default_rng(5)
    N, K = 64, 1024
    e = rng.integers(-6, 3, size=(N, K // 128))
    k = rng.integers(-15, 15, size=(N, K)).astype(np.float32) / 2
    k[:, ::128] = 7.0
    x = (k * np.repeat(2.0 ** e, 128, axis=1)).astype(np.float32)
    W = synthetic.to_bf16(x)
    for seed in (3, 4):
        packed, scales = w4.w4a16_quantize(W.cuda(), seed=seed)
        torch.cuda.synchronize()
        check_sr_exact(W, seed, packed, scales)


@pytest.mark.parametrize("N,K", [(8, 128), (136, 384), (1000, 1152)])
def test_ragged_shapes(w4, N, K):
    W = synthetic.draw_weight_only(N + K, N, K, "t4")
    packed, scales = w4.w4a16_quantize(W.cuda(), seed=N * K)
    torch.cuda.synchronize()
    check_sr_exact(W, N * K, packed, scales)


def test_scales_are_rtn_and_seeds(w4):
    W = synthetic.draw_weight_only(9, 512, 2048).cuda()
    p_rtn, s_rtn = w4.w4a16_quantize(W)
    p1, s1 = w4.w4a16_quantize(W, seed=11)
    p2, s2 = w4.w4a16_quantize(W, seed=11)
    p3, s3 = w4.w4a16_quantize(W, seed=12)
    torch.cuda.synchronize()
    assert torch.equal(s1, s_rtn) and torch.equal(s3, s_rtn)
    assert torch.equal(p1, p2) and not torch.equal(p1, p3) and not torch.equal(p1, p_rtn)
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


@pytest.mark.parametrize("case", synthetic.WORKLOADS["expert_m50"], ids=lambda c: f"{c.N}x{c.K}")
def test_expert_weights_full(w4, case):
    W = synthetic.draw_weight_only(case.seed, case.N, case.K)
    packed, scales = w4.w4a16_quantize(W.cuda(), seed=case.seed)
    torch.cuda.synchronize()
    check_sr_exact(W, case.seed, packed, scales)


def test_large_weight_sampled_tiles(w4):
    # the 8192 x 8192 weight of the compute-bound case, in the launch the
    # bench times; compared on the first and last 128-row storage tiles
    c = synthetic.WORKLOADS["large"][0]
    W = synthetic.draw_weight_only(c.seed, c.N, c.K)
    seed = 0xFEEDFACE
    packed, scales = w4.w4a16_quantize(W.cuda(), seed=seed)
    torch.cuda.synchronize()
    for row0 in (0, c.N - 128):
        check_sr_exact(W, seed, packed, scales, row0=row0, rows=128)
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


def test_rtn_unchanged(w4):
    # the round-to-nearest path is untouched by the new mode
    W = synthetic.draw_weight_only(21, 256, 1024, "t4")
    packed, scales = w4.w4a16_quantize(W.cuda())
    torch.cuda.synchronize()
    check_quantize_exact(W, packed, scales)


def test_bad_seed_rejected(w4):
    W = torch.zeros(8, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        w4.w4a16_quantize(W, seed=-1)
