"""RTN quantize/pack on the GPU against the oracle: codes and scales bit-exact."""

import numpy as np
import pytest
import torch

import pins
from gpu_helpers import check_quantize_exact, guarded
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu


def run_quantize(w4, W_cpu):
    W = W_cpu.cuda()
    packed, scales = w4.w4a16_quantize(W)
    torch.cuda.synchronize()
    return packed, scales


def test_tiny(w4):
    W, _, _ = synthetic.draw(synthetic.TINY[0])
    packed, scales = run_quantize(w4, W)
    check_quantize_exact(W, packed, scales)


def test_special_groups(w4):
    # zero groups, spikes, exact ties, subnormal and underflowing scales, large values
    x = pins.special_groups(64).reshape(16, 512)
    W = synthetic.to_bf16(x)
    packed, scales = run_quantize(w4, W)
    check_quantize_exact(W, packed, scales)


def test_ties_everywhere(w4):
    # every element an exact half-integer multiple of its (power-of-two) scale
    rng = np.random.default_rng(5)
    N, K = 64, 1024
    e = rng.integers(-6, 3, size=(N, K // 128))
    k = rng.integers(-15, 15, size=(N, K)).astype(np.float32) + 0.5
    k[:, ::128] = 7.0
    x = (k * np.repeat(2.0 ** e, 128, axis=1)).astype(np.float32)
    W = synthetic.to_bf16(x)
    packed, scales = run_quantize(w4, W)
    check_quantize_exact(W, packed, scales)


@pytest.mark.parametrize("N,K", [(8, 128), (24, 256), (136, 384), (1000, 1152)])
def test_small_and_ragged_shapes(w4, N, K):
    W = synthetic.draw_weight_only(N + K, N, K, "t4")
    packed, scales = run_quantize(w4, W)
    check_quantize_exact(W, packed, scales)


def test_outputs_stay_in_bounds(w4):
    N, K = 40, 640
    W = synthetic.draw_weight_only(3, N, K).cuda()
    packed, p_ok = guarded((w4.w4a16_packed_bytes(N, K),), torch.uint8, W.device, 0xA5)
    scales, s_ok = guarded((K // 128, N), torch.float16, W.device, 0x7E00)
    w4.w4a16_quantize(W, packed=packed, scales=scales)
    torch.cuda.synchronize()
    assert p_ok() and s_ok()
    check_quantize_exact(W.cpu(), packed, scales)


ALL_WEIGHTS = sorted({(c.N, c.K, c.seed, c.wdist): c for cfg in synthetic.WORKLOADS.values()
                      for c in cfg}.values(), key=lambda c: c.N * c.K)


@pytest.mark.parametrize("case", ALL_WEIGHTS, ids=[c.name for c in ALL_WEIGHTS])
def test_workload_weights_full_size(w4, case):
    W = synthetic.draw_weight_only(case.seed, case.N, case.K, case.wdist)
    packed, scales = run_quantize(w4, W)
    check_quantize_exact(W, packed, scales)


def test_scale_overflow_matches_oracle(w4):
    # amax / 7 above fp16's range (outside the preconditions): the kernel
    # takes the IEEE division for an infinite scale, as the oracle does
    # (scale 0x7C00, codes 0); the other groups are unaffected
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((16, 512)) * 0.02).astype(np.float32)
    x[3, 5] = 524288.0          # group 0 of row 3
    x[7, 300] = -1048576.0      # group 2 of row 7
    x[9, 128:256] = 0.0
    x[9, 130] = 600000.0        # group 1 of row 9
    W = synthetic.to_bf16(x)
    packed, scales = run_quantize(w4, W)
    s = scales.cpu().view(torch.int16).numpy().view(np.uint16)
    assert s[0, 3] == 0x7C00 and s[2, 7] == 0x7C00 and s[1, 9] == 0x7C00
    with np.errstate(over="ignore"):
        check_quantize_exact(W, packed, scales)
