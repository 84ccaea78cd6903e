"""W4A16 GEMM with FP16 activations (A, bias and Y in fp16) on the GPU
against the oracle's FP32 GEMM on identical packed operands:
|y - y_ref| <= 1e-2 |y_ref| + 1e-2 rms(y_ref) element by element."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bits, check_gemm_close
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu

SHAPES = [
    synthetic.Case("tiny", 16, 256, 512, 0),
    synthetic.Case("m1_ragged_n", 1, 264, 384, 11, bias=True),
    synthetic.Case("m50_ragged", 50, 520, 640, 12, "t4", bias=True),
    synthetic.Case("m300_multi_tile", 300, 384, 1024, 14, bias=True),
    # the row-block kernel's fp16 MMAs with several activation columns: teams
    # (2056 rows, ragged) and a cluster K split (few rows, long K)
    synthetic.Case("m7_n2056", 7, 2056, 2048, 19, bias=True),
    synthetic.Case("m3_long_k", 3, 264, 16384, 20, "t4"),
]


def make_operands(w4, case):
    W, A, b = synthetic.draw(case, act="f16")
    packed, scales = w4.w4a16_quantize(W.cuda())
    return W, A, b, packed, scales


def reference(A, packed, scales, b, rows=None):
    s = scales.cpu().view(torch.int16).numpy().view(np.uint16)
    K, N = s.shape[0] * 128, s.shape[1]
    p = oracle.from_tile_layout(packed.cpu().numpy(), N, K)
    return oracle.gemm(bits(A), p, s, None if b is None else bits(b), rows=rows, act="f16")


@pytest.mark.parametrize("case", SHAPES, ids=[c.name for c in SHAPES])
def test_every_variant_f16(w4, case):
    W, A, b, packed, scales = make_operands(w4, case)
    y_ref = reference(A, packed, scales, b)
    Ad = A.cuda()
    bd = None if b is None else b.cuda()
    for v in range(w4.w4a16_variant_count()):
        if not w4.w4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        Y = w4.w4a16_gemm(Ad, packed, scales, bias=bd, variant=v)
        assert Y.dtype == torch.float16
        assert w4.w4a16_get_device_error() == w4.W4A16_OK
        check_gemm_close(Y, y_ref, what=w4.w4a16_variant_name(v) + " f16")


def test_long_pipelines_f16(w4):
    # 128 units per tile: every variant's stage rings wrap many times
    case = synthetic.Case("m200_k16384", 200, 256, 16384, 17, bias=True)
    W, A, b, packed, scales = make_operands(w4, case)
    y_ref = reference(A, packed, scales, b)
    Ad, bd = A.cuda(), b.cuda()
    for v in range(w4.w4a16_variant_count()):
        if not w4.w4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        Y = w4.w4a16_gemm(Ad, packed, scales, bias=bd, variant=v)
        assert w4.w4a16_get_device_error() == w4.W4A16_OK
        check_gemm_close(Y, y_ref, what=w4.w4a16_variant_name(v) + " f16")


def test_integer_exact_f16(w4):
    # power-of-two scales and small-integer activations: every product and
    # partial sum is exact in fp32, so every variant returns the exact sum
    # rounded once to fp16
    rng = np.random.default_rng(32)
    M, N, K = 40, 256, 512
    codes = rng.integers(-3, 4, size=(N, K))
    codes[:, ::128] = 7
    e = rng.integers(-3, 0, size=(N, K // 128))
    x = (codes * np.repeat(2.0 ** e, 128, axis=1)).astype(np.float32)
    a = rng.integers(-1, 2, size=(M, K)).astype(np.float32)
    W = synthetic.to_bf16(x).cuda()
    A = synthetic.to_f16(a)
    packed, scales = w4.w4a16_quantize(W)
    exact = a.astype(np.float64) @ x.astype(np.float64).T
    assert np.all(exact == np.round(exact * 8) / 8) and np.abs(exact).max() < 4096
    expected = bits(synthetic.to_f16(exact.astype(np.float32)))
    for v in range(w4.w4a16_variant_count()):
        if not w4.w4a16_variant_eligible(v, M, N, K):
            continue
        Y = w4.w4a16_gemm(A.cuda(), packed, scales, variant=v)
        torch.cuda.synchronize()
        assert np.array_equal(bits(Y), expected), w4.w4a16_variant_name(v)


WORKLOAD_CASES = synthetic.WORKLOADS["expert_m50"] + [synthetic.WORKLOADS["sweep"][8]]


@pytest.mark.parametrize("case", WORKLOAD_CASES, ids=[c.name for c in WORKLOAD_CASES])
def test_workloads_f16_default_variant(w4, case):
    W, A, b, packed, scales = make_operands(w4, case)
    Y = w4.w4a16_gemm(A.cuda(), packed, scales)
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
    check_gemm_close(Y, reference(A, packed, scales, b), what=case.name + " f16")


@pytest.mark.parametrize("M", [1, 3, 5, 12, 16])
def test_integer_exact_f16_small_m(w4, M):
    # as test_integer_exact_f16 at M = 1, 3, 5, 12, 16: the streaming
    # variants for M <= 16 (the row-block kernel's fp16 MMAs on 1032 + q and
    # 1152 + 16 q, less their offsets times the activation sums, the second
    # class scaled by 1/16; two column tiles above M = 8) return the exact
    # sum rounded once to fp16
    rng = np.random.default_rng(33 + M)
    N, K = 264, 1024
    codes = rng.integers(-3, 4, size=(N, K))
    codes[:, ::128] = 7
    e = rng.integers(-3, 0, size=(N, K // 128))
    x = (codes * np.repeat(2.0 ** e, 128, axis=1)).astype(np.float32)
    a = rng.integers(-2, 3, size=(M, K)).astype(np.float32)
    W = synthetic.to_bf16(x).cuda()
    A = synthetic.to_f16(a)
    packed, scales = w4.w4a16_quantize(W)
    exact = a.astype(np.float64) @ x.astype(np.float64).T
    assert np.all(exact == np.round(exact * 8) / 8) and np.abs(exact).max() < 4096
    expected = bits(synthetic.to_f16(exact.astype(np.float32)))
    ran = 0
    for v in range(w4.w4a16_variant_count()):
        name = w4.w4a16_variant_name(v)
        if not name.startswith(("simt_", "rb_")) or not w4.w4a16_variant_eligible(v, M, N, K):
            continue
        Y = w4.w4a16_gemm(A.cuda(), packed, scales, variant=v)
        torch.cuda.synchronize()
        assert np.array_equal(bits(Y), expected), name
        ran += 1
    assert ran >= (4 if M <= 2 else 2 if M <= 8 else 1)
