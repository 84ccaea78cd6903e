"""INT8 weight-only scheme (W8A16) on the GPU against the oracle: quantize
bit-exact; GEMM within |y - y_ref| <= 1e-2 |y_ref| + 1e-2 rms(y_ref) on
identical packed operands, bit-exact on integer-exact inputs
("Kernel dispatch and Humming quantization in PhyAI", section "Choose
precision by layer and hardware": INT8 is one of the Humming weight schemes)."""

import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_helpers import bits, check_gemm_close, guarded
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC1


def check_q8_exact(W_cpu, packed, scales, row0=0, rows=None):
    wb = bits(W_cpu)
    N, K = wb.shape
    rows = N if rows is None else rows
    codes, s_ref = oracle.quantize8(wb[row0:row0 + rows])
    p_ref = oracle.to_tile_layout8(codes)
    p = packed.cpu().numpy().reshape(-1)
    if not (row0 == 0 and rows == N):
        G = K // 128
        p = p[(row0 // 128) * G * 16384:((row0 + rows) // 128) * G * 16384]
    s = scales.cpu().view(torch.int16).numpy().view(np.uint16)[:, row0:row0 + rows]
    assert np.array_equal(s, s_ref), "scale mismatch"
    bad = np.argwhere(p != p_ref)
    assert bad.size == 0, f"{len(bad)} code-byte mismatches, first {bad[:4].tolist()}"


def w8_variants(w4):
    return list(range(w4.lib().w8a16_variant_count()))


def vname(w4, v):
    return w4.lib().w8a16_variant_name(v).decode()


def test_quantize_special_and_ragged(w4):
    for x in (pins.special_groups(64).reshape(16, 512), pins.random_weights(136, 384, 5, "t4"),
              pins.random_weights(1000, 1152, 6, "normal")):
        W = synthetic.to_bf16(x)
        packed, scales = w4.w8a16_quantize(W.cuda())
        torch.cuda.synchronize()
        check_q8_exact(W, packed, scales)


def test_quantize_ties(w4):
    rng = np.random.default_rng(8)
    N, K = 64, 1024
    e = rng.integers(-6, 2, size=(N, K // 128))
    k = rng.integers(-250, 250, size=(N, K)).astype(np.float32) / 2
    k[:, ::128] = 127.0
    W = synthetic.to_bf16((k * np.repeat(2.0 ** e, 128, axis=1)).astype(np.float32))
    packed, scales = w4.w8a16_quantize(W.cuda())
    torch.cuda.synchronize()
    check_q8_exact(W, packed, scales)


def test_quantize_large_weight_sampled(w4):
    c = synthetic.WORKLOADS["large"][0]
    W = synthetic.draw_weight_only(c.seed, c.N, c.K)
    packed, scales = w4.w8a16_quantize(W.cuda())
    torch.cuda.synchronize()
    for row0 in (0, c.N - 128):
        check_q8_exact(W, packed, scales, row0=row0, rows=128)


def _reference(A, packed, scales, b, rows=None):
    s = scales.cpu().view(torch.int16).numpy().view(np.uint16)
    K, N = s.shape[0] * 128, s.shape[1]
    codes = oracle.from_tile_layout8(packed.cpu().numpy(), N, K)
    return oracle.gemm8(bits(A), codes, s, None if b is None else bits(b), rows=rows)


SHAPES = [
    synthetic.Case("tiny", 16, 256, 512, 0),
    synthetic.Case("m1_ragged_n", 1, 264, 384, 11, bias=True),
    synthetic.Case("m50_ragged", 50, 520, 640, 12, "t4", bias=True),
    synthetic.Case("m129", 129, 256, 256, 13),
    synthetic.Case("m300_multi_tile", 300, 384, 1024, 14, bias=True),
    synthetic.Case("m17_long_k", 17, 136, 4096, 15),
]


@pytest.mark.parametrize("case", SHAPES, ids=[c.name for c in SHAPES])
def test_every_w8_variant(w4, case):
    W, A, b = synthetic.draw(case)
    packed, scales = w4.w8a16_quantize(W.cuda())
    y_ref = _reference(A, packed, scales, b)
    Ad = A.cuda()
    bd = None if b is None else b.cuda()
    for v in w8_variants(w4):
        if not w4.lib().w8a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        Y, ok = guarded((case.M, case.N), torch.bfloat16, Ad.device, NAN_BF16)
        w4.w8a16_gemm(Ad, packed, scales, bias=bd, Y=Y, variant=v)
        torch.cuda.synchronize()
        assert ok(), f"{vname(w4, v)} wrote outside Y"
        check_gemm_close(Y, y_ref, what=vname(w4, v))
    y = w4.w8a16_gemm(Ad, packed, scales, bias=bd)      # the rule's choice
    torch.cuda.synchronize()
    check_gemm_close(y, y_ref, what="default")
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


def test_integer_exact(w4):
    # power-of-two scales, small integer activations: exact sums, bit-exact
    rng = np.random.default_rng(33)
    M, N, K = 40, 256, 512
    codes = rng.integers(-100, 101, size=(N, K))
    codes[:, ::128] = 127
    e = rng.integers(-3, 0, size=(N, K // 128))
    x = (codes * np.repeat(2.0 ** e, 128, axis=1)).astype(np.float32)
    a = rng.integers(-1, 2, size=(M, K)).astype(np.float32)
    W = synthetic.to_bf16(x).cuda()
    A = synthetic.to_bf16(a)
    packed, scales = w4.w8a16_quantize(W)
    exact = a.astype(np.float64) @ x.astype(np.float64).T
    assert np.abs(exact).max() < 2 ** 16
    expected = bits(synthetic.to_bf16(exact.astype(np.float32)))
    for v in w8_variants(w4):
        if not w4.lib().w8a16_variant_eligible(v, M, N, K):
            continue
        Y = w4.w8a16_gemm(A.cuda(), packed, scales, variant=v)
        torch.cuda.synchronize()
        assert np.array_equal(bits(Y), expected), vname(w4, v)


def test_long_pipelines_and_determinism(w4):
    """K = 16384: long stage rings; fresh workspaces whose partial slots hold
    NaN; split tiles summed in k order give bit-identical repeats."""
    case = synthetic.Case("m300_k16384", 300, 256, 16384, 16, bias=True)
    W, A, b = synthetic.draw(case)
    packed, scales = w4.w8a16_quantize(W.cuda())
    y_ref = _reference(A, packed, scales, b)
    Ad, bd = A.cuda(), b.cuda()
    for v in w8_variants(w4):
        if not w4.lib().w8a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        need = w4.lib().w8a16_variant_workspace_bytes(v, case.M, case.N, case.K)
        ys = []
        for _ in range(2):
            ws = torch.zeros(max(need, 8192), dtype=torch.uint8, device=Ad.device)
            ws[8192:].fill_(0xFF)   # partial slots (after the 8 KiB counter region)
            ys.append(w4.w8a16_gemm(Ad, packed, scales, bias=bd, workspace=ws, variant=v))
        torch.cuda.synchronize()
        assert w4.w4a16_get_device_error() == w4.W4A16_OK, vname(w4, v)
        check_gemm_close(ys[0], y_ref, what=vname(w4, v))
        assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16)), vname(w4, v)


@pytest.mark.parametrize("case", synthetic.WORKLOADS["expert_m50"] + [synthetic.WORKLOADS["sweep"][8]],
                         ids=lambda c: c.name)
def test_workload_shapes(w4, case):
    # full-size workload shapes with the rule's choice, compared on sampled rows
    W, A, b = synthetic.draw(case)
    packed, scales = w4.w8a16_quantize(W.cuda())
    torch.cuda.synchronize()
    check_q8_exact(W, packed, scales, row0=0, rows=128)
    Y = w4.w8a16_gemm(A.cuda(), packed, scales, bias=None if b is None else b.cuda())
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(case.N - 64, case.N),
                                     np.random.default_rng(1).integers(0, case.N, 64)]))
    y_ref = _reference(A, packed, scales, b, rows=rows)
    check_gemm_close(Y[:, torch.as_tensor(rows)], y_ref,
                     rms=float(np.sqrt(np.mean(y_ref.astype(np.float64) ** 2))), what=case.name)
