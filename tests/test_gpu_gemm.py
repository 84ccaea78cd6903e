"""W4A16 GEMM on the GPU against the oracle's FP32 GEMM on identical packed
operands: |y - y_ref| <= 1e-2 |y_ref| + 1e-2 rms(y_ref) element by element."""

import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_helpers import bits, check_gemm_close, guarded, oracle_quantize
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC1


def make_operands(w4, case):
    W, A, b = synthetic.draw(case)
    packed, scales = w4.w4a16_quantize(W.cuda())
    return W, A, b, packed, scales


def reference(A, packed, scales, b, rows=None):
    s = scales.cpu().view(torch.int16).numpy().view(np.uint16)
    K, N = s.shape[0] * 128, s.shape[1]
    p = oracle.from_tile_layout(packed.cpu().numpy(), N, K)
    return oracle.gemm(bits(A), p, s, None if b is None else bits(b), rows=rows)


SHAPES = [
    synthetic.Case("tiny", 16, 256, 512, 0),
    synthetic.Case("m1_ragged_n", 1, 264, 384, 11, bias=True),
    synthetic.Case("m50_ragged", 50, 520, 640, 12, "t4", bias=True),
    synthetic.Case("m129", 129, 256, 256, 13),
    synthetic.Case("m300_multi_tile", 300, 384, 1024, 14, bias=True),
    synthetic.Case("m17_long_k", 17, 136, 4096, 15),
    synthetic.Case("m3_ragged_n_even_groups", 3, 200, 768, 18, bias=True),
]


def variant_ids(w4):
    return list(range(w4.w4a16_variant_count()))


@pytest.mark.parametrize("case", SHAPES, ids=[c.name for c in SHAPES])
def test_every_variant(w4, case):
    W, A, b, packed, scales = make_operands(w4, case)
    y_ref = reference(A, packed, scales, b)
    Ad = A.cuda()
    bd = None if b is None else b.cuda()
    for v in variant_ids(w4):
        if not w4.w4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        Y, ok = guarded((case.M, case.N), torch.bfloat16, Ad.device, NAN_BF16)
        w4.w4a16_gemm(Ad, packed, scales, bias=bd, Y=Y, variant=v)
        torch.cuda.synchronize()
        assert ok(), f"variant {w4.w4a16_variant_name(v)} wrote outside Y"
        check_gemm_close(Y, y_ref, what=w4.w4a16_variant_name(v))
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


def test_every_variant_long_pipelines(w4):
    """Long runs through every variant's stage rings (K = 16384: 128 units
    per tile, up to 128 units per CTA), each launch on a fresh workspace whose
    partial slots hold NaN, three launches per variant: a stage reused before
    its copy landed, or a partial tile read before it was written, shows up
    as a wrong or non-finite output."""
    case = synthetic.Case("m300_k16384", 300, 256, 16384, 16, bias=True)
    W, A, b, packed, scales = make_operands(w4, case)
    y_ref = reference(A, packed, scales, b)
    Ad, bd = A.cuda(), b.cuda()
    for v in variant_ids(w4):
        if not w4.w4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        need = w4.w4a16_variant_workspace_bytes(v, case.M, case.N, case.K)
        for _ in range(3):
            ws = torch.zeros(max(need, 8192), dtype=torch.uint8, device=Ad.device)
            ws[8192:].fill_(0xFF)   # partial slots (after the 8 KiB counter region)
            Y = w4.w4a16_gemm(Ad, packed, scales, bias=bd, workspace=ws, variant=v)
            assert w4.w4a16_get_device_error() == w4.W4A16_OK, w4.w4a16_variant_name(v)
            check_gemm_close(Y, y_ref, what=w4.w4a16_variant_name(v))


def test_split_tiles_deterministic(w4):
    """A split tile is summed by whichever of its contributors arrives last,
    always in k order: repeated launches of every split variant give
    bit-identical outputs (K = 8192 spreads each tile over several CTAs)."""
    case = synthetic.Case("m17_k8192", 17, 384, 8192, 17, bias=True)
    W, A, b, packed, scales = make_operands(w4, case)
    y_ref = reference(A, packed, scales, b)
    Ad, bd = A.cuda(), b.cuda()
    checked = 0
    for v in variant_ids(w4):
        if not w4.w4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        if w4.w4a16_variant_workspace_bytes(v, case.M, case.N, case.K) == 0:
            continue   # whole tiles only
        ys = [w4.w4a16_gemm(Ad, packed, scales, bias=bd, variant=v) for _ in range(3)]
        torch.cuda.synchronize()
        check_gemm_close(ys[0], y_ref, what=w4.w4a16_variant_name(v))
        for y in ys[1:]:
            assert torch.equal(ys[0].view(torch.int16), y.view(torch.int16)), w4.w4a16_variant_name(v)
        checked += 1
    assert checked > 0
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


def test_default_selection_and_determinism(w4):
    case = synthetic.Case("det", 64, 2048, 2048, 21, bias=True)
    W, A, b, packed, scales = make_operands(w4, case)
    Ad, bd = A.cuda(), b.cuda()
    y1 = w4.w4a16_gemm(Ad, packed, scales, bias=bd).clone()
    y2 = w4.w4a16_gemm(Ad, packed, scales, bias=bd).clone()
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    check_gemm_close(y1, reference(A, packed, scales, b))


def test_hand_worked_example(w4):
    # A = ones(1, 128); W rows r0..r3 (and zero rows up to N = 8):
    # Y = 6, 0, 3 * 0.142822265625, -14 -> bf16 6, 0, 0.427734375, -14
    rows, _ = pins.load_golden()
    x = np.zeros((8, 128), np.float32)
    for i, n in enumerate(["r0", "r1", "r2", "r3"]):
        x[i] = pins.golden_row_values(rows[n])
    W = synthetic.to_bf16(x).cuda()
    packed, scales = w4.w4a16_quantize(W)
    A = torch.ones(1, 128, dtype=torch.bfloat16, device="cuda")
    for v in variant_ids(w4):
        if not w4.w4a16_variant_eligible(v, 1, 8, 128):
            # units of two groups need an even number of groups along K
            with pytest.raises(w4.W4A16Error) as ei:
                w4.w4a16_gemm(A, packed, scales, variant=v)
            assert ei.value.status == w4.W4A16_ERR_NO_VARIANT
            continue
        Y = w4.w4a16_gemm(A, packed, scales, variant=v)
        torch.cuda.synchronize()
        got = Y.float().cpu().numpy()[0]
        assert got[0] == 6.0 and got[1] == 0.0 and got[3] == -14.0, (w4.w4a16_variant_name(v), got)
        assert got[2] == np.float32(0.427734375), (w4.w4a16_variant_name(v), got)
        assert not got[4:].any()


def test_integer_exact(w4):
    # power-of-two scales and small-integer activations: every product and
    # partial sum is exact in fp32 (multiples of 1/8 below 2^12), so every
    # variant must return the exact sum rounded once to bf16
    rng = np.random.default_rng(31)
    M, N, K = 40, 256, 512
    codes = rng.integers(-3, 4, size=(N, K))
    codes[:, ::128] = 7
    e = rng.integers(-3, 0, size=(N, K // 128))
    x = (codes * np.repeat(2.0 ** e, 128, axis=1)).astype(np.float32)
    a = rng.integers(-1, 2, size=(M, K)).astype(np.float32)
    W = synthetic.to_bf16(x).cuda()
    A = synthetic.to_bf16(a)
    packed, scales = w4.w4a16_quantize(W)
    exact = a.astype(np.float64) @ x.astype(np.float64).T
    assert np.all(exact == np.round(exact * 8) / 8) and np.abs(exact).max() < 4096
    expected = bits(synthetic.to_bf16(exact.astype(np.float32)))
    for v in variant_ids(w4):
        if not w4.w4a16_variant_eligible(v, M, N, K):
            continue
        Y = w4.w4a16_gemm(A.cuda(), packed, scales, variant=v)
        torch.cuda.synchronize()
        assert np.array_equal(bits(Y), expected), w4.w4a16_variant_name(v)


@pytest.mark.parametrize("N", [128, 256, 512, 1024, 2048])
def test_split_fixup_modes_integer_exact(w4, N):
    """Split tiles with few and with very many contributors, summed by the
    readout warps in the middle of a run or by the whole CTA at its exit: with
    M = 50, K = 8192 the tiles of the different activation widths are spread
    over roughly 5 to 80 CTAs.  Integer-valued inputs make every partial and
    every order of summing them exact, so a partial summed twice or missed
    changes the result: every split variant must return the exact sum rounded
    once to bf16, twice, each launch on a workspace whose partial slots hold
    NaN."""
    rng = np.random.default_rng(33 + N)
    M, K = 50, 8192
    codes = rng.integers(-3, 4, size=(N, K))
    codes[:, ::128] = 7
    e = rng.integers(-3, 0, size=(N, K // 128))
    x = (codes * np.repeat(2.0 ** e, 128, axis=1)).astype(np.float32)
    a = rng.integers(-1, 2, size=(M, K)).astype(np.float32)
    W = synthetic.to_bf16(x).cuda()
    Ad = synthetic.to_bf16(a).cuda()
    packed, scales = w4.w4a16_quantize(W)
    exact = a.astype(np.float64) @ x.astype(np.float64).T
    assert np.all(exact == np.round(exact * 8) / 8) and np.abs(exact).max() < 2 ** 20
    expected = bits(synthetic.to_bf16(exact.astype(np.float32)))
    checked = 0
    for v in variant_ids(w4):
        if not w4.w4a16_variant_eligible(v, M, N, K):
            continue
        need = w4.w4a16_variant_workspace_bytes(v, M, N, K)
        if need == 0:
            continue   # whole tiles only
        for _ in range(2):
            ws = torch.zeros(need, dtype=torch.uint8, device=Ad.device)
            ws[8192:].fill_(0xFF)   # partial slots (after the 8 KiB counter region)
            Y = w4.w4a16_gemm(Ad, packed, scales, workspace=ws, variant=v)
            torch.cuda.synchronize()
            assert np.array_equal(bits(Y), expected), (w4.w4a16_variant_name(v), N)
        checked += 1
    assert checked > 0
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


def test_workspace_too_small_is_an_error(w4):
    M, N, K = 16, 2048, 2048
    v = w4.variant_id("tc_a16_grp_sk")
    need = w4.w4a16_variant_workspace_bytes(v, M, N, K)
    assert need > 0
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    packed = torch.zeros(w4.w4a16_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    scales = torch.ones(K // 128, N, dtype=torch.float16, device="cuda")
    ws = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(w4.W4A16Error) as ei:
        w4.w4a16_gemm(A, packed, scales, workspace=ws, variant=v)
    assert ei.value.status == w4.W4A16_ERR_WORKSPACE


FULL = [c for name in ("tiny", "expert_m50", "prefix_m816", "sweep", "large")
        for c in synthetic.WORKLOADS[name]]


@pytest.mark.parametrize("case", FULL, ids=[c.name for c in FULL])
def test_workloads_full_size_sampled(w4, case):
    """Full-size workloads through the default (table/rule) variant, which is
    the launch configuration the benchmark times; rows sampled for the
    oracle (all rows when M <= 64)."""
    W, A, b, packed, scales = make_operands(w4, case)
    Y = w4.w4a16_gemm(A.cuda(), packed, scales)
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
    M = case.M
    rows = np.arange(M) if M <= 64 else np.unique(np.r_[0, 1, M // 2, M - 2, M - 1,
                                                       np.random.default_rng(0).integers(0, M, 11)])
    y_ref = reference(A, packed, scales, b, rows=rows)
    check_gemm_close(Y[torch.as_tensor(rows, device=Y.device)], y_ref, what=case.name)


def test_static_weights_prefetch_back_to_back(w4):
    """With the weights declared static (w4a16_set_weights_static), each GEMM
    copies its first codes and scales before the previous kernel on the
    stream finishes.  Back-to-back launches in one CUDA graph, every launch on
    other weights and activations and each writing its own output, must still
    give each launch's own result (every variant, a stream-K and a
    data-parallel shape); a launch that used another launch's operands would
    miss the tolerance."""
    cases = [synthetic.Case("static_m16_n1024_k2048", 16, 1024, 2048, 31, bias=True),
             synthetic.Case("static_m64_n256_k4096", 64, 256, 4096, 32),
             # the CUDA-core kernels for M <= 4 (ragged last row block)
             synthetic.Case("static_m1_n2056_k2048", 1, 2056, 2048, 33, bias=True),
             synthetic.Case("static_m3_n1032_k4096", 3, 1032, 4096, 34)]
    try:
        w4.w4a16_set_weights_static(True)
        assert w4.w4a16_weights_static()
        for case in cases:
            ops = []
            for r in range(3):
                c = synthetic.Case(case.name, case.M, case.N, case.K, case.seed + 10 * r, bias=case.bias)
                W, A, b, packed, scales = make_operands(w4, c)
                ops.append((A.cuda(), None if b is None else b.cuda(), packed, scales,
                            reference(A, packed, scales, b)))
            torch.cuda.synchronize()   # the quantizes are done before any GEMM reads early
            for v in variant_ids(w4):
                if not w4.w4a16_variant_eligible(v, case.M, case.N, case.K):
                    continue
                need = w4.w4a16_variant_workspace_bytes(v, case.M, case.N, case.K)
                ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
                Ys = [torch.full((case.M, case.N), float("nan"), dtype=torch.bfloat16, device="cuda")
                      for _ in ops]
                for (A, b, p, s, _), Y in zip(ops, Ys):   # outside the capture: attributes
                    w4.w4a16_gemm(A, p, s, bias=b, Y=Y, workspace=ws, variant=v)
                g = torch.cuda.CUDAGraph()
                cs = torch.cuda.Stream()
                cs.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(cs):
                    with torch.cuda.graph(g, stream=cs):
                        for _ in range(2):
                            for (A, b, p, s, _), Y in zip(ops, Ys):
                                w4.w4a16_gemm(A, p, s, bias=b, Y=Y, workspace=ws, variant=v, stream=cs)
                torch.cuda.current_stream().wait_stream(cs)
                for Y in Ys:
                    Y.fill_(float("nan"))
                g.replay()
                torch.cuda.synchronize()
                for (_, _, _, _, y_ref), Y in zip(ops, Ys):
                    check_gemm_close(Y, y_ref, what=f"static {w4.w4a16_variant_name(v)}")
    finally:
        w4.w4a16_set_weights_static(False)
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
