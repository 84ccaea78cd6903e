"""FP4 weight-only schemes (MXFP4, NVFP4) on the GPU against the oracle:
codes, block-scale codes and NVFP4's tensor scale bit-exact; GEMM within
|y - y_ref| <= 1e-2 |y_ref| + 1e-2 rms(y_ref) on identical packed operands,
bit-exact on integer-exact inputs ("Kernel dispatch and Humming quantization
in PhyAI", section "Choose precision by layer and hardware": MXFP4 and NVFP4
are Humming weight schemes; "Piper Kernels", section "NVFP4 construction":
blocks of 16, a per-tensor scale applied with the bias in FP32)."""

import numpy as np
import pytest
import torch

import oracle
import pins
from gpu_helpers import bits, check_gemm_close, guarded
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC1
FORMATS = ["mxfp4", "nvfp4"]


def oracle_fp4(x: np.ndarray, fmt: str, g=None):
    """(row-major packed bytes, scale codes, g) of the oracle for float32 x."""
    if fmt == "mxfp4":
        p, s = oracle.quantize_mxfp4_f32(x)
        return p, s, None
    return oracle.quantize_nvfp4_f32(x, tensor_scale=g)


def check_fp4_exact(W_cpu, fmt, packed, scales, ts, row0=0, rows=None):
    x = oracle.bf16_bits_to_f32(bits(W_cpu))
    N, K = x.shape
    rows = N if rows is None else rows
    g = None
    if fmt == "nvfp4":
        amax = np.float32(np.max(np.abs(x)))
        t = ts.cpu().numpy()
        assert t[1] == amax, ("tensor absmax", t[1], amax)
        g = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(2688.0))
        assert t[0] == g, ("tensor scale", t[0], g)
    p_rm, s_ref, _ = oracle_fp4(x[row0:row0 + rows], fmt, g)
    p_ref = oracle.to_tile_layout(p_rm)
    p = packed.cpu().numpy().reshape(-1)
    if not (row0 == 0 and rows == N):
        G = K // 128
        p = p[(row0 // 128) * G * 8192:((row0 + rows) // 128) * G * 8192]
    s = scales.cpu().numpy()[:, row0:row0 + rows]
    bad_s = np.argwhere(s != s_ref)
    assert bad_s.size == 0, f"{fmt}: {len(bad_s)} scale-code mismatches, first {bad_s[:4].tolist()}"
    bad = np.argwhere(p != p_ref)
    assert bad.size == 0, f"{fmt}: {len(bad)} code-byte mismatches, first {bad[:4].tolist()}"


def dequant_ref(fmt, packed, scales, ts, N, K):
    p_rm = oracle.from_tile_layout(packed.cpu().numpy(), N, K)
    s = scales.cpu().numpy()
    if fmt == "mxfp4":
        return oracle.dequantize_mxfp4(p_rm, s)
    return oracle.dequantize_nvfp4(p_rm, s, np.float32(ts.cpu().numpy()[0]))


def reference(fmt, A, packed, scales, ts, b, N, K, rows=None):
    wd = dequant_ref(fmt, packed, scales, ts, N, K)
    return oracle.gemm_fp4(bits(A), wd, None if b is None else bits(b), rows=rows)


def variants(w4):
    return list(range(w4.fp4a16_variant_count()))


def vname(w4, v):
    return w4.fp4a16_variant_name(v)


@pytest.mark.parametrize("fmt", FORMATS)
def test_quantize_special_and_ragged(w4, fmt):
    for x in (pins.special_groups(64).reshape(16, 512), pins.random_weights(144, 384, 5, "t4"),
              pins.random_weights(1008, 1152, 6, "normal")):
        W = synthetic.to_bf16(x)
        packed, scales, ts = w4.fp4a16_quantize(W.cuda(), fmt)
        torch.cuda.synchronize()
        check_fp4_exact(W, fmt, packed, scales, ts)


@pytest.mark.parametrize("fmt", FORMATS)
def test_gemm_on_special_groups(w4, fmt):
    # zero blocks, spikes, ties, blocks of tiny values (MXFP4 exponent codes
    # 0 and 1: subnormal bf16 operands), large values: every variant within
    # tolerance of the oracle on the same codes and scales
    x = pins.special_groups(64).reshape(16, 512)
    W = synthetic.to_bf16(x)
    A = synthetic.to_bf16(np.random.default_rng(61).standard_normal((9, 512)).astype(np.float32))
    packed, scales, ts = w4.fp4a16_quantize(W.cuda(), fmt)
    y_ref = reference(fmt, A, packed, scales, ts, None, 16, 512)
    for v in variants(w4):
        if not w4.fp4a16_variant_eligible(v, 9, 16, 512):
            continue
        Y = w4.fp4a16_gemm(A.cuda(), packed, scales, fmt, tensor_scale=ts, variant=v)
        torch.cuda.synchronize()
        check_gemm_close(Y, y_ref, what=f"{fmt} {vname(w4, v)}")
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


@pytest.mark.parametrize("fmt", FORMATS)
def test_quantize_ties_and_saturation(w4, fmt):
    # block scales that are powers of two (MXFP4: amax 6 * 2^e; NVFP4: g = 1
    # from one value 2688 and block amax 6 * 2^j, so s_b = 2^j), elements on
    # the quarter grid: every E2M1 midpoint occurs; MXFP4 blocks with amax in
    # (6, 8) * 2^e saturate
    rng = np.random.default_rng(8)
    N, K = 64, 1024
    bs = 32 if fmt == "mxfp4" else 16
    q = rng.integers(-24, 25, size=(N, K)).astype(np.float32) / 4      # [-6, 6] on 0.25 steps
    q[:, ::bs] = 6.0
    if fmt == "mxfp4":
        q[::3, 1::bs] = -7.5                                            # saturating blocks
        e = rng.integers(-8, 8, size=(N, K // bs))
    else:
        e = rng.integers(-6, 7, size=(N, K // bs))
    x = q * np.repeat(2.0 ** e, bs, axis=1)
    if fmt == "nvfp4":
        x[0, 0] = 2688.0                                                # g = 1
    W = synthetic.to_bf16(x.astype(np.float32))
    packed, scales, ts = w4.fp4a16_quantize(W.cuda(), fmt)
    torch.cuda.synchronize()
    check_fp4_exact(W, fmt, packed, scales, ts)


def test_nvfp4_zero_tensor(w4):
    W = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    packed, scales, ts = w4.fp4a16_quantize(W, "nvfp4")
    torch.cuda.synchronize()
    assert ts.cpu().tolist() == [1.0, 0.0]
    assert not packed[: 128 * 128].any() and not scales.any()
    A = torch.ones((3, 256), dtype=torch.bfloat16, device="cuda")
    b = torch.arange(128, dtype=torch.float32).to(torch.bfloat16).cuda()
    Y = w4.fp4a16_gemm(A, packed, scales, "nvfp4", tensor_scale=ts, bias=b)
    torch.cuda.synchronize()
    assert torch.equal(Y, b.expand(3, 128))


@pytest.mark.parametrize("fmt", FORMATS)
def test_quantize_large_weight_sampled(w4, fmt):
    c = synthetic.WORKLOADS["large"][0]
    W = synthetic.draw_weight_only(c.seed, c.N, c.K)
    packed, scales, ts = w4.fp4a16_quantize(W.cuda(), fmt)
    torch.cuda.synchronize()
    for row0 in (0, c.N - 128):
        check_fp4_exact(W, fmt, packed, scales, ts, row0=row0, rows=128)


SHAPES = [
    synthetic.Case("tiny", 16, 256, 512, 0),
    synthetic.Case("m1_ragged_n", 1, 272, 384, 11, bias=True),
    synthetic.Case("m50_ragged", 50, 528, 640, 12, "t4", bias=True),
    synthetic.Case("m129", 129, 256, 256, 13),
    synthetic.Case("m300_multi_tile", 300, 384, 1024, 14, bias=True),
    synthetic.Case("m17_long_k", 17, 144, 4096, 15),
]


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("case", SHAPES, ids=[c.name for c in SHAPES])
def test_every_fp4_variant(w4, case, fmt):
    W, A, b = synthetic.draw(case)
    packed, scales, ts = w4.fp4a16_quantize(W.cuda(), fmt)
    torch.cuda.synchronize()
    check_fp4_exact(W, fmt, packed, scales, ts)
    y_ref = reference(fmt, A, packed, scales, ts, b, case.N, case.K)
    Ad = A.cuda()
    bd = None if b is None else b.cuda()
    for v in variants(w4):
        if not w4.fp4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        Y, ok = guarded((case.M, case.N), torch.bfloat16, Ad.device, NAN_BF16)
        w4.fp4a16_gemm(Ad, packed, scales, fmt, tensor_scale=ts, bias=bd, Y=Y, variant=v)
        torch.cuda.synchronize()
        assert ok(), f"{vname(w4, v)} wrote outside Y"
        check_gemm_close(Y, y_ref, what=f"{fmt} {vname(w4, v)}")
    y = w4.fp4a16_gemm(Ad, packed, scales, fmt, tensor_scale=ts, bias=bd)   # the rule's choice
    torch.cuda.synchronize()
    check_gemm_close(y, y_ref, what=f"{fmt} default")
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


@pytest.mark.parametrize("fmt", FORMATS)
def test_integer_exact(w4, fmt):
    # power-of-two scales (MXFP4: block amax 6 * 2^e; NVFP4: tensor amax 42
    # gives g = 2^-6, block amax 6 * 2^j gives s_b = 2^(j + 6)), activations
    # in {-1, 0, 1}: every product and partial sum is exact in fp32, so Y is
    # the bf16 rounding of the exact sum
    rng = np.random.default_rng(33)
    M, N, K = 40, 256, 512
    bs = 32 if fmt == "mxfp4" else 16
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    q = mags[rng.integers(0, 8, size=(N, K))] * rng.choice([-1.0, 1.0], size=(N, K))
    q[:, ::bs] = 6.0
    e = rng.integers(-3, 1, size=(N, K // bs))
    x = (q * np.repeat(2.0 ** e, bs, axis=1)).astype(np.float32)
    if fmt == "nvfp4":
        x[0, 0] = 42.0          # = 6 * 7, not a block amax of the 6 * 2^j form: that block
        x[0, 1:16] = 0.0        # holds only this value; 42 / 6 / 2^-6 = 448, s_b g = 7
    a = rng.integers(-1, 2, size=(M, K)).astype(np.float32)
    W = synthetic.to_bf16(x).cuda()
    A = synthetic.to_bf16(a)
    packed, scales, ts = w4.fp4a16_quantize(W, fmt)
    torch.cuda.synchronize()
    wd = dequant_ref(fmt, packed, scales, ts, N, K).astype(np.float64)
    assert np.array_equal(wd, x.astype(np.float64))            # every weight is exact
    exact = a.astype(np.float64) @ x.astype(np.float64).T
    expected = bits(synthetic.to_bf16(exact.astype(np.float32)))
    for v in variants(w4):
        if not w4.fp4a16_variant_eligible(v, M, N, K):
            continue
        Y = w4.fp4a16_gemm(A.cuda(), packed, scales, fmt, tensor_scale=ts, variant=v)
        torch.cuda.synchronize()
        assert np.array_equal(bits(Y), expected), f"{fmt} {vname(w4, v)}"


@pytest.mark.parametrize("fmt", FORMATS)
def test_long_pipelines_and_determinism(w4, fmt):
    """K = 16384: long stage rings; fresh workspaces whose partial slots hold
    NaN; split tiles summed in k order give bit-identical repeats."""
    case = synthetic.Case("m300_k16384", 300, 256, 16384, 16, bias=True)
    W, A, b = synthetic.draw(case)
    packed, scales, ts = w4.fp4a16_quantize(W.cuda(), fmt)
    y_ref = reference(fmt, A, packed, scales, ts, b, case.N, case.K)
    Ad, bd = A.cuda(), b.cuda()
    for v in variants(w4):
        if not w4.fp4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        need = w4.lib().fp4a16_variant_workspace_bytes(v, case.M, case.N, case.K)
        ys = []
        for _ in range(2):
            ws = torch.zeros(max(need, 8192), dtype=torch.uint8, device=Ad.device)
            ws[8192:].fill_(0xFF)   # partial slots (after the 8 KiB counter region)
            ys.append(w4.fp4a16_gemm(Ad, packed, scales, fmt, tensor_scale=ts, bias=bd,
                                     workspace=ws, variant=v))
        torch.cuda.synchronize()
        assert w4.w4a16_get_device_error() == w4.W4A16_OK, vname(w4, v)
        check_gemm_close(ys[0], y_ref, what=f"{fmt} {vname(w4, v)}")
        assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16)), vname(w4, v)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("case", synthetic.WORKLOADS["expert_m50"][:2] + [synthetic.WORKLOADS["sweep"][8]],
                         ids=lambda c: c.name)
def test_workload_shapes(w4, case, fmt):
    # full-size workload shapes with the rule's choice, compared on sampled rows
    W, A, b = synthetic.draw(case)
    packed, scales, ts = w4.fp4a16_quantize(W.cuda(), fmt)
    torch.cuda.synchronize()
    check_fp4_exact(W, fmt, packed, scales, ts, row0=0, rows=128)
    Y = w4.fp4a16_gemm(A.cuda(), packed, scales, fmt, tensor_scale=ts,
                       bias=None if b is None else b.cuda())
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(case.N - 64, case.N),
                                     np.random.default_rng(1).integers(0, case.N, 64)]))
    y_ref = reference(fmt, A, packed, scales, ts, b, case.N, case.K, rows=rows)
    check_gemm_close(Y[:, torch.as_tensor(rows)], y_ref,
                     rms=float(np.sqrt(np.mean(y_ref.astype(np.float64) ** 2))), what=case.name)


def test_fp4_argument_errors(w4):
    L = w4.lib()
    W = torch.zeros((24, 256), dtype=torch.bfloat16, device="cuda")       # N % 16 != 0
    p = torch.empty(L.fp4a16_packed_bytes(24, 256), dtype=torch.uint8, device="cuda")
    s = torch.empty(L.fp4a16_scales_bytes(2, 24, 256), dtype=torch.uint8, device="cuda")
    ts = torch.empty(2, dtype=torch.float32, device="cuda")
    sh = torch.cuda.current_stream().cuda_stream
    assert L.fp4a16_quantize(1, W.data_ptr(), 24, 256, p.data_ptr(), s.data_ptr(), None, sh) == \
        w4.W4A16_ERR_UNSUPPORTED
    assert L.fp4a16_quantize(3, W.data_ptr(), 32, 256, p.data_ptr(), s.data_ptr(), None, sh) == \
        w4.W4A16_ERR_UNSUPPORTED
    assert L.fp4a16_quantize(2, W.data_ptr(), 16, 256, p.data_ptr(), s.data_ptr(), None, sh) == \
        w4.W4A16_ERR_INVALID_ARG                                            # NVFP4 needs the pair
    assert L.fp4a16_quantize(2, W.data_ptr(), 16, 256, p.data_ptr(), s.data_ptr(),
                             ts.data_ptr() + 4, sh) == w4.W4A16_ERR_ALIGNMENT
    A = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((2, 16), dtype=torch.bfloat16, device="cuda")
    assert L.fp4a16_gemm(2, A.data_ptr(), 2, 16, 256, p.data_ptr(), s.data_ptr(), None, None,
                         Y.data_ptr(), None, 0, sh) == w4.W4A16_ERR_INVALID_ARG
    assert L.fp4a16_gemm(1, A.data_ptr(), 2, 24, 256, p.data_ptr(), s.data_ptr(), None, None,
                         Y.data_ptr(), None, 0, sh) == w4.W4A16_ERR_UNSUPPORTED


@pytest.mark.parametrize("fmt", FORMATS)
def test_fp4_graph_capture(w4, fmt):
    # the whole FP4 path (NVFP4: the memset of the tensor-scale pair, the
    # absmax kernel, the quantize kernel; then the GEMM) captured in a CUDA
    # graph and replayed: the same codes, scales and Y as eager calls
    case = synthetic.Case("fp4_graph", 50, 1024, 1024, 9, bias=True)
    W, A, b = synthetic.draw(case)
    Wd, Ad, bd = W.cuda(), A.cuda(), b.cuda()
    p_e, s_e, t_e = w4.fp4a16_quantize(Wd, fmt)
    y_e = w4.fp4a16_gemm(Ad, p_e, s_e, fmt, tensor_scale=t_e, bias=bd)
    torch.cuda.synchronize()
    packed, scales = torch.zeros_like(p_e), torch.zeros_like(s_e)
    ts = torch.zeros(2, dtype=torch.float32, device="cuda")
    Y = torch.empty_like(y_e)
    ws = torch.zeros(max(w4.lib().fp4a16_gemm_workspace_bytes(w4.FP4_FORMATS[fmt], 50, 1024, 1024), 16),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):          # warm-up outside capture
        w4.fp4a16_quantize(Wd, fmt, packed=packed, scales=scales, tensor_scale=ts)
        w4.fp4a16_gemm(Ad, packed, scales, fmt, tensor_scale=ts, bias=bd, Y=Y, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    packed.zero_(), scales.zero_(), ts.fill_(-1.0), Y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w4.fp4a16_quantize(Wd, fmt, packed=packed, scales=scales, tensor_scale=ts)
        w4.fp4a16_gemm(Ad, packed, scales, fmt, tensor_scale=ts, bias=bd, Y=Y, workspace=ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(packed, p_e) and torch.equal(scales, s_e)
    if fmt == "nvfp4":
        assert torch.equal(ts, t_e)
    assert torch.equal(Y.view(torch.int16), y_e.view(torch.int16))
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


@pytest.mark.parametrize("fmt", FORMATS)
def test_quantize_extreme_magnitudes(w4, fmt):
    # the special groups scaled to amax 1e-35 (NVFP4: a subnormal tensor scale,
    # so both zero and subnormal steps s_b g, the quantizer's IEEE-division
    # branches; MXFP4: exponent codes near 0) and to amax 4e37 (MXFP4 exponent
    # codes up to 249): codes, scale codes and the tensor scale bit-exact
    base = pins.special_groups(64).reshape(16, 512).astype(np.float64)
    for factor in (2.5e-41, 1e32):
        W = synthetic.to_bf16((base * factor).astype(np.float32))
        packed, scales, ts = w4.fp4a16_quantize(W.cuda(), fmt)
        torch.cuda.synchronize()
        check_fp4_exact(W, fmt, packed, scales, ts)
