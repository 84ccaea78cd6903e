"""W4A16 GEMM with the SwiGLU epilogue on the GPU against the oracle's
gemm_swiglu on identical packed operands (weight rows interleave up and
gate), for every tcgen05 variant, whole and split tiles, with and without
bias.  The bound is the GEMM's tolerance on the pre-activations, tol(y) =
1e-2 |y| + 1e-2 rms(y), carried through h = silu(g) u (first order, the
second-order term in g and the cross term) plus the final bf16 rounding:
    |h - h_ref| <= |silu'(g) u| tol(g) + 0.25 tol(g)^2 |u|
                   + (|silu(g)| + 1.1 tol(g)) tol(u) + 2^-8 |h_ref|
(|silu'| <= 1.1 and |silu''| <= 0.5 everywhere)."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bits, guarded
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC1

SHAPES = [
    synthetic.Case("tiny", 16, 256, 512, 40),
    synthetic.Case("m1_ragged_n", 1, 264, 384, 41, bias=True),
    synthetic.Case("m50_ragged", 50, 520, 640, 42, "t4", bias=True),
    synthetic.Case("m300_multi_tile", 300, 384, 1024, 43, bias=True),
    synthetic.Case("m17_k8192_split", 17, 384, 8192, 44, bias=True),
]


def check_swiglu_close(Y, y_pre, rms_y=None, what=""):
    """Y [M, N/2] from the GPU against swiglu(y_pre) (y_pre: the oracle's FP32
    GEMM with bias, [M, N], interleaved up/gate columns)."""
    y = np.asarray(y_pre, dtype=np.float64)
    h_ref = oracle.swiglu(y)
    hg = Y.float().cpu().numpy().astype(np.float64)
    assert hg.shape == h_ref.shape, (hg.shape, h_ref.shape)
    assert np.isfinite(hg).all(), f"{what}: non-finite output"
    if rms_y is None:
        rms_y = float(np.sqrt(np.mean(y ** 2)))
    up, gate = y[:, 0::2], y[:, 1::2]
    sig = 1.0 / (1.0 + np.exp(-gate))
    dsilu = sig * (1.0 + gate * (1.0 - sig))
    tol_g = 1e-2 * np.abs(gate) + 1e-2 * rms_y
    tol_u = 1e-2 * np.abs(up) + 1e-2 * rms_y
    lim = (np.abs(dsilu * up) * tol_g + 0.25 * tol_g ** 2 * np.abs(up)
           + (np.abs(gate * sig) + 1.1 * tol_g) * tol_u + 2.0 ** -8 * np.abs(h_ref))
    err = np.abs(hg - h_ref)
    bad = np.argwhere(err > lim)
    assert bad.size == 0, (
        f"{what}: {len(bad)} of {err.size} outside tolerance; worst excess "
        f"{float(np.max(err - lim)):.4g} at {bad[:3].tolist()}")


def operands(w4, case):
    W, A, b = synthetic.draw(case)
    packed, scales = w4.w4a16_quantize(W.cuda())
    s = scales.cpu().view(torch.int16).numpy().view(np.uint16)
    p = oracle.from_tile_layout(packed.cpu().numpy(), case.N, case.K)
    y_pre = oracle.gemm(bits(A), p, s, None if b is None else bits(b))
    return A.cuda(), None if b is None else b.cuda(), packed, scales, y_pre


def tc_variants(w4):
    # tcgen05 variants with a SwiGLU form: not the CUDA-core streaming ones,
    # not cluster split-K (its exit reduction stores plain outputs)
    return [v for v in range(w4.w4a16_variant_count())
            if not w4.w4a16_variant_name(v).startswith(("simt_", "rb_"))
            and "csk" not in w4.w4a16_variant_name(v)]


@pytest.mark.parametrize("case", SHAPES, ids=[c.name for c in SHAPES])
def test_every_variant(w4, case):
    Ad, bd, packed, scales, y_pre = operands(w4, case)
    checked = 0
    for v in tc_variants(w4):
        if not w4.w4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        Y, untouched = guarded((case.M, case.N // 2), torch.bfloat16, Ad.device, NAN_BF16)
        w4.w4a16_gemm_swiglu(Ad, packed, scales, bias=bd, Y=Y, variant=v)
        torch.cuda.synchronize()
        assert untouched(), f"variant {w4.w4a16_variant_name(v)} wrote outside Y"
        check_swiglu_close(Y, y_pre, what=w4.w4a16_variant_name(v))
        checked += 1
    assert checked > 0
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


def test_default_selection_small_m(w4):
    """For M <= 8 the rule may prefer a CUDA-core streaming variant; the
    SwiGLU call then takes the best tcgen05 variant instead."""
    for M in (1, 4, 8):
        case = synthetic.Case(f"m{M}", M, 2048, 1024, 45 + M, bias=True)
        Ad, bd, packed, scales, y_pre = operands(w4, case)
        Y = w4.w4a16_gemm_swiglu(Ad, packed, scales, bias=bd)
        torch.cuda.synchronize()
        check_swiglu_close(Y, y_pre, what=f"default M={M}")
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


def test_streaming_variants_are_rejected(w4):
    case = SHAPES[0]
    Ad, bd, packed, scales, _ = operands(w4, case)
    for v in range(w4.w4a16_variant_count()):
        name = w4.w4a16_variant_name(v)
        if not (name.startswith(("simt_", "rb_")) or "csk" in name):
            continue
        with pytest.raises(w4.W4A16Error):
            w4.w4a16_gemm_swiglu(Ad[:1].contiguous(), packed, scales, variant=v)


def test_split_tiles_deterministic(w4):
    case = SHAPES[-1]
    Ad, bd, packed, scales, _ = operands(w4, case)
    checked = 0
    for v in tc_variants(w4):
        if not w4.w4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        if w4.w4a16_variant_workspace_bytes(v, case.M, case.N, case.K) == 0:
            continue
        ys = [w4.w4a16_gemm_swiglu(Ad, packed, scales, bias=bd, variant=v).clone() for _ in range(3)]
        torch.cuda.synchronize()
        for y in ys[1:]:
            assert torch.equal(ys[0].view(torch.int16), y.view(torch.int16)), w4.w4a16_variant_name(v)
        checked += 1
    assert checked > 0


@pytest.mark.parametrize("case", [c for c in synthetic.WORKLOADS["expert_m50"] + synthetic.WORKLOADS["prefix_m816"]
                                  if "gate_up" in c.name], ids=lambda c: c.name)
def test_workload_gate_up_shapes(w4, case):
    """The workloads' gate/up projections at full size with the default
    selection; the M = 816 case is checked on sampled activation rows."""
    W, A, b = synthetic.draw(case)
    packed, scales = w4.w4a16_quantize(W.cuda())
    Y = w4.w4a16_gemm_swiglu(A.cuda(), packed, scales, bias=None if b is None else b.cuda())
    torch.cuda.synchronize()
    s = scales.cpu().view(torch.int16).numpy().view(np.uint16)
    p = oracle.from_tile_layout(packed.cpu().numpy(), case.N, case.K)
    rows = None if case.M <= 64 else np.sort(np.random.default_rng(0).choice(case.M, 12, replace=False))
    y_pre = oracle.gemm(bits(A), p, s, None if b is None else bits(b), rows=rows)
    got = Y if rows is None else Y[torch.as_tensor(rows, device=Y.device)]
    check_swiglu_close(got, y_pre, what=case.name)
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


def test_graph_capture(w4):
    """The SwiGLU call is capture-safe: a captured quantize + SwiGLU GEMM,
    replayed, gives the eager result bit for bit."""
    case = synthetic.Case("m50_capture", 50, 2048, 1024, 49, bias=True)
    W, A, b = synthetic.draw(case)
    Wd, Ad, bd = W.cuda(), A.cuda(), b.cuda()
    p_e, s_e = w4.w4a16_quantize(Wd)
    y_e = w4.w4a16_gemm_swiglu(Ad, p_e, s_e, bias=bd).clone()
    torch.cuda.synchronize()
    packed, scales = torch.zeros_like(p_e), torch.zeros_like(s_e)
    Y = torch.empty_like(y_e)
    ws = torch.zeros(max(w4.lib().w4a16_gemm_swiglu_workspace_bytes(case.M, case.N, case.K), 16),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):          # warm-up outside capture
        w4.w4a16_quantize(Wd, packed=packed, scales=scales)
        w4.w4a16_gemm_swiglu(Ad, packed, scales, bias=bd, Y=Y, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    packed.zero_(), scales.zero_(), Y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w4.w4a16_quantize(Wd, packed=packed, scales=scales)
        w4.w4a16_gemm_swiglu(Ad, packed, scales, bias=bd, Y=Y, workspace=ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(packed, p_e) and torch.equal(scales, s_e)
    assert torch.equal(Y.view(torch.int16), y_e.view(torch.int16))
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
