"""The streaming GEMM variants for small M (the CUDA-core stream-K workers
simt_m{1,2,4,8}_sk and the row-block warp-MMA kernels rb_m{1,2,4,8,16})
against the oracle's FP32 GEMM on identical packed operands: M from 1 to 16
on ragged, multi-tile and long-K shapes within |y - y_ref| <= 1e-2 |y_ref|
+ 1e-2 rms(y_ref); bit-exact on integer-exact inputs; split tiles
bit-identical across runs with NaN-filled partial slots."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bits, check_gemm_close, guarded
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC1


def simt_variants(w4):
    return [v for v in range(w4.w4a16_variant_count()) if w4.w4a16_variant_name(v).startswith(("simt_", "rb_"))]


def reference(A, packed, scales, b, rows=None):
    s = scales.cpu().view(torch.int16).numpy().view(np.uint16)
    K, N = s.shape[0] * 128, s.shape[1]
    p = oracle.from_tile_layout(packed.cpu().numpy(), N, K)
    return oracle.gemm(bits(A), p, s, None if b is None else bits(b), rows=rows)


SHAPES = [synthetic.Case(f"m{m}_{n}x{k}", m, n, k, 40 + m + k // 128, "t4" if m % 2 else "normal",
                         bias=(m % 3 != 0))
          for m in (1, 2, 3, 4, 5, 7, 8, 9, 12, 16)
          for (n, k) in ((264, 384), (2048, 4096), (136, 16384))]


@pytest.mark.parametrize("case", SHAPES, ids=[c.name for c in SHAPES])
def test_simt_variants(w4, case):
    W, A, b = synthetic.draw(case)
    packed, scales = w4.w4a16_quantize(W.cuda())
    y_ref = reference(A, packed, scales, b)
    Ad = A.cuda()
    bd = None if b is None else b.cuda()
    ran = 0
    for v in simt_variants(w4):
        if not w4.w4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        Y, ok = guarded((case.M, case.N), torch.bfloat16, Ad.device, NAN_BF16)
        w4.w4a16_gemm(Ad, packed, scales, bias=bd, Y=Y, variant=v)
        torch.cuda.synchronize()
        assert ok(), f"{w4.w4a16_variant_name(v)} wrote outside Y"
        check_gemm_close(Y, y_ref, what=w4.w4a16_variant_name(v))
        ran += 1
    assert ran >= 1
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


def test_simt_ineligible_above_its_m(w4):
    for v in simt_variants(w4):
        mt = int(w4.w4a16_variant_name(v).split("_")[1][1:])
        assert w4.w4a16_variant_eligible(v, mt, 256, 512)
        assert not w4.w4a16_variant_eligible(v, mt + 1, 256, 512)


def test_simt_integer_exact(w4):
    # power-of-two scales, activations in {-1, 0, 1}: every product, the
    # offset corrections and every partial sum are exact in fp32, so Y is the
    # exact sum rounded once to bf16
    rng = np.random.default_rng(35)
    M, N, K = 16, 384, 2048
    codes = rng.integers(-7, 8, size=(N, K))
    codes[:, ::128] = 7
    e = rng.integers(-3, 0, size=(N, K // 128))
    x = (codes * np.repeat(2.0 ** e, 128, axis=1)).astype(np.float32)
    a = rng.integers(-1, 2, size=(M, K)).astype(np.float32)
    W = synthetic.to_bf16(x).cuda()
    packed, scales = w4.w4a16_quantize(W)
    for m in range(1, M + 1):
        A = synthetic.to_bf16(a[:m])
        exact = a[:m].astype(np.float64) @ x.astype(np.float64).T
        expected = bits(synthetic.to_bf16(exact.astype(np.float32)))
        for v in simt_variants(w4):
            if not w4.w4a16_variant_eligible(v, m, N, K):
                continue
            Y = w4.w4a16_gemm(A.cuda(), packed, scales, variant=v)
            torch.cuda.synchronize()
            assert np.array_equal(bits(Y), expected), (m, w4.w4a16_variant_name(v))


def test_simt_split_tiles_deterministic(w4):
    """Every tile split over several CTAs; fresh workspaces whose partial
    slots hold NaN; the k-ordered sums give bit-identical repeats."""
    case = synthetic.Case("m4_k16384", 4, 1024, 16384, 47, bias=True)
    W, A, b = synthetic.draw(case)
    packed, scales = w4.w4a16_quantize(W.cuda())
    y_ref = reference(A, packed, scales, b)
    Ad, bd = A.cuda(), b.cuda()
    for v in simt_variants(w4):
        if not w4.w4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        need = w4.w4a16_variant_workspace_bytes(v, case.M, case.N, case.K)
        # the stream-K workers split tiles through the workspace; the
        # row-block variants (rb_m*) split K inside a CTA and a cluster and
        # need none
        rowblock = w4.w4a16_variant_name(v).startswith("rb_")
        assert need == 0 if rowblock else need > 8192
        ys = []
        for _ in range(2):
            ws = None
            if need:
                ws = torch.zeros(need, dtype=torch.uint8, device=Ad.device)
                ws[8192:].fill_(0xFF)
            ys.append(w4.w4a16_gemm(Ad, packed, scales, bias=bd, workspace=ws, variant=v))
        torch.cuda.synchronize()
        assert w4.w4a16_get_device_error() == w4.W4A16_OK
        check_gemm_close(ys[0], y_ref, what=w4.w4a16_variant_name(v))
        assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16)), w4.w4a16_variant_name(v)


@pytest.mark.parametrize("case", [c for c in synthetic.WORKLOADS["sweep"] if c.M <= 16],
                         ids=lambda c: c.name)
def test_simt_sweep_shapes(w4, case):
    # the sweep's M <= 16 shapes through every eligible streaming variant,
    # all rows against the oracle
    W, A, b = synthetic.draw(case)
    packed, scales = w4.w4a16_quantize(W.cuda())
    y_ref = reference(A, packed, scales, b)
    Ad = A.cuda()
    for v in simt_variants(w4):
        if not w4.w4a16_variant_eligible(v, case.M, case.N, case.K):
            continue
        Y = w4.w4a16_gemm(Ad, packed, scales, variant=v)
        torch.cuda.synchronize()
        check_gemm_close(Y, y_ref, what=f"{case.name} {w4.w4a16_variant_name(v)}")


def test_simt_graph_capture(w4):
    # a streaming variant captured in a CUDA graph and replayed: Y identical
    # to the eager call (k-ordered split-tile sums are deterministic)
    case = synthetic.Case("simt_graph", 1, 2048, 4096, 51, bias=True)
    W, A, b = synthetic.draw(case)
    packed, scales = w4.w4a16_quantize(W.cuda())
    Ad, bd = A.cuda(), b.cuda()
    v = w4.variant_id("simt_m1_sk")
    y_e = w4.w4a16_gemm(Ad, packed, scales, bias=bd, variant=v)
    torch.cuda.synchronize()
    Y = torch.zeros_like(y_e)
    ws = torch.zeros(max(w4.w4a16_variant_workspace_bytes(v, 1, 2048, 4096), 16), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        w4.w4a16_gemm(Ad, packed, scales, bias=bd, Y=Y, workspace=ws, variant=v)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    Y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w4.w4a16_gemm(Ad, packed, scales, bias=bd, Y=Y, workspace=ws, variant=v)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int16), y_e.view(torch.int16))
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


# shapes whose row-block launch takes each form (team of 1, 2, 4 or 8 warps;
# cluster K split), the last row block ragged (N = 32 k + 8)
FORM_SHAPES = [(4104, 128), (4104, 256), (4104, 512), (4104, 1024), (264, 4096), (264, 16384),
               (16392, 2048)]


@pytest.mark.parametrize("M,variant", [(1, "rb_m1"), (3, "rb_m4"), (8, "rb_m8"), (11, "rb_m16"),
                                       (16, "rb_m16")])
def test_row_block_every_form(w4, M, variant):
    """Every launch form of the row-block kernel against the oracle: the
    forms are the host's choice for these shapes on this GPU, and together
    they cover teams of 1, 2, 4, 8 warps and the cluster split,
    bit-identical across repeats."""
    v = w4.variant_id(variant)
    forms = set()
    for i, (N, K) in enumerate(FORM_SHAPES):
        sch = w4.w4a16_variant_schedule(v, M, N, K)
        forms.add("cluster" if sch["cluster"] > 1 else "team%d" % sch["team"])
        assert w4.w4a16_variant_workspace_bytes(v, M, N, K) == 0
        case = synthetic.Case(f"form_m{M}_{N}x{K}", M, N, K, 70 + i, bias=(i % 2 == 0))
        W, A, b = synthetic.draw(case)
        packed, scales = w4.w4a16_quantize(W.cuda())
        y_ref = reference(A, packed, scales, b)
        bd = None if b is None else b.cuda()
        Y = w4.w4a16_gemm(A.cuda(), packed, scales, bias=bd, variant=v)
        Y2 = w4.w4a16_gemm(A.cuda(), packed, scales, bias=bd, variant=v)
        torch.cuda.synchronize()
        assert w4.w4a16_get_device_error() == w4.W4A16_OK
        check_gemm_close(Y, y_ref, what=f"{variant} {N}x{K} {sch}")
        assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
    assert forms == {"team1", "team2", "team4", "team8", "cluster"}, forms
