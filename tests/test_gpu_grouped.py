"""Grouped launches: several independent quantize / GEMM problems in one
kernel, each checked against the oracle exactly as a single call is."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bits, check_gemm_close, check_quantize_exact
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu

MIXED = [
    synthetic.Case("g_tiny", 16, 256, 512, 40),
    synthetic.Case("g_m50_ragged", 50, 520, 640, 41, "t4", bias=True),
    synthetic.Case("g_m1_ragged_n", 1, 264, 384, 42, bias=True),
    synthetic.Case("g_m300", 300, 384, 1024, 43, bias=True),
]


def _operands(w4, cases, act="bf16"):
    drawn = [synthetic.draw(c, act=act) for c in cases]
    q = w4.w4a16_quantize_grouped([W.cuda() for W, _, _ in drawn])
    return drawn, q


def _reference(A, packed, scales, b, act="bf16", rows=None):
    s = scales.cpu().view(torch.int16).numpy().view(np.uint16)
    K, N = s.shape[0] * 128, s.shape[1]
    p = oracle.from_tile_layout(packed.cpu().numpy(), N, K)
    return oracle.gemm(bits(A), p, s, None if b is None else bits(b), rows=rows, act=act)


def test_grouped_quantize_is_bit_exact(w4):
    cases = synthetic.WORKLOADS["expert_m50"] + [synthetic.Case("ragged", 1, 136, 384, 44, "t4")]
    drawn, q = _operands(w4, cases)
    torch.cuda.synchronize()
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
    for (W, _, _), (packed, scales) in zip(drawn, q):
        check_quantize_exact(W, packed, scales)


@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_grouped_gemm_every_variant(w4, act):
    drawn, q = _operands(w4, MIXED, act)
    refs = [_reference(A, p, s, b, act) for (_, A, b), (p, s) in zip(drawn, q)]
    As = [A.cuda() for _, A, _ in drawn]
    bs = [None if b is None else b.cuda() for _, _, b in drawn]
    for v in range(w4.w4a16_variant_count()):
        if "csk" in w4.w4a16_variant_name(v) or not all(
                w4.w4a16_variant_eligible(v, c.M, c.N, c.K) for c in MIXED):
            continue   # cluster split-K runs single problems only
        Ys = w4.w4a16_gemm_grouped(As, [p for p, _ in q], [s for _, s in q], biases=bs, variant=v)
        assert w4.w4a16_get_device_error() == w4.W4A16_OK, w4.w4a16_variant_name(v)
        for c, Y, ref in zip(MIXED, Ys, refs):
            check_gemm_close(Y, ref, what=f"{w4.w4a16_variant_name(v)} {c.name} {act}")


# the action-expert block's projections and a ragged one, at decode sizes
SMALL = [(2048, 1024), (1024, 1024), (8192, 1024), (1024, 4096), (136, 384)]


@pytest.mark.parametrize("M,act", [(1, "bf16"), (3, "bf16"), (8, "bf16"), (16, "bf16"), (5, "f16"),
                                   (13, "f16")])
def test_grouped_small_m_row_block(w4, M, act):
    """Projections of a decode step (M <= 16) in one grouped launch of the
    row-block kernel (problem i on its own sub-grid, persistent form):
    every eligible rb variant against the oracle, bit-identical repeats, and
    the library's own plan."""
    cases = [synthetic.Case(f"gs_m{M}_{n}x{k}", M, n, k, 60 + i, "t4" if i % 2 else "normal",
                            bias=(i % 2 == 0)) for i, (n, k) in enumerate(SMALL)]
    drawn, q = _operands(w4, cases, act)
    refs = [_reference(A, p, s, b, act) for (_, A, b), (p, s) in zip(drawn, q)]
    As = [A.cuda() for _, A, _ in drawn]
    bs = [None if b is None else b.cuda() for _, _, b in drawn]
    ps, ss = [p for p, _ in q], [s for _, s in q]
    ran = 0
    for v in range(w4.w4a16_variant_count()):
        name = w4.w4a16_variant_name(v)
        if not name.startswith("rb_") or not all(w4.w4a16_variant_eligible(v, c.M, c.N, c.K) for c in cases):
            continue
        Y1 = w4.w4a16_gemm_grouped(As, ps, ss, biases=bs, variant=v)
        Y2 = w4.w4a16_gemm_grouped(As, ps, ss, biases=bs, variant=v)
        torch.cuda.synchronize()
        assert w4.w4a16_get_device_error() == w4.W4A16_OK, name
        for c, ya, yb, ref in zip(cases, Y1, Y2, refs):
            check_gemm_close(ya, ref, what=f"{name} {c.name} {act}")
            assert torch.equal(ya.view(torch.int16), yb.view(torch.int16)), f"{name} {c.name}"
        ran += 1
    assert ran >= 1
    Ys = w4.w4a16_gemm_grouped(As, ps, ss, biases=bs)
    torch.cuda.synchronize()
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
    for c, y, ref in zip(cases, Ys, refs):
        check_gemm_close(y, ref, what=f"default plan {c.name} {act}")


def test_grouped_expert_block_default_variant(w4):
    cases = synthetic.WORKLOADS["expert_m50"]
    drawn, q = _operands(w4, cases)
    Ys = w4.w4a16_gemm_grouped([A.cuda() for _, A, _ in drawn], [p for p, _ in q], [s for _, s in q])
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
    for c, (_, A, b), (p, s), Y in zip(cases, drawn, q, Ys):
        check_gemm_close(Y, _reference(A, p, s, b), what=c.name)


def test_group_of_one_matches_single_call(w4):
    case = synthetic.Case("one", 64, 2048, 2048, 45, bias=True)
    (W, A, b), = [synthetic.draw(case)]
    packed, scales = w4.w4a16_quantize(W.cuda())
    for name in ("tc_a16_grp_sk", "tc_a64_deq_sk", "tc_a256_deq_sk"):
        v = w4.variant_id(name)
        Y1 = w4.w4a16_gemm(A.cuda(), packed, scales, bias=b.cuda(), variant=v)
        Yg, = w4.w4a16_gemm_grouped([A.cuda()], [packed], [scales], biases=[b.cuda()], variant=v)
        torch.cuda.synchronize()
        assert torch.equal(Y1, Yg), name


def test_grouped_split_k_on_fresh_workspaces(w4):
    # every problem split over its sub-grid; partial slots start as NaN
    cases = [synthetic.Case("s0", 16, 256, 16384, 46), synthetic.Case("s1", 50, 1024, 4096, 47, bias=True),
             synthetic.Case("s2", 1, 512, 8192, 48, bias=True)]
    drawn, q = _operands(w4, cases)
    refs = [_reference(A, p, s, b) for (_, A, b), (p, s) in zip(drawn, q)]
    As = [A.cuda() for _, A, _ in drawn]
    bs = [None if b is None else b.cuda() for _, _, b in drawn]
    probs = [(p, s) for p, s in q]
    for name in ("tc_a16_grp_sk", "tc_a64_deq_sk"):
        v = w4.variant_id(name)
        P, _, _ = w4._gemm_problems(As, [p for p, _ in probs], [s for _, s in probs], bs, None)
        need = w4.lib().w4a16_gemm_grouped_workspace_bytes(P, len(cases), v)
        assert need > 8192
        for _ in range(2):
            ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
            ws[8192:].fill_(0xFF)   # partial slots (after the 8 KiB counter region)
            Ys = w4.w4a16_gemm_grouped(As, [p for p, _ in probs], [s for _, s in probs], biases=bs,
                                       workspace=ws, variant=v)
            assert w4.w4a16_get_device_error() == w4.W4A16_OK, name
            for c, Y, ref in zip(cases, Ys, refs):
                check_gemm_close(Y, ref, what=f"{name} {c.name}")
