"""SwiGLU inside the grouped launch: an MLP block's gate/up projection takes
the SwiGLU epilogue ("Piper Kernels", section "ConvRot INT8": SwiGLU of a raw
[up | gate] tensor; here its rows interleave up and gate) while the block's
other projections store their plain GEMM, all in one launch.  Each output is
checked against the oracle: the GEMM tolerance for the plain problems, the
same tolerance carried through silu(g) u for the SwiGLU one."""

import pytest
import torch

from test_gpu_grouped import _operands, _reference
from test_gpu_swiglu import check_swiglu_close
from gpu_helpers import check_gemm_close
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu

BLOCK = [
    synthetic.Case("qkv_m50", 50, 2048, 1024, 1),
    synthetic.Case("o_m50", 50, 1024, 1024, 2, bias=True),
    synthetic.Case("gate_up_m50", 50, 8192, 1024, 3, bias=True),   # the SwiGLU problem
    synthetic.Case("down_m50", 50, 1024, 4096, 4),
]
EPI = [0, 0, 1, 0]


def _check(w4, cases, drawn, q, Ys, what):
    for c, e, (_, A, b), (p, s), Y in zip(cases, EPI, drawn, q, Ys):
        ref = _reference(A, p, s, b)
        if e:
            assert Y.shape == (c.M, c.N // 2)
            check_swiglu_close(Y, ref, what=f"{what} {c.name}")
        else:
            check_gemm_close(Y, ref, what=f"{what} {c.name}")


def test_grouped_block_with_swiglu_every_variant(w4):
    drawn, q = _operands(w4, BLOCK)
    As = [A.cuda() for _, A, _ in drawn]
    bs = [None if b is None else b.cuda() for _, _, b in drawn]
    ran = 0
    for v in range(w4.w4a16_variant_count()):
        name = w4.w4a16_variant_name(v)
        if name.startswith(("simt_", "rb_")) or "csk" in name or not all(
                w4.w4a16_variant_eligible(v, c.M, c.N, c.K) for c in BLOCK):
            continue
        Ys = w4.w4a16_gemm_grouped(As, [p for p, _ in q], [s for _, s in q], biases=bs, variant=v,
                                   epilogues=EPI)
        torch.cuda.synchronize()
        assert w4.w4a16_get_device_error() == w4.W4A16_OK, name
        _check(w4, BLOCK, drawn, q, Ys, name)
        ran += 1
    assert ran >= 10


def test_grouped_block_with_swiglu_tuned_plan(w4):
    v = w4.w4a16_tune_grouped([(c.M, c.N, c.K, e) for c, e in zip(BLOCK, EPI)])
    assert not w4.w4a16_variant_name(v).startswith(("simt_", "rb_"))
    drawn, q = _operands(w4, BLOCK)
    Ys = w4.w4a16_gemm_grouped([A.cuda() for _, A, _ in drawn], [p for p, _ in q], [s for _, s in q],
                               biases=[None if b is None else b.cuda() for _, _, b in drawn],
                               epilogues=EPI)
    torch.cuda.synchronize()
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
    _check(w4, BLOCK, drawn, q, Ys, "tuned")


def test_grouped_swiglu_matches_single_launch_bits(w4):
    # the grouped SwiGLU output equals the single-problem SwiGLU launch of the
    # same variant bit for bit (same schedule: the problem alone in the group)
    c = BLOCK[2]
    drawn, q = _operands(w4, [c])
    (_, A, b), (p, s) = drawn[0], q[0]
    Ad, bd = A.cuda(), b.cuda()
    for v in (w4.variant_id("tc_a64_deq2_dp"), w4.variant_id("tc_a16_grp_sk")):
        Yg = w4.w4a16_gemm_grouped([Ad], [p], [s], biases=[bd], variant=v, epilogues=[1])[0]
        Ys = w4.w4a16_gemm_swiglu(Ad, p, s, bias=bd, variant=v)
        torch.cuda.synchronize()
        assert torch.equal(Yg, Ys), w4.w4a16_variant_name(v)
