"""Grouped-GEMM plan chosen by measurement ("Kernel dispatch and Humming
quantization in PhyAI", section "Keep selection work out of repeated
inference"): the tuned, memoized plan runs and matches the oracle."""

import pytest
import torch

from gpu_helpers import check_gemm_close
from test_gpu_grouped import _operands, _reference
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu


def test_tuned_grouped_expert_block(w4):
    cases = synthetic.WORKLOADS["expert_m50"]
    v = w4.w4a16_tune_grouped([(c.M, c.N, c.K) for c in cases])
    assert 0 <= v < w4.w4a16_variant_count()
    drawn, q = _operands(w4, cases)
    Ys = w4.w4a16_gemm_grouped([A.cuda() for _, A, _ in drawn], [p for p, _ in q], [s for _, s in q],
                               biases=[None if b is None else b.cuda() for _, _, b in drawn])
    torch.cuda.synchronize()
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
    for c, (_, A, b), (p, s), Y in zip(cases, drawn, q, Ys):
        check_gemm_close(Y, _reference(A, p, s, b), what=c.name)
