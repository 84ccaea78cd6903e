"""Cluster split-K: a tile's K range split over the CTAs of one thread-block
cluster, the partials summed through distributed shared memory in rank (k)
order.  Checked three ways: integer-valued inputs, for which every partial
and every order of summing is exact (so a partial missed, summed twice or
read from the wrong rank changes the bits); random inputs against the oracle
at the GEMM tolerance; and repeated launches, which must give the same bits
(the order of the sum does not depend on timing)."""

import numpy as np
import pytest
import torch

from gpu_helpers import bits, check_gemm_close
from test_gpu_gemm import make_operands, reference
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu


def csk_variants(w4, M, N, K):
    return [v for v in range(w4.w4a16_variant_count())
            if "csk" in w4.w4a16_variant_name(v) and w4.w4a16_variant_eligible(v, M, N, K)]


@pytest.mark.parametrize("M,N,K", [(50, 1024, 4096), (1, 2048, 8192), (64, 256, 2048), (130, 384, 1024)])
def test_cluster_splitk_integer_exact(w4, M, N, K):
    rng = np.random.default_rng(M + N + K)
    codes = rng.integers(-3, 4, size=(N, K))
    codes[:, ::128] = 7
    e = rng.integers(-3, 0, size=(N, K // 128))
    x = (codes * np.repeat(2.0 ** e, 128, axis=1)).astype(np.float32)
    a = rng.integers(-1, 2, size=(M, K)).astype(np.float32)
    W = synthetic.to_bf16(x).cuda()
    Ad = synthetic.to_bf16(a).cuda()
    b = synthetic.to_bf16(rng.integers(-4, 5, size=N).astype(np.float32)).cuda()
    packed, scales = w4.w4a16_quantize(W)
    exact = a.astype(np.float64) @ x.astype(np.float64).T + b.float().cpu().numpy()[None, :]
    assert np.all(exact == np.round(exact * 8) / 8) and np.abs(exact).max() < 2 ** 20
    expected = bits(synthetic.to_bf16(exact.astype(np.float32)))
    vs = csk_variants(w4, M, N, K)
    assert vs, "no cluster split-K variant is eligible"
    for v in vs:
        assert w4.w4a16_variant_workspace_bytes(v, M, N, K) == 0
        for _ in range(2):
            Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            w4.w4a16_gemm(Ad, packed, scales, bias=b, Y=Y, variant=v)
            torch.cuda.synchronize()
            assert np.array_equal(bits(Y), expected), w4.w4a16_variant_name(v)
    assert w4.w4a16_get_device_error() == w4.W4A16_OK


@pytest.mark.parametrize("case", [
    synthetic.Case("csk_down_m50", 50, 1024, 4096, 4, bias=True),
    synthetic.Case("csk_m1_n2048_k16384", 1, 2048, 16384, 0),
    synthetic.Case("csk_m17_ragged", 17, 136, 4096, 15, "t4", bias=True),
], ids=lambda c: c.name)
def test_cluster_splitk_matches_oracle_and_repeats(w4, case):
    W, A, b, packed, scales = make_operands(w4, case)
    y_ref = reference(A, packed, scales, b)
    Ad, bd = A.cuda(), None if b is None else b.cuda()
    for v in csk_variants(w4, case.M, case.N, case.K):
        Y1 = w4.w4a16_gemm(Ad, packed, scales, bias=bd, variant=v)
        Y2 = w4.w4a16_gemm(Ad, packed, scales, bias=bd, variant=v)
        torch.cuda.synchronize()
        check_gemm_close(Y1, y_ref, what=w4.w4a16_variant_name(v))
        assert torch.equal(Y1, Y2), w4.w4a16_variant_name(v)
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
