"""Failure detection without a GPU fault: a bounded device-side wait that
nothing completes runs out, the kernel records W4A16_ERR_TIMEOUT and
returns, and the context stays usable."""

import pytest
import torch

from gpu_helpers import check_gemm_close
from test_gpu_gemm import make_operands, reference
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_cleared(w4):
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
    w4.w4a16_selftest_wait_timeout(2_000_000)        # 2 ms limit; nobody arrives
    assert w4.w4a16_get_device_error() == w4.W4A16_ERR_TIMEOUT
    assert w4.w4a16_get_device_error() == w4.W4A16_OK  # read clears it
    # the context still works
    case = synthetic.Case("after", 16, 256, 512, 7)
    W, A, b, packed, scales = make_operands(w4, case)
    Y = w4.w4a16_gemm(A.cuda(), packed, scales)
    torch.cuda.synchronize()
    check_gemm_close(Y, reference(A, packed, scales, b))


def test_graph_capture(w4):
    case = synthetic.Case("graph", 50, 1024, 1024, 8, bias=True)
    W, A, b, _, _ = make_operands(w4, case)
    Wd, Ad, bd = W.cuda(), A.cuda(), b.cuda()
    packed = torch.empty(w4.w4a16_packed_bytes(1024, 1024), dtype=torch.uint8, device="cuda")
    scales = torch.empty(8, 1024, dtype=torch.float16, device="cuda")
    Y = torch.empty(50, 1024, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(max(w4.w4a16_gemm_workspace_bytes(50, 1024, 1024), 16), dtype=torch.uint8,
                     device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):          # warm-up outside capture
        w4.w4a16_quantize(Wd, packed=packed, scales=scales)
        w4.w4a16_gemm(Ad, packed, scales, bias=bd, Y=Y, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    Y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w4.w4a16_quantize(Wd, packed=packed, scales=scales)
        w4.w4a16_gemm(Ad, packed, scales, bias=bd, Y=Y, workspace=ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    check_gemm_close(Y, reference(A, packed, scales, b))
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
