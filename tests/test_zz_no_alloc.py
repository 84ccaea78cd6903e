"""The allocation-free GEMM entry point, called through the C ABI, gives the
same result as the regular entry point (which gets its workspace from the
caller), on two calls in a row.

Some callers cannot allocate device memory (their memory belongs to another
allocator, or allocation is forbidden once a control loop runs); for them
w4a16_gemm_noalloc keeps its split-K scratch in a static device array.  This
file is named to be collected last, so that a run stopping at the first
failure has run every other test before it."""

import ctypes

import pytest
import torch

from gpu_helpers import check_gemm_close
from test_gpu_gemm import reference
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu


def test_noalloc_matches_regular_entry_point_twice(w4):
    L = w4.lib()
    # a stream-K variant for this shape, so that the call uses the scratch
    # (the library's own choice for a shape may need none)
    case = synthetic.Case("noalloc_m16_n2048_k2048", 16, 2048, 2048, 41, bias=True)
    M, N, K = case.M, case.N, case.K
    w4.w4a16_table_set(M, N, K, w4.variant_id("tc_a16_grp_sk"))
    assert w4.w4a16_gemm_workspace_bytes(M, N, K) > 0
    W, A, b = synthetic.draw(case)
    packed, scales = w4.w4a16_quantize(W.cuda())
    Ad, bd = A.cuda(), b.cuda()
    y_regular = w4.w4a16_gemm(Ad, packed, scales, bias=bd)
    stream = torch.cuda.current_stream().cuda_stream
    y_ref = reference(A, packed, scales, b)
    for call in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = L.w4a16_gemm_noalloc(ctypes.c_void_p(Ad.data_ptr()), M, N, K,
                                  ctypes.c_void_p(packed.data_ptr()),
                                  ctypes.c_void_p(scales.data_ptr()), 128,
                                  ctypes.c_void_p(bd.data_ptr()), ctypes.c_void_p(Y.data_ptr()),
                                  ctypes.c_void_p(stream))
        assert st == w4.W4A16_OK, (call, w4.status_string(st), L.w4a16_last_error_detail())
        torch.cuda.synchronize()
        # same tolerance as every GEMM test, against the regular entry point's output
        check_gemm_close(Y, y_regular.float().cpu().numpy(), what=f"noalloc call {call}")
        check_gemm_close(Y, y_ref, what=f"noalloc call {call} vs oracle")
    assert w4.w4a16_get_device_error() == w4.W4A16_OK
    w4.w4a16_table_clear()


def test_noalloc_rejects_shapes_beyond_its_scratch(w4):
    L = w4.lib()
    # a shape whose selected variant needs more than the 16 MiB static
    # scratch: searched, so that the rejection path is always exercised
    limit = 16 << 20
    over = [(M, N, K) for M in (816, 2048, 4096, 8192) for (N, K) in
            ((2048, 16384), (1024, 65536), (2048, 65536), (4096, 32768))
            if w4.w4a16_gemm_workspace_bytes(M, N, K) > limit]
    assert over, "no searched shape needs more scratch than the static array holds"
    M, N, K = over[0]
    # real (zero) buffers, although the call must return before any launch
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    packed = torch.zeros(w4.w4a16_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    scales = torch.ones(K // 128, N, dtype=torch.float16, device="cuda")
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    st = L.w4a16_gemm_noalloc(ctypes.c_void_p(A.data_ptr()), M, N, K,
                              ctypes.c_void_p(packed.data_ptr()), ctypes.c_void_p(scales.data_ptr()),
                              128, None, ctypes.c_void_p(Y.data_ptr()),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == w4.W4A16_ERR_WORKSPACE
    assert b"scratch" in L.w4a16_last_error_detail()
