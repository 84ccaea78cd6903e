"""Row-major packed codes -> tiled storage (w4a16_repack_rowmajor), byte for
byte against the oracle's own tiling of the same bytes, and the GEMM run on
the repacked codes.

"Kernel dispatch and Humming quantization in PhyAI", section "Humming makes
the separation useful": a packed INT4 layout runs only through the kernel
that understands it; the row-major [N, K/2] bytes are the plain interchange
form, and the repack is a pure permutation of them."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bits, check_gemm_close
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K", [(256, 512), (264, 384), (8, 128), (2048, 1024), (1032, 2176)])
def test_repack_matches_oracle_tiling(w4, N, K):
    rng = np.random.default_rng(N * 7 + K)
    rm = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    expect = oracle.to_tile_layout(rm)
    src = torch.from_numpy(rm).cuda()
    # poisoned output: padding rows must come back zero
    out = torch.full((w4.w4a16_packed_bytes(N, K),), 0xA5, dtype=torch.uint8, device="cuda")
    w4.w4a16_repack_rowmajor(src, N, K, packed=out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    bad = np.flatnonzero(got != expect)
    assert bad.size == 0, f"{bad.size} bytes differ, first offsets {bad[:4].tolist()}"


def test_gemm_on_repacked_oracle_codes(w4):
    case = synthetic.Case("repack_m16_n512_k1024", 16, 512, 1024, 9, bias=True)
    W, A, b = synthetic.draw(case)
    p_rm, s_ref = oracle.quantize(bits(W))
    packed = w4.w4a16_repack_rowmajor(torch.from_numpy(p_rm).cuda(), case.N, case.K)
    # the quantizer writes the same storage
    packed_q, _ = w4.w4a16_quantize(W.cuda())
    assert torch.equal(packed, packed_q)
    scales = torch.from_numpy(s_ref.view(np.int16)).view(torch.float16).cuda()
    Y = w4.w4a16_gemm(A.cuda(), packed, scales, bias=b.cuda())
    torch.cuda.synchronize()
    y_ref = oracle.gemm(bits(A), p_rm, s_ref, bits(b))
    check_gemm_close(Y, y_ref, what="gemm on repacked codes")
