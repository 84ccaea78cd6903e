"""Measured selection for the SwiGLU, INT8 and FP4 catalogues ("Kernel
dispatch and Humming quantization in PhyAI", section "Keep selection work out
of repeated inference": prepared kernel choices are tuned and memoized): each
tuner stores its measured choice, the public GEMM then uses it, and the
result still matches the oracle."""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bits, check_gemm_close
from test_gpu_gemm import make_operands, reference
from weight_only_int4_rtn_gb300 import synthetic

pytestmark = pytest.mark.gpu


def test_tuned_swiglu(w4):
    case = synthetic.Case("tune_sw_m50_n2048_k1024", 50, 2048, 1024, 3, bias=True)
    v = w4.w4a16_tune_swiglu(case.M, case.N, case.K)
    assert w4.w4a16_variant_eligible(v, case.M, case.N, case.K)
    assert not w4.w4a16_variant_name(v).startswith(("simt_", "rb_"))
    W, A, b, packed, scales = make_operands(w4, case)
    Yh = w4.w4a16_gemm_swiglu(A.cuda(), packed, scales, bias=b.cuda())
    Yv = w4.w4a16_gemm_swiglu(A.cuda(), packed, scales, bias=b.cuda(), variant=v)
    torch.cuda.synchronize()
    # the public call took the tuned variant: identical bits
    assert torch.equal(Yh, Yv)
    y = reference(A, packed, scales, b).astype(np.float64)
    h_ref = oracle.swiglu(y)
    # the GEMM tolerance carried through silu(g) u (the SwiGLU tests' bound)
    up, gate = y[:, 0::2], y[:, 1::2]
    rms = float(np.sqrt(np.mean(y ** 2)))
    sig = 1.0 / (1.0 + np.exp(-gate))
    tol_g, tol_u = 1e-2 * np.abs(gate) + 1e-2 * rms, 1e-2 * np.abs(up) + 1e-2 * rms
    lim = (np.abs(sig * (1.0 + gate * (1.0 - sig)) * up) * tol_g + 0.25 * tol_g ** 2 * np.abs(up)
           + (np.abs(gate * sig) + 1.1 * tol_g) * tol_u + 2.0 ** -8 * np.abs(h_ref))
    assert np.all(np.abs(Yh.float().cpu().numpy() - h_ref) <= lim)


def test_tuned_int8(w4):
    L = w4.lib()
    M, N, K = 16, 2048, 2048
    v = w4.w8a16_tune(M, N, K)
    assert L.w8a16_select_variant(M, N, K) == v
    W, A, _ = synthetic.draw(synthetic.Case("tune8", M, N, K, 5))
    packed, scales = w4.w8a16_quantize(W.cuda())
    Y = w4.w8a16_gemm(A.cuda(), packed, scales)
    torch.cuda.synchronize()
    p_ref, s_ref = oracle.quantize8(bits(W))
    check_gemm_close(Y, oracle.gemm8(bits(A), p_ref, s_ref), what="tuned int8")


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_tuned_fp4(w4, fmt):
    L = w4.lib()
    M, N, K = 16, 2048, 2048
    v = w4.fp4a16_tune(M, N, K, fmt)
    assert L.fp4a16_select_variant(M, N, K) == v
    W, A, _ = synthetic.draw(synthetic.Case("tunef4", M, N, K, 6))
    packed, scales, ts = w4.fp4a16_quantize(W.cuda(), fmt)
    Y = w4.fp4a16_gemm(A.cuda(), packed, scales, fmt, tensor_scale=ts)
    torch.cuda.synchronize()
    wf = oracle.bf16_bits_to_f32(bits(W))
    if fmt == "mxfp4":
        p, s = oracle.quantize_mxfp4_f32(wf)
        wd = oracle.dequantize_mxfp4(p, s)
    else:
        p, s, g = oracle.quantize_nvfp4_f32(wf)
        wd = oracle.dequantize_nvfp4(p, s, g)
    check_gemm_close(Y, oracle.gemm_fp4(bits(A), wd), what=f"tuned {fmt}")
