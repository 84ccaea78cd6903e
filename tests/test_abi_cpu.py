"""The C ABI loads, exports what include/w4a16.h declares, and rejects bad
arguments from metadata alone (no GPU needed: nothing here launches)."""

import ctypes
import os
import re

import pytest

import weight_only_int4_rtn_gb300 as w4

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "w4a16.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:w[48]|fp4)a16_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("w4a16_quantize", "w4a16_gemm", "w4a16_tune", "w4a16_get_device_error",
                     "w4a16_status_string", "w4a16_packed_bytes", "w4a16_scales_bytes",
                     "w4a16_gemm_workspace_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol(built_lib):
    handle = ctypes.CDLL(built_lib)
    missing = [n for n in declared_functions() if not hasattr(handle, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    bound = {name for name, _, _ in w4.SIGNATURES}
    assert set(declared_functions()) == bound


def test_sizes(built_lib):
    assert w4.w4a16_packed_bytes(256, 512) == 256 * 256
    assert w4.w4a16_packed_bytes(264, 512) == 384 * 256     # rows padded to whole 128-row tiles
    assert w4.w4a16_scales_bytes(256, 512) == 4 * 256 * 2
    assert w4.w4a16_scales_bytes(256, 512, 64) == 0
    assert w4.lib().fp4a16_packed_bytes(256, 512) == 256 * 256
    assert w4.lib().fp4a16_scales_bytes(1, 256, 512) == 16 * 256      # MXFP4: K/32 bytes per row
    assert w4.lib().fp4a16_scales_bytes(2, 256, 512) == 32 * 256      # NVFP4: K/16 bytes per row
    assert w4.lib().fp4a16_scales_bytes(3, 256, 512) == 0


def test_status_strings(built_lib):
    for st in range(8):
        assert w4.status_string(st).startswith("W4A16_")
    assert "unknown" in w4.status_string(99)


def _gemm(L, **kw):
    args = dict(A=16, M=4, N=256, K=512, packed=16, scales=16, group=128, bias=None, Y=16,
                ws=None, ws_bytes=0, stream=None)
    args.update(kw)
    return L.w4a16_gemm(args["A"], args["M"], args["N"], args["K"], args["packed"], args["scales"],
                        args["group"], args["bias"], args["Y"], args["ws"], args["ws_bytes"],
                        args["stream"])


def test_gemm_argument_errors_before_any_launch(built_lib):
    L = w4.lib()
    assert _gemm(L, A=None) == w4.W4A16_ERR_INVALID_ARG
    assert _gemm(L, Y=None) == w4.W4A16_ERR_INVALID_ARG
    assert _gemm(L, M=0) == w4.W4A16_ERR_INVALID_ARG
    assert _gemm(L, group=64) == w4.W4A16_ERR_UNSUPPORTED
    assert _gemm(L, K=500) == w4.W4A16_ERR_UNSUPPORTED
    assert _gemm(L, N=250) == w4.W4A16_ERR_UNSUPPORTED
    assert _gemm(L, A=18) == w4.W4A16_ERR_ALIGNMENT
    assert _gemm(L, packed=8) == w4.W4A16_ERR_ALIGNMENT
    assert _gemm(L, bias=4) == w4.W4A16_ERR_ALIGNMENT
    assert _gemm(L, Y=2) == w4.W4A16_ERR_ALIGNMENT


def test_quantize_argument_errors_before_any_launch(built_lib):
    L = w4.lib()
    assert L.w4a16_quantize(None, 256, 512, 128, 16, 16, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_quantize(16, 256, 512, 32, 16, 16, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_quantize(16, 256, 130, 128, 16, 16, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_quantize(16, 12, 512, 128, 16, 16, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_quantize(17, 256, 512, 128, 16, 16, None) == w4.W4A16_ERR_ALIGNMENT
    assert L.w4a16_quantize(16, 256, 512, 128, 16, 24, None) == w4.W4A16_ERR_ALIGNMENT


def test_fp4_argument_errors_before_any_launch(built_lib):
    L = w4.lib()
    # quantize: format, nulls (NVFP4 needs the tensor-scale pair), sizes, alignment
    assert L.fp4a16_quantize(3, 16, 256, 512, 16, 16, 16, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.fp4a16_quantize(1, None, 256, 512, 16, 16, None, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.fp4a16_quantize(2, 16, 256, 512, 16, 16, None, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.fp4a16_quantize(1, 16, 264, 512, 16, 16, None, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.fp4a16_quantize(1, 16, 256, 500, 16, 16, None, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.fp4a16_quantize(1, 24, 256, 512, 16, 16, None, None) == w4.W4A16_ERR_ALIGNMENT
    assert L.fp4a16_quantize(2, 16, 256, 512, 16, 16, 20, None) == w4.W4A16_ERR_ALIGNMENT
    # GEMM: format, NVFP4 without its tensor scale, N % 16, alignment
    g = lambda f, N=256, ts=16, A=16: L.fp4a16_gemm(f, A, 4, N, 512, 16, 16, ts, None, 16, None, 0, None)
    assert g(0) == w4.W4A16_ERR_UNSUPPORTED
    assert g(2, ts=None) == w4.W4A16_ERR_INVALID_ARG
    assert g(1, N=264) == w4.W4A16_ERR_UNSUPPORTED
    assert g(1, A=18) == w4.W4A16_ERR_ALIGNMENT
    assert g(2, ts=18) == w4.W4A16_ERR_ALIGNMENT
    assert L.fp4a16_gemm_workspace_bytes(5, 1, 256, 512) == 0


def test_swiglu_argument_errors_before_any_launch(built_lib):
    L = w4.lib()
    names = [w4.w4a16_variant_name(i) for i in range(w4.w4a16_variant_count())]
    args = (16, 4, 256, 512, 16, 16, 128, None, 16, None, 0, None)
    simt = [i for i, n in enumerate(names) if n.startswith(("simt_", "rb_"))]
    assert simt
    for v in simt:   # the streaming variants have no SwiGLU epilogue
        assert L.w4a16_gemm_swiglu_variant(v, *args) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_gemm_swiglu_variant(len(names), *args) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_gemm_swiglu(16, 4, 250, 512, 16, 16, 128, None, 16, None, 0, None) == \
        w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_gemm_swiglu(18, 4, 256, 512, 16, 16, 128, None, 16, None, 0, None) == \
        w4.W4A16_ERR_ALIGNMENT
    assert L.w4a16_gemm_swiglu(None, 4, 256, 512, 16, 16, 128, None, 16, None, 0, None) == \
        w4.W4A16_ERR_INVALID_ARG


def test_variant_catalogue_is_host_only(built_lib):
    n = w4.w4a16_variant_count()
    assert n >= 4
    names = [w4.w4a16_variant_name(i) for i in range(n)]
    assert len(set(names)) == n and all(names)
    assert w4.w4a16_variant_name(n) is None
    for i in range(n):
        # the CUDA-core streaming variants take M up to their own tile
        m = int(names[i].split("_")[1][1:]) if names[i].startswith(("simt_", "rb_")) else 16
        assert w4.w4a16_variant_eligible(i, m, 256, 512)
        assert not w4.w4a16_variant_eligible(i, m, 256, 500)
        assert not names[i].startswith(("simt_", "rb_")) or not w4.w4a16_variant_eligible(i, m + 1, 256, 512)
    for M in (1, 4, 16, 50, 64, 816, 8192):
        v = w4.w4a16_select_variant(M, 8192, 8192)
        assert 0 <= v < n


def test_table_roundtrip(built_lib, tmp_path):
    w4.w4a16_table_clear()
    rule = w4.w4a16_select_variant(50, 2048, 1024)
    v = w4.variant_id("tc_a16_grp_sk")
    assert v != rule
    w4.w4a16_table_set(50, 2048, 1024, v)
    assert w4.w4a16_select_variant(50, 2048, 1024) == v
    p = str(tmp_path / "table.txt")
    w4.w4a16_table_save(p)
    w4.w4a16_table_clear()
    assert w4.w4a16_select_variant(50, 2048, 1024) == rule
    w4.w4a16_table_load(p)
    assert w4.w4a16_select_variant(50, 2048, 1024) == v
    with open(p, "a") as f:
        f.write("16 256 512 no_such_variant\n")
    with pytest.raises(w4.W4A16Error):
        w4.w4a16_table_load(p)
    w4.w4a16_table_clear()


def test_binding_rejects_cpu_tensors(built_lib):
    import torch
    W = torch.zeros(256, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        w4.w4a16_quantize(W)


def test_group_structs_match_the_header():
    # five pointers, three int64 and the int epilogue (padded to 8 bytes)
    assert ctypes.sizeof(w4.GemmProblem) == 5 * 8 + 3 * 8 + 8
    assert w4.GemmProblem.epilogue.offset == 64
    assert ctypes.sizeof(w4.QuantizeProblem) == 8 + 2 * 8 + 2 * 8
    text = open(HEADER).read()
    assert "#define W4A16_MAX_GROUP 8" in text and w4.MAX_GROUP == 8


def test_grouped_argument_errors_before_launch(built_lib):
    L = w4.lib()
    P = (w4.GemmProblem * 9)()
    for i in range(9):
        P[i] = w4.GemmProblem(16, 16, 16, None, 16, 4, 256, 512)
    assert L.w4a16_gemm_grouped(P, 0, 128, 0, -1, None, 0, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_gemm_grouped(P, 9, 128, 0, -1, None, 0, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_gemm_grouped(P, 2, 64, 0, -1, None, 0, None) == w4.W4A16_ERR_UNSUPPORTED
    P[1] = w4.GemmProblem(16, 16, 16, None, 16, 4, 256, 500)      # K not a multiple of 128
    assert L.w4a16_gemm_grouped(P, 2, 128, 0, -1, None, 0, None) == w4.W4A16_ERR_UNSUPPORTED
    P[1] = w4.GemmProblem(24, 16, 16, None, 16, 4, 256, 512)      # A not 16-byte aligned
    assert L.w4a16_gemm_grouped(P, 2, 128, 0, -1, None, 0, None) == w4.W4A16_ERR_ALIGNMENT
    Q = (w4.QuantizeProblem * 2)()
    Q[0] = w4.QuantizeProblem(16, 256, 512, 16, 16)
    Q[1] = w4.QuantizeProblem(16, 250, 512, 16, 16)               # N not a multiple of 8
    assert L.w4a16_quantize_grouped(Q, 2, 128, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_quantize_grouped(Q, 0, 128, None) == w4.W4A16_ERR_INVALID_ARG


def test_rowmajor_sizes(built_lib):
    L = w4.lib()
    assert L.w4a16_packed_rowmajor_bytes(256, 512) == 256 * 256
    assert L.w4a16_packed_rowmajor_bytes(264, 512) == 264 * 256   # no padding rows
    assert L.w4a16_packed_rowmajor_bytes(-1, 512) == 0


def test_repack_argument_errors_before_any_launch(built_lib):
    L = w4.lib()
    assert L.w4a16_repack_rowmajor(None, 256, 512, 16, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_repack_rowmajor(16, 256, 512, None, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_repack_rowmajor(16, 0, 512, 16, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_repack_rowmajor(16, 256, 500, 16, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_repack_rowmajor(16, 250, 512, 16, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_repack_rowmajor(8, 256, 512, 16, None) == w4.W4A16_ERR_ALIGNMENT
    assert L.w4a16_repack_rowmajor(16, 256, 512, 24, None) == w4.W4A16_ERR_ALIGNMENT


def test_quotient_selftest_argument_errors(built_lib):
    L = w4.lib()
    assert L.w4a16_selftest_quotient(0, None, None) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_selftest_quotient(3, 16, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_selftest_quotient(-1, 16, None) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w4a16_selftest_quotient(0, 12, None) == w4.W4A16_ERR_ALIGNMENT


def test_table_roundtrip_every_catalogue(built_lib, tmp_path):
    """Entries of the INT4, SwiGLU, INT8 and FP4 catalogues are kept apart,
    selected, saved and loaded back (no GPU: selection is host logic)."""
    L = w4.lib()
    w4.w4a16_table_clear()
    M, N, K = 16, 2048, 2048
    rule4, rule_sw = w4.w4a16_select_variant(M, N, K), None
    rule8 = L.w8a16_select_variant(M, N, K)
    rulef4 = L.fp4a16_select_variant(M, N, K)
    v4 = w4.variant_id("tc_a32_grp_sk")
    vsw = w4.variant_id("tc_a64_deq2_sk")
    v8 = next(i for i in range(L.w8a16_variant_count())
              if L.w8a16_variant_eligible(i, M, N, K) and i != rule8)
    vf4 = next(i for i in range(L.fp4a16_variant_count())
               if L.fp4a16_variant_eligible(i, M, N, K) and i != rulef4)
    w4.w4a16_table_set(M, N, K, v4)
    w4.w4a16_swiglu_table_set(M, N, K, vsw)
    w4.w8a16_table_set(M, N, K, v8)
    w4.fp4a16_table_set(M, N, K, vf4)
    assert w4.w4a16_select_variant(M, N, K) == v4
    assert L.w8a16_select_variant(M, N, K) == v8
    assert L.fp4a16_select_variant(M, N, K) == vf4
    p = str(tmp_path / "table_all.txt")
    w4.w4a16_table_save(p)
    text = open(p).read()
    assert "swiglu 16 2048 2048 tc_a64_deq2_sk" in text
    assert f"int8 16 2048 2048 {L.w8a16_variant_name(v8).decode()}" in text
    assert f"fp4 16 2048 2048 {L.fp4a16_variant_name(vf4).decode()}" in text
    w4.w4a16_table_clear()
    assert w4.w4a16_select_variant(M, N, K) == rule4
    assert L.w8a16_select_variant(M, N, K) == rule8
    assert L.fp4a16_select_variant(M, N, K) == rulef4
    w4.w4a16_table_load(p)
    assert w4.w4a16_select_variant(M, N, K) == v4
    assert L.w8a16_select_variant(M, N, K) == v8
    assert L.fp4a16_select_variant(M, N, K) == vf4
    # a variant of another catalogue is refused
    with pytest.raises(w4.W4A16Error):
        w4.w8a16_table_set(M, N, K, 10 ** 6)
    with open(p, "a") as f:
        f.write("int8 16 256 512 tc_a16_grp_sk\n")   # an INT4 name in the INT8 catalogue
    with pytest.raises(w4.W4A16Error):
        w4.w4a16_table_load(p)
    with open(p, "w") as f:
        f.write("nosuchtag 16 256 512 tc_a16_grp_sk\n")
    with pytest.raises(w4.W4A16Error):
        w4.w4a16_table_load(p)
    w4.w4a16_table_clear()
    del rule_sw


def test_tuners_refuse_bad_shapes(built_lib):
    L = w4.lib()
    out = ctypes.c_int(-1)
    assert L.w4a16_tune_swiglu(16, 250, 512, None, ctypes.byref(out)) == w4.W4A16_ERR_UNSUPPORTED
    assert L.w8a16_tune(16, 256, 500, None, ctypes.byref(out)) == w4.W4A16_ERR_UNSUPPORTED
    assert L.fp4a16_tune(1, 16, 264, 512, None, ctypes.byref(out)) == w4.W4A16_ERR_UNSUPPORTED
    assert L.fp4a16_tune(7, 16, 256, 512, None, ctypes.byref(out)) == w4.W4A16_ERR_UNSUPPORTED


def test_grouped_epilogue_argument_errors(built_lib):
    L = w4.lib()
    P = (w4.GemmProblem * 2)()
    P[0] = w4.GemmProblem(16, 16, 16, None, 16, 4, 256, 512, 0)
    P[1] = w4.GemmProblem(16, 16, 16, None, 16, 4, 256, 512, 2)        # no such epilogue
    assert L.w4a16_gemm_grouped(P, 2, 128, 0, -1, None, 0, None) == w4.W4A16_ERR_UNSUPPORTED
    P[1] = w4.GemmProblem(16, 16, 16, None, 16, 4, 264, 512, 1)        # SwiGLU needs N even...
    P[1].N = 260
    assert L.w4a16_gemm_grouped(P, 2, 128, 0, -1, None, 0, None) == w4.W4A16_ERR_UNSUPPORTED
    P[1] = w4.GemmProblem(16, 16, 16, None, 16, 4, 256, 512, 1)
    assert L.w4a16_gemm_grouped(P, 2, 128, 1, -1, None, 0, None) == w4.W4A16_ERR_UNSUPPORTED  # fp16


def test_row_block_schedule_forms(built_lib):
    """The row-block kernel's launch form chosen by the host cost model (on a
    152-SM GB300): the busiest SM's group-items at 16 per unit of time with
    two busy CTAs and 8 / 0.65 with one, the cluster split at 1.3 items a
    wave (items at 1.4 when its clusters put two CTAs on an SM).  Each team size and the cluster form is the choice for some
    shape."""
    rb1 = w4.variant_id("rb_m1")
    sched = lambda N, K: w4.w4a16_variant_schedule(rb1, 1, N, K, 152)
    # K/128 groups bound the team: one group (team 1) up to eight (team 8)
    assert sched(4096, 128)["team"] == 1 and sched(4096, 128)["grid"] == 16
    assert sched(4096, 256)["team"] == 2 and sched(4096, 256)["grid"] == 32
    assert sched(4096, 512)["team"] == 4 and sched(4096, 512)["grid"] == 64
    assert sched(4096, 1024) == dict(grid=128, dp_tiles=0, sk_units=0, cluster=1, team=8)
    # the metric's sweep shapes: the measured-best forms
    assert sched(8192, 8192) == dict(grid=256, dp_tiles=0, sk_units=0, cluster=1, team=8)
    assert sched(16384, 2048) == dict(grid=256, dp_tiles=0, sk_units=0, cluster=1, team=4)
    assert sched(4096, 4096) == dict(grid=128, dp_tiles=0, sk_units=0, cluster=1, team=8)
    assert w4.w4a16_variant_workspace_bytes(rb1, 1, 8192, 8192) == 0
    # few row blocks, long K: a cluster K split (grid = row blocks x cluster)
    # (a split of 2 on 128 CTAs: measured 7.7 us against 8.2 us for 4 on 256)
    assert sched(2048, 16384) == dict(grid=128, dp_tiles=0, sk_units=0, cluster=2, team=8)
    assert sched(256, 4096) == dict(grid=32, dp_tiles=0, sk_units=0, cluster=4, team=8)
    assert sched(256, 16384) == dict(grid=64, dp_tiles=0, sk_units=0, cluster=8, team=8)
    # a tcgen05 variant reports no team; argument errors
    tc = w4.variant_id("tc_a16_grp_sk")
    assert w4.w4a16_variant_schedule(tc, 16, 8192, 8192, 152)["team"] == 0
    out = (ctypes.c_int * 5)()
    L = w4.lib()
    assert L.w4a16_variant_schedule(rb1, 2, 4096, 1024, 152, out) == w4.W4A16_ERR_NO_VARIANT
    assert L.w4a16_variant_schedule(rb1, 1, 4096, 1024, -1, out) == w4.W4A16_ERR_INVALID_ARG
    assert L.w4a16_variant_schedule(rb1, 1, 4096, 1024, 152, None) == w4.W4A16_ERR_INVALID_ARG


def test_row_block_two_column_tiles(built_lib):
    """rb_m16 (two MMA column tiles, one CTA of 8 warps per SM): persistent
    grids stay within the SMs, few row blocks with long K take the cluster
    split, and the rule leaves the sweep's M = 16 shapes, where it measured
    slower than the tcgen05 kernel, to the tcgen05 variants."""
    rb16 = w4.variant_id("rb_m16")
    assert w4.w4a16_variant_eligible(rb16, 16, 8192, 8192)
    assert not w4.w4a16_variant_eligible(rb16, 17, 8192, 8192)
    for N, K in ((8192, 8192), (16384, 2048), (28672, 4096), (4104, 1024)):
        s = w4.w4a16_variant_schedule(rb16, 16, N, K, 152)
        assert s["cluster"] == 1 and 1 <= s["grid"] <= 152, (N, K, s)
    assert w4.w4a16_variant_schedule(rb16, 16, 264, 16384, 152) == dict(
        grid=72, dp_tiles=0, sk_units=0, cluster=8, team=8)
    for N, K in ((16384, 2048), (2048, 16384), (8192, 8192)):
        name = w4.w4a16_variant_name(w4.w4a16_select_variant(16, N, K))
        assert name.startswith("tc_"), (N, K, name)
