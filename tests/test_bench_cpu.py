"""Host logic of bench.py: the algorithmic bytes behind `value` and the
roofline, and the rule that ncu traffic is reported only for the kernel
sources it was taken on.  No GPU: bench.py imports without one."""

import os
import sys
from fractions import Fraction

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

# bytes per weight from the formats: a 4-bit code is 1/2 byte, an 8-bit code
# 1; an fp16 scale (2 bytes) per 128 weights, an E8M0 byte per 32 (MXFP4), an
# E4M3 byte per 16 (NVFP4)
STORED = {"int4": Fraction(1, 2) + Fraction(2, 128), "int8": 1 + Fraction(2, 128),
          "mxfp4": Fraction(1, 2) + Fraction(1, 32), "nvfp4": Fraction(1, 2) + Fraction(1, 16)}


@pytest.mark.parametrize("fmt", sorted(STORED))
def test_weight_and_gemm_bytes(fmt):
    N, K, M = 8192, 1024, 50
    assert Fraction(bench.weight_bytes(N, K, fmt)) == STORED[fmt] * N * K
    # the GEMM reads the stored weight and the bf16 activations
    assert Fraction(bench.gemm_bytes(M, N, K, fmt)) == STORED[fmt] * N * K + 2 * M * K
    assert bench.gemm_flops(M, N, K) == 2 * M * N * K


@pytest.mark.parametrize("fmt", sorted(STORED))
def test_quantize_bytes(fmt):
    N, K = 4096, 2048
    reads = 2 * (2 if fmt == "nvfp4" else 1)      # bf16 in; NVFP4 reads it twice
    assert Fraction(bench.quant_bytes(N, K, fmt)) == (reads + STORED[fmt]) * N * K


def test_quantize_bytes_per_weight_as_documented():
    # the per-weight figures the measurement notes quote
    per = {f: Fraction(bench.quant_bytes(128, 128, f)) / (128 * 128) for f in STORED}
    assert per == {"int4": Fraction(2515625, 1000000), "int8": Fraction(3015625, 1000000),
                   "mxfp4": Fraction(253125, 100000), "nvfp4": Fraction(45625, 10000)}


def test_traffic_only_for_the_recorded_sources(monkeypatch):
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")
    rows = [line.split() for line in open(path) if line.strip() and not line.startswith("#")]
    assert rows, "no traffic rows"
    kernel, workload, nbytes, src = rows[0][:4]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: src)
    assert bench.dram_traffic(kernel, workload) == float(nbytes)
    assert bench.dram_traffic(kernel, "no_such_workload") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 12)
    assert bench.dram_traffic(kernel, workload) is None


def test_source_hash_covers_every_kernel_source(tmp_path, monkeypatch):
    # the hash changes when the code of any .cu, .cuh or .h file under csrc
    # changes, and not when only a comment does
    h0 = bench.kernel_source_hash()
    csrc = os.path.join(bench.ROOT, "weight_only_int4_rtn_gb300", "csrc")
    names = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    real_open = open
    extra = {"text": ""}

    def fake_open(p, mode="r", *a, **k):
        f = real_open(p, mode, *a, **k)
        if "b" not in mode and os.path.basename(str(p)) == names[-1]:
            data = f.read() + extra["text"]
            f.close()
            import io
            return io.StringIO(data)
        return f

    monkeypatch.setattr("builtins.open", fake_open)
    extra["text"] = "\n// a comment only\n"
    assert bench.kernel_source_hash() == h0
    extra["text"] = "\nstatic int w4a16_probe_value = 1;\n"
    assert bench.kernel_source_hash() != h0
