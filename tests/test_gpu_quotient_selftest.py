"""The quantizer's division, exhaustively: the corrected reciprocal quotient
that every quantize mode uses against the IEEE division, on the device.

The codes must equal rint(fl32(w / s)) bit for bit (reading P2 of the
method: an IEEE fp32 division).  The kernels compute the quotient as a
reciprocal product plus one remainder correction; Markstein's theorem says
that is the correctly rounded quotient, and this test checks it on every
(scale, weight) pair the INT4 and INT8 modes can meet (every normal finite
fp16 scale, every finite bf16 weight within the code range), and on a fixed
sample of NVFP4 steps."""

import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,min_pairs", [(0, 10**9), (1, 10**9), (2, 10**8)])
def test_corrected_quotient_equals_ieee_division(w4, mode, min_pairs):
    checked, bad = w4.selftest_quotient(mode)
    assert checked >= min_pairs, checked
    assert bad == 0, f"{bad} of {checked} quotients differ from the IEEE division"
