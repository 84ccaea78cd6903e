"""The quantizer's division, exhaustively: the corrected reciprocal quotient
that every quantize mode uses against the IEEE division, on the device.

The codes must equal rint(fl32(w / s)) bit for bit (reading P2 of the
method: an IEEE fp32 division, then rounding half to even).  The kernels
compute the quotient as a reciprocal product plus one remainder correction;
Markstein's theorem says that is the correctly rounded quotient wherever the
remainder is exact.  This test checks it on every (scale, weight) pair the
INT4 and INT8 modes can meet (every normal finite fp16 scale, every finite
bf16 weight within the code range):

* no stored code may differ (the bit-exactness claim);
* no quotient may differ where |w| >= 2^-100.  Below that the remainder can
  fall in the subnormal range and lose bits, so the quotient may be off by
  an ulp there, but such a quotient is far below 1/4 and its code is 0 on
  both sides (the first check).

With full fp32 divisors (the NVFP4 steps) the same correction does give
different codes on a fixed sample, which is why the NVFP4 quantize uses the
IEEE division instead."""

import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [0, 1])
def test_corrected_quotient_equals_ieee_division(w4, mode):
    c = w4.selftest_quotient(mode)
    assert c["checked"] >= 10**9, c
    assert c["code_mismatches"] == 0, c
    assert c["quotient_mismatches_normal"] == 0, c


def test_fp32_divisors_need_the_ieee_division(w4):
    # the same correction with full fp32 divisors of the NVFP4 form is not
    # always correctly rounded; the NVFP4 quantize therefore divides with the
    # IEEE division (its codes are checked bit for bit in test_gpu_fp4.py)
    c = w4.selftest_quotient(2)
    assert c["checked"] >= 10**9, c
    assert c["code_mismatches"] > 0, c
