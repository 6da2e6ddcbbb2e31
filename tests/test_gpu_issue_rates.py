"""Premises of the GEMM kernel's arithmetic, checked on the GPU: the packed f32x2
multiply (round to nearest and toward zero) and add, which pass 2 issues on two
adjacent k at once, round every half bit for bit as the scalar instruction does,
subnormal results included.  The measured instruction rates (libemupeaks, the
denominators bench.py reports its roofline against) are printed, not asserted:
on a shared GPU they can move for reasons unrelated to this code."""
import pytest

pytestmark = pytest.mark.gpu


def test_packed_f32x2_rounds_like_scalar_and_rates_are_measurable():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_exact_fp8_gb300 import build, peaks
    build.build()
    assert peaks.f32x2_agreement(1 << 23) == (0, 0, 0)
    rates = peaks.issue_rates()
    print(rates)
    assert all(r > 0 for r in rates.values())
