"""The tensor cores as a source of exact products: the self-test behind the opt-in
tensor-core W tile ("User guide" section 6: the tensor-core kernels rest on what the
tensor cores compute; the one property used here is that a bf16 x bf16 product of two
pre-scaled FP8 values, alone in its output, comes back exact in fp32)."""
import pytest

pytestmark = pytest.mark.gpu


def test_tensor_core_products_are_exact():
    import __graft_entry__
    __graft_entry__.build()
    from bit_exact_fp8_gb300 import _lib
    assert _lib.emu_tc_selftest() == 0
    assert _lib.emu_device_status() == 0
