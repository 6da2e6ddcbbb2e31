"""The kernels' waits for their TMA loads are bounded: a wait that cannot complete
gives up, sets the library's device status word and returns instead of hanging.
The self-test kernel makes a wait run out on purpose (its barrier never
completes), the status reports it, and the context stays usable: a GEMM after it
still matches the oracle and leaves the status at 0."""
import pytest
import torch

from bit_exact_fp8_gb300 import workloads as W
from helpers import assert_bits_equal, gpu_run, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from bit_exact_fp8_gb300 import _lib
    return _lib


def test_gemms_leave_the_status_clear(lib):
    lib.emu_device_status(reset=True)
    for cs in (W.case("tiny"), W.Case("st", 70, 96, 528, out_dtype="f32", split_S=3, gen="mixed",
                                      fast_accum=False, seed=6)):
        a, b = W.make_inputs(cs)
        assert_bits_equal(gpu_run(cs, a, b), oracle_full(cs, a, b), cs.name)
    assert lib.emu_device_status() == 0


def test_a_wait_that_cannot_complete_gives_up_and_reports(lib):
    lib.emu_device_status(reset=True)
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.emu_selftest_wait_timeout(stream) == 0
    torch.cuda.synchronize()
    assert lib.emu_device_status(reset=True) == 1
    assert lib.emu_device_status() == 0
    cs = W.case("tiny")
    a, b = W.make_inputs(cs)
    assert_bits_equal(gpu_run(cs, a, b), oracle_full(cs, a, b), "after the self-test")
    assert lib.emu_device_status() == 0
