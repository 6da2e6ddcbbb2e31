"""Several host threads call the library at once, each on its own CUDA stream:
the device entry point (scaled_mm) and the host-buffer one (scaled_mm_host, whose
enqueue is serialised by the library; its first use, which creates the library's
stream pool, happens inside the threads).
ctypes releases the GIL during the C calls, so the calls overlap.  Every result
must equal the single-threaded one bit for bit."""
import threading

import numpy as np
import pytest
import torch

from bit_exact_fp8_gb300 import workloads as W
from helpers import TORCH_FP8, TORCH_OUT, gpu_run, out_bits

pytestmark = pytest.mark.gpu


def test_concurrent_host_threads_give_single_threaded_bits():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_exact_fp8_gb300 import build, scaled_mm, scaled_mm_host
    build.build()
    dev = torch.device("cuda:0")
    cases = [W.shrink(W.case("linear"), 48, 640, 512),
             W.shrink(W.case("splitk-hopper-S8-fast-bf16"), 16, 128, 4096),
             W.shrink(W.case("splitk-ada-S8-slow-f32"), 16, 64, 2048),
             W.case("tiny")]
    inputs = [W.make_inputs(cs) for cs in cases]
    want = [gpu_run(cs, a, b) for cs, (a, b) in zip(cases, inputs)]
    errors = []

    def worker(t):
        try:
            stream = torch.cuda.Stream(dev)
            for rep in range(3):
                i = (t + rep) % len(cases)
                cs, (a, b) = cases[i], inputs[i]
                od = TORCH_OUT[cs.out_dtype]
                with torch.cuda.stream(stream):
                    if (t + rep) % 2 == 0:
                        A = torch.from_numpy(a).to(dev).view(TORCH_FP8[cs.fmt_a])
                        B = torch.from_numpy(b).to(dev).view(TORCH_FP8[cs.fmt_b])
                        sa = torch.tensor(cs.scale_a, dtype=torch.float32, device=dev)
                        sb = torch.tensor(cs.scale_b, dtype=torch.float32, device=dev)
                        y = scaled_mm(A, B.t(), sa, sb, out_dtype=od,
                                      use_fast_accum=cs.fast_accum, splitk=cs.split_S,
                                      preset=cs.preset)
                        stream.synchronize()
                    else:
                        A = torch.from_numpy(a).view(TORCH_FP8[cs.fmt_a]).pin_memory()
                        B = torch.from_numpy(b).view(TORCH_FP8[cs.fmt_b]).pin_memory()
                        y = scaled_mm_host(A, B.t(), cs.scale_a, cs.scale_b, out_dtype=od,
                                           use_fast_accum=cs.fast_accum, splitk=cs.split_S,
                                           preset=cs.preset, device=dev)
                got = out_bits(y)
                if not np.array_equal(got, want[i]):
                    errors.append(f"thread {t} rep {rep} case {cs.name}: "
                                  f"{int(np.sum(got != want[i]))} outputs differ")
        except Exception as e:                          # reported below, with the thread
            errors.append(f"thread {t}: {e!r}")

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
    assert not any(th.is_alive() for th in threads), "a worker thread did not finish"
    assert not errors, errors
