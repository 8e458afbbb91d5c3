"""Failure detection on the device: every mbarrier wait in the kernels is bounded, so a wait
that never completes ends in a status the host reads, not in a hang.  The library's
self-test waits on an mbarrier that nothing arrives on; the wait gives up after its limit
(about 2 s), the host reads wait code 8 through qlora_device_status, and the same context
then still computes a layer that matches the oracle.  Nothing here faults or hangs the GPU:
the wait is bounded by design and the kernel returns."""
import time

import numpy as np
import pytest
import torch

import oracle
import bit_nf4_quantized_37_b300 as qn
from bit_nf4_quantized_37_b300 import workloads as wl
from gpu_helpers import TOL, Problem, f32_host, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_37_b300 import build
    build.build()
    qn.lib()


def test_wait_that_never_completes_ends_in_a_status_and_the_device_stays_usable():
    assert qn.device_status() == 0
    t0 = time.perf_counter()
    qn.wait_timeout_selftest()
    code = qn.device_status()  # synchronizes: returns once the wait has given up
    elapsed = time.perf_counter() - t0
    assert code == 8
    assert 1.9 <= elapsed <= 60.0, elapsed
    assert qn.device_status() == 0  # the read cleared the word
    pb = Problem(wl.config1())
    Y, _ = qn.qlora_linear_fwd(pb.Xd, pb.qd, pb.Ad, pb.Bd, pb.p.scale)
    Yo, _ = oracle.lora_fwd(pb.X, pb.Wd, pb.A, pb.B, pb.p.scale)
    assert rel_fro(f32_host(Y), Yo) <= TOL
    assert qn.device_status() == 0
