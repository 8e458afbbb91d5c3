"""nf4_quantize_noalloc: the quantizer for callers that must not allocate device memory
(a plugin whose host application owns all device allocations, or a service that reserved
its memory at start-up and keeps cudaMalloc off the request path).  The call keeps its
scratch in a fixed device array of the library, so it must give bit-for-bit what the
workspace-taking nf4_quantize gives -- also on a second call, when the array still holds
the first call's contents.

This file is collected last on purpose, and passes both on its own in a fresh process and
after the rest of the suite."""
import ctypes

import numpy as np
import pytest
import torch

import bit_nf4_quantized_37_b300 as qn
from bit_nf4_quantized_37_b300 import _binding, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_37_b300 import build
    build.build()
    qn.lib()


def _via_c_abi(W: torch.Tensor, rows: int, cols: int) -> qn.NF4Tensor:
    out = qn.NF4Tensor.empty(rows, cols, W.device)
    for t in (out.codes, out.scale_codes, out.scale_steps, out.scale_mean):
        t.fill_(0x5A if t.dtype in (torch.uint8, torch.int8) else 7.0)  # not zero: catch holes
    s = out.c_struct()
    st = qn.lib().nf4_quantize_noalloc(ctypes.c_void_p(W.data_ptr()), ctypes.byref(s),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, qn.status_str(st)
    return out


def _same(a: qn.NF4Tensor, b: qn.NF4Tensor):
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes)
    assert torch.equal(a.scale_codes, b.scale_codes)
    assert torch.equal(a.scale_steps.view(torch.int32), b.scale_steps.view(torch.int32))
    assert torch.equal(a.scale_mean.view(torch.int32), b.scale_mean.view(torch.int32))


def test_noalloc_matches_workspace_quantize_on_two_calls_in_a_row():
    # a large tensor first (fills most of the scratch), then a small ragged one that reuses
    # the head of the same scratch
    shapes = [(4096, 4096), (1001, 333)]
    for i, (rows, cols) in enumerate(shapes):
        W = torch.from_numpy(wl.weight((rows, cols), seed=900 + i, sigma=0.02,
                                       outlier_frac=0.001)).cuda()
        want = qn.nf4_quantize(W)
        got = _via_c_abi(W, rows, cols)
        _same(got, want)


def test_noalloc_at_its_largest_size():
    """Exactly NF4_NOALLOC_MAX_NUMEL weights (8192 x 8192): the whole scratch, the mean's
    tail included, is in use; bit-exact with the oracle."""
    import oracle
    rows, cols = 8192, 8192
    assert rows * cols == _binding.NF4_NOALLOC_MAX_NUMEL
    Wh = wl.weight((rows, cols), seed=917, sigma=0.02, outlier_frac=0.001)
    W = torch.from_numpy(Wh).cuda()
    got = _via_c_abi(W, rows, cols)
    torch.cuda.synchronize()
    o = oracle.quantize(Wh)
    assert np.array_equal(got.codes.cpu().numpy(), o["codes"])
    assert np.array_equal(got.scale_codes.cpu().numpy(), o["qscale"])
    assert np.array_equal(got.scale_steps.cpu().numpy().view(np.uint32), o["steps"].view(np.uint32))
    assert got.scale_mean.cpu().numpy()[0].view(np.uint32) == np.float32(o["mean"]).view(np.uint32)


def test_noalloc_rejects_tensors_beyond_its_scratch():
    rows, cols = 8193, 8192  # one row past NF4_NOALLOC_MAX_NUMEL
    assert rows * cols > _binding.NF4_NOALLOC_MAX_NUMEL
    fake = _binding._NF4Struct(16, 32, 48, 64, rows, cols, 64, 256)
    st = qn.lib().nf4_quantize_noalloc(ctypes.c_void_p(16), ctypes.byref(fake), None)
    assert st == -8 and "scratch" in qn.status_str(st)
