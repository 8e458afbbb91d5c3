"""The bounds-checked build of the library (build.py --checked, QLORA_CHECK_BOUNDS=1) on the
small parity cases: every result within the usual bounds and no failed index check (the
kernels would record it in their device error word).  Runs the cases in a process of its
own, with QLORA_NF4_LIB naming the checked library."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_small_cases():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_37_b300 import build
    lib = build.build(checked=True)
    assert lib.endswith("libqlora_nf4_checked.so")
    env = dict(os.environ, QLORA_NF4_LIB=lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_cases.py")],
                       env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-4000:] + r.stderr[-4000:])
    assert "CHECKED_OK" in r.stdout
