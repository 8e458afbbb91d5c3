"""CPU-side checks of the C-ABI library: it loads, exports every declared symbol, its
constant tables equal the oracle's construction, and host-side validation answers without
touching a GPU.  No compute calls (there is no GPU here)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import bit_nf4_quantized_37_b300 as qn
from bit_nf4_quantized_37_b300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qlora_nf4.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_0-9]+)\s*\(", src, re.M)
    return sorted(set(n for n in names if n.startswith(("nf4_", "qlora_"))))


@pytest.fixture(scope="module")
def lib():
    from bit_nf4_quantized_37_b300 import build
    build.build()
    return qn.lib()


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert len(declared) >= 11
    assert sorted(declared) == sorted(_binding.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_level_table_equals_oracle_construction(lib):
    L, T = qn.level_table()
    Lo, To = oracle.levels()
    assert np.array_equal(np.array(L, np.float32), Lo)
    assert np.array_equal(np.array(T, np.float32), To)


def test_storage_bytes_formula(lib):
    for rows, cols in ((1, 1), (3, 5), (256, 256), (4096, 11008), (28672, 8192), (7, 64 * 256 + 3)):
        sizes, total = qn.nf4_storage_bytes(rows, cols)
        n = rows * cols
        nb = -(-n // 64)
        ng = -(-nb // 256)
        assert sizes == [(n + 1) // 2, nb, 4 * ng, 4]
        assert total == sum(sizes)
    # 4.127 bits per weight on a large tensor (infivelines.com "QLoRA": ~0.127 bits/weight)
    _, total = qn.nf4_storage_bytes(4096, 11008)
    assert abs(total * 8 / (4096 * 11008) - 4.127) < 0.001
    # without double quantization: fp32 absmax per 64 weights, 0.5 bits/weight of scales
    sizes, total = qn.nf4_storage_bytes(4096, 11008, 0)
    n = 4096 * 11008
    assert sizes == [n // 2, 0, 4 * (n // 64), 0] and total * 8 / n == 4.5


def test_host_validation_without_device(lib):
    u64 = ctypes.c_uint64(0)
    assert lib.nf4_storage_bytes(0, 5, 64, 256, None, ctypes.byref(u64)) == -1
    assert lib.nf4_storage_bytes(5, 5, 32, 256, None, ctypes.byref(u64)) == -2
    assert lib.nf4_storage_bytes(5, 5, 64, 128, None, ctypes.byref(u64)) == -2
    assert lib.qlora_workspace_bytes(16, 256, 256, 129, ctypes.byref(u64)) == -2
    assert lib.qlora_workspace_bytes(16, 256, 256, 8, ctypes.byref(u64)) == 0 and u64.value > 0
    S = _binding._NF4Struct
    good = S(16, 32, 48, 64, 256, 256, 64, 256)
    assert lib.nf4_dequantize(ctypes.byref(S(16, 32, 48, 64, 256, 256, 32, 256)), 16, None) == -2
    assert lib.nf4_dequantize(ctypes.byref(S(17, 32, 48, 64, 256, 256, 64, 256)), 16, None) == -3
    assert lib.nf4_dequantize(ctypes.byref(S(0, 32, 48, 64, 256, 256, 64, 256)), 16, None) == -1
    assert lib.nf4_dequantize(ctypes.byref(good), 24, None) == -3
    # fused path needs N, K multiples of 64
    bad_shape = S(16, 32, 48, 64, 250, 256, 64, 256)
    assert lib.qlora_linear_fwd(16, 16, ctypes.byref(bad_shape), 16, 16, 8, ctypes.c_float(2.0),
                                16, None, 16, 1 << 30, None) == -2
    # well-formed arguments reach the device check, which fails cleanly on a CPU-only host
    st = lib.nf4_dequantize(ctypes.byref(good), 16, None)
    assert st in (-7, 0)
    assert lib.qlora_status_str(-4).decode() == "workspace too small"
    # the wait self-test needs a device; without one it answers at once
    import torch
    if not torch.cuda.is_available():
        assert lib.qlora_wait_timeout_selftest(None) == -7


def test_f16_entry_points_validate_like_the_bf16_ones(lib):
    """The fp16 compute-type entry points share the bf16 ones' host validation: the same
    status for the same bad argument, before any device work."""
    S = _binding._NF4Struct
    good = S(16, 32, 48, 64, 256, 256, 64, 256)
    for f in (lib.nf4_dequantize, lib.nf4_dequantize_f16):
        assert f(ctypes.byref(S(16, 32, 48, 64, 256, 256, 32, 256)), 16, None) == -2
        assert f(ctypes.byref(S(17, 32, 48, 64, 256, 256, 64, 256)), 16, None) == -3
        assert f(ctypes.byref(good), 24, None) == -3
        assert f(ctypes.byref(good), 16, None) in (-7, 0)
    bad_shape = S(16, 32, 48, 64, 250, 256, 64, 256)
    f32 = ctypes.c_float
    for fwd in (lib.qlora_linear_fwd, lib.qlora_linear_fwd_f16):
        assert fwd(16, 16, ctypes.byref(bad_shape), 16, 16, 8, f32(2.0), 16, None, 16, 1 << 30,
                   None) == -2
        assert fwd(16, 16, ctypes.byref(good), 16, 16, 129, f32(2.0), 16, None, 16, 1 << 30,
                   None) == -2                                   # rank above 128
        assert fwd(16, 16, ctypes.byref(good), 16, 16, 8, f32(float("nan")), 16, None, 16,
                   1 << 30, None) == -1                          # NaN scale
        assert fwd(24, 16, ctypes.byref(good), 16, 16, 8, f32(2.0), 16, None, 16, 1 << 30,
                   None) == -3                                   # X not 16-byte aligned
        assert fwd(16, 16, ctypes.byref(good), 16, 16, 8, f32(2.0), 16, None, 16, 1, None) == -4
    for bwd in (lib.qlora_linear_bwd, lib.qlora_linear_bwd_f16):
        assert bwd(16, 16, 16, ctypes.byref(bad_shape), 16, 16, 8, f32(2.0), None, 16, 16, 16,
                   16, 1 << 30, None) == -2
        assert bwd(16, 16, 16, ctypes.byref(good), 16, 16, 8, f32(2.0), None, 16, None, 16,
                   16, 1 << 30, None) == -1                      # dA missing
        assert bwd(16, 16, 16, ctypes.byref(good), 16, 16, 8, f32(2.0), None, 16, 16, 16,
                   16, 1, None) == -4


def test_f16_wrappers_refuse_host_tensors(lib):
    import torch
    q = _cpu_nf4(64, 64)  # never reaches a kernel
    x = torch.zeros(4, 64, dtype=torch.float16)
    a = torch.zeros(4, 64, dtype=torch.float16)
    b = torch.zeros(64, 4, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        qn.qlora_linear_fwd_f16(x, q, a, b, 1.0)       # host tensors
    with pytest.raises(ValueError, match="CUDA tensor"):
        qn.qlora_linear_bwd_f16(x, x, q, a, b, 1.0)


def test_workspace_grows_with_problem(lib):
    a = qn.qlora_workspace_bytes(16, 256, 256, 8)
    b = qn.qlora_workspace_bytes(4096, 4096, 4096, 16)
    c = qn.qlora_workspace_bytes(4096, 4096, 4096, 128)
    assert 0 < a < b < c
    assert qn.nf4_quantize_workspace_bytes(28672 * 8192) >= 28672 * 8192 // 64 * 4


# ------------------------------------------------------------------ binding shape checks
# A buffer whose shape does not match the NF4 base would make a kernel read or write past
# its allocation; the binding refuses it with ValueError before anything is launched.  The
# checks run before the device checks, so CPU tensors of the wrong shape exercise them here.
def _cpu_nf4(rows, cols, dq=True):
    import torch
    sizes, _ = qn.nf4_storage_bytes(rows, cols, 256 if dq else 0)
    return qn.NF4Tensor(torch.zeros(sizes[0], dtype=torch.uint8),
                        torch.zeros(sizes[1], dtype=torch.int8),
                        torch.zeros(sizes[2] // 4, dtype=torch.float32),
                        torch.zeros(sizes[3] // 4, dtype=torch.float32), rows, cols,
                        256 if dq else 0)


def _bf(*shape):
    import torch
    return torch.zeros(*shape, dtype=torch.bfloat16)


SHAPE_WORDS = r"shape|columns|elements|holds"


def test_linear_fwd_refuses_mismatched_shapes(lib):
    q = _cpu_nf4(256, 128)
    cases = [
        (_bf(16, 64), _bf(8, 64), _bf(256, 8), None),     # X has K = 64, base has 128
        (_bf(16, 128), _bf(8, 64), _bf(256, 8), None),    # A [r, 64]
        (_bf(16, 128), _bf(8, 128), _bf(128, 8), None),   # B rows != N
        (_bf(16, 128), _bf(8, 128), _bf(256, 4), None),   # B columns != r
        (_bf(16, 128), _bf(8, 128), _bf(256, 8), _bf(16, 128)),  # out [M, K] instead of [M, N]
        (_bf(2, 8, 128), _bf(8, 128), _bf(256, 8), None),  # X not 2-D
    ]
    for X, A, B, out in cases:
        for fn in (qn.qlora_linear_fwd, qn.qlora_linear_fwd_f16):
            with pytest.raises(ValueError, match=SHAPE_WORDS + "|2-D"):
                fn(X, q, A, B, 2.0, out=out)


def test_linear_bwd_refuses_mismatched_shapes(lib):
    import torch
    q = _cpu_nf4(256, 128)
    X, A, B = _bf(16, 128), _bf(8, 128), _bf(256, 8)
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.qlora_linear_bwd(_bf(16, 128), X, q, A, B, 2.0)           # dY [M, K]
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.qlora_linear_bwd(_bf(8, 256), X, q, A, B, 2.0)            # dY with other M
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.qlora_linear_bwd(_bf(16, 256), X, q, A, B, 2.0,
                            U=torch.zeros(16, 4, dtype=torch.float32))  # U [M, r'] r' != r
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.qlora_linear_bwd_f16(_bf(16, 256), _bf(16, 64), q, A, B, 2.0)  # X columns


def test_quantize_and_dequantize_refuse_mismatched_sizes(lib):
    import torch
    q = _cpu_nf4(64, 64)
    W = torch.zeros(64, 65, dtype=torch.float32)
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.nf4_quantize(W, out=q)
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.nf4_quantize_noalloc(W, q)
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.nf4_dequantize(q, out=_bf(64, 63))
    short = qn.NF4Tensor(q.codes[:100], q.scale_codes, q.scale_steps, q.scale_mean, 64, 64)
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.nf4_dequantize(short)
    nodq_short = _cpu_nf4(64, 64, dq=False)
    nodq_short.scale_steps = nodq_short.scale_steps[:10]  # 64 blocks need 64 fp32 absmax
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.nf4_dequantize(nodq_short)


def test_multi_and_merge_refuse_mismatched_shapes(lib):
    import torch
    q = _cpu_nf4(256, 128)
    X = _bf(4, 128)
    A_all, B_all = _bf(3, 8, 128), _bf(3, 256, 8)
    idx = torch.zeros(4, dtype=torch.int32)
    sc = torch.ones(3, dtype=torch.float32)
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.qlora_linear_fwd_multi(X, q, A_all, _bf(2, 256, 8), idx, sc)
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.qlora_linear_fwd_multi(X, q, A_all, B_all, torch.zeros(5, dtype=torch.int32), sc)
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.qlora_linear_fwd_multi(X, q, A_all, B_all, idx, torch.ones(2, dtype=torch.float32))
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.nf4_merge_lora(q, _bf(8, 64), _bf(256, 8), 2.0)
    with pytest.raises(ValueError, match=SHAPE_WORDS):
        qn.nf4_merge_lora(q, _bf(8, 128), _bf(256, 8), 2.0, out=_bf(128, 256))


def test_matching_cpu_tensors_reach_the_device_check(lib):
    """With every shape right, the first refusal is the device check (CPU tensors)."""
    q = _cpu_nf4(256, 128)
    with pytest.raises(ValueError, match="CUDA tensor"):
        qn.qlora_linear_fwd(_bf(16, 128), q, _bf(8, 128), _bf(256, 8), 2.0)


def test_per_device_setup_cache_keying(tmp_path):
    """The per-device set-up cache (csrc/device_cache.h): one entry per device ordinal, a
    new set-up when that device's context changes (cudaDeviceReset), nothing stored when the
    set-up fails or no context id exists.  Built with g++ against a fake key; no GPU."""
    import subprocess
    src = os.path.join(ROOT, "tests", "device_cache_test.cpp")
    exe = str(tmp_path / "device_cache_test")
    subprocess.run(["g++", "-std=c++17", "-O1", "-Wall", "-Werror", "-pthread", src, "-o", exe],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr


def test_checked_variant_builds_and_exports_every_symbol():
    """The bounds-checked build (QLORA_CHECK_BOUNDS=1) compiles for sm_103a and exports the
    same C ABI (its GPU test runs the small parity cases through it)."""
    from bit_nf4_quantized_37_b300 import build
    lib = ctypes.CDLL(build.build(checked=True))
    for name in _declared_functions():
        assert hasattr(lib, name), name
