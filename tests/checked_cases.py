"""Small parity cases run against the bounds-checked library (QLORA_NF4_LIB names
libqlora_nf4_checked.so; started by tests/test_checked_build.py in a process of its own).
Every case must match the oracle within the usual bounds and leave the device error word
clear: a failed index check would set it (codes 9-11) and skip the access."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
import bit_nf4_quantized_37_b300 as qn  # noqa: E402
from bit_nf4_quantized_37_b300 import _binding, workloads as wl  # noqa: E402
from gpu_helpers import TOL, Problem, bf16_dev, f32_host, rel_fro  # noqa: E402


def status_clear(what):
    st = qn.device_status()
    assert st == 0, f"{what}: device error word {st}"


def main():
    assert _binding.LIB_PATH.endswith("_checked.so"), _binding.LIB_PATH
    qn.lib()
    # quantize / dequantize (bit-exact)
    for n in (65, 64 * 256 + 1, 1 << 18):
        W = wl.weight((1, n), seed=900 + n, sigma=0.02)
        q = qn.nf4_quantize(torch.from_numpy(W).cuda())
        o = oracle.quantize(W)
        assert np.array_equal(q.codes.cpu().numpy(), o["codes"])
        assert np.array_equal(q.scale_codes.cpu().numpy(), o["qscale"])
        got = qn.nf4_dequantize(q).contiguous().view(torch.int16).cpu().numpy().view(np.uint16).ravel()
        assert np.array_equal(got, oracle.dequantize(o))
        status_clear(f"quantize {n}")
    # forward / backward: single-CTA tiles with and without a split contraction, CTA pairs
    # with and without one, the decode path (whole and split row blocks)
    cases = [("small", 200, 320, 448, 16), ("split2", 520, 1024, 1088, 16),
             ("split4_pairs", 2000, 320, 4800, 40), ("pairs_split", 512, 3072, 3072, 16),
             ("decode1", 1, 2048, 4096, 64), ("decode5", 5, 1088, 2560, 24),
             ("decode16", 16, 2048, 4096, 64), ("rank3", 40, 192, 128, 3)]
    for name, M, N, K, r in cases:
        p = wl.LinearProblem(name, M, N, K, r, 2.0 * r, 0.02, 0.001, config=70 + len(name))
        pb = Problem(p)
        Y, U = qn.qlora_linear_fwd(pb.Xd, pb.qd, pb.Ad, pb.Bd, p.scale)
        Yo, _ = oracle.lora_fwd(pb.X, pb.Wd, pb.A, pb.B, p.scale)
        assert rel_fro(f32_host(Y), Yo) <= TOL, name
        status_clear(f"{name} forward")
        dX, dA, dB = qn.qlora_linear_bwd(pb.dYd, pb.Xd, pb.qd, pb.Ad, pb.Bd, p.scale, U)
        status_clear(f"{name} backward")
        dXo, _ = oracle.lora_dx(pb.dY, pb.Wd, pb.A, pb.B, p.scale)
        dAo, dBo = oracle.lora_dadb(pb.dY, pb.X, pb.A, pb.B, p.scale)
        assert rel_fro(f32_host(dX), dXo) <= TOL, name
        assert rel_fro(f32_host(dA), dAo) <= TOL, name
        assert rel_fro(f32_host(dB), dBo) <= TOL, name
    # per-token adapters on the decode path
    N, K, M, r, nad = 1024, 2048, 6, 16, 3
    W = wl.weight((N, K), seed=95, sigma=0.015)
    Wd = oracle.dequantize(oracle.quantize(W)).reshape(N, K)
    qd = qn.nf4_quantize(torch.from_numpy(W).cuda())
    A = [wl.bf16_normal((r, K), seed=96 + i, sigma=0.01) for i in range(nad)]
    B = [wl.bf16_normal((N, r), seed=99 + i, sigma=0.01) for i in range(nad)]
    X = wl.bf16_normal((M, K), seed=102)
    idx = np.array([t % nad for t in range(M)], np.int32)
    sc = np.array([0.5, 1.0, 2.0], np.float32)
    Y = qn.qlora_linear_fwd_multi(bf16_dev(X), qd, bf16_dev(np.stack(A)), bf16_dev(np.stack(B)),
                                  torch.from_numpy(idx).cuda(), torch.from_numpy(sc).cuda())
    ref = np.stack([oracle.lora_fwd(X[t:t + 1], Wd, A[idx[t]], B[idx[t]], float(sc[idx[t]]))[0][0]
                    for t in range(M)])
    assert rel_fro(f32_host(Y), ref) <= TOL
    status_clear("per-token adapters")
    print("CHECKED_OK")


if __name__ == "__main__":
    main()
