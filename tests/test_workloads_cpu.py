"""The seeded input recipe the design notes state: seeds, shapes, distributions, the exact
outlier count and the bf16 rounding of the 16-bit inputs.  CPU only."""
import numpy as np
import torch

from bit_nf4_quantized_37_b300 import workloads as wl


def test_seeds_follow_the_stated_formula():
    assert wl.seed_for(2, "W") == 2001 and wl.seed_for(2, "dY") == 2005
    assert wl.seed_for(5, "X", layer=3) == 5000 + 2 + 30
    # a seed fixes the draw; another seed changes it
    a = wl.weight((64, 64), seed=7, sigma=0.02)
    assert np.array_equal(a, wl.weight((64, 64), seed=7, sigma=0.02))
    assert not np.array_equal(a, wl.weight((64, 64), seed=8, sigma=0.02))


def test_weight_distribution_and_exact_outlier_count():
    n = 1 << 20
    w = wl.weight((n,), seed=11, sigma=0.02)
    assert w.dtype == np.float32
    assert abs(w.std() / 0.02 - 1) < 0.01 and abs(w.mean()) < 1e-4
    wo = wl.weight((n,), seed=11, sigma=0.02, outlier_frac=0.001)
    changed = np.count_nonzero(wo != w)
    assert changed <= int(np.floor(0.001 * n))          # exactly floor(frac*n) positions drawn
    assert changed >= int(np.floor(0.001 * n)) - 2       # (a t-draw may equal the normal one)
    # the outliers are heavy-tailed: far more mass beyond 5 sigma than a normal has
    assert np.count_nonzero(np.abs(wo) > 0.1) > 100 * max(1, np.count_nonzero(np.abs(w) > 0.1))


def test_16_bit_inputs_are_bf16_rounded_normals():
    bits = wl.bf16_normal((256, 256), seed=3, sigma=1.0)
    assert bits.dtype == np.uint16
    v = wl.bf16_bits_to_f32(bits)
    raw = wl.rng(3).standard_normal(size=(256, 256), dtype=np.float32)
    want = torch.from_numpy(raw).to(torch.bfloat16).float().numpy()
    assert np.array_equal(v, want)
    assert abs(v.std() - 1.0) < 0.02


def test_config_shapes():
    c1, c2 = wl.config1(), wl.config2()
    assert (c1.M, c1.N, c1.K, c1.r) == (16, 256, 256, 8)
    assert (c2.M, c2.N, c2.K, c2.r, c2.alpha) == (4096, 4096, 4096, 16, 32.0)
    assert c2.scale == 2.0
    for M in (1, 4, 16):
        c4 = wl.config4(M)
        assert (c4.M, c4.N, c4.K, c4.r) == (M, 28672, 8192, 64)
    assert all(p.M == 2048 and p.r == 16 for p in wl.config3())
    assert len(wl.config5(layer=0)) == 7
