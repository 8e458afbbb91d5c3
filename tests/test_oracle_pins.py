"""Pins for the CPU oracle: checks against what the QLoRA pages and the mathematics fix,
never against the oracle itself.  CPU only (not marked gpu).

Pages cited: infivelines.com "QLoRA" (mechanism paragraphs), junaidshaukat.com
"QLoRA -- the democratization event" (recipe), aicurriculum "QLoRA -- Module 12.4"
(Design Details: NF4), addaly.com "QLoRA on one card" (What each setting is doing),
digipro.cn "QLoRA: Fine-Tuning a 7B Model on a 16GB GPU".
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special as sp
import torch

import oracle
from bit_nf4_quantized_37_b300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            key, val, tol, src = [p.strip() for p in line.split("|", 3)]
            out[key] = (float(val), float(tol), src)
    return out


def _exact_nearest(x: np.ndarray, L: np.ndarray) -> np.ndarray:
    """Brute force: index of the nearest level in exact fp64 arithmetic, ties -> lower."""
    d = np.abs(x.astype(np.float64)[:, None] - L.astype(np.float64)[None, :])
    return np.argmin(d, axis=1)  # argmin returns the first (lower) index on ties


def _unpack(codes: np.ndarray, numel: int) -> np.ndarray:
    c = np.stack([codes >> 4, codes & 0xF], axis=1).reshape(-1)
    return c[:numel].astype(np.int64)


# ---------------------------------------------------------------- levels (NF4 data type)

def test_levels_structure():
    """16 levels (4 bits), ascending, 0 exact, block absmax maps to -1 / +1."""
    L, T = oracle.levels()
    assert L.shape == (16,) and L.dtype == np.float32
    assert np.all(np.diff(L) > 0)
    assert L[0] == -1.0 and L[15] == 1.0 and L[7] == 0.0
    assert (L > 0).sum() == 8 and (L < 0).sum() == 7


def test_levels_sit_at_equally_spaced_normal_probabilities():
    """infivelines 'QLoRA': NF4 places its 16 levels at quantiles of a normal
    distribution.  Mapped back through the normal CDF (scipy ndtr, not the oracle's
    quantile routine), the positive levels sit at equally spaced probabilities and so do
    the negative ones."""
    L, _ = oracle.levels()
    delta = 0.5 * ((1 - 1 / 32) + (1 - 1 / 30))
    zmax = sp.ndtri(delta)
    p_pos = sp.ndtr(L[8:].astype(np.float64) * zmax)       # ascending
    p_neg = sp.ndtr(-L[:7].astype(np.float64) * zmax)      # -L ascending magnitude reversed
    dp = np.diff(p_pos)
    assert np.allclose(dp, (delta - 0.5) / 8, rtol=2e-6, atol=0)
    dn = np.diff(p_neg[::-1])
    assert np.allclose(dn, (delta - 0.5) / 7, rtol=2e-6, atol=0)
    # the construction through scipy's own quantile gives the same fp32 table
    pos = sp.ndtri(np.linspace(delta, 0.5, 9)[:-1])
    neg = -sp.ndtri(np.linspace(delta, 0.5, 8)[:-1])
    v = np.sort(np.concatenate([pos, neg, [0.0]]))
    assert np.array_equal((v / np.abs(v).max()).astype(np.float32), L)


def test_nf4_levels_used_about_equally_and_beat_int4():
    """infivelines 'QLoRA': each NF4 level is about equally likely on normal weights;
    aicurriculum 'Design Details' and addaly 'What each setting is doing': NF4 keeps more
    information than plain 4-bit integers.  Compare with a uniform 16-level grid."""
    W = wl.weight((512, 1024), seed=7, sigma=0.02)
    q = oracle.quantize(W)
    c = _unpack(q["codes"], W.size)
    h = np.bincount(c, minlength=16) / c.size
    inner = h[1:15]
    ent = -(h * np.log2(h)).sum()
    L, _ = oracle.levels()
    a = q["absmax"][:, None]
    Wb = W.reshape(-1, 64)
    nf4 = L[c].reshape(-1, 64) * a
    grid = np.linspace(-1, 1, 16)
    gi = np.abs((Wb / a)[..., None] - grid).argmin(-1)
    hi = np.bincount(gi.ravel(), minlength=16) / gi.size
    ent_int4 = -(hi * np.log2(hi)).sum()
    assert inner.max() / inner.min() < 3.0
    assert ent > 3.85 and ent > ent_int4 + 0.2
    rmse_nf4 = np.sqrt(((nf4 - Wb) ** 2).mean())
    rmse_int4 = np.sqrt(((grid[gi] * a - Wb) ** 2).mean())
    assert rmse_nf4 < 0.95 * rmse_int4


def test_thresholds_round_midpoints_down():
    L, T = oracle.levels()
    for i in range(15):
        m = (Fraction(float(L[i])) + Fraction(float(L[i + 1]))) / 2
        assert Fraction(float(T[i])) <= m
        assert Fraction(float(np.nextafter(T[i], np.float32(2)))) > m


# ---------------------------------------------------------------- quantize (blockwise absmax)

def _blocks_with_unit_absmax(x: np.ndarray) -> np.ndarray:
    """Blocks of 64 whose first entry is 1.0, so w / absmax == w exactly."""
    n = len(x)
    nb = -(-n // 63)
    W = np.zeros((nb, 64), np.float32)
    W[:, 0] = 1.0
    flat = np.zeros(nb * 63, np.float32)
    flat[:n] = x
    W[:, 1:] = flat.reshape(nb, 63)
    return W, n


def _codes_of_unit_blocks(x):
    W, n = _blocks_with_unit_absmax(x)
    q = oracle.quantize(W)
    c = _unpack(q["codes"], W.size).reshape(-1, 64)
    assert np.all(c[:, 0] == 15)
    return c[:, 1:].reshape(-1)[:n]


def test_nearest_level_brute_force_around_every_midpoint():
    """Every fp32 value within 3000 ulps of each midpoint, plus random values, gets the
    exactly nearest level (ties to the lower index)."""
    L, T = oracle.levels()
    xs = []
    for t in T:
        base = np.float32(t).view(np.int32)
        ints = base + np.arange(-3000, 3001, dtype=np.int64)  # both sides of the midpoint
        xs.append(ints.astype(np.int32).view(np.float32))
    g = wl.rng(11)
    xs.append(g.uniform(-1, 1, size=200_000).astype(np.float32))
    x = np.concatenate(xs)
    x = x[(x >= -1) & (x <= 1)]
    got = _codes_of_unit_blocks(x)
    want = _exact_nearest(x, L)
    assert np.array_equal(got, want)


def test_exact_midpoint_ties_go_down():
    L, T = oracle.levels()
    ties = []
    for i in range(15):
        m = (np.float64(L[i]) + np.float64(L[i + 1])) / 2
        if np.float64(np.float32(m)) == m:
            ties.append((i, np.float32(m)))
    for i, m in ties:
        assert _codes_of_unit_blocks(np.array([m], np.float32))[0] == i


def test_quantize_brute_force_small_ragged():
    """Random weights with a ragged last block and odd length: codes equal the brute-force
    nearest level of the fp32 quotient w / absmax (numpy's IEEE fp32 division)."""
    L, _ = oracle.levels()
    for n in (1, 63, 64, 65, 1001, 64 * 300 + 37):
        W = wl.weight((n,), seed=100 + n, sigma=0.02)
        q = oracle.quantize(W)
        nb = -(-n // 64)
        pad = np.zeros(nb * 64, np.float32)
        pad[:n] = W
        a = np.abs(pad.reshape(nb, 64)).max(1)
        assert np.array_equal(q["absmax"], a)
        x = (pad.reshape(nb, 64) / a[:, None]).astype(np.float32).reshape(-1)[:n]
        want = _exact_nearest(x, L)
        assert np.array_equal(_unpack(q["codes"], n), want)
        if n % 2:
            assert q["codes"][-1] & 0xF == 0


def test_absmax_element_and_zero_block():
    W = wl.weight((64 * 8,), seed=5, sigma=1.0).reshape(8, 64)
    W[3] = 0.0
    W[5, 17] = -abs(W[5]).max() * 2
    q = oracle.quantize(W)
    c = _unpack(q["codes"], W.size).reshape(8, 64)
    for b in range(8):
        if b == 3:
            assert np.all(c[b] == 7)  # 0 is a level: an all-zero block is all code 7
            continue
        j = np.argmax(np.abs(W[b]))
        assert c[b, j] == (15 if W[b, j] > 0 else 0)


def test_requantize_is_idempotent():
    """Quantizing the level-times-absmax reconstruction returns the same codes."""
    L, _ = oracle.levels()
    W = wl.weight((64 * 500,), seed=9, sigma=0.02)
    q = oracle.quantize(W)
    c = _unpack(q["codes"], W.size)
    rec = (L[c].reshape(-1, 64) * q["absmax"][:, None]).astype(np.float32).reshape(-1)
    q2 = oracle.quantize(rec)
    assert np.array_equal(q2["codes"], q["codes"])


# ---------------------------------------------------------------- double quantization

def test_mean_equals_exact_rational_mean():
    for n_blocks in (1, 7, 256, 1000, 5000):
        a = np.abs(wl.weight((n_blocks,), seed=n_blocks, sigma=0.05)) + np.float32(1e-3)
        exact = sum(Fraction(float(v)) for v in a) / n_blocks
        mu = oracle.absmax_mean(a.astype(np.float32))
        # the mean is rounded twice (fp64 then fp32); it must be one of the two fp32
        # neighbours of the exact value and the nearest one unless exact is a near-tie
        lo = np.float32(float(exact))
        cands = {lo, np.nextafter(lo, np.float32(-1)), np.nextafter(lo, np.float32(1))}
        assert mu in cands
        assert abs(Fraction(float(mu)) - exact) <= abs(Fraction(float(np.float32(float(exact)))) - exact) + Fraction(1, 2**60)


def test_double_quant_constant_group_has_zero_step():
    W = np.zeros((256, 64), np.float32)
    W[:, 5] = 0.125  # every block absmax == 0.125
    q = oracle.quantize(W)
    assert q["mean"] == np.float32(0.125)
    assert q["steps"][0] == 0.0 and np.all(q["qscale"] == 0)


def test_double_quant_two_value_group():
    W = np.zeros((256, 64), np.float32)
    W[:128, 0] = 0.25
    W[128:, 0] = 0.75
    q = oracle.quantize(W)
    assert q["mean"] == np.float32(0.5)
    assert q["steps"][0] == np.float32(np.float32(0.25) / np.float32(127))
    assert np.all(q["qscale"][:128] == -127) and np.all(q["qscale"][128:] == 127)


def test_double_quant_ties_round_half_to_even():
    """Reading R5 rounds the second-level quotient half to even.  dq_ties builds one group
    whose quotients (a - mu) / step are exact half-integers (mu = 1, step = 2^-7, both exact),
    so each code is fixed by the tie rule alone: 0.5 -> 0, 2.5 -> 2, 126.5 -> 126 (even k, where
    rounding half away from zero would give k + 1), 1.5 -> 2, 3.5 -> 4 (odd k), and the same
    with the signs flipped."""
    from dq_ties import tie_tensor, tie_offsets
    W, expect = tie_tensor()
    q = oracle.quantize(W)
    assert q["mean"] == np.float32(1.0)
    assert q["steps"][0] == np.float32(2.0 ** -7)
    assert np.array_equal(q["qscale"], expect)
    u = tie_offsets()
    got = dict(zip(u.tolist(), q["qscale"][:128].tolist()))
    assert got[0.5] == 0 and got[2.5] == 2 and got[10.5] == 10 and got[62.5] == 62
    assert got[126.5] == 126
    assert got[1.5] == 2 and got[3.5] == 4 and got[11.5] == 12 and got[63.5] == 64
    assert got[127.0] == 127 and got[64.0] == 64 and got[0.0] == 0
    neg = dict(zip((-u).tolist(), q["qscale"][128:].tolist()))
    assert neg[-0.5] == 0 and neg[-2.5] == -2 and neg[-126.5] == -126 and neg[-1.5] == -2
    # half away from zero would differ on every even k: the pin separates the two rules
    away = np.sign(u) * np.floor(np.abs(u) + 0.5)
    even_k = np.isin(u, [0.5, 2.5, 10.5, 62.5, 126.5])
    assert np.all(q["qscale"][:128][even_k] != away[even_k])


def test_double_quant_error_bound_and_range():
    """|ahat - a| <= step/2 (plus fp32 rounding); codes in [-127, 127]; the block with the
    largest |a - mu| in each group gets |q| = 127."""
    W = wl.weight((64 * 256 * 5 + 64 * 3 + 11,), seed=21, sigma=0.02, outlier_frac=0.001)
    q = oracle.quantize(W)
    a, qs, st, mu = q["absmax"], q["qscale"].astype(np.int64), q["steps"], q["mean"]
    g = np.arange(a.size) // 256
    # q * step is exact in fp64 (8-bit times 24-bit significands)
    ahat = (qs.astype(np.float64) * st[g].astype(np.float64) + np.float64(mu)).astype(np.float32)
    err = np.abs(ahat.astype(np.float64) - a.astype(np.float64))
    tol = st[g].astype(np.float64) * (0.5 + 1e-5) + 4 * np.spacing(np.abs(a)).astype(np.float64)
    assert np.all(err <= tol)
    assert qs.min() >= -127 and qs.max() <= 127
    for gi in range(st.size):
        sel = g == gi
        d = np.abs(a[sel].astype(np.float64) - np.float64(mu))
        assert np.abs(qs[sel][np.argmax(d)]) == 127


# ---------------------------------------------------------------- dequantize

def test_bf16_rne_matches_torch_conversion():
    g = wl.rng(3)
    x = np.concatenate([g.standard_normal(20000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, -1.0, 3.4e38, 1e-40, -1e-40], np.float32),
                        (np.arange(1, 3000, dtype=np.uint32) * 0x8000 + 0x3F800000).view(np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_rne(x), want)


def test_dequant_error_bound_and_values():
    """Dequantized weights stay within half the largest level gap times the block scale,
    plus the second-level and bf16 rounding errors (infivelines: each block of 64 weights
    carries its own scale, quantized again in blocks of 256)."""
    L, _ = oracle.levels()
    W = wl.weight((300, 512), seed=31, sigma=0.02, outlier_frac=0.001)
    q = oracle.quantize(W)
    wd = wl.bf16_bits_to_f32(oracle.dequantize(q)).astype(np.float64)
    n = W.size
    b = np.arange(n) // 64
    g = b // 256
    a = q["absmax"][b].astype(np.float64)
    ahat = (q["qscale"][b].astype(np.float64) * q["steps"][g] + np.float64(q["mean"]))
    gap = np.diff(L.astype(np.float64)).max() / 2
    bound = gap * a + np.abs(ahat - a) + np.abs(wd) * 2.0 ** -8 + 1e-12
    assert np.all(np.abs(wd - W.reshape(-1).astype(np.float64)) <= bound)
    # level times recovered scale, rounded to bf16 by torch (a library conversion)
    c = _unpack(q["codes"], n)
    ahat32 = np.array([np.float32(np.float64(qq) * np.float64(s) + np.float64(q["mean"]))
                       for qq, s in zip(q["qscale"][b[::997]], q["steps"][g[::997]])], np.float32)
    prod = (L[c[::997]] * ahat32).astype(np.float32)
    want = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.dequantize(q)[::997], want)


# ---------------------------------------------------------------- storage accounting

def test_storage_matches_the_pages():
    gold = _golden("storage_accounting.txt")
    numel = 4096 * 11008
    q = oracle.quantize(np.zeros(64 * 256 * 2, np.float32))  # shapes only
    assert q["codes"].size == 64 * 256 and q["qscale"].size == 512 and q["steps"].size == 2
    nb, ng = -(-numel // 64), -(-numel // (64 * 256))
    meta_bits = (8 * nb + 32 * ng) / numel
    v, tol, _ = gold["metadata_bits_per_weight"]
    assert abs(meta_bits - v) <= tol * v
    assert meta_bits == pytest.approx(8 / 64 + 32 / (64 * 256), rel=1e-12)
    assert gold["storage_shrink_vs_16bit"][0] == 16 / 4
    for size, k16, k4 in ((7e9, "base_7b_16bit_gb", "base_7b_4bit_gb"),
                          (70e9, "base_70b_16bit_gb", "base_70b_4bit_gb")):
        assert 2 * size / 1e9 == gold[k16][0]
        assert 0.5 * size / 1e9 == gold[k4][0]
    saving = (32 / 64 - meta_bits) * 7e9 / 8 / 1e9  # fp32 absmax per block vs double quant
    assert gold["double_quant_saving_7b_gb_min"][0] < saving < gold["double_quant_saving_7b_gb_max"][0]


# ---------------------------------------------------------------- LoRA forward / backward

def _f(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


@pytest.fixture(scope="module")
def small():
    p = wl.config1()
    W = p.W()
    q = oracle.quantize(W)
    Wd = oracle.dequantize(q).reshape(p.N, p.K)
    return p, Wd, p.X(), p.A(), p.B(), p.dY()


def test_forward_matches_numpy_matmul(small):
    p, Wd, X, A, B, dY = small
    Y, U = oracle.lora_fwd(X, Wd, A, B, p.scale)
    Uref = _f(X) @ _f(A).T
    Yref = _f(X) @ _f(Wd).T + p.scale * (Uref @ _f(B).T)
    assert np.allclose(U, Uref, rtol=1e-12, atol=1e-12)
    assert np.allclose(Y, Yref, rtol=1e-12, atol=1e-12)
    rows = np.array([3, 0, 15], np.int64)
    Ys, _ = oracle.lora_fwd(X, Wd, A, B, p.scale, rows)
    assert np.array_equal(Ys, Y[rows])


def test_zero_b_reduces_to_base_matmul(small):
    p, Wd, X, A, B, dY = small
    B0 = np.zeros_like(B)
    Y, _ = oracle.lora_fwd(X, Wd, A, B0, p.scale)
    assert np.allclose(Y, _f(X) @ _f(Wd).T, rtol=1e-12, atol=1e-12)
    dA, dB = oracle.lora_dadb(dY, X, A, B0, p.scale)
    assert np.all(dA == 0.0)
    A0 = np.zeros_like(A)
    dA, dB = oracle.lora_dadb(dY, X, A0, B, p.scale)
    assert np.all(dB == 0.0)


def test_backward_is_adjoint_of_forward(small):
    """<dY, Y> pairs with the gradients: Y is linear in X, in A and in B separately, so
    <dY, dY/dX-direction> identities pin every transpose and index of the backward."""
    p, Wd, X, A, B, dY = small
    s = p.scale
    g = _f(dY)
    Y, _ = oracle.lora_fwd(X, Wd, A, B, s)
    dX, V = oracle.lora_dx(dY, Wd, A, B, s)
    dA, dB = oracle.lora_dadb(dY, X, A, B, s)
    lhs = (g * Y).sum()
    assert lhs == pytest.approx((dX * _f(X)).sum(), rel=1e-10)
    Y_noA, _ = oracle.lora_fwd(X, Wd, np.zeros_like(A), B, s)
    lora = (g * (Y - Y_noA)).sum()
    assert lora == pytest.approx((dA * _f(A)).sum(), rel=1e-9)
    assert lora == pytest.approx((dB * _f(B)).sum(), rel=1e-9)
    assert np.allclose(V, g @ _f(B), rtol=1e-12, atol=1e-12)
    assert np.allclose(dX, g @ _f(Wd) + s * (g @ _f(B)) @ _f(A), rtol=1e-12, atol=1e-12)


def test_backward_finite_difference(small):
    """Central differences of L = <dY, Y> in fp64 along random directions."""
    p, Wd, X, A, B, dY = small
    s = p.scale
    g = _f(dY)
    Xf, Af, Bf, Wf = _f(X), _f(A), _f(B), _f(Wd)

    def loss(Xv, Av, Bv):
        return (g * (Xv @ Wf.T + s * (Xv @ Av.T) @ Bv.T)).sum()

    dX, _ = oracle.lora_dx(dY, Wd, A, B, s)
    dA, dB = oracle.lora_dadb(dY, X, A, B, s)
    r = wl.rng(77)
    for grad, which in ((dX, 0), (dA, 1), (dB, 2)):
        D = r.standard_normal(grad.shape)
        h = 1e-3
        args_p = [Xf, Af, Bf]
        args_m = [Xf, Af, Bf]
        args_p[which] = args_p[which] + h * D
        args_m[which] = args_m[which] - h * D
        fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert fd == pytest.approx((grad * D).sum(), rel=1e-6)


# ---------------------------------------------------------------- merge (reading R11)

def _bf16_nearest_exact(x: Fraction) -> int:
    """Brute force: bits of the bf16 nearest to the rational x, ties to the even pattern."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    ax = -x if x < 0 else x
    # bracket ax between consecutive positive bf16 values by bisection on the bit pattern
    lo, hi = 0, 0x7F80  # +0 .. +inf
    val = lambda b: Fraction(float(wl.bf16_bits_to_f32(np.array([b], np.uint16))[0]))
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if val(mid) <= ax:
            lo = mid
        else:
            hi = mid
    dl, dh = ax - val(lo), val(hi) - ax
    b = lo if dl < dh or (dl == dh and lo % 2 == 0) else hi
    return sign | b


def test_bf16_rne_double_against_exact_rounding():
    g = wl.rng(11)
    xs = list(g.standard_normal(300) * 10.0 ** g.integers(-30, 30, 300))
    xs += [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 3e-39, 2.0 ** -133,
           1.5 * 2.0 ** -133, 1.0 + 2.0 ** -8 + 2.0 ** -40]
    want = np.array([_bf16_nearest_exact(Fraction(float(x))) for x in xs], np.uint16)
    assert np.array_equal(oracle.bf16_rne_double(xs), want)


def test_merge_with_zero_adapter_is_the_dequantization():
    W = wl.weight((64, 128), seed=21, sigma=0.02)
    q = oracle.quantize(W)
    A = wl.bf16_normal((8, 128), seed=22, sigma=0.01)
    B = np.zeros((64, 8), np.uint16)
    got = oracle.merge(oracle.dequantize(q).reshape(64, 128), A, B, 2.0)
    assert np.array_equal(got.ravel(), oracle.dequantize(q))


def test_merge_brute_force_small():
    """Every element from exact rational arithmetic rounded once (R11)."""
    N, K, r, s = 6, 64, 3, 0.75
    W = wl.weight((N, K), seed=23, sigma=0.02)
    q = oracle.quantize(W)
    Wd = wl.bf16_bits_to_f32(oracle.dequantize(q)).reshape(N, K)
    A = wl.bf16_normal((r, K), seed=24, sigma=0.01)
    B = wl.bf16_normal((N, r), seed=25, sigma=0.01)
    Af, Bf = wl.bf16_bits_to_f32(A), wl.bf16_bits_to_f32(B)
    want = np.zeros((N, K), np.uint16)
    for n in range(N):
        for k in range(K):
            d = sum(Fraction(float(Bf[n, j])) * Fraction(float(Af[j, k])) for j in range(r))
            want[n, k] = _bf16_nearest_exact(Fraction(float(Wd[n, k])) + Fraction(s) * d)
    assert np.array_equal(oracle.merge(oracle.dequantize(q).reshape(N, K), A, B, s), want)


# ---------------------------------------------------------------- NF4 vs INT4 (reading R12)

def test_int4_error_zero_on_each_grid_and_sum_of_squares():
    L, _ = oracle.levels()
    g = wl.rng(31)
    a = np.float32(0.5)
    # every block holds the absmax and otherwise NF4 levels times it: NF4 error is exactly 0
    c = g.integers(0, 16, size=(64, 64))
    c[:, 0] = 15
    Wn = (L[c] * a).astype(np.float32).ravel()
    s = oracle.int4_error(Wn)
    assert s[1] == 0.0 and s[2] > 0.0
    assert s[0] == pytest.approx(float(np.sum(Wn.astype(np.float64) ** 2)), rel=1e-12)
    # absmax 7 * 2^-6 and multiples of 2^-6: exactly on the INT4 grid
    qv = g.integers(-7, 8, size=(64, 64)).astype(np.float32)
    qv[:, 0] = 7
    Wi = (qv * np.float32(2.0 ** -6)).ravel()
    assert oracle.int4_error(Wi)[2] == 0.0


def test_int4_error_brute_force_small():
    """Exact nearest level (fp64 argmin, ties down) and plain rint for INT4."""
    W = wl.weight((16, 64), seed=32, sigma=0.02)
    L, _ = oracle.levels()
    Wb = W.reshape(-1, 64)
    a = np.abs(Wb).max(axis=1, keepdims=True)
    x = (Wb / a).astype(np.float32)
    c = _exact_nearest(x.ravel(), L).reshape(x.shape)
    en = Wb.astype(np.float64) - L[c].astype(np.float64) * a.astype(np.float64)
    qv = np.clip(np.rint((np.float32(7.0) * x).astype(np.float32)), -7, 7)
    ei = Wb.astype(np.float64) - qv.astype(np.float64) * (a / np.float32(7.0)).astype(np.float32).astype(np.float64)
    got = oracle.int4_error(W)
    assert got[1] == pytest.approx(float((en ** 2).sum()), rel=1e-12)
    assert got[2] == pytest.approx(float((ei ** 2).sum()), rel=1e-12)


def test_nf4_beats_int4_on_normal_weights():
    """aicurriculum 'Design Details That Matter': NF4 (normal quantiles) is often better
    than naive INT4; on normally distributed weights its squared error is clearly lower."""
    W = wl.weight((256, 1024), seed=33, sigma=0.02)
    s = oracle.int4_error(W)
    assert s[1] < 0.9 * s[2]


# ---------------------------------------------------------------- no double quantization (R14)

def test_dequantize_nodq_is_level_times_true_absmax():
    """Without the second level the block scale is the stored absmax: every weight
    dequantizes to bf16(L[c] * absmax) (numpy fp32 product, torch's bf16 rounding)."""
    W = wl.weight((1, 64 * 40 + 13), seed=91, sigma=0.02).ravel()
    q = oracle.quantize(W)
    L, _ = oracle.levels()
    c = _unpack(q["codes"], W.size)
    a = np.repeat(q["absmax"], 64)[:W.size]
    want = wl.to_bf16_bits((L[c] * a).astype(np.float32))
    assert np.array_equal(oracle.dequantize_nodq(q), want)
    assert np.array_equal(q["absmax"], np.abs(np.pad(W, (0, (-W.size) % 64))).reshape(-1, 64).max(1))


# ---------------------------------------------------------------- fp8 second level (R15)

def test_e4m3_codec_matches_torch_and_the_format():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    fin = ~np.isnan(want)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(got[fin], want[fin])
    assert got[0x7E] == 448.0 and got[0x38] == 1.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9
    g = wl.rng(61)
    x = np.concatenate([g.standard_normal(3000) * 10.0 ** g.integers(-3, 3, 3000),
                        got[fin][::3] + 1e-9, (got[1:0x7E] + got[2:0x7F]) / 2]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    want_enc = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), want_enc)
    assert list(oracle.e4m3_encode(np.array([500.0, -1e9, 449.0], np.float32))) == [0x7E, 0xFE, 0x7E]


def test_fp8_second_level_error_bound_and_extremes():
    """Every block scale is recovered within half an E4M3 step of its distance from the
    mean (relative 2^-4), and the largest |a - mean| of a group maps to +-448."""
    W = wl.weight((64 * 256 * 3 + 640,), seed=62, sigma=0.02)
    q = oracle.quantize(W, fp8=True)
    a = q["absmax"].astype(np.float64)
    qv = oracle.e4m3_decode(q["qscale"].view(np.uint8))
    step = np.repeat(q["steps"].astype(np.float64), 256)[:a.size]
    ahat = qv * step + np.float64(q["mean"])
    d = np.abs(a - np.float64(q["mean"]))
    assert np.all(np.abs(ahat - a) <= d * 2.0 ** -4 + step * 2.0 ** -9 + 1e-12)
    for gidx in range(q["steps"].size):
        seg = slice(256 * gidx, min(256 * gidx + 256, a.size))
        assert np.max(np.abs(qv[seg])) == 448.0


# ---------------------------------------------------------------- fp16 compute type (R16)
# digipro.cn "QLoRA: Fine-Tuning a 7B Model on a 16GB GPU", "The QLoRA insight": the
# compute-dtype flag dequantizes to fp16 for the matrix multiplies.

def test_f16_decode_matches_numpy_on_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_double(bits)
    want = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    assert np.array_equal(got[fin], want[fin])
    assert got[0x3C00] == 1.0 and got[0x0001] == 2.0 ** -24 and got[0x7BFF] == 65504.0


def test_f16_rne_double_matches_numpy_and_ties():
    """numpy converts fp64 to binary16 with one round-to-nearest-even; so must the oracle,
    through normals, subnormals, exact ties and the overflow edge."""
    g = wl.rng(71)
    vals = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (vals[:-1] + vals[1:]) / 2            # exact ties (representable in fp64)
    x = np.concatenate([g.standard_normal(4000) * 10.0 ** g.integers(-9, 5, 4000),
                        mids[::7], -mids[::11], mids[::13] * (1 + 2.0 ** -40),
                        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -25,
                         2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26]])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f16_rne_double(x), want)


def test_dequantize_f16_is_library_rounding_of_the_same_product():
    """The fp16 dequantization rounds the same fp32 product L[c] * ahat as the bf16 one:
    numpy's binary16 conversion of it (a library rounding) for double-quantized and for
    absmax scales, with values small enough to reach binary16 subnormals."""
    L, _ = oracle.levels()
    W = wl.weight((3, 64 * 90 + 17), seed=72, sigma=0.02, outlier_frac=0.001).ravel()
    W[: 64 * 3] *= 2.0 ** -14                    # blocks whose products are fp16 subnormals
    q = oracle.quantize(W)
    n = W.size
    c = _unpack(q["codes"], n)
    b = np.arange(n) // 64
    ahat = np.array([np.float32(np.float64(qq) * np.float64(s) + np.float64(q["mean"]))
                     for qq, s in zip(q["qscale"], np.repeat(q["steps"], 256)[:q["qscale"].size])],
                    np.float32)
    prod = (L[c] * ahat[b]).astype(np.float32)
    assert np.array_equal(oracle.dequantize(q, f16=True), prod.astype(np.float16).view(np.uint16))
    prod0 = (L[c] * np.repeat(q["absmax"], 64)[:n]).astype(np.float32)
    assert np.array_equal(oracle.dequantize_nodq(q, f16=True),
                          prod0.astype(np.float16).view(np.uint16))
    sub = oracle.dequantize(q, f16=True)[: 64 * 3]
    assert np.any((sub & 0x7C00) == 0) and np.any(sub & 0x3FF)


def test_lora_f16_inputs_match_numpy_matmul():
    """With f16 every 16-bit input is read as binary16: forward, dX, dA and dB equal the fp64
    numpy products of the binary16 values."""
    g = wl.rng(73)
    M, N, K, r, s = 24, 64, 128, 8, 0.75
    h = lambda *shape: (g.standard_normal(shape) * 0.5).astype(np.float16)
    X, Wd, A, B, dY = h(M, K), h(N, K), h(r, K), h(N, r), h(M, N)
    u = lambda a: a.view(np.uint16)
    d = lambda a: a.astype(np.float64)
    Y, U = oracle.lora_fwd(u(X), u(Wd), u(A), u(B), s, f16=True)
    assert np.allclose(U, d(X) @ d(A).T, rtol=1e-12, atol=1e-12)
    assert np.allclose(Y, d(X) @ d(Wd).T + s * (d(X) @ d(A).T) @ d(B).T, rtol=1e-12, atol=1e-12)
    dX, V = oracle.lora_dx(u(dY), u(Wd), u(A), u(B), s, f16=True)
    assert np.allclose(V, d(dY) @ d(B), rtol=1e-12, atol=1e-12)
    assert np.allclose(dX, d(dY) @ d(Wd) + s * (d(dY) @ d(B)) @ d(A), rtol=1e-12, atol=1e-12)
    dA, dB = oracle.lora_dadb(u(dY), u(X), u(A), u(B), s, f16=True)
    assert np.allclose(dA, s * (d(dY) @ d(B)).T @ d(X), rtol=1e-12, atol=1e-12)
    assert np.allclose(dB, s * d(dY).T @ (d(X) @ d(A).T), rtol=1e-12, atol=1e-12)
    # the same bits read as bf16 give a different answer: the flag is live
    Yb, _ = oracle.lora_fwd(u(X), u(Wd), u(A), u(B), s)
    assert not np.allclose(Yb, Y)
