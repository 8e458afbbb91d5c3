"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: packed codes, second-level scale codes, steps, mean, dequantized bf16 weights.
Relative Frobenius error <= 5e-3 against the fp64 oracle: Y, U, dX, dA, dB.
"""
import os
import zlib

import numpy as np
import pytest
import torch

import oracle
import bit_nf4_quantized_37_b300 as qn
from bit_nf4_quantized_37_b300 import workloads as wl
from gpu_helpers import (TOL, Problem, bf16_dev, bits_host, f32_host, rel_fro,
                         upload_oracle_tensor)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_37_b300 import build
    build.build()
    qn.lib()
    yield
    assert qn.device_status() == 0


def _quant_parity(W: np.ndarray):
    q = qn.nf4_quantize(torch.from_numpy(W).cuda())
    o = oracle.quantize(W)
    assert np.array_equal(q.codes.cpu().numpy(), o["codes"])
    assert np.array_equal(q.scale_codes.cpu().numpy(), o["qscale"])
    assert np.array_equal(q.scale_steps.cpu().numpy().view(np.uint32), o["steps"].view(np.uint32))
    assert q.scale_mean.cpu().numpy()[0].view(np.uint32) == np.float32(o["mean"]).view(np.uint32)
    return q, o


# ------------------------------------------------------------------ quantize / dequantize
@pytest.mark.parametrize("n", [1, 2, 63, 64, 65, 127, 1001, 64 * 256, 64 * 256 + 1,
                               64 * 300 + 37, 64 * 256 * 5 + 3, 1 << 20])
def test_quantize_bit_exact_ragged(n):
    W = wl.weight((1, n), seed=500 + n, sigma=0.02, outlier_frac=0.001 if n > 5000 else 0.0)
    _quant_parity(W)


def test_quantize_special_blocks():
    W = wl.weight((64 * 512,), seed=3, sigma=0.02).reshape(512, 64)
    W[5] = 0.0                      # all-zero block
    W[9] = 0.125                    # constant block
    W[11, 3] = 1e-30                # tiny absmax
    W[12, :] = -W[12, :]
    W[200:456] = W[200]             # a whole group of identical blocks
    _quant_parity(W.reshape(1, -1))


def test_quantize_second_level_ties():
    """A group whose second-level quotients are exact half-integers (tests/dq_ties.py): the
    int8 codes follow rounding half to even, bit for bit with the oracle."""
    from dq_ties import tie_tensor
    W, expect = tie_tensor()
    q, o = _quant_parity(W)
    assert np.array_equal(q.scale_codes.cpu().numpy(), expect)


def test_quantize_near_thresholds():
    """Weights planted within a few ulps of level boundaries (w ~ T_i * absmax): the
    quotient w / absmax lands next to a threshold, where the quantizer must take its exact
    division path to stay bit-exact."""
    L, T = oracle.levels()
    g = wl.rng(44)
    nb = 64 * 256 * 4  # whole groups of 256 blocks
    a = g.uniform(0.005, 1.5, size=nb).astype(np.float32)
    i = g.integers(0, 15, size=(nb, 64))
    base = (T[i].astype(np.float32) * a[:, None]).astype(np.float32)
    k = g.integers(-3, 4, size=(nb, 64)).astype(np.int32)
    W = (base.view(np.int32) + k).view(np.float32)
    W[:, 0] = np.where(g.integers(0, 2, size=nb) == 1, a, -a)  # absmax element
    W = np.clip(W, -a[:, None], a[:, None]).astype(np.float32)
    _quant_parity(W.reshape(1, -1))


def test_quantize_config_tensors_bit_exact():
    _quant_parity(wl.config1().W())
    _quant_parity(wl.config2().W())
    _quant_parity(wl.config3()[2].W())


def test_quantize_decode_tensor_bit_exact():
    _quant_parity(wl.config4(1).W())


@pytest.mark.parametrize("rows", [2048, 5000, 9000])
def test_quantize_mean_partitions(rows):
    """The mean's pairwise tree cut into 16, 64 and 128 subtree sums (8.4 M, 20.5 M and
    36.9 M weights), the last of which the final CTA of that pass combines."""
    _quant_parity(wl.weight((rows, 4096), seed=rows, sigma=0.02, outlier_frac=0.001))


@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 17), (3, 333), (256, 256), (64, 64 * 256 + 64),
                                       (4096, 4096)])
def test_dequantize_bit_exact(rows, cols):
    W = wl.weight((rows, cols), seed=rows * 7 + cols, sigma=0.02, outlier_frac=0.001)
    o = oracle.quantize(W)
    want = oracle.dequantize(o)
    # from the oracle's own encoding (independent of the GPU quantizer)
    qd = upload_oracle_tensor(o, rows, cols)
    got = bits_host(qn.nf4_dequantize(qd)).reshape(-1)
    assert np.array_equal(got, want)
    # and round trip through the GPU quantizer
    q = qn.nf4_quantize(torch.from_numpy(W).cuda())
    assert np.array_equal(bits_host(qn.nf4_dequantize(q)).reshape(-1), want)


def test_dequantize_decode_tensor_bit_exact():
    p = wl.config4(1)
    W = p.W()
    o = oracle.quantize(W)
    want = oracle.dequantize(o)
    q = qn.nf4_quantize(torch.from_numpy(W).cuda())
    got = bits_host(qn.nf4_dequantize(q)).reshape(-1)
    assert np.array_equal(got, want)


# ------------------------------------------------------------------ forward / backward
def _check_fwd(pb: Problem, rows=None):
    p = pb.p
    fwd = qn.qlora_linear_fwd_f16 if pb.half else qn.qlora_linear_fwd
    Y, U = fwd(pb.Xd, pb.qd, pb.Ad, pb.Bd, p.scale)
    assert Y.dtype == (torch.float16 if pb.half else torch.bfloat16)
    Yo, Uo = oracle.lora_fwd(pb.X, pb.Wd, pb.A, pb.B, p.scale, rows, f16=pb.half)
    Yg = f32_host(Y)
    Ug = f32_host(U)
    if rows is not None:
        Yg, Ug = Yg[rows], Ug[rows]
    ey, eu = rel_fro(Yg, Yo), rel_fro(Ug, Uo)
    assert ey <= TOL, ey
    assert eu <= TOL, eu
    return Y, U


def _check_bwd(pb: Problem, U, rows=None):
    p = pb.p
    bwd = qn.qlora_linear_bwd_f16 if pb.half else qn.qlora_linear_bwd
    dX, dA, dB = bwd(pb.dYd, pb.Xd, pb.qd, pb.Ad, pb.Bd, p.scale, U)
    dXo, _ = oracle.lora_dx(pb.dY, pb.Wd, pb.A, pb.B, p.scale, rows, f16=pb.half)
    dAo, dBo = oracle.lora_dadb(pb.dY, pb.X, pb.A, pb.B, p.scale, f16=pb.half)
    dXg = f32_host(dX)
    if rows is not None:
        dXg = dXg[rows]
    ex = rel_fro(dXg, dXo)
    assert ex <= TOL, ex
    if np.linalg.norm(dAo) > 0:
        ea = rel_fro(f32_host(dA), dAo)
        assert ea <= TOL, ea
    else:
        assert np.all(f32_host(dA) == 0)
    eb = rel_fro(f32_host(dB), dBo)
    assert eb <= TOL, eb
    return dX, dA, dB


SMALL = [
    # name, M, N, K, r, alpha
    ("cfg1", 16, 256, 256, 8, 16.0),
    ("ragged", 200, 320, 448, 16, 32.0),
    ("rank40", 130, 512, 256, 40, 16.0),
    ("rank72", 129, 256, 320, 72, 16.0),
    ("rank128", 300, 384, 512, 128, 64.0),
    ("tokens17", 17, 640, 192, 16, 32.0),
    ("tokens1", 1, 576, 320, 8, 16.0),
    ("tokens5", 5, 256, 1024, 64, 16.0),
    ("multi_tile", 520, 1024, 1088, 16, 32.0),
    ("rank12", 150, 256, 320, 12, 24.0),     # rank not a multiple of 8: padded B path
    ("rank3", 40, 192, 128, 3, 6.0),
    ("tokens9_rank13", 9, 320, 256, 13, 26.0),
    # few tokens, long contractions: the input gradient on 128-row tiles with a split
    # contraction (its workspace is needed below the decode path's token limit too)
    ("tokens1_split", 1, 2048, 4096, 64, 16.0),
    ("tokens5_split", 5, 1088, 2560, 24, 48.0),
    # more row tiles than a quarter of the SMs: U and V with the split contraction and the
    # last-CTA sum (below that they take one CTA per row tile and the whole contraction)
    ("tall_split_side", 4800, 256, 320, 16, 32.0),
]


@pytest.mark.parametrize("name,M,N,K,r,alpha", SMALL)
def test_fwd_bwd_small(name, M, N, K, r, alpha):
    p = wl.LinearProblem(name, M, N, K, r, alpha, 0.02, 0.001, config=90 + len(name))
    pb = Problem(p)
    Y, U = _check_fwd(pb)
    _check_bwd(pb, U)
    _check_bwd(pb, None)  # U recomputed in the backward


@pytest.mark.parametrize("M,N,K,r", [(2000, 4800, 320, 24),    # forward on CTA pairs
                                     (2000, 320, 4800, 40),    # input gradient on CTA pairs
                                     (2100, 4864, 256, 16),    # forward pairs, 5th pair row partial
                                     (2100, 256, 4864, 16),    # input gradient, the same
                                     (512, 3072, 3072, 16),    # 128-row tiles, 3-way split contraction
                                     (400, 3072, 2560, 24),    # the same, rows past M in the tile
                                     (700, 768, 640, 16),      # staged base, six row tiles, ragged
                                     (384, 640, 576, 24),      # staged base, three row tiles
                                     (512, 4096, 4096, 16),    # two splits as a cluster, both ways
                                     (300, 2048, 1024, 16),    # the same with a ragged row tile
                                     (1024, 4864, 512, 128),   # narrow U at rank 128 (unswizzled rows)
                                     (1024, 512, 4864, 128)])  # narrow V at rank 128
def test_pair_tiles_every_output(M, N, K, r):
    """The fused GEMMs against the oracle on every output element: the CTA pairs (512 x 256
    tiles: all 16 row classes of a pair tile -- 2 CTAs x 2 accumulators x 4 TMEM lane groups
    -- and partial last tiles in M and in the output columns), and single-CTA tiles with the
    contraction split (fp32 tiles summed in split order by the CTA completing the tile) in
    both directions."""
    p = wl.LinearProblem(f"pairs-{M}-{N}-{K}", M, N, K, r, 2.0 * r, 0.02, 0.001, config=60 + r)
    pb = Problem(p)
    Y, U = _check_fwd(pb)
    _check_bwd(pb, U)
    if M == 2100:
        _check_bwd(pb, None)  # U recomputed (split form) before the narrow V


def test_base_past_staging_limit():
    """One-CTA tiles over two row tiles with a base too large to stage in the workspace
    (8192 x 8256 > 64 Mi weights): W' is dequantized inside both GEMMs, once per row tile,
    with a two-way split contraction.  (Smaller bases at more than 128 tokens on one-CTA
    tiles are dequantized once into the workspace and streamed by TMA: the ragged, rank and
    multi-tile cases above and the 7B-stack layers.)  Sampled rows of Y and dX, U / dA / dB
    in full."""
    p = wl.LinearProblem("unstaged-160-8192-8256", 160, 8192, 8256, 16, 32.0, 0.02, 0.001,
                         config=77)
    pb = Problem(p)
    rows = _sample_rows(p.M, 24, p.name)
    Y, U = _check_fwd(pb, rows)
    _check_bwd(pb, U, rows)


def test_arrival_tickets_zeroed_without_memset():
    """A call whose U / V take the narrow form (one CTA per 128-row tile beside a pair GEMM)
    launches no ticket memset: the narrow kernel zeroes the arrival counters that split-form
    kernels later in the call use (dA here).  The cached workspace is filled with 0xFF bytes
    before each call, so a counter left unzeroed would lose dA's split sums.  The backward
    also recomputes U (split form, with the memset) once."""
    from bit_nf4_quantized_37_b300 import _binding as bnd
    p = wl.LinearProblem("tickets-1024-4864-4864", 1024, 4864, 4864, 16, 32.0, 0.02, 0.001,
                         config=78)
    pb = Problem(p)
    rows = _sample_rows(p.M, 16, p.name)

    def dirty():
        torch.cuda.synchronize()
        for buf in bnd._ws_cache.values():
            buf.fill_(0xFF)
        torch.cuda.synchronize()

    qn.qlora_linear_fwd(pb.Xd, pb.qd, pb.Ad, pb.Bd, p.scale)  # sizes the cached workspace
    dirty()
    Y, U = _check_fwd(pb, rows)
    dirty()
    _check_bwd(pb, U, rows)
    dirty()
    _check_bwd(pb, None, rows)


def test_zero_b_equals_base_matmul():
    pb = Problem(wl.config1(b_zero=True))
    p = pb.p
    Y, U = qn.qlora_linear_fwd(pb.Xd, pb.qd, pb.Ad, pb.Bd, p.scale)
    base = wl.bf16_bits_to_f32(pb.X).astype(np.float64) @ wl.bf16_bits_to_f32(pb.Wd).astype(np.float64).T
    assert rel_fro(f32_host(Y), base) <= TOL
    dX, dA, dB = qn.qlora_linear_bwd(pb.dYd, pb.Xd, pb.qd, pb.Ad, pb.Bd, p.scale, U)
    assert np.all(dA.cpu().numpy() == 0.0)
    # same with the fused GEMM path (M > 16)
    p2 = wl.LinearProblem("bzero-fused", 96, 256, 256, 8, 16.0, config=1, b_zero=True)
    pb2 = Problem(p2)
    Y2, _ = qn.qlora_linear_fwd(pb2.Xd, pb2.qd, pb2.Ad, pb2.Bd, p2.scale)
    base2 = wl.bf16_bits_to_f32(pb2.X).astype(np.float64) @ wl.bf16_bits_to_f32(pb2.Wd).astype(np.float64).T
    assert rel_fro(f32_host(Y2), base2) <= TOL


def test_base_is_frozen_and_results_reproducible():
    p = wl.LinearProblem("repro", 300, 512, 512, 16, 32.0, config=77)
    pb = Problem(p)
    before = [t.clone() for t in (pb.qd.codes, pb.qd.scale_codes, pb.qd.scale_steps, pb.qd.scale_mean)]
    Y1, U1 = qn.qlora_linear_fwd(pb.Xd, pb.qd, pb.Ad, pb.Bd, p.scale)
    g1 = qn.qlora_linear_bwd(pb.dYd, pb.Xd, pb.qd, pb.Ad, pb.Bd, p.scale, U1)
    Y2, U2 = qn.qlora_linear_fwd(pb.Xd, pb.qd, pb.Ad, pb.Bd, p.scale)
    g2 = qn.qlora_linear_bwd(pb.dYd, pb.Xd, pb.qd, pb.Ad, pb.Bd, p.scale, U2)
    after = (pb.qd.codes, pb.qd.scale_codes, pb.qd.scale_steps, pb.qd.scale_mean)
    for b, a in zip(before, after):
        assert torch.equal(b, a)
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    assert torch.equal(U1, U2)
    for x, y in zip(g1, g2):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)


# ------------------------------------------------------------------ full-size workloads
def _sample_rows(M, n, key: str):
    """Sampled token rows for the oracle: the first and last row plus n rows drawn with a
    seed of their own for every test (key), so tests on one shape check different rows."""
    r = np.random.default_rng(zlib.crc32(key.encode()))
    rows = np.unique(np.concatenate([[0, M - 1], r.choice(M, size=min(n, M), replace=False)]))
    return rows.astype(np.int64)


def test_config2_attention_projection():
    """The headline shape on the CTA-pair kernels, every output element of Y and dX."""
    pb = Problem(wl.config2())
    Y, U = _check_fwd(pb)
    _check_bwd(pb, U)


@pytest.mark.parametrize("which", [0, 1, 2])
def test_config3_mlp_projection(which):
    pb = Problem(wl.config3()[which])
    rows = _sample_rows(pb.p.M, 64, f"config3-{which}")
    Y, U = _check_fwd(pb, rows)
    _check_bwd(pb, U, rows)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_config4_decode(M):
    pb = Problem(wl.config4(M))
    _check_fwd(pb)


@pytest.mark.parametrize("layer", [0, 15, 31])
def test_config5_layer_gemms(layer):
    """Every projection of three layers of the 32-layer stack at M = 512 (all-linear LoRA):
    Y and dX on sampled rows, U, dA and dB in full."""
    for p in wl.config5(layer=layer):
        pb = Problem(p)
        rows = _sample_rows(p.M, 24, p.name)
        Y, U = _check_fwd(pb, rows)
        _check_bwd(pb, U, rows)


def test_config5_quantize_every_layer_bit_exact():
    """nf4_quantize on all 224 weight matrices of the 32-layer stack (6.48 G weights), each
    bit-exact with the oracle.  The oracle runs in spawned worker processes (no GPU state)."""
    import concurrent.futures as cf
    import multiprocessing as mp

    import oracle_pool
    workers = max(1, min(8, (os.cpu_count() or 2) // 2))
    with cf.ProcessPoolExecutor(workers, mp_context=mp.get_context("spawn")) as ex, \
            cf.ThreadPoolExecutor(7) as gen:
        for layer, ref in enumerate(ex.map(oracle_pool.quantize_stack_layer, range(32))):
            projs = wl.config5(layer=layer)
            weights = list(gen.map(lambda p: p.W(), projs))  # the seeded draws, in threads
            for p, W, (name, codes, qs, steps, mean) in zip(projs, weights, ref):
                assert p.name == name
                q = qn.nf4_quantize(torch.from_numpy(W).cuda())
                assert np.array_equal(q.codes.cpu().numpy(), codes), name
                assert np.array_equal(q.scale_codes.cpu().numpy(), qs), name
                assert np.array_equal(q.scale_steps.cpu().numpy().view(np.uint32),
                                      steps.view(np.uint32)), name
                assert q.scale_mean.cpu().numpy()[0].view(np.uint32) == mean.view(np.uint32), name


# ------------------------------------------------------------------ error paths
def test_bad_arguments_raise():
    pb = Problem(wl.config1())
    with pytest.raises(ValueError):
        qn.qlora_linear_fwd(pb.Xd.float(), pb.qd, pb.Ad, pb.Bd, 2.0)
    # N = 250 is not a multiple of 64: the library refuses the shape (the binding's own shape
    # checks pass: B has N rows)
    bad = qn.NF4Tensor(pb.qd.codes, pb.qd.scale_codes, pb.qd.scale_steps, pb.qd.scale_mean, 250, 256)
    with pytest.raises(qn.QLoRAError):
        qn.qlora_linear_fwd(pb.Xd[:, :256], bad, pb.Ad, pb.Bd[:250].contiguous(), 2.0)
    with pytest.raises(ValueError):  # B rows do not match the base's N
        qn.qlora_linear_fwd(pb.Xd, pb.qd, pb.Ad, pb.Bd[:128].contiguous(), 2.0)


# ------------------------------------------------------------------ merge / requantize
def _ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 steps between two arrays of bf16 bits (sign-magnitude order)."""
    def key(h):
        h = h.astype(np.int64)
        return np.where(h & 0x8000, -(h & 0x7FFF), h & 0x7FFF)
    return np.abs(key(a) - key(b))


def _check_merge(p):
    """bf16(W' + s B A): the device's fp32 bracket against the oracle's fp64 one, each rounded
    once to bf16.  Bound from the fp32 arithmetic: the r exact bf16 x bf16 products summed on
    the tensor cores (r additions; their fp32 accumulation is not specified as
    round-to-nearest, so a unit of 2^-23 each), one multiply and one add leave at most
    (2 r + 2) 2^-24 (|W'| + s sum_j |B A|) before the final rounding, so the two results differ
    by at most that plus one bf16 step of the result; more than one step only where W' and
    s B A nearly cancel.  Differences of any size are rare (~2^-16)."""
    W = p.W()
    qo = oracle.quantize(W)
    qd = qn.nf4_quantize(torch.from_numpy(W).cuda())
    A, B = p.A(), p.B()
    m16, m32 = qn.nf4_merge_lora(qd, bf16_dev(A), bf16_dev(B), p.scale, f32=True)
    got = bits_host(m16)
    want = oracle.merge(oracle.dequantize(qo).reshape(p.N, p.K), A, B, p.scale)
    d = _ulp_diff(got, want)
    assert (d > 0).mean() <= 1e-3
    gv = wl.bf16_bits_to_f32(got).astype(np.float64)
    wv = wl.bf16_bits_to_f32(want).astype(np.float64)
    wd = wl.bf16_bits_to_f32(oracle.dequantize(qo)).astype(np.float64).reshape(p.N, p.K)
    mag = np.abs(wd) + p.scale * (np.abs(wl.bf16_bits_to_f32(B).astype(np.float64)) @
                                  np.abs(wl.bf16_bits_to_f32(A).astype(np.float64)))
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(wv), 2.0 ** -126))) - 7)
    bound = (2 * p.r + 2) * 2.0 ** -24 * mag + step
    assert np.all(np.abs(gv - wv) <= bound)
    assert np.array_equal(m32.cpu().numpy(), wl.bf16_bits_to_f32(got))


@pytest.mark.parametrize("cfg", ["config1", "config2"])
def test_merge_matches_oracle(cfg):
    """The merge on the config shapes (ranks 8 and 16: the persistent form)."""
    _check_merge(getattr(wl, cfg)())


@pytest.mark.parametrize("N,K,r", [(200, 320, 24),    # persistent form, rank 24 (32-wide slices)
                                   (200, 320, 12),    # one-tile form: rank not a multiple of 8
                                   (130, 448, 40),    # one-tile form: rank past 32
                                   (64, 8192, 128)])  # one-tile form at the largest rank
def test_merge_ranks_and_ragged(N, K, r):
    """The merge's two forms on ragged tiles (rows past N, columns past K in the last tiles)."""
    p = wl.LinearProblem(f"merge-{N}-{K}-{r}", 16, N, K, r, 2.0 * r, 0.02, 0.001, config=79)
    _check_merge(p)


def test_merge_zero_adapter_is_dequantize():
    p = wl.config1()
    qd = qn.nf4_quantize(torch.from_numpy(p.W()).cuda())
    B = np.zeros((p.N, p.r), np.uint16)
    m16, _ = qn.nf4_merge_lora(qd, bf16_dev(p.A()), bf16_dev(B), p.scale)
    assert np.array_equal(bits_host(m16), bits_host(qn.nf4_dequantize(qd)))


def test_requantized_merge_bit_exact_and_loses_the_adapter():
    """Requantizing the merged weights (the pages' dequantize -> merge -> requantize path) is
    bit-exact with the oracle's quantization of the same merged values; its reconstruction
    error is of the size of the adapter update, so most of that update is lost."""
    p = wl.config2()
    qd = qn.nf4_quantize(torch.from_numpy(p.W()).cuda())
    _, m32 = qn.nf4_merge_lora(qd, bf16_dev(p.A()), bf16_dev(p.B()), p.scale, bf16=False, f32=True)
    q2 = qn.nf4_quantize(m32)
    o2 = oracle.quantize(m32.cpu().numpy())
    assert np.array_equal(q2.codes.cpu().numpy(), o2["codes"])
    assert np.array_equal(q2.scale_codes.cpu().numpy(), o2["qscale"])
    base = f32_host(qn.nf4_dequantize(qd))
    merged = m32.cpu().numpy().astype(np.float64)
    requant = f32_host(qn.nf4_dequantize(q2))
    delta = np.linalg.norm(merged - base)
    loss = np.linalg.norm(requant - merged)
    assert delta > 0 and loss > 0.5 * delta


# ------------------------------------------------------------------ NF4 vs INT4 error
@pytest.mark.parametrize("kind,n", [("normal", 4096 * 4096), ("student_t", 1 << 20),
                                    ("normal", 1001), ("normal", 64 * 3 + 5)])
def test_int4_error_stats_match_oracle(kind, n):
    if kind == "normal":
        W = wl.weight((n,), seed=41, sigma=0.02)
    else:
        W = wl.student_t_weight((n,), seed=42, df=3.0, sigma=0.02)
    got = qn.nf4_int4_error_stats(torch.from_numpy(W).cuda()).cpu().numpy()
    want = oracle.int4_error(W)
    assert got[0] == pytest.approx(want[0], rel=1e-6)
    assert got[1] == pytest.approx(want[1], rel=1e-5)
    assert got[2] == pytest.approx(want[2], rel=1e-5)
    if kind == "normal" and n >= 4096:
        assert got[1] < 0.9 * got[2]


# ------------------------------------------------------------------ per-token adapters
def _multi_case(N, K, M, r, nad, seed):
    W = wl.weight((N, K), seed=seed, sigma=0.015)
    qo = oracle.quantize(W)
    Wd = oracle.dequantize(qo).reshape(N, K)
    qd = qn.nf4_quantize(torch.from_numpy(W).cuda())
    A = [wl.bf16_normal((r, K), seed=seed + 10 + i, sigma=0.01) for i in range(nad)]
    B = [wl.bf16_normal((N, r), seed=seed + 20 + i, sigma=0.01) for i in range(nad)]
    scales = np.array([0.25, 0.5, 2.0, 1.0][:nad], np.float32)
    X = wl.bf16_normal((M, K), seed=seed + 30)
    idx = np.array([(t % (nad + 1)) - 1 for t in range(M)], np.int32)  # -1: no adapter
    Y = qn.qlora_linear_fwd_multi(bf16_dev(X), qd, bf16_dev(np.stack(A)), bf16_dev(np.stack(B)),
                                  torch.from_numpy(idx).cuda(), torch.from_numpy(scales).cuda())
    ref = np.zeros((M, N))
    zeroB = np.zeros((N, r), np.uint16)
    for t in range(M):
        a = int(idx[t])
        if 0 <= a < nad:
            ref[t] = oracle.lora_fwd(X[t:t + 1], Wd, A[a], B[a], float(scales[a]))[0][0]
        else:
            ref[t] = oracle.lora_fwd(X[t:t + 1], Wd, A[0], zeroB, 1.0)[0][0]
    return f32_host(Y), ref


@pytest.mark.parametrize("M,r", [(1, 16), (5, 64), (16, 64), (16, 24), (9, 128)])
def test_multi_adapter_decode(M, r):
    got, ref = _multi_case(2048, 4096, M, r, 3, seed=51)
    assert rel_fro(got, ref) <= TOL
    for t in range(M):  # every token against its own adapter, not only the whole batch
        assert rel_fro(got[t], ref[t]) <= TOL


def test_multi_adapter_decode_full_size():
    got, ref = _multi_case(28672, 8192, 4, 64, 3, seed=52)
    assert rel_fro(got, ref) <= TOL


# ------------------------------------------------------------------ no double quantization
@pytest.mark.parametrize("n", [1, 63, 65, 1001, 64 * 256 + 1, 1 << 20])
def test_quantize_nodq_bit_exact(n):
    W = wl.weight((n,), seed=80 + n % 7, sigma=0.02)
    q = qn.nf4_quantize(torch.from_numpy(W).cuda(), double_quant=False)
    o = oracle.quantize(W)
    assert q.dq_block == 0 and q.scale_codes.numel() == 0 and q.scale_mean.numel() == 0
    assert np.array_equal(q.codes.cpu().numpy(), o["codes"])
    assert np.array_equal(q.scale_steps.cpu().numpy().view(np.uint32), o["absmax"].view(np.uint32))
    got = bits_host(qn.nf4_dequantize(q)).reshape(-1)
    assert np.array_equal(got, oracle.dequantize_nodq(o))


def test_dequantize_nodq_decode_tensor_bit_exact():
    W = wl.config4(1).W()
    o = oracle.quantize(W)
    q = qn.nf4_quantize(torch.from_numpy(W).cuda(), double_quant=False)
    assert np.array_equal(bits_host(qn.nf4_dequantize(q)).reshape(-1), oracle.dequantize_nodq(o))


@pytest.mark.parametrize("name,M,N,K,r,alpha", [s for s in SMALL if s[0] in
                                                ("cfg1", "ragged", "rank72", "tokens5",
                                                 "multi_tile", "rank12")])
def test_fwd_bwd_nodq(name, M, N, K, r, alpha):
    p = wl.LinearProblem(name, M, N, K, r, alpha, 0.02, 0.001, config=90 + len(name))
    pb = Problem(p, double_quant=False)
    Y, U = _check_fwd(pb)
    _check_bwd(pb, U)


def test_config2_nodq():
    pb = Problem(wl.config2(), double_quant=False)
    rows = _sample_rows(pb.p.M, 48, "config2-nodq")
    Y, U = _check_fwd(pb, rows)
    _check_bwd(pb, U, rows)


@pytest.mark.parametrize("M", [1, 16])
def test_config4_decode_nodq(M):
    pb = Problem(wl.config4(M), double_quant=False)
    _check_fwd(pb)


def test_merge_and_noalloc_nodq():
    p = wl.config1()
    W = p.W()
    o = oracle.quantize(W)
    q = qn.nf4_quantize(torch.from_numpy(W).cuda(), double_quant=False)
    m16, _ = qn.nf4_merge_lora(q, bf16_dev(p.A()), bf16_dev(p.B()), p.scale)
    want = oracle.merge(oracle.dequantize_nodq(o).reshape(p.N, p.K), p.A(), p.B(), p.scale)
    assert (_ulp_diff(bits_host(m16), want) > 0).mean() <= 1e-3
    q2 = qn.nf4_quantize_noalloc(torch.from_numpy(W).cuda(),
                                 qn.NF4Tensor.empty(p.N, p.K, "cuda", double_quant=False))
    assert torch.equal(q2.codes, q.codes) and torch.equal(q2.scale_steps, q.scale_steps)


@pytest.mark.parametrize("variant", ["nodq", "fp8"])
def test_merge_format_variants(variant):
    """The merge's scale decoding in both format variants (fp32 absmax per block, E4M3 second
    level), on the persistent form at rank 24 with a ragged row tile."""
    N, K, r = 200, 1024, 24
    W = wl.weight((N, K), seed=61, sigma=0.02, outlier_frac=0.001)
    A = wl.bf16_normal((r, K), seed=62, sigma=0.01)
    B = wl.bf16_normal((N, r), seed=63, sigma=0.01)
    scale = 2.0
    if variant == "nodq":
        o = oracle.quantize(W)
        q = qn.nf4_quantize(torch.from_numpy(W).cuda(), double_quant=False)
        wd = oracle.dequantize_nodq(o)
    else:
        o = oracle.quantize(W, fp8=True)
        q = qn.nf4_quantize(torch.from_numpy(W).cuda(), fp8_second_level=True)
        wd = oracle.dequantize(o)
    m16, m32 = qn.nf4_merge_lora(q, bf16_dev(A), bf16_dev(B), scale, f32=True)
    got = bits_host(m16)
    want = oracle.merge(wd.reshape(N, K), A, B, scale)
    assert (_ulp_diff(got, want) > 0).mean() <= 1e-3
    assert np.array_equal(m32.cpu().numpy(), wl.bf16_bits_to_f32(got))


# ------------------------------------------------------------------ fp8 second level
@pytest.mark.parametrize("n", [1, 65, 1001, 64 * 256 + 1, 64 * 300 + 37, 1 << 20])
def test_quantize_fp8_second_level_bit_exact(n):
    W = wl.weight((n,), seed=85 + n % 5, sigma=0.02)
    q = qn.nf4_quantize(torch.from_numpy(W).cuda(), fp8_second_level=True)
    o = oracle.quantize(W, fp8=True)
    assert q.dq_type == 1
    assert np.array_equal(q.codes.cpu().numpy(), o["codes"])
    assert np.array_equal(q.scale_codes.cpu().numpy(), o["qscale"])
    assert np.array_equal(q.scale_steps.cpu().numpy().view(np.uint32), o["steps"].view(np.uint32))
    assert q.scale_mean.cpu().numpy()[0].view(np.uint32) == np.float32(o["mean"]).view(np.uint32)
    assert np.array_equal(bits_host(qn.nf4_dequantize(q)).reshape(-1), oracle.dequantize(o))


def test_quantize_fp8_second_level_decode_tensor_bit_exact():
    W = wl.config4(1).W()
    q = qn.nf4_quantize(torch.from_numpy(W).cuda(), fp8_second_level=True)
    o = oracle.quantize(W, fp8=True)
    assert np.array_equal(q.scale_codes.cpu().numpy(), o["qscale"])
    assert np.array_equal(bits_host(qn.nf4_dequantize(q)).reshape(-1), oracle.dequantize(o))


@pytest.mark.parametrize("name,M,N,K,r,alpha", [s for s in SMALL if s[0] in
                                                ("cfg1", "ragged", "tokens5", "multi_tile")])
def test_fwd_bwd_fp8_second_level(name, M, N, K, r, alpha):
    p = wl.LinearProblem(name, M, N, K, r, alpha, 0.02, 0.001, config=90 + len(name))
    pb = Problem(p, fp8_second_level=True)
    Y, U = _check_fwd(pb)
    _check_bwd(pb, U)


def test_config2_fp8_second_level():
    pb = Problem(wl.config2(), fp8_second_level=True)
    rows = _sample_rows(pb.p.M, 48, "config2-fp8")
    Y, U = _check_fwd(pb, rows)
    _check_bwd(pb, U, rows)


@pytest.mark.parametrize("M", [1, 16])
def test_config4_decode_fp8_second_level(M):
    pb = Problem(wl.config4(M), fp8_second_level=True)
    _check_fwd(pb)


# ------------------------------------------------------------------ fp16 compute type
# digipro.cn "QLoRA: Fine-Tuning a 7B Model on a 16GB GPU", "The QLoRA insight": the
# compute-dtype flag dequantizes to fp16 for the matrix multiplies.
@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 17), (3, 333), (256, 256), (4096, 4096)])
def test_dequantize_f16_bit_exact(rows, cols):
    W = wl.weight((rows, cols), seed=rows * 5 + cols, sigma=0.02, outlier_frac=0.001)
    W.reshape(-1)[:128] *= 2.0 ** -14   # two blocks whose weights are binary16 subnormals
    o = oracle.quantize(W)
    got = bits_host(qn.nf4_dequantize_f16(upload_oracle_tensor(o, rows, cols))).reshape(-1)
    assert np.array_equal(got, oracle.dequantize(o, f16=True))
    for dq, fp8 in ((False, False), (True, True)):
        q = qn.nf4_quantize(torch.from_numpy(W).cuda(), double_quant=dq, fp8_second_level=fp8)
        o = oracle.quantize(W, fp8=fp8)
        want = oracle.dequantize(o, f16=True) if dq else oracle.dequantize_nodq(o, f16=True)
        out = qn.nf4_dequantize_f16(q)
        assert out.dtype == torch.float16
        assert np.array_equal(bits_host(out).reshape(-1), want)


def test_dequantize_f16_decode_tensor_bit_exact():
    W = wl.config4(1).W()
    q = qn.nf4_quantize(torch.from_numpy(W).cuda())
    got = bits_host(qn.nf4_dequantize_f16(q)).reshape(-1)
    assert np.array_equal(got, oracle.dequantize(oracle.quantize(W), f16=True))


@pytest.mark.parametrize("name,M,N,K,r,alpha", [s for s in SMALL if s[0] in
                                                ("cfg1", "ragged", "rank72", "rank128",
                                                 "tokens17", "tokens1", "tokens5",
                                                 "multi_tile", "rank12", "tokens9_rank13")])
def test_fwd_bwd_f16(name, M, N, K, r, alpha):
    p = wl.LinearProblem(name, M, N, K, r, alpha, 0.02, 0.001, config=90 + len(name))
    pb = Problem(p, half=True)
    Y, U = _check_fwd(pb)
    _check_bwd(pb, U)
    _check_bwd(pb, None)


@pytest.mark.parametrize("variant", ["nodq", "fp8"])
def test_fwd_bwd_f16_format_variants(variant):
    p = wl.LinearProblem(f"f16-{variant}", 200, 320, 448, 16, 32.0, 0.02, 0.001, config=93)
    pb = Problem(p, double_quant=variant != "nodq", fp8_second_level=variant == "fp8",
                 half=True)
    Y, U = _check_fwd(pb)
    _check_bwd(pb, U)
    p1 = wl.LinearProblem(f"f16-{variant}-decode", 4, 576, 320, 8, 16.0, 0.02, 0.001, config=94)
    _check_fwd(Problem(p1, double_quant=variant != "nodq", fp8_second_level=variant == "fp8",
                       half=True))


def test_config2_f16():
    pb = Problem(wl.config2(), half=True)
    rows = _sample_rows(pb.p.M, 48, "config2-f16")
    Y, U = _check_fwd(pb, rows)
    _check_bwd(pb, U, rows)


@pytest.mark.parametrize("M", [1, 16])
def test_config4_decode_f16(M):
    pb = Problem(wl.config4(M), half=True)
    _check_fwd(pb)


def test_f16_and_bf16_entry_points_refuse_each_others_dtype():
    pb = Problem(wl.config1(), half=True)
    with pytest.raises(ValueError):
        qn.qlora_linear_fwd(pb.Xd, pb.qd, pb.Ad, pb.Bd, pb.p.scale)
    pbb = Problem(wl.config1())
    with pytest.raises(ValueError):
        qn.qlora_linear_fwd_f16(pbb.Xd, pbb.qd, pbb.Ad, pbb.Bd, pbb.p.scale)
