"""Helpers for the GPU parity tests: moving seeded inputs to the device and comparing the
CUDA path against the CPU oracle."""
import numpy as np
import torch

import oracle
import bit_nf4_quantized_37_b300 as qn
from bit_nf4_quantized_37_b300 import workloads as wl

TOL = 5e-3  # relative Frobenius bound for Y, dX, dA, dB against the fp64 oracle


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def f16_dev(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16).cuda()


def f16_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """binary16 bits of bf16-valued inputs (numpy's round to nearest even; exact for the
    normal range, which the seeded inputs stay in apart from their smallest values)."""
    return wl.bf16_bits_to_f32(bits).astype(np.float16).view(np.uint16)


def bits_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32_host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return wl.bf16_bits_to_f32(bits_host(t)).astype(np.float64)
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    d = np.linalg.norm((got - ref).ravel())
    n = np.linalg.norm(ref.ravel())
    return float(d / n) if n > 0 else float(d)


def upload_oracle_tensor(q: dict, rows: int, cols: int) -> qn.NF4Tensor:
    dev = "cuda"
    return qn.NF4Tensor(torch.from_numpy(q["codes"]).to(dev),
                        torch.from_numpy(q["qscale"]).to(dev),
                        torch.from_numpy(q["steps"]).to(dev),
                        torch.tensor([q["mean"]], dtype=torch.float32, device=dev), rows, cols)


class Problem:
    """A LinearProblem with its oracle quantization and device copies."""

    def __init__(self, p: wl.LinearProblem, quantize_on_gpu: bool = True,
                 double_quant: bool = True, fp8_second_level: bool = False, half: bool = False):
        self.p = p
        self.half = half
        W = p.W()
        self.qo = oracle.quantize(W, fp8=fp8_second_level)
        if double_quant:
            self.Wd = oracle.dequantize(self.qo, f16=half).reshape(p.N, p.K)
        else:
            self.Wd = oracle.dequantize_nodq(self.qo, f16=half).reshape(p.N, p.K)
        if quantize_on_gpu or not double_quant or fp8_second_level:
            self.qd = qn.nf4_quantize(torch.from_numpy(W).cuda(), double_quant=double_quant,
                                      fp8_second_level=fp8_second_level)
        else:
            self.qd = upload_oracle_tensor(self.qo, p.N, p.K)
        self.X, self.A, self.B, self.dY = p.X(), p.A(), p.B(), p.dY()
        dev = bf16_dev
        if half:
            self.X, self.A, self.B, self.dY = (f16_from_bf16_bits(t)
                                               for t in (self.X, self.A, self.B, self.dY))
            dev = f16_dev
        self.Xd, self.Ad, self.Bd, self.dYd = (dev(self.X), dev(self.A), dev(self.B),
                                               dev(self.dY))
