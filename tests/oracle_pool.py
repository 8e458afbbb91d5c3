"""Oracle work for the GPU tests that runs in spawned worker processes (no GPU state)."""
import numpy as np

import oracle
from bit_nf4_quantized_37_b300 import workloads as wl


def quantize_stack_layer(layer: int):
    """Oracle quantization of every projection of one layer of the 32-layer 7B stack:
    [(name, codes, scale codes, steps, mean)]."""
    out = []
    for p in wl.config5(layer=layer):
        o = oracle.quantize(p.W())
        out.append((p.name, o["codes"], o["qscale"], o["steps"], np.float32(o["mean"])))
    return out
