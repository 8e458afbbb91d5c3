"""A weight tensor whose second-level (int8) scale quotients land exactly on half-integers.

One group of 256 blocks.  Block b holds a single nonzero weight, its absmax a_b = 1 + d_b,
with the offsets d_b in mirrored pairs (+d, -d) so the mean of the absmax values is exactly 1.
The largest offset is 127/128, so the group's step is (127/128) / 127 = 2^-7 exactly, and
every quotient (a_b - 1) / 2^-7 = 128 d_b is computed without rounding.  Offsets of
(k + 1/2)/128 put the quotient on a tie for even and odd k alike: rounding half to even and
rounding half away from zero give different codes for every even k.
"""
import numpy as np

# k + 1/2 for even and odd k, the step's own block (127) and a few exact integers
TIE_HALVES = [0.5, 1.5, 2.5, 3.5, 10.5, 11.5, 62.5, 63.5, 125.5, 126.5]
EXACT = [0.0, 1.0, 64.0, 127.0]


def tie_offsets() -> np.ndarray:
    """128 d_b values (in units of 1/128) for the first half of the group; the second half
    holds their negatives."""
    base = TIE_HALVES + EXACT
    reps = [base[i % len(base)] for i in range(128)]
    return np.array(reps, np.float64)


def tie_tensor() -> tuple[np.ndarray, np.ndarray]:
    """(W fp32 [256, 64], expected int8 codes [256]) with codes from rounding half to even."""
    u = tie_offsets()
    units = np.concatenate([u, -u])               # 128 d_b in units of 1/128
    a = (1.0 + units / 128.0).astype(np.float32)  # exact: at most 15 significant bits
    assert np.all(a.astype(np.float64) == 1.0 + units / 128.0)
    W = np.zeros((256, 64), np.float32)
    W[:, 7] = a
    W[1::2, 7] *= -1.0                            # the sign of the absmax element is free
    expect = np.rint(units).astype(np.int64)      # numpy's rint: half to even
    return W, np.clip(expect, -127, 127).astype(np.int8)
