"""Philox4x32-10, written from the SC'11 paper (test infrastructure only).

Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
(SC'11), section 3.2 "Philox".  One Philox-4x32 round takes the counter
words (x0, x1, x2, x3) and the two key words (k0, k1), forms the two
32x32->64-bit products M0*x0 and M1*x2, and returns

    (hi(M1*x2) ^ x1 ^ k0,  lo(M1*x2),  hi(M0*x0) ^ x3 ^ k1,  lo(M0*x0))

The key is bumped by the Weyl constants (W0, W1) between rounds; ten
rounds make Philox4x32-10.  The multipliers and Weyl constants are the
ones the paper publishes for Philox-4x32.

How the verify step draws (a reading; the pages define no generator):

    key     = (seed mod 2^32, seed div 2^32)
    counter = (request b, position j (1-based), draw, 0)
    draw 0  = the accept test at position j: u = uniform of word 0
    draw 1  = the correction at the first rejected position j*, or the
              bonus at position j = N + 1: four uniforms, one per word,
              one for each level of the grouped inverse CDF
    uniform of a word w = (w >> 8) * 2^-24     in [0, 1 - 2^-24]

A uniform has 24 significant bits, so it is exact in both float32 and
float64 and both sides of a comparison see the same number.

Everything here is vectorised over numpy uint64 arrays so that it also
works on scalars.
"""

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF


def _u64(x):
    return np.asarray(x, dtype=np.uint64)


def philox4x32_10(c0, c1, c2, c3, k0, k1, rounds=10):
    """Return the four output words of Philox4x32-``rounds``.

    Arguments are 32-bit counter words c0..c3 and key words k0, k1 (ints or
    numpy arrays, broadcast together).  Output: tuple of four uint64 arrays
    holding 32-bit values.
    """
    m = np.uint64(MASK32)
    x0, x1, x2, x3 = (_u64(c) & m for c in (c0, c1, c2, c3))
    key0, key1 = _u64(k0) & m, _u64(k1) & m
    x0, x1, x2, x3, key0, key1 = np.broadcast_arrays(x0, x1, x2, x3, key0, key1)
    x0, x1, x2, x3 = (a.copy() for a in (x0, x1, x2, x3))
    key0, key1 = key0.copy(), key1.copy()
    for r in range(rounds):
        if r > 0:
            key0 = (key0 + np.uint64(W0)) & m
            key1 = (key1 + np.uint64(W1)) & m
        p0 = np.uint64(M0) * x0  # < 2^64: exact in uint64
        p1 = np.uint64(M1) * x2
        hi0, lo0 = p0 >> np.uint64(32), p0 & m
        hi1, lo1 = p1 >> np.uint64(32), p1 & m
        x0, x1, x2, x3 = hi1 ^ x1 ^ key0, lo1, hi0 ^ x3 ^ key1, lo0
    return x0, x1, x2, x3


def split_seed(seed):
    """Key words (k0, k1) = (low 32 bits, high 32 bits) of a 64-bit seed."""
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & MASK32, seed >> 32


def uniform(seed, b, j, draw):
    """The uniform in [0, 1) used for (request b, position j, draw).

    Returns a Python float (vectorised callers get a float64 array) equal to
    (word0 >> 8) * 2^-24.
    """
    k0, k1 = split_seed(seed)
    w0, _, _, _ = philox4x32_10(b, j, draw, 0, k0, k1)
    u = (w0 >> np.uint64(8)).astype(np.float64) * 2.0 ** -24
    if np.ndim(u) == 0:
        return float(u)
    return u


def uniforms4(seed, b, j, draw):
    """The four uniforms of (request b, position j, draw), one per output
    word, as a tuple of Python floats."""
    k0, k1 = split_seed(seed)
    words = philox4x32_10(b, j, draw, 0, k0, k1)
    return tuple(float(int(w) >> 8) * 2.0 ** -24 for w in words)


ACCEPT_DRAW = 0
SAMPLE_DRAW = 1
