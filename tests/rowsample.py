"""Query rows that the sampled O checks compare with the oracle.

Besides random rows, every sample holds rows of the first query tile, of the
last tile (the only one with rows beyond N and, on the key side, the masked
keys), and of the tile before it (at an odd tile count the last CTA of a
kernel that takes two query tiles per CTA holds the last tile alone, at an
even count the last two), each at both ends of the tile.
"""
import numpy as np

BLOCK = 128


def sampled_rows(N, rng, n_random):
    nb = (N + BLOCK - 1) // BLOCK
    parts = [rng.choice(N, min(n_random, N), replace=False), np.arange(0, min(4, N)),
             np.arange(max(0, N - 6), N)]
    for t in (nb - 2, nb - 1):
        if t >= 0:
            lo, hi = t * BLOCK, min(N, (t + 1) * BLOCK)
            parts += [np.arange(lo, min(lo + 3, hi)), np.arange(max(lo, hi - 3), hi),
                      np.array([lo + (hi - lo) // 2])]
    return np.unique(np.concatenate(parts)).astype(np.int32)
