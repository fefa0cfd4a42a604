"""Derive the per-piece beta of the range-adaptive ExpCast byte (oracle reading).

The paper summary's own analysis (paper.rainbus.top, 独立分析的弱点, weakness
two) suggests choosing beta by score range instead of one constant.  This
library's reading, for both the oracle and the kernel (expcast = 3):

    t0 = fmaf(acc, 8 sigma, fmaf(-8, m', 120))        (ExpCast's t without beta)
    p  = (rint(t0) >> 1) & 3                            (which pair of codes of its octave)
    c  = clip(rint(fl(t0 + beta_p)), 0, 120)

Each beta_p is chosen here to maximise agreement with the exp-then-cast byte
E4M3_RNE(2^((t0 - 120)/8 + 8)) for t0 uniform over one normal octave, the
criterion the single beta = -0.35 of the pages is measured by (79.6 %
agreement).  Only the oracle's E4M3 encoder is used.  Run from the repository
root: python -m oracle.derive_beta_pieces
"""
import numpy as np

import oracle


def exact_codes(t0):
    """Exp-then-cast byte for the log-domain position t0 (float64 -> fp32 value -> E4M3)."""
    v = np.exp2((t0 - 120.0) / 8.0 + 8.0).astype(np.float32)
    return oracle.e4m3_encode(v).astype(np.int64)


def pieces(t0):
    return (np.rint(t0).astype(np.int64) >> 1) & 3


def derive(n=400000, lo=64.0):
    t0 = (lo + 8.0 * (np.arange(n) + 0.5) / n).astype(np.float32)   # one normal octave of codes [64, 72)
    ex = exact_codes(t0.astype(np.float64))
    p = pieces(t0.astype(np.float64))
    cands = np.round(np.arange(-1.0, 0.5 + 1e-9, 0.005), 3).astype(np.float32)
    betas = []
    for q in range(4):
        sel = p == q
        agree = [np.mean(np.rint((t0[sel] + b).astype(np.float32)).astype(np.int64) == ex[sel]) for b in cands]
        betas.append(float(cands[int(np.argmax(agree))]))
    b = np.array(betas, np.float32)[p]
    c = np.rint((t0 + b).astype(np.float32)).astype(np.int64)
    return betas, float(np.mean(c == ex)), int(np.max(np.abs(c - ex)))


if __name__ == "__main__":
    betas, agree, maxdiff = derive()
    print("beta per piece:", betas)
    print("agreement with exp-then-cast over one octave: %.4f, max |code difference| %d" % (agree, maxdiff))
