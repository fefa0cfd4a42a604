"""Pins of the oracle's hybrid probability bytes (expcast = 2).

The pages' own analysis (paper summary, 独立分析的弱点, weakness two) suggests
keeping the exact exponent on high-weight tiles.  The reading: per group of 32
query rows and key tile, exp-then-cast if some row of the group has its tile
maximum within `margin` (log2) of its running maximum, else the ExpCast byte.
The pins check the composition rule against the two pinned modes:

* margin -> -inf gives ExpCast everywhere, margin -> +inf exp-then-cast
  everywhere (bit for bit, O and bytes);
* the first key tile is always high-weight (its maximum is the running max);
* a planted score pattern selects exactly the tiles and groups the rule
  names, one high row turning its whole group (and only it) exact;
* requesting part of a group is refused.
"""
import numpy as np
import pytest

from bit_fp8_attention_means_gb300 import inputs

N, D = 512, 64


@pytest.fixture(scope="module")
def qz(oracle_mod):
    w = inputs.WORKLOADS["tiny"]
    Q, K, V = inputs.make_qkv(w, "cpu", H=1, N=N, d=D, seed=31)
    return oracle_mod.quantize(*(inputs.to_u16(t) for t in (Q, K, V)), None, 1)


def _codes(oracle_mod, qz, expcast, margin=0.0, rows=None, acc=None):
    return oracle_mod.attn(qz, N, expcast=expcast, margin=margin, rows=rows, acc_in=acc, want_codes=True)


def test_margin_limits_reduce_to_the_two_modes(oracle_mod, qz):
    O1, P1 = _codes(oracle_mod, qz, 1)
    O0, P0 = _codes(oracle_mod, qz, 0)
    Oh, Ph = _codes(oracle_mod, qz, 2, margin=-1e30)
    np.testing.assert_array_equal(Ph, P1)
    np.testing.assert_array_equal(Oh, O1)
    Oh, Ph = _codes(oracle_mod, qz, 2, margin=1e30)
    np.testing.assert_array_equal(Ph, P0)
    np.testing.assert_array_equal(Oh, O0)


def test_first_tile_always_exact(oracle_mod, qz):
    _, P0 = _codes(oracle_mod, qz, 0)
    _, Ph = _codes(oracle_mod, qz, 2, margin=0.0)
    np.testing.assert_array_equal(Ph[..., :128], P0[..., :128])


def _planted_acc(sq, sk, kscale):
    """Scores (in units of each tile's sigma) that put every row's tile-1
    maximum 3 (log2 units) below its tile-0 maximum, except row 37 (group 1),
    whose tile-1 maximum is 0.5 below; tiles 2 and 3 stay 9 below."""
    acc = np.zeros((1, 1, N, 4 * 128), np.float32)
    rng = np.random.default_rng(2)
    for i in range(N):
        sig = [np.float32(np.float32(sq[i // 128] * sk[j]) * kscale) for j in range(4)]
        u = rng.uniform(-20, -9, 4 * 128).astype(np.float32)   # log2-domain values
        u[5] = 0.0                                              # tile 0 max
        gap = 0.5 if i == 37 else 3.0
        u[130] = -gap                                           # tile 1 max
        for j in range(4):
            acc[0, 0, i, 128 * j:128 * (j + 1)] = u[128 * j:128 * (j + 1)] / sig[j]
    return acc


def test_planted_tiles_and_groups(oracle_mod, qz):
    kscale = oracle_mod.kscale_of(0.0, D)
    rows = np.arange(N, dtype=np.int32)
    acc = _planted_acc(qz["sq"][0, 0], qz["sk"][0, 0], kscale)
    _, P0 = _codes(oracle_mod, qz, 0, rows=rows, acc=acc)
    _, P1 = _codes(oracle_mod, qz, 1, rows=rows, acc=acc)
    _, Ph = _codes(oracle_mod, qz, 2, margin=2.0, rows=rows, acc=acc)
    t1 = slice(128, 256)
    group1 = slice(32, 64)
    # tile 1: exact for group 1 (row 37 is within the margin), ExpCast for every other group
    np.testing.assert_array_equal(Ph[0, 0, group1, t1], P0[0, 0, group1, t1])
    others = np.r_[0:32, 64:N]
    np.testing.assert_array_equal(Ph[0, 0, others, t1], P1[0, 0, others, t1])
    # tiles 2, 3: 9 below the running max everywhere -> ExpCast
    np.testing.assert_array_equal(Ph[0, 0, :, 256:], P1[0, 0, :, 256:])
    # the planted gap is what separates the modes there
    assert np.any(P0[0, 0, others, t1] != P1[0, 0, others, t1])
    # a wider margin turns tile 1 exact for all groups
    _, Pw = _codes(oracle_mod, qz, 2, margin=4.0, rows=rows, acc=acc)
    np.testing.assert_array_equal(Pw[0, 0, :, t1], P0[0, 0, :, t1])


def test_partial_group_is_refused(oracle_mod, qz):
    with pytest.raises(AssertionError):
        _codes(oracle_mod, qz, 2, margin=1.0, rows=np.arange(0, 40, dtype=np.int32))
