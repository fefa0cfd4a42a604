"""Pins for the oracle's E4M3 and bf16 codecs (CPU only).

The E4M3 decoder is pinned to the log-affine byte relation the pages print
(paper.rainbus.top summary, 前置知识 "E4M3 浮点格式": the byte read as an
integer equals 8 log2 v + 56 + eps(m)); the encoder is pinned by brute force
(nearest finite code, ties to the even code, saturation at 448); bf16
rounding is pinned to torch's CPU conversion.
"""
import json
import math
import os

import numpy as np
import torch

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")))


def test_decode_log_affine_relation(oracle_mod):
    slope = GOLD["byte_slope"]["value"]
    offset = GOLD["byte_offset"]["value"]
    codes = np.arange(0x08, 0x7F, dtype=np.uint8)        # the 119 positive normal codes
    assert codes.size == 119
    v = oracle_mod.e4m3_decode(codes)
    m = (codes & 7) / 8.0
    eps = slope * (m - np.log2(1.0 + m))
    assert np.all(eps <= 1e-15) and eps.min() > -0.69
    np.testing.assert_allclose(codes.astype(np.float64), slope * np.log2(v) + offset + eps,
                               rtol=0, atol=1e-12)


def test_decode_remaining_codes(oracle_mod):
    dec = oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert dec[0] == 0.0
    # 7 positive subnormals are multiples of 2^-9
    np.testing.assert_array_equal(dec[1:8], np.arange(1, 8) * 2.0 ** -9)
    assert math.isnan(dec[0x7F]) and math.isnan(dec[0xFF])
    # negative codes mirror the positive ones
    pos = dec[:0x7F]
    np.testing.assert_array_equal(dec[0x80:0xFF], -pos)
    assert dec[0x38] == 1.0 and dec[0x7E] == 448.0 and dec[0x08] == 2.0 ** -6
    # the ExpCast top byte: 120 = 2^8, the probability of the row maximum
    assert dec[GOLD["clip_hi"]["value"]] == 256.0
    finite = dec[~np.isnan(dec)]
    assert np.all(np.diff(dec[:0x7F]) > 0)      # strictly increasing on the positive side
    assert finite.size == 254


def _brute_encode(x):
    """Nearest finite E4M3 value, ties to the even code, |x| >= 448 saturates."""
    codes = np.arange(0, 0x7F, dtype=np.int64)
    vals = np.array([_dec_py(c) for c in codes])
    a = np.abs(x.astype(np.float64))
    out = np.empty(x.size, np.uint8)
    dist = np.abs(a[:, None] - vals[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # prefer the even code among ties
    even = cand & ((codes[None, :] & 1) == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    out[:] = codes[pick]
    out[a >= 448.0] = 0x7E
    out |= np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    return out


def _dec_py(c):
    e, m = (c >> 3) & 15, c & 7
    if e == 0:
        return m * 2.0 ** -9
    return (1 + m / 8.0) * 2.0 ** (e - 7)


def test_encode_bruteforce(oracle_mod):
    rng = np.random.default_rng(7)
    logu = rng.uniform(-13, 9.5, 60000)
    x = (np.exp2(logu) * rng.choice([-1, 1], logu.size)).astype(np.float32)
    # exact midpoints between neighbouring codes (ties) and the codes themselves
    vals = np.array([_dec_py(c) for c in range(0, 0x7F)])
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    extra = np.concatenate([vals.astype(np.float32), mids, -mids,
                            np.array([0.0, -0.0, 447.9, 448.0, 449.0, 464.0, 1e30, 2.0 ** -10,
                                      2.0 ** -10 * 1.0001, 3 * 2.0 ** -11], np.float32)])
    x = np.concatenate([x, extra])
    got = oracle_mod.e4m3_encode(x)
    want = _brute_encode(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_encode_decode_roundtrip(oracle_mod):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle_mod.e4m3_decode(codes).astype(np.float32)
    np.testing.assert_array_equal(oracle_mod.e4m3_encode(vals), codes)


def test_bf16_rne_matches_torch(oracle_mod):
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    # keep finite values, add exact ties (low half = 0x8000)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ties = ((rng.integers(0, 2 ** 16, 5000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    x = np.concatenate([x, ties, np.array([0.0, -0.0, 1.0, 65504.0], np.float32)])
    got = oracle_mod.bf16_rne(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(oracle_mod.bf16_to_f32(got),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())
