"""Pins for the oracle's quantizer (CPU only).

Block scales ([R] 前置知识: one scale per hardware block) and the V-Smooth
residual ([R] 方法步骤详情 step 2; dimensionstp.github.io 2-2: mu_j =
(1/B_v) V'_j^T 1, R_j = V'_j - 1 mu_j^T, per-channel E4M3 residual).  The pins
are format error bounds, gather identities and special cases, not a retyping
of the quantizer.
"""
import json
import os

import numpy as np
import pytest

from bit_fp8_attention_means_gb300 import inputs

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")))
BLK = GOLD["block_tokens"]["value"]


def _e4m3_err_bound(y):
    """Half the E4M3 spacing at |y| (|y| <= 448): 2^(floor(log2|y|)-4), >= 2^-10."""
    a = np.abs(y)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return np.exp2(e - 4)


def _data(N=1000, d=64, H=2, seed=3):
    Q, K, V = inputs.make_qkv(inputs.WORKLOADS["tiny"], "cpu", H=H, N=N, d=d, seed=seed)
    return inputs.to_u16(Q), inputs.to_u16(K), inputs.to_u16(V)


def test_block_scale_and_error_bound(oracle_mod):
    N, d = 1000, 64
    Q, K, V = _data(N, d)
    qz = oracle_mod.quantize(Q, K, V, None, 1)
    x = oracle_mod.bf16_to_f32(Q).astype(np.float64).transpose(0, 2, 1, 3)   # [B,H,N,d]
    nb = (N + BLK - 1) // BLK
    dec = oracle_mod.e4m3_decode(qz["Q8"])
    for j in range(nb):
        blk = x[:, :, j * BLK:(j + 1) * BLK]
        amax = np.abs(blk).max(axis=(2, 3))
        np.testing.assert_allclose(qz["sq"][:, :, j], amax / 448.0, rtol=2 ** -23)
        codes = qz["Q8"][:, :, j * BLK:(j + 1) * BLK]
        # the element at the block maximum lands on the largest code
        assert np.all((codes & 0x7F).reshape(codes.shape[0], codes.shape[1], -1).max(axis=2) == 0x7E)
        s = qz["sq"][:, :, j][:, :, None, None]
        y = blk / s
        err = np.abs(dec[:, :, j * BLK:j * BLK + blk.shape[2]] - y)
        assert np.all(err <= _e4m3_err_bound(y) * (1 + 1e-6) + 1e-6)
    # padding rows are code 0
    assert np.all(qz["Q8"][:, :, N:] == 0) and np.all(qz["K8"][:, :, N:] == 0)
    assert np.all(qz["V8T"][..., N:] == 0)


@pytest.mark.parametrize("vsmooth", [0, 1])
def test_permutation_is_a_gather(oracle_mod, vsmooth):
    N = 777
    Q, K, V = _data(N, 64, seed=8)
    rng = np.random.default_rng(1)
    B, _, H, _ = Q.shape
    perm = np.stack([np.stack([rng.permutation(N) for _ in range(H)]) for _ in range(B)]).astype(np.int32)
    a = oracle_mod.quantize(Q, K, V, perm, vsmooth)
    Kp = np.empty_like(K)
    Vp = np.empty_like(V)
    for b in range(B):
        for h in range(H):
            Kp[b, :, h] = K[b, perm[b, h], h]
            Vp[b, :, h] = V[b, perm[b, h], h]
    c = oracle_mod.quantize(Q, Kp, Vp, None, vsmooth)
    for key in a:
        np.testing.assert_array_equal(a[key], c[key], err_msg=key)


def test_block_mean_and_residual(oracle_mod):
    N, d = 1000, 64
    Q, K, V = _data(N, d, seed=12)
    qz = oracle_mod.quantize(Q, K, V, None, 1)
    v = oracle_mod.bf16_to_f32(V).astype(np.float64).transpose(0, 2, 1, 3)   # [B,H,N,d]
    mu = oracle_mod.bf16_to_f32(qz["mu"]).astype(np.float64)
    nb = mu.shape[2]
    for j in range(nb):
        blk = v[:, :, j * BLK:(j + 1) * BLK]
        mean = blk.mean(axis=2)
        # bf16 rounding (2^-8 relative) plus the fp32 running-sum error
        tol = np.abs(mean) * 2.0 ** -8 + np.abs(blk).sum(axis=2) / blk.shape[2] * blk.shape[2] * 2.0 ** -23
        assert np.all(np.abs(mu[:, :, j] - mean) <= tol + 1e-30)
    # dequantized V' = s_v * R_q + mu, within the E4M3 bound on the residual
    sv = qz["sv"][:, :, None, :]
    rq = oracle_mod.e4m3_decode(qz["V8T"]).transpose(0, 1, 3, 2)[:, :, :N] * sv
    r = v - np.repeat(mu, BLK, axis=2)[:, :, :N]
    bound = _e4m3_err_bound(r / sv) * sv
    assert np.all(np.abs(rq - r) <= bound * (1 + 1e-5) + 1e-7)
    # each channel's largest residual reaches code 448
    assert np.all((qz["V8T"] & 0x7F).max(axis=3) == 0x7E)


def test_mean_costs_an_eighth_bit_per_element(oracle_mod):
    N, d = 1024, 64
    Q, K, V = _data(N, d)
    qz = oracle_mod.quantize(Q, K, V, None, 1)
    bits = qz["mu"].size * 16 / (qz["V8T"].shape[0] * qz["V8T"].shape[1] * N * d)
    assert bits == GOLD["mean_bits_per_element"]["value"]


def test_vsmooth_off_quantizes_v_directly(oracle_mod):
    N, d = 500, 64
    Q, K, V = _data(N, d, seed=2)
    qz = oracle_mod.quantize(Q, K, V, None, 0)
    assert np.all(qz["mu"] == 0)
    v = oracle_mod.bf16_to_f32(V).astype(np.float64).transpose(0, 2, 1, 3)
    np.testing.assert_allclose(qz["sv"], np.abs(v).max(axis=2) / 448.0, rtol=2 ** -23)


def test_single_cluster_is_sequence_order(oracle_mod):
    """k = 1: every label is 0, pi is the identity, mu is the plain block mean."""
    N, d = 400, 64
    Q, K, V = _data(N, d, seed=6)
    cent, lab = oracle_mod.kmeans(V, 1, 2)
    assert np.all(lab == 0)
    perm = oracle_mod.argsort_labels(lab, 1)
    assert np.all(perm == np.arange(N))
    a = oracle_mod.quantize(Q, K, V, perm, 1)
    b = oracle_mod.quantize(Q, K, V, None, 1)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])
    v = oracle_mod.bf16_to_f32(V).astype(np.float64).transpose(0, 2, 1, 3)
    np.testing.assert_allclose(cent[:, :, 0], v.mean(axis=2), rtol=1e-6, atol=1e-7)


def test_zero_block(oracle_mod):
    N, d = 256, 64
    Q, K, V = _data(N, d)
    Q[:, :128] = 0
    qz = oracle_mod.quantize(Q, K, V, None, 1)
    assert np.all(qz["sq"][:, :, 0] == 0) and np.all(qz["Q8"][:, :, :128] == 0)
