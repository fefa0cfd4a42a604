"""Pins for the oracle's attention (CPU only).

* P'V' = PV (dimensionstp.github.io, 2-1): the fp64 fidelity reference is
  invariant under a joint permutation of K and V.
* Closed forms: equal scores give the plain mean of the dequantized values;
  two dominant keys in different tiles give (alpha v1 + v2)/(alpha + 1) with
  alpha = 2^(s1 - s2), which pins the rescale, the running max and the
  per-tile mean restore ([R] step 3; dimensionstp.github.io, 2-3).
* Error bound: with the row maximum in the first tile, |O - O_exact| <=
  2 TV(p_hat, p) max|v| and TV <= 3.64% + underflow tail (the pages' bound).
"""
import math

import numpy as np
import pytest
import torch

from bit_fp8_attention_means_gb300 import inputs

LN2 = np.float32(math.log(2.0))   # softmax_scale whose kscale = fp32(ln2 * log2 e) = 1


def _dequant_v(oracle_mod, qz, vsmooth):
    """V'_q[b,h,t,c] = s_v[c] * dec(v8[c,t]) + mu_j[c] (fp64)."""
    V8T, sv, mu = qz["V8T"], qz["sv"], qz["mu"]
    B, H, d, Npad = V8T.shape
    v = oracle_mod.e4m3_decode(V8T).transpose(0, 1, 3, 2) * sv[:, :, None, :]
    if vsmooth:
        m = oracle_mod.bf16_to_f32(mu).astype(np.float64)       # [B,H,nblk,d]
        v = v + np.repeat(m, 128, axis=2)
    return v


def _small(N=300, d=64, H=2, seed=5):
    w = inputs.WORKLOADS["tiny"]
    Q, K, V = inputs.make_qkv(w, "cpu", H=H, N=N, d=d, seed=seed)
    return inputs.to_u16(Q), inputs.to_u16(K), inputs.to_u16(V)


def test_mean_restore_identity(oracle_mod):
    """P (R + 1 mu_j) = P R + r_ij mu_j ([R] step 3; dimensionstp.github.io, 2-3).

    With every row's maximum planted in the first tile no rescale ever happens,
    so the oracle's output (which adds r_ij mu_j per tile) must equal the fp64
    weighted mean of the dequantized V' = s_v R_q + mu_j under its own bytes.
    A dropped mean term, a wrong block index or a wrong channel scale fails.
    """
    N, d = 700, 64
    Q, K, V = _small(N=N, d=d, seed=21)
    qz = oracle_mod.quantize(Q, K, V, None, 1)
    B, H, Npad, _ = qz["Q8"].shape
    rng = np.random.default_rng(3)
    rows = np.arange(0, N, 7, dtype=np.int32)
    acc = rng.normal(0.0, 20.0, (B, H, rows.size, Npad)).astype(np.float32)
    acc[..., 0] = 200.0   # the running max is fixed by tile 0
    O, P = oracle_mod.attn(qz, N, softmax_scale=LN2, rows=rows, acc_in=acc, want_codes=True)
    w = oracle_mod.e4m3_decode(P)                     # [B,H,nrows,Npad]
    v = _dequant_v(oracle_mod, qz, 1)                 # [B,H,Npad,d]
    want = np.einsum("bhrt,bhtd->bhrd", w, v) / w.sum(axis=-1, keepdims=True)
    assert np.all(w[..., N:] == 0)
    np.testing.assert_allclose(O, want, rtol=1e-10, atol=1e-12)


def test_reference_permutation_identity(oracle_mod):
    Q, K, V = _small(N=260)
    rng = np.random.default_rng(0)
    pi = rng.permutation(Q.shape[1])
    O1 = oracle_mod.attn_ref(Q, K, V)
    O2 = oracle_mod.attn_ref(Q, K[:, pi], V[:, pi])
    np.testing.assert_allclose(O2, O1, rtol=1e-12, atol=1e-12)


def test_reference_is_softmax(oracle_mod):
    # brute force in torch fp64 on a tiny case
    Q, K, V = _small(N=37, d=64, H=1)
    f = lambda a: torch.from_numpy(oracle_mod.bf16_to_f32(a)).double()[0, :, 0]
    q, k, v = f(Q), f(K), f(V)
    O = torch.softmax(q @ k.T / 8.0, dim=-1) @ v
    np.testing.assert_allclose(oracle_mod.attn_ref(Q, K, V)[0, 0], O.numpy(), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("expcast", [0, 1])
@pytest.mark.parametrize("vsmooth", [0, 1])
def test_equal_scores_give_mean(oracle_mod, expcast, vsmooth):
    N = 300                                  # 3 tiles, ragged tail of 44 keys
    Q, K, V = _small(N=N)
    Q[:] = 0                                 # every score is 0
    qz = oracle_mod.quantize(Q, K, V, None, vsmooth)
    O = oracle_mod.attn(qz, N, expcast=expcast, vsmooth=vsmooth)
    vq = _dequant_v(oracle_mod, qz, vsmooth)[:, :, :N]
    want = vq.mean(axis=2, keepdims=True)
    np.testing.assert_allclose(O, np.broadcast_to(want, O.shape), rtol=1e-12, atol=1e-12)


def _two_key_case(oracle_mod, s1, s2, t1, t2, N=700, d=64, vsmooth=1):
    """Q = e0, key t1 has score s1, key t2 has score s2, all others 0."""
    _, K, V = _small(N=N, d=d, H=1)
    Q = np.zeros_like(K)
    qz = oracle_mod.quantize(Q, K, V, None, vsmooth)
    qz["Q8"][:] = 0
    qz["Q8"][..., 0] = 0x38                       # q = (1, 0, ..., 0)
    qz["sq"][:] = 1.0
    qz["K8"][:] = 0
    qz["sk"][:] = 1.0
    enc = lambda s: oracle_mod.e4m3_encode(np.array([s], np.float32))[0]
    qz["K8"][0, 0, t1, 0] = enc(s1)
    qz["K8"][0, 0, t2, 0] = enc(s2)
    return qz


@pytest.mark.parametrize("expcast", [0, 1])
@pytest.mark.parametrize("vsmooth", [0, 1])
def test_two_dominant_keys_closed_form(oracle_mod, expcast, vsmooth):
    N = 700
    t1, t2, s1, s2 = 5, 3 * 128 + 17, 32.0, 48.0   # max rises in the 4th tile
    qz = _two_key_case(oracle_mod, s1, s2, t1, t2, N=N, vsmooth=vsmooth)
    O = oracle_mod.attn(qz, N, softmax_scale=float(LN2), expcast=expcast, vsmooth=vsmooth)
    vq = _dequant_v(oracle_mod, qz, vsmooth)[0, 0]
    alpha = 2.0 ** (s1 - s2)
    want = (alpha * vq[t1] + vq[t2]) / (alpha + 1.0)
    np.testing.assert_allclose(O[0, 0], np.broadcast_to(want, O[0, 0].shape), rtol=1e-12, atol=1e-12)
    # equal scores: both keys at byte 120, no rescale
    qz = _two_key_case(oracle_mod, s2, s2, t1, t2, N=N, vsmooth=vsmooth)
    O = oracle_mod.attn(qz, N, softmax_scale=float(LN2), expcast=expcast, vsmooth=vsmooth)
    np.testing.assert_allclose(O[0, 0], np.broadcast_to((vq[t1] + vq[t2]) / 2, O[0, 0].shape),
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("expcast", [0, 1])
def test_each_query_block_takes_its_own_scale(oracle_mod, expcast):
    """sigma_ij = s_q,i s_k,j: rows of query block b see the scores s1 sq_b and
    s2 sq_b, so alpha_b = 2^(sq_b (s1 - s2)) in the two-key closed form.  The
    block scales are exact binary fractions; every other key underflows."""
    N = 700
    t1, t2, s1, s2 = 5, 3 * 128 + 17, 32.0, 48.0
    qz = _two_key_case(oracle_mod, s1, s2, t1, t2, N=N, vsmooth=1)
    sq = np.array([1.0, 0.75, 1.5, 1.25, 0.875, 2.0], np.float32)
    qz["sq"][0, 0, :] = sq
    O = oracle_mod.attn(qz, N, softmax_scale=float(LN2), expcast=expcast, vsmooth=1)
    vq = _dequant_v(oracle_mod, qz, 1)[0, 0]
    for b, s in enumerate(sq):
        alpha = 2.0 ** (float(s) * (s1 - s2))
        want = (alpha * vq[t1] + vq[t2]) / (alpha + 1.0)
        rows = O[0, 0, 128 * b:min(N, 128 * (b + 1))]
        np.testing.assert_allclose(rows, np.broadcast_to(want, rows.shape), rtol=1e-12, atol=1e-12)


def test_error_bound_against_exact_softmax(oracle_mod):
    """Row max in tile 0 for every row, so every code is relative to the final max."""
    N, d = 640, 64
    Q, K, V = _small(N=N, d=d, H=1, seed=9)
    qz = oracle_mod.quantize(Q, K, V, None, 1)
    dec = oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))
    rng = np.random.default_rng(2)
    # q = e0 for every row; key t has score dec(k8[t,0]) (sigma = 1 with sq = sk = 1)
    qz["Q8"][:] = 0
    qz["Q8"][..., 0] = 0x38
    qz["sq"][:] = 1.0
    qz["sk"][:] = 1.0
    qz["K8"][:] = 0
    kv = rng.uniform(-6, 6, N).astype(np.float32)
    kv[3] = 8.0                                    # the maximum, in tile 0
    qz["K8"][0, 0, :N, 0] = oracle_mod.e4m3_encode(kv)
    O, P = oracle_mod.attn(qz, N, softmax_scale=float(LN2), expcast=1, vsmooth=1, want_codes=True)
    s = dec[qz["K8"][0, 0, :N, 0]]                 # exact scores in log2 units
    assert np.argmax(s) == 3 and s[3] == 8.0
    p = np.exp2(s - s.max())
    p /= p.sum()
    vq = _dequant_v(oracle_mod, qz, 1)[0, 0, :N]
    exact = p @ vq
    codes = P[0, 0][:, :N]
    ph = dec[codes]
    ph /= ph.sum(axis=1, keepdims=True)
    tv = 0.5 * np.abs(ph - p[None, :]).sum(axis=1)
    tau = np.where(codes < 8, p[None, :], 0).sum(axis=1)
    assert np.all(tv <= 0.0364 + tau)
    assert tv.max() > 0.001                        # the case is not degenerate
    err = np.abs(O[0, 0] - exact[None, :]).max(axis=1)
    assert np.all(err <= 2 * tv * np.abs(vq).max() + 1e-9)


def test_expcast_codes_within_one_of_exp_then_cast(oracle_mod):
    """Same scores, same running max: the two P paths differ by <= 1 code on normals."""
    N = 900
    Q, K, V = _small(N=N, seed=21)
    qz = oracle_mod.quantize(Q, K, V, None, 1)
    _, P1 = oracle_mod.attn(qz, N, expcast=1, vsmooth=1, want_codes=True)
    _, P0 = oracle_mod.attn(qz, N, expcast=0, vsmooth=1, want_codes=True)
    P0, P1 = P0.astype(int), P1.astype(int)
    normal = P0 >= 8
    assert np.abs(P1 - P0)[normal].max() <= 1
    assert 0.70 < np.mean(P1[normal] == P0[normal]) < 0.90
    assert np.all(P1[..., N:] == 0) and np.all(P0[..., N:] == 0)
    assert P1.max() == 120


def test_acc_override_reproduces_codes(oracle_mod):
    """Feeding the oracle's own fp32 scores back gives identical codes and output."""
    N = 260
    Q, K, V = _small(N=N, seed=4)
    qz = oracle_mod.quantize(Q, K, V, None, 1)
    dec = oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))
    q = dec[qz["Q8"]]
    k = dec[qz["K8"]]
    acc = np.einsum("bhic,bhjc->bhij", q, k).astype(np.float32)
    O1, P1 = oracle_mod.attn(qz, N, want_codes=True)
    O2, P2 = oracle_mod.attn(qz, N, want_codes=True, acc_in=acc[:, :, :N])
    np.testing.assert_array_equal(P1, P2)
    np.testing.assert_array_equal(O1, O2)


def test_quantized_close_to_reference(oracle_mod):
    """End-to-end fidelity sanity: quantized path vs fp64 reference on bf16 inputs."""
    N = 1024
    w = inputs.WORKLOADS["tiny"]
    Q, K, V = (inputs.to_u16(t) for t in inputs.make_qkv(w, "cpu"))
    ref = oracle_mod.attn_ref(Q, K, V)
    for ec in (0, 1):
        for vs in (0, 1):
            qz = oracle_mod.quantize(Q, K, V, None, vs)
            O = oracle_mod.attn(qz, N, expcast=ec, vsmooth=vs)
            rel = np.linalg.norm(O - ref) / np.linalg.norm(ref)
            assert rel < 0.1, (ec, vs, rel)
