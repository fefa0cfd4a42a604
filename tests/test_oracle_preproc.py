"""Pins of the oracle's Q/K preprocessing: the rotary transform and the
Hadamard rotation ahead of the quantizer.

The pages list both among the steps of their fused quantization kernel (paper
summary, 核心方法; study note 3-1 "Fused CuTe kernel" and 3-3 "Kernel
fusion") and name the Hadamard rotation of the Q/K channels as
FlashAttention-3's (paper summary, 研究动机) without formulas.  The pins tie
the oracle to what the mathematics fixes, independently of its own code:

* Hadamard: equals the Sylvester matrix built by the Kronecker recursion
  (exactly on integer rows, within the summation-tree bound on real rows);
* rotary: equals complex multiplication by e^{i theta} in fp64, has the
  counter-clockwise sign, preserves the pair norms and makes scores depend on
  the position difference only; K rows rotate at their own token's position;
* with an identity table and no Hadamard the quantizer is the plain one,
  bit for bit;
* the dequantized scores, and attention, match fp64 on the rotated inputs,
  which fails if the 1/d of the Hadamard is lost or one side is not rotated.
"""
import numpy as np
import pytest
import torch

from bit_fp8_attention_means_gb300 import inputs

U = 2.0 ** -24  # unit roundoff of fp32


def _sylvester(d: int) -> np.ndarray:
    H = np.array([[1]], dtype=np.int64)
    while H.shape[0] < d:
        H = np.kron(np.array([[1, 1], [1, -1]], dtype=np.int64), H)
    return H


def _bf16_rows(x: np.ndarray) -> np.ndarray:
    return inputs.to_u16(torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16))


def _f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("d", [64, 128])
def test_hadamard_integer_rows_exact(oracle_mod, d):
    rng = np.random.default_rng(d)
    X = rng.integers(-8, 9, size=(50, d)).astype(np.float32)
    got = oracle_mod.preproc_rows(_bf16_rows(X), hadamard=1)
    want = X.astype(np.int64) @ _sylvester(d).T
    np.testing.assert_array_equal(got, want.astype(np.float32))


@pytest.mark.parametrize("d", [64, 128])
def test_hadamard_real_rows_within_tree_bound(oracle_mod, d):
    rng = np.random.default_rng(7 + d)
    bits = _bf16_rows(rng.standard_normal((200, d)) * np.exp(rng.uniform(-3, 3, (200, 1))))
    x = _f32(bits).astype(np.float64)
    got = oracle_mod.preproc_rows(bits, hadamard=1).astype(np.float64)
    want = x @ _sylvester(d).T.astype(np.float64)
    k = int(np.log2(d))
    bound = (k * U / (1 - k * U)) * np.abs(x).sum(axis=1, keepdims=True)
    assert np.all(np.abs(got - want) <= bound)
    # and it is not the identity or a permutation: the energy grows by d
    np.testing.assert_allclose((got ** 2).sum(1), d * (x ** 2).sum(1), rtol=1e-5)


def test_rotary_sign_and_pairs(oracle_mod):
    d = 8
    rope = np.zeros((1, d // 2, 2), np.float32)
    rope[0, :, 0] = 1.0          # identity on pairs 1..3
    rope[0, 0] = (0.0, 1.0)      # +90 degrees on pair (0, 1)
    x = np.array([[1, 0, 2, 3, 4, 5, 6, 7]], np.float32)
    got = oracle_mod.preproc_rows(_bf16_rows(x), rope=rope)
    np.testing.assert_array_equal(got, [[0, 1, 2, 3, 4, 5, 6, 7]])


@pytest.mark.parametrize("d", [64, 128])
def test_rotary_is_complex_multiplication(oracle_mod, d):
    rng = np.random.default_rng(11)
    n = 300
    bits = _bf16_rows(rng.standard_normal((n, d)) * 4)
    theta = rng.uniform(-np.pi, np.pi, (n, d // 2))
    rope = np.stack([np.cos(theta), np.sin(theta)], -1).astype(np.float32)
    got = oracle_mod.preproc_rows(bits, rope=rope).astype(np.float64)
    x = _f32(bits).astype(np.float64)
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * (rope[..., 0].astype(np.float64) + 1j * rope[..., 1].astype(np.float64))
    want = np.empty_like(got)
    want[:, 0::2], want[:, 1::2] = z.real, z.imag
    mag = np.repeat(np.abs(x[:, 0::2]) + np.abs(x[:, 1::2]), 2, axis=1)
    assert np.all(np.abs(got - want) <= 2.01 * U * mag)
    # a rotation: pair norms kept (up to the table's own rounding)
    np.testing.assert_allclose(np.abs(z), np.hypot(x[:, 0::2], x[:, 1::2]), rtol=1e-6)


def test_rotary_scores_depend_on_position_difference(oracle_mod):
    d, N = 64, 600
    rope = inputs.rope_table(N, d)
    rng = np.random.default_rng(3)
    q = _bf16_rows(rng.standard_normal((1, d)))
    k = _bf16_rows(rng.standard_normal((1, d)))
    qm = oracle_mod.preproc_rows(np.repeat(q, N, 0), rope=rope).astype(np.float64)
    kn = oracle_mod.preproc_rows(np.repeat(k, N, 0), rope=rope).astype(np.float64)
    base = float(np.linalg.norm(_f32(q)) * np.linalg.norm(_f32(k)))
    for m, n, shift in [(10, 3, 250), (0, 500, 77), (123, 123, 400)]:
        s0 = qm[m] @ kn[n]
        s1 = qm[m + shift] @ kn[n + shift] if max(m, n) + shift < N else qm[m - shift] @ kn[n - shift]
        assert abs(s0 - s1) <= 1e-4 * base, (m, n, s0, s1)
    # and they do change with the difference
    assert abs(qm[10] @ kn[3] - qm[10] @ kn[40]) > 1e-3 * base


def test_identity_preprocessing_is_the_plain_quantizer(oracle_mod):
    w = inputs.WORKLOADS["tiny"]
    Q, K, V = inputs.make_qkv(w, "cpu", H=2, N=700, seed=4)
    Q, K, V = (inputs.to_u16(t) for t in (Q, K, V))
    rng = np.random.default_rng(1)
    perm = np.stack([rng.permutation(700) for _ in range(2)])[None].astype(np.int32)
    ident = np.zeros((700, 32, 2), np.float32)
    ident[..., 0] = 1.0
    a = oracle_mod.quantize(Q, K, V, perm, 1)
    b = oracle_mod.quantize(Q, K, V, perm, 1, rope=ident, hadamard=0)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_k_rows_rotate_at_their_own_position(oracle_mod):
    w = inputs.WORKLOADS["tiny"]
    N, d = 500, 64
    Q, K, V = inputs.make_qkv(w, "cpu", H=1, N=N, seed=9)
    Q, K, V = (inputs.to_u16(t) for t in (Q, K, V))
    pi = np.random.default_rng(2).permutation(N).astype(np.int32)
    rope = inputs.rope_table(N, d)
    a = oracle_mod.quantize(Q, K, V, pi[None, None], 1, rope=rope, hadamard=1)
    # gathering first and carrying each token's table row along gives the same K'
    b = oracle_mod.quantize(Q, K[:, pi], V[:, pi], None, 1, rope=rope[pi], hadamard=1)
    np.testing.assert_array_equal(a["K8"], b["K8"])
    np.testing.assert_array_equal(a["sk"], b["sk"])


def _rotated_f64(X_bits, rope):
    x = _f32(X_bits).astype(np.float64)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * (rope[:, None, :, 0] + 1j * rope[:, None, :, 1])
    y = np.empty_like(x)
    y[..., 0::2], y[..., 1::2] = z.real, z.imag
    return y  # [B, N, H, d]


@pytest.mark.parametrize("hadamard", [0, 1])
def test_dequantized_scores_match_rotated_inputs(oracle_mod, hadamard):
    w = inputs.WORKLOADS["medium"]
    N, d = 300, 128
    Q, K, V = inputs.make_qkv(w, "cpu", H=1, N=N, seed=13)
    Q, K, V = (inputs.to_u16(t) for t in (Q, K, V))
    rope = inputs.rope_table(N, d)
    qz = oracle_mod.quantize(Q, K, V, None, 1, rope=rope, hadamard=hadamard)
    nb = oracle_mod.nblk_of(N)
    blk = np.arange(N) // 128
    q = oracle_mod.e4m3_decode(qz["Q8"][0, 0, :N]) * qz["sq"][0, 0, blk][:, None]
    k = oracle_mod.e4m3_decode(qz["K8"][0, 0, :N]) * qz["sk"][0, 0, blk][:, None]
    S = q @ k.T
    y = _rotated_f64(np.concatenate([Q, K], 2), rope.astype(np.float64))
    S_ref = y[0, :, 0] @ y[0, :, 1].T
    rel = np.linalg.norm(S - S_ref) / np.linalg.norm(S_ref)
    assert rel < 0.06, rel
    assert nb == 3
    if hadamard:
        # s_q carries the 1/d of H H = d I: s_q * d is the block amax / 448
        rows = oracle_mod.preproc_rows(Q[0, :, 0], rope=rope, hadamard=1)
        for j in range(nb):
            amax = np.float32(np.abs(rows[128 * j:128 * (j + 1)]).max())
            assert qz["sq"][0, 0, j] * np.float32(d) == amax / np.float32(448.0)


@pytest.mark.parametrize("hadamard", [0, 1])
def test_attention_on_preprocessed_inputs(oracle_mod, hadamard):
    w = inputs.WORKLOADS["medium"]
    N, d = 384, 128
    Q, K, V = inputs.make_qkv(w, "cpu", H=1, N=N, seed=17)
    Q, K, V = (inputs.to_u16(t) for t in (Q, K, V))
    rope = inputs.rope_table(N, d)
    pi = np.random.default_rng(5).permutation(N).astype(np.int32)[None, None]
    qz = oracle_mod.quantize(Q, K, V, pi, 1, rope=rope, hadamard=hadamard)
    O = oracle_mod.attn(qz, N, expcast=0, vsmooth=1)[0, 0]
    y = _rotated_f64(np.concatenate([Q, K], 2), rope.astype(np.float64))
    S = y[0, :, 0] @ y[0, :, 1].T / np.sqrt(d)
    P = np.exp(S - S.max(1, keepdims=True))
    ref = (P / P.sum(1, keepdims=True)) @ _f32(V[0, :, 0]).astype(np.float64)
    rel = np.linalg.norm(O - ref) / np.linalg.norm(ref)
    assert rel < 0.05, rel
