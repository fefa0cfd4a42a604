"""Pins of the oracle's 4-bit V residual (vco_quantize_v4) and its codec (CPU only).

The pages' 4-bit path keeps the V residual in 4 bits with a per-block scale
(paper summary, 方法步骤详情 step 2, "4 比特 NVFP4"); with FP8 probabilities
this build reads it as E2M1 with a power-of-two scale per 32 tokens of a
channel (the OCP MX rule) under the per-channel scale amax/6.  Pins:

* the E2M1 code table (OCP FP4: 1 sign, 2 exponent bits with bias 1, 1
  mantissa bit) written out by value, and every E2M1 value times 2^e,
  e in [-8, 0], is an E4M3 value (so the E4M3 carrier is exact);
* round to nearest, ties to the even code, saturating at 6: the tie and
  saturation cases by value, decode/encode round trips, sign symmetry;
* the quantizer's output: one scale per channel = amax/6; within every
  32-token group the values share one power of two 2^e with
  e = floor(log2 max|x|) - 2 (clamped to [-8, 0]), lie on the E2M1 grid
  scaled by it, carry the group maximum to 4 or 6 (times 2^e), and stay
  within 2^(e+1) of x (half the widest step, or the saturation above 6);
* values that are exactly E2M1 times powers of two survive the round trip;
* the mean restore P(R_q + 1 mu) = P R_q + r mu still holds: the oracle's
  attention on the 4-bit operands equals the fp64 weighted mean of its own
  dequantized V'.
"""
import math

import numpy as np

from bit_fp8_attention_means_gb300 import inputs

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # OCP FP4 (E2M1) magnitudes, codes 0-7
LN2 = np.float32(math.log(2.0))


def test_e2m1_table(oracle_mod):
    for c in range(16):
        want = E2M1[c & 7] * (-1.0 if c & 8 else 1.0)
        assert oracle_mod.e2m1_decode(c) == want, c
    # every scaled E2M1 value is exactly an E4M3 value
    for e in range(-8, 1):
        for v in E2M1[1:]:
            x = np.float32(v * 2.0 ** e)
            assert oracle_mod.e4m3_decode(oracle_mod.e4m3_encode(np.array([x]))[0]) == x, (v, e)


def test_e2m1_rounding(oracle_mod):
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    just = {0.2499: 0.0, 0.2501: 0.5, 0.7499: 0.5, 2.4999: 2.0, 2.5001: 3.0, 4.999: 4.0, 5.001: 6.0}
    sat = {6.0: 6.0, 6.9: 6.0, 7.0: 6.0, 8.0: 6.0, 1e30: 6.0}
    for table in (ties, just, sat):
        for x, v in table.items():
            for s in (1.0, -1.0):
                c = oracle_mod.e2m1_encode(np.array([s * x], np.float32))[0]
                assert oracle_mod.e2m1_decode(c) == s * v, (s * x, c)
    for c in range(16):
        assert oracle_mod.e2m1_encode(np.array([oracle_mod.e2m1_decode(c)], np.float32))[0] == c or c == 8
    x = np.linspace(-7.0, 7.0, 20001, dtype=np.float32)
    dec = np.array([oracle_mod.e2m1_decode(c) for c in oracle_mod.e2m1_encode(x)])
    assert np.all(np.diff(dec) >= 0)                              # monotone
    grid = np.array(E2M1)
    err = np.abs(np.abs(x.astype(np.float64)) - np.abs(dec))
    nearest = np.min(np.abs(np.abs(x.astype(np.float64))[:, None] - grid[None]), axis=1)
    assert np.all(err <= nearest + 1e-12)                          # a nearest value


def _case(N, d, H, seed, vmul=1.0):
    w = inputs.WORKLOADS["tiny"]
    Q, K, V = inputs.make_qkv(w, "cpu", H=H, N=N, d=d, seed=seed)
    V = (V.float() * vmul).to(V.dtype)
    return inputs.to_u16(Q), inputs.to_u16(K), inputs.to_u16(V)


def test_quantizer_mx_structure(oracle_mod):
    N, d, H = 700, 64, 2
    Q, K, V = _case(N, d, H, seed=61)
    rng = np.random.default_rng(1)
    perm = np.stack([rng.permutation(N) for _ in range(H)])[None].astype(np.int32)
    qz = oracle_mod.quantize(Q, K, V, perm, 1, vbits=4)
    q8 = oracle_mod.quantize(Q, K, V, perm, 1)
    for key in ("Q8", "sq", "K8", "sk", "mu"):                     # only V's residual changes
        np.testing.assert_array_equal(qz[key], q8[key])
    v = oracle_mod.bf16_to_f32(V).transpose(0, 2, 1, 3)[0]          # [H, N, d]
    mu = oracle_mod.bf16_to_f32(qz["mu"])[0]                         # [H, nblk, d]
    Npad = qz["V8T"].shape[-1]
    for h in range(H):
        vp = v[h][perm[0, h]]                                        # V' = V[pi]
        R = (vp - np.repeat(mu[h], 128, axis=0)[:N]).astype(np.float32)
        amax = np.abs(R).max(axis=0)
        np.testing.assert_array_equal(qz["sv"][0, h], (amax / np.float32(6.0)).astype(np.float32))
        inv = np.where(amax > 0, np.float32(6.0) / amax, np.float32(0.0)).astype(np.float32)
        x = (R * inv[None]).astype(np.float32)                       # [N, d]
        val = oracle_mod.e4m3_decode(qz["V8T"][0, h]).T              # [Npad, d]
        assert np.all(val[N:] == 0)
        for g0 in range(0, N, 32):
            xs = x[g0:g0 + 32].astype(np.float64)
            vs = val[g0:min(g0 + 32, N)]
            a = np.abs(xs).max(axis=0)
            e = np.where(a > 0, np.floor(np.log2(np.where(a > 0, a, 1.0))) - 2, -8)
            e = np.clip(e, -8, 0)
            scaled = vs / 2.0 ** e[None]
            assert np.all(np.isin(np.abs(scaled), E2M1)), g0           # on the grid of 2^e
            top = np.abs(scaled).max(axis=0)
            live = (a > 0) & (e > -8)
            assert np.all(np.isin(top[live], [4.0, 6.0])), g0           # the maximum lands on 4 or 6
            assert np.all(np.abs(xs - vs) <= 2.0 ** (e + 1)[None] + 1e-12), g0


def test_exact_values_round_trip(oracle_mod):
    """V = g * q * 2^e exactly (vsmooth off): the residual comes back bit for bit."""
    N, d = 256, 64
    rng = np.random.default_rng(2)
    g = 0.25
    q = rng.choice(E2M1, size=(N, d)) * rng.choice([-1.0, 1.0], size=(N, d))
    e = rng.integers(-3, 1, size=(N // 32, d))
    q[::32] = 4.0                                                    # every group's maximum is 4 * 2^e
    q[0] = 6.0                                                       # and one 6 per channel fixes amax = 6 g
    e[0] = 0
    V = (g * q * 2.0 ** np.repeat(e, 32, axis=0)).astype(np.float32)
    Vb = oracle_mod.bf16_rne(V)
    assert np.array_equal(oracle_mod.bf16_to_f32(Vb), V)              # exactly representable
    Vb = Vb.reshape(1, N, 1, d)
    qz = oracle_mod.quantize(Vb, Vb, Vb, None, 0, vbits=4)
    np.testing.assert_array_equal(qz["sv"][0, 0], np.full(d, np.float32(6.0 * g / 6.0)))
    back = oracle_mod.e4m3_decode(qz["V8T"][0, 0]).T[:N] * qz["sv"][0, 0][None]
    np.testing.assert_array_equal(back, V)


def test_mean_restore_with_4bit_residual(oracle_mod):
    """P (R_q + 1 mu_j) = P R_q + r_ij mu_j with the 4-bit residual: the oracle's
    output equals the fp64 weighted mean of s_v dec(V8T) + mu_j under its own bytes."""
    N, d = 700, 64
    Q, K, V = _case(N, d, 2, seed=21)
    qz = oracle_mod.quantize(Q, K, V, None, 1, vbits=4)
    B, H, Npad, _ = qz["Q8"].shape
    rng = np.random.default_rng(3)
    rows = np.arange(0, N, 7, dtype=np.int32)
    acc = rng.normal(0.0, 20.0, (B, H, rows.size, Npad)).astype(np.float32)
    acc[..., 0] = 200.0   # the running max is fixed by tile 0: no rescale
    O, P = oracle_mod.attn(qz, N, softmax_scale=LN2, rows=rows, acc_in=acc, want_codes=True)
    w = oracle_mod.e4m3_decode(P)
    v = oracle_mod.e4m3_decode(qz["V8T"]).transpose(0, 1, 3, 2) * qz["sv"][:, :, None, :]
    v = v + np.repeat(oracle_mod.bf16_to_f32(qz["mu"]).astype(np.float64), 128, axis=2)
    want = np.einsum("bhrt,bhtd->bhrd", w, v) / w.sum(axis=-1, keepdims=True)
    np.testing.assert_allclose(O, want, rtol=1e-10, atol=1e-12)
