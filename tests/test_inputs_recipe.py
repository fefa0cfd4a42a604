"""The seeded input generator follows its stated recipe (CPU only).

Checked on CPU draws: determinism per seed, the [B, N, H, d] bf16 layout,
unit-variance Q/K, the per-(head, channel) bias of variance 2 on the
Wan2.2-shaped workload, the 1 % outlier tokens at x20 on 4 channels per head
(drifting by 3 channels per head on the Wan shape), the N(0, 0.05) drift of
the schedule, and the rotary table's split of the channel pairs over the
latent grid's frame, height and width coordinates.
"""
import math

import numpy as np
import pytest
import torch

from bit_fp8_attention_means_gb300 import inputs


def test_deterministic_and_layout():
    w = inputs.WORKLOADS["tiny"]
    a = inputs.make_qkv(w, "cpu")
    b = inputs.make_qkv(w, "cpu")
    c = inputs.make_qkv(w, "cpu", seed=w.seed + 1)
    for x, y, z in zip(a, b, c):
        assert x.dtype == torch.bfloat16 and tuple(x.shape) == (w.B, w.N, w.H, w.d)
        assert torch.equal(x, y) and not torch.equal(x, z)


def test_qk_unit_variance_and_wan_bias():
    tiny = inputs.WORKLOADS["tiny"]
    Q, K, _ = inputs.make_qkv(tiny, "cpu", N=8192)
    for t in (Q, K):
        x = t.float()
        assert abs(x.mean().item()) < 0.02 and abs(x.var().item() - 1.0) < 0.02
    # the Wan shape adds a per-(head, channel) bias ~ N(0, 2): channel means spread with variance ~2
    wan = inputs.WORKLOADS["wan"]
    Q, K, _ = inputs.make_qkv(wan, "cpu", H=8, N=4096)
    for t in (Q, K):
        x = t.float()
        mu = x.mean(dim=1)                                  # [B, H, d]: the bias of each (head, channel)
        assert 1.6 < mu.var().item() < 2.4
        assert abs((x - mu[:, None]).var().item() - 1.0) < 0.03


@pytest.mark.parametrize("name", ["tiny", "wan"])
def test_outlier_tokens_and_channels(name):
    w = inputs.WORKLOADS[name]
    N, H = 20000, 4
    _, _, V = inputs.make_qkv(w, "cpu", H=H, N=N)
    v = V.float()[0]                                        # [N, H, d]
    chans = []
    for h in range(H):
        # x20 of an O(1) value exceeds 12 on some of its channels; an unscaled one
        # (the mixture and noise have a standard deviation below 2) never does
        big = v[:, h].abs() > 12.0
        ch = torch.nonzero(big.any(dim=0)).flatten()
        assert ch.numel() == 4                              # 4 outlier channels
        frac = big.any(dim=1).float().mean().item()
        assert 0.007 < frac < 0.013, frac                   # on ~1 % of the tokens
        chans.append(ch)
    # each head draws its own outlier channels
    sets = {tuple(sorted(c.tolist())) for c in chans}
    assert len(sets) == H


def test_schedule_drift_variance():
    w = inputs.WORKLOADS["tiny"]
    _, _, V = inputs.make_qkv(w, "cpu", N=8192)
    V1 = inputs.drift_v(V, 1, seed=5)
    diff = V1.float() - V.float()
    # bf16 rounding of the result adds a little variance on top of 0.05
    assert 0.045 < diff.var().item() < 0.06
    assert torch.equal(V1, inputs.drift_v(V, 1, seed=5)) and not torch.equal(V1, inputs.drift_v(V, 2, seed=5))


def test_rope_table_grid_split():
    F, Hh, Ww = inputs.WAN_GRID
    N, d = F * Hh * Ww, 128
    T = inputs.rope_table(N, d, grid=inputs.WAN_GRID)
    assert T.shape == (N, d // 2, 2) and T.dtype == np.float32
    np.testing.assert_allclose(T[..., 0] ** 2 + T[..., 1] ** 2, 1.0, atol=1e-6)
    ps = (d // 2) // 3
    nf = d // 2 - 2 * ps                                    # 22 / 21 / 21 pairs
    assert (nf, ps) == (22, 21)

    def ang(n, pair):
        return math.atan2(float(T[n, pair, 1]), float(T[n, pair, 0]))

    # token (f, y, x) = (2, 3, 5): each axis's pair 0 rotates by its own coordinate
    n = 2 * Hh * Ww + 3 * Ww + 5
    assert ang(n, 0) == pytest.approx(2.0, abs=1e-6)
    assert ang(n, nf) == pytest.approx(3.0, abs=1e-6)
    assert ang(n, nf + ps) == pytest.approx(5.0 - 2 * math.pi, abs=1e-6)
    # the frame axis's pair i has frequency 10^4^(-2i/44)
    i = 7
    want = (2.0 * 1e4 ** (-2 * i / (2 * nf)))
    assert ang(n, i) == pytest.approx(want, abs=1e-6)
    # without a grid every pair follows the token index
    T1 = inputs.rope_table(64, 64)
    assert math.atan2(float(T1[1, 0, 1]), float(T1[1, 0, 0])) == pytest.approx(1.0, abs=1e-6)
    np.testing.assert_allclose(T1[0, :, 0], 1.0)
    np.testing.assert_allclose(T1[0, :, 1], 0.0)
