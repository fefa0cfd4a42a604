"""Pins for the oracle's grouping step (CPU only).

[R] 方法步骤详情 step 1: online k-means labels per (batch, head), pi =
argsort(z).  Pins: every label is a nearest centroid (fp64 brute force), the
centroids are the means of their members (an empty cluster keeps its
centroid), the objective does not increase, the cold start uses tokens
floor(i N / k), and pi matches numpy's stable sort.
"""
import numpy as np

from bit_fp8_attention_means_gb300 import inputs


def _v(N=900, d=64, H=2, seed=4):
    _, _, V = inputs.make_qkv(inputs.WORKLOADS["tiny"], "cpu", H=H, N=N, d=d, seed=seed)
    return inputs.to_u16(V)


def _vf(oracle_mod, V):
    return oracle_mod.bf16_to_f32(V).astype(np.float64).transpose(0, 2, 1, 3)   # [B,H,N,d]


def _d2(v, c):
    return ((v[:, None, :] - c[None, :, :].astype(np.float64)) ** 2).sum(axis=2)


def test_labels_nearest_and_centroids_are_means(oracle_mod):
    V = _v()
    k = 8
    c_prev, _ = oracle_mod.kmeans(V, k, 2)
    cent, lab = oracle_mod.kmeans(V, k, 1, centroids=c_prev)      # one warm iteration
    v = _vf(oracle_mod, V)
    for b in range(v.shape[0]):
        for h in range(v.shape[1]):
            d2 = _d2(v[b, h], c_prev[b, h])
            np.testing.assert_array_equal(lab[b, h], np.argmin(d2, axis=1))   # argmin: lowest index on ties
            for i in range(k):
                mem = lab[b, h] == i
                if mem.any():
                    np.testing.assert_allclose(cent[b, h, i], v[b, h][mem].mean(axis=0), rtol=1e-6, atol=1e-6)
                else:
                    np.testing.assert_array_equal(cent[b, h, i], c_prev[b, h, i])


def test_empty_cluster_keeps_its_centroid(oracle_mod):
    """A centroid no token is nearest to owns no label and is returned unchanged."""
    V = _v(N=500)
    k = 6
    c_prev, _ = oracle_mod.kmeans(V, k, 2)
    c_prev[:, :, 4] = 1.0e4              # far from every token: cluster 4 stays empty
    c_prev[0, 1, 2] = -3.0e4             # and cluster 2 of head 1
    cent, lab = oracle_mod.kmeans(V, k, 1, centroids=c_prev)
    assert not np.any(lab == 4) and not np.any(lab[0, 1] == 2)
    np.testing.assert_array_equal(cent[:, :, 4], c_prev[:, :, 4])
    np.testing.assert_array_equal(cent[0, 1, 2], c_prev[0, 1, 2])


def test_cold_start_rule(oracle_mod):
    V = _v(N=300)
    k = 7
    _, lab = oracle_mod.kmeans(V, k, 1)
    v = _vf(oracle_mod, V)
    N = v.shape[2]
    init = v[:, :, [(i * N) // k for i in range(k)]]
    for b in range(v.shape[0]):
        for h in range(v.shape[1]):
            np.testing.assert_array_equal(lab[b, h], np.argmin(_d2(v[b, h], init[b, h]), axis=1))


def test_each_token_its_own_cluster(oracle_mod):
    V = _v(N=64)
    _, lab = oracle_mod.kmeans(V, 64, 1)
    assert np.all(lab == np.arange(64))


def test_objective_non_increasing(oracle_mod):
    V = _v(N=1200, seed=9)
    v = _vf(oracle_mod, V)
    k = 16
    cent, _ = oracle_mod.kmeans(V, k, 1)
    prev = None
    for it in range(6):
        c_in = cent.copy()
        cent, lab = oracle_mod.kmeans(V, k, 1, centroids=c_in)
        obj = sum(_d2(v[b, h], c_in[b, h]).min(axis=1).sum() for b in range(v.shape[0]) for h in range(v.shape[1]))
        if prev is not None:
            assert obj <= prev * (1 + 1e-12)
        prev = obj


def test_argsort_is_stable_sort(oracle_mod):
    rng = np.random.default_rng(5)
    lab = rng.integers(0, 13, (2, 3, 1000)).astype(np.int32)
    perm = oracle_mod.argsort_labels(lab, 13)
    for b in range(2):
        for h in range(3):
            np.testing.assert_array_equal(perm[b, h], np.argsort(lab[b, h], kind="stable"))
            assert np.all(np.diff(lab[b, h][perm[b, h]]) >= 0)
            assert np.array_equal(np.sort(perm[b, h]), np.arange(1000))
