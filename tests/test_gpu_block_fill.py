"""GPU parity of the block-fill permutation (vc_cluster_ex, block_fill = 1).

Bars: given the labels and centroids the device returns, the permutation is
bit-exact against the oracle's block fill (fp32 chain distances in the same
order); the k-means part is unchanged by the flag; attention on the filled
permutation matches the oracle within 2e-3.
"""
import numpy as np
import pytest
import torch

from bit_fp8_attention_means_gb300 import inputs, vc

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
u16 = inputs.to_u16

CASES = [dict(w="tiny", N=1000, d=64, H=2, k=8), dict(w="medium", N=3000, d=128, H=3, k=37),
         dict(w="medium", N=8192, d=128, H=2, k=64), dict(w="tiny", N=130, d=64, H=1, k=3)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "N%d_d%d_k%d" % (c["N"], c["d"], c["k"]))
def test_block_fill_bitexact(oracle_mod, case):
    w = inputs.WORKLOADS[case["w"]]
    _, _, V = inputs.make_qkv(w, DEV, H=case["H"], N=case["N"], d=case["d"])
    c0, l0, p0 = vc.vc_cluster(V, case["k"], 3)
    c1, l1, p1 = vc.vc_cluster(V, case["k"], 3, block_fill=1)
    torch.cuda.synchronize()
    assert torch.equal(l0, l1) and torch.equal(c0, c1)
    want = oracle_mod.block_fill(l1.cpu().numpy(), c1.cpu().numpy())
    np.testing.assert_array_equal(p1.cpu().numpy(), want)
    # the plain permutation is still the stable argsort of the same labels
    np.testing.assert_array_equal(p0.cpu().numpy(), oracle_mod.argsort_labels(l0.cpu().numpy(), case["k"]))


def test_block_fill_wan_size(oracle_mod):
    w = inputs.WORKLOADS["wan"]
    _, _, V = inputs.make_qkv(w, DEV)
    cent, _, _ = vc.vc_cluster(V, w.k, w.iters)
    cent, lab, perm = vc.vc_cluster(V, w.k, 1, warm_start=True, centroids=cent, block_fill=1)
    torch.cuda.synchronize()
    for h in (0, 21, 39):
        want = oracle_mod.block_fill(lab[:, h:h + 1].cpu().numpy(), cent[:, h:h + 1].cpu().numpy())
        np.testing.assert_array_equal(perm[:, h:h + 1].cpu().numpy(), want)


def test_attention_on_block_fill(oracle_mod):
    w = inputs.WORKLOADS["medium"]
    Q, K, V = inputs.make_qkv(w, DEV, H=2, N=2000)
    _, _, perm = vc.vc_cluster(V, 16, 3, block_fill=1)
    qz = vc.vc_quantize(Q, K, V, perm, 1)
    O = vc.vc_attn_fwd(qz, vc.shape_of(Q))
    torch.cuda.synchronize()
    want = oracle_mod.quantize(u16(Q), u16(K), u16(V), perm.cpu().numpy(), 1)
    for key in ("Q8", "sq", "K8", "sk", "V8T", "sv"):
        np.testing.assert_array_equal(qz[key].cpu().numpy(), want[key], err_msg=key)
    ref = oracle_mod.attn(want, 2000)
    got = O.float().cpu().numpy().transpose(0, 2, 1, 3)
    oracle_mod.check_o(got, ref, "block fill")


def test_block_fill_batched_warm(oracle_mod):
    """B = 2, d = 64, warm start: the filled permutation of every (b, h)."""
    w = inputs.WORKLOADS["tiny"]
    _, _, V = inputs.make_qkv(w, DEV, B=2, H=3, N=2500, d=64)
    cent, _, _ = vc.vc_cluster(V, 20, 3)
    cent, lab, perm = vc.vc_cluster(V, 20, 1, warm_start=True, centroids=cent, block_fill=1)
    torch.cuda.synchronize()
    want = oracle_mod.block_fill(lab.cpu().numpy(), cent.cpu().numpy())
    np.testing.assert_array_equal(perm.cpu().numpy(), want)
