"""Full-size parity on the Wan2.2-shaped workload (B=1, H=40, N=75,600, d=128).

The whole path runs at full size in the launch configuration the benchmark
times; the oracle checks what it can compute one by one: the quantizer
bit-exactly for two heads, O on sampled query rows of those heads (including
the ragged last tile), and the grouping invariants on sampled tokens.
"""
import numpy as np
import pytest
import torch

from bit_fp8_attention_means_gb300 import inputs, vc
from rowsample import sampled_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
u16 = inputs.to_u16


def test_wan_full_size_sampled(oracle_mod):
    w = inputs.WORKLOADS["wan"]
    Q, K, V = inputs.make_qkv(w, DEV)
    cent, _, _ = vc.vc_cluster(V, w.k, w.iters)
    c_prev = cent.clone()
    cent, lab, perm = vc.vc_cluster(V, w.k, 1, warm_start=True, centroids=cent)
    qz = vc.vc_quantize(Q, K, V, perm, 1)
    O = vc.vc_attn_fwd(qz, vc.shape_of(Q), expcast=1, vsmooth=1)
    torch.cuda.synchronize()
    N = w.N
    rng = np.random.default_rng(0)
    for h in (0, 23, 39):
        Qh, Kh, Vh = (u16(t[:, :, h:h + 1]) for t in (Q, K, V))
        ph = perm[:, h:h + 1].cpu().numpy()
        lh = lab[:, h:h + 1].cpu().numpy()
        # pi is the stable argsort of the labels
        np.testing.assert_array_equal(ph[0, 0], np.argsort(lh[0, 0], kind="stable"))
        # labels are nearest centroids on sampled tokens
        v = oracle_mod.bf16_to_f32(Vh).astype(np.float64)[0, :, 0]
        cp = c_prev[0, h].cpu().numpy().astype(np.float64)
        toks = rng.choice(N, 512, replace=False)
        d2 = ((v[toks][:, None] - cp[None]) ** 2).sum(-1)
        chosen = d2[np.arange(toks.size), lh[0, 0, toks]]
        scale = (v[toks] ** 2).sum(-1) + (cp ** 2).sum(-1)[lh[0, 0, toks]]
        assert np.all(chosen - d2.min(1) <= 4 * 128 * 2.0 ** -24 * scale + 1e-6)
        # quantizer bit-exact for this head
        want = oracle_mod.quantize(Qh, Kh, Vh, ph, 1)
        for key in ("Q8", "sq", "K8", "sk", "V8T", "sv"):
            np.testing.assert_array_equal(qz[key][:, h:h + 1].cpu().numpy(), want[key], err_msg=key)
        np.testing.assert_array_equal(qz["mu"][:, h:h + 1].cpu().numpy().view(np.uint16), want["mu"])
        # O on sampled rows, including the first tile, the last (80-row) tile and the one before it
        rows = sampled_rows(N, rng, 40)
        ref = oracle_mod.attn(want, N, rows=rows)[0, 0]
        got = O[0, rows, h].float().cpu().numpy()
        oracle_mod.check_o(got, ref, "wan head %d" % h)


@pytest.mark.parametrize("mode", ["exp_then_cast", "hybrid_m2"])
def test_wan_full_size_other_bytes(oracle_mod, mode):
    """The exp-then-cast and hybrid probability bytes at the full Wan2.2 shape:
    O on sampled rows of the last head (incl. the masked last tile) within
    the oracle's bars for exponential-derived bytes."""
    w = inputs.WORKLOADS["wan"]
    Q, K, V = inputs.make_qkv(w, DEV)
    perm = vc.vc_cluster(V, w.k, w.iters)[2]
    qz = vc.vc_quantize(Q, K, V, perm, 1)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    if mode == "exp_then_cast":
        O = vc.vc_attn_fwd(qz, vc.shape_of(Q), expcast=0, vsmooth=1, dev_status=status)
        kw = dict(expcast=0)
    else:
        O = vc.vc_attn_fwd(qz, vc.shape_of(Q), vsmooth=1, exact_margin=2.0, dev_status=status)
        kw = dict(expcast=2, margin=2.0)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    h = w.H - 1
    one = {k: qz[k][:, h:h + 1].cpu().numpy() for k in ("Q8", "sq", "K8", "sk", "V8T", "sv")}
    one["mu"] = qz["mu"][:, h:h + 1].cpu().numpy().view(np.uint16)
    rng = np.random.default_rng(11)
    # the hybrid votes over whole 32-row groups: sample whole groups
    groups = np.unique(sampled_rows(w.N, rng, 6) // 32)
    rows = np.concatenate([np.arange(g * 32, min(w.N, g * 32 + 32)) for g in groups]).astype(np.int32)
    ref = oracle_mod.attn(one, w.N, vsmooth=1, rows=rows, **kw)[0, 0]
    oracle_mod.check_o(O[0, rows, h].float().cpu().numpy(), ref, "wan %s head %d" % (mode, h), exp_bytes=True)
