"""GPU parity of the 4-bit V residual (vc_quantize_v4) against the oracle.

Bars: every output of the quantizer (Q8, sq, K8, sk, the V residual bytes,
its channel scales and the block means) bit-exact against the oracle's
4-bit form (E2M1 with a power-of-two scale per 32 tokens of a channel, each
value stored as its E4M3 byte); attention on those operands within the
oracle's O bars (oracle.check_o), including the full Wan2.2 shape on sampled
rows; fidelity against unquantized fp64 attention reported beside the 8-bit
residual's.
"""
import numpy as np
import pytest
import torch

from bit_fp8_attention_means_gb300 import inputs, vc
from rowsample import sampled_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
u16 = inputs.to_u16
KEYS = ("Q8", "sq", "K8", "sk", "V8T", "sv")

CASES = [dict(N=1000, d=128, H=3, B=1, seed=1), dict(N=129, d=64, H=2, B=1, seed=2),
         dict(N=1, d=128, H=1, B=1, seed=3), dict(N=700, d=64, H=2, B=2, seed=4),
         dict(N=2500, d=128, H=1, B=1, seed=5)]


def _np(qz):
    out = {k: qz[k].cpu().numpy() for k in KEYS}
    out["mu"] = qz["mu"].cpu().numpy().view(np.uint16) if qz.get("mu") is not None else None
    return out


@pytest.mark.parametrize("case", CASES, ids=lambda c: "N%d_d%d_H%d_B%d" % (c["N"], c["d"], c["H"], c["B"]))
@pytest.mark.parametrize("vsmooth", [1, 0])
def test_v4_quantizer_bitexact(oracle_mod, case, vsmooth):
    w = inputs.WORKLOADS["tiny"]
    Q, K, V = inputs.make_qkv(w, "cpu", B=case["B"], H=case["H"], N=case["N"], d=case["d"], seed=case["seed"])
    B, N, H, d = Q.shape
    g = torch.Generator().manual_seed(case["seed"])
    perm = torch.stack([torch.stack([torch.randperm(N, generator=g) for _ in range(H)]) for _ in range(B)])
    perm = perm.to(torch.int32)
    qz = vc.vc_quantize(Q.to(DEV), K.to(DEV), V.to(DEV), perm.to(DEV), vsmooth, vbits=4)
    got = _np(qz)
    want = oracle_mod.quantize(u16(Q), u16(K), u16(V), perm.numpy(), vsmooth, vbits=4)
    for key in KEYS:
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)
    if vsmooth:
        np.testing.assert_array_equal(got["mu"], want["mu"], err_msg="mu")


@pytest.mark.parametrize("N,d", [(1000, 128), (700, 64), (1300, 128)])
def test_v4_attention_matches_oracle(oracle_mod, N, d):
    w = inputs.WORKLOADS["tiny"]
    Q, K, V = inputs.make_qkv(w, "cpu", H=2, N=N, d=d, seed=9)
    Qd, Kd, Vd = Q.to(DEV), K.to(DEV), V.to(DEV)
    perm = vc.vc_cluster(Vd, 8, 2)[2]
    qz = vc.vc_quantize(Qd, Kd, Vd, perm, 1, vbits=4)
    O = vc.vc_attn_fwd(qz, vc.shape_of(Qd), expcast=1, vsmooth=1)
    torch.cuda.synchronize()
    want = oracle_mod.quantize(u16(Q), u16(K), u16(V), perm.cpu().numpy(), 1, vbits=4)
    ref = oracle_mod.attn(want, N, expcast=1, vsmooth=1)
    oracle_mod.check_o(O.float().cpu().numpy().transpose(0, 2, 1, 3), ref, "4-bit V N%d d%d" % (N, d))


def test_v4_fidelity_reported(oracle_mod, capsys):
    """Against unquantized fp64 attention: the 4-bit residual costs accuracy
    (reported, loosely bounded), the 8-bit one beside it."""
    w = inputs.WORKLOADS["tiny"]
    Q, K, V = inputs.make_qkv(w, "cpu")
    ref = oracle_mod.attn_ref(u16(Q), u16(K), u16(V))
    Qd, Kd, Vd = Q.to(DEV), K.to(DEV), V.to(DEV)
    perm = vc.vc_cluster(Vd, w.k, w.iters)[2]
    err = {}
    for vbits in (8, 4):
        qz = vc.vc_quantize(Qd, Kd, Vd, perm, 1, vbits=vbits)
        O = vc.vc_attn_fwd(qz, vc.shape_of(Qd))
        torch.cuda.synchronize()
        got = O.float().cpu().numpy().transpose(0, 2, 1, 3)
        err[vbits] = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    with capsys.disabled():
        print("\nfidelity rel-L2 vs fp64, V residual 8 / 4 bits:", {k: round(v, 5) for k, v in err.items()})
    assert err[8] < err[4] < 0.25


def test_v4_wan_size_sampled(oracle_mod):
    w = inputs.WORKLOADS["wan"]
    Q, K, V = inputs.make_qkv(w, DEV)
    perm = vc.vc_cluster(V, w.k, w.iters)[2]
    qz = vc.vc_quantize(Q, K, V, perm, 1, vbits=4)
    O = vc.vc_attn_fwd(qz, vc.shape_of(Q))
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    for h in (0, 39):
        Qh, Kh, Vh = (u16(t[:, :, h:h + 1]) for t in (Q, K, V))
        want = oracle_mod.quantize(Qh, Kh, Vh, perm[:, h:h + 1].cpu().numpy(), 1, vbits=4)
        for key in KEYS:
            np.testing.assert_array_equal(qz[key][:, h:h + 1].cpu().numpy(), want[key], err_msg=key)
        rows = sampled_rows(w.N, rng, 24)
        ref = oracle_mod.attn(want, w.N, rows=rows)[0, 0]
        oracle_mod.check_o(O[0, rows, h].float().cpu().numpy(), ref, "4-bit V wan head %d" % h)
