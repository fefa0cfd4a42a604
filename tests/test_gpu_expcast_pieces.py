"""GPU parity of the range-adaptive ExpCast bytes (expcast = 3).

Bars: the probability bytes the kernel feeds to its P V product equal, bit
for bit, the oracle's range-adaptive bytes computed from the kernel's own
fp32 scores (the debug dump), on a ragged last tile of the full Wan2.2 shape;
O on sampled rows of that shape within the oracle's O bars; fidelity against
unquantized fp64 attention reported beside ExpCast and exp-then-cast (the
smaller-size byte and O parity cases live with the other attention tests).
"""
import numpy as np
import pytest
import torch

from bit_fp8_attention_means_gb300 import inputs, vc
from rowsample import sampled_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
u16 = inputs.to_u16
KEYS = ("Q8", "sq", "K8", "sk", "V8T", "sv", "mu")


def _head_np(qz, h):
    out = {k: qz[k][:, h:h + 1].cpu().numpy() for k in KEYS}
    out["mu"] = out["mu"].view(np.uint16)
    return out


def test_wan_size_bytes_and_rows(oracle_mod):
    w = inputs.WORKLOADS["wan"]
    Q, K, V = inputs.make_qkv(w, DEV)
    perm = vc.vc_cluster(V, w.k, w.iters)[2]
    qz = vc.vc_quantize(Q, K, V, perm, 1)
    shape = vc.shape_of(Q)
    O = vc.vc_attn_fwd(qz, shape, expcast=3, vsmooth=1)
    nblk = vc.nblk_of(w.N)
    h, qtile = 39, nblk - 1
    _, S, P = vc.vc_attn_fwd(qz, shape, expcast=3, vsmooth=1, debug=(h, qtile))
    torch.cuda.synchronize()
    one = _head_np(qz, h)
    rows = np.arange(qtile * 128, w.N, dtype=np.int32)
    acc = S.cpu().numpy()[: rows.size][None, None]
    _, codes = oracle_mod.attn(one, w.N, expcast=3, rows=rows, acc_in=acc, want_codes=True)
    np.testing.assert_array_equal(P.cpu().numpy()[: rows.size], codes[0, 0])
    rng = np.random.default_rng(8)
    for hh in (0, 39):
        r = sampled_rows(w.N, rng, 24)
        ref = oracle_mod.attn(_head_np(qz, hh), w.N, expcast=3, rows=r)[0, 0]
        oracle_mod.check_o(O[0, r, hh].float().cpu().numpy(), ref, "adaptive beta wan head %d" % hh)


def test_fidelity_beside_expcast(oracle_mod, capsys):
    """Against unquantized fp64 attention: the adaptive bytes are not worse than
    ExpCast's single beta (reported with exp-then-cast beside them)."""
    w = inputs.WORKLOADS["tiny"]
    Q, K, V = inputs.make_qkv(w, "cpu")
    ref = oracle_mod.attn_ref(u16(Q), u16(K), u16(V))
    Qd, Kd, Vd = Q.to(DEV), K.to(DEV), V.to(DEV)
    perm = vc.vc_cluster(Vd, w.k, w.iters)[2]
    qz = vc.vc_quantize(Qd, Kd, Vd, perm, 1)
    err = {}
    for ec in (0, 1, 3):
        O = vc.vc_attn_fwd(qz, vc.shape_of(Qd), expcast=ec)
        torch.cuda.synchronize()
        got = O.float().cpu().numpy().transpose(0, 2, 1, 3)
        err[ec] = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    with capsys.disabled():
        print("\nfidelity rel-L2 vs fp64 by expcast (0 exact, 1 ExpCast, 3 adaptive):",
              {k: round(v, 6) for k, v in err.items()})
    assert err[3] <= err[1] * 1.01 and err[3] < 0.05
