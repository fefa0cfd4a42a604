"""Parity on the sequence-sweep shapes (B=1, H=24, d=128, N from 4,096 to 131,072).

The whole path runs at the sweep's full sizes; the oracle checks the first
and the last head: the quantizer bit-exactly and O on sampled query rows
(first, last and second-to-last tiles included) row by row, with ExpCast and V-Smooth on at every N and in
all four modes at the smallest N.
"""
import numpy as np
import pytest
import torch

from bit_fp8_attention_means_gb300 import inputs, vc
from rowsample import sampled_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
u16 = inputs.to_u16


def _check(oracle_mod, w, Q, K, V, perm, expcast, vsmooth, heads, rng):
    qz = vc.vc_quantize(Q, K, V, perm if vsmooth else None, vsmooth)
    O = vc.vc_attn_fwd(qz, vc.shape_of(Q), expcast=expcast, vsmooth=vsmooth)
    torch.cuda.synchronize()
    N = w.N
    for h in heads:
        Qh, Kh, Vh = (u16(t[:, :, h:h + 1]) for t in (Q, K, V))
        ph = perm[:, h:h + 1].cpu().numpy() if vsmooth else None
        want = oracle_mod.quantize(Qh, Kh, Vh, ph, vsmooth)
        for key in ("Q8", "sq", "K8", "sk", "V8T", "sv"):
            np.testing.assert_array_equal(qz[key][:, h:h + 1].cpu().numpy(), want[key], err_msg=key)
        if vsmooth:
            np.testing.assert_array_equal(qz["mu"][:, h:h + 1].cpu().numpy().view(np.uint16), want["mu"])
        rows = sampled_rows(N, rng, 24)
        ref = oracle_mod.attn(want, N, expcast=expcast, vsmooth=vsmooth, rows=rows)[0, 0]
        got = O[0, rows, h].float().cpu().numpy()
        oracle_mod.check_o(got, ref, "N %d head %d expcast %d vsmooth %d" % (N, h, expcast, vsmooth),
                           exp_bytes=expcast == 0)


@pytest.mark.parametrize("N", [4096, 16384, 32768, 65536, 131072])
def test_sweep_sizes_sampled(oracle_mod, N):
    w = inputs.sweep_workload(N)
    Q, K, V = inputs.make_qkv(w, DEV)
    perm = vc.vc_cluster(V, w.k, w.iters)[2]
    rng = np.random.default_rng(N)
    modes = [(1, 1), (0, 1), (1, 0), (0, 0), (3, 1)] if N == 4096 else [(1, 1)]
    for expcast, vsmooth in modes:
        _check(oracle_mod, w, Q, K, V, perm, expcast, vsmooth, (0, w.H - 1), rng)
