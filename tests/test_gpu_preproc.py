"""GPU parity of the fused preprocessing (rotary transform + Hadamard rotation
of Q and K inside the quantizer) and of its unfused chain, against the oracle.

Bars: codes, scales and means bit-exact against the oracle given the same
permutation and rotary table; the unfused chain bit-identical to the fused
kernels; O after the preprocessing within the oracle's bars (2e-3 relative L2 over
the tensor, and row by row and element by element: oracle.check_o).
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

CASES = [
    dict(N=1000, d=64, H=2, B=1, seed=1),
    dict(N=2000, d=128, H=3, B=1, seed=2),
    dict(N=129, d=128, H=1, B=2, seed=3),
    dict(N=1, d=64, H=2, B=1, seed=4),
]


def _inputs(case):
    w = inputs.WORKLOADS["medium"]
    Q, K, V = inputs.make_qkv(w, "cpu", B=case["B"], H=case["H"], N=case["N"], d=case["d"], seed=case["seed"])
    B, N, H, _ = Q.shape
    g = torch.Generator().manual_seed(case["seed"])
    perm = torch.stack([torch.stack([torch.randperm(N, generator=g) for _ in range(H)]) for _ in range(B)])
    return Q, K, V, perm.to(torch.int32), inputs.rope_table(N, case["d"])


def _np(qz, vsmooth):
    out = {k: qz[k].cpu().numpy() for k in KEYS}
    if vsmooth:
        out["mu"] = qz["mu"].cpu().numpy().view(np.uint16)
    return out


def _assert_same(got, want, vsmooth, tag):
    for key in KEYS:
        np.testing.assert_array_equal(got[key], want[key], err_msg="%s %s" % (tag, key))
    if vsmooth:
        np.testing.assert_array_equal(got["mu"], want["mu"], err_msg="%s mu" % tag)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "N%d_d%d_H%d_B%d" % (c["N"], c["d"], c["H"], c["B"]))
@pytest.mark.parametrize("use_rope,hadamard", [(True, 1), (True, 0), (False, 1)])
@pytest.mark.parametrize("vsmooth", [0, 1])
def test_preproc_bitexact(oracle_mod, case, use_rope, hadamard, vsmooth):
    Q, K, V, perm, rope = _inputs(case)
    rope_np = rope if use_rope else None
    rope_d = torch.from_numpy(rope).to(DEV) if use_rope else None
    args = (Q.to(DEV), K.to(DEV), V.to(DEV), perm.to(DEV), vsmooth)
    fused = _np(vc.vc_quantize_ex(*args, rope=rope_d, hadamard=hadamard), vsmooth)
    staged = _np(vc.vc_quantize_staged(*args, rope=rope_d, hadamard=hadamard), vsmooth)
    want = oracle_mod.quantize(u16(Q), u16(K), u16(V), perm.numpy(), vsmooth, rope=rope_np, hadamard=hadamard)
    _assert_same(fused, want, vsmooth, "fused")
    _assert_same(staged, want, vsmooth, "staged")


def test_no_preproc_is_vc_quantize():
    Q, K, V, perm, _ = _inputs(CASES[1])
    args = (Q.to(DEV), K.to(DEV), V.to(DEV), perm.to(DEV), 1)
    a = _np(vc.vc_quantize(*args), 1)
    b = _np(vc.vc_quantize_ex(*args, rope=None, hadamard=0), 1)
    c = _np(vc.vc_quantize_staged(*args, rope=None, hadamard=0), 1)
    _assert_same(b, a, 1, "ex")
    _assert_same(c, a, 1, "staged")


@pytest.mark.parametrize("expcast", [0, 1])
def test_attention_after_preproc(oracle_mod, expcast):
    case = dict(N=1500, d=128, H=2, B=1, seed=7)
    Q, K, V, perm, rope = _inputs(case)
    qz = vc.vc_quantize_ex(Q.to(DEV), K.to(DEV), V.to(DEV), perm.to(DEV), 1,
                           rope=torch.from_numpy(rope).to(DEV), hadamard=1)
    O = vc.vc_attn_fwd(qz, vc.shape_of(Q.to(DEV)), expcast=expcast, vsmooth=1)
    torch.cuda.synchronize()
    want = oracle_mod.quantize(u16(Q), u16(K), u16(V), perm.numpy(), 1, rope=rope, hadamard=1)
    ref = oracle_mod.attn(want, case["N"], expcast=expcast, vsmooth=1)
    got = O.float().cpu().numpy().transpose(0, 2, 1, 3)
    oracle_mod.check_o(got, ref, "after preprocessing, expcast %d" % expcast, exp_bytes=expcast != 1)


def test_wan_size_preproc(oracle_mod):
    """Full Wan2.2 shape with the 21 x 45 x 80 rotary grid: fused and unfused
    bit-identical on the device, oracle bit-exact on two heads, O sampled."""
    w = inputs.WORKLOADS["wan"]
    Q, K, V = inputs.make_qkv(w, DEV)
    rope = inputs.rope_table(w.N, w.d, inputs.WAN_GRID)
    rope_d = torch.from_numpy(rope).to(DEV)
    perm = vc.vc_cluster(V, w.k, w.iters)[2]
    fused = vc.vc_quantize_ex(Q, K, V, perm, 1, rope=rope_d, hadamard=1)
    staged = vc.vc_quantize_staged(Q, K, V, perm, 1, rope=rope_d, hadamard=1)
    for key in KEYS + ("mu",):
        assert torch.equal(fused[key], staged[key]), key
    O = vc.vc_attn_fwd(fused, vc.shape_of(Q), expcast=1, vsmooth=1)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    N = w.N
    for h in (0, 39):
        Qh, Kh, Vh = (u16(t[:, :, h:h + 1]) for t in (Q, K, V))
        want = oracle_mod.quantize(Qh, Kh, Vh, perm[:, h:h + 1].cpu().numpy(), 1, rope=rope, hadamard=1)
        got = {k: fused[k][:, h:h + 1] for k in KEYS + ("mu",)}
        _assert_same(_np(got, 1), want, 1, "head %d" % h)
        rows = sampled_rows(N, rng, 24)
        ref = oracle_mod.attn(want, N, rows=rows)[0, 0]
        o = O[0, rows, h].float().cpu().numpy()
        oracle_mod.check_o(o, ref, "wan preprocessing head %d" % h)


@pytest.mark.parametrize("d", [64, 128])
def test_preproc_strided_batched(oracle_mod, d):
    """Q/K/V as views into one [B, N, H, 3, d] buffer (strided heads), B = 2,
    with a permutation: fused and unfused chains against the oracle."""
    w = inputs.WORKLOADS["medium"]
    B, N, H = 2, 900, 3
    Q, K, V = inputs.make_qkv(w, "cpu", B=B, H=H, N=N, d=d, seed=23)
    packed = torch.stack([Q, K, V], dim=3).to(DEV)
    Qv, Kv, Vv = packed[:, :, :, 0], packed[:, :, :, 1], packed[:, :, :, 2]
    g = torch.Generator().manual_seed(3)
    perm = torch.stack([torch.stack([torch.randperm(N, generator=g) for _ in range(H)]) for _ in range(B)])
    perm = perm.to(torch.int32)
    rope = inputs.rope_table(N, d)
    rope_d = torch.from_numpy(rope).to(DEV)
    want = oracle_mod.quantize(u16(Q), u16(K), u16(V), perm.numpy(), 1, rope=rope, hadamard=1)
    for fn in (vc.vc_quantize_ex, vc.vc_quantize_staged):
        got = _np(fn(Qv, Kv, Vv, perm.to(DEV), 1, rope=rope_d, hadamard=1), 1)
        _assert_same(got, want, 1, fn.__name__)
