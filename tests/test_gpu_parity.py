"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Bars: quantizer codes/scales/means bit-exact given the same permutation;
ExpCast bytes bit-exact when both sides see the same fp32 scores; O within
2e-3 relative L2 of the oracle over the compared tensor, and row by row and
element by element within the bars of oracle.check_o (O is bf16: its rounding
alone is ~1.1e-3 relative, at most 2^-8 of an element);
grouping checked by invariants (labels are nearest centroids, pi is the stable
argsort of the labels, centroids are the means of their members).
"""
import numpy as np
import pytest
import torch

import oracle
from bit_fp8_attention_means_gb300 import inputs, vc
from rowsample import sampled_rows

pytestmark = pytest.mark.gpu

O_TOL = 2e-3
DEV = "cuda:0"
u16 = inputs.to_u16


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _gpu_quant_np(qz):
    out = {k: v.cpu().numpy() for k, v in qz.items() if v is not None and k != "mu"}
    out["mu"] = qz["mu"].cpu().numpy().view(np.uint16) if qz.get("mu") is not None else None
    return out


def _case(N, d, H, seed, B=1, wname="tiny"):
    w = inputs.WORKLOADS[wname]
    return inputs.make_qkv(w, "cpu", B=B, H=H, N=N, d=d, seed=seed)


# ---------------------------------------------------------------- E4M3 conversion

def test_device_e4m3_conversion_exhaustive(oracle_mod):
    """The hardware cvt.rn.satfinite.e4m3 equals the oracle encoder on every non-NaN fp32."""
    chunk = 1 << 28
    for c in range(16):
        bits = torch.arange(c * chunk, (c + 1) * chunk, dtype=torch.int64, device=DEV).to(torch.int32)
        x = bits.view(torch.float32)
        got = vc.vc_debug_e4m3_encode(x).cpu().numpy()
        xh = x.cpu().numpy()
        want = oracle_mod.e4m3_encode(xh)
        ok = (got == want) | np.isnan(xh)
        bad = np.nonzero(~ok)[0]
        assert bad.size == 0, (c, xh[bad[:4]], got[bad[:4]], want[bad[:4]])


# ---------------------------------------------------------------- quantizer

QUANT_CASES = [
    dict(N=1024, d=64, H=2, seed=1),
    dict(N=1000, d=128, H=3, seed=2),
    dict(N=129, d=128, H=1, seed=3),
    dict(N=1, d=64, H=2, seed=4),
    dict(N=300, d=128, H=2, seed=5, B=2),
]


@pytest.mark.parametrize("case", QUANT_CASES, ids=lambda c: "N%d_d%d_H%d" % (c["N"], c["d"], c["H"]))
@pytest.mark.parametrize("vsmooth", [0, 1])
@pytest.mark.parametrize("use_perm", [False, True])
def test_quantize_bitexact(oracle_mod, case, vsmooth, use_perm):
    Q, K, V = _case(**case)
    B, N, H, d = Q.shape
    perm = None
    if use_perm:
        g = torch.Generator().manual_seed(case["seed"])
        perm = torch.stack([torch.stack([torch.randperm(N, generator=g) for _ in range(H)]) for _ in range(B)])
        perm = perm.to(torch.int32)
    qz = vc.vc_quantize(Q.to(DEV), K.to(DEV), V.to(DEV), None if perm is None else perm.to(DEV), vsmooth)
    got = _gpu_quant_np(qz)
    want = oracle_mod.quantize(u16(Q), u16(K), u16(V), None if perm is None else perm.numpy(), vsmooth)
    for key in ("Q8", "sq", "K8", "sk", "V8T", "sv"):
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)
    if vsmooth:
        np.testing.assert_array_equal(got["mu"], want["mu"], err_msg="mu")


@pytest.mark.parametrize("N,d", [(300, 128), (1000, 64)])
def test_quantize_poisoned_outputs(oracle_mod, N, d):
    """Every output buffer pre-filled with 0xFF bytes: the whole of each array,
    padding rows and columns included, comes out equal to the oracle's."""
    Q, K, V = _case(N=N, d=d, H=2, seed=31)
    Qd, Kd, Vd = Q.to(DEV), K.to(DEV), V.to(DEV)
    out = vc.alloc_quantized(vc.shape_of(Qd), Qd.device, 1)
    for t in out.values():
        t.view(torch.uint8).fill_(0xFF)
    g = torch.Generator().manual_seed(3)
    perm = torch.stack([torch.randperm(N, generator=g) for _ in range(2)])[None].to(torch.int32)
    qz = vc.vc_quantize(Qd, Kd, Vd, perm.to(DEV), 1, out=out)
    got = _gpu_quant_np(qz)
    want = oracle_mod.quantize(u16(Q), u16(K), u16(V), perm.numpy(), 1)
    for key in ("Q8", "sq", "K8", "sk", "V8T", "sv", "mu"):
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)


def test_quantize_strided_input(oracle_mod):
    """Q/K/V views into a larger [B, N, H, 3, d] buffer (strided heads)."""
    Q, K, V = _case(N=700, d=128, H=2, seed=7)
    packed = torch.stack([Q, K, V], dim=3).to(DEV)          # [B,N,H,3,d]
    Qv, Kv, Vv = packed[:, :, :, 0], packed[:, :, :, 1], packed[:, :, :, 2]
    qz = vc.vc_quantize(Qv, Kv, Vv, None, 1)
    want = oracle_mod.quantize(u16(Q), u16(K), u16(V), None, 1)
    got = _gpu_quant_np(qz)
    for key in ("Q8", "sq", "K8", "sk", "V8T", "sv", "mu"):
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)


# ---------------------------------------------------------------- grouping

# k <= 256 takes the tensor-core assignment (k = 250 pads the centroid rows to
# 256), k > 256 the fp32 CUDA-core one
@pytest.mark.parametrize("N,d,H,k,iters", [(1024, 64, 2, 8, 5), (5000, 128, 2, 64, 3), (700, 128, 1, 1, 2),
                                           (4096 * 2 + 77, 128, 1, 37, 2), (2048, 64, 1, 250, 2),
                                           (4000, 128, 1, 256, 2), (3000, 128, 1, 257, 2), (2000, 64, 1, 1000, 1),
                                           (2100, 64, 1, 1024, 1)])
def test_cluster_invariants(oracle_mod, N, d, H, k, iters):
    Q, K, V = _case(N=N, d=d, H=H, seed=11)
    Vd = V.to(DEV)
    c_prev, _, _ = vc.vc_cluster(Vd, k, iters)
    cent, lab, perm = vc.vc_cluster(Vd, k, 1, warm_start=True, centroids=c_prev.clone())
    lab, perm, cent, c_prev = (t.cpu().numpy() for t in (lab, perm, cent, c_prev))
    v = oracle_mod.bf16_to_f32(u16(V)).astype(np.float64).transpose(0, 2, 1, 3)
    for b in range(v.shape[0]):
        for h in range(v.shape[1]):
            np.testing.assert_array_equal(perm[b, h], np.argsort(lab[b, h], kind="stable"))
            cp = c_prev[b, h].astype(np.float64)
            d2 = (v[b, h] ** 2).sum(-1)[:, None] + (cp ** 2).sum(-1)[None] - 2.0 * v[b, h] @ cp.T
            best = d2.min(axis=1)
            chosen = d2[np.arange(N), lab[b, h]]
            # |c|^2 - 2 v.c: the two-part bf16 centroid split errs by <= 2^-17 (|v|^2 + |c|^2)
            # and fp32 accumulation by ~d 2^-25 (|v|^2 + |c|^2); both fit 4 d 2^-24 (|v|^2 + |c|^2)
            scale = (v[b, h] ** 2).sum(-1) + (c_prev[b, h].astype(np.float64) ** 2).sum(-1)[lab[b, h]]
            assert np.all(chosen - best <= 4 * d * 2.0 ** -24 * scale + 1e-6)
            for i in range(k):
                mem = lab[b, h] == i
                if mem.any():
                    np.testing.assert_allclose(cent[b, h, i], v[b, h][mem].mean(0), rtol=1e-5, atol=1e-5)
                else:
                    np.testing.assert_array_equal(cent[b, h, i], c_prev[b, h, i])


def test_cluster_cold_start(oracle_mod):
    """iters=1 from the cold start: labels are nearest to tokens floor(i N / k)."""
    Q, K, V = _case(N=900, d=64, H=1, seed=13)
    k = 9
    _, lab, _ = vc.vc_cluster(V.to(DEV), k, 1)
    v = oracle_mod.bf16_to_f32(u16(V)).astype(np.float64)[0, :, 0]
    init = v[[(i * 900) // k for i in range(k)]]
    d2 = ((v[:, None] - init[None]) ** 2).sum(-1)
    chosen = d2[np.arange(900), lab.cpu().numpy()[0, 0]]
    assert np.all(chosen <= d2.min(1) * (1 + 1e-5) + 1e-6)


# ---------------------------------------------------------------- attention

def _pipeline(Q, K, V, k, iters, vsmooth, expcast, debug=None, use_cluster=True, margin=None):
    Qd, Kd, Vd = Q.to(DEV), K.to(DEV), V.to(DEV)
    perm = vc.vc_cluster(Vd, k, iters)[2] if use_cluster else None
    qz = vc.vc_quantize(Qd, Kd, Vd, perm, vsmooth)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = vc.vc_attn_fwd(qz, vc.shape_of(Qd), expcast=expcast, vsmooth=vsmooth, debug=debug, exact_margin=margin,
                         dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a device wait ran out (status %d)" % int(status.item())
    return perm, qz, res


def _slice_bh(qz_np, b, h):
    return {k: (v[b:b + 1, h:h + 1] if v is not None else None) for k, v in qz_np.items()}


@pytest.mark.parametrize("expcast", [1, 0, 3])
@pytest.mark.parametrize("N,d,qtile", [(1024, 64, 3), (1000, 128, 7), (300, 128, 0), (300, 128, 2)])
def test_expcast_bytes_bitexact(oracle_mod, expcast, N, d, qtile):
    Q, K, V = _case(N=N, d=d, H=2, seed=17)
    bh = 1
    _, qz, (O, S, P) = _pipeline(Q, K, V, 8, 2, 1, expcast, debug=(bh, qtile))
    qn = _gpu_quant_np(qz)
    one = _slice_bh(qn, 0, bh)
    rows = np.arange(qtile * 128, min(N, qtile * 128 + 128), dtype=np.int32)
    acc = S.cpu().numpy()[: rows.size][None, None]
    _, codes = oracle_mod.attn(one, N, expcast=expcast, vsmooth=1, rows=rows, acc_in=acc, want_codes=True)
    got = P.cpu().numpy()[: rows.size]
    want = codes[0, 0]
    if expcast:
        np.testing.assert_array_equal(got, want)
    else:
        # exp-then-cast: the GPU's exp2 is not correctly rounded; codes agree up to one step
        diff = np.abs(got.astype(int) - want.astype(int))
        assert diff.max() <= 1 and np.mean(diff == 0) > 0.999
    assert np.all(got[:, N:] == 0)


# tile counts 8, 8, 2, 1, 20 and two odd counts with ragged tails (11 tiles)
ATTN_CASES = [dict(N=1024, d=64, H=2, k=8), dict(N=1000, d=128, H=2, k=16), dict(N=129, d=128, H=1, k=4),
              dict(N=1, d=64, H=1, k=1), dict(N=2500, d=128, H=1, k=32), dict(N=1300, d=64, H=1, k=8),
              dict(N=1400, d=128, H=2, k=16)]


@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: "N%d_d%d" % (c["N"], c["d"]))
@pytest.mark.parametrize("expcast,vsmooth", [(1, 1), (1, 0), (0, 1), (0, 0), (3, 1), (3, 0)])
def test_attention_matches_oracle(oracle_mod, case, expcast, vsmooth):
    Q, K, V = _case(N=case["N"], d=case["d"], H=case["H"], seed=19)
    N = case["N"]
    _, qz, O = _pipeline(Q, K, V, case["k"], 2, vsmooth, expcast, use_cluster=vsmooth == 1)
    qn = _gpu_quant_np(qz)
    if not vsmooth:
        qn["mu"] = np.zeros(qn["sq"].shape + (case["d"],), np.uint16)
    ref = oracle_mod.attn(qn, N, expcast=expcast, vsmooth=vsmooth)
    got = O.float().cpu().numpy().transpose(0, 2, 1, 3)
    oracle_mod.check_o(got, ref, "N%d d%d expcast %d vsmooth %d" % (N, case["d"], expcast, vsmooth),
                        exp_bytes=expcast == 0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("expcast", [1, 0, 3])
def test_attention_batched_with_scale(oracle_mod, d, expcast):
    """B = 2 and a softmax scale other than 1/sqrt(d): every (b, h) against the oracle."""
    N, scale = 700, 0.05
    Q, K, V = _case(N=N, d=d, H=2, seed=29, B=2)
    Qd, Kd, Vd = Q.to(DEV), K.to(DEV), V.to(DEV)
    perm = vc.vc_cluster(Vd, 8, 2)[2]
    qz = vc.vc_quantize(Qd, Kd, Vd, perm, 1)
    O = vc.vc_attn_fwd(qz, vc.shape_of(Qd), softmax_scale=scale, expcast=expcast, vsmooth=1)
    torch.cuda.synchronize()
    ref = oracle_mod.attn(_gpu_quant_np(qz), N, softmax_scale=scale, expcast=expcast, vsmooth=1)
    got = O.float().cpu().numpy().transpose(0, 2, 1, 3)
    for b in range(2):
        for h in range(2):
            oracle_mod.check_o(got[b, h], ref[b, h], "b%d h%d" % (b, h), exp_bytes=expcast == 0)


def test_output_rows_beyond_n_untouched(oracle_mod):
    Q, K, V = _case(N=200, d=128, H=2, seed=23)
    Qd, Kd, Vd = Q.to(DEV), K.to(DEV), V.to(DEV)
    qz = vc.vc_quantize(Qd, Kd, Vd, None, 1)
    big = torch.full((1, 256, 2, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    O = big[:, :200]
    vc.vc_attn_fwd(qz, vc.shape_of(Qd), O=O)
    torch.cuda.synchronize()
    assert torch.all(big[:, 200:] == 7.0)
    assert torch.isfinite(O.float()).all()


def test_medium_sampled_rows(oracle_mod):
    w = inputs.WORKLOADS["medium"]
    Q, K, V = inputs.make_qkv(w, "cpu")
    _, qz, O = _pipeline(Q, K, V, w.k, w.iters, 1, 1)
    qn = _gpu_quant_np(qz)
    rows = sampled_rows(w.N, np.random.default_rng(5), 80)
    ref = oracle_mod.attn(qn, w.N, rows=rows)
    got = O.float().cpu().numpy().transpose(0, 2, 1, 3)[:, :, rows]
    oracle_mod.check_o(got, ref, "medium")


def test_fidelity_vs_fp64_reported(oracle_mod, capsys):
    """Fidelity against unquantized fp64 attention, V-Smooth on and off (reported, loosely bounded)."""
    w = inputs.WORKLOADS["tiny"]
    Q, K, V = inputs.make_qkv(w, "cpu")
    ref = oracle_mod.attn_ref(u16(Q), u16(K), u16(V))
    out = {}
    for vs in (0, 1):
        for ec in (0, 1):
            _, _, O = _pipeline(Q, K, V, w.k, w.iters, vs, ec, use_cluster=vs == 1)
            out[(vs, ec)] = _rel(O.float().cpu().numpy().transpose(0, 2, 1, 3), ref)
    with capsys.disabled():
        print("\nfidelity rel-L2 vs fp64 (vsmooth, expcast):", {k: round(v, 5) for k, v in out.items()})
    assert all(v < 0.05 for v in out.values())


# ---------------------------------------------------------------- failure detection

def test_bounded_wait_reports_timeout():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    vc.vc_debug_wait_timeout(status, 20000)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    # the context is still usable
    Q, K, V = _case(N=256, d=64, H=1, seed=29)
    qz = vc.vc_quantize(Q.to(DEV), K.to(DEV), V.to(DEV), None, 1)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    O = vc.vc_attn_fwd(qz, vc.shape_of(Q.to(DEV)), dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0 and torch.isfinite(O.float()).all()


def test_attention_from_two_host_threads(oracle_mod):
    """Two host threads launch vc_attn_fwd at the same time on one device, each
    on its own stream and with its own output (the first launch of a kernel in
    a context sets its shared-memory limit under the library's lock): every
    result equals the single-threaded one bit for bit, and that one matches the
    oracle."""
    import threading
    Q, K, V = _case(N=1000, d=128, H=2, seed=37)
    _, qz, O_ref = _pipeline(Q, K, V, 8, 2, 1, 1)
    qn = _gpu_quant_np(qz)
    oracle_mod.check_o(O_ref.float().cpu().numpy().transpose(0, 2, 1, 3), oracle_mod.attn(qn, 1000), "reference")
    shape = vc.shape_of(Q.to(DEV))
    results, errors = {}, []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            outs = []
            with torch.cuda.stream(s):
                for _ in range(4):
                    outs.append(vc.vc_attn_fwd(qz, shape, expcast=1, vsmooth=1, stream=s))
            s.synchronize()
            results[i] = outs
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(2):
        for o in results[i]:
            assert torch.equal(o, O_ref)


@pytest.mark.parametrize("N,d,skip", [(256, 128, 1), (700, 64, 2)])
def test_attention_wait_timeout_and_recovery(oracle_mod, N, d, skip):
    """The attention kernel's own failure path: its K loader never delivers key
    tile `skip`, so the MMA warp's wait for it runs out (2 ms bound).  The
    kernel records VC_ERR_TIMEOUT, every warp stops waiting, the copies and
    products in flight drain, tensor memory is freed and the call returns; the
    next normal call on the same context matches the oracle."""
    Q, K, V = _case(N=N, d=d, H=1, seed=43)
    Qd = Q.to(DEV)
    qz = vc.vc_quantize(Qd, K.to(DEV), V.to(DEV), None, 1)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    vc.vc_debug_attn_timeout(qz, vc.shape_of(Qd), status, skip, 2000)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    O = vc.vc_attn_fwd(qz, vc.shape_of(Qd), dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    ref = oracle_mod.attn(_gpu_quant_np(qz), N)
    oracle_mod.check_o(O.float().cpu().numpy().transpose(0, 2, 1, 3), ref, "after a timed-out call")


def test_invalid_arguments_raise():
    Q, K, V = _case(N=256, d=64, H=1, seed=31)
    Qd = Q.to(DEV)
    qz = vc.vc_quantize(Qd, K.to(DEV), V.to(DEV), None, 1)
    with pytest.raises(vc.VcError):
        vc.vc_attn_fwd(qz, vc.shape_of(Qd), expcast=2)
    with pytest.raises(vc.VcError):
        vc.vc_cluster(V.to(DEV), 0, 1)
    bad = vc.shape_of(Qd)
    bad.d = 96
    with pytest.raises(vc.VcError):
        vc.vc_attn_fwd(qz, bad)


# ---------------------------------------------------------------- hybrid bytes

def _planted_peaky(N, d, H, seed):
    """Queries sharing one direction b; the keys of tiles 0 and 3 aligned with
    b, all other keys small noise: every row's running maximum is set in tile
    0, tile 3 stays within ~1 of it, the other tiles ~8 (log2) below."""
    g = torch.Generator().manual_seed(seed)
    b = torch.randn(d, generator=g)
    Q = torch.randn(1, N, H, d, generator=g) * 0.5 + b
    K = torch.randn(1, N, H, d, generator=g) * 0.3
    K[:, 0:128] += 0.5 * b
    K[:, 384:512] += 0.5 * b
    V = torch.randn(1, N, H, d, generator=g)
    return tuple(t.to(torch.bfloat16) for t in (Q, K, V))


@pytest.mark.parametrize("N,d,qtile", [(700, 64, 5), (1000, 128, 2), (1000, 128, 7)])
def test_hybrid_bytes_match_oracle(oracle_mod, N, d, qtile):
    """Hybrid mode: given the kernel's fp32 scores, the tiles the oracle writes
    with ExpCast match bit for bit, the exp-then-cast tiles within one code."""
    margin = 2.0
    Q, K, V = _planted_peaky(N, d, 2, seed=17)
    bh = 1
    _, qz, (O, S, P) = _pipeline(Q, K, V, 8, 2, 1, 2, debug=(bh, qtile), margin=margin, use_cluster=False)
    one = _slice_bh(_gpu_quant_np(qz), 0, bh)
    rows = np.arange(qtile * 128, min(N, qtile * 128 + 128), dtype=np.int32)
    acc = S.cpu().numpy()[: rows.size][None, None]
    kw = dict(vsmooth=1, rows=rows, acc_in=acc, want_codes=True)
    want_h = oracle_mod.attn(one, N, expcast=2, margin=margin, **kw)[1][0, 0]
    want_1 = oracle_mod.attn(one, N, expcast=1, **kw)[1][0, 0]
    want_0 = oracle_mod.attn(one, N, expcast=0, **kw)[1][0, 0]
    got = P.cpu().numpy()[: rows.size]
    diff = np.abs(got.astype(int) - want_h.astype(int))
    assert diff.max() <= 1 and np.mean(diff == 0) > 0.999
    nb = (N + 127) // 128
    kinds = {}
    for g in range(0, rows.size, 32):
        for j in range(nb):
            blk = np.s_[g:g + 32, 128 * j:128 * (j + 1)]
            if np.array_equal(want_h[blk], want_1[blk]) and not np.array_equal(want_1[blk], want_0[blk]):
                np.testing.assert_array_equal(got[blk], want_h[blk])   # an ExpCast tile: bit-exact
                kinds[j] = "expcast"
            elif not np.array_equal(want_h[blk], want_1[blk]):
                kinds[j] = "exact"
    # the planted pattern: tiles 0 and 3 exact, the rest ExpCast
    assert kinds.get(0) == "exact" and kinds.get(3) == "exact", kinds
    assert all(v == "expcast" for j, v in kinds.items() if j not in (0, 3)), kinds
    assert sum(v == "expcast" for v in kinds.values()) >= 2, kinds


@pytest.mark.parametrize("margin", [1.0, 3.0])
def test_hybrid_attention_matches_oracle(oracle_mod, margin):
    N, d = 1000, 128
    Q, K, V = _case(N=N, d=d, H=2, seed=19)
    _, qz, O = _pipeline(Q, K, V, 16, 2, 1, 2, margin=margin)
    qn = _gpu_quant_np(qz)
    ref = oracle_mod.attn(qn, N, expcast=2, margin=margin, vsmooth=1)
    got = O.float().cpu().numpy().transpose(0, 2, 1, 3)
    oracle_mod.check_o(got, ref, "hybrid margin %g" % margin, exp_bytes=True)
