"""vc_quantize_static: the quantizer entry point that allocates nothing.

It exists for callers that cannot hand the library device memory: programs
embedding it inside a framework whose pool owns all device memory, or code
running where an allocation would synchronize the device or is not allowed.
Its scratch is a fixed array inside the library.  These tests call it through
the C ABI and require bit-identical results to vc_quantize (the tolerance the
other quantizer tests use for codes, scales and means), on two calls in a row
so that the second call proves the shared array is cleared between calls.
"""
import ctypes

import numpy as np
import pytest
import torch

from bit_fp8_attention_means_gb300 import inputs, vc

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
_vp = ctypes.c_void_p


def _entry():
    L = vc.lib()
    fn = L.vc_quantize_static
    fn.restype = ctypes.c_int
    fn.argtypes = [_vp, _vp, _vp, vc.VcShape, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    return fn


def _call_static(Q, K, V, perm, vsmooth, out=None):
    s = vc.shape_of(Q)
    if out is None:
        out = vc.alloc_quantized(s, Q.device, vsmooth)
    p = lambda t: None if t is None else _vp(t.data_ptr())
    rc = _entry()(p(Q), p(K), p(V), s, p(perm), vsmooth, p(out["Q8"]), p(out["sq"]), p(out["K8"]),
                  p(out["sk"]), p(out["V8T"]), p(out["sv"]), p(out["mu"]),
                  _vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, vc.STATUS.get(rc, rc)
    return out


def _same(a, b, vsmooth):
    keys = ["Q8", "sq", "K8", "sk", "V8T", "sv"] + (["mu"] if vsmooth else [])
    for k in keys:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("vsmooth", [1, 0])
def test_static_matches_workspace_version_twice(vsmooth):
    w = inputs.WORKLOADS["tiny"]
    # The first call's V is scaled by 100, so every channel maximum it leaves in
    # the shared array exceeds the second call's own: a second call that did
    # not clear the array would certainly get scales and codes wrong.
    for call, (N, d, H, seed, vmul) in enumerate([(1000, 128, 3, 41, 100.0), (777, 64, 2, 42, 1.0)]):
        Q, K, V = (t.to(DEV) for t in inputs.make_qkv(w, "cpu", H=H, N=N, d=d, seed=seed))
        V = (V.float() * vmul).to(torch.bfloat16)
        g = torch.Generator().manual_seed(seed)
        perm = torch.stack([torch.randperm(N, generator=g) for _ in range(H)])[None].to(torch.int32).to(DEV)
        want = vc.vc_quantize(Q, K, V, perm, vsmooth)
        got = _call_static(Q, K, V, perm, vsmooth)
        torch.cuda.synchronize()
        _same(got, want, vsmooth)
        # the largest residual of every channel lands on the top code, which a
        # stale (uncleared) maximum from the previous call would prevent
        assert int((got["V8T"] & 0x7F).amax(dim=3).min()) == 0x7E, call


def test_static_call_allocates_nothing():
    """Once warmed up, a call changes neither PyTorch's allocation count nor
    the device's free memory."""
    w = inputs.WORKLOADS["tiny"]
    Q, K, V = (t.to(DEV) for t in inputs.make_qkv(w, "cpu", H=2, N=900, d=128, seed=43))
    out = vc.alloc_quantized(vc.shape_of(Q), Q.device, 1)
    _call_static(Q, K, V, None, 1, out=out)
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    _call_static(Q, K, V, None, 1, out=out)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    want = vc.vc_quantize(Q, K, V, None, 1)
    torch.cuda.synchronize()
    _same(out, want, 1)


def test_static_rejects_shapes_beyond_its_array():
    s = vc.VcShape(1, 513, 256, 128, 256 * 513 * 128, 513 * 128, 128)   # B*H*d = 65664 > 65536
    fake = _vp(0x10000)
    rc = _entry()(fake, fake, fake, s, None, 1, fake, fake, fake, fake, fake, fake, fake, None)
    assert rc == 3   # VC_ERR_WORKSPACE, nothing launched
