"""CPU-side checks of the C ABI library: it loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from bit_fp8_attention_means_gb300 import build, vc
    build.build()
    return vc.lib()


def _declared():
    hdr = open(os.path.join(ROOT, "include", "vc.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(vc_[a-z0-9_]+)\s*\(", hdr)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code, name in [(0, b"VC_OK"), (1, b"VC_ERR_INVALID_ARG"), (2, b"VC_ERR_UNSUPPORTED"),
                       (3, b"VC_ERR_WORKSPACE"), (4, b"VC_ERR_CUDA"), (5, b"VC_ERR_TIMEOUT")]:
        assert L.vc_status_string(code) == name
    assert L.vc_version() >= 100


def _shape(B=1, H=2, N=1000, d=128):
    from bit_fp8_attention_means_gb300.vc import VcShape
    return VcShape(B, H, N, d, N * H * d, H * d, d)


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: validation fails first


def test_workspace_queries(L):
    s = _shape()
    assert L.vc_quantize_workspace(s) == 1 * 2 * 128 * 4
    assert L.vc_cluster_workspace(s, 64) > 0
    bad = _shape(d=96)
    assert L.vc_quantize_workspace(bad) == 0


def test_attn_argument_errors(L):
    s = _shape()
    args = [FAKE] * 7
    assert L.vc_attn_fwd(*args, _shape(d=96), 0.0, 1, 1, FAKE, None, None) == 2
    assert L.vc_attn_fwd(*args, s, 0.0, 2, 1, FAKE, None, None) == 1
    assert L.vc_attn_fwd(*args, s, 0.0, 4, 1, FAKE, None, None) == 1
    assert L.vc_attn_fwd(*args, s, 0.0, -1, 1, FAKE, None, None) == 1
    assert L.vc_attn_fwd_hybrid(*args, s, 0.0, float("nan"), 1, FAKE, None, None) == 1
    assert L.vc_attn_fwd_hybrid(*args, s, 0.0, 2.0, 3, FAKE, None, None) == 1
    assert L.vc_attn_fwd_hybrid(*args, _shape(d=96), 0.0, 2.0, 1, FAKE, None, None) == 2
    assert L.vc_attn_fwd(*args, s, 0.0, 1, 3, FAKE, None, None) == 1
    assert L.vc_attn_fwd(None, *args[1:], s, 0.0, 1, 1, FAKE, None, None) == 1
    assert L.vc_attn_fwd(*args, s, 0.0, 1, 1, None, None, None) == 1
    unaligned = ctypes.c_void_p(0x10008)
    assert L.vc_attn_fwd(unaligned, *args[1:], s, 0.0, 1, 1, FAKE, None, None) == 1
    neg = _shape()
    neg.N = 0
    assert L.vc_attn_fwd(*args, neg, 0.0, 1, 1, FAKE, None, None) == 1
    st = _shape()
    st.s_n = 100   # not a multiple of 8 elements
    assert L.vc_attn_fwd(*args, st, 0.0, 1, 1, FAKE, None, None) == 1
    big = _shape(N=(1 << 24) + 1)
    assert L.vc_attn_fwd(*args, big, 0.0, 1, 1, FAKE, None, None) == 2
    # O is written 16 bytes at a time
    assert L.vc_attn_fwd(*args, s, 0.0, 1, 1, unaligned, None, None) == 1
    # B*H*Npad rows must stay below 2^31 (32-bit TMA row coordinates)
    many = _shape(H=140000, N=16384)
    assert L.vc_attn_fwd(*args, many, 0.0, 1, 1, FAKE, None, None) == 2


def test_quantize_and_cluster_argument_errors(L):
    s = _shape()
    f = [FAKE] * 3
    outs = [FAKE] * 7
    ws_need = L.vc_quantize_workspace(s)
    assert L.vc_quantize(*f, s, None, 1, *outs, FAKE, ws_need - 1, None) == 3
    assert L.vc_quantize(*f, s, None, 1, *outs, None, ws_need, None) == 3
    assert L.vc_quantize(*f, s, None, 2, *outs, FAKE, ws_need, None) == 1
    assert L.vc_quantize(*f, s, None, 1, *outs[:6], None, FAKE, ws_need, None) == 1   # mu needed
    ws_odd = ctypes.c_void_p(0x10000 + 128)   # workspace must be 256-byte aligned
    assert L.vc_quantize(*f, s, None, 1, *outs, ws_odd, ws_need, None) == 3
    # the 4-bit residual entry point checks the same way
    assert L.vc_quantize_v4(*f, s, None, 1, *outs, FAKE, ws_need - 1, None) == 3
    assert L.vc_quantize_v4(*f, s, None, 2, *outs, FAKE, ws_need, None) == 1
    assert L.vc_quantize_v4(*f, s, None, 1, *outs[:6], None, FAKE, ws_need, None) == 1
    assert L.vc_quantize_v4(*f, _shape(d=96), None, 1, *outs, FAKE, ws_need, None) == 2
    cw = L.vc_cluster_workspace(s, 8)
    assert L.vc_cluster(FAKE, s, 0, 1, 0, FAKE, FAKE, FAKE, FAKE, cw, None, None) == 2
    assert L.vc_cluster(FAKE, s, 2000, 1, 0, FAKE, FAKE, FAKE, FAKE, cw, None, None) == 2
    assert L.vc_cluster(FAKE, s, 8, 0, 0, FAKE, FAKE, FAKE, FAKE, cw, None, None) == 1
    assert L.vc_cluster(FAKE, s, 8, 1, 0, FAKE, FAKE, FAKE, FAKE, cw - 1, None, None) == 3
    unaligned = ctypes.c_void_p(0x10008)
    assert L.vc_cluster(FAKE, s, 8, 1, 0, unaligned, FAKE, FAKE, FAKE, cw, None, None) == 1
    small = _shape(N=4)
    assert L.vc_cluster(FAKE, small, 8, 1, 0, FAKE, FAKE, FAKE, FAKE, 1 << 20, None, None) == 1
    assert L.vc_debug_wait_timeout(None, 10, None) == 1
    s3 = _shape(N=300)   # 3 key tiles
    args = [FAKE] * 7
    assert L.vc_debug_attn_timeout(*args, s3, 1, FAKE, None, None, 1, 1000) == 1     # dev_status required
    assert L.vc_debug_attn_timeout(*args, s3, 1, FAKE, FAKE, None, 3, 1000) == 1     # tile out of range
    assert L.vc_debug_attn_timeout(*args, s3, 1, FAKE, FAKE, None, 0, 0) == 1        # zero bound
    assert L.vc_debug_attn_timeout(*args, _shape(d=96), 1, FAKE, FAKE, None, 0, 10) == 2
    assert L.vc_cluster_ex(FAKE, s, 8, 1, 0, 2, FAKE, FAKE, FAKE, FAKE, cw, None, None) == 1   # block_fill flag
    assert L.vc_cluster_ex(FAKE, s, 8, 1, 0, 1, FAKE, FAKE, FAKE, FAKE, cw - 1, None, None) == 3


def test_quantize_ex_and_staged_argument_errors(L):
    s = _shape()
    f = [FAKE] * 3
    outs = [FAKE] * 7
    ws_need = L.vc_quantize_workspace(s)
    staged_need = L.vc_quantize_staged_workspace(s)
    elems = 1 * 1000 * 2 * 128
    assert staged_need >= ws_need + 14 * elems
    unaligned = ctypes.c_void_p(0x10008)
    for fn, need in ((L.vc_quantize_ex, ws_need), (L.vc_quantize_staged, staged_need)):
        assert fn(*f, s, None, 1, None, 2, *outs, FAKE, need, None) == 1        # hadamard flag
        assert fn(*f, s, None, 1, unaligned, 1, *outs, FAKE, need, None) == 1   # rope alignment
        assert fn(*f, s, None, 1, FAKE, 1, *outs, FAKE, need - 1, None) == 3
        assert fn(*f, _shape(d=96), None, 1, FAKE, 1, *outs, FAKE, need, None) == 2
    assert L.vc_quantize_staged_workspace(_shape(d=96)) == 0
