"""Thin ctypes binding over libvc_gb300.so (the C ABI in include/vc.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no
fallback: if the library has not been built, every call raises.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libvc_gb300.so")
BLOCK = 128

STATUS = {0: "VC_OK", 1: "VC_ERR_INVALID_ARG", 2: "VC_ERR_UNSUPPORTED", 3: "VC_ERR_WORKSPACE",
          4: "VC_ERR_CUDA", 5: "VC_ERR_TIMEOUT"}


class VcError(RuntimeError):
    def __init__(self, code, where):
        super().__init__("%s failed: %s" % (where, STATUS.get(code, code)))
        self.code = code


class VcShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32), ("d", ctypes.c_int32),
                ("s_b", ctypes.c_int64), ("s_n", ctypes.c_int64), ("s_h", ctypes.c_int64)]


_lib = None
_vp = ctypes.c_void_p


def lib():
    """Load the CUDA library; raises if it was not built (no silent fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libvc_gb300.so is missing: build it with `python -c \"import __graft_entry__ as g; "
                               "g.build()\"` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        L.vc_status_string.restype = ctypes.c_char_p
        L.vc_status_string.argtypes = [ctypes.c_int]
        L.vc_version.restype = ctypes.c_int
        L.vc_cluster_workspace.restype = ctypes.c_size_t
        L.vc_cluster_workspace.argtypes = [VcShape, ctypes.c_int]
        L.vc_cluster.restype = ctypes.c_int
        L.vc_cluster.argtypes = [_vp, VcShape, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp,
                                 ctypes.c_size_t, _vp, _vp]
        L.vc_cluster_ex.restype = ctypes.c_int
        L.vc_cluster_ex.argtypes = [_vp, VcShape, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                    _vp, _vp, ctypes.c_size_t, _vp, _vp]
        L.vc_quantize_workspace.restype = ctypes.c_size_t
        L.vc_quantize_workspace.argtypes = [VcShape]
        L.vc_quantize.restype = ctypes.c_int
        L.vc_quantize.argtypes = [_vp, _vp, _vp, VcShape, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                  _vp, ctypes.c_size_t, _vp]
        L.vc_quantize_ex.restype = ctypes.c_int
        L.vc_quantize_ex.argtypes = [_vp, _vp, _vp, VcShape, _vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp, _vp,
                                     _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
        L.vc_quantize_v4.restype = ctypes.c_int
        L.vc_quantize_v4.argtypes = L.vc_quantize.argtypes
        L.vc_quantize_staged_workspace.restype = ctypes.c_size_t
        L.vc_quantize_staged_workspace.argtypes = [VcShape]
        L.vc_quantize_staged.restype = ctypes.c_int
        L.vc_quantize_staged.argtypes = L.vc_quantize_ex.argtypes
        L.vc_attn_fwd.restype = ctypes.c_int
        L.vc_attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, VcShape, ctypes.c_float, ctypes.c_int,
                                  ctypes.c_int, _vp, _vp, _vp]
        L.vc_attn_fwd_hybrid.restype = ctypes.c_int
        L.vc_attn_fwd_hybrid.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, VcShape, ctypes.c_float,
                                         ctypes.c_float, ctypes.c_int, _vp, _vp, _vp]
        L.vc_attn_fwd_debug.restype = ctypes.c_int
        L.vc_attn_fwd_debug.argtypes = L.vc_attn_fwd.argtypes + [ctypes.c_int, ctypes.c_int, _vp, _vp,
                                                                 ctypes.c_float]
        L.vc_debug_e4m3_encode.restype = ctypes.c_int
        L.vc_debug_e4m3_encode.argtypes = [_vp, ctypes.c_int64, _vp, _vp]
        L.vc_debug_wait_timeout.restype = ctypes.c_int
        L.vc_debug_wait_timeout.argtypes = [_vp, ctypes.c_uint32, _vp]
        L.vc_debug_attn_timeout.restype = ctypes.c_int
        L.vc_debug_attn_timeout.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, VcShape, ctypes.c_int, _vp, _vp, _vp,
                                            ctypes.c_int, ctypes.c_uint32]
        _lib = L
    return _lib


def _check(code, where):
    if code != 0:
        raise VcError(code, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def nblk_of(N):
    return (N + BLOCK - 1) // BLOCK


def shape_of(X: torch.Tensor) -> VcShape:
    """[B, N, H, d] bf16 tensor with unit channel stride -> vc_shape."""
    if X.dim() != 4 or X.stride(3) != 1:
        raise ValueError("expected [B, N, H, d] with unit channel stride")
    B, N, H, d = X.shape
    return VcShape(B, H, N, d, X.stride(0), X.stride(1), X.stride(2))


def _empty(shape, dtype, device, fill=None):
    t = torch.empty(shape, dtype=dtype, device=device)
    if fill is not None:
        t.fill_(fill)
    return t


def quantize_workspace_bytes(shape: VcShape) -> int:
    return lib().vc_quantize_workspace(shape)


def cluster_workspace_bytes(shape: VcShape, k: int) -> int:
    return lib().vc_cluster_workspace(shape, k)


def _workspace(nbytes, device):
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def vc_cluster(V, k, iters, warm_start=False, centroids=None, labels=None, perm=None, workspace=None,
               dev_status=None, stream=None, block_fill=0):
    """Grouping step. Returns (centroids fp32 [B,H,k,d], labels int32 [B,H,N], perm int32 [B,H,N]).

    block_fill=1 calls vc_cluster_ex: perm keeps whole 128-token blocks per
    cluster and chains the clusters' leftovers by centroid distance."""
    s = shape_of(V)
    dev = V.device
    if centroids is None:
        if warm_start:
            raise ValueError("warm start needs centroids")
        centroids = _empty((s.B, s.H, k, s.d), torch.float32, dev)
    if labels is None:
        labels = _empty((s.B, s.H, s.N), torch.int32, dev)
    if perm is None:
        perm = _empty((s.B, s.H, s.N), torch.int32, dev)
    need = lib().vc_cluster_workspace(s, k)
    if workspace is None:
        workspace = _workspace(need, dev)
    if block_fill:
        rc = lib().vc_cluster_ex(_ptr(V), s, k, iters, int(bool(warm_start)), int(block_fill), _ptr(centroids),
                                 _ptr(labels), _ptr(perm), _ptr(workspace), workspace.numel(), _ptr(dev_status),
                                 _stream(stream))
        _check(rc, "vc_cluster_ex")
        return centroids, labels, perm
    rc = lib().vc_cluster(_ptr(V), s, k, iters, int(bool(warm_start)), _ptr(centroids), _ptr(labels), _ptr(perm),
                          _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(stream))
    _check(rc, "vc_cluster")
    return centroids, labels, perm


def alloc_quantized(shape: VcShape, device, vsmooth=1):
    nb = nblk_of(shape.N)
    npad = nb * BLOCK
    B, H, d = shape.B, shape.H, shape.d
    return dict(
        Q8=_empty((B, H, npad, d), torch.uint8, device), sq=_empty((B, H, nb), torch.float32, device),
        K8=_empty((B, H, npad, d), torch.uint8, device), sk=_empty((B, H, nb), torch.float32, device),
        V8T=_empty((B, H, d, npad), torch.uint8, device), sv=_empty((B, H, d), torch.float32, device),
        mu=_empty((B, H, nb, d), torch.int16, device) if vsmooth else None)


def _check_qkv(Q, K, V):
    s = shape_of(Q)
    if shape_of(K).N != s.N or shape_of(V).N != s.N:
        raise ValueError("Q, K, V shapes differ")
    if (K.stride(), V.stride()) != (Q.stride(), Q.stride()):
        raise ValueError("Q, K, V must share strides")
    return s


def _check_rope(rope, s: VcShape):
    if rope is None:
        return
    if rope.dtype != torch.float32 or tuple(rope.shape) != (s.N, s.d // 2, 2) or not rope.is_contiguous():
        raise ValueError("rope must be a contiguous fp32 [N, d/2, 2] (cos, sin) table")


def _quantize_call(fn, name, Q, K, V, perm, vsmooth, rope, hadamard, out, workspace, need, stream):
    s = _check_qkv(Q, K, V)
    _check_rope(rope, s)
    dev = Q.device
    if out is None:
        out = alloc_quantized(s, dev, vsmooth)
    if workspace is None:
        workspace = _workspace(need(s), dev)
    args = [_ptr(Q), _ptr(K), _ptr(V), s, _ptr(perm), int(vsmooth), _ptr(rope), int(hadamard),
             _ptr(out["Q8"]), _ptr(out["sq"]), _ptr(out["K8"]), _ptr(out["sk"]), _ptr(out["V8T"]), _ptr(out["sv"]),
             _ptr(out["mu"]) if vsmooth else None, _ptr(workspace), workspace.numel(), _stream(stream)]
    _check(fn(*args), name)
    return out


def vc_quantize(Q, K, V, perm=None, vsmooth=1, out=None, workspace=None, stream=None, vbits=8):
    """Fused quantizer. Returns a dict with Q8, sq, K8, sk, V8T, sv, mu (mu is bf16 bits as int16).
    vbits=4 calls vc_quantize_v4: the V residual in 4 bits (E2M1 with a power-of-two
    scale per 32 tokens of a channel), stored as E4M3 bytes for vc_attn_fwd."""
    L = lib()
    s = _check_qkv(Q, K, V)
    dev = Q.device
    if out is None:
        out = alloc_quantized(s, dev, vsmooth)
    if workspace is None:
        workspace = _workspace(L.vc_quantize_workspace(s), dev)
    if vbits not in (4, 8):
        raise ValueError("vbits must be 4 or 8")
    fn, name = (L.vc_quantize_v4, "vc_quantize_v4") if vbits == 4 else (L.vc_quantize, "vc_quantize")
    rc = fn(_ptr(Q), _ptr(K), _ptr(V), s, _ptr(perm), int(vsmooth), _ptr(out["Q8"]),
            _ptr(out["sq"]), _ptr(out["K8"]), _ptr(out["sk"]), _ptr(out["V8T"]), _ptr(out["sv"]),
            _ptr(out["mu"]) if vsmooth else None, _ptr(workspace), workspace.numel(),
            _stream(stream))
    _check(rc, name)
    return out


def vc_quantize_ex(Q, K, V, perm=None, vsmooth=1, rope=None, hadamard=0, out=None, workspace=None, stream=None):
    """vc_quantize with the rotary transform (``rope``: fp32 [N, d/2, 2] (cos, sin)
    table on the device) and/or the Hadamard rotation of Q and K fused in."""
    L = lib()
    return _quantize_call(L.vc_quantize_ex, "vc_quantize_ex", Q, K, V, perm, vsmooth, rope, hadamard, out,
                          workspace, L.vc_quantize_workspace, stream)


def vc_quantize_staged(Q, K, V, perm=None, vsmooth=1, rope=None, hadamard=0, out=None, workspace=None,
                       stream=None):
    """The same computation as vc_quantize_ex as the unfused chain of kernels
    (intermediates in device memory); bit-identical outputs."""
    L = lib()
    return _quantize_call(L.vc_quantize_staged, "vc_quantize_staged", Q, K, V, perm, vsmooth, rope, hadamard, out,
                          workspace, L.vc_quantize_staged_workspace, stream)


def quantize_staged_workspace_bytes(shape: VcShape) -> int:
    return lib().vc_quantize_staged_workspace(shape)


def vc_attn_fwd(qz, shape: VcShape, softmax_scale=0.0, expcast=1, vsmooth=1, O=None, dev_status=None,
                stream=None, debug=None, exact_margin=None):
    """FP8 attention on vc_quantize outputs. O is bf16 [B,N,H,d] laid out with `shape`'s strides.

    exact_margin (float) selects the hybrid bytes (vc_attn_fwd_hybrid):
    exp-then-cast on the key tiles within that many log2 units of a row's
    running maximum, ExpCast elsewhere; expcast is then ignored.
    expcast: 0 exp-then-cast, 1 ExpCast, 3 range-adaptive ExpCast (a beta per
    pair of codes of the octave).
    debug=(bh, qtile) additionally returns the fp32 scores and probability bytes
    of that one query tile: (O, S_dump [128, Npad], P_dump [128, Npad]).
    """
    dev = qz["Q8"].device
    if O is None:
        O = torch.empty((shape.B, shape.N, shape.H, shape.d), dtype=torch.bfloat16, device=dev)
        if (O.stride(0), O.stride(1), O.stride(2)) != (shape.s_b, shape.s_n, shape.s_h):
            O = torch.empty_strided((shape.B, shape.N, shape.H, shape.d), (shape.s_b, shape.s_n, shape.s_h, 1),
                                    dtype=torch.bfloat16, device=dev)
    ops = [_ptr(qz["Q8"]), _ptr(qz["sq"]), _ptr(qz["K8"]), _ptr(qz["sk"]), _ptr(qz["V8T"]), _ptr(qz["sv"]),
           _ptr(qz["mu"]) if vsmooth else None, shape, float(softmax_scale)]
    tail = [_ptr(O), _ptr(dev_status), _stream(stream)]
    if exact_margin is not None:
        expcast = 2
    if debug is None:
        if exact_margin is not None:
            _check(lib().vc_attn_fwd_hybrid(*ops, float(exact_margin), int(vsmooth), *tail), "vc_attn_fwd_hybrid")
        else:
            _check(lib().vc_attn_fwd(*ops, int(expcast), int(vsmooth), *tail), "vc_attn_fwd")
        return O
    npad = nblk_of(shape.N) * BLOCK
    S = torch.zeros((BLOCK, npad), dtype=torch.float32, device=dev)
    P = torch.zeros((BLOCK, npad), dtype=torch.uint8, device=dev)
    _check(lib().vc_attn_fwd_debug(*ops, int(expcast), int(vsmooth), *tail, int(debug[0]), int(debug[1]), _ptr(S),
                                   _ptr(P), float(exact_margin or 0.0)), "vc_attn_fwd_debug")
    return O, S, P


def vc_debug_e4m3_encode(x: torch.Tensor, out=None, stream=None):
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(lib().vc_debug_e4m3_encode(_ptr(x), x.numel(), _ptr(out), _stream(stream)), "vc_debug_e4m3_encode")
    return out


def vc_debug_wait_timeout(dev_status: torch.Tensor, timeout_us: int, stream=None):
    _check(lib().vc_debug_wait_timeout(_ptr(dev_status), int(timeout_us), _stream(stream)), "vc_debug_wait_timeout")


def vc_debug_attn_timeout(qz, shape: VcShape, dev_status: torch.Tensor, skip_k_tile: int, timeout_us: int,
                          vsmooth=1, O=None, stream=None):
    """vc_attn_fwd whose K loader never delivers key tile `skip_k_tile`, every
    device wait bounded by timeout_us: the kernel must record VC_ERR_TIMEOUT in
    dev_status and return.  Returns O (unspecified contents)."""
    if O is None:
        O = torch.empty((shape.B, shape.N, shape.H, shape.d), dtype=torch.bfloat16, device=qz["Q8"].device)
    _check(lib().vc_debug_attn_timeout(_ptr(qz["Q8"]), _ptr(qz["sq"]), _ptr(qz["K8"]), _ptr(qz["sk"]),
                                       _ptr(qz["V8T"]), _ptr(qz["sv"]), _ptr(qz["mu"]) if vsmooth else None, shape,
                                       int(vsmooth), _ptr(O), _ptr(dev_status), _stream(stream), int(skip_k_tile),
                                       int(timeout_us)), "vc_debug_attn_timeout")
    return O
