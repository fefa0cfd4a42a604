"""CPU oracle for the VC-Attention hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  It shares no code with the CUDA
library (``bit_fp8_attention_means_gb300``) and never imports it; both sides
receive the same seeded inputs from ``bit_fp8_attention_means_gb300.inputs``.

Every function takes / returns numpy arrays.  bf16 tensors are passed as their
raw ``uint16`` bit patterns.  Layouts follow the C-ABI of the library:
Q/K/V ``[B, N, H, d]`` (any strides with unit channel stride), Q8/K8
``[B, H, Npad, d]``, V8T ``[B, H, d, Npad]``, scales ``[B, H, nblk]`` /
``[B, H, d]``, means ``[B, H, nblk, d]``.

Parity status of each function is pinned by ``tests/test_oracle_*.py``;
see the file header of ``vc_oracle.c`` for the passages each step follows.
"""
import ctypes
import math
import os

import numpy as np

from . import build as _build

BLOCK = 128
_lib = None

_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64
_int = ctypes.c_int


# Test aid: the mutation tests point this variable at a build of a copy of
# vc_oracle.c with one planted mistake, to show that the pins catch it.
LIB_OVERRIDE_ENV = "VC_ORACLE_LIB_OVERRIDE"


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(os.environ.get(LIB_OVERRIDE_ENV) or _build.build())
        L = _lib
        L.vco_e4m3_decode.restype = ctypes.c_double
        L.vco_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.vco_e4m3_encode.restype = ctypes.c_uint8
        L.vco_e4m3_encode.argtypes = [ctypes.c_float]
        L.vco_expcast_C.restype = ctypes.c_float
        L.vco_expcast_C.argtypes = [ctypes.c_float]
        L.vco_expcast_code.restype = ctypes.c_uint8
        L.vco_expcast_code.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_float]
        L.vco_e4m3_encode_arr.argtypes = [_f32p, _i64, _u8p]
        L.vco_e4m3_decode_arr.argtypes = [_u8p, _i64, _f64p]
        L.vco_bf16_rne_arr.argtypes = [_f32p, _i64, _u16p]
        L.vco_expcast_arr.argtypes = [_f32p, _i64, ctypes.c_float, ctypes.c_float, _u8p]
        L.vco_expcast_piece_arr.argtypes = [_f32p, _i64, ctypes.c_float, ctypes.c_float, _u8p]
        L.vco_expcast_C0.restype = ctypes.c_float
        L.vco_expcast_C0.argtypes = [ctypes.c_float]
        L.vco_kmeans.restype = _int
        L.vco_kmeans.argtypes = [_u16p, _int, _int, _int, _int, _i64, _i64, _i64,
                                 _int, _int, _int, _f32p, _i32p]
        L.vco_argsort_labels.restype = _int
        L.vco_argsort_labels.argtypes = [_i32p, _int, _int, _int, _i32p]
        L.vco_block_fill.restype = _int
        L.vco_block_fill.argtypes = [_i32p, _f32p, _int, _int, _int, _int, _i32p]
        L.vco_quantize.restype = _int
        L.vco_quantize.argtypes = [_u16p, _u16p, _u16p, _int, _int, _int, _int, _i64, _i64, _i64,
                                   ctypes.c_void_p, _int, _u8p, _f32p, _u8p, _f32p, _u8p, _f32p,
                                   ctypes.c_void_p]
        L.vco_e2m1_decode.restype = ctypes.c_double
        L.vco_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.vco_e2m1_encode.restype = ctypes.c_uint8
        L.vco_e2m1_encode.argtypes = [ctypes.c_float]
        L.vco_e2m1_encode_arr.argtypes = [_f32p, _i64, _u8p]
        L.vco_quantize_v4.restype = _int
        L.vco_quantize_v4.argtypes = [_u16p, _u16p, _u16p, _int, _int, _int, _int, _i64, _i64, _i64,
                                      ctypes.c_void_p, _int, _u8p, _f32p, _u8p, _f32p, _u8p, _f32p,
                                      ctypes.c_void_p]
        L.vco_quantize_ex.restype = _int
        L.vco_quantize_ex.argtypes = [_u16p, _u16p, _u16p, _int, _int, _int, _int, _i64, _i64, _i64,
                                      ctypes.c_void_p, _int, ctypes.c_void_p, _int,
                                      _u8p, _f32p, _u8p, _f32p, _u8p, _f32p, ctypes.c_void_p]
        L.vco_preproc_rows.restype = _int
        L.vco_preproc_rows.argtypes = [_u16p, _i64, _int, ctypes.c_void_p, ctypes.c_void_p, _int, _f32p]
        L.vco_attn.restype = _int
        L.vco_attn.argtypes = [_u8p, _f32p, _u8p, _f32p, _u8p, _f32p, ctypes.c_void_p,
                               _int, _int, _int, _int, ctypes.c_float, _int, _int,
                               _i32p, _int, ctypes.c_void_p, _f64p, ctypes.c_void_p]
        L.vco_attn_ex.restype = _int
        L.vco_attn_ex.argtypes = [_u8p, _f32p, _u8p, _f32p, _u8p, _f32p, ctypes.c_void_p,
                                  _int, _int, _int, _int, ctypes.c_float, _int, ctypes.c_float, _int,
                                  _i32p, _int, ctypes.c_void_p, _f64p, ctypes.c_void_p]
        L.vco_attn_ref.restype = _int
        L.vco_attn_ref.argtypes = [_u16p, _u16p, _u16p, _int, _int, _int, _int, _i64, _i64, _i64,
                                   ctypes.c_double, _i32p, _int, _f64p]
        L.vco_num_threads.restype = _int
    return _lib


def num_threads() -> int:
    return lib().vco_num_threads()


def nblk_of(N: int) -> int:
    return (N + BLOCK - 1) // BLOCK


# ---------------------------------------------------------------- codecs

def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    out = np.empty(c.size, np.float64)
    lib().vco_e4m3_decode_arr(c, c.size, out)
    return out.reshape(np.shape(codes))


def e4m3_encode(x) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(a.size, np.uint8)
    lib().vco_e4m3_encode_arr(a, a.size, out)
    return out.reshape(np.shape(x))


def e2m1_decode(code) -> float:
    return lib().vco_e2m1_decode(int(code))


def e2m1_encode(x) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(a.size, np.uint8)
    lib().vco_e2m1_encode_arr(a, a.size, out)
    return out.reshape(np.shape(x))


def bf16_rne(x) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.empty(a.size, np.uint16)
    lib().vco_bf16_rne_arr(a, a.size, out)
    return out.reshape(np.shape(x))


def bf16_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def kscale_of(softmax_scale: float, d: int) -> np.float32:
    """fp32(softmax_scale * log2 e); softmax_scale <= 0 means 1/sqrt(d)."""
    s = np.float32(softmax_scale) if softmax_scale > 0 else np.float32(1.0 / math.sqrt(d))
    return np.float32(float(s) * (1.0 / math.log(2.0)))


def expcast_C(m_new: float) -> np.float32:
    return np.float32(lib().vco_expcast_C(float(m_new)))


def expcast_C0(m_new: float) -> np.float32:
    return np.float32(lib().vco_expcast_C0(float(m_new)))


def expcast_piece_codes(acc, sigma8: float, C0: float) -> np.ndarray:
    """Range-adaptive ExpCast bytes (expcast = 3) for fp32 scores acc."""
    a = np.ascontiguousarray(acc, dtype=np.float32).ravel()
    out = np.empty(a.size, np.uint8)
    lib().vco_expcast_piece_arr(a, a.size, float(sigma8), float(C0), out)
    return out.reshape(np.shape(acc))


def expcast_codes(acc, sigma8: float, C: float) -> np.ndarray:
    a = np.ascontiguousarray(acc, dtype=np.float32).ravel()
    out = np.empty(a.size, np.uint8)
    lib().vco_expcast_arr(a, a.size, float(sigma8), float(C), out)
    return out.reshape(np.shape(acc))


# ---------------------------------------------------------------- path

def _bnhd(X):
    """uint16 [B,N,H,d] (any layout) -> (contiguous array, strides in elements)."""
    X = np.ascontiguousarray(X, dtype=np.uint16)
    B, N, H, d = X.shape
    return X, (N * H * d, H * d, d)


def kmeans(V, k: int, iters: int, centroids=None):
    """Lloyd k-means per (b,h). Returns (centroids fp32 [B,H,k,d], labels int32 [B,H,N])."""
    V, (sb, sn, sh) = _bnhd(V)
    B, N, H, d = V.shape
    warm = centroids is not None
    cent = (np.ascontiguousarray(centroids, dtype=np.float32).copy() if warm
            else np.zeros((B, H, k, d), np.float32))
    labels = np.zeros((B, H, N), np.int32)
    rc = lib().vco_kmeans(V, B, H, N, d, sb, sn, sh, k, iters, int(warm), cent, labels)
    assert rc == 0
    return cent, labels


def argsort_labels(labels, k: int) -> np.ndarray:
    z = np.ascontiguousarray(labels, dtype=np.int32)
    B, H, N = z.shape
    perm = np.zeros_like(z)
    assert lib().vco_argsort_labels(z, B * H, N, k, perm) == 0
    return perm


def _rope_table(rope, N: int, d: int):
    """fp32 [N, d/2, 2] (cos, sin) table -> (array kept alive, pointer)."""
    if rope is None:
        return None, None
    r = np.ascontiguousarray(rope, dtype=np.float32)
    assert r.shape == (N, d // 2, 2), r.shape
    return r, r.ctypes.data_as(ctypes.c_void_p)


def preproc_rows(X, pos=None, rope=None, hadamard: int = 0) -> np.ndarray:
    """Rotary transform (row r at position pos[r]) then Hadamard rotation of
    bf16 rows X [n, d]; returns the fp32 rows the Q/K quantizer encodes."""
    X = np.ascontiguousarray(X, dtype=np.uint16)
    n, d = X.shape
    out = np.zeros((n, d), np.float32)
    pp = None
    if pos is not None:
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        pp = pos.ctypes.data_as(ctypes.c_void_p)
    r = np.ascontiguousarray(rope, dtype=np.float32) if rope is not None else None
    rp = r.ctypes.data_as(ctypes.c_void_p) if r is not None else None
    assert lib().vco_preproc_rows(X, n, d, pp, rp, int(hadamard), out) == 0
    return out


def block_fill(labels, centroids) -> np.ndarray:
    """Block-fill permutation [B,H,N] from labels [B,H,N] and centroids [B,H,k,d]:
    whole 128-token blocks of each cluster in label order, then the clusters'
    leftovers along a greedy nearest-centroid chain."""
    z = np.ascontiguousarray(labels, dtype=np.int32)
    C = np.ascontiguousarray(centroids, dtype=np.float32)
    B, H, N = z.shape
    k, d = C.shape[2], C.shape[3]
    perm = np.zeros_like(z)
    assert lib().vco_block_fill(z, C, B * H, N, k, d, perm) == 0
    return perm


def quantize(Q, K, V, perm=None, vsmooth: int = 1, rope=None, hadamard: int = 0, vbits: int = 8):
    """Q/K/V quantizer.  With ``rope`` (fp32 [N, d/2, 2]) and/or ``hadamard``
    the Q and K rows are rotated / Hadamard-transformed before quantization
    and sq carries the factor 1/d.  vbits = 4 keeps the V residual in the 4-bit
    form (E2M1 with a power-of-two scale per 32 tokens of a channel, stored as
    the equal E4M3 byte; sv = amax/6); it takes no rotary table or Hadamard."""
    Q, (sb, sn, sh) = _bnhd(Q)
    K, _ = _bnhd(K)
    V, _ = _bnhd(V)
    B, N, H, d = Q.shape
    nb = nblk_of(N)
    Npad = nb * BLOCK
    out = dict(
        Q8=np.zeros((B, H, Npad, d), np.uint8), sq=np.zeros((B, H, nb), np.float32),
        K8=np.zeros((B, H, Npad, d), np.uint8), sk=np.zeros((B, H, nb), np.float32),
        V8T=np.zeros((B, H, d, Npad), np.uint8), sv=np.zeros((B, H, d), np.float32),
        mu=np.zeros((B, H, nb, d), np.uint16))
    p = None
    if perm is not None:
        perm = np.ascontiguousarray(perm, dtype=np.int32)
        p = perm.ctypes.data_as(ctypes.c_void_p)
    r, rp = _rope_table(rope, N, d)
    if vbits == 4:
        assert rope is None and not hadamard
        rc = lib().vco_quantize_v4(Q, K, V, B, H, N, d, sb, sn, sh, p, int(vsmooth),
                                   out["Q8"], out["sq"], out["K8"], out["sk"], out["V8T"], out["sv"],
                                   out["mu"].ctypes.data_as(ctypes.c_void_p))
    else:
        assert vbits == 8
        rc = lib().vco_quantize_ex(Q, K, V, B, H, N, d, sb, sn, sh, p, int(vsmooth), rp, int(hadamard),
                                   out["Q8"], out["sq"], out["K8"], out["sk"], out["V8T"], out["sv"],
                                   out["mu"].ctypes.data_as(ctypes.c_void_p))
    assert rc == 0
    return out


def attn(qz: dict, N: int, softmax_scale: float = 0.0, expcast: int = 1, vsmooth: int = 1,
         rows=None, acc_in=None, want_codes: bool = False, margin: float = 0.0):
    """Quantized-path attention for the query rows ``rows`` of every (b,h).

    expcast: 0 exp-then-cast, 1 ExpCast, 2 hybrid (exp-then-cast on the key
    tiles that are high-weight for a 32-row group: some row's tile maximum
    within ``margin`` (log2 units) of its running maximum; ``rows`` must then
    hold whole groups), 3 range-adaptive ExpCast (a beta per pair of codes
    of the octave).  Returns O fp64 [B,H,nrows,d] (and codes uint8
    [B,H,nrows,Npad] if asked).
    """
    B, H, Npad, d = qz["Q8"].shape
    if rows is None:
        rows = np.arange(N, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    nr = rows.size
    O = np.zeros((B, H, nr, d), np.float64)
    P = np.zeros((B, H, nr, Npad), np.uint8) if want_codes else None
    acc_p = None
    if acc_in is not None:
        acc_in = np.ascontiguousarray(acc_in, dtype=np.float32)
        assert acc_in.shape == (B, H, nr, Npad)
        acc_p = acc_in.ctypes.data_as(ctypes.c_void_p)
    mu = np.ascontiguousarray(qz["mu"], dtype=np.uint16)
    rc = lib().vco_attn_ex(np.ascontiguousarray(qz["Q8"]), np.ascontiguousarray(qz["sq"]),
                           np.ascontiguousarray(qz["K8"]), np.ascontiguousarray(qz["sk"]),
                           np.ascontiguousarray(qz["V8T"]), np.ascontiguousarray(qz["sv"]),
                           mu.ctypes.data_as(ctypes.c_void_p),
                           B, H, N, d, float(kscale_of(softmax_scale, d)), int(expcast), float(margin),
                           int(vsmooth), rows, nr, acc_p, O,
                           P.ctypes.data_as(ctypes.c_void_p) if P is not None else None)
    assert rc == 0
    return (O, P) if want_codes else O


def attn_ref(Q, K, V, softmax_scale: float = 0.0, rows=None) -> np.ndarray:
    """fp64 softmax(Q K^T * scale) V on the bf16 inputs. Returns [B,H,nrows,d]."""
    Q, (sb, sn, sh) = _bnhd(Q)
    K, _ = _bnhd(K)
    V, _ = _bnhd(V)
    B, N, H, d = Q.shape
    scale = softmax_scale if softmax_scale > 0 else 1.0 / math.sqrt(d)
    if rows is None:
        rows = np.arange(N, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    O = np.zeros((B, H, rows.size, d), np.float64)
    assert lib().vco_attn_ref(Q, K, V, B, H, N, d, sb, sn, sh, float(scale), rows, rows.size, O) == 0
    return O


# ---------------------------------------------------------------- O comparison

# Bars for comparing a bf16 attention output with this oracle's fp64 output on
# the same quantized inputs (see check_o).
O_TOL = 2e-3                 # relative L2 over the whole compared tensor
O_ROW_TOL = 2.0 ** -8 + 5e-4  # relative L2 of every query row
O_ELEM_REL = 2.0 ** -8       # per element: bf16 rounding of the kernel's value ...
O_ELEM_ROWRMS = 2e-3         # ... plus this fraction of the row's RMS
O_ELEM_ROWRMS_EXP = 2e-2     # ... or this one where the bytes come from an exponential (see check_o)
O_ROW_TOL_EXP = 1e-2         # row bar where the bytes come from an exponential


def check_o(got, ref, where="", exp_bytes=False):
    """Compare a kernel output with the oracle, element by element.

    got, ref: arrays [..., rows, d] (got the kernel's bf16 values as floats,
    ref this oracle's fp64 output for the same rows).  Three bars, each
    derived from what separates the two:
      * bf16 rounding of the kernel's output: half an ulp is at most 2^-8 of
        the element, so no element can differ by more than 2^-8 |ref| for
        that reason, and no row's relative L2 by more than 2^-8;
      * the kernel's arithmetic (fp32 tensor-core sums in another order, the
        rescale factor from a hardware exp2, the mean term through bf16
        hi/lo parts) moves O by ~1e-4 of the row's RMS, well inside
        O_ELEM_ROWRMS = 2e-3 and the 5e-4 added to the row bar.
    Bars: the whole tensor within O_TOL (2e-3) relative L2; every query row
    within O_ROW_TOL; every element within O_ELEM_REL |ref| + O_ELEM_ROWRMS
    rms(ref row).  A row that is wrong by a few percent passes the first bar
    but fails the other two.  Returns the worst ratios (observed / bar).

    exp_bytes: the compared output took some probability bytes from an
    exponential (exp-then-cast, or the exact tiles of the hybrid bytes).  The
    kernel's hardware exp2 is not correctly rounded, so up to about one byte
    in 10^3 lands one E4M3 step away from the oracle's; one step moves that
    probability by at most 1/8 of itself, and a heavy key moved so shifts
    its row by up to ~1/8 of its weight times its distance from the row's
    output -- a few 1e-3 of the row on the test workloads, whose largest
    single-key weights are a few percent.  The row bar is then
    O_ROW_TOL_EXP (1e-2) and the per-element allowance O_ELEM_ROWRMS_EXP
    (2e-2) of the row's RMS; the tensor bar stays 2e-3, and a row wrong by a
    few percent still fails.
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    diff = got - ref
    tot = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    rnorm = np.linalg.norm(ref, axis=-1)
    rrel = np.linalg.norm(diff, axis=-1) / np.maximum(rnorm, 1e-300)
    rms = (rnorm / math.sqrt(ref.shape[-1]))[..., None]
    bound = O_ELEM_REL * np.abs(ref) + (O_ELEM_ROWRMS_EXP if exp_bytes else O_ELEM_ROWRMS) * rms
    row_tol = O_ROW_TOL_EXP if exp_bytes else O_ROW_TOL
    eratio = np.abs(diff) / np.maximum(bound, 1e-300)
    stats = {"total": tot / O_TOL, "row": float(rrel.max()) / row_tol, "elem": float(eratio.max())}
    msg = "%s: rel-L2 %.3e (bar %.1e), worst row %.3e at %s (bar %.2e), worst element %.2f x its bar at %s" % (
        where, tot, O_TOL, float(rrel.max()), np.unravel_index(int(np.argmax(rrel)), rrel.shape), row_tol,
        float(eratio.max()), np.unravel_index(int(np.argmax(eratio)), eratio.shape))
    assert tot <= O_TOL and float(rrel.max()) <= row_tol and float(eratio.max()) <= 1.0, msg
    return stats
