"""Python binding of libqmm (the C ABI declared in include/qmm.h).

Argument marshalling only: every function here has the name of the C entry
point it calls, converts tensors to device pointers and the current torch
stream to a cudaStream_t, and raises QmmError on a non-OK status.  All
arithmetic runs in the CUDA kernels of libqmm.so; there is no other path.
Tensors may be torch CUDA tensors or raw integer device addresses.
"""
from __future__ import annotations

import ctypes
import os

from .buildlib import LIB, build  # noqa: F401

QMM_Q4_0, QMM_Q8_0, QMM_Q4_K, QMM_Q6_K, QMM_Q2_K, QMM_Q8_K, QMM_Q4_1, QMM_Q5_0, QMM_Q5_1, QMM_Q5_K = range(10)
TYPES = {"q4_0": QMM_Q4_0, "q8_0": QMM_Q8_0, "q4_K": QMM_Q4_K, "q6_K": QMM_Q6_K, "q2_K": QMM_Q2_K,
         "q8_K": QMM_Q8_K, "q4_1": QMM_Q4_1, "q5_0": QMM_Q5_0, "q5_1": QMM_Q5_1, "q5_K": QMM_Q5_K}
WEIGHT_TYPES = ("q4_0", "q8_0", "q4_K", "q6_K", "q2_K", "q4_1", "q5_0", "q5_1", "q5_K")

STATUS = {0: "QMM_OK", 1: "QMM_E_NULL", 2: "QMM_E_SHAPE", 3: "QMM_E_TYPE", 4: "QMM_E_ALIGN",
          5: "QMM_E_SCRATCH", 6: "QMM_E_CUDA", 7: "QMM_E_TIMEOUT", 8: "QMM_E_BOUNDS"}

# every entry point the header declares, with its argument kinds
# p: pointer, i: int64, s: size_t, t: int (type code), c: int, q: stream
SIGNATURES = {
    "qmm_block_bytes": ("t", ctypes.c_size_t),
    "qmm_block_values": ("t", ctypes.c_int),
    "qmm_row_bytes": ("ti", ctypes.c_size_t),
    "qmm_act_type": ("t", ctypes.c_int),
    "qmm_status_str": ("c", ctypes.c_char_p),
    "qmm_quantize_q8_0": ("ppiiq", ctypes.c_int),
    "qmm_quantize_q8_K": ("ppiiq", ctypes.c_int),
    "qmm_quantize_q4_0": ("ppiiq", ctypes.c_int),
    "qmm_quantize_q4_K": ("ppiiq", ctypes.c_int),
    "qmm_quantize_q6_K": ("ppiiq", ctypes.c_int),
    "qmm_quantize_q2_K": ("ppiiq", ctypes.c_int),
    "qmm_quantize_q4_1": ("ppiiq", ctypes.c_int),
    "qmm_quantize_q5_0": ("ppiiq", ctypes.c_int),
    "qmm_quantize_q5_1": ("ppiiq", ctypes.c_int),
    "qmm_quantize_q5_K": ("ppiiq", ctypes.c_int),
    "qmm_matvec_q4_0": ("pppiiq", ctypes.c_int),
    "qmm_matvec_q8_0": ("pppiiq", ctypes.c_int),
    "qmm_matvec_q4_K": ("pppiiq", ctypes.c_int),
    "qmm_matvec_q6_K": ("pppiiq", ctypes.c_int),
    "qmm_matvec_q2_K": ("pppiiq", ctypes.c_int),
    "qmm_matvec_q4_1": ("pppiiq", ctypes.c_int),
    "qmm_matvec_q5_0": ("pppiiq", ctypes.c_int),
    "qmm_matvec_q5_1": ("pppiiq", ctypes.c_int),
    "qmm_matvec_q5_K": ("pppiiq", ctypes.c_int),
    "qmm_linear_q4_0": ("pppspiiiq", ctypes.c_int),
    "qmm_linear_q8_0": ("pppspiiiq", ctypes.c_int),
    "qmm_linear_q4_K": ("pppspiiiq", ctypes.c_int),
    "qmm_linear_q6_K": ("pppspiiiq", ctypes.c_int),
    "qmm_linear_q2_K": ("pppspiiiq", ctypes.c_int),
    "qmm_linear_q4_1": ("pppspiiiq", ctypes.c_int),
    "qmm_linear_q5_0": ("pppspiiiq", ctypes.c_int),
    "qmm_linear_q5_1": ("pppspiiiq", ctypes.c_int),
    "qmm_linear_q5_K": ("pppspiiiq", ctypes.c_int),
    "qmm_matmul_q4_0": ("pppiiiq", ctypes.c_int),
    "qmm_matmul_q8_0": ("pppiiiq", ctypes.c_int),
    "qmm_matmul_q4_1": ("pppiiiq", ctypes.c_int),
    "qmm_matmul_q5_0": ("pppiiiq", ctypes.c_int),
    "qmm_matmul_q5_1": ("pppiiiq", ctypes.c_int),
    "qmm_get_rows": ("tpppiiiq", ctypes.c_int),
    "qmm_linear_host": ("tppppsppiiiq", ctypes.c_int),
    "qmm_rmsnorm_quantize": ("tppfpiiq", ctypes.c_int),
    "qmm_linear_norm": ("ttppppfpspiiq", ctypes.c_int),
    "qmm_kv_row_bytes": ("i", ctypes.c_size_t),
    "qmm_kv_quantize": ("ppiiq", ctypes.c_int),
    "qmm_kv_scores": ("pppiiiifq", ctypes.c_int),
    "qmm_kv_wsum_scratch_bytes": ("iii", ctypes.c_size_t),
    "qmm_kv_wsum": ("pppps" + "iiiiq", ctypes.c_int),
    "qmm_matmul_q4_K": ("pppiiiq", ctypes.c_int),
    "qmm_matmul_q6_K": ("pppiiiq", ctypes.c_int),
    "qmm_matmul_q5_K": ("pppiiiq", ctypes.c_int),
    "qmm_matmul_q2_K": ("pppiiiq", ctypes.c_int),
    "qmm_linear_noalloc": ("tpppiiiq", ctypes.c_int),
    "qmm_linear_group": ("ttppppspiiq", ctypes.c_int),
    "qmm_blocksums": ("tpppiiiq", ctypes.c_int),
    "qmm_test_wait_timeout": ("uq", ctypes.c_int),
    "qmm_device_status": ("c", ctypes.c_int),
}
_CT = {"p": ctypes.c_void_p, "i": ctypes.c_int64, "s": ctypes.c_size_t, "t": ctypes.c_int, "c": ctypes.c_int,
       "q": ctypes.c_void_p, "f": ctypes.c_float, "u": ctypes.c_uint64}

_lib = None


class QmmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (fn, STATUS.get(status, status), _status_str(status)))


def load(path: str = None):
    """Load libqmm.so (built in-tree by build()); raises if it is missing.  The environment
    variable QMM_LIBRARY names another build of the same library to load instead (the
    bounds-checked variant, block_quantized_weight_q8_gb300.buildlib.CHECKED_LIB)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("QMM_LIBRARY") or LIB
    if not os.path.exists(path):
        raise ImportError("libqmm.so is not built (%s): run block_quantized_weight_q8_gb300.build()" % path)
    L = ctypes.CDLL(path)
    for name, (kinds, res) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.argtypes = [_CT[k] for k in kinds]
        fn.restype = res
    _lib = L
    return L


def _status_str(status: int) -> str:
    try:
        return load().qmm_status_str(int(status)).decode()
    except Exception:
        return "?"


def ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def stream_handle(stream=None) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _call(name, *args):
    r = getattr(load(), name)(*args)
    if r != 0:
        raise QmmError(name, r)


def _type(t) -> int:
    return TYPES[t] if isinstance(t, str) else int(t)


# ---- formats
def qmm_block_bytes(t) -> int:
    return int(load().qmm_block_bytes(_type(t)))


def qmm_block_values(t) -> int:
    return int(load().qmm_block_values(_type(t)))


def qmm_row_bytes(t, K: int) -> int:
    return int(load().qmm_row_bytes(_type(t), int(K)))


def qmm_act_type(wtype) -> int:
    return int(load().qmm_act_type(_type(wtype)))


# ---- quantizers
def qmm_quantize_q8_0(x, xq, M, K, stream=None):
    _call("qmm_quantize_q8_0", ptr(x), ptr(xq), int(M), int(K), stream_handle(stream))


def qmm_quantize_q8_K(x, xq, M, K, stream=None):
    _call("qmm_quantize_q8_K", ptr(x), ptr(xq), int(M), int(K), stream_handle(stream))


def qmm_quantize_q4_0(w, wq, N, K, stream=None):
    _call("qmm_quantize_q4_0", ptr(w), ptr(wq), int(N), int(K), stream_handle(stream))


def qmm_quantize_q4_K(w, wq, N, K, stream=None):
    _call("qmm_quantize_q4_K", ptr(w), ptr(wq), int(N), int(K), stream_handle(stream))


def qmm_quantize_q6_K(w, wq, N, K, stream=None):
    _call("qmm_quantize_q6_K", ptr(w), ptr(wq), int(N), int(K), stream_handle(stream))


def qmm_quantize_q2_K(w, wq, N, K, stream=None):
    _call("qmm_quantize_q2_K", ptr(w), ptr(wq), int(N), int(K), stream_handle(stream))


def quantize(t, x, out, rows, K, stream=None):
    """qmm_quantize_<t> by type name (q8_0 also quantizes Q8_0 weights)."""
    _call("qmm_quantize_" + t, ptr(x), ptr(out), int(rows), int(K), stream_handle(stream))


# ---- matvec / linear / matmul
def _mv(name):
    def f(W, xq, y, N, K, stream=None):
        _call(name, ptr(W), ptr(xq), ptr(y), int(N), int(K), stream_handle(stream))
    f.__name__ = name
    return f


qmm_matvec_q4_0 = _mv("qmm_matvec_q4_0")
qmm_matvec_q8_0 = _mv("qmm_matvec_q8_0")
qmm_matvec_q4_K = _mv("qmm_matvec_q4_K")
qmm_matvec_q6_K = _mv("qmm_matvec_q6_K")
qmm_matvec_q2_K = _mv("qmm_matvec_q2_K")
qmm_matvec_q4_1 = _mv("qmm_matvec_q4_1")
qmm_matvec_q5_0 = _mv("qmm_matvec_q5_0")
qmm_matvec_q5_1 = _mv("qmm_matvec_q5_1")
qmm_matvec_q5_K = _mv("qmm_matvec_q5_K")


def matvec(wtype, W, xq, y, N, K, stream=None):
    _call("qmm_matvec_" + wtype, ptr(W), ptr(xq), ptr(y), int(N), int(K), stream_handle(stream))


def _lin(name):
    def f(W, x, scratch, scratch_bytes, y, M, N, K, stream=None):
        _call(name, ptr(W), ptr(x), ptr(scratch), int(scratch_bytes), ptr(y), int(M), int(N), int(K),
              stream_handle(stream))
    f.__name__ = name
    return f


qmm_linear_q4_0 = _lin("qmm_linear_q4_0")
qmm_linear_q8_0 = _lin("qmm_linear_q8_0")
qmm_linear_q4_K = _lin("qmm_linear_q4_K")
qmm_linear_q6_K = _lin("qmm_linear_q6_K")
qmm_linear_q2_K = _lin("qmm_linear_q2_K")
qmm_linear_q4_1 = _lin("qmm_linear_q4_1")
qmm_linear_q5_0 = _lin("qmm_linear_q5_0")
qmm_linear_q5_1 = _lin("qmm_linear_q5_1")
qmm_linear_q5_K = _lin("qmm_linear_q5_K")


def linear(wtype, W, x, scratch, scratch_bytes, y, M, N, K, stream=None):
    _call("qmm_linear_" + wtype, ptr(W), ptr(x), ptr(scratch), int(scratch_bytes), ptr(y), int(M), int(N), int(K),
          stream_handle(stream))


def qmm_linear_host(wtype, W, x_host, x_dev, scratch, scratch_bytes, y_dev, y_host, M, N, K, stream=None):
    """qmm_linear_<wtype> with host buffers: x_host (pinned) -> x_dev, the multiply, y_dev -> y_host, queued on
    the stream (synchronize it before reading y_host)."""
    _call("qmm_linear_host", _type(wtype), ptr(W), ptr(x_host), ptr(x_dev), ptr(scratch), int(scratch_bytes), ptr(y_dev),
          ptr(y_host), int(M), int(N), int(K), stream_handle(stream))


def qmm_linear_noalloc(wtype, W, x, y, M, N, K, stream=None):
    """qmm_linear_<wtype> without a workspace argument: the library's own 1 MiB device array holds the
    quantized rows (see include/qmm.h for the limit and the sharing rules)."""
    _call("qmm_linear_noalloc", _type(wtype), ptr(W), ptr(x), ptr(y), int(M), int(N), int(K), stream_handle(stream))


def qmm_linear_group(wtype, Ws, Ns, x, scratch, scratch_bytes, ys, M, K, stream=None):
    """qmm_linear_<wtype> for several matrices Ws (rows Ns) on the same rows x, outputs ys, one launch
    per token (see include/qmm.h)."""
    G = len(Ws)
    if not (len(Ns) == G and len(ys) == G):
        raise ValueError("Ws, Ns and ys must have the same length")
    w_arr = (ctypes.c_void_p * max(G, 1))(*[ptr(w) for w in Ws])
    n_arr = (ctypes.c_int64 * max(G, 1))(*[int(n) for n in Ns])
    y_arr = (ctypes.c_void_p * max(G, 1))(*[ptr(y) for y in ys])
    _call("qmm_linear_group", _type(wtype), G, ctypes.cast(w_arr, ctypes.c_void_p), ctypes.cast(n_arr, ctypes.c_void_p),
          ptr(x), ptr(scratch), int(scratch_bytes), ctypes.cast(y_arr, ctypes.c_void_p), int(M), int(K),
          stream_handle(stream))


def qmm_rmsnorm_quantize(act, x, w, eps, xq, M, K, stream=None):
    """Quantize the RMSNormed rows (x * s) * w to act ("q8_0" or "q8_K")."""
    _call("qmm_rmsnorm_quantize", _type(act), ptr(x), ptr(w), float(eps), ptr(xq), int(M), int(K), stream_handle(stream))


def qmm_linear_norm(wtype, Ws, Ns, x, w, eps, scratch, scratch_bytes, ys, M, K, stream=None):
    """qmm_linear_group on the RMSNormed rows of x (norm weight w, eps)."""
    G = len(Ws)
    if not (len(Ns) == G and len(ys) == G):
        raise ValueError("Ws, Ns and ys must have the same length")
    w_arr = (ctypes.c_void_p * max(G, 1))(*[ptr(m) for m in Ws])
    n_arr = (ctypes.c_int64 * max(G, 1))(*[int(n) for n in Ns])
    y_arr = (ctypes.c_void_p * max(G, 1))(*[ptr(y) for y in ys])
    _call("qmm_linear_norm", _type(wtype), G, ctypes.cast(w_arr, ctypes.c_void_p), ctypes.cast(n_arr, ctypes.c_void_p),
          ptr(x), ptr(w), float(eps), ptr(scratch), int(scratch_bytes), ctypes.cast(y_arr, ctypes.c_void_p), int(M),
          int(K), stream_handle(stream))


def qmm_matmul_q4_0(W, xq, Y, M, N, K, stream=None):
    _call("qmm_matmul_q4_0", ptr(W), ptr(xq), ptr(Y), int(M), int(N), int(K), stream_handle(stream))


def matmul(wtype, W, xq, Y, M, N, K, stream=None):
    """qmm_matmul_<wtype>: Y[M][N] for M quantized activation rows (Q8_0 for the 32-value formats, Q8_K for
    the K-quants)."""
    _call("qmm_matmul_" + wtype, ptr(W), ptr(xq), ptr(Y), int(M), int(N), int(K), stream_handle(stream))


def qmm_get_rows(wtype, W, ids, out, R, N, K, stream=None):
    """out[r] = dequantized row ids[r] of W (ids: int32 device tensor)."""
    _call("qmm_get_rows", _type(wtype), ptr(W), ptr(ids), ptr(out), int(R), int(N), int(K), stream_handle(stream))


# ---- the Q8 KV cache
def qmm_kv_row_bytes(hd):
    return int(load().qmm_kv_row_bytes(int(hd)))


def qmm_kv_quantize(x, out, rows, hd, stream=None):
    """rows head vectors (f32 [rows][hd]) into quantized rows (f32 d + int8 codes) at out."""
    _call("qmm_kv_quantize", ptr(x), ptr(out), int(rows), int(hd), stream_handle(stream))


def qmm_kv_scores(q, kc, scores, Hq, Hkv, P, hd, scale, stream=None):
    """scores[h][p] for the quantized query rows q against positions 0..P-1 of the K cache kc."""
    _call("qmm_kv_scores", ptr(q), ptr(kc), ptr(scores), int(Hq), int(Hkv), int(P), int(hd), float(scale),
          stream_handle(stream))


def qmm_kv_wsum_scratch_bytes(Hq, P, hd):
    return int(load().qmm_kv_wsum_scratch_bytes(int(Hq), int(P), int(hd)))


def qmm_kv_wsum(w, vc, out, scratch, scratch_bytes, Hq, Hkv, P, hd, stream=None):
    """out[h] = sum_p w[h][p] * (dequantized V row of position p, KV head h / (Hq/Hkv))."""
    _call("qmm_kv_wsum", ptr(w), ptr(vc), ptr(out), ptr(scratch), int(scratch_bytes), int(Hq), int(Hkv), int(P),
          int(hd), stream_handle(stream))


def qmm_blocksums(wtype, W, xq, s, M, N, K, stream=None):
    _call("qmm_blocksums", _type(wtype), ptr(W), ptr(xq), ptr(s), int(M), int(N), int(K), stream_handle(stream))


def qmm_test_wait_timeout(limit_ns: int, stream=None):
    _call("qmm_test_wait_timeout", int(limit_ns), stream_handle(stream))


def qmm_device_status(clear: bool = False) -> int:
    return int(load().qmm_device_status(1 if clear else 0))
