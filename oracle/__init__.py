"""The CPU oracle for the block-quantized weight x Q8 activation matmul.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never imports it, and it imports nothing from the
product: the two share no code.  The arithmetic lives in ``qmm_oracle.c`` (plain
scalar C, -O2 -ffp-contract=off); this module only compiles it with gcc and
marshals numpy arrays through ctypes.

Type codes: 0 Q4_0, 1 Q8_0, 2 Q4_K, 3 Q6_K, 4 Q2_K, 5 Q8_K, 6 Q4_1, 7 Q5_0, 8 Q5_1, 9 Q5_K.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qmm_oracle.c")
LIB = os.path.join(HERE, "_build", "liboracle.so")

Q4_0, Q8_0, Q4_K, Q6_K, Q2_K, Q8_K, Q4_1, Q5_0, Q5_1, Q5_K = range(10)
TYPES = {"q4_0": Q4_0, "q8_0": Q8_0, "q4_K": Q4_K, "q6_K": Q6_K, "q2_K": Q2_K, "q8_K": Q8_K,
         "q4_1": Q4_1, "q5_0": Q5_0, "q5_1": Q5_1, "q5_K": Q5_K}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile qmm_oracle.c into _build/liboracle.so (gcc, no fast-math, no FMA contraction)."""
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def load(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    L = ctypes.CDLL(path)
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.orc_block_bytes.argtypes = [i32]
    L.orc_block_values.argtypes = [i32]
    L.orc_act_type.argtypes = [i32]
    L.orc_f32_to_f16.argtypes = [ctypes.c_float]
    L.orc_f32_to_f16.restype = ctypes.c_uint16
    L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_f16_to_f32.restype = ctypes.c_float
    for name in ("orc_quantize_q8_0", "orc_quantize_q8_K", "orc_quantize_q4_0",
                 "orc_quantize_q4_K", "orc_quantize_q6_K", "orc_quantize_q2_K", "orc_quantize_q4_1",
                 "orc_quantize_q5_0", "orc_quantize_q5_1", "orc_quantize_q5_K"):
        getattr(L, name).argtypes = [p, p, i64]
        getattr(L, name).restype = None
    L.orc_dequantize.argtypes = [i32, p, p, i64]
    L.orc_dequantize.restype = None
    L.orc_codes.argtypes = [i32, p, p, i64]
    L.orc_codes.restype = None
    L.orc_q4_K_unpack_scales.argtypes = [p, p, p]
    L.orc_q4_K_unpack_scales.restype = None
    L.orc_blocksums_row.argtypes = [i32, p, p, i64, p]
    L.orc_blocksums_row.restype = None
    L.orc_dot_row.argtypes = [i32, p, p, i64]
    L.orc_dot_row.restype = ctypes.c_float
    L.orc_dot_row_exact.argtypes = [i32, p, p, i64]
    L.orc_dot_row_exact.restype = ctypes.c_double
    L.orc_dot_row_bruteforce.argtypes = [i32, p, p, i64]
    L.orc_dot_row_bruteforce.restype = ctypes.c_double
    L.orc_matmul.argtypes = [i32, p, p, p, i64, i64, i64, i32]
    L.orc_blocksums.argtypes = [i32, p, p, p, i64, i64, i64]
    L.orc_blocksums.restype = None
    L.orc_matmul_exact.argtypes = [i32, p, p, p, i64, i64, i64, i32]
    L.orc_matmul_exact.restype = None
    L.orc_rmsnorm.argtypes = [p, p, ctypes.c_float, p, i64, i64]
    L.orc_rmsnorm.restype = None
    L.orc_kv_row_bytes.argtypes = [i32]
    L.orc_kv_quantize.argtypes = [p, p, i64, i32]
    L.orc_kv_quantize.restype = None
    L.orc_kv_scores.argtypes = [p, p, p, i32, i32, i64, i32, ctypes.c_float]
    L.orc_kv_scores.restype = None
    L.orc_kv_wsum.argtypes = [p, p, p, i32, i32, i64, i32]
    L.orc_kv_wsum.restype = None
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
        return _lib


def _t(wtype) -> int:
    return TYPES[wtype] if isinstance(wtype, str) else int(wtype)


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def block_bytes(t) -> int:
    return lib().orc_block_bytes(_t(t))


def block_values(t) -> int:
    return lib().orc_block_values(_t(t))


def act_type(wtype) -> int:
    return lib().orc_act_type(_t(wtype))


def row_bytes(t, K: int) -> int:
    return (K // block_values(t)) * block_bytes(t)


def f32_to_f16_bits(x: float) -> int:
    return int(lib().orc_f32_to_f16(ctypes.c_float(x)))


def f16_bits_to_f32(h: int) -> float:
    return float(lib().orc_f16_to_f32(ctypes.c_uint16(h)))


def quantize(t, x: np.ndarray) -> np.ndarray:
    """Quantize a float32 [rows, K] (or [K]) array; returns uint8 [rows, row_bytes]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    rows, K = x2.shape
    t = _t(t)
    if K % block_values(t):
        raise ValueError("K must be a multiple of the block size")
    out = np.zeros((rows, row_bytes(t, K)), dtype=np.uint8)
    fn = {Q8_0: "orc_quantize_q8_0", Q8_K: "orc_quantize_q8_K", Q4_0: "orc_quantize_q4_0",
          Q4_K: "orc_quantize_q4_K", Q6_K: "orc_quantize_q6_K", Q2_K: "orc_quantize_q2_K",
          Q4_1: "orc_quantize_q4_1", Q5_0: "orc_quantize_q5_0", Q5_1: "orc_quantize_q5_1",
          Q5_K: "orc_quantize_q5_K"}[t]
    getattr(lib(), fn)(_ptr(x2), _ptr(out), rows * K)
    return out


def dequantize(t, q: np.ndarray, K: int) -> np.ndarray:
    """Exact dequantized values (float64) of a uint8 [rows, row_bytes] array."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    rows = q.size // row_bytes(t, K)
    out = np.zeros((rows, K), dtype=np.float64)
    lib().orc_dequantize(_t(t), _ptr(q), _ptr(out), rows * K)
    return out


def get_rows(t, W: np.ndarray, ids, K: int) -> np.ndarray:
    """The embedding lookup ([minfer] s3.2, "The embedding 'matmul'"): for each token id, that row
    of the quantized matrix dequantized block by block, exact (float64).  An id outside the matrix
    is an error here; the device entry point writes a zero row and reports it."""
    rb = row_bytes(t, K)
    W = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1, rb)
    ids = np.asarray(ids, dtype=np.int64)
    if ids.size and (ids.min() < 0 or ids.max() >= W.shape[0]):
        raise IndexError("token id outside the matrix")
    return dequantize(t, W[ids], K)


def codes(t, q: np.ndarray, K: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    rows = q.size // row_bytes(t, K)
    out = np.zeros((rows, K), dtype=np.int32)
    lib().orc_codes(_t(t), _ptr(q), _ptr(out), rows * K)
    return out


def q4_K_scales(block6: bytes):
    b = np.frombuffer(bytes(block6), dtype=np.uint8).copy()
    sc = np.zeros(8, dtype=np.int32)
    mn = np.zeros(8, dtype=np.int32)
    lib().orc_q4_K_unpack_scales(_ptr(b), _ptr(sc), _ptr(mn))
    return sc, mn


def matmul(wtype, W: np.ndarray, xq: np.ndarray, M: int, N: int, K: int, nthreads: int = 1) -> np.ndarray:
    """y[M, N] float32 with the pages' fp32 fold, rows split over nthreads."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    at = act_type(wtype)
    assert W.size == N * row_bytes(wtype, K) and xq.size == M * row_bytes(at, K)
    out = np.zeros((M, N), dtype=np.float32)
    lib().orc_matmul(_t(wtype), _ptr(W), _ptr(xq), _ptr(out), M, N, K, nthreads)
    return out


def matmul_exact(wtype, W, xq, M, N, K, bruteforce=False) -> np.ndarray:
    """Diagnostics in float64: the factorized sum (default) or the brute-force dequantized dot."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    out = np.zeros((M, N), dtype=np.float64)
    lib().orc_matmul_exact(_t(wtype), _ptr(W), _ptr(xq), _ptr(out), M, N, K, int(bruteforce))
    return out


def blocksums_per_row(wtype, K: int) -> int:
    return K // 32 if act_type(wtype) == Q8_0 else 2 * (K // 256)


def blocksums(wtype, W, xq, M, N, K) -> np.ndarray:
    """int32 [M, N, per] exact block sums (K-quants: value, min pairs)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    per = blocksums_per_row(wtype, K)
    out = np.zeros((M, N, per), dtype=np.int32)
    lib().orc_blocksums(_t(wtype), _ptr(W), _ptr(xq), _ptr(out), M, N, K)
    return out


def dot_row(wtype, wrow, xrow, K) -> float:
    wrow = np.ascontiguousarray(wrow, dtype=np.uint8)
    xrow = np.ascontiguousarray(xrow, dtype=np.uint8)
    return float(lib().orc_dot_row(_t(wtype), _ptr(wrow), _ptr(xrow), K))


# ---- the Q8 KV cache ([krafla] "Architecture", Attention: "Q8 cache")
def kv_row_bytes(hd: int) -> int:
    """Bytes of one quantized head vector: f32 scale + hd int8 codes."""
    return int(lib().orc_kv_row_bytes(hd))


def kv_quantize(x: np.ndarray, hd: int) -> np.ndarray:
    """f32 [..., hd] head vectors -> uint8 [rows, 4 + hd] (f32 d, int8 codes), the activations' rule."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, hd)
    out = np.zeros((x.shape[0], kv_row_bytes(hd)), dtype=np.uint8)
    lib().orc_kv_quantize(_ptr(x), _ptr(out), x.shape[0], hd)
    return out


def kv_scores(q8: np.ndarray, k8: np.ndarray, Hq: int, Hkv: int, P: int, hd: int, scale: float = 1.0) -> np.ndarray:
    """f32 [Hq, P]: ((dq * dk) * isum) * scale, query head h against KV head h // (Hq // Hkv);
    k8 holds row (p, kvh) at index p * Hkv + kvh."""
    q8 = np.ascontiguousarray(q8, dtype=np.uint8)
    k8 = np.ascontiguousarray(k8, dtype=np.uint8)
    assert q8.size == Hq * kv_row_bytes(hd) and k8.size >= P * Hkv * kv_row_bytes(hd) and Hq % Hkv == 0
    out = np.zeros((Hq, P), dtype=np.float32)
    lib().orc_kv_scores(_ptr(q8), _ptr(k8), _ptr(out), Hq, Hkv, P, hd, ctypes.c_float(scale))
    return out


def kv_wsum(w: np.ndarray, v8: np.ndarray, Hq: int, Hkv: int, P: int, hd: int) -> np.ndarray:
    """float64 [Hq, hd]: sum_p w[h, p] * dv[p, kvh] * v[p, kvh, :], exact up to binary64 rounding."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    v8 = np.ascontiguousarray(v8, dtype=np.uint8)
    assert w.size == Hq * P and v8.size >= P * Hkv * kv_row_bytes(hd) and Hq % Hkv == 0
    out = np.zeros((Hq, hd), dtype=np.float64)
    lib().orc_kv_wsum(_ptr(w), _ptr(v8), _ptr(out), Hq, Hkv, P, hd)
    return out


# ---- RMSNorm ahead of the quantizer ([krafla] "Architecture", "Data flow for one token")
def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """f32 [M, K]: (x * s) * w with s = 1/sqrt(ss/K + eps) in f32, ss = sum of x^2 taken left to
    right in binary64 and rounded once to f32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    M, K = x2.shape
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(-1)
    assert w.size == K
    out = np.zeros((M, K), dtype=np.float32)
    lib().orc_rmsnorm(_ptr(x2), _ptr(w), ctypes.c_float(eps), _ptr(out), M, K)
    return out
