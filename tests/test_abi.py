"""The C-ABI boundary on the CPU: the library builds, loads, exports every entry point
include/qmm.h declares, and rejects bad arguments on the host before any CUDA call (these
checks run without a GPU).  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

import block_quantized_weight_q8_gb300 as qmm

HEADER = os.path.join(ROOT, "include", "qmm.h")


@pytest.fixture(scope="module")
def lib():
    qmm.build()
    return qmm.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"QMM_API\s+[\w\s\*]+?\b(qmm_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("qmm_quantize_q8_0", "qmm_quantize_q8_K", "qmm_matvec_q4_0", "qmm_matvec_q8_0",
                 "qmm_matvec_q4_K", "qmm_matvec_q6_K", "qmm_matvec_q2_K", "qmm_matmul_q4_0", "qmm_matmul_q4_K",
                 "qmm_matmul_q6_K", "qmm_matmul_q2_K",
                 "qmm_linear_q4_0", "qmm_blocksums", "qmm_status_str", "qmm_row_bytes", "qmm_matvec_q4_1",
                 "qmm_matvec_q5_0", "qmm_matvec_q5_1", "qmm_matvec_q5_K", "qmm_get_rows", "qmm_kv_quantize",
                 "qmm_kv_scores", "qmm_kv_wsum", "qmm_rmsnorm_quantize", "qmm_linear_norm", "qmm_linear_host",
                 "qmm_matmul_q8_0", "qmm_matmul_q4_1", "qmm_matmul_q5_0", "qmm_matmul_q5_1", "qmm_matmul_q5_K"):
        assert want in names
    assert set(names) == set(qmm.SIGNATURES), set(names) ^ set(qmm.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", qmm.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(qmm_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "qmm.h"\nint main(void){return (int)qmm_block_bytes(QMM_Q4_0) - 18;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.dirname(HEADER), str(src)],
                   check=True)


def test_formats(lib):
    sizes = {"q4_0": (18, 32), "q8_0": (34, 32), "q4_K": (144, 256), "q6_K": (210, 256), "q2_K": (84, 256),
             "q8_K": (292, 256), "q4_1": (20, 32), "q5_0": (22, 32), "q5_1": (24, 32), "q5_K": (176, 256)}
    for t, (bb, bv) in sizes.items():
        assert qmm.qmm_block_bytes(t) == bb and qmm.qmm_block_values(t) == bv
    for t in ("q4_1", "q5_0", "q5_1"):
        assert qmm.qmm_act_type(t) == qmm.QMM_Q8_0
    assert qmm.qmm_act_type("q5_K") == qmm.QMM_Q8_K
    assert qmm.qmm_block_bytes(10) == 0
    assert qmm.qmm_row_bytes("q4_0", 896) == 504
    assert qmm.qmm_row_bytes("q8_0", 4096) == 4352
    assert qmm.qmm_row_bytes("q4_K", 4096) == 16 * 144
    assert qmm.qmm_row_bytes("q4_K", 4000) == 0
    assert qmm.qmm_block_bytes(99) == 0
    assert qmm.qmm_act_type("q4_0") == qmm.QMM_Q8_0 and qmm.qmm_act_type("q6_K") == qmm.QMM_Q8_K
    assert qmm.qmm_act_type(99) == -1
    for s in range(8):
        assert lib.qmm_status_str(s)
    assert lib.qmm_status_str(1234) == b"unknown status"


# Host-side validation: every one of these returns before any CUDA call.
A = 1 << 20          # a fake, 16-byte aligned address that is never dereferenced
U = A + 4            # a fake misaligned address


@pytest.mark.parametrize("name", ["qmm_matvec_q4_0", "qmm_matvec_q8_0", "qmm_matvec_q4_K", "qmm_matvec_q6_K",
                                  "qmm_matvec_q2_K"])
def test_matvec_rejects_bad_arguments(lib, name):
    f = getattr(lib, name)
    K = 256
    assert f(None, A, A, 8, K, None) == 1          # NULL
    assert f(A, None, A, 8, K, None) == 1
    assert f(A, A, None, 8, K, None) == 1
    assert f(A, A, A, 0, K, None) == 2             # N < 1
    assert f(A, A, A, 8, 0, None) == 2             # K < 1
    assert f(A, A, A, 8, K + 16, None) == 2        # K not a multiple of the block
    assert f(A, A, A, 8, 65536 + 256, None) == 2   # K above the limit
    assert f(A, A, A, 1 << 31, K, None) == 2       # N above the limit
    assert f(U, A, A, 8, K, None) == 4             # misaligned
    assert f(A, U, A, 8, K, None) == 4
    assert f(A, A, U, 8, K, None) == 4


def test_quantizers_reject_bad_arguments(lib):
    for name, bv in (("qmm_quantize_q8_0", 32), ("qmm_quantize_q8_K", 256), ("qmm_quantize_q4_0", 32),
                     ("qmm_quantize_q4_K", 256), ("qmm_quantize_q6_K", 256), ("qmm_quantize_q2_K", 256)):
        f = getattr(lib, name)
        assert f(None, A, 1, bv, None) == 1
        assert f(A, None, 1, bv, None) == 1
        assert f(A, A, 0, bv, None) == 2
        assert f(A, A, 1, bv + 16, None) == 2
        assert f(U, A, 1, bv, None) == 4


def test_linear_rejects_bad_arguments(lib):
    f = lib.qmm_linear_q4_K
    need = 3 * qmm.qmm_row_bytes("q8_K", 512)
    assert f(A, A, A, need - 1, A, 3, 64, 512, None) == 5      # scratch too small
    assert f(A, A, None, need, A, 3, 64, 512, None) == 1
    assert f(A, A, A, need, A, 3, 64, 500, None) == 2
    assert f(A, A, U, need, A, 3, 64, 512, None) == 4
    g = lib.qmm_linear_q4_0
    assert g(A, A, A, 34 * 8 - 1, A, 1, 64, 256, None) == 5


def test_linear_group_rejects_bad_arguments(lib):
    import ctypes
    f = lib.qmm_linear_group
    W = (ctypes.c_void_p * 2)(A, A)
    N = (ctypes.c_int64 * 2)(64, 32)
    Y = (ctypes.c_void_p * 2)(A, A)
    need = 2 * qmm.qmm_row_bytes("q8_K", 512)
    args = lambda wt, G, w, n, y, sb, M, K: f(wt, G, ctypes.cast(w, ctypes.c_void_p), ctypes.cast(n, ctypes.c_void_p),
                                               A, A, sb, ctypes.cast(y, ctypes.c_void_p), M, K, None)
    assert args(qmm.QMM_Q4_K, 2, W, N, Y, need - 1, 2, 512) == 5          # scratch too small
    assert args(qmm.QMM_Q4_K, 0, W, N, Y, need, 2, 512) == 2              # no matrices
    assert args(qmm.QMM_Q4_K, 9, W, N, Y, need, 2, 512) == 2              # more than 8
    assert args(qmm.QMM_Q8_K, 2, W, N, Y, need, 2, 512) == 3              # not a weight type
    assert args(qmm.QMM_Q4_K, 2, W, N, Y, need, 2, 500) == 2              # K not a multiple of 256
    Wn = (ctypes.c_void_p * 2)(A, None)
    assert args(qmm.QMM_Q4_K, 2, Wn, N, Y, need, 2, 512) == 1             # a NULL matrix
    Nz = (ctypes.c_int64 * 2)(64, 0)
    assert args(qmm.QMM_Q4_K, 2, W, Nz, Y, need, 2, 512) == 2             # an empty matrix
    Yu = (ctypes.c_void_p * 2)(A, U)
    assert args(qmm.QMM_Q4_K, 2, W, N, Yu, need, 2, 512) == 4             # unaligned output


def test_get_rows_rejects_bad_arguments(lib):
    f = lib.qmm_get_rows
    assert f(qmm.QMM_Q8_K, A, A, A, 1, 4, 256, None) == 3     # not a weight type
    assert f(qmm.QMM_Q4_0, None, A, A, 1, 4, 256, None) == 1
    assert f(qmm.QMM_Q4_0, A, A, A, 0, 4, 256, None) == 2
    assert f(qmm.QMM_Q4_K, A, A, A, 1, 4, 128, None) == 2
    assert f(qmm.QMM_Q4_0, A, A + 2, A, 1, 4, 256, None) == 4  # ids not 4-byte aligned
    assert f(qmm.QMM_Q4_0, A, A, U, 1, 4, 256, None) == 4


def test_linear_host_rejects_bad_arguments(lib):
    f = lib.qmm_linear_host
    need = qmm.qmm_row_bytes("q8_0", 256)
    assert f(qmm.QMM_Q8_0, A, None, A, A, need, A, A, 1, 64, 256, None) == 1   # no host x
    assert f(qmm.QMM_Q8_0, A, A, A, A, need, A, None, 1, 64, 256, None) == 1   # no host y
    assert f(qmm.QMM_Q8_0, A, A, A, A, need, A, A, 1, 64, 100, None) == 2
    assert f(qmm.QMM_Q8_K, A, A, A, A, need, A, A, 1, 64, 256, None) in (2, 3)


def test_norm_calls_reject_bad_arguments(lib):
    f = lib.qmm_rmsnorm_quantize
    e = ctypes.c_float(1e-6)
    assert f(qmm.QMM_Q4_0, A, A, e, A, 1, 256, None) == 3     # not an activation type
    assert f(qmm.QMM_Q8_0, A, None, e, A, 1, 256, None) == 1
    assert f(qmm.QMM_Q8_K, A, A, e, A, 1, 96, None) == 2
    assert f(qmm.QMM_Q8_0, A, A, e, A, 1, 131072, None) == 2  # beyond the 65536 limit
    assert f(qmm.QMM_Q8_0, A, U, e, A, 1, 256, None) == 4
    W = (ctypes.c_void_p * 2)(A, A)
    N = (ctypes.c_int64 * 2)(64, 32)
    Y = (ctypes.c_void_p * 2)(A, A)
    g = lib.qmm_linear_norm
    need = 2 * qmm.qmm_row_bytes("q8_K", 512)
    assert g(qmm.QMM_Q4_K, 2, W, N, A, None, e, A, need, Y, 2, 512, None) == 1
    assert g(qmm.QMM_Q4_K, 2, W, N, A, U, e, A, need, Y, 2, 512, None) == 4
    assert g(qmm.QMM_Q4_K, 2, W, N, A, A, e, A, need - 1, Y, 2, 512, None) == 5
    assert g(qmm.QMM_Q4_K, 9, W, N, A, A, e, A, need, Y, 2, 512, None) == 2
    assert g(qmm.QMM_Q8_K, 2, W, N, A, A, e, A, need, Y, 2, 512, None) == 3


def test_kv_cache_calls_reject_bad_arguments(lib):
    assert qmm.qmm_kv_row_bytes(64) == 68 and qmm.qmm_kv_row_bytes(128) == 132
    assert qmm.qmm_kv_row_bytes(72) == 0 and qmm.qmm_kv_row_bytes(512) == 0 and qmm.qmm_kv_row_bytes(0) == 0
    q = lib.qmm_kv_quantize
    assert q(None, A, 4, 64, None) == 1
    assert q(A, A, 0, 64, None) == 2
    assert q(A, A, 4, 60, None) == 2
    assert q(A + 2, A, 4, 64, None) == 4
    s = lib.qmm_kv_scores
    f = ctypes.c_float(0.125)
    assert s(A, A, None, 32, 8, 100, 128, f, None) == 1
    assert s(A, A, A, 32, 6, 100, 128, f, None) == 2    # Hq not a multiple of Hkv
    assert s(A, A, A, 32, 2, 100, 128, f, None) == 2    # 16 query heads per KV head
    assert s(A, A, A, 32, 8, 0, 128, f, None) == 2
    assert s(A, A, A, 32, 8, 100, 120, f, None) == 2
    assert s(A, A + 1, A, 32, 8, 100, 128, f, None) == 4
    need = qmm.qmm_kv_wsum_scratch_bytes(32, 300, 128)
    assert need == 32 * 10 * 128 * 4                           # 32-position chunks
    w = lib.qmm_kv_wsum
    assert w(A, A, A, None, need, 32, 8, 300, 128, None) == 1
    assert w(A, A, A, A, need - 4, 32, 8, 300, 128, None) == 5
    assert w(A, A, A, A + 4, need, 32, 8, 300, 128, None) == 4  # scratch must be 16-byte aligned
    assert w(A, A, A, A, need, 32, 8, 300, 100, None) == 2


def test_matmul_and_blocksums_reject_bad_arguments(lib):
    assert lib.qmm_matmul_q4_0(A, A, A, 0, 64, 256, None) == 2
    assert lib.qmm_matmul_q4_0(A, A, None, 4, 64, 256, None) == 1
    assert lib.qmm_matmul_q4_0(A, U, A, 4, 64, 256, None) == 4
    assert lib.qmm_matmul_q4_0(A, A, A, 4, 64, 48, None) == 2
    for f in (lib.qmm_matmul_q8_0, lib.qmm_matmul_q4_1, lib.qmm_matmul_q5_0, lib.qmm_matmul_q5_1):
        assert f(A, A, A, 0, 64, 256, None) == 2
        assert f(None, A, A, 8, 64, 256, None) == 1
        assert f(A, U, A, 8, 64, 256, None) == 4
        assert f(A, A, A, 8, 64, 48, None) == 2
    for f in (lib.qmm_matmul_q4_K, lib.qmm_matmul_q6_K, lib.qmm_matmul_q2_K, lib.qmm_matmul_q5_K):
        assert f(A, A, A, 0, 64, 2048, None) == 2
        assert f(A, A, None, 8, 64, 2048, None) == 1
        assert f(A, U, A, 8, 64, 2048, None) == 4
        assert f(A, A, A, 8, 64, 1000, None) == 2
    assert lib.qmm_blocksums(10, A, A, A, 1, 1, 256, None) == 3
    assert lib.qmm_blocksums(qmm.QMM_Q8_K, A, A, A, 1, 1, 256, None) == 3   # not a weight type
    assert lib.qmm_blocksums(qmm.QMM_Q4_K, A, A, A, 1, 1, 128, None) == 2


def test_binding_raises(lib):
    with pytest.raises(qmm.QmmError) as e:
        qmm.qmm_matvec_q4_0(0, A, A, 8, 256, stream=0)
    assert e.value.status == 1 and "NULL" in str(e.value)
