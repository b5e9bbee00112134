"""qmm_linear_noalloc: the quantize-and-multiply call for callers that cannot give the library a
device workspace (for example a plugin that only receives its input and output buffers from the
application that owns the device memory, or a loop that must never call cudaMalloc).  It keeps the
quantized activation in the library's own fixed 1 MiB device array instead.

Checked through the C ABI on two calls in a row: bit for bit against qmm_linear_<wtype> (the call
that takes a caller workspace and runs the same kernels), and against the CPU oracle within the
tolerance the other GPU tests use.  The cases cover both routes: a launch per token (M < 8) and the
tensor-core prefill (M >= 8), whose TMA tensor maps are then built over the library's array.  This
file is collected last so a run that stops at the first failure has already run every other test;
it also passes on its own."""
import ctypes

import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
import block_quantized_weight_q8_gb300 as qmm  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("these tests need a CUDA GPU")
    qmm.build()
    return qmm.load()


def _close(y, ref):
    ref = np.asarray(ref, dtype=np.float64)
    norm = np.linalg.norm(ref, axis=-1, keepdims=True)
    assert np.all(np.abs(np.asarray(y, dtype=np.float64).reshape(ref.shape) - ref) <= TOL * norm + 1e-30)


@pytest.mark.parametrize("wtype,M,N,K", [("q8_0", 1, 12288, 4096), ("q4_0", 1, 4864, 896), ("q4_K", 1, 4096, 4096),
                                         ("q6_K", 1, 1024, 12288), ("q2_K", 3, 777, 1024), ("q4_0", 5, 300, 1024),
                                         ("q5_1", 2, 500, 4096), ("q5_K", 1, 4096, 4096),
                                         ("q4_0", 16, 300, 1024), ("q8_0", 8, 500, 4096), ("q4_K", 8, 300, 2048),
                                         ("q6_K", 9, 200, 4096), ("q5_0", 200, 129, 4096),
                                         ("q2_K", 16, 130, 2048), ("q5_K", 8, 200, 4096), ("q4_1", 8, 300, 4096),
                                         ("q5_1", 130, 77, 2048)])
def test_noalloc_matches_linear_twice(lib, wtype, M, N, K):
    """qmm_linear_noalloc against qmm_linear_<w>, bit for bit.  At M >= 8 the K-quant (Q4_K, Q2_K,
    Q5_K, Q6_K), Q4_1 and Q5_1 prefills of qmm_linear_<w> take the activation pre-pass and those
    of qmm_linear_noalloc convert the activation in the kernel: the two paths must agree exactly."""
    act = "q8_0" if wtype in ("q4_0", "q8_0", "q4_1", "q5_0", "q5_1") else "q8_K"
    Wq = oracle.quantize(wtype, workloads.weights_f32(N, K, seed=31, row_jitter=True))
    W = torch.from_numpy(Wq).cuda()
    sb = M * qmm.qmm_row_bytes(act, K)
    assert sb <= 1 << 20
    scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    f = lib.qmm_linear_noalloc
    lin = getattr(lib, "qmm_linear_" + wtype)
    for call in range(2):  # the shared array keeps the previous call's contents: both must be right
        xh = workloads.activations_f32(M, K, seed=100 + call)
        x = torch.from_numpy(xh).cuda()
        y_ref = torch.empty(M, N, dtype=torch.float32, device="cuda")
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert lin(W.data_ptr(), x.data_ptr(), scratch.data_ptr(), sb, y_ref.data_ptr(), M, N, K, stream) == 0
        assert f(qmm.TYPES[wtype], W.data_ptr(), x.data_ptr(), y.data_ptr(), M, N, K, stream) == 0
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32))
        _close(y.cpu().numpy(), oracle.matmul(wtype, Wq, oracle.quantize(act, xh), M, N, K, nthreads=8))
    assert qmm.qmm_device_status(clear=True) == 0


def test_noalloc_rejects_too_many_rows(lib):
    K = 4096
    rows_max = (1 << 20) // qmm.qmm_row_bytes("q8_0", K)
    A = 1 << 20
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.qmm_linear_noalloc(qmm.QMM_Q8_0, A, A, A, rows_max + 1, 64, K, stream) == 5   # QMM_E_SCRATCH
    assert lib.qmm_linear_noalloc(qmm.QMM_Q8_K, A, A, A, 1, 64, K, stream) == 3              # not a weight type
