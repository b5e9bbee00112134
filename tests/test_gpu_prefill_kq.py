"""The K-quant prefill (qmm_matmul_q4_K / q6_K / q2_K) against the CPU oracle.

Shapes on the tensor-core path (K a multiple of 2048, M >= 8) span several 128 x 128 tiles with
ragged edges in both directions; the others take one matvec per token.  The bar: each token's
output row within 1e-5 of its L2 norm."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
import block_quantized_weight_q8_gb300 as qmm  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 1e-5
KQ = ["q4_K", "q6_K", "q2_K", "q5_K"]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("these tests need a CUDA GPU")
    qmm.build()
    qmm.load()
    yield
    assert qmm.qmm_device_status(clear=True) == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_rows_close(y, ref, tol=TOL):
    y = np.asarray(y, dtype=np.float64).reshape(ref.shape)
    ref = np.asarray(ref, dtype=np.float64)
    norm = np.linalg.norm(ref, axis=-1, keepdims=True)
    err = np.abs(y - ref)
    bad = err > tol * norm + 1e-30
    assert not bad.any(), "max err/norm %.3g at %s" % ((err / np.maximum(norm, 1e-30)).max(),
                                                     np.argwhere(bad)[:3].tolist())


def inputs(wtype, M, N, K, seed):
    w = workloads.weights_f32(N, K, seed, row_jitter=True)
    x = workloads.activations_f32(M, K, seed + 1)
    return oracle.quantize(wtype, w), oracle.quantize("q8_K", x), x


@pytest.mark.parametrize("wtype", KQ)
@pytest.mark.parametrize("M,N,K", [(8, 128, 2048), (130, 390, 2048), (17, 300, 4096), (256, 129, 4096),
                                   (3, 77, 1024), (9, 50, 768)])
def test_matmul_kq_matches_oracle(wtype, M, N, K):
    W, X, _ = inputs(wtype, M, N, K, seed=11000 + M + N)
    ref = oracle.matmul(wtype, W, X, M, N, K, nthreads=8)
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    qmm.matmul(wtype, dev(W), dev(X), Y, M, N, K)
    assert_rows_close(host(Y), ref)


@pytest.mark.parametrize("wtype", KQ)
def test_linear_kq_many_tokens(wtype):
    """qmm_linear_<k-quant> with M >= 8 quantizes all rows, then runs the tensor-core prefill."""
    M, N, K = 40, 200, 4096
    W, X, x = inputs(wtype, M, N, K, seed=12000)
    ref = oracle.matmul(wtype, W, X, M, N, K, nthreads=8)
    xrb = qmm.qmm_row_bytes("q8_K", K)
    scratch = torch.empty(M * xrb, dtype=torch.uint8, device="cuda")
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    qmm.linear(wtype, dev(W), dev(x), scratch, scratch.numel(), Y, M, N, K)
    assert np.array_equal(host(scratch), X.reshape(-1))
    assert_rows_close(host(Y), ref)


@pytest.mark.parametrize("wtype,N,K", [("q4_K", 4096, 4096), ("q6_K", 4096, 12288), ("q2_K", 12288, 4096),
                                       ("q5_K", 12288, 4096)])
def test_full_size_kq_prefill_sampled(wtype, N, K):
    """M = 512 at the layer's shapes; rows and tokens sampled for the oracle."""
    M = 512
    W, X, _ = inputs(wtype, M, N, K, seed=13000 + N)
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    qmm.matmul(wtype, dev(W), dev(X), Y, M, N, K)
    got = host(Y)
    g = np.random.default_rng(N)
    tokens = np.unique(np.concatenate([[0, M - 1], g.integers(0, M, 4)]))
    for t in tokens:
        ref = oracle.matmul(wtype, W, X.reshape(M, -1)[t:t + 1], 1, N, K, nthreads=16)[0]
        assert_rows_close(got[t], ref)
