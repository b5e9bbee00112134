"""RMSNorm fused ahead of the quantizer ([krafla] "Architecture", "Data flow for one token":
h = rmsnorm(x) ; qa = quantize_q8(h)) on the GPU against the CPU oracle: the quantized normed
rows bit-exact (both sides sum the squares in the same fixed order), the products within 1e-5
of each token row's L2 norm."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
import block_quantized_weight_q8_gb300 as qmm  # noqa: E402

pytestmark = pytest.mark.gpu
TOL = 1e-5


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


def act_name(wtype):
    return "q8_0" if wtype in ("q4_0", "q8_0", "q4_1", "q5_0", "q5_1") else "q8_K"


def assert_rows_close(y, ref, tol=TOL):
    y = np.asarray(y, dtype=np.float64).reshape(ref.shape)
    ref = np.asarray(ref, dtype=np.float64)
    norm = np.linalg.norm(ref, axis=-1, keepdims=True)
    bad = np.abs(y - ref) > tol * norm + 1e-30
    assert not bad.any(), (np.abs(y - ref) / np.maximum(norm, 1e-30)).max()


def norm_weight(K, seed):
    return np.random.default_rng(seed).uniform(0.5, 1.5, size=K).astype(np.float32)


@pytest.mark.parametrize("act,M,K,eps", [("q8_0", 1, 4096, 1e-6), ("q8_0", 3, 896, 1e-5), ("q8_0", 2, 96, 0.5),
                                         ("q8_K", 5, 256, 1e-6), ("q8_K", 2, 12288, 1e-6), ("q8_0", 1, 65536, 1e-6),
                                         ("q8_K", 1, 65536, 0.0)])
def test_rmsnorm_quantize_bitexact(act, M, K, eps):
    x = workloads.activations_f32(M, K, seed=900 + K)
    if M >= 3:
        x[1] = 0.0 if eps > 0 else 1.0      # an all-zero row (eps keeps the scale finite)
        x[2] = -0.5                          # a constant row
    w = norm_weight(K, K)
    want = oracle.quantize(act, oracle.rmsnorm(x, w, eps))
    out = torch.empty(want.size, dtype=torch.uint8, device="cuda")
    qmm.qmm_rmsnorm_quantize(act, dev(x), dev(w), eps, out, M, K)
    got = host(out).reshape(want.shape)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5].tolist()


@pytest.mark.parametrize("wtype,Ns,K,M", [("q8_0", (12288,), 4096, 1), ("q4_K", (300, 77, 1024), 4096, 1),
                                          ("q6_K", (257,), 12288, 2), ("q2_K", (129, 64), 1024, 1),
                                          ("q4_0", (64, 33), 896, 3), ("q5_1", (100,), 512, 1),
                                          ("q5_K", (333, 20), 4096, 2), ("q4_K", (512, 300), 4096, 16),
                                          ("q4_0", (512,), 4096, 16), ("q8_0", (300, 77), 2048, 16),
                                          ("q5_1", (130,), 1024, 9)])
def test_linear_norm_matches_oracle(wtype, Ns, K, M):
    """Decode tokens (one fused launch each) and the prefill route (M = 16: norm-quantize all rows,
    then the tensor-core matmul) against the oracle on the same f32 inputs; the scratch holds the
    quantized normed rows."""
    eps = 1e-6
    x = workloads.activations_f32(M, K, seed=950 + K)
    w = norm_weight(K, 7)
    X = oracle.quantize(act_name(wtype), oracle.rmsnorm(x, w, eps))
    Ws, refs = [], []
    for g, N in enumerate(Ns):
        Wq = oracle.quantize(wtype, workloads.weights_f32(N, K, seed=960 + g, row_jitter=True))
        Ws.append(dev(Wq))
        refs.append(oracle.matmul(wtype, Wq, X, M, N, K, nthreads=8))
    ys = [torch.empty(M, N, dtype=torch.float32, device="cuda") for N in Ns]
    sb = M * qmm.qmm_row_bytes(act_name(wtype), K)
    scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
    qmm.qmm_linear_norm(wtype, Ws, Ns, dev(x), dev(w), eps, scratch, sb, ys, M, K)
    assert np.array_equal(host(scratch), X.reshape(-1))
    for g in range(len(Ns)):
        assert_rows_close(host(ys[g]), refs[g])


def test_linear_norm_equals_matvec_on_the_normed_row():
    """The fused launch gives, bit for bit, the plain matvec of the row it stored."""
    wtype, N, K = "q4_K", 4096, 4096
    x = workloads.activations_f32(1, K, seed=990)
    w = norm_weight(K, 8)
    Wd = dev(oracle.quantize(wtype, workloads.weights_f32(N, K, seed=991)))
    sb = qmm.qmm_row_bytes("q8_K", K)
    scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
    y = torch.empty(1, N, dtype=torch.float32, device="cuda")
    qmm.qmm_linear_norm(wtype, [Wd], [N], dev(x), dev(w), 1e-6, scratch, sb, [y], 1, K)
    y2 = torch.empty(N, dtype=torch.float32, device="cuda")
    qmm.matvec(wtype, Wd, scratch, y2, N, K)
    assert np.array_equal(host(y).reshape(-1).view(np.uint32), host(y2).view(np.uint32))
