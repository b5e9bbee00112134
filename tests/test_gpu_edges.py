"""Edge cases of the decode path on the GPU, against the CPU oracle.

The largest K the library accepts (65536: every format's row is cut into segments whose
partial sums meet in shared memory), rows whose last segment is short, rows whose blocks do
not group into 16-byte aligned super-units, and the quantize-inside-the-matvec path of
qmm_linear_* on all of these, with its stored activation row compared byte for byte; the
grouped linear; and the embedding lookup qmm_get_rows."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
import block_quantized_weight_q8_gb300 as qmm  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 1e-5
WTYPES = ["q4_0", "q8_0", "q4_K", "q6_K", "q2_K", "q4_1", "q5_0", "q5_1", "q5_K"]


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
    err = np.abs(y - ref)
    bad = err > tol * norm + 1e-30
    assert not bad.any(), "max err/norm %.3g at %s" % ((err / np.maximum(norm, 1e-30)).max(),
                                                     np.argwhere(bad)[:3].tolist())


def check_matvec_and_linear(wtype, M, N, K, seed):
    w = workloads.weights_f32(N, K, seed, row_jitter=True)
    x = workloads.activations_f32(M, K, seed + 1)
    W = oracle.quantize(wtype, w)
    X = oracle.quantize(act_name(wtype), x)
    ref = oracle.matmul(wtype, W, X, M, N, K, nthreads=8)
    Wd = dev(W)
    xrb = qmm.qmm_row_bytes(act_name(wtype), K)
    # the multiply on quantized rows, one token at a time
    for t in range(M):
        y = torch.empty(N, dtype=torch.float32, device="cuda")
        qmm.matvec(wtype, Wd, dev(X.reshape(M, -1)[t]), y, N, K)
        assert_rows_close(host(y), ref[t])
    # quantize + multiply through the linear entry point
    scratch = torch.empty(M * xrb, dtype=torch.uint8, device="cuda")
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    qmm.linear(wtype, Wd, dev(x), scratch, scratch.numel(), Y, M, N, K)
    assert_rows_close(host(Y), ref)
    assert np.array_equal(host(scratch), X.reshape(-1))


@pytest.mark.parametrize("wtype", WTYPES)
def test_max_k(wtype):
    """K = 65536, the header's limit: 256 units per row for every format."""
    check_matvec_and_linear(wtype, 1, 19, 65536, seed=70)


@pytest.mark.parametrize("wtype,K", [("q8_0", 4128), ("q4_0", 4128), ("q8_0", 4160), ("q4_0", 96),
                                     ("q4_K", 4352), ("q6_K", 4352), ("q2_K", 4352), ("q6_K", 12288),
                                     ("q4_1", 4160), ("q5_0", 4128), ("q5_1", 4096), ("q5_K", 4352)])
def test_short_last_segment(wtype, K):
    """Rows cut into segments with a shorter last one (129 Q8_0 blocks: 16 segments of 8 and one
    of 1; 17 super-blocks: 3 segments of 6, 6, 5), and rows of blocks that do not form aligned
    super-units (K % 256 != 0)."""
    check_matvec_and_linear(wtype, 2, 301, K, seed=80 + K)


@pytest.mark.parametrize("wtype", WTYPES)
def test_one_row_per_cta_and_idle_warps(wtype):
    """Fewer rows than SMs x warps: most warps of most CTAs have no item."""
    K = 256 if wtype in ("q4_K", "q6_K", "q2_K", "q5_K") else 64
    check_matvec_and_linear(wtype, 3, 150, K, seed=90)


def test_linear_token_rows_of_odd_alignment():
    """Q8_0 rows of 34 * 3 bytes: token t's quantized row starts 2 bytes past a 16-byte boundary
    for odd t, so the in-kernel quantizer stores it with 16-bit writes."""
    check_matvec_and_linear("q8_0", 5, 67, 96, seed=95)


@pytest.mark.parametrize("wtype,Ns,K,M", [("q4_K", (300, 77, 1024), 4096, 1), ("q4_K", (4096, 1024, 1024), 4096, 2),
                                          ("q8_0", (129, 4096), 4096, 1), ("q4_0", (64, 33, 5, 700), 896, 3),
                                          ("q6_K", (512, 257), 12288, 1), ("q2_K", (12288,), 4096, 1),
                                          ("q5_1", (64, 33), 896, 2), ("q5_K", (300, 77), 4096, 1),
                                          ("q4_0", (300, 77), 1024, 16), ("q4_K", (300, 77), 2048, 16),
                                          ("q5_0", (64, 33), 512, 9)])
def test_linear_group_matches_oracle_and_linear(wtype, Ns, K, M):
    """qmm_linear_group: every matrix's output equals the oracle within tolerance and qmm_linear_<w> on
    that matrix alone bit for bit; the scratch holds the quantized rows."""
    x = workloads.activations_f32(M, K, seed=100 + K)
    X = oracle.quantize(act_name(wtype), x)
    xrb = qmm.qmm_row_bytes(act_name(wtype), K)
    Ws, refs = [], []
    for g, N in enumerate(Ns):
        W = oracle.quantize(wtype, workloads.weights_f32(N, K, seed=200 + g, row_jitter=True))
        Ws.append(dev(W))
        refs.append(oracle.matmul(wtype, W, X, M, N, K, nthreads=8))
    ys = [torch.empty(M, N, dtype=torch.float32, device="cuda") for N in Ns]
    scratch = torch.empty(M * xrb, dtype=torch.uint8, device="cuda")
    xd = dev(x)
    qmm.qmm_linear_group(wtype, Ws, Ns, xd, scratch, scratch.numel(), ys, M, K)
    assert np.array_equal(host(scratch), X.reshape(-1))
    for g, N in enumerate(Ns):
        got = host(ys[g])
        assert_rows_close(got, refs[g])
        y1 = torch.empty(M, N, dtype=torch.float32, device="cuda")
        qmm.linear(wtype, Ws[g], xd, scratch, scratch.numel(), y1, M, N, K)
        assert np.array_equal(host(y1).view(np.uint32), got.view(np.uint32))


@pytest.mark.parametrize("wtype,N,K", [("q4_0", 300, 896), ("q8_0", 129, 4096), ("q4_K", 77, 4096), ("q6_K", 50, 12288),
                                       ("q2_K", 33, 768), ("q4_1", 40, 896), ("q5_0", 41, 4096), ("q5_1", 9, 96),
                                       ("q5_K", 20, 4096)])
def test_get_rows_bitexact(wtype, N, K):
    """qmm_get_rows equals the oracle's exact dequantized rows rounded once to f32, bit for bit; ids repeat
    and cover the first and last rows."""
    W = oracle.quantize(wtype, workloads.weights_f32(N, K, seed=300 + N, row_jitter=True))
    ids = np.array([0, N - 1, 5 % N, 5 % N, N // 2, 1 % N, N - 2], dtype=np.int32)
    want = oracle.get_rows(wtype, W, ids, K).astype(np.float32)
    out = torch.empty(len(ids), K, dtype=torch.float32, device="cuda")
    qmm.qmm_get_rows(wtype, dev(W), dev(ids), out, len(ids), N, K)
    got = host(out)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), np.argwhere(got != want)[:5].tolist()


def test_get_rows_index_out_of_range_is_reported():
    """An id outside [0, N) gives a zero row and QMM_E_SHAPE from qmm_device_status."""
    N, K = 16, 256
    W = oracle.quantize("q8_0", workloads.weights_f32(N, K, seed=9))
    ids = np.array([3, N, -1], dtype=np.int32)
    out = torch.full((3, K), 7.0, dtype=torch.float32, device="cuda")
    assert qmm.qmm_device_status(clear=True) == 0
    qmm.qmm_get_rows("q8_0", dev(W), dev(ids), out, 3, N, K)
    got = host(out)
    assert np.array_equal(got[0], oracle.get_rows("q8_0", W, [3], K)[0].astype(np.float32))
    assert np.all(got[1:] == 0.0)
    assert qmm.qmm_device_status(clear=True) == 2   # QMM_E_SHAPE


@pytest.mark.parametrize("wtype,M,N,K,pinned", [("q4_K", 2, 300, 4096, True), ("q8_0", 1, 12288, 4096, True),
                                                 ("q4_0", 16, 300, 1024, True), ("q8_0", 1, 70000, 256, True),
                                                 ("q4_K", 2, 300, 4096, False)])
def test_linear_host_matches_linear(wtype, M, N, K, pinned):
    """qmm_linear_host (x in from host memory, the multiply, y out on one stream) gives qmm_linear_<w>'s result
    bit for bit: pinned buffers with a small output take the direct path (the kernels read x and write y in
    host memory), a large output or pageable buffers the copying one."""
    W = dev(oracle.quantize(wtype, workloads.weights_f32(N, K, seed=71)))
    x = workloads.activations_f32(M, K, seed=72)
    x_host = torch.from_numpy(x)
    y_host = torch.full((M, N), float("nan"), dtype=torch.float32)
    if pinned:
        x_host, y_host = x_host.pin_memory(), y_host.pin_memory()
    x_dev = torch.empty(M, K, dtype=torch.float32, device="cuda")
    sb = M * qmm.qmm_row_bytes(act_name(wtype), K)
    scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
    y_dev = torch.empty(M, N, dtype=torch.float32, device="cuda")
    qmm.qmm_linear_host(wtype, W, x_host, x_dev, scratch, sb, y_dev, y_host, M, N, K)
    torch.cuda.synchronize()
    y2 = torch.empty(M, N, dtype=torch.float32, device="cuda")
    qmm.linear(wtype, W, dev(x), scratch, sb, y2, M, N, K)
    assert np.array_equal(y_host.numpy().view(np.uint32), host(y2).view(np.uint32))


# ------------------------------------------------------------------ failure path
def test_bounded_wait_runs_out_and_reports():
    """[krafla] "Architecture", Error handling (status codes, nothing aborts): a wait on an
    mbarrier that nothing arrives at, limited to 1 ms, ends, records QMM_E_TIMEOUT for
    qmm_device_status, and leaves the context usable (a multiply right after is still correct
    and the cleared status reads OK)."""
    assert qmm.qmm_device_status(clear=True) == 0
    qmm.qmm_test_wait_timeout(1_000_000)
    assert qmm.qmm_device_status(clear=False) == 7  # QMM_E_TIMEOUT, still set until cleared
    assert qmm.qmm_device_status(clear=True) == 7
    assert qmm.qmm_device_status(clear=False) == 0
    N, K = 300, 1024
    W = oracle.quantize("q8_0", workloads.weights_f32(N, K, seed=70))
    X = oracle.quantize("q8_0", workloads.activations_f32(1, K, seed=71))
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    qmm.matvec("q8_0", dev(W), dev(X), y, N, K)
    assert_rows_close(host(y), oracle.matmul("q8_0", W, X, 1, N, K))
    assert qmm.qmm_device_status(clear=True) == 0
