"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on the same seeded inputs.

Bar: quantized codes, scales, bsums and int32 block sums bit-exact; fp32 outputs within
1e-5 of the L2 norm of the oracle's output row (per token).  Shapes span several CTA
stages, ragged tails (N not a multiple of the rows per stage, W not a multiple of 16
bytes), the smallest cases (N = 1, K = one block) and the full workload sizes."""
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


def u8(n):
    return torch.empty(int(n), dtype=torch.uint8, device="cuda")


def f32(*shape):
    return torch.empty(*shape, dtype=torch.float32, device="cuda")


def bv(t):
    return 256 if t in ("q4_K", "q6_K", "q2_K", "q8_K", "q5_K") else 32


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


def special_activations(K, seed):
    """Rows with the degenerate cases: zeros, exact ties (amax 127), huge and tiny values."""
    g = np.random.default_rng(seed)
    rows = [np.zeros(K, np.float32)]
    t = np.zeros(K, np.float32)
    t[0::32] = 127.0
    t[1::32] = 2.5
    t[2::32] = -3.5
    t[3::32] = 0.5
    rows.append(t)
    rows.append((g.standard_normal(K) * 1e30).astype(np.float32))
    rows.append((g.standard_normal(K) * 1e-30).astype(np.float32))
    z = g.standard_normal(K).astype(np.float32)
    z[: K // 2] = -0.0
    rows.append(z)
    return np.stack(rows)


# ------------------------------------------------------------------ activation quantizers
@pytest.mark.parametrize("t,M,K", [("q8_0", 1, 32), ("q8_0", 1, 896), ("q8_0", 3, 4096), ("q8_0", 17, 544),
                                   ("q8_0", 512, 4096), ("q8_K", 1, 256), ("q8_K", 1, 4096), ("q8_K", 5, 12288),
                                   ("q8_K", 2, 768)])
def test_activation_quantizer_bitexact(t, M, K):
    x = workloads.activations_f32(M, K, seed=1000 + M + K)
    if M >= 5:
        x[:5] = special_activations(K, seed=K)
    want = oracle.quantize(t, x)
    out = u8(want.size)
    qmm.quantize(t, dev(x), out, M, K)
    got = host(out).reshape(want.shape)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5].tolist()


# ------------------------------------------------------------------ weight quantizers
@pytest.mark.parametrize("t", ["q4_0", "q8_0", "q4_K", "q6_K", "q2_K", "q4_1", "q5_0", "q5_1", "q5_K"])
@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (33, 1024)])
def test_weight_quantizer_bitexact(t, N, K):
    w = workloads.weights_f32(N, K, seed=2000 + N, row_jitter=True)
    if N >= 7:
        w[0] = 0.0                      # all-zero row
        w[1] = 0.013                    # constant row
        w[2, ::2] = -w[2, ::2]
        w[3] *= 1e-6                    # tiny scales (f16 subnormal d)
    want = oracle.quantize(t, w)
    out = u8(want.size)
    qmm.quantize(t, dev(w), out, N, K)
    got = host(out).reshape(want.shape)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5].tolist()


# ------------------------------------------------------------------ block sums
def make_inputs(wtype, M, N, K, seed, jitter=True):
    w = workloads.weights_f32(N, K, seed, row_jitter=jitter)
    x = workloads.activations_f32(M, K, seed)
    return oracle.quantize(wtype, w), oracle.quantize(act_name(wtype), x)


@pytest.mark.parametrize("wtype", WTYPES)
@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (2, 37, 512), (3, 300, 1024), (1, 64, 4096)])
def test_blocksums_bitexact(wtype, M, N, K):
    W, X = make_inputs(wtype, M, N, K, seed=3000 + N)
    want = oracle.blocksums(wtype, W, X, M, N, K)
    s = torch.empty(want.size, dtype=torch.int32, device="cuda")
    qmm.qmm_blocksums(wtype, dev(W), dev(X), s, M, N, K)
    got = host(s).reshape(want.shape)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5].tolist()


# ------------------------------------------------------------------ matvec
MV_SHAPES = [(1, 256), (7, 256), (37, 512), (129, 768), (1000, 1024), (4096, 2048), (515, 4352)]


@pytest.mark.parametrize("wtype", WTYPES)
@pytest.mark.parametrize("N,K", MV_SHAPES)
def test_matvec_matches_oracle(wtype, N, K):
    if K % bv(wtype):
        K = (K // bv(wtype) + 1) * bv(wtype)
    W, X = make_inputs(wtype, 1, N, K, seed=4000 + N + K)
    ref = oracle.matmul(wtype, W, X, 1, N, K, nthreads=8)
    y = f32(N)
    qmm.matvec(wtype, dev(W), dev(X), y, N, K)
    assert_rows_close(host(y), ref)


@pytest.mark.parametrize("wtype,N,K", [("q4_0", 7, 32), ("q4_0", 3, 96), ("q8_0", 5, 32), ("q6_K", 3, 256),
                                       ("q2_K", 1, 256), ("q6_K", 1, 768), ("q4_0", 1, 32), ("q4_1", 3, 32),
                                       ("q5_0", 5, 96), ("q5_1", 1, 32), ("q5_0", 1, 32), ("q5_K", 3, 256)])
def test_matvec_unaligned_tail(wtype, N, K):
    """W of N * row_bytes bytes that is not a multiple of 16: the last bytes take the plain path."""
    W, X = make_inputs(wtype, 1, N, K, seed=5000 + N)
    ref = oracle.matmul(wtype, W, X, 1, N, K)
    y = f32(N)
    qmm.matvec(wtype, dev(W), dev(X), y, N, K)
    assert_rows_close(host(y), ref)


def test_matvec_zero_activation_gives_zero():
    for wtype in WTYPES:
        N, K = 33, 512
        W, _ = make_inputs(wtype, 1, N, K, seed=6)
        X = oracle.quantize(act_name(wtype), np.zeros((1, K), np.float32))
        y = f32(N)
        qmm.matvec(wtype, dev(W), dev(X), y, N, K)
        assert np.all(host(y) == 0.0)


def test_matvec_deterministic():
    for wtype in WTYPES:
        N, K = 4099, 4096
        W, X = make_inputs(wtype, 1, N, K, seed=7)
        Wd, Xd = dev(W), dev(X)
        y1, y2 = f32(N), f32(N)
        qmm.matvec(wtype, Wd, Xd, y1, N, K)
        qmm.matvec(wtype, Wd, Xd, y2, N, K)
        assert np.array_equal(host(y1).view(np.uint32), host(y2).view(np.uint32))


# ------------------------------------------------------------------ linear (quantize + matvec)
@pytest.mark.parametrize("wtype", WTYPES)
@pytest.mark.parametrize("M", [1, 3])
def test_linear_matches_quantize_then_matvec(wtype, M):
    N, K = 777, 1024
    w = workloads.weights_f32(N, K, seed=8, row_jitter=True)
    x = workloads.activations_f32(M, K, seed=9)
    W = oracle.quantize(wtype, w)
    ref = oracle.matmul(wtype, W, oracle.quantize(act_name(wtype), x), M, N, K, nthreads=8)
    sb = M * qmm.qmm_row_bytes(act_name(wtype), K)
    scratch = u8(sb)
    y = f32(M, N)
    qmm.linear(wtype, dev(W), dev(x), scratch, sb, y, M, N, K)
    got = host(y)
    assert_rows_close(got, ref)
    assert np.array_equal(host(scratch), oracle.quantize(act_name(wtype), x).reshape(-1))
    if M == 1:
        y2 = f32(N)
        qmm.matvec(wtype, dev(W), scratch, y2, N, K)
        assert np.array_equal(host(y2).view(np.uint32), got.reshape(-1).view(np.uint32))


# ------------------------------------------------------------------ prefill matmul
@pytest.mark.parametrize("wtype", ["q4_0", "q8_0", "q4_1", "q5_0", "q5_1"])
@pytest.mark.parametrize("M,N,K", [(1, 64, 256), (3, 100, 512), (17, 300, 1024), (128, 256, 4096),
                                   (130, 390, 2048), (8, 129, 256), (255, 17, 768)])
def test_matmul_q_matches_oracle(wtype, M, N, K):
    """The 32-value-block prefill (Q4_0, Q8_0, Q4_1, Q5_0 or Q5_1 weights x Q8_0 rows): several tiles in
    both directions, ragged last tiles of rows and tokens, and the per-token fallback shapes."""
    W, X = make_inputs(wtype, M, N, K, seed=9000 + M)
    ref = oracle.matmul(wtype, W, X, M, N, K, nthreads=8)
    Y = f32(M, N)
    qmm.matmul(wtype, dev(W), dev(X), Y, M, N, K)
    assert_rows_close(host(Y), ref)


@pytest.mark.parametrize("wtype", ["q4_0", "q8_0", "q4_1", "q5_0", "q5_1", "q4_K", "q6_K", "q2_K", "q5_K"])
def test_matmul_deterministic(wtype):
    """Each output element has one owner and a fixed order of operations, so reruns of a prefill are bit
    for bit the same (a stage handed back to the copy engine too early showed up here first)."""
    M, N, K = 256, 390, 2048
    W, X = make_inputs(wtype, M, N, K, seed=6000)
    Wd, Xd = dev(W), dev(X)
    ys = []
    for _ in range(4):
        Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        qmm.matmul(wtype, Wd, Xd, Y, M, N, K)
        ys.append(host(Y).view(np.uint32))
    for y in ys[1:]:
        assert np.array_equal(y, ys[0])
    assert_rows_close(ys[0].view(np.float32), oracle.matmul(wtype, W, X, M, N, K, nthreads=8))


# integer weight ranges whose quantization gives d = 1 (and m = 0) exactly, codes equal to the values,
# given the extremes each block is forced to hold
INT_RANGES = {"q4_0": (-8, 7, (-8,)), "q8_0": (-127, 127, (127, -127)), "q5_0": (-16, 15, (-16,)),
              "q4_1": (0, 15, (0, 15)), "q5_1": (0, 31, (0, 31))}


@pytest.mark.parametrize("wtype", ["q4_0", "q8_0", "q5_0", "q4_1", "q5_1"])
@pytest.mark.parametrize("M,N,K", [(8, 128, 256), (130, 300, 1024)])
def test_matmul_integer_sums_exact(wtype, M, N, K):
    """Integer-valued rows quantize to d = 1 (m = 0) with codes equal to the values (weights: the format's
    code range with its extremes in every block; activations: -127..127 with a +-127 in every block), so
    Y is the plain integer matrix product (at most 1024 * 127 * 127 < 2^24: exact in f32) and must match
    it bit for bit: each block's sum of 32 products is exact on the tensor cores."""
    lo, hi, ext = INT_RANGES[wtype]
    g = np.random.default_rng(77 + M)
    w = g.integers(lo, hi + 1, size=(N, K)).astype(np.float32)
    x = g.integers(-127, 128, size=(M, K)).astype(np.float32)
    for i, e in enumerate(ext):  # the extremes at the start of every block (the first max-|x| wins)
        w[:, i::32] = e
    x[:, ::32] = np.where(g.random((M, K // 32)) < 0.5, 127.0, -127.0)
    w[0, len(ext):] = hi if abs(hi) >= abs(lo) else lo  # the largest block sums, both signs
    x[0, :] = 127.0
    x[1, :] = -127.0
    W = oracle.quantize(wtype, w)
    X = oracle.quantize("q8_0", x)
    assert np.array_equal(oracle.get_rows(wtype, W, np.arange(N, dtype=np.int32), K), w)  # d = 1, codes = values
    want = (x.astype(np.int64) @ w.astype(np.int64).T).astype(np.float32)
    Y = f32(M, N)
    qmm.matmul(wtype, dev(W), dev(X), Y, M, N, K)
    assert np.array_equal(host(Y), want)
    # and through the quantize + multiply entry point, with the GPU quantizer
    Y2 = f32(M, N)
    xrb = qmm.qmm_row_bytes("q8_0", K)
    scratch = u8(M * xrb)
    qmm.linear(wtype, dev(W), dev(x), scratch, scratch.numel(), Y2, M, N, K)
    assert np.array_equal(host(scratch), X.reshape(-1))
    assert np.array_equal(host(Y2), want)


@pytest.mark.parametrize("wtype", ["q8_0", "q4_1", "q5_0", "q5_1"])
@pytest.mark.parametrize("M", [8, 64])
def test_linear_prefill_route(wtype, M):
    """qmm_linear_<w> with M >= 8 quantizes all rows, then runs the prefill: bit for bit the same as
    qmm_quantize_q8_0 followed by qmm_matmul_<w>."""
    N, K = 300, 2048
    W, _ = make_inputs(wtype, 1, N, K, seed=4242)
    x = workloads.activations_f32(M, K, seed=4243)
    Wd, xd = dev(W), dev(x)
    xrb = qmm.qmm_row_bytes("q8_0", K)
    s1, s2 = u8(M * xrb), u8(M * xrb)
    y1, y2 = f32(M, N), f32(M, N)
    qmm.linear(wtype, Wd, xd, s1, s1.numel(), y1, M, N, K)
    qmm.qmm_quantize_q8_0(xd, s2, M, K)
    qmm.matmul(wtype, Wd, s2, y2, M, N, K)
    assert np.array_equal(host(s1), host(s2))
    assert np.array_equal(host(y1).view(np.uint32), host(y2).view(np.uint32))
    assert_rows_close(host(y1), oracle.matmul(wtype, W, oracle.quantize("q8_0", x), M, N, K, nthreads=8))


# ------------------------------------------------------------------ full workload sizes
def _full_matvec(name):
    cfg = workloads.WORKLOADS[name]
    N, K, wtype = cfg["N"], cfg["K"], cfg["wtype"]
    w = workloads.weights_f32(N, K, cfg["seed"])
    x = workloads.activations_f32(1, K, cfg["seed"])
    W = oracle.quantize(wtype, w)
    X = oracle.quantize(act_name(wtype), x)
    ref = oracle.matmul(wtype, W, X, 1, N, K, nthreads=16)
    # the GPU weight quantizer on the same f32 weights gives the same bytes
    Wg = u8(W.size)
    qmm.quantize(wtype, dev(w), Wg, N, K)
    assert np.array_equal(host(Wg), W.reshape(-1))
    y = f32(N)
    sb = qmm.qmm_row_bytes(act_name(wtype), K)
    scratch = u8(sb)
    qmm.linear(wtype, Wg, dev(x), scratch, sb, y, 1, N, K)
    assert_rows_close(host(y), ref)


@pytest.mark.parametrize("name", ["q4_0_matvec_4864x896", "q8_0_matvec_12288x4096", "q2_K_matvec_12288x4096",
                                  "q4_1_matvec_12288x4096", "q5_0_matvec_12288x4096", "q5_1_matvec_12288x4096",
                                  "q5_K_matvec_12288x4096"])
def test_full_size_matvec(name):
    _full_matvec(name)


def test_full_size_layer_set():
    cfg = workloads.WORKLOADS["q4_K_M_layer_4096"]
    for i, (label, wtype, N, K) in enumerate(cfg["matrices"]):
        w = workloads.weights_f32(N, K, cfg["seed"], stream=i, row_jitter=True)
        x = workloads.activations_f32(1, K, cfg["seed"], stream=i)
        W = oracle.quantize(wtype, w)
        X = oracle.quantize("q8_K", x)
        ref = oracle.matmul(wtype, W, X, 1, N, K, nthreads=16)
        y = f32(N)
        qmm.matvec(wtype, dev(W), dev(X), y, N, K)
        assert_rows_close(host(y), ref)


@pytest.mark.parametrize("wtype,M", [("q4_0", 128), ("q4_0", 512), ("q4_0", 2048), ("q8_0", 512), ("q4_1", 512),
                                     ("q5_0", 512), ("q5_1", 512)])
def test_full_size_prefill_sampled(wtype, M):
    cfg = workloads.WORKLOADS["q4_0_prefill_512x12288x4096"]
    N, K = cfg["N"], cfg["K"]
    w = workloads.weights_f32(N, K, cfg["seed"])
    x = workloads.activations_f32(M, K, cfg["seed"])
    W = oracle.quantize(wtype, w)
    X = oracle.quantize("q8_0", x)
    Y = f32(M, N)
    qmm.matmul(wtype, dev(W), dev(X), Y, M, N, K)
    got = host(Y)
    g = np.random.default_rng(M)
    tokens = np.unique(np.concatenate([[0, M - 1], g.integers(0, M, 6)]))
    rows = np.unique(np.concatenate([[0, N - 1], g.integers(0, N, 200)]))
    Wr = W.reshape(N, -1)[rows]
    for t in tokens:
        ref_full = oracle.matmul(wtype, W, X.reshape(M, -1)[t:t + 1], 1, N, K, nthreads=16)[0]
        assert_rows_close(got[t], ref_full)
        ref_rows = oracle.matmul(wtype, Wr, X.reshape(M, -1)[t:t + 1], 1, len(rows), K)[0]
        assert np.array_equal(ref_rows, ref_full[rows])
